"""The split-K work list that plan_units_kernel writes into the decode workspace
(GPU): every (item, split) with visible keys exactly once, the full 2048-row
splits first in item order, then the partial splits longest first."""
import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"
SPLIT = 2048
BUCKETS = 64


def test_unit_list_is_complete_and_longest_first(gpu_lib):
    g = gpu_lib
    lens = [100, 2048, 2049, 5000, 4096, 7000, 1, 6143]
    B, H, Hkv, d, L = len(lens), 32, 8, 128, 8192
    c = W.make_contig(B=B, H=H, Hkv=Hkv, dk=d, dv=d, max_len=L, lens=lens, seed=103, device=DEV)
    out = torch.empty(B, H, d, dtype=torch.bfloat16, device=DEV)
    ws = g.decode_workspace(B, H, d, L)
    g.attn_decode_contig(c.q, c.k, c.v, c.seq_lens, out, c.scale, workspace=ws)
    assert g.attn_get_device_error() == g.OK
    raw = ws.cpu().numpy()
    header = raw[:256].view(np.int32)
    total = int(header[1])
    units = raw[256:256 + 8 * total].view(np.int32).reshape(total, 2)
    # items: (sequence, KV head) with the whole group of 4 heads in one item
    items_per_seq = Hkv
    assert units[:, 0].max() < B * items_per_seq
    want = {}
    for b, n in enumerate(lens):
        for kvh in range(Hkv):
            item = b * items_per_seq + kvh
            for s in range((n + SPLIT - 1) // SPLIT):
                want[(item, s)] = min(SPLIT, n - s * SPLIT)
    got = [tuple(u) for u in units.tolist()]
    assert len(got) == len(set(got)) == len(want)
    assert set(got) == set(want)
    rows = [want[u] for u in got]
    n_full = sum(r == SPLIT for r in rows)
    assert all(r == SPLIT for r in rows[:n_full])  # full splits first ...
    assert [u[0] for u in got[:n_full]] == sorted(u[0] for u in got[:n_full])  # ... in item order
    buckets = [((SPLIT - r) * BUCKETS) // SPLIT for r in rows[n_full:]]
    assert buckets == sorted(buckets)  # then the partial ones, longest first
