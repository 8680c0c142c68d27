"""The paged decode entry point that allocates nothing (GPU).

attn_decode_paged_static_workspace serves callers that cannot allocate device
memory -- e.g. a program whose HBM is all reserved up front by another
component, or a plugin without access to its host's allocator. Its split-K
scratch is a fixed array inside the library. This file is collected last so
that a failure here cannot hide any other test; it passes alone in a fresh
process as well as after the rest of the suite.
"""
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _case():
    # several splits per sequence (up to 2600 rows), block size 16, a shuffled pool
    c = W.make_paged(B=6, H=32, Hkv=8, dk=128, dv=128, block_size=16, num_blocks=2000,
                     lens=[0, 15, 1023, 1024, 2047, 2599], mbps=170, seed=90)
    lens = (c.seq_lens + 1).to(DEV)  # the decode sees history + 1 rows
    return c, lens


def test_static_workspace_matches_workspace_call_twice(gpu_lib):
    g = gpu_lib
    c, lens = _case()
    q, kp, vp, tab = c.q.to(DEV), c.k_pool.to(DEV), c.v_pool.to(DEV), c.tables.to(DEV)
    ws = g.decode_workspace(6, 32, 128, 170 * 16)
    assert ws is not None and ws.numel() <= g.STATIC_WORKSPACE_BYTES
    want = torch.empty(6, 32, 128, dtype=torch.bfloat16, device=DEV)
    g.attn_decode_paged(q, kp, vp, tab, lens, want, c.scale, workspace=ws)
    for _ in range(2):  # two calls in a row share the same static scratch
        out = torch.full_like(want, float("nan"))
        g.attn_decode_paged_static_workspace(q, kp, vp, tab, lens, out, c.scale)
        assert g.attn_get_device_error() == g.OK
        assert (out.float() - want.float()).abs().max().item() <= 2e-2
        assert torch.isfinite(out.float()).all()


def test_static_workspace_rejects_too_large_problem(gpu_lib):
    g = gpu_lib
    c, lens = _case()
    # 256 sequences of up to 32784 rows need ~140 MB of scratch: beyond the fixed size
    need = g.attn_decode_workspace_bytes(256, 32, 128, 2049 * 16)
    assert need > g.STATIC_WORKSPACE_BYTES
    q = torch.empty(256, 32, 128, dtype=torch.bfloat16, device=DEV)
    tables = torch.zeros(256, 2049, dtype=torch.int32, device=DEV)
    with pytest.raises(g.GqaError) as e:
        g.attn_decode_paged_static_workspace(q, c.k_pool.to(DEV), c.v_pool.to(DEV), tables,
                                             torch.ones(256, dtype=torch.int32, device=DEV),
                                             torch.empty_like(q), c.scale)
    assert e.value.status == g.ERR_WORKSPACE
