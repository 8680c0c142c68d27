"""The paged decode entry point that allocates nothing (GPU).

attn_decode_paged_static_workspace serves callers that cannot allocate device
memory -- e.g. a program whose HBM is all reserved up front by another
component, or a plugin without access to its host's allocator. Its split-K
scratch is a fixed array inside the library. This file is collected last so
that a failure here cannot hide any other test; it passes alone in a fresh
process as well as after the rest of the suite.
"""
import numpy as np
import pytest
import torch

import workloads as W
from margins import check
from oracle import core

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _case():
    # several splits per sequence (up to 2600 rows), block size 16, a shuffled pool
    c = W.make_paged(B=6, H=32, Hkv=8, dk=128, dv=128, block_size=16, num_blocks=2000,
                     lens=[0, 15, 1023, 1024, 2047, 2599], mbps=170, seed=90)
    lens = c.seq_lens + 1  # the decode sees history + 1 rows
    return c, lens


def _set_up(g):
    """The documented set-up call: B = 0, which only places the scratch array
    on the current device."""
    q = torch.empty(0, 32, 128, dtype=torch.bfloat16, device=DEV)
    pool = torch.empty(1, 8, 16, 128, dtype=torch.bfloat16, device=DEV)
    g.attn_decode_paged_static_workspace(q, pool, pool, torch.zeros(0, 4, dtype=torch.int32, device=DEV),
                                         torch.zeros(0, dtype=torch.int32, device=DEV), torch.empty_like(q), 0.1)


def test_static_workspace_matches_workspace_call_twice(gpu_lib):
    g = gpu_lib
    _set_up(g)
    c, lens = _case()
    q, kp, vp, tab, dl = c.q.to(DEV), c.k_pool.to(DEV), c.v_pool.to(DEV), c.tables.to(DEV), lens.to(DEV)
    ws = g.decode_workspace(6, 32, 128, 170 * 16)
    assert ws is not None and ws.numel() <= g.STATIC_WORKSPACE_BYTES
    want = torch.empty(6, 32, 128, dtype=torch.bfloat16, device=DEV)
    g.attn_decode_paged(q, kp, vp, tab, dl, want, c.scale, workspace=ws)
    outs = [torch.full_like(want, float("nan")) for _ in range(2)]
    torch.cuda.synchronize()
    free0, alloc0 = torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated()
    for out in outs:  # two calls in a row share the same static scratch
        g.attn_decode_paged_static_workspace(q, kp, vp, tab, dl, out, c.scale)
    torch.cuda.synchronize()
    # nothing was allocated on the device by the two calls
    assert torch.cuda.mem_get_info()[0] == free0 and torch.cuda.memory_allocated() == alloc0
    assert g.attn_get_device_error() == g.OK
    oracle = core.decode_paged(W.to_oracle(c.q), W.to_oracle(c.k_pool), W.to_oracle(c.v_pool),
                               W.to_oracle(c.tables), lens.numpy(), c.scale)
    for out in outs:
        # the same kernels and split rule as the workspace call: the same bits
        assert torch.equal(out, want)
        check(float(np.abs(out.float().cpu().numpy() - oracle).max()), 2e-2, "static-scratch call vs oracle")


def test_static_workspace_rejects_too_large_problem(gpu_lib):
    g = gpu_lib
    c, _ = _case()
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
