"""Device-detected errors: out-of-range inputs and a bounded wait that runs out.
Nothing here faults or hangs the GPU: bad entries are caught before any copy is
issued, and the withheld-tile hook makes a one-second bounded wait give up."""
import numpy as np
import pytest
import torch

import workloads as W
from margins import check
from oracle import core

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _paged_case(g):
    c = W.make_paged(B=3, H=8, Hkv=2, dk=64, dv=64, block_size=16, num_blocks=64, lens=[10, 200, 33], mbps=20,
                     seed=60)
    lens = (c.seq_lens + 1).to(DEV)
    out = torch.empty(3, 8, 64, dtype=torch.bfloat16, device=DEV)
    return c, lens, out


def test_bad_block_table_entry_sets_bounds_error(gpu_lib):
    g = gpu_lib
    assert g.attn_get_device_error() == g.OK
    c, lens, out = _paged_case(g)
    tables = c.tables.clone()
    tables[1, 3] = 64          # one past the pool
    tables[2, 0] = -7
    g.attn_decode_paged(c.q.to(DEV), c.k_pool.to(DEV), c.v_pool.to(DEV), tables.to(DEV), lens, out, c.scale)
    assert g.attn_get_device_error() == g.ERR_DEVICE_BOUNDS
    assert g.attn_get_device_error() == g.OK  # read-and-clear
    # the untouched sequence is still right
    ref = torch.empty_like(out)
    g.attn_decode_paged(c.q.to(DEV), c.k_pool.to(DEV), c.v_pool.to(DEV), c.tables.to(DEV), lens, ref, c.scale)
    assert torch.equal(out[0], ref[0])
    assert g.attn_get_device_error() == g.OK


@pytest.mark.parametrize("bad", [0, -3, 20 * 16 + 1])
def test_bad_length_sets_bounds_error(gpu_lib, bad):
    g = gpu_lib
    c, lens, out = _paged_case(g)
    lens[1] = bad
    g.attn_decode_paged(c.q.to(DEV), c.k_pool.to(DEV), c.v_pool.to(DEV), c.tables.to(DEV), lens, out, c.scale)
    assert g.attn_get_device_error() == g.ERR_DEVICE_BOUNDS
    assert torch.all(out[1] == 0)


def test_append_out_of_range_position_is_skipped(gpu_lib):
    g = gpu_lib
    c = W.make_paged(B=2, H=4, Hkv=2, dk=64, dv=64, block_size=16, num_blocks=8, lens=[3, 5], mbps=2, seed=61)
    kp = c.k_pool.to(DEV)
    before = kp.clone()
    lens = torch.tensor([3, 32], dtype=torch.int32, device=DEV)  # 32 = capacity: no slot
    g.kv_append_paged(c.q.to(DEV), c.k_new.to(DEV), c.v_new.to(DEV), kp, c.v_pool.to(DEV), c.tables.to(DEV),
                      lens, lens, c.theta)
    assert g.attn_get_device_error() == g.ERR_DEVICE_BOUNDS
    assert lens.cpu().tolist() == [4, 32]
    changed = (kp != before).any(dim=-1).nonzero().tolist()
    assert {(blk, r) for blk, _, r in changed} <= {(int(c.tables[0, 0]), 3)}


def test_prefill_offset_past_cache_sets_bounds_error(gpu_lib):
    g = gpu_lib
    c = W.make_prefill(B=1, S=8, H=4, Hkv=2, dk=16, dv=16, dtype=torch.float32, seed=62, S_kv=10, offsets=[5])
    out = torch.empty(1, 8, 4, 16, device=DEV)
    g.attn_prefill_causal(c.q.to(DEV), c.k.to(DEV), c.v.to(DEV), out, c.scale, position_offset=c.offsets.to(DEV))
    assert g.attn_get_device_error() == g.ERR_DEVICE_BOUNDS


def test_withheld_tile_times_out_and_context_survives(gpu_lib):
    g = gpu_lib
    c = W.make_contig(B=1, H=8, Hkv=2, dk=64, dv=64, max_len=100, lens=[100], seed=63)
    args = [t.to(DEV) for t in (c.q, c.k, c.v, c.seq_lens)]
    out = torch.empty(1, 8, 64, dtype=torch.bfloat16, device=DEV)
    prev = g.gqa_debug_withhold_first_tile(True)
    try:
        g.attn_decode_contig(*args, out, c.scale)
    finally:
        g.gqa_debug_withhold_first_tile(prev)
    assert g.attn_get_device_error() == g.ERR_DEVICE_TIMEOUT
    # the context is still usable and the same call now succeeds
    g.attn_decode_contig(*args, out, c.scale)
    assert g.attn_get_device_error() == g.OK
    want = core.decode_contig(W.to_oracle(c.q), W.to_oracle(c.k), W.to_oracle(c.v), [100], c.scale)
    check(float(np.abs(out.float().cpu().numpy() - want).max()), 2e-2, "decode after the timeout")


def _withheld(g, call):
    prev = g.gqa_debug_withhold_first_tile(True)
    try:
        call()
    finally:
        g.gqa_debug_withhold_first_tile(prev)
    return g.attn_get_device_error()


@pytest.mark.parametrize("d", [64, 128])
def test_prefill_tensor_core_withheld_tile_times_out(gpu_lib, d):
    """The tensor-core prefill's first K tile is never loaded: its one-second
    waits give up, the call reports the timeout, and the CTA still releases its
    tensor memory (the next call allocates it again and matches the oracle)."""
    g = gpu_lib
    c = W.make_prefill(B=1, S=200, H=2, Hkv=1, dk=d, dv=d, seed=64)
    q, k, v = c.q.to(DEV), c.k.to(DEV), c.v.to(DEV)
    out = torch.empty(1, 200, 2, d, dtype=torch.bfloat16, device=DEV)
    assert _withheld(g, lambda: g.attn_prefill_causal(q, k, v, out, c.scale)) == g.ERR_DEVICE_TIMEOUT
    for _ in range(2):  # every CTA of the timed-out launch freed its TMEM: these allocate it again
        g.attn_prefill_causal(q, k, v, out, c.scale)
        assert g.attn_get_device_error() == g.OK
    want = core.prefill_causal(W.to_oracle(c.q), W.to_oracle(c.k), W.to_oracle(c.v), c.scale)
    check(float(np.abs(out.float().cpu().numpy() - want).max()), 2e-2, "prefill after the timeout")


def test_mla_absorbed_withheld_tile_times_out_and_pair_drains(gpu_lib):
    """The second CTA of each absorbed-MLA pair never gets its first cache tile:
    it gives up, its peer gives up waiting for the tile maxima it would have
    sent, both let what they sent each other land before leaving, and both free
    their tensor memory. The call reports the timeout; the next call matches
    the oracle."""
    g = gpu_lib
    B, H, L, D_C, D_R = 2, 128, 100, 512, 64
    c = W.make_mla_absorbed(B=B, H=H, max_len=L, lens=[100, 70], seed=65)
    q_abs = torch.empty(B, H, D_C + D_R, dtype=torch.bfloat16, device=DEV)
    g.mla_absorb_q(c.q.to(DEV), c.k_b.to(DEV), q_abs)
    latent, lens = c.latent.to(DEV), c.lens.to(DEV)
    out = torch.empty(B, H, D_C, dtype=torch.bfloat16, device=DEV)
    assert g.attn_get_device_error() == g.OK
    call = lambda: g.attn_decode_mla_absorbed(q_abs, latent, lens, out, c.scale)
    assert _withheld(g, call) == g.ERR_DEVICE_TIMEOUT
    for _ in range(2):
        call()
        assert g.attn_get_device_error() == g.OK
    want = core.decode_mla_absorbed(W.to_oracle(q_abs), W.to_oracle(c.latent), W.to_oracle(c.lens), D_C, c.scale)
    check(float(np.abs(out.float().cpu().numpy() - want).max()), 2e-2, "absorbed MLA after the timeout")
