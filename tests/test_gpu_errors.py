"""Device-detected errors: out-of-range inputs and a bounded wait that runs out.
Nothing here faults or hangs the GPU: bad entries are caught before any copy is
issued, and the withheld-tile hook makes a one-second bounded wait give up."""
import pytest
import torch

import workloads as W

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
    assert torch.isfinite(out.float()).all()
