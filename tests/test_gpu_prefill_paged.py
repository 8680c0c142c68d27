"""Chunked prefill against the paged pool (include/gqa_attn.h, attn_prefill_paged):
new rows at explicit position offsets attend to a history that lives in pool
blocks reached through a block table. Paging changes where rows live and nothing
else (frink-models src/decoder/attn_block.rs, `push_and_attend_row`, paged arm),
so the paged call must equal attn_prefill_causal on the same history bit for bit
-- on the tcgen05 kernel (bf16, d = 64, block gather by TMA) and on the SIMT
kernel alike -- and both must match the oracle."""
import numpy as np
import pytest
import torch

import workloads as W
from margins import check
from oracle import core

pytestmark = pytest.mark.gpu
DEV = "cuda"
TOL = {torch.bfloat16: 2e-2, torch.float32: 1e-4}


def ok(g):
    assert g.attn_get_device_error() == g.OK


def page(c, bs, spare=7, seed=0):
    """Scatter the contiguous history of a prefill case (k, v [B, Hkv, S_kv, d])
    into a pool of bs-row blocks taken from a seeded permutation; entries past a
    sequence's last block are -1. Returns (k_pool, v_pool, tables)."""
    B, Hkv, S_kv, dk = c.k.shape
    dv = c.v.shape[-1]
    nblk = (S_kv + bs - 1) // bs
    nb = B * nblk + spare
    perm = torch.randperm(nb, generator=W.generator(seed + 500)).to(torch.int32)
    kp = W.randn((nb, Hkv, bs, dk), W.generator(seed + 501), c.k.dtype)  # junk outside the history
    vp = W.randn((nb, Hkv, bs, dv), W.generator(seed + 502), c.v.dtype)
    tables = torch.full((B, nblk + 3), -1, dtype=torch.int32)
    at = 0
    for b in range(B):
        used = (int(c.offsets[b]) + c.q.shape[1] + bs - 1) // bs  # blocks holding keys the rows see
        for t in range(used):
            e = int(perm[at])
            at += 1
            tables[b, t] = e
            r = min(bs, S_kv - t * bs)
            kp[e, :, :r] = c.k[b, :, t * bs:t * bs + r]
            vp[e, :, :r] = c.v[b, :, t * bs:t * bs + r]
    return kp, vp, tables


def run_both(g, c, bs, **arms):
    kp, vp, tables = page(c, bs, seed=int(bs))
    B, S, H, _ = c.q.shape
    dv = c.v.shape[-1]
    out_p = torch.empty(B, S, H, dv, dtype=c.q.dtype, device=DEV)
    g.attn_prefill_paged(c.q.to(DEV), kp.to(DEV), vp.to(DEV), tables.to(DEV), out_p, c.scale,
                         position_offset=c.offsets.to(DEV), **arms)
    ok(g)
    out_c = torch.empty_like(out_p)
    g.attn_prefill_causal(c.q.to(DEV), c.k.to(DEV), c.v.to(DEV), out_c, c.scale, position_offset=c.offsets.to(DEV),
                          **arms)
    ok(g)
    return out_p, out_c


def oracle(c, window=0, softcap=0.0, sinks=None, slopes=None):
    base = [int(o) + c.q.shape[1] for o in c.offsets]
    return core.attention_arms(W.to_oracle(c.q), W.to_oracle(c.k), W.to_oracle(c.v), base, c.scale, window, softcap,
                               sinks, slopes)


def err(out, want):
    return np.abs(out.float().cpu().numpy().astype(np.float64) - want).max()


@pytest.mark.parametrize("bs", [8, 16, 32, 128])
def test_tensor_core_paged_equals_contig_bits(gpu_lib, bs):
    """bf16, d = 64: both calls on the tcgen05 kernel; ragged chunk (200 rows =
    two query tiles, the second partial) at offsets inside and across key tiles."""
    g = gpu_lib
    offs = [0, 300, 1000]
    S = 200
    c = W.make_prefill(B=3, S=S, H=14, Hkv=2, dk=64, dv=64, seed=150 + bs, S_kv=S + max(offs) + 5, offsets=offs)
    out_p, out_c = run_both(g, c, bs)
    assert torch.equal(out_p, out_c)
    check(err(out_p, oracle(c)), TOL[torch.bfloat16])


@pytest.mark.parametrize("dtype,d,bs", [(torch.float32, 64, 16), (torch.bfloat16, 128, 16),
                                        (torch.bfloat16, 64, 24)])
def test_simt_paged_equals_contig_and_oracle(gpu_lib, dtype, d, bs):
    """Shapes the tensor-core kernel does not take: f32, d = 128, and a block
    size that does not divide a 128-key tile (bf16 d = 64 contiguous goes to the
    tensor cores then, so the comparison is against the oracle only)."""
    g = gpu_lib
    offs = [0, 37, 900]
    S = 70
    c = W.make_prefill(B=3, S=S, H=8, Hkv=2, dk=d, dv=d, dtype=dtype, seed=160 + d + bs, S_kv=S + max(offs) + 3,
                       offsets=offs)
    out_p, out_c = run_both(g, c, bs)
    if not (dtype == torch.bfloat16 and d == 64):
        assert torch.equal(out_p, out_c)
    check(err(out_p, oracle(c)), TOL[dtype])


def test_paged_prefill_arms(gpu_lib):
    """Window, sinks, softcap and ALiBi with the paged history (SIMT kernel)."""
    g = gpu_lib
    H = 8
    offs = [5, 400]
    S = 48
    c = W.make_prefill(B=2, S=S, H=H, Hkv=2, dk=64, dv=64, seed=170, S_kv=S + 401, offsets=offs)
    rng = np.random.default_rng(171)
    sinks = rng.standard_normal(H).astype(np.float32)
    slopes = np.array([2.0 ** (-8.0 * (h + 1) / H) for h in range(H)], np.float32)
    arms = dict(window=130, softcap=3.0, sinks=torch.from_numpy(sinks).to(DEV),
                alibi_slopes=torch.from_numpy(slopes).to(DEV))
    out_p, out_c = run_both(g, c, 16, **arms)
    assert torch.equal(out_p, out_c)
    check(err(out_p, oracle(c, 130, 3.0, sinks.astype(np.float64), slopes.astype(np.float64))), 2e-2)


def test_decode_step_is_a_one_row_chunk(gpu_lib):
    """seq_q = 1 at offset len - 1 is the decode step: attn_prefill_paged equals
    attn_decode_paged on the same pool within the bf16 tolerance (different
    kernels, so not bit for bit)."""
    g = gpu_lib
    c = W.make_paged(B=4, H=8, Hkv=2, dk=64, dv=64, block_size=16, num_blocks=400, lens=[1, 15, 700, 2100],
                     mbps=140, seed=175)
    lens = c.seq_lens.to(DEV)  # rows present, the query's own included
    out_d = torch.empty(4, 8, 64, dtype=torch.bfloat16, device=DEV)
    g.attn_decode_paged(c.q.to(DEV), c.k_pool.to(DEV), c.v_pool.to(DEV), c.tables.to(DEV), lens, out_d, c.scale,
                        workspace=g.decode_workspace(4, 8, 64, 140 * 16))
    ok(g)
    out_p = torch.empty(4, 1, 8, 64, dtype=torch.bfloat16, device=DEV)
    g.attn_prefill_paged(c.q.view(4, 1, 8, 64).to(DEV), c.k_pool.to(DEV), c.v_pool.to(DEV), c.tables.to(DEV), out_p,
                         c.scale, position_offset=(lens - 1).to(torch.int32))
    ok(g)
    check((out_p[:, 0].float() - out_d.float()).abs().max().item(), 2e-2)


@pytest.mark.parametrize("dtype,dk,dv", [(torch.bfloat16, 64, 64), (torch.float32, 64, 64),
                                         (torch.bfloat16, 128, 128), (torch.bfloat16, 192, 128)])
def test_bad_table_entry_and_offset_are_flagged(gpu_lib, dtype, dk, dv):
    """An out-of-range entry in a block the rows read is skipped and reported; so
    is an offset that puts the chunk past the table's capacity (whose rows are
    written as zeros). Nothing is read out of range. Both kernels, every
    tensor-core width."""
    g = gpu_lib
    offs = [0, 150]
    S = 100
    c = W.make_prefill(B=2, S=S, H=4, Hkv=2, dk=dk, dv=dv, dtype=dtype, seed=180, S_kv=S + 150, offsets=offs)
    kp, vp, tables = page(c, 16, seed=181)
    bad = tables.clone()
    bad[1, 2] = kp.shape[0]  # one past the pool
    out = torch.empty(2, S, 4, dv, dtype=dtype, device=DEV)
    g.attn_prefill_paged(c.q.to(DEV), kp.to(DEV), vp.to(DEV), bad.to(DEV), out, c.scale,
                         position_offset=c.offsets.to(DEV))
    assert g.attn_get_device_error() == g.ERR_DEVICE_BOUNDS
    assert g.attn_get_device_error() == g.OK
    cap = tables.shape[1] * 16
    far = torch.tensor([0, cap - S + 1], dtype=torch.int32, device=DEV)
    g.attn_prefill_paged(c.q.to(DEV), kp.to(DEV), vp.to(DEV), tables.to(DEV), out, c.scale, position_offset=far)
    assert g.attn_get_device_error() == g.ERR_DEVICE_BOUNDS
    assert torch.all(out[1] == 0)


@pytest.mark.parametrize("H,Hkv,d", [(14, 2, 64), (32, 8, 128)])
def test_full_size_chunked_prefill_sampled_rows(gpu_lib, H, Hkv, d):
    """The chunked-prefill workloads the bench times (4 sequences, 2048-row chunks
    at offsets up to 6144, bs = 16; d = 64 at the prefill config's heads, d = 128
    at the decode configs'): sampled rows -- first, last and seeded others of each
    chunk, every head -- against the oracle, each row computed on its own over the
    history gathered from the pool through the table."""
    g = gpu_lib
    q, kp, vp, tables, off, scale = W.make_prefill_paged(H=H, Hkv=Hkv, d=d)
    B, S, H, d = q.shape
    bs = kp.shape[2]
    out = torch.empty(B, S, H, d, dtype=torch.bfloat16, device=DEV)
    g.attn_prefill_paged(q.to(DEV), kp.to(DEV), vp.to(DEV), tables.to(DEV), out, scale,
                         position_offset=off.to(DEV))
    ok(g)
    out = out.cpu()
    rng = np.random.default_rng(190)
    worst = 0.0
    for b in range(B):
        o = int(off[b])
        n = o + S
        blocks = tables[b, :(n + bs - 1) // bs].long()
        k_hist = kp[blocks].permute(1, 0, 2, 3).reshape(1, kp.shape[1], -1, d)[:, :, :n].contiguous()
        v_hist = vp[blocks].permute(1, 0, 2, 3).reshape(1, vp.shape[1], -1, d)[:, :, :n].contiguous()
        for i in sorted({0, S - 1, *rng.integers(0, S, 3).tolist()}):
            want = core.attention_arms(W.to_oracle(q[b:b + 1, i:i + 1].contiguous()), W.to_oracle(k_hist),
                                       W.to_oracle(v_hist), [o + i + 1], scale)
            worst = max(worst, err(out[b:b + 1, i:i + 1], want))
    check(worst, 2e-2)


@pytest.mark.parametrize("dk,dv,bs", [(128, 128, 16), (128, 128, 8), (192, 128, 8), (192, 128, 32)])
def test_tensor_core_paged_wide_heads_equal_contig_bits(gpu_lib, dk, dv, bs):
    """d = 128 and the MLA widths (d_k = 192, d_v = 128) on the tensor cores: a
    key tile is several 64-column blocks per pool block (bs = 8 with d_k = 192
    needs more boxes than a warp has lanes)."""
    g = gpu_lib
    offs = [0, 260]
    S = 150
    c = W.make_prefill(B=2, S=S, H=8, Hkv=2, dk=dk, dv=dv, seed=185 + dk + bs, S_kv=S + max(offs) + 3,
                       offsets=offs)
    out_p, out_c = run_both(g, c, bs)
    assert torch.equal(out_p, out_c)
    check(err(out_p, oracle(c)), TOL[torch.bfloat16])
