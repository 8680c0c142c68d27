"""CUDA path against the fp64 oracle on identical seeded inputs (GPU).

Tolerances: max abs error <= 1e-4 for fp32 inputs, <= 2e-2 for bf16 inputs
(fp32 accumulation; the oracle reads the same bf16 values widened to fp64).
Paged vs contiguous, block permutation and run-to-run results are bit-exact.
"""
import math

import numpy as np
import pytest
import torch

import workloads as W
from margins import check
from oracle import core

pytestmark = pytest.mark.gpu

TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2}
DEV = "cuda"


def maxerr(gpu, want):
    return float(np.abs(gpu.float().cpu().numpy().astype(np.float64) - want).max())


def ok(g):
    assert g.attn_get_device_error() == g.OK


# ---------------------------------------------------------------------------
# tiny fp32: H=4, Hkv=2, d=16, scale 1/4, 8-row prefill, then one decode step

def test_tiny_prefill(gpu_lib):
    g = gpu_lib
    pre, _ = W.make_tiny()
    out = torch.empty(1, 8, 4, 16, device=DEV)
    g.attn_prefill_causal(pre.q.to(DEV), pre.k.to(DEV), pre.v.to(DEV), out, pre.scale)
    want = core.prefill_causal(W.to_oracle(pre.q), W.to_oracle(pre.k)[:, :, :8], W.to_oracle(pre.v)[:, :, :8],
                               pre.scale)
    ok(g)
    check(maxerr(out, want), 1e-4)


def test_tiny_decode_reading_last_prefill_row(gpu_lib):
    """Reading (i): the decode step at cache length 8 is prefill row 7."""
    g = gpu_lib
    pre, _ = W.make_tiny()
    k8, v8 = pre.k[:, :, :8].contiguous(), pre.v[:, :, :8].contiguous()
    out = torch.empty(1, 4, 16, device=DEV)
    g.attn_decode_contig(pre.q[:, 7].contiguous().to(DEV), k8.to(DEV), v8.to(DEV),
                         torch.tensor([8], dtype=torch.int32, device=DEV), out, pre.scale)
    want = core.prefill_causal(W.to_oracle(pre.q), W.to_oracle(k8), W.to_oracle(v8), pre.scale)[:, 7]
    ok(g)
    check(maxerr(out, want), 1e-4)


def test_tiny_decode_appended_ninth_row_contig_and_paged(gpu_lib):
    """Reading (ii): a ninth row is pushed at position 8, then the step attends
    over 9 rows -- contiguous and paged (block size 4, seeded table) give the same
    bits, and both match the last row of a 9-row prefill."""
    g = gpu_lib
    pre, q9 = W.make_tiny()
    lens = torch.tensor([9], dtype=torch.int32, device=DEV)
    out_c = torch.empty(1, 4, 16, device=DEV)
    g.attn_decode_contig(q9.to(DEV), pre.k.to(DEV), pre.v.to(DEV), lens, out_c, pre.scale)
    # paged: 3 blocks of 4 rows at seeded positions of a 7-block pool
    perm = torch.randperm(7, generator=W.generator(5))[:3].to(torch.int32)
    kp = torch.randn(7, 2, 4, 16, generator=W.generator(6))
    vp = torch.randn(7, 2, 4, 16, generator=W.generator(7))
    for blk in range(3):
        n = min(4, 9 - 4 * blk)
        kp[perm[blk], :, :n] = pre.k[0, :, 4 * blk:4 * blk + n]
        vp[perm[blk], :, :n] = pre.v[0, :, 4 * blk:4 * blk + n]
    tables = torch.cat([perm, torch.full((2,), -1, dtype=torch.int32)])[None]
    out_p = torch.empty(1, 4, 16, device=DEV)
    g.attn_decode_paged(q9.to(DEV), kp.to(DEV), vp.to(DEV), tables.to(DEV), lens, out_p, pre.scale)
    ok(g)
    assert torch.equal(out_c, out_p)
    q_all = torch.cat([pre.q[0], q9], 0)[None]  # the new query is row 8 of a 9-row prefill
    want = core.prefill_causal(W.to_oracle(q_all), W.to_oracle(pre.k), W.to_oracle(pre.v), pre.scale)[:, 8]
    check(maxerr(out_c, want), 1e-4)
    want_p = core.decode_paged(W.to_oracle(q9), W.to_oracle(kp), W.to_oracle(vp), W.to_oracle(tables), [9],
                               pre.scale)
    check(maxerr(out_p, want_p), 1e-4)


# ---------------------------------------------------------------------------
# decode, several splits and ragged lengths

@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("H,Hkv,d", [(32, 8, 128), (8, 8, 128), (16, 2, 64), (12, 4, 32), (8, 1, 16),
                                     (6, 3, 128), (4, 2, 256)])
def test_decode_contig(gpu_lib, dtype, H, Hkv, d):
    g = gpu_lib
    # lengths around the 2048-row split boundary and past two of them
    lens = [1, 31, 1024, 2047, 2048, 2049, 4500]
    c = W.make_contig(B=len(lens), H=H, Hkv=Hkv, dk=d, dv=d, max_len=4600, lens=lens, dtype=dtype, seed=20)
    out = torch.empty(len(lens), H, d, dtype=dtype, device=DEV)
    ws = g.decode_workspace(len(lens), H, d, 4600)
    g.attn_decode_contig(c.q.to(DEV), c.k.to(DEV), c.v.to(DEV), c.seq_lens.to(DEV), out, c.scale, workspace=ws)
    ok(g)
    want = core.decode_contig(W.to_oracle(c.q), W.to_oracle(c.k), W.to_oracle(c.v), lens, c.scale)
    check(maxerr(out, want), TOL[dtype])


@pytest.mark.parametrize("bs", [16, 4, 5, 64])
def test_decode_paged_matches_oracle_and_contig_bits(gpu_lib, bs):
    g = gpu_lib
    lens = [1, 16, 17, 1023, 2047, 2048, 2049, 4200]
    B, H, Hkv, d, L = len(lens), 32, 8, 128, 4200
    c = W.make_contig(B=B, H=H, Hkv=Hkv, dk=d, dv=d, max_len=L, lens=lens, seed=21)
    mbps = (L + bs - 1) // bs + 1
    need = sum((n + bs - 1) // bs for n in lens)
    nb = need + 37
    perm = torch.randperm(nb, generator=W.generator(22)).to(torch.int32)
    kp = torch.randn(nb, Hkv, bs, d, generator=W.generator(23)).to(torch.bfloat16)
    vp = torch.randn(nb, Hkv, bs, d, generator=W.generator(24)).to(torch.bfloat16)
    tables = torch.full((B, mbps), -1, dtype=torch.int32)
    at = 0
    for b, n in enumerate(lens):
        for blk in range((n + bs - 1) // bs):
            e = perm[at]
            at += 1
            tables[b, blk] = e
            r = min(bs, n - blk * bs)
            kp[e, :, :r] = c.k[b, :, blk * bs:blk * bs + r]
            vp[e, :, :r] = c.v[b, :, blk * bs:blk * bs + r]
    ws = g.decode_workspace(B, H, d, mbps * bs)
    out_p = torch.empty(B, H, d, dtype=torch.bfloat16, device=DEV)
    g.attn_decode_paged(c.q.to(DEV), kp.to(DEV), vp.to(DEV), tables.to(DEV), c.seq_lens.to(DEV), out_p, c.scale,
                        workspace=ws)
    out_c = torch.empty_like(out_p)
    wsc = g.decode_workspace(B, H, d, L)
    g.attn_decode_contig(c.q.to(DEV), c.k.to(DEV), c.v.to(DEV), c.seq_lens.to(DEV), out_c, c.scale, workspace=wsc)
    ok(g)
    assert torch.equal(out_p, out_c), "paged and contiguous decode must be bit-identical"
    want = core.decode_paged(W.to_oracle(c.q), W.to_oracle(kp), W.to_oracle(vp), W.to_oracle(tables), lens,
                             c.scale)
    check(maxerr(out_p, want), 2e-2)


def test_decode_mla_shared_rot(gpu_lib):
    """MLA shape: group 1, d_k = 128 + 64 with the 64 shared per position; the
    oracle copies k_rot into every head (the naive form)."""
    g = gpu_lib
    c = W.make_mla(B=2, H=16, cache_len=1500, seed=25)
    c.seq_lens = torch.tensor([1500, 700], dtype=torch.int32)
    out = torch.empty(2, 16, 128, dtype=torch.bfloat16, device=DEV)
    ws = g.decode_workspace(2, 16, 128, 1500)
    g.attn_decode_contig(c.q.to(DEV), c.k.to(DEV), c.v.to(DEV), c.seq_lens.to(DEV), out, c.scale, workspace=ws,
                         k_rot_shared=c.k_rot.to(DEV))
    ok(g)
    want = core.decode_mla_naive(W.to_oracle(c.q), W.to_oracle(c.k), W.to_oracle(c.k_rot), W.to_oracle(c.v),
                                 [1500, 700], c.scale)
    check(maxerr(out, want), 2e-2)


# ---------------------------------------------------------------------------
# prefill

@pytest.mark.parametrize("dtype,H,Hkv,d,S,off", [
    (torch.bfloat16, 14, 2, 64, 300, 0), (torch.float32, 14, 2, 64, 200, 0), (torch.bfloat16, 8, 2, 128, 150, 0),
    (torch.float32, 4, 4, 32, 70, 33), (torch.bfloat16, 6, 2, 64, 129, 100), (torch.float32, 4, 1, 16, 1, 50)])
def test_prefill(gpu_lib, dtype, H, Hkv, d, S, off):
    g = gpu_lib
    c = W.make_prefill(B=2, S=S, H=H, Hkv=Hkv, dk=d, dv=d, dtype=dtype, seed=30, S_kv=S + off + 3,
                       offsets=[off, off + 3])
    out = torch.empty(2, S, H, d, dtype=dtype, device=DEV)
    g.attn_prefill_causal(c.q.to(DEV), c.k.to(DEV), c.v.to(DEV), out, c.scale,
                          position_offset=c.offsets.to(DEV))
    ok(g)
    want = core.prefill_causal(W.to_oracle(c.q), W.to_oracle(c.k), W.to_oracle(c.v), c.scale,
                               offsets=[off, off + 3])
    check(maxerr(out, want), TOL[dtype])


def test_prefill_mla_shape(gpu_lib):
    g = gpu_lib
    c = W.make_prefill(B=1, S=90, H=4, Hkv=4, dk=192, dv=128, seed=31)
    out = torch.empty(1, 90, 4, 128, dtype=torch.bfloat16, device=DEV)
    g.attn_prefill_causal(c.q.to(DEV), c.k.to(DEV), c.v.to(DEV), out, c.scale)
    ok(g)
    want = core.prefill_causal(W.to_oracle(c.q), W.to_oracle(c.k), W.to_oracle(c.v), c.scale)
    check(maxerr(out, want), 2e-2)


# ---------------------------------------------------------------------------
# RoPE and append

def rope_close(got_bits, want_bits, x_in_bits):
    """GPU RoPE (fp32 rotation of an fp64-reduced angle, rounded once) against the
    oracle (exact rotation, rounded once). Before rounding the two differ by at most
    a few fp32 roundings of the pair's norm (sincosf, the fp32 angle, two FMAs), so
    after rounding: |got - want| <= 1 bf16 ulp of want + 2^-20 * |(x0, x1)|."""
    got, want, x = core.widen(got_bits), core.widen(want_bits), core.widen(x_in_bits)
    pair = np.sqrt(x[..., 0::2] ** 2 + x[..., 1::2] ** 2)
    norm = np.repeat(pair, 2, axis=-1)
    mag = np.maximum(np.abs(want), 1e-30)
    ulp = 2.0 ** (np.floor(np.log2(mag)) - 7)
    return bool(np.all(np.abs(got - want) <= ulp + 2.0 ** -20 * norm))


@pytest.mark.parametrize("heads_outer", [False, True])
def test_rope_bf16_within_one_ulp(gpu_lib, heads_outer):
    g = gpu_lib
    B, T, Hh, d = 2, 300, 3, 64
    x = W.randn((B, Hh, T, d) if heads_outer else (B, T, Hh, d), W.generator(40), torch.bfloat16)
    pos = torch.randint(0, 40000, (B, T), generator=W.generator(41), dtype=torch.int32)
    xg = x.to(DEV)
    g.attn_rope_interleaved(xg, pos.to(DEV), 1e6, heads_outer=heads_outer)
    ok(g)
    xo = W.to_oracle(x)
    if heads_outer:
        xo = np.ascontiguousarray(xo.transpose(0, 2, 1, 3))
    want = core.rope_interleaved(xo, W.to_oracle(pos), 0, d, 1e6)
    got = W.to_oracle(xg)
    if heads_outer:
        got = np.ascontiguousarray(got.transpose(0, 2, 1, 3))
    assert rope_close(got, want, xo)


def test_rope_positions_around_float_exactness(gpu_lib):
    """Positions below 2^24 take the angle in fp32 arithmetic (the product formed
    without error, Cody-Waite reduction), positions from 2^24 on (no longer exact
    as a float) in fp64: both within the same bound as above."""
    g = gpu_lib
    pos = torch.tensor([[0, 1, 7, 4095, 32767, 40000, 99999, 2 ** 20, 2 ** 24 - 2, 2 ** 24 - 1, 2 ** 24, 2 ** 24 + 1,
                         2 ** 24 + 7, 2 ** 25 + 3, 2 ** 30, 2 ** 31 - 1]], dtype=torch.int32)
    x = W.randn((1, pos.shape[1], 2, 64), W.generator(45), torch.bfloat16)
    xg = x.to(DEV)
    g.attn_rope_interleaved(xg, pos.to(DEV), 1e4)
    ok(g)
    want = core.rope_interleaved(W.to_oracle(x), W.to_oracle(pos), 0, 64, 1e4)
    assert rope_close(W.to_oracle(xg), want, W.to_oracle(x))


def test_rope_f32_slice(gpu_lib):
    g = gpu_lib
    x = W.randn((1, 50, 4, 192), W.generator(42), torch.float32)
    pos = torch.arange(4046, 4096, dtype=torch.int32)[None]
    xg = x.to(DEV)
    g.attn_rope_interleaved(xg, pos.to(DEV), 1e4, rot_offset=128, rot_dim=64)
    ok(g)
    want = core.rope_interleaved(W.to_oracle(x).astype(np.float64), W.to_oracle(pos), 128, 64, 1e4)
    assert np.abs(xg.cpu().numpy() - want).max() <= 2e-5


@pytest.mark.parametrize("dt,hq,hk,q_outer,k_outer,off,rot", [
    (torch.bfloat16, 14, 2, False, True, 0, 64),    # the 2048-row prefill's layout and heads
    (torch.bfloat16, 5, 7, True, False, 0, 64),     # more k heads than in flight at once, both layouts swapped
    (torch.bfloat16, 20, 1, False, False, 16, 32),  # a partial slice; q heads past the in-flight group
    (torch.float32, 3, 2, False, True, 128, 64),    # fp32, the MLA-style rope slice of a 192-wide head
])
def test_rope_qk_equals_two_calls(gpu_lib, dt, hq, hk, q_outer, k_outer, off, rot):
    """One launch over q and k gives bit for bit what two attn_rope_interleaved
    calls give (the same angle per pair and token, the same arithmetic); the k
    result is also checked against the oracle."""
    g = gpu_lib
    B, T = 2, 333
    d = off + rot if off else 64
    d = max(d, 64)
    shape = lambda h, outer: (B, h, T, d) if outer else (B, T, h, d)
    q = W.randn(shape(hq, q_outer), W.generator(46), dt)
    k = W.randn(shape(hk, k_outer), W.generator(47), dt)
    pos = torch.randint(0, 50000, (B, T), generator=W.generator(48), dtype=torch.int32)
    q1, k1, q2, k2 = q.to(DEV), k.to(DEV), q.to(DEV), k.to(DEV)
    g.attn_rope_interleaved(q1, pos.to(DEV), 1e6, rot_offset=off, rot_dim=rot, heads_outer=q_outer)
    g.attn_rope_interleaved(k1, pos.to(DEV), 1e6, rot_offset=off, rot_dim=rot, heads_outer=k_outer)
    g.attn_rope_interleaved_qk(q2, k2, pos.to(DEV), 1e6, rot_offset=off, rot_dim=rot, q_heads_outer=q_outer,
                               k_heads_outer=k_outer)
    ok(g)
    assert torch.equal(q1, q2) and torch.equal(k1, k2)
    tok = lambda a: np.ascontiguousarray(a.transpose(0, 2, 1, 3)) if k_outer else a  # to [B, T, heads, d]
    if dt == torch.bfloat16:  # the oracle's bf16 values, as bits
        ko = tok(W.to_oracle(k))
        want = core.rope_interleaved(ko, W.to_oracle(pos), off, rot, 1e6)
        assert rope_close(tok(W.to_oracle(k2)), want, ko)
    else:
        want = core.rope_interleaved(tok(W.to_oracle(k).astype(np.float64)), W.to_oracle(pos), off, rot, 1e6)
        assert np.abs(tok(k2.cpu().numpy()) - want).max() <= 2e-5


def test_append_writes_only_target_slots(gpu_lib):
    g = gpu_lib
    c = W.make_paged(B=6, H=8, Hkv=2, dk=128, dv=128, block_size=16, num_blocks=300, lens=[0, 15, 16, 17, 700, 1],
                     mbps=50, seed=43)
    kp0, vp0 = W.to_oracle(c.k_pool), W.to_oracle(c.v_pool)
    q, kp, vp = c.q.to(DEV), c.k_pool.to(DEV), c.v_pool.to(DEV)
    lin = c.seq_lens.to(DEV)
    lout = torch.empty_like(lin)
    g.kv_append_paged(q, c.k_new.to(DEV), c.v_new.to(DEV), kp, vp, c.tables.to(DEV), lin, lout, c.theta)
    ok(g)
    q2, kp2, vp2, l2 = core.kv_append_paged(W.to_oracle(c.q), W.to_oracle(c.k_new), W.to_oracle(c.v_new), kp0, vp0,
                                            W.to_oracle(c.tables), W.to_oracle(c.seq_lens), c.theta)
    assert lout.cpu().tolist() == list(l2) == [n + 1 for n in c.seq_lens.tolist()]
    gk, gv = W.to_oracle(kp), W.to_oracle(vp)
    assert np.array_equal(gv, vp2)                      # V is copied bit for bit
    diff = np.argwhere(np.any(gk != kp0, axis=-1))      # K rows that changed
    targets = {(int(c.tables[b, n // 16]), n % 16) for b, n in enumerate(c.seq_lens.tolist())}
    assert {(int(a), int(r)) for a, _, r in diff} <= targets
    k_in = kp2.copy()                                    # unrotated new rows at the targets
    for b, n in enumerate(c.seq_lens.tolist()):
        k_in[int(c.tables[b, n // 16]), :, n % 16] = W.to_oracle(c.k_new[b])
    assert rope_close(gk, kp2, k_in)                     # rotated k
    assert rope_close(W.to_oracle(q), q2, W.to_oracle(c.q))


@pytest.mark.parametrize("dtype,rot_offset,rot_dim", [
    (torch.bfloat16, 0, None),   # every column rotated: the 16-byte chunk path
    (torch.bfloat16, 16, 32),    # an aligned middle range: chunks rotated or copied as they fall
    (torch.bfloat16, 2, 12),     # not on a chunk boundary: the element-wise form
    (torch.float32, 4, 8),       # fp32 rows, 4-element chunks
])
def test_append_partial_rotary(gpu_lib, dtype, rot_offset, rot_dim):
    """kv_append_paged with only part of each row rotated, through both of its
    forms: V copied bit for bit, K and q rotated within the RoPE bound where the
    range says and bit for bit elsewhere, no other pool slot written."""
    g = gpu_lib
    c = W.make_paged(B=5, H=8, Hkv=2, dk=64, dv=64, block_size=16, num_blocks=200, lens=[0, 15, 16, 300, 1],
                     mbps=40, seed=44, dtype=dtype)
    kp0, vp0 = W.to_oracle(c.k_pool), W.to_oracle(c.v_pool)
    q, kp, vp = c.q.to(DEV), c.k_pool.to(DEV), c.v_pool.to(DEV)
    lin = c.seq_lens.to(DEV)
    lout = torch.empty_like(lin)
    g.kv_append_paged(q, c.k_new.to(DEV), c.v_new.to(DEV), kp, vp, c.tables.to(DEV), lin, lout, c.theta,
                      rot_offset=rot_offset, rot_dim=rot_dim)
    ok(g)
    q2, kp2, vp2, l2 = core.kv_append_paged(W.to_oracle(c.q), W.to_oracle(c.k_new), W.to_oracle(c.v_new), kp0, vp0,
                                            W.to_oracle(c.tables), W.to_oracle(c.seq_lens), c.theta,
                                            rot_offset=rot_offset, rot_dim=rot_dim)
    assert lout.cpu().tolist() == list(l2)
    gk, gv, gq = W.to_oracle(kp), W.to_oracle(vp), W.to_oracle(q)
    assert np.array_equal(gv, vp2)
    rd = 64 - rot_offset if rot_dim is None else rot_dim
    cols = np.zeros(64, dtype=bool)
    cols[rot_offset:rot_offset + rd] = True
    assert np.array_equal(gk[..., ~cols], kp2[..., ~cols])   # columns outside the range: copied
    assert np.array_equal(gq[..., ~cols], q2[..., ~cols])
    k_in = kp2.copy()
    for b, n in enumerate(c.seq_lens.tolist()):
        k_in[int(c.tables[b, n // 16]), :, n % 16] = W.to_oracle(c.k_new[b])
    if dtype == torch.bfloat16:
        assert rope_close(gk[..., cols], kp2[..., cols], k_in[..., cols])
        assert rope_close(gq[..., cols], q2[..., cols], W.to_oracle(c.q)[..., cols])
    else:  # fp32: a few fp32 roundings of the pair's norm
        for got, want, x in ((gk, kp2, k_in), (gq, q2, W.to_oracle(c.q))):
            x = core.widen(x[..., cols])
            norm = np.repeat(np.sqrt(x[..., 0::2] ** 2 + x[..., 1::2] ** 2), 2, axis=-1)
            assert np.all(np.abs(core.widen(got[..., cols]) - core.widen(want[..., cols])) <= 2.0 ** -20 * norm + 1e-30)


# ---------------------------------------------------------------------------
# invariants

def test_determinism_and_batch_invariance(gpu_lib):
    g = gpu_lib
    lens = [3000, 1, 1500, 2049]
    c = W.make_contig(B=4, H=32, Hkv=8, dk=128, dv=128, max_len=3000, lens=lens, seed=50)
    args = [t.to(DEV) for t in (c.q, c.k, c.v, c.seq_lens)]
    ws = g.decode_workspace(4, 32, 128, 3000)
    o1 = torch.empty(4, 32, 128, dtype=torch.bfloat16, device=DEV)
    o2 = torch.empty_like(o1)
    g.attn_decode_contig(*args[:4], o1, c.scale, workspace=ws)
    g.attn_decode_contig(*args[:4], o2, c.scale, workspace=ws)
    assert torch.equal(o1, o2)
    # sequence 2 alone gives the same bits as inside the batch
    o3 = torch.empty(1, 32, 128, dtype=torch.bfloat16, device=DEV)
    g.attn_decode_contig(args[0][2:3].contiguous(), args[1][2:3].contiguous(), args[2][2:3].contiguous(),
                         args[3][2:3].contiguous(), o3, c.scale, workspace=ws)
    ok(g)
    assert torch.equal(o3[0], o1[2])


def test_gqa_equals_mha_on_repeated_kv(gpu_lib):
    g = gpu_lib
    c = W.make_contig(B=2, H=16, Hkv=4, dk=64, dv=64, max_len=1300, lens=[1300, 77], seed=51)
    q, k, v, lens = (t.to(DEV) for t in (c.q, c.k, c.v, c.seq_lens))
    ws = g.decode_workspace(2, 16, 64, 1300)
    o_gqa = torch.empty(2, 16, 64, dtype=torch.bfloat16, device=DEV)
    g.attn_decode_contig(q, k, v, lens, o_gqa, c.scale, workspace=ws)
    o_mha = torch.empty_like(o_gqa)
    g.attn_decode_contig(q, k.repeat_interleave(4, dim=1).contiguous(), v.repeat_interleave(4, dim=1).contiguous(),
                         lens, o_mha, c.scale, workspace=ws)
    ok(g)
    assert torch.equal(o_gqa, o_mha)  # the same arithmetic per (head, key row)


def test_decode_equals_last_prefill_row(gpu_lib):
    g = gpu_lib
    c = W.make_prefill(B=1, S=40, H=8, Hkv=2, dk=128, dv=128, seed=52)
    pre = torch.empty(1, 40, 8, 128, dtype=torch.bfloat16, device=DEV)
    g.attn_prefill_causal(c.q.to(DEV), c.k.to(DEV), c.v.to(DEV), pre, c.scale)
    dec = torch.empty(1, 8, 128, dtype=torch.bfloat16, device=DEV)
    g.attn_decode_contig(c.q[:, 39].contiguous().to(DEV), c.k.to(DEV), c.v.to(DEV),
                         torch.tensor([40], dtype=torch.int32, device=DEV), dec, c.scale)
    ok(g)
    check((dec.float() - pre[:, 39].float()).abs().max().item(), 2e-2, "decode vs prefill row")


def test_empty_batch_is_a_no_op(gpu_lib):
    g = gpu_lib
    z = torch.empty(0, 4, 16, device=DEV)
    g.attn_decode_contig(z, torch.empty(0, 2, 8, 16, device=DEV), torch.empty(0, 2, 8, 16, device=DEV),
                         torch.empty(0, dtype=torch.int32, device=DEV), z, 0.25)
    ok(g)
