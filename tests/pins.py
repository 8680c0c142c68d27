"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Each ``pin_*`` function takes the oracle's C binding module (``oracle.core`` or a
stand-in with a planted mistake) and raises AssertionError when the oracle is
wrong. ``tests/test_oracle_pins.py`` runs them on the real oracle and
``tests/test_oracle_mutants.py`` checks that every planted mistake trips at
least one of them.
"""
import math
import os
import re

import numpy as np

from oracle import dense

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
_MATH = {k: getattr(math, k) for k in ("cos", "sin", "log", "exp", "sqrt", "pi")}


def _expr(tok: str) -> float:
    if tok == "-inf":
        return -math.inf
    if not re.fullmatch(r"[0-9a-z_.*/+\-() ]+", tok):
        raise ValueError(tok)
    return float(eval(tok, {"__builtins__": {}}, _MATH))


def golden_blocks(name):
    """Parse a golden file into a list of blocks (lists of non-comment lines)."""
    blocks, cur = [], []
    for line in open(os.path.join(GOLDEN, name)):
        line = line.rstrip("\n")
        if line.startswith("#"):
            continue
        if not line.strip():
            if cur:
                blocks.append(cur)
            cur = []
            continue
        cur.append(line)
    if cur:
        blocks.append(cur)
    return blocks


def _vec(s):
    return np.array([_expr(t) for t in s.split()], np.float64)


def rng(seed):
    return np.random.default_rng(seed)


# ---------------------------------------------------------------------------
# closed forms through the C loops

def _closed_cases():
    cases = {}
    for blk in golden_blocks("closed_form_attention.txt"):
        d = {}
        for line in blk:
            key, _, rest = line.partition(" ")
            d[key] = rest
        cases[d["case"]] = d
    return cases


def pin_closed_form_two_keys(core):
    c = _closed_cases()["two_keys"]
    rows = [[_vec(h) for h in r.split("|")] for r in c["q"].split("||")]
    q = np.array(rows)[None]                                     # [1, 2, 2, 2]
    k = np.array([_vec(r) for r in c["k"].split(";")])[None, None]  # [1, 1, 2, 2]
    v = np.array([_vec(r) for r in c["v"].split(";")])[None, None]
    want = np.array([[_vec(h) for h in r.split("|")] for r in c["out"].split("||")])[None]
    got = core.prefill_causal(q, k, v, float(c["scale"]))
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-13)


def pin_closed_form_head_mapping(core):
    c = _closed_cases()["head_mapping"]
    q = np.array([_vec(h) for h in c["q"].split("|")])[None]                      # [1, 4, 1]
    k = np.array([[_vec(r) for r in kv.split(";")] for kv in c["k"].split(";;")])[None]  # [1,2,2,1]
    v = np.array([[_vec(r) for r in kv.split(";")] for kv in c["v"].split(";;")])[None]
    want = np.array([_vec(h) for h in c["out"].split("|")])[None]
    got = core.decode_contig(q, k, v, [2], float(c["scale"]))
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-13)


def pin_zero_kv_gives_zero(core):
    """kopitiam-runtime src/attention.rs, test `attention_forward_with_zeroed_kv_weights_
    produces_zero_output`: K = V = 0 gives exactly zero output (uniform weights over zeros)."""
    r = rng(1)
    q = r.standard_normal((1, 2, 2, 2))
    z = np.zeros((1, 1, 2, 2))
    assert np.all(core.prefill_causal(q, z, z, 1 / math.sqrt(2)) == 0.0)


def pin_zero_keys_give_prefix_mean(core):
    """K = 0 (or scale 0): every visible key scores 0, so row i returns the mean of
    V[0..=p] -- the non-zero-V extension of the same test."""
    r = rng(2)
    B, S, H, Hkv, d = 2, 7, 4, 2, 8
    q = r.standard_normal((B, S, H, d))
    k = np.zeros((B, Hkv, S + 3, d))
    v = r.standard_normal((B, Hkv, S + 3, d))
    off = [0, 3]
    got = core.prefill_causal(q, k, v, 0.7, offsets=off)
    got0 = core.prefill_causal(q, r.standard_normal(k.shape), v, 0.0, offsets=off)
    for b in range(B):
        for i in range(S):
            p = off[b] + i
            for h in range(H):
                want = v[b, h // (H // Hkv), :p + 1].mean(axis=0)
                np.testing.assert_allclose(got[b, i, h], want, rtol=0, atol=1e-13)
                np.testing.assert_allclose(got0[b, i, h], want, rtol=0, atol=1e-13)


def pin_first_row_is_v0(core):
    """Position 0 sees key 0 only: output is V[0] exactly (decode at seq_len 1 too)."""
    r = rng(3)
    q = r.standard_normal((1, 3, 4, 8))
    k = r.standard_normal((1, 2, 3, 8))
    v = r.standard_normal((1, 2, 3, 8))
    got = core.prefill_causal(q, k, v, 0.35)
    for h in range(4):
        assert np.array_equal(got[0, 0, h], v[0, h // 2, 0])
    got = core.decode_contig(q[:, 0], k, v, [1], 0.35)
    for h in range(4):
        assert np.array_equal(got[0, h], v[0, h // 2, 0])


def pin_constant_v(core):
    """Softmax rows sum to 1: V = c everywhere gives c."""
    r = rng(4)
    q = r.standard_normal((1, 5, 2, 4))
    k = r.standard_normal((1, 1, 5, 4))
    v = np.full((1, 1, 5, 4), 2.5)
    np.testing.assert_allclose(core.prefill_causal(q, k, v, 0.9), 2.5, rtol=1e-15, atol=0)


def pin_one_hot_v_gives_probabilities(core):
    """With V = identity rows (seq_kv <= d_v) the output row IS the probability row:
    non-negative, sums to 1, exactly zero past the row's position, and equal to the
    dense softmax of the mask-matrix formulation."""
    r = rng(5)
    S, H, Hkv, d = 6, 4, 2, 6
    q = r.standard_normal((1, S, H, d))
    k = r.standard_normal((1, Hkv, S, d))
    v = np.broadcast_to(np.eye(S)[None, None], (1, Hkv, S, S)).copy()
    got = core.prefill_causal(q, k, v, 0.5)[0]                     # [S, H, S]
    probs = dense.probabilities(q[0], k[0], 0, 0.5)                # [H, S, S]
    for i in range(S):
        for h in range(H):
            row = got[i, h]
            assert np.all(row[i + 1:] == 0.0)
            assert np.all(row >= 0.0)
            assert abs(row.sum() - 1.0) < 1e-14
            np.testing.assert_allclose(row, probs[h, i], rtol=0, atol=1e-14)


def pin_loops_equal_dense(core):
    """The C loops and the mask-matrix formulation agree to 1e-12 over a sweep."""
    r = rng(6)
    for (H, Hkv, dk, dv, S, off) in [(4, 2, 16, 16, 8, 0), (8, 1, 8, 12, 5, 7), (6, 6, 4, 4, 9, 2),
                                     (12, 3, 32, 16, 3, 20), (2, 1, 24, 8, 1, 30)]:
        q = r.standard_normal((1, S, H, dk))
        k = r.standard_normal((1, Hkv, off + S, dk))
        v = r.standard_normal((1, Hkv, off + S, dv))
        scale = 1 / math.sqrt(dk)
        got = core.prefill_causal(q, k, v, scale, offsets=[off])[0]
        want = dense.attention(q[0], k[0], v[0], off, scale)
        np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)


def pin_gqa_equals_mha_on_repeated_kv(core):
    """GQA(H, Hkv) equals MHA(H, H) on K/V repeated per `repeat_kv_heads` (head g of
    the repeated cache is KV head g // group)."""
    r = rng(7)
    B, H, Hkv, d, L = 2, 8, 2, 16, 11
    q = r.standard_normal((B, H, d))
    k = r.standard_normal((B, Hkv, L, d))
    v = r.standard_normal((B, Hkv, L, d))
    lens = [L, 4]
    got = core.decode_contig(q, k, v, lens, 0.25)
    k_rep = np.stack([dense.repeat_kv_heads(k[b], H // Hkv) for b in range(B)])
    v_rep = np.stack([dense.repeat_kv_heads(v[b], H // Hkv) for b in range(B)])
    assert np.array_equal(got, core.decode_contig(q, k_rep, v_rep, lens, 0.25))
    # Hkv = 1 is MQA: every head reads the same KV head.
    got1 = core.decode_contig(q, k[:, :1], v[:, :1], lens, 0.25)
    for h in range(H):
        assert np.array_equal(got1[:, h], core.decode_contig(q[:, h:h + 1], k[:, :1], v[:, :1], lens,
                                                             0.25)[:, 0])


def pin_paged_equals_contig(core):
    """Paging changes where rows live and nothing else: a shuffled pool with its
    table gives the contiguous answer bit for bit."""
    r = rng(8)
    B, H, Hkv, d, bs, L = 3, 4, 2, 8, 4, 13
    q = r.standard_normal((B, H, d))
    k = r.standard_normal((B, Hkv, L, d))
    v = r.standard_normal((B, Hkv, L, d))
    lens = [13, 1, 6]
    nblk = (L + bs - 1) // bs
    pool_n = B * nblk + 5
    perm = r.permutation(pool_n)
    kp = r.standard_normal((pool_n, Hkv, bs, d))
    vp = r.standard_normal((pool_n, Hkv, bs, d))
    tables = np.full((B, nblk + 2), -1, np.int32)
    for b in range(B):
        for blk in range(nblk):
            e = perm[b * nblk + blk]
            tables[b, blk] = e
            rows = slice(blk * bs, min(L, (blk + 1) * bs))
            n = rows.stop - rows.start
            kp[e, :, :n] = k[b, :, rows]
            vp[e, :, :n] = v[b, :, rows]
    assert np.array_equal(core.decode_paged(q, kp, vp, tables, lens, 0.3),
                          core.decode_contig(q, k, v, lens, 0.3))


def pin_decode_equals_last_prefill_row(core):
    """One decode step at position p equals row p of the matching prefill
    (kopitiam-runtime src/attention.rs, module doc: one mask rule serves both)."""
    r = rng(9)
    S, H, Hkv, d = 9, 4, 2, 16
    q = r.standard_normal((1, S, H, d))
    k = r.standard_normal((1, Hkv, S, d))
    v = r.standard_normal((1, Hkv, S, d))
    pre = core.prefill_causal(q, k, v, 0.25)
    for p in range(S):
        dec = core.decode_contig(q[:, p], k, v, [p + 1], 0.25)
        assert np.array_equal(dec, pre[:, p])
    # the same step via the offset form: seq_q = 1 at position_offset = p
    dec = core.prefill_causal(q[:, 5:6], k, v, 0.25, offsets=[5])
    assert np.array_equal(dec, pre[:, 5:6])


# ---------------------------------------------------------------------------
# RoPE

def pin_rope_closed_forms(core):
    for blk in golden_blocks("rope_closed_form.txt"):
        theta, d, off, rd, pos = blk[0].split()[1:]
        x = _vec(blk[1].partition(" ")[2])
        want = _vec(blk[2].partition(" ")[2])
        got = core.rope_interleaved(x.reshape(1, 1, 1, -1), [[int(pos)]], int(off), int(rd), float(theta))
        np.testing.assert_allclose(got.reshape(-1), want, rtol=0, atol=1e-12)


def pin_rope_invariants(core):
    r = rng(10)
    x = r.standard_normal((2, 5, 3, 16))
    zero = np.zeros((2, 5), np.int32)
    assert np.array_equal(core.rope_interleaved(x, zero, 0, 16, 1e4), x)        # pos 0: identity
    pos = r.integers(0, 40000, (2, 5)).astype(np.int32)
    y = core.rope_interleaved(x, pos, 0, 16, 1e6)
    n_x = x[..., 0::2] ** 2 + x[..., 1::2] ** 2                                  # pair norms kept
    n_y = y[..., 0::2] ** 2 + y[..., 1::2] ** 2
    np.testing.assert_allclose(n_y, n_x, rtol=1e-12, atol=1e-12)
    # <R(p) q, R(s) k> depends on p - s only
    qv = r.standard_normal((1, 1, 1, 16))
    kv = r.standard_normal((1, 1, 1, 16))
    dots = []
    for (p, s) in [(7, 3), (104, 100), (4, 0), (1004, 1000)]:
        a = core.rope_interleaved(qv, [[p]], 0, 16, 1e4).reshape(-1)
        b = core.rope_interleaved(kv, [[s]], 0, 16, 1e4).reshape(-1)
        dots.append(a @ b)
    np.testing.assert_allclose(dots, dots[0], rtol=0, atol=1e-10)


def pin_shared_rot_once_equals_per_head(core):
    """frink-models src/mla/mod.rs, module doc point 2: rotating the shared k_rot
    once and copying it into every head equals rotating each head's copy."""
    r = rng(11)
    L, H, dr = 6, 5, 8
    k_rot = r.standard_normal((1, L, 1, dr))
    pos = np.arange(L, dtype=np.int32)[None]
    once = core.rope_interleaved(k_rot, pos, 0, dr, 1e4)
    per_head = core.rope_interleaved(np.broadcast_to(k_rot, (1, L, H, dr)).copy(), pos, 0, dr, 1e4)
    for h in range(H):
        assert np.array_equal(per_head[:, :, h], once[:, :, 0])


# ---------------------------------------------------------------------------
# MLA, absorbed (latent) form

def _mla_case(seed, B=2, H=3, dn=8, dr=4, dc=12, dv=6, L=9):
    r = rng(seed)
    return dict(q=r.standard_normal((B, H, dn + dr)), k_b=r.standard_normal((H, dc, dn)),
                v_b=r.standard_normal((H, dv, dc)), c=r.standard_normal((B, L, dc)),
                k_rot=r.standard_normal((B, L, dr)), dn=dn, dc=dc, scale=1.0 / np.sqrt(dn + dr))


def pin_mla_absorbed_equals_naive(core):
    """frink-models src/mla/mod.rs, `MlaKvB`: the absorbed and the naive forms
    compute the same attention. The naive cache is the latent expanded per head:
    k_nope[b, h, j] = k_b[h]^T c_j (k_b maps qk_nope to the latent, so its
    transpose expands the latent into the nope key) and v[b, h, j] = v_b[h] c_j,
    with the shared k_rot copied into every head."""
    m = _mla_case(21)
    k_nope = np.einsum("hcn,bjc->bhjn", m["k_b"], m["c"])
    v = np.einsum("hvc,bjc->bhjv", m["v_b"], m["c"])
    for lens in ([9, 5], [1, 9]):
        naive = core.decode_mla_naive(m["q"], k_nope, m["k_rot"], v, lens, m["scale"])
        q_abs = core.mla_absorb_q(m["q"], m["k_b"], m["dn"])
        lat = np.concatenate([m["c"], m["k_rot"]], axis=-1)
        out = core.mla_unabsorb_out(core.decode_mla_absorbed(q_abs, lat, lens, m["dc"], m["scale"]), m["v_b"])
        np.testing.assert_allclose(out, naive, rtol=0, atol=1e-10)


def pin_mla_latent_closed_forms(core):
    """Attention over the latent rows (c_j, k_rot_j) with value c_j: (1) a zero
    query weighs the visible rows equally, so each head gets the mean of c_j over
    j < seq_len; (2) one visible row gives c_0 exactly; (3) two rows with c_0 =
    e_0 and c_1 = e_1 give (p, 1 - p, 0, ...), p = 1 / (1 + e^(s_1 - s_0)), where
    s_j = scale * (q_c . c_j + q_r . k_rot_j) takes the rope slices too."""
    r = rng(22)
    B, H, dc, dr, L = 2, 3, 8, 4, 7
    lat = r.standard_normal((B, L, dc + dr))
    lens = [7, 3]
    zero = core.decode_mla_absorbed(np.zeros((B, H, dc + dr)), lat, lens, dc, 0.3)
    for b, n in enumerate(lens):
        np.testing.assert_allclose(zero[b], np.broadcast_to(lat[b, :n, :dc].mean(axis=0), (H, dc)), rtol=0,
                                   atol=1e-12)
    q = r.standard_normal((B, H, dc + dr))
    one = core.decode_mla_absorbed(q, lat, [1, 1], dc, 0.3)
    for b in range(B):
        assert np.array_equal(one[b], np.broadcast_to(lat[b, 0, :dc], (H, dc)))
    lat2 = np.zeros((1, 2, dc + dr))
    lat2[0, 0, 0] = lat2[0, 1, 1] = 1.0
    lat2[0, :, dc:] = r.standard_normal((2, dr))
    q2 = r.standard_normal((1, H, dc + dr))
    got = core.decode_mla_absorbed(q2, lat2, [2], dc, 0.7)
    for h in range(H):
        s = [0.7 * (q2[0, h, :dc] @ lat2[0, j, :dc] + q2[0, h, dc:] @ lat2[0, j, dc:]) for j in range(2)]
        p = 1.0 / (1.0 + np.exp(s[1] - s[0]))
        np.testing.assert_allclose(got[0, h], [p, 1.0 - p] + [0.0] * (dc - 2), rtol=0, atol=1e-12)


def pin_mla_projections(core):
    """The absorb and unabsorb maps on basis vectors: the absorbed nope slice of
    q = e_n is column n of k_b[h] and the rope slice passes through unchanged;
    out_lat = e_c maps to column c of v_b[h]."""
    m = _mla_case(23, B=1)
    H, dn, dc = m["k_b"].shape[0], m["dn"], m["dc"]
    for n in (0, dn - 1):
        q = np.zeros((1, H, dn + 4))
        q[0, :, n] = 1.0
        q[0, :, dn:] = [1.5, -2.0, 0.25, 3.0]
        got = core.mla_absorb_q(q, m["k_b"], dn)
        for h in range(H):
            assert np.array_equal(got[0, h, :dc], m["k_b"][h, :, n])
            assert np.array_equal(got[0, h, dc:], [1.5, -2.0, 0.25, 3.0])
    for c in (0, dc - 1):
        lat = np.zeros((1, H, dc))
        lat[0, :, c] = 1.0
        got = core.mla_unabsorb_out(lat, m["v_b"])
        for h in range(H):
            assert np.array_equal(got[0, h], m["v_b"][h, :, c])


# ---------------------------------------------------------------------------
# paged append

def pin_append(core):
    """Push then attend (frink-models src/decoder/attn_block.rs, `push_and_attend_row`):
    the row goes to (table[b][p / bs], kvh, p % bs) with p = seq_lens_in[b], rotated
    at p; nothing else in the pool changes; seq_lens_out = p + 1."""
    r = rng(12)
    B, H, Hkv, d, bs, nb = 3, 4, 2, 8, 4, 20
    q = r.standard_normal((B, H, d))
    kn = r.standard_normal((B, Hkv, d))
    vn = r.standard_normal((B, Hkv, d))
    kp = r.standard_normal((nb, Hkv, bs, d))
    vp = r.standard_normal((nb, Hkv, bs, d))
    tables = np.array([[3, 7, 1, -1], [11, -1, -1, -1], [0, 2, 19, 5]], np.int32)
    lens = np.array([9, 0, 15], np.int32)
    q2, kp2, vp2, lout = core.kv_append_paged(q, kn, vn, kp, vp, tables, lens, 1e4)
    assert list(lout) == [10, 1, 16]
    touched = np.zeros((nb, bs), bool)
    for b in range(B):
        p = int(lens[b])
        blk, row = tables[b, p // bs], p % bs
        touched[blk, row] = True
        want_k = core.rope_interleaved(kn[b][None, None], [[p]], 0, d, 1e4)[0, 0]
        want_q = core.rope_interleaved(q[b][None, None], [[p]], 0, d, 1e4)[0, 0]
        assert np.array_equal(kp2[blk, :, row], want_k)
        assert np.array_equal(vp2[blk, :, row], vn[b])
        assert np.array_equal(q2[b], want_q)
    for blk in range(nb):
        for row in range(bs):
            if not touched[blk, row]:
                assert np.array_equal(kp2[blk, :, row], kp[blk, :, row])
                assert np.array_equal(vp2[blk, :, row], vp[blk, :, row])


def pin_append_then_decode_is_attention_over_history(core):
    """Append + paged decode equals the definition on the history plus the new row
    (the new query sits at position len and sees rows 0..=len)."""
    r = rng(13)
    H, Hkv, d, bs = 4, 2, 8, 4
    L = 6
    hist_k = r.standard_normal((1, Hkv, L + 1, d))
    hist_v = r.standard_normal((1, Hkv, L + 1, d))
    q = r.standard_normal((1, H, d))
    kn = r.standard_normal((1, Hkv, d))
    vn = r.standard_normal((1, Hkv, d))
    tables = np.array([[2, 0, 1]], np.int32)
    kp = np.zeros((3, Hkv, bs, d))
    vp = np.zeros((3, Hkv, bs, d))
    for j in range(L):
        kp[tables[0, j // bs], :, j % bs] = hist_k[0, :, j]
        vp[tables[0, j // bs], :, j % bs] = hist_v[0, :, j]
    q2, kp2, vp2, lout = core.kv_append_paged(q, kn, vn, kp, vp, tables, [L], 0.0)  # no rotation
    got = core.decode_paged(q2, kp2, vp2, tables, lout, 0.5)
    hist_k[0, :, L] = kn[0]
    hist_v[0, :, L] = vn[0]
    want = dense.attention(q[:, None][0], hist_k[0], hist_v[0], L, 0.5)[0]
    np.testing.assert_allclose(got[0], want, rtol=0, atol=1e-13)


# ---------------------------------------------------------------------------
# bf16 storage

def pin_bf16_rounding(core):
    """Nearest-even rounding to bf16 (8 significant bits): ties go to the even code."""
    cases = [(1.0, 0x3F80), (1.0 + 2 ** -8, 0x3F80), (1.0 + 3 * 2 ** -8, 0x3F82),
             (1.0 + 2 ** -8 + 2 ** -20, 0x3F81), (-2.0, 0xC000), (0.0, 0x0000),
             (3.0e38, 0x7F62), (1e39, 0x7F80), (2 ** -130, 0x0008), (2 ** -134, 0x0000),
             (3 * 2 ** -134, 0x0002)]
    for x, bits in cases:
        assert core.bf16_bits(x) == bits, (x, hex(core.bf16_bits(x)), hex(bits))
        assert core.bf16_bits(-x) == bits ^ 0x8000 or x == 0.0


def pin_bf16_storage_widens_exactly(core):
    """bf16 inputs are widened exactly: the oracle on bf16 bits equals the oracle on
    the same values held as float64."""
    r = rng(14)
    q = r.standard_normal((1, 3, 2, 8)).astype(np.float32)
    k = r.standard_normal((1, 1, 3, 8)).astype(np.float32)
    v = r.standard_normal((1, 1, 3, 8)).astype(np.float32)
    bits = lambda a: (a.view(np.uint32) >> 16).astype(np.uint16)  # truncation: a valid bf16 value
    qb, kb, vb = bits(q), bits(k), bits(v)
    wide = lambda a: (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert np.array_equal(core.prefill_causal(qb, kb, vb, 0.3),
                          core.prefill_causal(wide(qb), wide(kb), wide(vb), 0.3))


# ---- the arms of the attention row (window, sink logits, softcap, ALiBi) ---
# The pages print no formula for these; the readings are stated in
# oracle/gqa_oracle.c (`oracle_attention_arms`).

def _arms_case(seed, B=2, S=5, H=4, Hkv=2, d=8, L=12):
    r = rng(seed)
    return r.standard_normal((B, S, H, d)), r.standard_normal((B, Hkv, L, d)), r.standard_normal((B, Hkv, L, d))


def pin_arms_loops_equal_mask_matrix(core):
    """The loops with every combination of arms equal the mask-matrix form with one
    bias matrix and the sink as an extra key of zero value (oracle/dense.py)."""
    from oracle import dense
    q, k, v = _arms_case(31)
    S = q.shape[1]
    sinks, slopes = np.array([0.4, -1.2, 2.0, 0.0]), np.array([0.25, 0.125, 0.0625, 0.5])
    base = [9, 12]
    for window, cap, sk, sl in [(3, 0.0, None, None), (0, 1.7, None, None), (0, 0.0, sinks, None),
                                (0, 0.0, None, slopes), (4, 2.5, sinks, slopes), (1, 0.9, sinks, slopes)]:
        out = core.attention_arms(q, k, v, base, 0.35, window, cap, sk, sl)
        for b in range(2):
            ref = dense.attention_arms(q[b], k[b, :, :base[b]], v[b, :, :base[b]], base[b] - S, 0.35, window, cap,
                                       sk, sl)
            assert np.abs(out[b] - ref).max() <= 1e-12


def pin_arms_vanish_at_their_limits(core):
    """No arms equals the plain oracle; a window wider than the history, a sink of
    -inf, an infinite cap and a zero slope each change nothing."""
    q, k, v = _arms_case(32)
    S, H = q.shape[1], q.shape[2]
    base = np.array([9, 12], np.int32)
    plain = core.attention_arms(q, k, v, base, 0.5)
    assert np.abs(plain - core.prefill_causal(q, k, v, 0.5, offsets=base - S)).max() <= 1e-13
    assert np.abs(core.attention_arms(q, k, v, base, 0.5, window=100) - plain).max() <= 1e-13
    assert np.abs(core.attention_arms(q, k, v, base, 0.5, sinks=[-1e300] * H) - plain).max() <= 1e-13
    assert np.abs(core.attention_arms(q, k, v, base, 0.5, softcap=1e9) - plain).max() <= 1e-9
    assert np.abs(core.attention_arms(q, k, v, base, 0.5, slopes=[0.0] * H) - plain).max() <= 1e-13


def pin_arms_closed_forms(core):
    """One or two visible keys: window 1 gives v_p; window 2 with ALiBi weighs key
    p-1 by e^(s - a); a sink z gives v_p / (1 + e^(z - s)); a softcap c maps s to
    c tanh(s / c) and leaves the sink alone."""
    q, k, v = _arms_case(33)
    B, S, H, _ = q.shape
    G = H // k.shape[1]
    base, scale, cap = [9, 12], 0.45, 0.8
    slopes, sinks = np.array([0.3, 0.7, 1.1, 0.05]), np.array([0.5, -0.7, 1.9, 0.0])
    w1 = core.attention_arms(q, k, v, base, scale, window=1)
    w2 = core.attention_arms(q, k, v, base, scale, window=2, slopes=slopes)
    ws = core.attention_arms(q, k, v, base, scale, window=1, sinks=sinks)
    wc = core.attention_arms(q, k, v, base, scale, window=1, sinks=sinks, softcap=cap)
    sc = lambda b, i, h, j: scale * float(np.dot(q[b, i, h], k[b, h // G, j]))
    for b in range(B):
        for i in range(S):
            p = base[b] - S + i
            for h in range(H):
                vp = v[b, h // G, p]
                assert np.abs(w1[b, i, h] - vp).max() <= 1e-14
                s = sc(b, i, h, p)
                assert np.abs(ws[b, i, h] - vp / (1.0 + math.exp(sinks[h] - s))).max() <= 1e-13
                assert np.abs(wc[b, i, h] - vp / (1.0 + math.exp(sinks[h] - cap * math.tanh(s / cap)))).max() <= 1e-13
                if p > 0:
                    s0, s1 = sc(b, i, h, p - 1) - slopes[h], s
                    mx = max(s0, s1)
                    e0, e1 = math.exp(s0 - mx), math.exp(s1 - mx)
                    want = (e0 * v[b, h // G, p - 1] + e1 * vp) / (e0 + e1)
                    assert np.abs(w2[b, i, h] - want).max() <= 1e-13


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
