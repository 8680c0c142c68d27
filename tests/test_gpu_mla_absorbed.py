"""The absorbed (latent) MLA decode -- absorb, attention over the latent rows,
unabsorb -- against the fp64 oracle (GPU, through the C ABI)."""
import numpy as np
import pytest
import torch

import workloads as W
from margins import check
from oracle import core

pytestmark = pytest.mark.gpu
DEV = "cuda"
D_C, D_R, D_NOPE = 512, 64, 128


def attend(g, q_abs, latent, lens, scale):
    B, H, _ = q_abs.shape
    out = torch.full((B, H, D_C), float("nan"), dtype=torch.bfloat16, device=DEV)
    ws = g.mla_absorbed_workspace(B, H, D_C, latent.shape[1])
    g.attn_decode_mla_absorbed(q_abs, latent, lens, out, scale, workspace=ws)
    return out


def absorbed_q(g, c):
    q_abs = torch.empty(c.q.shape[0], c.q.shape[1], D_C + D_R, dtype=torch.bfloat16, device=DEV)
    return g.mla_absorb_q(c.q.to(DEV), c.k_b.to(DEV), q_abs)


def oracle_latent(q_abs, latent, lens, scale):
    return core.decode_mla_absorbed(W.to_oracle(q_abs), W.to_oracle(latent), W.to_oracle(lens.cpu()), D_C, scale)


@pytest.mark.parametrize("B,H,L,lens", [
    (3, 128, 200, [1, 77, 200]),        # one split each; ragged last tiles; a single row
    (4, 128, 3000, [3000, 1025, 1024, 2049]),  # split boundaries 1024 / 2048 and the combine
    (2, 16, 300, [300, 33]),            # fewer heads than the 128-row tile
    (2, 200, 1100, [1100, 31]),         # two head tiles, the second ragged
])
def test_latent_attention_matches_oracle(gpu_lib, B, H, L, lens):
    g = gpu_lib
    c = W.make_mla_absorbed(B=B, H=H, max_len=L, lens=lens, seed=80 + H + L)
    q_abs = absorbed_q(g, c)
    latent = c.latent.to(DEV)
    out = attend(g, q_abs, latent, c.lens.to(DEV), c.scale)
    assert g.attn_get_device_error() == g.OK
    want = oracle_latent(q_abs, latent, c.lens, c.scale)
    err = np.abs(out.float().cpu().numpy() - want).max()
    check(err, 2e-2)


def test_rows_past_seq_len_never_reach_the_output(gpu_lib):
    """Rows at or past seq_len inside the last tile (and up to the capacity) hold
    NaN: the outputs stay finite and equal those of a clean cache bit for bit."""
    g = gpu_lib
    c = W.make_mla_absorbed(B=3, H=128, max_len=1100, lens=[45, 1030, 1100], seed=90)
    q_abs = absorbed_q(g, c)
    clean = c.latent.to(DEV)
    dirty = clean.clone()
    for b, n in enumerate(c.lens.tolist()):
        dirty[b, n:] = float("nan")
    lens = c.lens.to(DEV)
    a = attend(g, q_abs, clean, lens, c.scale)
    d = attend(g, q_abs, dirty, lens, c.scale)
    assert g.attn_get_device_error() == g.OK
    assert torch.isfinite(d.float()).all()
    assert torch.equal(a, d)


def test_zero_query_gives_prefix_mean(gpu_lib):
    """q_abs = 0: every visible row weighs the same, so each head gets the mean
    of c_j over j < seq_len (one split and several)."""
    g = gpu_lib
    c = W.make_mla_absorbed(B=2, H=128, max_len=2500, lens=[700, 2500], seed=91)
    latent = c.latent.to(DEV)
    out = attend(g, torch.zeros(2, 128, D_C + D_R, dtype=torch.bfloat16, device=DEV), latent, c.lens.to(DEV), 0.1)
    assert g.attn_get_device_error() == g.OK
    lat = W.to_oracle(c.latent)
    for b, n in enumerate(c.lens.tolist()):
        mean = core.widen(lat[b, :n, :D_C]).mean(axis=0)
        err = np.abs(out[b].float().cpu().numpy() - mean[None]).max()
        check(err, 1e-2)


def test_batch_composition_does_not_change_a_sequence(gpu_lib):
    """A sequence's output is the same bits alone and inside a batch (the split
    size is fixed, so its arithmetic does not depend on the other sequences)."""
    g = gpu_lib
    c = W.make_mla_absorbed(B=3, H=128, max_len=2100, lens=[2100, 900, 1500], seed=92)
    q_abs = absorbed_q(g, c)
    latent = c.latent.to(DEV)
    full = attend(g, q_abs, latent, c.lens.to(DEV), c.scale)
    for b in range(3):
        one = attend(g, q_abs[b:b + 1].contiguous(), latent[b:b + 1].contiguous(), c.lens[b:b + 1].to(DEV), c.scale)
        assert torch.equal(one[0], full[b])
    assert g.attn_get_device_error() == g.OK


def test_bad_lengths_give_zero_rows_and_flag(gpu_lib):
    g = gpu_lib
    c = W.make_mla_absorbed(B=3, H=128, max_len=256, lens=[0, 256, 257], seed=93)
    q_abs = absorbed_q(g, c)
    latent = c.latent.to(DEV)
    out = attend(g, q_abs, latent, c.lens.to(DEV), c.scale)
    assert g.attn_get_device_error() == g.ERR_DEVICE_BOUNDS
    assert torch.count_nonzero(out[0]) == 0 and torch.count_nonzero(out[2]) == 0
    want = core.decode_mla_absorbed(W.to_oracle(q_abs[1:2]), W.to_oracle(latent[1:2]), [256], D_C, c.scale)
    check(np.abs(out[1:2].float().cpu().numpy() - want).max(), 2e-2)


def test_projections_match_oracle(gpu_lib):
    """mla_absorb_q and mla_unabsorb_out: each output within the bf16 rounding of
    the fp64 product (|err| <= 2^-8 |y| + 1e-3); the rope slice copied exactly."""
    g = gpu_lib
    c = W.make_mla_absorbed(B=37, H=20, max_len=4, seed=94)  # B past one 32-row block
    q_abs = absorbed_q(g, c)
    want = core.mla_absorb_q(W.to_oracle(c.q), W.to_oracle(c.k_b), D_NOPE)
    got = q_abs.float().cpu().numpy()
    assert np.all(np.abs(got[..., :D_C] - want[..., :D_C]) <= 2.0 ** -8 * np.abs(want[..., :D_C]) + 1e-3)
    assert torch.equal(q_abs[..., D_C:].cpu(), c.q[..., D_NOPE:])
    lat = W.randn((37, 20, D_C), W.generator(95), torch.bfloat16)
    out = torch.empty(37, 20, 128, dtype=torch.bfloat16, device=DEV)
    g.mla_unabsorb_out(lat.to(DEV), c.v_b.to(DEV), out)
    want = core.mla_unabsorb_out(W.to_oracle(lat), W.to_oracle(c.v_b))
    assert np.all(np.abs(out.float().cpu().numpy() - want) <= 2.0 ** -8 * np.abs(want) + 1e-3)
    assert g.attn_get_device_error() == g.OK


def test_absorbed_chain_equals_naive_form(gpu_lib):
    """The three calls end to end against the oracle's naive form (per-head
    k_nope = k_b^T c_j and v = v_b c_j expanded in fp64, the shared k_rot copied
    into every head): the two forms are the same attention."""
    g = gpu_lib
    c = W.make_mla_absorbed(B=2, H=128, max_len=1500, lens=[1500, 600], seed=96)
    q_abs = absorbed_q(g, c)
    out_lat = attend(g, q_abs, c.latent.to(DEV), c.lens.to(DEV), c.scale)
    out = torch.empty(2, 128, 128, dtype=torch.bfloat16, device=DEV)
    g.mla_unabsorb_out(out_lat, c.v_b.to(DEV), out)
    assert g.attn_get_device_error() == g.OK
    lat = core.widen(W.to_oracle(c.latent))
    kb, vb = core.widen(W.to_oracle(c.k_b)), core.widen(W.to_oracle(c.v_b))
    k_nope = np.einsum("hcn,bjc->bhjn", kb, lat[..., :D_C])
    v = np.einsum("hvc,bjc->bhjv", vb, lat[..., :D_C])
    want = core.decode_mla_naive(core.widen(W.to_oracle(c.q)), k_nope, np.ascontiguousarray(lat[..., D_C:]), v,
                                 c.lens.numpy(), c.scale)
    err = np.abs(out.float().cpu().numpy() - want).max()
    check(err, 2e-2)


def test_full_size_sampled_sequences(gpu_lib):
    """The benchmarked workload (32 sequences, 128 heads, 4096 latent rows each),
    in the bench's launch configuration; three sequences checked against the
    oracle on every head."""
    g = gpu_lib
    c = W.make_mla_absorbed(seed=9, device=DEV)
    q_abs = absorbed_q(g, c)
    out = attend(g, q_abs, c.latent, c.lens, c.scale)
    assert g.attn_get_device_error() == g.OK
    for b in (0, 13, 31):
        want = oracle_latent(q_abs[b:b + 1], c.latent[b:b + 1], c.lens[b:b + 1], c.scale)
        err = np.abs(out[b:b + 1].float().cpu().numpy() - want).max()
        check(err, 2e-2, f"sequence {b}")


def page_latent(latent, lens, bs, seed, spare=3):
    """The latent rows of each sequence scattered over a pool of bs-row blocks in
    a seeded permuted order; table entries past a sequence's rows are -1."""
    B, L, w = latent.shape
    mbps = (L + bs - 1) // bs
    need = [(int(n) + bs - 1) // bs for n in lens]
    nb = sum(need) + spare
    perm = torch.randperm(nb, generator=W.generator(seed)).to(torch.int32)
    pool = torch.full((nb, bs, w), float("nan"), dtype=latent.dtype, device=latent.device)
    tables = torch.full((B, mbps), -1, dtype=torch.int32)
    at = 0
    for b, n in enumerate(need):
        for i in range(n):
            blk = int(perm[at])
            rows = latent[b, i * bs:(i + 1) * bs]
            pool[blk, :rows.shape[0]] = rows
            tables[b, i] = blk
            at += 1
    return pool, tables.to(latent.device)


@pytest.mark.parametrize("bs", [8, 16, 32, 64])
def test_paged_equals_contiguous_bit_for_bit(gpu_lib, bs):
    """The same rows through a permuted pool of bs-row blocks give the same bits
    as the contiguous cache (the slots past each sequence's rows hold NaN)."""
    g = gpu_lib
    L = 2112
    lens = [1, 63, 1025, 2100, L]
    c = W.make_mla_absorbed(B=5, H=128, max_len=L, lens=lens, seed=97)
    q_abs = absorbed_q(g, c)
    latent = c.latent.to(DEV)
    lens_d = c.lens.to(DEV)
    want = attend(g, q_abs, latent, lens_d, c.scale)
    pool, tables = page_latent(latent, lens, bs, seed=98 + bs)
    out = torch.full((5, 128, D_C), float("nan"), dtype=torch.bfloat16, device=DEV)
    ws = g.mla_absorbed_workspace(5, 128, D_C, tables.shape[1] * bs)
    g.attn_decode_mla_absorbed_paged(q_abs, pool, tables, lens_d, out, c.scale, workspace=ws)
    assert g.attn_get_device_error() == g.OK
    assert torch.equal(out, want)
    ref = oracle_latent(q_abs[3:4], latent[3:4], c.lens[3:4], c.scale)
    check(np.abs(out[3:4].float().cpu().numpy() - ref).max(), 2e-2)


def test_paged_equals_contiguous_at_2048_row_splits(gpu_lib):
    """A batch large enough for 2048-row splits (32 sequences of capacity 2112:
    32 * ceil(2112 / 2048) = 64 clusters at that size): paged equals contiguous
    bit for bit, lengths across the 2048-row boundary, one sequence against the
    oracle."""
    g = gpu_lib
    B, L = 32, 2112
    lens = [int(x) for x in torch.randint(1, L + 1, (B,), generator=W.generator(130))]
    lens[0], lens[1], lens[2] = 2048, 2049, L
    c = W.make_mla_absorbed(B=B, H=128, max_len=L, lens=lens, seed=131)
    q_abs = absorbed_q(g, c)
    latent = c.latent.to(DEV)
    lens_d = c.lens.to(DEV)
    want = attend(g, q_abs, latent, lens_d, c.scale)
    assert g.attn_get_device_error() == g.OK
    assert g.attn_decode_mla_absorbed_workspace_bytes(B, 128, D_C, L) == B * 128 * 2 * (D_C + 2) * 4  # two splits
    pool, tables = page_latent(latent, lens, 16, seed=132)
    out = torch.full((B, 128, D_C), float("nan"), dtype=torch.bfloat16, device=DEV)
    ws = g.mla_absorbed_workspace(B, 128, D_C, tables.shape[1] * 16)
    g.attn_decode_mla_absorbed_paged(q_abs, pool, tables, lens_d, out, c.scale, workspace=ws)
    assert g.attn_get_device_error() == g.OK
    assert torch.equal(out, want)
    ref = oracle_latent(q_abs[1:2], latent[1:2], c.lens[1:2], c.scale)
    check(np.abs(out[1:2].float().cpu().numpy() - ref).max(), 2e-2)


def test_paged_bad_entry_is_flagged(gpu_lib):
    """A table entry outside the pool for a visible row sets the bounds error; the
    other sequences' outputs are unaffected."""
    g = gpu_lib
    lens = [300, 700]
    c = W.make_mla_absorbed(B=2, H=128, max_len=704, lens=lens, seed=99)
    q_abs = absorbed_q(g, c)
    latent = c.latent.to(DEV)
    pool, tables = page_latent(latent, lens, 16, seed=100)
    good = torch.empty(2, 128, D_C, dtype=torch.bfloat16, device=DEV)
    g.attn_decode_mla_absorbed_paged(q_abs, pool, tables, c.lens.to(DEV), good, c.scale)
    assert g.attn_get_device_error() == g.OK
    tables[0, 5] = pool.shape[0] + 7
    out = torch.empty(2, 128, D_C, dtype=torch.bfloat16, device=DEV)
    g.attn_decode_mla_absorbed_paged(q_abs, pool, tables, c.lens.to(DEV), out, c.scale)
    assert g.attn_get_device_error() == g.ERR_DEVICE_BOUNDS
    assert torch.equal(out[1], good[1])


def test_projections_other_widths_match_oracle(gpu_lib):
    """Widths the tensor-core projection does not take (rows not a multiple of
    128, K not a multiple of 64) go through the SIMT kernel: same bound."""
    g = gpu_lib
    B, H, dn, dr, dc, dv = 5, 3, 40, 16, 96, 24
    gen = W.generator(101)
    q = W.randn((B, H, dn + dr), gen, torch.bfloat16)
    k_b = (W.randn((H, dc, dn), gen) / 6.0).to(torch.bfloat16)
    v_b = (W.randn((H, dv, dc), gen) / 10.0).to(torch.bfloat16)
    q_abs = torch.empty(B, H, dc + dr, dtype=torch.bfloat16, device=DEV)
    g.mla_absorb_q(q.to(DEV), k_b.to(DEV), q_abs)
    want = core.mla_absorb_q(W.to_oracle(q), W.to_oracle(k_b), dn)
    got = q_abs.float().cpu().numpy()
    assert np.all(np.abs(got - want) <= 2.0 ** -8 * np.abs(want) + 1e-3)
    out = torch.empty(B, H, dv, dtype=torch.bfloat16, device=DEV)
    g.mla_unabsorb_out(q_abs[..., :dc].contiguous(), v_b.to(DEV), out)
    want = core.mla_unabsorb_out(W.to_oracle(q_abs[..., :dc]), W.to_oracle(v_b))
    assert np.all(np.abs(out.float().cpu().numpy() - want) <= 2.0 ** -8 * np.abs(want) + 1e-3)
    assert g.attn_get_device_error() == g.OK


def test_long_sequence_many_splits(gpu_lib):
    """One 40,000-row sequence (40 splits: the combine walks its split weights in
    two passes of 32) and a short one beside it, against the oracle."""
    g = gpu_lib
    c = W.make_mla_absorbed(B=2, H=128, max_len=40000, lens=[40000, 5], seed=102, device=DEV)
    q_abs = absorbed_q(g, c)
    out = attend(g, q_abs, c.latent, c.lens, c.scale)
    assert g.attn_get_device_error() == g.OK
    want = oracle_latent(q_abs, c.latent, c.lens, c.scale)
    err = np.abs(out.float().cpu().numpy() - want).max()
    check(err, 2e-2)
