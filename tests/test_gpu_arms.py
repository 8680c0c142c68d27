"""The arms of the attention row on the GPU (sliding window, sink logits, logit
softcap, ALiBi slopes; include/gqa_attn.h, `gqa_arms`) against the oracle's
`attention_arms` (oracle/gqa_oracle.c), and paged against contiguous bit for bit
with every arm on."""
import math

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


def alibi_slopes(H):
    # the usual geometric slopes 2^(-8 (h + 1) / H)
    return np.array([2.0 ** (-8.0 * (h + 1) / H) for h in range(H)], np.float32)


ARMS = [dict(window=1000), dict(sinks=True), dict(softcap=2.0), dict(alibi=True),
        dict(window=700, sinks=True, softcap=1.5, alibi=True), dict(window=1, sinks=True)]


def _arms_args(a, H):
    rng = np.random.default_rng(7)
    sinks = rng.standard_normal(H).astype(np.float32) if a.get("sinks") else None
    slopes = alibi_slopes(H) if a.get("alibi") else None
    return a.get("window", 0), a.get("softcap", 0.0), sinks, slopes


def _dev(x):
    return None if x is None else torch.from_numpy(x).to(DEV)


@pytest.mark.parametrize("dtype,H,Hkv,d", [(torch.bfloat16, 32, 8, 128), (torch.float32, 16, 2, 64)])
@pytest.mark.parametrize("arm", range(len(ARMS)))
def test_decode_contig_arms_match_oracle(gpu_lib, dtype, H, Hkv, d, arm):
    g = gpu_lib
    lens = [1, 300, 2047, 2049, 5000]
    L = 5100
    c = W.make_contig(B=len(lens), H=H, Hkv=Hkv, dk=d, dv=d, max_len=L, lens=lens, dtype=dtype, seed=70 + arm)
    window, cap, sinks, slopes = _arms_args(ARMS[arm], H)
    out = torch.empty(len(lens), H, d, dtype=dtype, device=DEV)
    g.attn_decode_contig(c.q.to(DEV), c.k.to(DEV), c.v.to(DEV), c.seq_lens.to(DEV), out, c.scale,
                         workspace=g.decode_workspace(len(lens), H, d, L), window=window, softcap=cap,
                         sinks=_dev(sinks), alibi_slopes=_dev(slopes))
    ok(g)
    want = core.attention_arms(W.to_oracle(c.q), W.to_oracle(c.k), W.to_oracle(c.v), lens, c.scale, window, cap,
                               None if sinks is None else sinks.astype(np.float64),
                               None if slopes is None else slopes.astype(np.float64))
    err = np.abs(out.float().cpu().numpy().astype(np.float64) - want).max()
    check(err, TOL[dtype])


def test_paged_equals_contig_bitwise_with_every_arm(gpu_lib):
    """Every arm on, lengths across split boundaries; the block-table entries of
    blocks wholly below a sequence's window are -1 (evicted): they must be neither
    read nor reported."""
    g = gpu_lib
    lens = [1, 17, 2047, 2049, 4500]
    B, H, Hkv, d, bs, window = len(lens), 32, 8, 128, 16, 1500
    L = 4600
    c = W.make_contig(B=B, H=H, Hkv=Hkv, dk=d, dv=d, max_len=L, lens=lens, seed=80)
    mbps = (L + bs - 1) // bs
    need = sum((n + bs - 1) // bs for n in lens)
    nb = need + 11
    perm = torch.randperm(nb, generator=W.generator(81)).to(torch.int32)
    kp = torch.randn(nb, Hkv, bs, d, generator=W.generator(82)).to(torch.bfloat16)
    vp = torch.randn(nb, Hkv, bs, d, generator=W.generator(83)).to(torch.bfloat16)
    tables = torch.full((B, mbps), -1, dtype=torch.int32)
    at = 0
    for b, n in enumerate(lens):
        lo = max(0, n - window)  # the first key the decode row sees
        for blk in range((n + bs - 1) // bs):
            e = perm[at]
            at += 1
            if (blk + 1) * bs <= lo:
                continue  # below the window: left as -1
            tables[b, blk] = e
            r = min(bs, n - blk * bs)
            kp[e, :, :r] = c.k[b, :, blk * bs:blk * bs + r]
            vp[e, :, :r] = c.v[b, :, blk * bs:blk * bs + r]
    _, cap, sinks, slopes = _arms_args(dict(sinks=True, alibi=True), H)
    arms = dict(window=window, softcap=1.75, sinks=_dev(sinks), alibi_slopes=_dev(slopes))
    out_p = torch.empty(B, H, d, dtype=torch.bfloat16, device=DEV)
    g.attn_decode_paged(c.q.to(DEV), kp.to(DEV), vp.to(DEV), tables.to(DEV), c.seq_lens.to(DEV), out_p, c.scale,
                        workspace=g.decode_workspace(B, H, d, mbps * bs), **arms)
    ok(g)
    out_c = torch.empty_like(out_p)
    g.attn_decode_contig(c.q.to(DEV), c.k.to(DEV), c.v.to(DEV), c.seq_lens.to(DEV), out_c, c.scale,
                         workspace=g.decode_workspace(B, H, d, L), **arms)
    ok(g)
    assert torch.equal(out_p, out_c)
    want = core.attention_arms(W.to_oracle(c.q), W.to_oracle(c.k), W.to_oracle(c.v), lens, c.scale, window, 1.75,
                               sinks.astype(np.float64), slopes.astype(np.float64))
    check(np.abs(out_c.float().cpu().numpy() - want).max(), 2e-2)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_prefill_arms_match_oracle(gpu_lib, dtype):
    g = gpu_lib
    B, S, H, Hkv, d = 2, 40, 8, 2, 64
    offs = [0, 17]
    c = W.make_prefill(B=B, S=S, H=H, Hkv=Hkv, dk=d, dv=d, dtype=dtype, seed=90, S_kv=S + 17, offsets=offs)
    _, cap, sinks, slopes = _arms_args(dict(sinks=True, alibi=True), H)
    out = torch.empty(B, S, H, d, dtype=dtype, device=DEV)
    g.attn_prefill_causal(c.q.to(DEV), c.k.to(DEV), c.v.to(DEV), out, c.scale, position_offset=c.offsets.to(DEV),
                          window=9, softcap=2.5, sinks=_dev(sinks), alibi_slopes=_dev(slopes))
    ok(g)
    base = [o + S for o in offs]
    want = core.attention_arms(W.to_oracle(c.q), W.to_oracle(c.k), W.to_oracle(c.v), base, c.scale, 9, 2.5,
                               sinks.astype(np.float64), slopes.astype(np.float64))
    check(np.abs(out.float().cpu().numpy() - want).max(), TOL[dtype])


def test_plain_call_equals_zero_arms(gpu_lib):
    """The arms switched off through the _ex call are the plain call, bit for bit."""
    g = gpu_lib
    lens = [5, 2600]
    c = W.make_contig(B=2, H=32, Hkv=8, dk=128, dv=128, max_len=2700, lens=lens, seed=95)
    ws = g.decode_workspace(2, 32, 128, 2700)
    a = torch.empty(2, 32, 128, dtype=torch.bfloat16, device=DEV)
    b = torch.empty_like(a)
    args = (c.q.to(DEV), c.k.to(DEV), c.v.to(DEV), c.seq_lens.to(DEV))
    g.attn_decode_contig(*args, a, c.scale, workspace=ws)
    g.attn_decode_contig(*args, b, c.scale, workspace=ws, window=100000, alibi_slopes=torch.zeros(32, device=DEV))
    ok(g)
    assert torch.equal(a, b)


def test_decode_softcap_saturates(gpu_lib):
    """Logits far beyond the softcap: q scaled so that |scale q.k| reaches the
    hundreds with a cap of 1, so cap * tanh(s / cap) saturates to +-cap (e^(2t)
    overflowing to infinity, or to 0) for most keys and is still checked against
    the oracle's tanh for the rest."""
    g = gpu_lib
    lens = [5, 700, 2049]
    B, H, Hkv, d, L = len(lens), 32, 8, 128, 2100
    c = W.make_contig(B=B, H=H, Hkv=Hkv, dk=d, dv=d, max_len=L, lens=lens, seed=95)
    q = (c.q.float() * 60.0).to(torch.bfloat16)
    out = torch.empty(B, H, d, dtype=torch.bfloat16, device=DEV)
    g.attn_decode_contig(q.to(DEV), c.k.to(DEV), c.v.to(DEV), c.seq_lens.to(DEV), out, c.scale,
                         workspace=g.decode_workspace(B, H, d, L), softcap=1.0)
    ok(g)
    s_max = float((q.float()[2, 0] @ c.k.float()[2, 0, :lens[2]].T).abs().max() * c.scale)
    assert s_max > 50.0  # the scores do reach far past the cap
    want = core.attention_arms(W.to_oracle(q), W.to_oracle(c.k), W.to_oracle(c.v), lens, c.scale, 0, 1.0, None, None)
    check(float(np.abs(out.float().cpu().numpy().astype(np.float64) - want).max()), TOL[torch.bfloat16])
