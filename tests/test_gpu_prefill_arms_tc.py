"""The arms of the attention row on the tensor-core prefill (GPU): sliding
window, sink logits, logit softcap and ALiBi slopes (frink-models
src/decoder/attn_block.rs, `push_and_attend_row`: one kernel for plain,
windowed, softcapped and sink-bearing layers) against the oracle's
`attention_arms`, for the three head shapes the kernel takes, windows smaller
and larger than a 128-key tile, several query tiles at non-zero offsets, and the
paged pool against the contiguous cache bit for bit."""
import numpy as np
import pytest
import torch

import workloads as W
from margins import check
from oracle import core

pytestmark = pytest.mark.gpu
DEV = "cuda"

ARMS = {
    "window": dict(window=200),
    "window_small": dict(window=37),
    "sinks": dict(sinks=True),
    "softcap": dict(softcap=5.0),
    "alibi": dict(alibi=True),
    "all": dict(window=300, sinks=True, softcap=30.0, alibi=True),
}


def _arms(a, H, seed):
    rng = np.random.default_rng(seed)
    sinks = (2.0 * rng.standard_normal(H)).astype(np.float32) if a.get("sinks") else None
    slopes = np.array([2.0 ** (-8.0 * (h + 1) / H) for h in range(H)], np.float32) if a.get("alibi") else None
    return a.get("window", 0), a.get("softcap", 0.0), sinks, slopes


def _t(x):
    return None if x is None else torch.from_numpy(x).to(DEV)


def _f64(x):
    return None if x is None else x.astype(np.float64)


@pytest.mark.parametrize("dk,dv,H,Hkv", [(64, 64, 8, 2), (128, 128, 8, 4), (192, 128, 4, 4)])
@pytest.mark.parametrize("name", list(ARMS))
def test_tc_prefill_arms_match_oracle(gpu_lib, dk, dv, H, Hkv, name):
    g = gpu_lib
    S, offs = 520, [0, 75]
    c = W.make_prefill(B=2, S=S, H=H, Hkv=Hkv, dk=dk, dv=dv, seed=300, S_kv=S + 75, offsets=offs)
    window, cap, sinks, slopes = _arms(ARMS[name], H, 301)
    out = torch.empty(2, S, H, dv, dtype=torch.bfloat16, device=DEV)
    g.attn_prefill_causal(c.q.to(DEV), c.k.to(DEV), c.v.to(DEV), out, c.scale, position_offset=c.offsets.to(DEV),
                          window=window, softcap=cap, sinks=_t(sinks), alibi_slopes=_t(slopes))
    assert g.attn_get_device_error() == g.OK
    want = core.attention_arms(W.to_oracle(c.q), W.to_oracle(c.k), W.to_oracle(c.v), [o + S for o in offs], c.scale,
                               window, cap, _f64(sinks), _f64(slopes))
    check(float(np.abs(out.float().cpu().numpy() - want).max()), 2e-2, name)


@pytest.mark.parametrize("bs", [16, 64])
def test_tc_prefill_arms_paged_equals_contig_bits(gpu_lib, bs):
    """Every arm on: the chunk against the paged pool gives the contiguous
    cache's output bit for bit (same tiles, same arithmetic)."""
    g = gpu_lib
    H, Hkv, d, S = 8, 2, 64, 300
    offs = [40, 700]
    c = W.make_prefill(B=2, S=S, H=H, Hkv=Hkv, dk=d, dv=d, seed=310, S_kv=S + 700, offsets=offs)
    window, cap, sinks, slopes = _arms(ARMS["all"], H, 311)
    arms = dict(window=window, softcap=cap, sinks=_t(sinks), alibi_slopes=_t(slopes))
    out_c = torch.empty(2, S, H, d, dtype=torch.bfloat16, device=DEV)
    g.attn_prefill_causal(c.q.to(DEV), c.k.to(DEV), c.v.to(DEV), out_c, c.scale, position_offset=c.offsets.to(DEV),
                          **arms)
    # the same rows scattered over a shuffled pool of bs-row blocks
    L = S + 700
    nblk = (L + bs - 1) // bs
    perm = torch.randperm(2 * nblk + 5, generator=W.generator(312)).to(torch.int32)
    kp = torch.zeros(2 * nblk + 5, Hkv, bs, d, dtype=torch.bfloat16)
    vp = torch.zeros_like(kp)
    tables = torch.full((2, nblk), -1, dtype=torch.int32)
    for b in range(2):
        for blk in range(nblk):
            e = perm[b * nblk + blk]
            tables[b, blk] = e
            r = min(bs, L - blk * bs)
            kp[e, :, :r] = c.k[b, :, blk * bs:blk * bs + r]
            vp[e, :, :r] = c.v[b, :, blk * bs:blk * bs + r]
    out_p = torch.empty_like(out_c)
    g.attn_prefill_paged(c.q.to(DEV), kp.to(DEV), vp.to(DEV), tables.to(DEV), out_p, c.scale,
                         position_offset=c.offsets.to(DEV), **arms)
    assert g.attn_get_device_error() == g.OK
    assert torch.equal(out_p, out_c)
    want = core.attention_arms(W.to_oracle(c.q), W.to_oracle(c.k), W.to_oracle(c.v), [o + S for o in offs], c.scale,
                               window, cap, _f64(sinks), _f64(slopes))
    check(float(np.abs(out_c.float().cpu().numpy() - want).max()), 2e-2, "paged, every arm")


@pytest.mark.parametrize("dk,dv,H,Hkv", [(64, 64, 8, 2), (128, 128, 8, 4)])
def test_tc_prefill_softcap_saturates(gpu_lib, dk, dv, H, Hkv):
    """Logits far beyond the softcap (q scaled by 60, cap 1): most scores saturate
    to +-cap, where 2^x overflows to infinity or goes to 0 inside the kernel's tanh."""
    g = gpu_lib
    S = 300
    c = W.make_prefill(B=1, S=S, H=H, Hkv=Hkv, dk=dk, dv=dv, seed=310)
    q = (c.q.float() * 60.0).to(torch.bfloat16)
    out = torch.empty(1, S, H, dv, dtype=torch.bfloat16, device=DEV)
    g.attn_prefill_causal(q.to(DEV), c.k.to(DEV), c.v.to(DEV), out, c.scale, softcap=1.0)
    assert g.attn_get_device_error() == g.OK
    want = core.attention_arms(W.to_oracle(q), W.to_oracle(c.k), W.to_oracle(c.v), [S], c.scale, 0, 1.0, None, None)
    check(float(np.abs(out.float().cpu().numpy() - want).max()), 2e-2)
