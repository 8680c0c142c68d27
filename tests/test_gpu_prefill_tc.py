"""The tcgen05 causal prefill (bf16, d = 64 and d = 128) against the fp64 oracle (GPU)."""
import numpy as np
import pytest
import torch

import workloads as W
from margins import check
from oracle import core

pytestmark = pytest.mark.gpu
DEV = "cuda"


def run(g, c):
    B, S, H, _ = c.q.shape
    out = torch.full((B, S, H, c.v.shape[-1]), float("nan"), dtype=torch.bfloat16, device=DEV)
    g.attn_prefill_causal(c.q.to(DEV), c.k.to(DEV), c.v.to(DEV), out, c.scale, position_offset=c.offsets.to(DEV))
    assert g.attn_get_device_error() == g.OK
    return out


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("B,S,H,Hkv,offs", [
    (1, 128, 2, 1, [0]), (1, 256, 4, 2, [0]), (1, 300, 14, 2, [0]), (2, 200, 6, 3, [0, 37]),
    (1, 1, 2, 2, [5]), (2, 129, 8, 1, [128, 3]), (1, 520, 4, 4, [0])])
def test_prefill_tc_matches_oracle(gpu_lib, B, S, H, Hkv, offs, d):
    g = gpu_lib
    extra = max(offs)
    c = W.make_prefill(B=B, S=S, H=H, Hkv=Hkv, dk=d, dv=d, seed=70 + S + d, S_kv=S + extra + 5, offsets=offs)
    out = run(g, c)
    want = core.prefill_causal(W.to_oracle(c.q), W.to_oracle(c.k), W.to_oracle(c.v), c.scale, offsets=offs)
    err = np.abs(out.float().cpu().numpy() - want).max()
    check(err, 2e-2)


def test_prefill_tc_full_size_config(gpu_lib):
    """The causal prefill workload at full size: B=1, H=14, Hkv=2, d=64, 2048 rows,
    interleaved RoPE (theta 1e6) applied to q and k first; every output checked."""
    g = gpu_lib
    c = W.make_prefill(B=1, S=2048, H=14, Hkv=2, dk=64, dv=64, seed=1)
    pos = torch.arange(2048, dtype=torch.int32)[None]
    q, k = c.q.to(DEV), c.k.to(DEV)
    g.attn_rope_interleaved(q, pos.to(DEV), 1e6)
    g.attn_rope_interleaved(k, pos.to(DEV), 1e6, heads_outer=True)
    out = torch.empty(1, 2048, 14, 64, dtype=torch.bfloat16, device=DEV)
    g.attn_prefill_causal(q, k, c.v.to(DEV), out, c.scale)
    assert g.attn_get_device_error() == g.OK
    # oracle: its own RoPE of the raw inputs, rounded to bf16 as the cache stores them
    qo = core.rope_interleaved(W.to_oracle(c.q), W.to_oracle(pos), 0, 64, 1e6)
    ko = np.ascontiguousarray(core.rope_interleaved(np.ascontiguousarray(W.to_oracle(c.k).transpose(0, 2, 1, 3)),
                                                    W.to_oracle(pos), 0, 64, 1e6).transpose(0, 2, 1, 3))
    want = core.prefill_causal(qo, ko, W.to_oracle(c.v), c.scale)
    err = np.abs(out.float().cpu().numpy() - want).max()
    check(err, 2e-2)


@pytest.mark.parametrize("d", [64, 128])
def test_prefill_tc_zero_keys_give_prefix_mean(gpu_lib, d):
    """K = 0: every visible key scores 0, so row i is the mean of V[0..=i]."""
    g = gpu_lib
    c = W.make_prefill(B=1, S=300, H=4, Hkv=2, dk=d, dv=d, seed=71)
    c.k.zero_()
    out = run(g, c)
    v = c.v.float()[0]                                       # [Hkv, S, d]
    mean = torch.cumsum(v, dim=1) / torch.arange(1, 301)[None, :, None]
    want = mean.repeat_interleave(2, dim=0).permute(1, 0, 2)  # [S, H, d]
    check((out[0].float().cpu() - want).abs().max().item(), 2e-2)


@pytest.mark.parametrize("d", [64, 128])
def test_prefill_tc_decode_step_is_last_row(gpu_lib, d):
    g = gpu_lib
    c = W.make_prefill(B=1, S=640, H=8, Hkv=2, dk=d, dv=d, seed=72)
    out = run(g, c)
    dec = torch.empty(1, 8, d, dtype=torch.bfloat16, device=DEV)
    g.attn_decode_contig(c.q[:, 639].contiguous().to(DEV), c.k.to(DEV), c.v.to(DEV),
                         torch.tensor([640], dtype=torch.int32, device=DEV), dec, c.scale)
    check((dec.float() - out[:, 639].float()).abs().max().item(), 2e-2)


def test_prefill_tc_d128_model_shape(gpu_lib):
    """d = 128 at the decode configs' head shape (H=32, Hkv=8): two sequences, one
    at an offset inside the second key tile; every output against the oracle."""
    g = gpu_lib
    offs = [0, 200]
    c = W.make_prefill(B=2, S=1024, H=32, Hkv=8, dk=128, dv=128, seed=73, S_kv=1024 + 200, offsets=offs)
    out = run(g, c)
    want = core.prefill_causal(W.to_oracle(c.q), W.to_oracle(c.k), W.to_oracle(c.v), c.scale, offsets=offs)
    err = np.abs(out.float().cpu().numpy() - want).max()
    check(err, 2e-2)


@pytest.mark.parametrize("B,S,H,Hkv,offs", [(1, 90, 4, 4, [0]), (2, 300, 8, 8, [0, 140]), (1, 257, 6, 2, [5])])
def test_prefill_tc_mla_shape(gpu_lib, B, S, H, Hkv, offs):
    """The MLA shape on the tensor cores: d_k = 192 (Q and K rows of three 64-column
    blocks), d_v = 128; group size 1 as in the pages' MLA and a grouped case."""
    g = gpu_lib
    c = W.make_prefill(B=B, S=S, H=H, Hkv=Hkv, dk=192, dv=128, seed=75 + S, S_kv=S + max(offs) + 2, offsets=offs)
    out = run(g, c)
    want = core.prefill_causal(W.to_oracle(c.q), W.to_oracle(c.k), W.to_oracle(c.v), c.scale, offsets=offs)
    err = np.abs(out.float().cpu().numpy() - want).max()
    check(err, 2e-2)


@pytest.mark.parametrize("H,Hkv,dk,dv", [(32, 8, 128, 128), (32, 32, 192, 128)])
def test_prefill_tc_full_size_wide_heads_sampled_rows(gpu_lib, H, Hkv, dk, dv):
    """The d = 128 and MLA-shaped prefill workloads the bench times (2048 rows):
    sampled rows -- first, last and seeded others, every head -- against the
    oracle, each row computed on its own as a one-row chunk at its position."""
    g = gpu_lib
    S = 2048
    c = W.make_prefill(B=1, S=S, H=H, Hkv=Hkv, dk=dk, dv=dv, seed=7)
    out = run(g, c).cpu()
    rng = np.random.default_rng(76)
    worst = 0.0
    for i in sorted({0, 127, 128, S - 1, *rng.integers(0, S, 4).tolist()}):
        want = core.prefill_causal(W.to_oracle(c.q[:, i:i + 1].contiguous()),
                                   W.to_oracle(c.k[:, :, :i + 1].contiguous()),
                                   W.to_oracle(c.v[:, :, :i + 1].contiguous()), c.scale, offsets=[i])
        worst = max(worst, np.abs(out[:, i:i + 1].float().numpy() - want).max())
    check(worst, 2e-2)


@pytest.mark.parametrize("dk,dv", [(128, 128), (192, 128)])
def test_prefill_tc_wide_zero_keys_give_prefix_mean(gpu_lib, dk, dv):
    """K = 0 at the wide head shapes: every visible key scores 0, so row i is the
    mean of V[0..=i] (a closed form independent of the oracle)."""
    g = gpu_lib
    c = W.make_prefill(B=1, S=200, H=4, Hkv=2, dk=dk, dv=dv, seed=77)
    c.k.zero_()
    out = run(g, c)
    v = c.v.float()[0]                                       # [Hkv, S, dv]
    mean = torch.cumsum(v, dim=1) / torch.arange(1, 201)[None, :, None]
    want = mean.repeat_interleave(2, dim=0).permute(1, 0, 2)  # [S, H, dv]
    check((out[0].float().cpu() - want).abs().max().item(), 2e-2)
