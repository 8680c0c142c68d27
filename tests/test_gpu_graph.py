"""The decode and prefill steps captured in a CUDA graph and replayed: every
kernel of the library is launched as a programmatic dependent of the one before,
and a captured step must give the same bits as the same step run eagerly. (The
entry point that allocates nothing is left out: it makes no claim about graphs.)"""
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _restore(dst, src):
    for d, s in zip(dst, src):
        d.copy_(s)


def test_paged_decode_step_replays_in_a_graph(gpu_lib):
    """kv_append_paged + attn_decode_paged (plan, attention, combine) captured
    once, replayed twice from the same inputs: equal to the eager step."""
    g = gpu_lib
    c = W.make_paged(B=24, H=32, Hkv=8, dk=128, dv=128, block_size=16, num_blocks=12000, len_lo=1, len_hi=5000,
                     seed=140, device=DEV)
    lens = c.seq_lens.clone()
    state = [c.q, c.k_pool, c.v_pool, lens]
    saved = [t.clone() for t in state]
    out = torch.empty(24, 32, 128, dtype=torch.bfloat16, device=DEV)
    ws = g.decode_workspace(24, 32, 128, c.tables.shape[1] * 16, device=DEV)

    def step():
        g.kv_append_paged(c.q, c.k_new, c.v_new, c.k_pool, c.v_pool, c.tables, lens, lens, c.theta)
        g.attn_decode_paged(c.q, c.k_pool, c.v_pool, c.tables, lens, out, c.scale, workspace=ws)

    step()  # eager (also sets the kernels' attributes before any capture)
    torch.cuda.synchronize()
    assert g.attn_get_device_error() == g.OK
    want = out.clone()
    want_lens = lens.clone()

    _restore(state, saved)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for _ in range(2):
        _restore(state, saved)
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert g.attn_get_device_error() == g.OK
        assert torch.equal(out, want)
        assert torch.equal(lens, want_lens)


def test_prefill_step_replays_in_a_graph(gpu_lib):
    """RoPE of q and k, then the tensor-core prefill, captured once and replayed:
    equal to the eager step."""
    g = gpu_lib
    B, S, H, Hkv, d = 1, 1024, 14, 2, 64
    c = W.make_prefill(B=B, S=S, H=H, Hkv=Hkv, dk=d, dv=d, seed=141, device=DEV)
    pos = torch.arange(S, dtype=torch.int32, device=DEV)[None].repeat(B, 1).contiguous()
    state = [c.q, c.k]
    saved = [t.clone() for t in state]
    out = torch.empty(B, S, H, d, dtype=torch.bfloat16, device=DEV)

    def step():
        g.attn_rope_interleaved(c.q, pos, 1e6)
        g.attn_rope_interleaved(c.k, pos, 1e6, heads_outer=True)
        g.attn_prefill_causal(c.q, c.k, c.v, out, c.scale)

    step()
    torch.cuda.synchronize()
    assert g.attn_get_device_error() == g.OK
    want = out.clone()

    _restore(state, saved)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for _ in range(2):
        _restore(state, saved)
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert g.attn_get_device_error() == g.OK
        assert torch.equal(out, want)


def test_absorbed_mla_step_replays_in_a_graph(gpu_lib):
    """mla_absorb_q + attn_decode_mla_absorbed (two-CTA cluster kernel, split
    combine) + mla_unabsorb_out captured once and replayed: equal to the eager step."""
    g = gpu_lib
    B, H, L = 4, 128, 2500
    c = W.make_mla_absorbed(B=B, H=H, max_len=L, lens=[2500, 900, 1, 2049], seed=142, device=DEV)
    q_abs = torch.empty(B, H, 576, dtype=torch.bfloat16, device=DEV)
    out_lat = torch.empty(B, H, 512, dtype=torch.bfloat16, device=DEV)
    out = torch.empty(B, H, 128, dtype=torch.bfloat16, device=DEV)
    ws = g.mla_absorbed_workspace(B, H, 512, L, device=DEV)

    def step():
        g.mla_absorb_q(c.q, c.k_b, q_abs)
        g.attn_decode_mla_absorbed(q_abs, c.latent, c.lens, out_lat, c.scale, workspace=ws)
        g.mla_unabsorb_out(out_lat, c.v_b, out)

    step()
    torch.cuda.synchronize()
    assert g.attn_get_device_error() == g.OK
    want = out.clone()

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for _ in range(2):
        out.fill_(float("nan"))
        out_lat.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert g.attn_get_device_error() == g.OK
        assert torch.equal(out, want)
