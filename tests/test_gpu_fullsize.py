"""The three decode workloads at their full sizes, against the fp64 oracle (GPU).

Each test builds the workload exactly as the benchmark does (same generator,
seeds, shapes and launch: the same entry points with the same workspace), runs
it on the GPU, and compares sampled sequences with the oracle element by
element, within 2e-2 (bf16 inputs, fp32 accumulation; the oracle reads the same
bf16 values widened to fp64). The oracle finishes a sampled sequence in well
under a second, so the samples reach every length class of the workload: the
shortest and longest histories, ones that end at and just past a split
boundary, and seeded others.

* paged decode -- 256 sequences, H=32, Hkv=8, d=128, block size 16, a
  600,000-block pool (19.7 GB per pool: byte offsets far beyond 2^32), histories
  U[1, 32768] and one appended row (RoPE theta 1e6) per sequence. 32 sequences go
  through the oracle's append and decode from the pristine pool; the same 32 are
  also decoded from contiguous copies of their (appended) rows, which must give
  the paged output bit for bit (frink-models src/decoder/attn_block.rs,
  `push_and_attend_row`: paging changes where rows live and nothing else).
* contiguous decode -- all 64 sequences of the [64, 8, 8192, 128] cache.
* MLA-shaped decode -- 32 sequences, 128 heads, d_k = 128 + 64 shared rotated
  part (RoPE theta 1e4 as setup), d_v = 128, 4096 rows; four sequences through
  the oracle's naive per-head form (frink-models src/mla/mod.rs,
  `naive_attention`).
"""
import numpy as np
import pytest
import torch

import workloads as W
from margins import check
from oracle import core

pytestmark = pytest.mark.gpu
DEV = "cuda"
SPLIT = 2048  # rows of one split-K unit of the decode


def need_free(nbytes):
    free, _ = torch.cuda.mem_get_info()
    if free < nbytes:
        pytest.fail(f"the full-size workload needs {nbytes / 2**30:.1f} GiB free on the device, "
                    f"{free / 2**30:.1f} GiB are")


def maxerr(gpu_rows, want):
    return float(np.abs(gpu_rows.float().cpu().numpy().astype(np.float64) - want).max())


def pick_sequences(rows, n, seed):
    """Indices of the shortest and longest `rows`, those ending exactly at and
    just past a split boundary (closest available), then seeded others, n in all."""
    order = np.argsort(rows, kind="stable")
    pick = [int(order[0]), int(order[-1])]
    for target in (SPLIT, 2 * SPLIT, SPLIT + 1, 8 * SPLIT + 1):
        b = int(np.argmin(np.abs(rows - target)))
        if b not in pick:
            pick.append(b)
    for b in torch.randperm(len(rows), generator=W.generator(seed)).tolist():
        if len(pick) >= n:
            break
        if b not in pick:
            pick.append(b)
    return pick


def test_paged_decode_full_size(gpu_lib):
    g = gpu_lib
    B, H, Hkv, d, bs, nb = 256, 32, 8, 128, 16, 600_000
    need_free(2 * nb * Hkv * bs * d * 2 + (8 << 30))
    dev = torch.device(DEV)
    c = W.make_paged(B=B, H=H, Hkv=Hkv, dk=d, dv=d, block_size=bs, num_blocks=nb, seed=3, device=dev)
    gi = W.generator(77, dev)  # the benchmark's first step's new rows
    q = W.randn((B, H, d), gi, torch.bfloat16, dev)
    kn = W.randn((B, Hkv, d), gi, torch.bfloat16, dev)
    vn = W.randn((B, Hkv, d), gi, torch.bfloat16, dev)
    hist = c.seq_lens.cpu().numpy().astype(np.int64)
    pick = pick_sequences(hist + 1, 32, seed=5)
    # host copies of the sampled sequences' pristine blocks, in table order
    sample = []
    for b in pick:
        nblk = (int(hist[b]) + 1 + bs - 1) // bs
        blocks = c.tables[b, :nblk].long()
        sample.append(dict(b=b, blocks=blocks, kp=W.to_oracle(c.k_pool[blocks]), vp=W.to_oracle(c.v_pool[blocks]),
                           q=W.to_oracle(q[b:b + 1]), kn=W.to_oracle(kn[b:b + 1]), vn=W.to_oracle(vn[b:b + 1])))
    # the sampled blocks reach past 4 GiB into each pool (32 KiB per block)
    assert max(int(s["blocks"].max()) for s in sample) * Hkv * bs * d * 2 >= (1 << 32)

    lens_out = torch.empty_like(c.seq_lens)
    mbps = c.tables.shape[1]
    g.kv_append_paged(q, kn, vn, c.k_pool, c.v_pool, c.tables, c.seq_lens, lens_out, c.theta)
    out = torch.empty(B, H, d, dtype=torch.bfloat16, device=dev)
    ws = g.decode_workspace(B, H, d, mbps * bs, device=dev)
    g.attn_decode_paged(q, c.k_pool, c.v_pool, c.tables, lens_out, out, c.scale, workspace=ws)
    assert g.attn_get_device_error() == g.OK
    assert lens_out.cpu().numpy().tolist() == (hist + 1).tolist()

    worst = 0.0
    for s in sample:
        n = int(hist[s["b"]])
        table = np.arange(len(s["blocks"]), dtype=np.int32)[None]
        q2, kp2, vp2, l2 = core.kv_append_paged(s["q"], s["kn"], s["vn"], s["kp"], s["vp"], table, [n], c.theta)
        want = core.decode_paged(q2, kp2, vp2, table, l2, c.scale)
        worst = max(worst, maxerr(out[s["b"]:s["b"] + 1], want))
    check(worst, 2e-2, f"{len(sample)} sampled sequences, {int((hist[pick] + 1).sum())} rows")

    # the same sequences from contiguous copies of their rows: bit for bit
    L = int(hist[pick].max()) + 1
    kc = torch.zeros(len(pick), Hkv, L, d, dtype=torch.bfloat16, device=dev)
    vc = torch.zeros_like(kc)
    for i, s in enumerate(sample):
        n = int(hist[s["b"]]) + 1
        rows_k = c.k_pool[s["blocks"].to(dev)].permute(1, 0, 2, 3).reshape(Hkv, -1, d)[:, :n]
        rows_v = c.v_pool[s["blocks"].to(dev)].permute(1, 0, 2, 3).reshape(Hkv, -1, d)[:, :n]
        kc[i, :, :n] = rows_k
        vc[i, :, :n] = rows_v
    idx = torch.tensor(pick, device=dev)
    out_c = torch.empty(len(pick), H, d, dtype=torch.bfloat16, device=dev)
    wsc = g.decode_workspace(len(pick), H, d, L, device=dev)
    g.attn_decode_contig(q[idx].contiguous(), kc, vc, lens_out[idx].contiguous(), out_c, c.scale, workspace=wsc)
    assert g.attn_get_device_error() == g.OK
    assert torch.equal(out_c, out[idx]), "paged and contiguous decode of the same rows must be bit-identical"


def test_contig_decode_full_size(gpu_lib):
    g = gpu_lib
    B, H, Hkv, d, L = 64, 32, 8, 128, 8192
    need_free(2 * B * Hkv * L * d * 2 + (4 << 30))
    dev = torch.device(DEV)
    c = W.make_contig(B=B, H=H, Hkv=Hkv, dk=d, dv=d, max_len=L, seed=2, device=dev)
    out = torch.empty(B, H, d, dtype=torch.bfloat16, device=dev)
    ws = g.decode_workspace(B, H, d, L, device=dev)
    g.attn_decode_contig(c.q, c.k, c.v, c.seq_lens, out, c.scale, workspace=ws)
    assert g.attn_get_device_error() == g.OK
    lens = c.seq_lens.cpu().numpy()
    want = core.decode_contig(W.to_oracle(c.q), W.to_oracle(c.k), W.to_oracle(c.v), lens, c.scale)
    check(maxerr(out, want), 2e-2, f"all {B} sequences, {int(lens.sum())} rows")


def test_mla_shaped_decode_full_size(gpu_lib):
    g = gpu_lib
    B, H, L = 32, 128, 4096
    need_free(2 * B * H * L * 128 * 2 + (4 << 30))
    dev = torch.device(DEV)
    c = W.make_mla(B=B, H=H, cache_len=L, seed=4, device=dev)
    pos = torch.arange(L, dtype=torch.int32, device=dev)[None].repeat(B, 1)
    # setup, as the benchmark does it: RoPE theta 1e4 on the shared k_rot (once
    # per position) and on every head's q rot slice at position L - 1
    g.attn_rope_interleaved(c.k_rot.view(B, L, 1, 64), pos, 1e4)
    g.attn_rope_interleaved(c.q.view(B, 1, H, 192), pos[:, -1:].contiguous(), 1e4, rot_offset=128, rot_dim=64)
    out = torch.empty(B, H, 128, dtype=torch.bfloat16, device=dev)
    ws = g.decode_workspace(B, H, 128, L, device=dev)
    g.attn_decode_contig(c.q, c.k, c.v, c.seq_lens, out, c.scale, workspace=ws, k_rot_shared=c.k_rot)
    assert g.attn_get_device_error() == g.OK
    pick = [0, B - 1] + [b for b in torch.randperm(B, generator=W.generator(8)).tolist() if b not in (0, B - 1)][:2]
    worst = 0.0
    for b in pick:
        sl = slice(b, b + 1)
        want = core.decode_mla_naive(W.to_oracle(c.q[sl]), W.to_oracle(c.k[sl]), W.to_oracle(c.k_rot[sl]),
                                     W.to_oracle(c.v[sl]), [L], c.scale)
        worst = max(worst, maxerr(out[sl], want))
    check(worst, 2e-2, f"sequences {pick}")
