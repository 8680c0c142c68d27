"""Benchmark: paged GQA decode HBM GB/s (headline) and causal prefill TFLOP/s.

Headline step (the paged decode workload): kv_append_paged (one new row per
sequence, interleaved RoPE on q and k) + attn_decode_paged over 256 sequences
whose histories are U[1, 32768] rows in a 600,000-block shared pool. The K/V
working set (~17 GB per step) is far larger than L2, so steps need no flush.

The same run also measures, as secondary objects of the one JSON line:
  prefill  -- causal prefill bf16, B=1, H=14, Hkv=2, d=64, S=2048 (tcgen05),
              with RoPE on q and k in the step; TFLOP/s against the bf16 peak
  prefill_arms -- the same with a 512-row window, sinks, ALiBi and softcap
  contig   -- contiguous decode bf16, 64 sequences, len U[512, 8192]
  mla      -- MLA-shaped decode bf16, 32 sequences, 128 heads, d_k 128+64 shared
              rotated part, d_v 128, len 4096

`--impl reference` times the fp64 CPU oracle on the host cores on a bounded
sample of the paged workload. Under torchrun each rank runs its own replica
(its own seed) on its own GPU: sequences shard with no exchange (weak scaling);
only timings cross ranks.
"""
import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "paged GQA decode HBM GB/s (% of ~8 TB/s); causal prefill TFLOP/s (% peak)"
NOMINAL_HBM_GBS = 8000.0


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except OSError:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


# ---------------------------------------------------------------------------
# distributed plumbing (rank-local replicas; only timings cross ranks)

def dist_setup():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    if torch.cuda.is_available():
        torch.cuda.set_device(local)
    return rank, world


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def reduce_over_ranks(x, world, op="max"):
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX if op == "max" else dist.ReduceOp.SUM)
    return float(t.item())


# ---------------------------------------------------------------------------
# clocks during the timed region

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, index):
        self.index, self.proc, self.out = index, None, ""

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.out = self.proc.communicate(timeout=5)[0]
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        rows = [[p.strip() for p in line.split(",")] for line in (self.out or "").strip().splitlines()]
        rows = [r for r in rows if len(r) == 7]
        num = lambda s: float(s) if s.replace(".", "", 1).isdigit() else None
        sm = [v for v in (num(r[0]) for r in rows) if v is not None]
        mx = [v for v in (num(r[1]) for r in rows) if v is not None]
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        reasons = sorted({self.NAMES[i] for r in rows for i in range(4) if r[3 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(sm)}


def queue_ahead(n_launch_groups, us_per_group=100.0):
    """Keep the current stream busy long enough (a device-side spin of about
    n_launch_groups * us_per_group microseconds at ~2 GHz) for the host to queue
    the launches that follow."""
    torch.cuda._sleep(int(n_launch_groups * us_per_group * 2000))


def timed(fn, steps, st, sync_first=True):
    """Time `steps` calls of fn(k) with CUDA events on stream st (synchronised on
    both sides); returns ms per call."""
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if sync_first:
        torch.cuda.synchronize()
    t0.record(st)
    for k in range(steps):
        fn(k)
    t1.record(st)
    torch.cuda.synchronize()
    return t0.elapsed_time(t1) / steps


# ---------------------------------------------------------------------------
# paged decode (headline)

def paged_bytes(lens_after, B, H, Hkv, dk, dv, bs, es=2):
    """Algorithmic bytes of one step. Decode: every visible K/V row read once,
    the block-table entries those rows need, q read and out written. Append: q
    read and written back, the new k and v read, one K and one V row written per
    KV head."""
    rows = int(np.sum(lens_after))
    dec = rows * Hkv * (dk + dv) * es + int(np.sum((lens_after + bs - 1) // bs)) * 4 + B * H * (dk + dv) * es
    app = 2 * B * H * dk * es + 2 * B * Hkv * (dk + dv) * es
    return dec, app


def run_paged(args, rank, world):
    import causal_gqa_attention_row_gb300 as g
    g.load()
    dev = torch.device("cuda")
    B, H, Hkv, d, bs, nb = args.seqs, 32, 8, 128, 16, args.pool_blocks
    need = 2 * nb * Hkv * bs * d * 2
    free, _ = torch.cuda.mem_get_info()
    if free < need + (4 << 30):
        raise SystemExit(f"not enough free device memory: {free / 2**30:.1f} GiB free, "
                         f"{(need + (4 << 30)) / 2**30:.1f} GiB needed")
    c = W.make_paged(B=B, H=H, Hkv=Hkv, dk=d, dv=d, block_size=bs, num_blocks=nb, seed=3 + 1000 * rank, device=dev)
    n_sets = args.warmup + args.steps
    gi = W.generator(77 + rank, dev)
    # one fresh (q, k_new, v_new) per step: the append rotates q in place
    qs = [W.randn((B, H, d), gi, torch.bfloat16, dev) for _ in range(n_sets)]
    kns = [W.randn((B, Hkv, d), gi, torch.bfloat16, dev) for _ in range(n_sets)]
    vns = [W.randn((B, Hkv, d), gi, torch.bfloat16, dev) for _ in range(n_sets)]
    lens_in = c.seq_lens
    lens_out = torch.empty_like(lens_in)
    tables = c.tables
    mbps = tables.shape[1]
    out = torch.empty(B, H, d, dtype=torch.bfloat16, device=dev)
    ws = g.decode_workspace(B, H, d, mbps * bs, device=dev)
    st = torch.cuda.current_stream()
    lens_after = c.seq_lens.cpu().numpy().astype(np.int64) + 1
    dec_bytes, app_bytes = paged_bytes(lens_after, B, H, Hkv, d, d, bs)

    sample = None
    if rank == 0 and not args.no_cpu_baseline:  # gathered from the pristine pool, before any step
        sample = gather_paged_sample(c, qs[0], kns[0], vns[0], args.cpu_seqs)

    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_sets)]

    def step(i):
        g.kv_append_paged(qs[i], kns[i], vns[i], c.k_pool, c.v_pool, tables, lens_in, lens_out, c.theta)
        evs[i][0].record(st)
        g.attn_decode_paged(qs[i], c.k_pool, c.v_pool, tables, lens_out, out, c.scale, workspace=ws)
        evs[i][1].record(st)

    for i in range(args.warmup):
        step(i)
        if i == 0 and sample:  # the step the CPU-baseline sample replays: keep its output rows
            for s in sample:
                s["gpu_out"] = out[s["b"]:s["b"] + 1].float().cpu().numpy()
    torch.cuda.synchronize()
    assert g.attn_get_device_error() == g.OK
    with ClockSampler(torch.cuda.current_device()) as clk:
        barrier(world)
        ms = timed(lambda k: step(args.warmup + k), args.steps, st)
        barrier(world)
    assert g.attn_get_device_error() == g.OK
    dec_ms = statistics.mean(evs[args.warmup + k][0].elapsed_time(evs[args.warmup + k][1])
                             for k in range(args.steps))
    ms_max = reduce_over_ranks(ms, world, "max")
    total_bytes = reduce_over_ranks(dec_bytes + app_bytes, world, "sum")
    res = {"value": total_bytes / (ms_max * 1e-3) / 1e9, "ms_per_step": ms_max, "decode_ms": dec_ms,
           "achieved_decode_gbs": dec_bytes / (dec_ms * 1e-3) / 1e9, "decode_bytes": dec_bytes,
           "append_bytes": app_bytes, "clocks": clk.summary(), "sample": sample, "rows": int(lens_after.sum())}
    if not args.no_e2e:
        res["e2e"] = run_paged_e2e(args, g, c, tables, lens_in, lens_out, out, ws, dec_bytes + app_bytes, world)
    if not args.no_secondary:
        res["arms"] = run_paged_arms(args, g, c, qs[0], tables, lens_out, out, ws, lens_after)
    del c, qs, kns, vns
    torch.cuda.empty_cache()
    return res


def run_paged_arms(args, g, c, q, tables, lens, out, ws, lens_after, window=4096):
    """The paged decode with every arm on (a 4096-row sliding window, sink logits,
    ALiBi slopes, a logit softcap) over the same pool and lengths. Algorithmic
    bytes: the K/V rows inside each sequence's window, their table entries, q
    and out."""
    B, H, d = q.shape
    Hkv, bs = c.k_pool.shape[1], c.k_pool.shape[2]
    dev = q.device
    sinks = W.randn((H,), W.generator(123, dev), torch.float32, dev)
    slopes = torch.tensor([2.0 ** (-8.0 * (h + 1) / H) for h in range(H)], dtype=torch.float32, device=dev)
    arms = dict(window=window, softcap=30.0, sinks=sinks, alibi_slopes=slopes)
    vis = np.minimum(lens_after, window)
    first_blk = (lens_after - vis) // bs
    last_blk = (lens_after - 1) // bs
    nbytes = int(vis.sum()) * Hkv * 2 * d * 2 + int((last_blk - first_blk + 1).sum()) * 4 + B * H * 2 * d * 2
    st = torch.cuda.current_stream()

    def step(_):
        g.attn_decode_paged(q, c.k_pool, c.v_pool, tables, lens, out, c.scale, workspace=ws, **arms)

    for i in range(max(3, args.warmup)):
        step(i)
    torch.cuda.synchronize()
    ms = timed(step, max(5, args.steps), st)
    assert g.attn_get_device_error() == g.OK
    return {"workload": f"paged decode bf16 as above with window {window}, sink logits, ALiBi slopes and "
                        "softcap 30 (every arm on)", "gbs": nbytes / (ms * 1e-3) / 1e9, "ms": ms, "bytes": nbytes,
            "roofline": {"bound": "hbm", "achieved": nbytes / (ms * 1e-3) / 1e9}}


def run_paged_e2e(args, g, c, tables, lens_in, lens_out, out, ws, step_bytes, world):
    """The same step through the public API from pinned host buffers: q, k_new and
    v_new copied in, the attention output copied back, every step. The copies run
    on a stream of their own, pipelined with the compute as a serving loop would:
    step i + 1's inputs come in and step i's output goes out while step i + 1 /
    step i compute (two device buffers each, ordered by events); the timed region
    holds every step's copies in and out."""
    B, H, d = c.q.shape
    Hkv = c.k_new.shape[1]
    gi = W.generator(99)
    hq = [W.randn((B, H, d), gi, torch.bfloat16).pin_memory() for _ in range(2)]
    hk = [W.randn((B, Hkv, d), gi, torch.bfloat16).pin_memory() for _ in range(2)]
    hv = [W.randn((B, Hkv, d), gi, torch.bfloat16).pin_memory() for _ in range(2)]
    hout = [torch.empty(B, H, d, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    dq = [torch.empty(B, H, d, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    dk = [torch.empty(B, Hkv, d, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    dv = [torch.empty(B, Hkv, d, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    outs = [out, torch.empty_like(out)]
    st = torch.cuda.current_stream()
    cs = torch.cuda.Stream()
    in_ready = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]       # step's compute finished with its buffers
    out_read = [torch.cuda.Event() for _ in range(2)]   # its output is on the host
    used = [False, False]

    def inputs(i):  # step i's inputs into buffer i % 2, once the step before that used it is done
        b = i % 2
        with torch.cuda.stream(cs):
            if used[b]:
                cs.wait_event(done[b])
            dq[b].copy_(hq[b], non_blocking=True)
            dk[b].copy_(hk[b], non_blocking=True)
            dv[b].copy_(hv[b], non_blocking=True)
            in_ready[b].record(cs)

    def steps(first, count):
        inputs(first)
        for i in range(first, first + count):
            b = i % 2
            st.wait_event(in_ready[b])
            if used[b]:
                st.wait_event(out_read[b])  # the output buffer's last copy out is done
            g.kv_append_paged(dq[b], dk[b], dv[b], c.k_pool, c.v_pool, tables, lens_in, lens_out, c.theta)
            g.attn_decode_paged(dq[b], c.k_pool, c.v_pool, tables, lens_out, outs[b], c.scale, workspace=ws)
            done[b].record(st)
            used[b] = True
            if i + 1 < first + count:
                inputs(i + 1)
            with torch.cuda.stream(cs):
                cs.wait_event(done[b])
                hout[b].copy_(outs[b], non_blocking=True)
                out_read[b].record(cs)
        st.wait_stream(cs)  # the last output is on the host

    steps(0, args.warmup)
    torch.cuda.synchronize()
    barrier(world)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(st)
    cs.wait_stream(st)  # no copy of the timed steps starts before t0
    steps(args.warmup, args.steps)
    t1.record(st)
    torch.cuda.synchronize()
    ms = reduce_over_ranks(t0.elapsed_time(t1) / args.steps, world, "max")
    total = reduce_over_ranks(step_bytes, world, "sum")
    return {"value": total / (ms * 1e-3) / 1e9, "unit": "GB/s", "ms_per_step": ms,
            "h2d_bytes_per_step": (dq[0].numel() + dk[0].numel() + dv[0].numel()) * 2,
            "d2h_bytes_per_step": out.numel() * 2,
            "copies": "own stream, pipelined with the compute (step i+1 in, step i out)"}


def gather_paged_sample(c, q, kn, vn, nseq):
    """Host copies of the pristine history of a few sequences (the shortest, the
    longest, then seeded others), each as a mini-pool of its own blocks in table
    order, with the step's new q/k/v rows."""
    lens = c.seq_lens.cpu()
    order = torch.argsort(lens)
    pick = [int(order[0]), int(order[-1])]
    for b in torch.randperm(len(lens), generator=W.generator(5)).tolist():
        if len(pick) >= nseq:
            break
        if b not in pick:
            pick.append(b)
    bs, seqs = c.block_size, []
    for b in pick:
        n = int(lens[b]) + 1
        nblk = (n + bs - 1) // bs
        blocks = c.tables[b, :nblk].long()
        seqs.append(dict(b=b, q=W.to_oracle(q[b:b + 1]), kn=W.to_oracle(kn[b:b + 1]), vn=W.to_oracle(vn[b:b + 1]),
                         kp=W.to_oracle(c.k_pool[blocks]), vp=W.to_oracle(c.v_pool[blocks]),
                         table=np.arange(nblk, dtype=np.int32)[None], len=int(lens[b])))
    return seqs


def oracle_paged_sample(sample, theta, scale, max_seconds, min_seconds=10.0):
    """Run the oracle's append + decode over the sampled sequences, pass after
    pass until at least min_seconds of oracle time is spent (stopping early once
    max_seconds is); returns (algorithmic bytes, seconds, sequences run, passes).
    The first pass leaves each sequence's oracle output in s["want"]."""
    from oracle import core
    done, t_total, n, passes = 0, 0.0, 0, 0
    while passes == 0 or t_total < min_seconds:
        passes += 1
        for s in sample:
            t = time.perf_counter()
            q2, kp2, vp2, l2 = core.kv_append_paged(s["q"], s["kn"], s["vn"], s["kp"], s["vp"], s["table"],
                                                    [s["len"]], theta)
            want = core.decode_paged(q2, kp2, vp2, s["table"], l2, scale)
            t_total += time.perf_counter() - t
            if passes == 1:
                s["want"] = want
            H, (Hkv, d) = s["q"].shape[1], s["kn"].shape[1:]
            dec, app = paged_bytes(np.array([s["len"] + 1]), 1, H, Hkv, d, d, s["kp"].shape[2])
            done += dec + app
            n += 1
            if t_total > max_seconds:
                return done, t_total, n, passes
    return done, t_total, n, passes


# ---------------------------------------------------------------------------
# secondary workloads

def run_prefill(args, peaks, peak_kind):
    import causal_gqa_attention_row_gb300 as g
    g.load()
    dev = torch.device("cuda")
    B, S, H, Hkv, d = 1, 2048, 14, 2, 64
    c = W.make_prefill(B=B, S=S, H=H, Hkv=Hkv, dk=d, dv=d, seed=1, device=dev)
    pos = torch.arange(S, dtype=torch.int32, device=dev)[None].repeat(B, 1)
    n = max(args.steps, 20)
    # fresh q, k per step (the RoPE is in place)
    qs = [c.q.clone() for _ in range(n + 3)]
    ks = [c.k.clone() for _ in range(n + 3)]
    out = torch.empty(B, S, H, d, dtype=torch.bfloat16, device=dev)
    flops = 2.0 * H * (d + d) * S * (S + 1) / 2  # unmasked (query, key) pairs only
    st = torch.cuda.current_stream()

    def step(i):  # RoPE of q and k (one launch), then the prefill
        g.attn_rope_interleaved_qk(qs[i], ks[i], pos, 1e6, k_heads_outer=True)
        g.attn_prefill_causal(qs[i], ks[i], c.v, out, c.scale)

    for i in range(3):
        step(i)
    torch.cuda.synchronize()
    # The kernel runs for microseconds, less than the host needs to issue a
    # step, so the GPU is first held busy (a device-side sleep) while the host
    # queues every timed launch; the events then see GPU time, not host gaps.
    queue_ahead(n)
    step_ms = timed(lambda k: step(3 + k), n, st, sync_first=False)
    assert g.attn_get_device_error() == g.OK
    # The kernel's average launch duration: CUDA events around a run of
    # back-to-back launches on the step's (already rotated) inputs, queued ahead
    # of the GPU (one event pair per microsecond-long launch would be dominated by
    # the events' 0.5 us resolution and the launch gap in front of each).
    n_kern = 4 * n
    torch.cuda.synchronize()
    queue_ahead(n_kern, us_per_group=40.0)
    ms = timed(lambda k: g.attn_prefill_causal(qs[3], ks[3], c.v, out, c.scale), n_kern, st, sync_first=False)
    assert g.attn_get_device_error() == g.OK
    tflops = flops / (ms * 1e-3) / 1e12
    peak = peaks["bf16_tflops"]
    return {"workload": W.WORKLOADS["prefill"], "tflops": tflops, "kernel_ms": ms, "step_ms": step_ms,
            "step_tflops": flops / (step_ms * 1e-3) / 1e12, "flops": flops,
            "roofline": {"bound": "tensor", "achieved": tflops, "peak": peak, "unit": "TFLOP/s", "frac": tflops / peak,
                         "kernel": "prefill_tc_kernel", "peak_kind": f"bf16 dense burst, {peak_kind}"}}


def run_prefill_arms(args, peaks, peak_kind, window=512):
    """The headline prefill shape with every arm on (a 512-row sliding window,
    sink logits, ALiBi slopes, softcap 30) on the tensor-core kernel's arms
    instantiation. Algorithmic FLOPs: the (query, key) pairs inside each row's
    window only."""
    import causal_gqa_attention_row_gb300 as g
    g.load()
    dev = torch.device("cuda")
    B, S, H, Hkv, d = 1, 2048, 14, 2, 64
    c = W.make_prefill(B=B, S=S, H=H, Hkv=Hkv, dk=d, dv=d, seed=1, device=dev)
    out = torch.empty(B, S, H, d, dtype=torch.bfloat16, device=dev)
    sinks = W.randn((H,), W.generator(123, dev), torch.float32, dev)
    slopes = torch.tensor([2.0 ** (-8.0 * (h + 1) / H) for h in range(H)], dtype=torch.float32, device=dev)
    arms = dict(window=window, softcap=30.0, sinks=sinks, alibi_slopes=slopes)
    pairs = sum(min(i + 1, window) for i in range(S))
    flops = 2.0 * H * (d + d) * pairs
    st = torch.cuda.current_stream()
    call = lambda k: g.attn_prefill_causal(c.q, c.k, c.v, out, c.scale, **arms)
    for i in range(3):
        call(i)
    torch.cuda.synchronize()
    n = 4 * max(args.steps, 20)
    queue_ahead(n, us_per_group=40.0)
    ms = timed(call, n, st, sync_first=False)
    assert g.attn_get_device_error() == g.OK
    tflops = flops / (ms * 1e-3) / 1e12
    peak = peaks["bf16_tflops"]
    return {"workload": W.WORKLOADS["prefill"] + f", window {window}, sink logits, ALiBi slopes, softcap 30",
            "tflops": tflops, "kernel_ms": ms, "flops": flops,
            "roofline": {"bound": "tensor", "achieved": tflops, "peak": peak, "unit": "TFLOP/s", "frac": tflops / peak,
                         "kernel": "prefill_tc_kernel<64, 64, arms>", "peak_kind": f"bf16 dense burst, {peak_kind}"}}


def run_prefill_d128(args, peaks, peak_kind, H=32, Hkv=8, dk=128, dv=128, key="prefill_d128"):
    """Causal prefill at d = 128 (the decode configs' head shape), or at the MLA
    widths, on the tcgen05 kernel: the kernel's event average over back-to-back
    launches."""
    import causal_gqa_attention_row_gb300 as g
    g.load()
    dev = torch.device("cuda")
    S = 2048
    c = W.make_prefill(B=1, S=S, H=H, Hkv=Hkv, dk=dk, dv=dv, seed=7, device=dev)
    out = torch.empty(1, S, H, dv, dtype=torch.bfloat16, device=dev)
    flops = 2.0 * H * (dk + dv) * S * (S + 1) / 2
    st = torch.cuda.current_stream()
    call = lambda k: g.attn_prefill_causal(c.q, c.k, c.v, out, c.scale)
    for i in range(3):
        call(i)
    torch.cuda.synchronize()
    n = 4 * max(args.steps, 20)
    queue_ahead(n, us_per_group=60.0)
    ms = timed(call, n, st, sync_first=False)
    assert g.attn_get_device_error() == g.OK
    tflops = flops / (ms * 1e-3) / 1e12
    peak = peaks["bf16_tflops"]
    return {"workload": W.WORKLOADS[key], "tflops": tflops, "kernel_ms": ms, "flops": flops,
            "roofline": {"bound": "tensor", "achieved": tflops, "peak": peak, "unit": "TFLOP/s", "frac": tflops / peak,
                         "kernel": f"prefill_tc_kernel<{dk}, {dv}>", "peak_kind": f"bf16 dense burst, {peak_kind}"}}


def run_prefill_mla(args, peaks, peak_kind):
    return run_prefill_d128(args, peaks, peak_kind, H=32, Hkv=32, dk=192, dv=128, key="prefill_mla")


def run_prefill_paged(args, peaks, peak_kind, H=14, Hkv=2, d=64, key="prefill_paged"):
    """Chunked prefill against the paged pool on the tcgen05 kernel (each key
    tile gathered from the pool block by block)."""
    import causal_gqa_attention_row_gb300 as g
    g.load()
    dev = torch.device("cuda")
    offs, S = (0, 2048, 4096, 6144), 2048
    q, kp, vp, tables, off, scale = W.make_prefill_paged(offsets=offs, S=S, H=H, Hkv=Hkv, d=d, device=dev)
    out = torch.empty_like(q)
    # unmasked (query, key) pairs: row i of sequence b sees off_b + i + 1 keys
    flops = sum(2.0 * H * (d + d) * (S * o + S * (S + 1) / 2) for o in offs)
    st = torch.cuda.current_stream()
    call = lambda k: g.attn_prefill_paged(q, kp, vp, tables, out, scale, position_offset=off)
    for i in range(3):
        call(i)
    torch.cuda.synchronize()
    n = 4 * max(args.steps, 20)
    queue_ahead(n, us_per_group=60.0)
    ms = timed(call, n, st, sync_first=False)
    assert g.attn_get_device_error() == g.OK
    tflops = flops / (ms * 1e-3) / 1e12
    peak = peaks["bf16_tflops"]
    return {"workload": W.WORKLOADS[key], "tflops": tflops, "kernel_ms": ms, "flops": flops,
            "roofline": {"bound": "tensor", "achieved": tflops, "peak": peak, "unit": "TFLOP/s", "frac": tflops / peak,
                         "kernel": f"prefill_tc_kernel<{d}> (paged)", "peak_kind": f"bf16 dense burst, {peak_kind}"}}


def run_prefill_paged_d128(args, peaks, peak_kind):
    return run_prefill_paged(args, peaks, peak_kind, H=32, Hkv=8, d=128, key="prefill_paged_d128")


def run_contig(args, peaks, peak_kind):
    import causal_gqa_attention_row_gb300 as g
    dev = torch.device("cuda")
    B, H, Hkv, d, L = 64, 32, 8, 128, 8192
    c = W.make_contig(B=B, H=H, Hkv=Hkv, dk=d, dv=d, max_len=L, seed=2, device=dev)
    # two cache copies alternate so that consecutive steps do not hit in L2
    k2, v2 = c.k.clone(), c.v.clone()
    caches = [(c.k, c.v), (k2, v2)]
    out = torch.empty(B, H, d, dtype=torch.bfloat16, device=dev)
    ws = g.decode_workspace(B, H, d, L, device=dev)
    lens = c.seq_lens.cpu().numpy().astype(np.int64)
    nbytes = int(lens.sum()) * Hkv * 2 * d * 2 + B * H * 2 * d * 2
    st = torch.cuda.current_stream()

    def step(i):
        k, v = caches[i % 2]
        g.attn_decode_contig(c.q, k, v, c.seq_lens, out, c.scale, workspace=ws)

    for i in range(3):
        step(i)
    ms = timed(step, max(args.steps, 20), st)
    assert g.attn_get_device_error() == g.OK
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"workload": W.WORKLOADS["contig"], "gbs": gbs, "ms": ms, "bytes": nbytes,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": gbs / peaks["hbm_gbs"], "frac_of_8tbs": gbs / NOMINAL_HBM_GBS,
                         "peak_kind": peak_kind}}


def run_mla(args, peaks, peak_kind):
    import causal_gqa_attention_row_gb300 as g
    dev = torch.device("cuda")
    B, H, L = args.mla_seqs, 128, 4096
    c = W.make_mla(B=B, H=H, cache_len=L, seed=4, device=dev)
    pos = torch.arange(L, dtype=torch.int32, device=dev)[None].repeat(B, 1)
    # setup (untimed): RoPE theta 1e4 on the shared k_rot (once per position) and
    # on every head's q rot slice at position L - 1
    g.attn_rope_interleaved(c.k_rot.view(B, L, 1, 64), pos, 1e4)
    g.attn_rope_interleaved(c.q.view(B, 1, H, 192), pos[:, -1:].contiguous(), 1e4, rot_offset=128, rot_dim=64)
    out = torch.empty(B, H, 128, dtype=torch.bfloat16, device=dev)
    ws = g.decode_workspace(B, H, 128, L, device=dev)
    nbytes = B * L * (H * (128 + 128) + 64) * 2 + B * H * (192 + 128) * 2
    st = torch.cuda.current_stream()
    step = lambda i: g.attn_decode_contig(c.q, c.k, c.v, c.seq_lens, out, c.scale, workspace=ws,
                                          k_rot_shared=c.k_rot)
    for i in range(3):
        step(i)
    ms = timed(step, max(args.steps, 10), st)
    assert g.attn_get_device_error() == g.OK
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"workload": W.WORKLOADS["mla"] if B == 32 else W.WORKLOADS["mla"].replace("32 seqs", f"{B} seqs (reduced)"),
            "gbs": gbs, "ms": ms, "bytes": nbytes,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": gbs / peaks["hbm_gbs"], "frac_of_8tbs": gbs / NOMINAL_HBM_GBS,
                         "peak_kind": peak_kind}}


def run_mla_absorbed(args, peaks, peak_kind):
    """Absorbed (latent) MLA decode at the MLA-shaped config's model shape: the
    attention over the latent rows (mla_absorbed_tc_kernel + split combine) timed
    alone, and the whole absorbed step (absorb, attention, unabsorb). Two copies
    of the latent cache (2 x 151 MB) alternate, so no launch finds its rows in L2."""
    import causal_gqa_attention_row_gb300 as g
    g.load()
    dev = torch.device("cuda")
    B, H, L, D_C, D_R = 32, 128, 4096, 512, 64
    c = W.make_mla_absorbed(B=B, H=H, max_len=L, seed=9, device=dev)
    pos = torch.arange(L, dtype=torch.int32, device=dev)[None].repeat(B, 1).contiguous()
    # setup (untimed): RoPE theta 1e4 on each latent row's rot slice at its own
    # position, and on every head's q rot slice at position L - 1
    g.attn_rope_interleaved(c.latent.view(B, L, 1, D_C + D_R), pos, 1e4, rot_offset=D_C, rot_dim=D_R)
    g.attn_rope_interleaved(c.q.view(B, 1, H, 192), pos[:, -1:].contiguous(), 1e4, rot_offset=128, rot_dim=64)
    latents = [c.latent, c.latent.clone()]
    q_abs = torch.empty(B, H, D_C + D_R, dtype=torch.bfloat16, device=dev)
    out_lat = torch.empty(B, H, D_C, dtype=torch.bfloat16, device=dev)
    out = torch.empty(B, H, 128, dtype=torch.bfloat16, device=dev)
    ws = g.mla_absorbed_workspace(B, H, D_C, L, device=dev)
    k_b, v_b = c.k_b, c.v_b
    g.mla_absorb_q(c.q, k_b, q_abs)
    flops = 2.0 * B * H * L * (D_C + D_R + D_C)
    nbytes = B * L * (D_C + D_R) * 2 + B * H * (D_C + D_R) * 2 + B * H * D_C * 2
    st = torch.cuda.current_stream()
    attend = lambda k: g.attn_decode_mla_absorbed(q_abs, latents[k % 2], c.lens, out_lat, c.scale, workspace=ws)

    def step(k):
        g.mla_absorb_q(c.q, k_b, q_abs)
        attend(k)
        g.mla_unabsorb_out(out_lat, v_b, out)

    for i in range(4):
        step(i)
    torch.cuda.synchronize()
    n = 2 * max(args.steps, 20)
    queue_ahead(n, us_per_group=60.0)
    ms = timed(attend, n, st, sync_first=False)
    queue_ahead(n, us_per_group=80.0)
    ms_step = timed(step, n, st, sync_first=False)
    assert g.attn_get_device_error() == g.OK
    # the same rows in a paged pool of 64-row blocks (a seeded permutation of the
    # blocks; two pools alternate), through attn_decode_mla_absorbed_paged
    bs = 64
    mbps = L // bs
    gl = W.generator(10)
    pools, tables = [], []
    for lat in latents:
        perm = torch.randperm(B * mbps, generator=gl).to(torch.int32)
        tab = perm.view(B, mbps).to(dev)
        pool = torch.empty(B * mbps, bs, D_C + D_R, dtype=torch.bfloat16, device=dev)
        pool[tab.view(-1).long()] = lat.view(B * mbps, bs, D_C + D_R)
        pools.append(pool)
        tables.append(tab)
    del pool
    attend_paged = lambda k: g.attn_decode_mla_absorbed_paged(q_abs, pools[k % 2], tables[k % 2], c.lens, out_lat,
                                                              c.scale, workspace=ws)
    for i in range(3):
        attend_paged(i)
    torch.cuda.synchronize()
    queue_ahead(n, us_per_group=60.0)
    ms_paged = timed(attend_paged, n, st, sync_first=False)
    assert g.attn_get_device_error() == g.OK
    gbs = nbytes / (ms * 1e-3) / 1e9
    tflops = flops / (ms * 1e-3) / 1e12
    hbm, bf = peaks["hbm_gbs"], peaks["bf16_tflops"]
    return {"workload": W.WORKLOADS["mla_absorbed"], "ms": ms, "gbs": gbs, "tflops": tflops, "bytes": nbytes,
            "flops": flops, "step_ms": ms_step, "paged_bs64_ms": ms_paged,
            "paged_bs64_gbs": nbytes / (ms_paged * 1e-3) / 1e9,
            "step": "mla_absorb_q + attn_decode_mla_absorbed + mla_unabsorb_out",
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm,
                         "tensor_tflops": tflops, "tensor_frac": tflops / bf,
                         "note": f"{flops / nbytes:.0f} flop per byte, below the ridge of {bf * 1e3 / hbm:.0f}: the "
                                 "latent stream bounds it",
                         "kernel": "attn_decode_mla_absorbed (mla_absorbed_tc_kernel + split_combine_kernel)",
                         "peak_kind": f"{peak_kind} copy bandwidth; bf16 dense burst for tensor_frac"}}


# ---------------------------------------------------------------------------
# reference arm: the oracle on the host cores

def reference_arm(args, rank, world):
    if rank != 0:
        return
    from oracle import core
    # A host-side replica of the paged workload holding only the sampled
    # sequences; their history lengths are drawn exactly as in the full workload.
    lens_all = torch.randint(1, 32769, (256,), generator=W.generator(3 + 1000), dtype=torch.int32)
    pick = lens_all[:args.ref_seqs].tolist()
    cs = W.make_paged(B=len(pick), H=32, Hkv=8, dk=128, dv=128, block_size=16,
                      num_blocks=sum((n + 16) // 16 for n in pick) + 1, lens=pick, seed=3, device="cpu")
    sample = []
    for b, n in enumerate(pick):
        nblk = (n + 1 + 15) // 16
        blocks = cs.tables[b, :nblk].long()
        sample.append(dict(q=W.to_oracle(cs.q[b:b + 1]), kn=W.to_oracle(cs.k_new[b:b + 1]),
                           vn=W.to_oracle(cs.v_new[b:b + 1]), kp=W.to_oracle(cs.k_pool[blocks]),
                           vp=W.to_oracle(cs.v_pool[blocks]), table=np.arange(nblk, dtype=np.int32)[None], len=n))
    for _ in range(args.warmup):
        oracle_paged_sample(sample[:1], cs.theta, cs.scale, 1e9, min_seconds=0.0)
    times, nbytes = [], 0
    for _ in range(args.steps):
        nbytes, t, _, _ = oracle_paged_sample(sample, cs.theta, cs.scale, 1e9, min_seconds=0.0)
        times.append(t)
    ms = statistics.mean(times) * 1e3
    value = nbytes / (ms * 1e-3) / 1e9
    desc = f"append + decode of {len(pick)} sequences of the paged workload ({sum(pick)} history rows) per step"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": W.WORKLOADS["paged"], "sample": desc},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": core.threads(), "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# DRAM bytes (read + write) of the paged decode's attention kernel per algorithmic
# byte, from an ncu capture of a 32-sequence case of the paged workload:
# 2,085,826,048 B moved for 2,080,718,884 B of K/V rows, q, out and table entries.
DECODE_TRAFFIC_PER_ALG_BYTE = 2085826048 / 2080718884

# Kernels one paged step launches: append_kernel, then the decode's plan_units_kernel,
# attn_rows_kernel and split_combine_kernel (the workload's caches are long enough to split).
LAUNCHES_PER_PAGED_STEP = 4


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--seqs", type=int, default=256, help="sequences of the paged workload")
    ap.add_argument("--pool-blocks", type=int, default=600_000, help="blocks in the paged pool")
    ap.add_argument("--cpu-seqs", type=int, default=96, help="sequences in the CPU-baseline sample")
    ap.add_argument("--cpu-seconds", type=float, default=30.0, help="cap on CPU-baseline oracle time")
    ap.add_argument("--ref-seqs", type=int, default=4, help="sequences per reference-arm step")
    ap.add_argument("--mla-seqs", type=int, default=32,
                    help="sequences of the MLA-shaped decode (32 is the workload; fewer only for profiling captures)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-secondary", action="store_true", help="skip prefill, contig and mla")
    ap.add_argument("--only", choices=["paged", "prefill", "prefill_arms", "prefill_paged", "prefill_d128",
                                       "prefill_paged_d128", "prefill_mla", "contig", "mla", "mla_absorbed"],
                    default=None)
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    rank, world = dist_setup()
    if args.impl == "reference":
        reference_arm(args, rank, world)
        return
    peaks, peak_kind = measured_peaks()
    only = {"prefill": run_prefill, "prefill_arms": run_prefill_arms, "prefill_paged": run_prefill_paged,
            "prefill_d128": run_prefill_d128,
            "prefill_paged_d128": run_prefill_paged_d128, "prefill_mla": run_prefill_mla, "contig": run_contig,
            "mla": run_mla, "mla_absorbed": run_mla_absorbed}
    if args.only in only:
        r = only[args.only](args, peaks, peak_kind)
        if rank == 0:
            print(json.dumps(r), flush=True)
        return
    res = run_paged(args, rank, world)
    secondary = {}
    if not args.no_secondary and args.only is None:
        secondary = {"prefill": run_prefill(args, peaks, peak_kind),
                     "prefill_arms": run_prefill_arms(args, peaks, peak_kind),
                     "prefill_paged": run_prefill_paged(args, peaks, peak_kind),
                     "prefill_d128": run_prefill_d128(args, peaks, peak_kind),
                     "prefill_paged_d128": run_prefill_paged_d128(args, peaks, peak_kind),
                     "prefill_mla": run_prefill_mla(args, peaks, peak_kind),
                     "contig": run_contig(args, peaks, peak_kind), "mla": run_mla(args, peaks, peak_kind),
                     "mla_absorbed": run_mla_absorbed(args, peaks, peak_kind)}
    if res.get("arms"):
        arms = res["arms"]
        arms["roofline"].update({"peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": arms["gbs"] / peaks["hbm_gbs"],
                                 "peak_kind": peak_kind})
        secondary["paged_arms"] = arms
    if rank != 0:
        return
    cpu = None
    if res["sample"]:
        from oracle import core
        nbytes, secs, n, passes = oracle_paged_sample(res["sample"], 1e6, 1.0 / math.sqrt(128), args.cpu_seconds)
        cpu = {"value": nbytes / secs / 1e9, "unit": "GB/s", "cores": core.threads(), "kind": "oracle",
               "sample": f"append + decode of {len(res['sample'])} of the {args.seqs} sequences (the shortest, the "
                         f"longest, seeded others) of the paged workload, {passes} pass(es), {n} sequence runs; "
                         f"{secs:.1f} s of oracle time"}
        # the oracle's outputs against the GPU's for the same step (first warm-up
        # step: same history, same new rows), element by element
        compared = [s for s in res["sample"] if "want" in s and "gpu_out" in s]
        err = max(float(np.abs(s["gpu_out"] - s["want"]).max()) for s in compared)
        cpu["parity"] = {"sequences": len(compared), "max_abs_err": err, "tol": 2e-2}
        if not err <= 2e-2:
            raise SystemExit(f"GPU output disagrees with the oracle on the CPU-baseline sample: max abs err {err}")
    hbm = peaks["hbm_gbs"]
    line = {
        "metric": METRIC, "value": res["value"], "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": res["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": W.WORKLOADS["paged"] if args.seqs == 256 and args.pool_blocks == 600_000 else
                   f"paged decode bf16, {args.seqs} seqs, {args.pool_blocks}-block pool (reduced)",
                   "global_batch": args.seqs * world, "history_rows": res["rows"],
                   "step": "kv_append_paged + attn_decode_paged",
                   "l2": "no flush: the K/V working set per step (~17 GB) is larger than L2",
                   "parallelism": f"{world} independent replicas (one per GPU)"},
        "roofline": {"bound": "hbm", "achieved": res["achieved_decode_gbs"], "peak": hbm, "unit": "GB/s",
                     "frac": res["achieved_decode_gbs"] / hbm,
                     "traffic": round(DECODE_TRAFFIC_PER_ALG_BYTE * res["decode_bytes"]) if args.seqs == 256 else None,
                     "traffic_source": "dram__bytes_read.sum + dram__bytes_write.sum of attn_rows_kernel on a 32-sequence "
                                       "case of this workload (2.0858 GB for 2.0807 GB of algorithmic bytes), scaled by the "
                                       "K/V rows one launch processes",
                     "kernel": "attn_decode_paged (plan_units_kernel + attn_rows_kernel + split_combine_kernel)",
                     "algorithmic_bytes_per_launch": res["decode_bytes"], "decode_ms": res["decode_ms"],
                     "peak_kind": f"{peak_kind} copy bandwidth",
                     "frac_of_8tbs": res["achieved_decode_gbs"] / NOMINAL_HBM_GBS},
        "cpu_baseline": cpu, "e2e": res.get("e2e"), "gpu_launches": LAUNCHES_PER_PAGED_STEP * args.steps, "clocks": res["clocks"],
        **secondary,
    }
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
