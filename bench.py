"""Benchmark: paged GQA decode HBM GB/s (headline) and causal prefill TFLOP/s.

One step of the paged workload = kv_append_paged (one new row per sequence,
interleaved RoPE on q and k) + attn_decode_paged over 256 sequences whose
histories are U[1, 32768] rows in a 600,000-block shared pool (the K/V working
set, ~17 GB, is far larger than L2, so no flush is needed between steps).

`--impl reference` times the fp64 CPU oracle on the host cores on a bounded
sample of the same workload. Under torchrun each rank runs its own replica of
the workload (its own seed) on its own GPU: the batch shards with no exchange,
so scaling is weak.
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


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except OSError:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


# ---------------------------------------------------------------------------
# distributed plumbing (rank-local replicas; only timings cross ranks)

def dist_setup(n_gpus):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    if torch.cuda.is_available():
        torch.cuda.set_device(local)
    return rank, world


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x, world):
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ---------------------------------------------------------------------------
# clocks during the timed region

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.out = self.proc.communicate(timeout=5)[0]
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        rows = []
        for line in (self.out or "").strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) == 7:
                rows.append(parts)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        sm = [float(r[0]) for r in rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[3 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------------------
# the paged decode workload

def paged_bytes(lens_after, B, H, Hkv, dk, dv, bs, es=2):
    """Algorithmic bytes of one append + decode step: every visible K/V row read
    once, q read, out written, the block-table entries the decode reads, and the
    append's own reads and writes (q in/out, new k/v in, pool rows out)."""
    rows = int(lens_after.sum())
    kv = rows * Hkv * (dk + dv) * es
    tables = int(((lens_after + bs - 1) // bs).sum()) * 4
    qo = B * H * (dk + dv) * es
    append = B * H * dk * es * 2 + 2 * B * Hkv * (dk + dv) * es
    return kv + tables + qo, append


def run_paged(args, rank, world, peaks, peak_kind):
    import causal_gqa_attention_row_gb300 as g
    g.load()
    dev = torch.device("cuda")
    free, total = torch.cuda.mem_get_info()
    B, H, Hkv, d, bs, nb = 256, 32, 8, 128, 16, 600_000
    need = 2 * nb * Hkv * bs * d * 2
    if free < need + (4 << 30):
        raise SystemExit(f"not enough free device memory: {free / 2**30:.1f} GiB free, "
                         f"{(need + (4 << 30)) / 2**30:.1f} GiB needed")
    c = W.make_paged(B=B, H=H, Hkv=Hkv, dk=d, dv=d, block_size=bs, num_blocks=nb, seed=3 + 1000 * rank,
                     device="cpu" if False else dev)
    n_sets = args.warmup + args.steps
    gi = W.generator(77 + rank, dev)
    qs = [W.randn((B, H, d), gi, torch.bfloat16, dev) for _ in range(n_sets)]
    kns = [W.randn((B, Hkv, d), gi, torch.bfloat16, dev) for _ in range(n_sets)]
    vns = [W.randn((B, Hkv, d), gi, torch.bfloat16, dev) for _ in range(n_sets)]
    lens_in = c.seq_lens.to(dev)
    lens_out = torch.empty_like(lens_in)
    tables = c.tables.to(dev)
    mbps = tables.shape[1]
    out = torch.empty(B, H, d, dtype=torch.bfloat16, device=dev)
    ws = g.decode_workspace(B, H, d, mbps * bs, device=dev)
    st = torch.cuda.current_stream()

    lens_after = c.seq_lens.cpu().numpy().astype(np.int64) + 1
    dec_bytes, app_bytes = paged_bytes(lens_after, B, H, Hkv, d, d, bs)

    # CPU-baseline sample gathered before anything is timed (pristine pool)
    sample = None
    if rank == 0 and not args.no_cpu_baseline:
        sample = gather_paged_sample(c, qs[0], kns[0], vns[0], args.cpu_seqs)

    def step(i, ev=None):
        g.kv_append_paged(qs[i], kns[i], vns[i], c.k_pool, c.v_pool, tables, lens_in, lens_out, c.theta)
        if ev:
            ev[0].record(st)
        g.attn_decode_paged(qs[i], c.k_pool, c.v_pool, tables, lens_out, out, c.scale, workspace=ws)
        if ev:
            ev[1].record(st)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    assert g.attn_get_device_error() == g.OK
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(torch.cuda.current_device()) as clk:
        barrier(world)
        torch.cuda.synchronize()
        t0.record(st)
        for k in range(args.steps):
            step(args.warmup + k, evs[k])
        t1.record(st)
        torch.cuda.synchronize()
        barrier(world)
    ms = t0.elapsed_time(t1) / args.steps
    dec_ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
    assert g.attn_get_device_error() == g.OK
    ms_max = max_over_ranks(ms, world)
    total_bytes = sum_over_ranks(float(dec_bytes + app_bytes), world)
    value = total_bytes / (ms_max * 1e-3) / 1e9
    achieved = dec_bytes / (dec_ms * 1e-3) / 1e9

    # end to end through the public API with host buffers
    e2e = run_paged_e2e(args, g, c, tables, lens_in, lens_out, out, ws, dec_bytes + app_bytes, world)

    res = {
        "value": value, "ms_per_step": ms_max, "decode_ms": dec_ms, "achieved_decode_gbs": achieved,
        "bytes_per_step": dec_bytes + app_bytes, "decode_bytes": dec_bytes, "clocks": clk.summary(), "e2e": e2e,
        "sample": sample,
    }
    return res


def run_paged_e2e(args, g, c, tables, lens_in, lens_out, out, ws, step_bytes, world):
    B, H, d = c.q.shape
    Hkv = c.k_new.shape[1]
    gi = W.generator(99)
    hq = [W.randn((B, H, d), gi, torch.bfloat16).pin_memory() for _ in range(2)]
    hk = [W.randn((B, Hkv, d), gi, torch.bfloat16).pin_memory() for _ in range(2)]
    hv = [W.randn((B, Hkv, d), gi, torch.bfloat16).pin_memory() for _ in range(2)]
    hout = torch.empty(B, H, d, dtype=torch.bfloat16).pin_memory()
    dq = torch.empty(B, H, d, dtype=torch.bfloat16, device="cuda")
    dk = torch.empty(B, Hkv, d, dtype=torch.bfloat16, device="cuda")
    dv = torch.empty(B, Hkv, d, dtype=torch.bfloat16, device="cuda")
    st = torch.cuda.current_stream()

    def step(i):
        dq.copy_(hq[i % 2], non_blocking=True)
        dk.copy_(hk[i % 2], non_blocking=True)
        dv.copy_(hv[i % 2], non_blocking=True)
        g.kv_append_paged(dq, dk, dv, c.k_pool, c.v_pool, tables, lens_in, lens_out, c.theta)
        g.attn_decode_paged(dq, c.k_pool, c.v_pool, tables, lens_out, out, c.scale, workspace=ws)
        hout.copy_(out, non_blocking=True)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    t0.record(st)
    for i in range(args.steps):
        step(i)
    t1.record(st)
    torch.cuda.synchronize()
    ms = max_over_ranks(t0.elapsed_time(t1) / args.steps, world)
    total = sum_over_ranks(float(step_bytes), world)
    h2d = (dq.numel() + dk.numel() + dv.numel()) * 2
    return {"value": total / (ms * 1e-3) / 1e9, "unit": "GB/s", "ms_per_step": ms, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": out.numel() * 2}


def gather_paged_sample(c, q, kn, vn, nseq):
    """Copy the pristine history of a few sequences (shortest, longest, and
    seeded others) to the host, as mini-pools in table order."""
    lens = c.seq_lens.cpu()
    order = torch.argsort(lens)
    pick = [int(order[0]), int(order[-1])]
    rest = torch.randperm(len(lens), generator=W.generator(5))
    for b in rest.tolist():
        if len(pick) >= nseq:
            break
        if b not in pick:
            pick.append(b)
    bs = c.block_size
    seqs = []
    for b in pick:
        n = int(lens[b]) + 1
        nblk = (n + bs - 1) // bs
        blocks = c.tables[b, :nblk].long()
        seqs.append(dict(
            q=W.to_oracle(q[b:b + 1]), kn=W.to_oracle(kn[b:b + 1]), vn=W.to_oracle(vn[b:b + 1]),
            kp=W.to_oracle(c.k_pool[blocks]), vp=W.to_oracle(c.v_pool[blocks]),
            table=np.arange(nblk, dtype=np.int32)[None], len=int(lens[b])))
    return seqs


def oracle_paged_sample(sample, theta, scale, max_seconds):
    """Time the oracle (append + decode) over the sample; returns (bytes, seconds, n)."""
    from oracle import core
    done_bytes, t_total, n = 0, 0.0, 0
    for s in sample:
        t = time.perf_counter()
        q2, kp2, vp2, l2 = core.kv_append_paged(s["q"], s["kn"], s["vn"], s["kp"], s["vp"], s["table"],
                                                [s["len"]], theta)
        core.decode_paged(q2, kp2, vp2, s["table"], l2, scale)
        t_total += time.perf_counter() - t
        Hkv, d = s["kn"].shape[1], s["kn"].shape[2]
        H = s["q"].shape[1]
        dec, app = paged_bytes(np.array([s["len"] + 1]), 1, H, Hkv, d, d, s["kp"].shape[2])
        done_bytes += dec + app
        n += 1
        if t_total > max_seconds:
            break
    return done_bytes, t_total, n


# ---------------------------------------------------------------------------
# the prefill workload (secondary line of the metric)

def run_prefill(args, peaks, peak_kind):
    import causal_gqa_attention_row_gb300 as g
    dev = torch.device("cuda")
    B, S, H, Hkv, d = 1, 2048, 14, 2, 64
    c = W.make_prefill(B=B, S=S, H=H, Hkv=Hkv, dk=d, dv=d, seed=1, device=dev)
    q0, k0 = c.q.clone(), c.k.clone()
    pos = torch.arange(S, dtype=torch.int32, device=dev)[None].repeat(B, 1)
    out = torch.empty(B, S, H, d, dtype=torch.bfloat16, device=dev)
    flops = 2.0 * H * (d + d) * S * (S + 1) / 2
    st = torch.cuda.current_stream()
    # each step: RoPE on fresh copies of q and k, then the causal prefill
    def step(ev=None):
        c.q.copy_(q0)
        c.k.copy_(k0)
        g.attn_rope_interleaved(c.q, pos, 1e6)
        g.attn_rope_interleaved(c.k, pos, 1e6, heads_outer=True)
        if ev:
            ev[0].record(st)
        g.attn_prefill_causal(c.q, c.k, c.v, out, c.scale)
        if ev:
            ev[1].record(st)
    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    n = max(args.steps, 20)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    for i in range(n):
        step(evs[i])
    torch.cuda.synchronize()
    assert g.attn_get_device_error() == g.OK
    ms = statistics.median(a.elapsed_time(b) for a, b in evs)
    tflops = flops / (ms * 1e-3) / 1e12
    peak = peaks["bf16_tflops"]
    return {"workload": W.WORKLOADS["prefill"], "tflops": tflops, "ms": ms, "flops": flops,
            "roofline": {"bound": "tensor", "achieved": tflops, "peak": peak, "unit": "TFLOP/s",
                         "frac": tflops / peak, "peak_kind": f"bf16 dense burst, {peak_kind}"}}


# ---------------------------------------------------------------------------

def reference_arm(args, rank, world):
    """The fp64 oracle on the host cores, on bounded samples of the paged workload."""
    if rank != 0:
        return
    from oracle import core
    c = W.make_paged(B=256, H=32, Hkv=8, dk=128, dv=128, block_size=16, num_blocks=600_000, seed=3,
                     device="cpu") if False else None
    # A CPU-side replica of the same workload shape, generated small: the paged
    # pool here holds only the sampled sequences (history lengths drawn as in the
    # full workload).
    lens_all = torch.randint(1, 32769, (256,), generator=W.generator(3 + 1000), dtype=torch.int32)
    pick = lens_all[:args.cpu_seqs].tolist()
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
        oracle_paged_sample(sample[:1], cs.theta, cs.scale, 1e9)
    times, nbytes = [], 0
    for _ in range(args.steps):
        b_, t_, _ = oracle_paged_sample(sample, cs.theta, cs.scale, 1e9)
        times.append(t_)
        nbytes = b_
    ms = statistics.mean(times) * 1e3
    value = nbytes / (ms * 1e-3) / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": W.WORKLOADS["paged"], "sample": f"{len(pick)} sequences per step"},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": core.threads(), "kind": "oracle",
                             "sample": f"append + decode of {len(pick)} sequences of the paged workload "
                                       f"({sum(pick)} history rows) per step"},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seqs", type=int, default=8)
    ap.add_argument("--cpu-seconds", type=float, default=20.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    rank, world = dist_setup(args.gpus)
    if args.impl == "reference":
        reference_arm(args, rank, world)
        return
    peaks, peak_kind = measured_peaks()
    res = run_paged(args, rank, world, peaks, peak_kind)
    pre = None if args.no_prefill else run_prefill(args, peaks, peak_kind)
    if rank != 0:
        return
    cpu = None
    if res["sample"]:
        from oracle import core
        b_, t_, n_ = oracle_paged_sample(res["sample"], 1e6, 1.0 / math.sqrt(128), args.cpu_seconds)
        cpu = {"value": b_ / t_ / 1e9, "unit": "GB/s", "cores": core.threads(), "kind": "oracle",
               "sample": f"append + decode of {n_} sequences of the paged workload (shortest, longest and "
                         f"seeded others), {t_:.1f} s of oracle time"}
    hbm = peaks["hbm_gbs"]
    line = {
        "metric": METRIC, "value": res["value"], "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": res["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": W.WORKLOADS["paged"], "global_batch": 256 * world, "step": "kv_append_paged + "
                   "attn_decode_paged", "l2": "K/V working set ~17 GB per step, larger than L2 (no flush)",
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm", "achieved": res["achieved_decode_gbs"], "peak": hbm, "unit": "GB/s",
                     "frac": res["achieved_decode_gbs"] / hbm, "traffic": None,
                     "kernel": "attn_decode_paged (attn_rows_kernel + split_combine_kernel)",
                     "peak_kind": peak_kind, "frac_of_8tbs": res["achieved_decode_gbs"] / 8000.0},
        "cpu_baseline": cpu, "e2e": res["e2e"], "gpu_launches": 3 * args.steps, "clocks": res["clocks"],
        "prefill": pre,
    }
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
