"""Benchmark of the speculative-sampling verify step on GB300.

One step = one verify call (one kernel launch) over the whole batch of the
workload, inputs resident in HBM.  The default workload is the Qwen-vocabulary
batch the roofline is reported on: B=256 sequences, N=7 drafts, V=151936,
bf16 logits, T=0.8 (1.17 GB of logits per call, larger than L2, so no flush is
needed between steps).

Prints one JSON line.  `--impl reference` times the float64 CPU oracle on the
host cores instead (a bounded sample of the same workload per step).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "verified rows/s (B·(N+1) logit rows) and achieved HBM GB/s vs GB300 peak"
UNIT = "rows/s"
FALLBACK_HBM_GBS = 6800.0
KERNEL_SOURCES = ["speculative_decoding_verification_49_gb300/csrc/spec_verify.cu",
                  "speculative_decoding_verification_49_gb300/csrc/sv_device.cuh"]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "row_normaliser_traffic.txt")


def dominant_kernel(w, num_sms: int) -> str:
    """The kernel that streams all B(2N+1) logit rows (row normalisers and
    accept tests): one CTA per logit row (sv_row_kernel) from a full wave of
    positions (four CTAs per SM), and from two CTAs per SM for batches of at
    most 1024 sequences (the rows that are read packed at the front of the
    grid), else one CTA or cluster per position (sv_rows_kernel)."""
    units = w.B * (w.N + 1)
    if units >= 4 * num_sms or (units >= 2 * num_sms and w.B <= 1024):
        return "sv_row_kernel"
    return "sv_rows_kernel"
L2_BYTES = 129 * 10**6  # GB300 L2


def _code_only(text: str) -> str:
    """C++ source without its comments, whitespace runs collapsed to one space:
    an edit to a comment leaves the digest (and the counters it vouches for)
    valid, any change to the code does not."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":  # string or character literal, copied whole
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_digest() -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, f), encoding="utf-8") as fh:
            h.update(_code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def committed_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source; else None."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    vals = {}
    with open(TRAFFIC_FILE) as f:
        for line in f:
            if ":" in line and not line.startswith("#"):
                k, v = line.split(":", 1)
                vals[k.strip()] = v.strip()
    if vals.get("kernel_digest") != kernel_digest():
        return None
    v = vals.get(f"dram_bytes_per_launch[{workload}]")
    return float(v) if v else None


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def tensor_peak():
    """Dense bf16 tensor throughput: the measured cuBLAS burst figure, else the fallback."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        if "bf16_tflops" in d:
            return float(d["bf16_tflops"]), "measured (cuBLAS bf16 burst)"
    return 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 200 ms."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.idx = device_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits", "-lms", "200",
                 "-i", str(self.idx)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        rows = []
        for line in (self.out or "").splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), float(parts[3]), parts[5:9]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in rows for k, v in enumerate(r[3]) if v.lower() == "active"})
        loaded = [r for r in rows if r[2] > 0] or rows
        return {"sm_mhz": statistics.median(r[0] for r in loaded), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows), "power_w_max": max(r[2] for r in rows)}


def dist_init(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl == "ours" else "gloo"
        dist.init_process_group(backend=backend)
        pg = dist
    return world, rank, local, pg


def max_over_ranks(ms: float, pg, device) -> float:
    """The slowest rank's time: every rank ran the same number of steps on its
    own replica, so the job finishes when the slowest one does."""
    if pg is None:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_step: int, world: int, steps: int, ms: float) -> float:
    """Whole-job throughput: units every rank processed, over the slowest time."""
    return units_per_step * world * steps / (ms * 1e-3)


def workload_desc(w) -> str:
    extra = {"headline": "T=0.8, Zipf prior (-1.1 ln rank) on odd sequences",
             "stress": "T=1.0, 5% forced near-zero-q drafts",
             "mixed": "T in {0,0.7,1} per sequence, sigma_q in [0.3,2]",
             "small": "T=1.0, 10% spiky target rows",
             "tiny": "T=1.0"}.get(w.name, "")
    return f"{w.name}: B={w.B} N={w.N} V={w.V} {w.dtype} logits, {extra}"


def cpu_oracle_rate(w, budget_s: float, threads: int):
    """Time the oracle, as it stands, on a bounded sample of the workload's
    sequences (about budget_s of CPU work); returns (rows/s, sequence
    verifications, seconds)."""
    import oracle
    import torch
    orc = oracle.Oracle()

    def args(n):
        s = torch.arange(n, device=w.target.device)
        return (w.target[s].cpu(), w.draft[s].cpu(), w.draft_tokens[s].cpu(),
                w.uniforms[s].double().cpu(), w.temperature[s].double().cpu())

    probe = min(w.B, threads)
    a = args(probe)
    t0 = time.perf_counter()
    orc.verify(*a, dtype=w.dtype, threads=threads, diagnostics=False)
    t_probe = time.perf_counter() - t0
    if t_probe >= 0.5 * budget_s:
        return probe * (w.N + 1) / t_probe, probe, t_probe
    # more sequences (up to the whole batch), then repeats, to fill the budget
    n = min(w.B, max(probe, int(probe * budget_s / t_probe) // threads * threads))
    t_one = t_probe * n / probe
    reps = max(1, int(budget_s / max(t_one, 1e-6)))
    a = args(n)
    t0 = time.perf_counter()
    for _ in range(reps):
        orc.verify(*a, dtype=w.dtype, threads=threads, diagnostics=False)
    dt = time.perf_counter() - t0
    return reps * n * (w.N + 1) / dt, reps * n, dt


def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import synth
    full = synth.config(args.workload)
    # a bounded sample of the workload: the first sequences of the same recipe
    w = synth.make_workload(args.workload, seed=0, device="cpu", B=min(full["B"], 128))
    threads = os.cpu_count() or 1
    # each step a bounded sample, so that warm-up plus steps stay within ~150 s
    per_step = min(args.ref_budget, max(0.02, 150.0 / (args.warmup + args.steps)))
    rates = []
    n_used = 0
    t_used = 0.0
    t_start = time.perf_counter()
    timed = 0
    for k in range(args.warmup + args.steps):
        r, n, dt = cpu_oracle_rate(w, per_step, threads)
        if k >= args.warmup:
            rates.append(r)
            n_used, t_used = n, dt
            timed += 1
        if time.perf_counter() - t_start > 180.0 and rates:
            break  # a single sequence takes longer than the per-step budget
    value = statistics.median(rates)
    sample = (f"{n_used} sequence verifications per step ({w.B} of the workload's {full['B']} sequences, "
              f"repeated; {n_used * (w.N + 1)} verified rows, "
              f"{n_used * (2 * w.N + 1) * w.V * w.elt / 1e9:.3f} GB of logits) in {t_used:.1f} s")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * n_used * (w.N + 1) / value,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": workload_desc(w).replace(f"B={w.B}", f"B={full['B']}"), "B": full["B"],
                   "N": w.N, "V": w.V, "sample_sequences": n_used, "steps_timed": timed},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


# KV layout of the commit measurement: a 7B-class model with grouped-query
# attention, 28 layers x {K, V} planes, 4 KV heads x 128 bf16 per token entry
KV_PLANES, KV_HEADS, KV_DIM, KV_MAX_LEN = 56, 4, 128, 2048


def measure_kv_commit(sv, torch, dev, stream, nacc, N, max_len=KV_MAX_LEN, reps=100):
    """Times spec_verify_kv_commit for the batch's accepted counts.  Before
    each call the lengths are restored and L2 is flushed: a 256 MiB write,
    then a 256 MiB read of another buffer, so that the timed copy starts with
    a cold L2 and does not pay for write-backs of the flush's dirty lines.
    Each call is bracketed by CUDA events on the launching stream."""
    B = nacc.shape[0]
    gen = torch.Generator(device=dev).manual_seed(11)
    scratch = torch.randn((KV_PLANES, B, N, KV_HEADS, KV_DIM), generator=gen, device=dev).to(torch.bfloat16)
    cache = torch.empty((KV_PLANES, B, max_len, KV_HEADS, KV_DIM), dtype=torch.bfloat16, device=dev)
    lens0 = torch.randint(0, max_len - N + 1, (B,), generator=gen, device=dev, dtype=torch.int32)
    lens = lens0.clone()
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    clean = torch.ones(64 << 20, dtype=torch.float32, device=dev)
    row_bytes = KV_HEADS * KV_DIM * 2
    a = nacc.cpu().clamp(min=0)
    moved = 2 * int(a.sum()) * KV_PLANES * row_bytes  # each committed row read once, written once
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    for k in range(reps + 3):
        lens.copy_(lens0)
        flush.zero_()
        clean.sum()
        if k >= 3:
            evs[k - 3][0].record(stream)
        sv.kv_commit(scratch, cache, lens, nacc, status=status, stream=stream)
        if k >= 3:
            evs[k - 3][1].record(stream)
    torch.cuda.synchronize(dev)
    if int(status.item()) != 0:
        raise RuntimeError(f"kv commit status {int(status.item())}")
    # the mean: single calls last a few event-timer ticks, and a median of
    # such samples moves by whole ticks
    us = statistics.mean(1e3 * e0.elapsed_time(e1) for e0, e1 in evs)
    gbs = moved / (us * 1e-6) / 1e9
    peak, peak_kind = peaks()
    del cache, scratch, flush, clean
    return {"us_per_call": us, "bytes_moved": moved, "gbs": gbs, "frac": gbs / peak,
            "peak": peak, "peak_kind": f"{peak_kind} (burst copy)", "launches_per_call": 2,
            "layout": f"{KV_PLANES} planes (28 layers x K,V) x B={B} x N={N} scratch rows -> cache of "
                      f"{max_len} positions, {row_bytes} B rows ({KV_HEADS} KV heads x {KV_DIM} bf16)",
            "accepted_rows": int(a.sum()), "timing": f"mean of {reps} calls, L2 flushed (256 MiB write, then 256 MiB read) before each"}


def measure_tree(sv, torch, dev, stream, rank, steps=200, warmup=5, cpu=True):
    """Times spec_verify_tree_run on the 64-tree batch (16-node trees shaped
    like static Medusa/EAGLE trees, V = 151936 bf16).  Its 467 MB of logits
    exceed L2, so calls run back to back between two CUDA events."""
    import synth
    w = synth.make_tree_workload("tree", seed=rank, device=dev)
    ctx = sv.SpecVerify(w.B, w.M, w.V, w.dtype, device=dev.index or 0)
    out = torch.empty((w.B, w.M + 1), dtype=torch.int32, device=dev)
    path = torch.empty_like(out)
    nacc = torch.empty((w.B,), dtype=torch.int32, device=dev)

    def call():
        ctx.tree_run(w.target, w.draft, w.parent, w.tokens, w.uniforms, w.temperature, out_tokens=out,
                     path_nodes=path, num_accepted=nacc, stream=stream)

    for _ in range(warmup):
        call()
    ctx.acceptance_counts(reset=True)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        call()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    if ctx.status() != sv.SV_OK:
        raise RuntimeError("device status set during the tree measurement")
    us = 1e3 * e0.elapsed_time(e1) / steps
    counts = ctx.acceptance_counts()
    mean_path = sum(k * c for k, c in enumerate(counts[: w.M + 1])) / max(1, sum(counts[: w.M + 1]))
    peak, peak_kind = peaks()
    gbs = w.logit_bytes / (us * 1e-6) / 1e9
    res = {"workload": f"tree: B={w.B} trees of M+1={w.M + 1} nodes (fixed 16-node topology), V={w.V} {w.dtype}, "
                       f"T=0.8, Zipf prior on odd trees",
           "us_per_call": us, "nodes_per_s": w.B * (w.M + 1) / (us * 1e-6), "logit_bytes": w.logit_bytes,
           "gbs": gbs, "frac": gbs / peak, "peak": peak, "peak_kind": f"{peak_kind} (burst copy)",
           "mean_path_length": mean_path, "launches_per_call": 2, "steps": steps,
           "note": "bytes count every verifier row and the draft rows of nodes with children; the walk's "
                   "re-reads of rejected row pairs are not counted"}
    if cpu:
        import numpy as np
        import oracle
        args = [t.cpu() for t in (w.target, w.draft, w.parent, w.tokens)] + \
            [w.uniforms.double().cpu(), w.temperature.double().cpu()]
        done, t0 = 0, time.perf_counter()
        while time.perf_counter() - t0 < 3.0:  # the whole batch, repeated for about 3 s
            oracle.tree_verify(*args, dtype=w.dtype, threads=os.cpu_count() or 1, diagnostics=False)
            done += w.B
        dt = time.perf_counter() - t0
        res["cpu_baseline"] = {"value": done * (w.M + 1) / dt, "unit": "tree nodes/s", "cores": os.cpu_count() or 1,
                               "kind": "oracle",
                               "sample": f"{done} tree verifications ({done // w.B} passes over the batch) in {dt:.1f} s"}
    ctx.close()
    return res


def measure_fused(sv, torch, dev, stream, rank, steps=20, warmup=3, batch=0):
    """Times spec_verify_run_fused on the 256-sequence, 7-draft batch with
    Qwen-sized heads (V = 151936; verifier K = 3584, draft K = 896) against
    the unfused pipeline: cuBLAS (torch.matmul) writes bf16 logits, then
    spec_verify_run verifies them.  The fused path runs both ways: keeping
    the verifier rows' float32 logits (the default) and recomputing the
    sampled verifier rows too (no logits in HBM).  The hidden states and weights (1.4 GB) exceed L2;
    calls run back to back between two CUDA events."""
    import synth
    w = synth.make_fused_workload("fused", seed=rank, device=dev, **({"B": batch} if batch else {}))
    ctx = sv.SpecVerify(w.B, w.N, w.V, "f32", device=dev.index or 0)
    ctx_r = sv.SpecVerify(w.B, w.N, w.V, "f32", device=dev.index or 0)
    ctx_r.set_fused_logits(False)
    ctx_b = sv.SpecVerify(w.B, w.N, w.V, "bf16", device=dev.index or 0)
    out = torch.empty((w.B, w.N + 1), dtype=torch.int32, device=dev)
    nacc = torch.empty((w.B,), dtype=torch.int32, device=dev)
    zt = torch.empty((w.B * (w.N + 1), w.V), dtype=torch.bfloat16, device=dev)
    zd = torch.empty((w.B * w.N, w.V), dtype=torch.bfloat16, device=dev)

    def fused():
        ctx.run_fused(w.target_hidden, w.target_weight, w.draft_hidden, w.draft_weight, w.draft_tokens, w.uniforms,
                      w.temperature, out_tokens=out, num_accepted=nacc, stream=stream)

    def fused_recompute():
        ctx_r.run_fused(w.target_hidden, w.target_weight, w.draft_hidden, w.draft_weight, w.draft_tokens,
                        w.uniforms, w.temperature, out_tokens=out, num_accepted=nacc, stream=stream)

    def unfused():
        torch.matmul(w.target_hidden, w.target_weight.T, out=zt)
        torch.matmul(w.draft_hidden, w.draft_weight.T, out=zd)
        ctx_b.run(zt.view(w.B, w.N + 1, w.V), zd.view(w.B, w.N, w.V), w.draft_tokens, w.uniforms, w.temperature,
                  out_tokens=out, num_accepted=nacc, stream=stream)

    def gemm_only():
        torch.matmul(w.target_hidden, w.target_weight.T, out=zt)
        torch.matmul(w.draft_hidden, w.draft_weight.T, out=zd)

    res = {}
    for name, fn in (("fused", fused), ("fused_recompute", fused_recompute), ("cublas_then_verify", unfused),
                     ("cublas_gemms_alone", gemm_only)):
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        res[name] = 1e3 * e0.elapsed_time(e1) / steps
    if ctx.status() != sv.SV_OK or ctx_r.status() != sv.SV_OK or ctx_b.status() != sv.SV_OK:
        raise RuntimeError("device status set during the fused measurement")
    tc_peak, tc_kind = tensor_peak()
    tflops = w.flops / (res["fused"] * 1e-6) / 1e12
    ctx.close()
    ctx_r.close()
    ctx_b.close()
    return {"workload": f"fused: B={w.B} N={w.N} V={w.V}, verifier K={w.Kt}, draft K={w.Kd}, bf16 hidden states and "
                        f"heads, T=0.8",
            "us_per_call": res["fused"], "verified_rows_per_s": w.B * (w.N + 1) / (res["fused"] * 1e-6),
            "unfused_us_per_call": res["cublas_then_verify"], "cublas_gemms_us": res["cublas_gemms_alone"],
            "speedup_vs_unfused": res["cublas_then_verify"] / res["fused"],
            "logits": "every verifier row's float32 logits written by its statistics epilogue and the sampled rows "
                      "read back; the sampled draft rows recomputed",
            "recompute_us_per_call": res["fused_recompute"],
            "recompute_speedup_vs_unfused": res["cublas_then_verify"] / res["fused_recompute"],
            "roofline": {"bound": "tensor", "achieved": tflops, "peak": tc_peak, "unit": "TFLOP/s",
                         "frac": tflops / tc_peak, "flops_per_call": w.flops,
                         "peak_kind": tc_kind},
            "launches_per_call": 7, "recompute_launches_per_call": 8, "steps": steps}


def measure_fused_sweep(sv, torch, dev, stream, rank, batches=(32, 64, 128, 512)):
    """The fused path against the unfused pipeline at other batch sizes (the
    256-sequence batch is measure_fused's): where, if anywhere, fusing pays."""
    rows = []
    for B in batches:
        r = measure_fused(sv, torch, dev, stream, rank, steps=10, warmup=2, batch=B)
        rows.append({"B": B, "fused_us": r["us_per_call"], "unfused_us": r["unfused_us_per_call"],
                     "cublas_gemms_us": r["cublas_gemms_us"], "speedup_vs_unfused": r["speedup_vs_unfused"],
                     "recompute_us": r["recompute_us_per_call"],
                     "recompute_speedup_vs_unfused": r["recompute_speedup_vs_unfused"],
                     "tflops_frac": r["roofline"]["frac"]})
        torch.cuda.empty_cache()
    return rows


def run_ours(args):
    import torch
    world, rank, local, pg = dist_init(args)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import synth
    import speculative_decoding_verification_49_gb300 as sv
    from speculative_decoding_verification_49_gb300 import build as svbuild
    svbuild.build()

    over = {"B": args.batch} if args.batch else {}
    w = synth.make_workload(args.workload, seed=rank, device=dev, **over)
    ctx = sv.SpecVerify(w.B, w.N, w.V, w.dtype, device=local)
    if args.cluster:
        ctx.set_cluster_size(args.cluster)
    stream = torch.cuda.current_stream(dev)
    out = torch.empty((w.B, w.N + 1), dtype=torch.int32, device=dev)
    nacc = torch.empty((w.B,), dtype=torch.int32, device=dev)

    def step():
        ctx.run(w.target, w.draft, w.draft_tokens, w.uniforms, w.temperature, out_tokens=out,
                num_accepted=nacc, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if pg:
        pg.barrier()
    torch.cuda.synchronize(dev)

    # Inputs smaller than twice L2 would be served from L2 on repeated calls:
    # then every timed call follows an L2 flush (a 256 MiB write, then a
    # 256 MiB read of another buffer, so no dirty lines are left to write
    # back) and the calls' own event intervals are summed.
    flush = args.flush or w.logit_bytes < 2 * L2_BYTES
    if flush:
        fl_w = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        fl_r = torch.ones(64 << 20, dtype=torch.float32, device=dev)

        def clear_l2():
            fl_w.zero_()
            fl_r.sum()

    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        if flush:
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(args.steps)]
            start.record(stream)
            for e0, e1 in evs:
                clear_l2()
                e0.record(stream)
                step()
                e1.record(stream)
            end.record(stream)
            torch.cuda.synchronize(dev)
            ms_local = sum(e0.elapsed_time(e1) for e0, e1 in evs)
        else:
            start.record(stream)
            for _ in range(args.steps):
                step()
            end.record(stream)
            torch.cuda.synchronize(dev)
            ms_local = start.elapsed_time(end)
    ms = max_over_ranks(ms_local, pg, dev)
    if pg:
        pg.barrier()
    if ctx.status() != sv.SV_OK:
        raise RuntimeError("device status set during the timed region")

    ms_step = ms / args.steps
    rows = w.verified_rows
    value = job_rate(rows, world, args.steps, ms)
    gbs = w.logit_bytes / (ms_step * 1e-3) / 1e9
    peak, peak_kind = peaks()

    # per-kernel device time over the same number of steps: the library
    # records CUDA events on the launching stream around each of its kernels
    ctx.profile(True)
    for _ in range(args.steps):
        if flush:
            clear_l2()
        step()
    ms_rows, ms_sample, nprof = ctx.profile_read()
    ctx.profile(False)
    rows_us = 1e3 * ms_rows / nprof
    sample_us = 1e3 * ms_sample / nprof
    rows_gbs = w.logit_bytes / (rows_us * 1e-6) / 1e9
    # bytes kernel A actually reads: every verifier row, and the draft rows of
    # sampled sequences only (greedy ones need no draft probabilities)
    Tc = w.temperature.float().cpu()
    n_sampled = 0 if w.greedy else int(((Tc > 0) & torch.isfinite(Tc)).sum())
    bytes_read = w.B * (w.N + 1) * w.V * w.elt + n_sampled * w.N * w.V * w.elt
    rows_kernel = dominant_kernel(w, torch.cuda.get_device_properties(dev).multi_processor_count)
    kernels = {
        rows_kernel: {"us_per_launch": rows_us, "share": ms_rows / (ms_rows + ms_sample),
                           "algorithmic_bytes": w.logit_bytes, "gbs": rows_gbs,
                           "bytes_read": bytes_read, "gbs_read": bytes_read / (rows_us * 1e-6) / 1e9,
                           "sampled_sequences": n_sampled},
        "sv_mass_kernel+sv_pick_kernel": {
            "us_per_launch": sample_us, "share": ms_sample / (ms_rows + ms_sample),
            "note": "residual sampling; re-reads the rejected row pair of each sampled sequence "
                    "(not counted in the metric)"},
    }

    # end to end through the C ABI: pinned host inputs copied in, outputs read back
    e2e = None
    if not args.no_e2e:
        h = {k: getattr(w, k).cpu().pin_memory() for k in ("target", "draft", "draft_tokens", "uniforms",
                                                           "temperature")}
        ho = torch.empty((w.B, w.N + 1), dtype=torch.int32).pin_memory()
        hn = torch.empty((w.B,), dtype=torch.int32).pin_memory()
        h2d = sum(t.numel() * t.element_size() for t in h.values())
        d2h = ho.numel() * 4 + hn.numel() * 4
        # A serving loop's pipeline: two device copies of the inputs, so that
        # the host-to-device copy of call i+1 (on a copy stream) overlaps the
        # verify of call i (on the compute stream); each call's outputs are
        # read back after its verify.  Every call still copies its own inputs
        # in and its outputs out inside the timed region.
        cs = torch.cuda.Stream(dev)
        d = [{k: torch.empty_like(getattr(w, k)) for k in h} for _ in range(2)]
        copied = [torch.cuda.Event() for _ in range(2)]
        freed = [torch.cuda.Event() for _ in range(2)]

        def e2e_copy(i):
            cs.wait_event(freed[i % 2])  # the verify that last read this buffer has finished
            with torch.cuda.stream(cs):
                for k in h:
                    d[i % 2][k].copy_(h[k], non_blocking=True)
            copied[i % 2].record(cs)

        def e2e_verify(i):
            b = d[i % 2]
            stream.wait_event(copied[i % 2])
            ctx.run(b["target"], b["draft"], b["draft_tokens"], b["uniforms"], b["temperature"],
                    out_tokens=out, num_accepted=nacc, stream=stream)
            freed[i % 2].record(stream)
            with torch.cuda.stream(stream):
                ho.copy_(out, non_blocking=True)
                hn.copy_(nacc, non_blocking=True)

        def e2e_run(n, start=None):
            for e in freed:
                e.record(stream)
            if start is not None:
                start.record(stream)
            cs.wait_stream(stream)
            e2e_copy(0)
            for i in range(n):
                if i + 1 < n:
                    e2e_copy(i + 1)
                e2e_verify(i)

        e2e_run(2)
        torch.cuda.synchronize(dev)
        if pg:
            pg.barrier()
        es, ee = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        k2 = max(1, min(args.steps, 20))
        e2e_run(k2, start=es)
        ee.record(stream)
        torch.cuda.synchronize(dev)
        ems = max_over_ranks(es.elapsed_time(ee), pg, dev)
        e2e = {"value": job_rate(rows, world, k2, ems), "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "steps": k2,
               "pipeline": "two input buffers: call i+1's host-to-device copy (copy stream) overlaps call i's "
                           "verify; outputs read back after each call"}

    # acceptance telemetry kept by the library over every run so far
    counts = ctx.acceptance_counts()
    runs = sum(counts)
    acc = None
    if runs:
        mean = sum(k * c for k, c in enumerate(counts[: w.N + 1])) / runs
        acc = {"runs_x_sequences": runs, "invalid": counts[w.N + 1], "mean_accepted": mean,
               "mean_tokens_per_call": mean + 1,
               "position_accept_rate": [sum(counts[i + 1: w.N + 1]) / max(1, sum(counts[i: w.N + 1]))
                                        for i in range(w.N)]}

    kv = None
    if not args.no_kv:
        kv = measure_kv_commit(sv, torch, dev, stream, nacc, w.N, max_len=args.kv_max_len)
    # the tree walk is bound by SM arithmetic: measure it before the power-heavy GEMMs
    tree = None
    if not args.no_tree:
        tree = measure_tree(sv, torch, dev, stream, rank, cpu=(rank == 0 and not args.no_cpu))
    fused = None
    if not args.no_fused:
        fused = measure_fused(sv, torch, dev, stream, rank, batch=args.fused_batch)
        if not args.no_fused_sweep:
            fused["sweep"] = measure_fused_sweep(sv, torch, dev, stream, rank)

    cpu = None
    check = None
    if rank == 0 and not args.no_cpu:
        if not args.no_check:
            # the CPU-baseline leg's oracle also checks every sequence of the
            # launch timed above (same inputs; a debug call for the ratios)
            sys.path.insert(0, os.path.join(ROOT, "tests"))
            import parity
            rep = parity.compare(w, parity.run_gpu(ctx, w), parity.run_oracle(w, threads=os.cpu_count() or 1))
            check = {k: rep.get(k) for k in ("sequences", "exact", "decisions", "band_decisions",
                                              "band_sequences", "band_mismatch", "q_rel_max", "S_rel_max",
                                              "decision_ratio_err_max")}
            check["band_rate"] = rep["band_decisions"] / max(1, rep["decisions"])
            check["mismatch_rate"] = rep["band_mismatch"] / max(1, rep["decisions"])
        rate, n, dt = cpu_oracle_rate(w, args.cpu_budget, os.cpu_count() or 1)
        rate1, n1, dt1 = cpu_oracle_rate(w, args.cpu_budget / 2, 1)
        cpu = {"value": rate, "unit": UNIT, "cores": os.cpu_count() or 1, "kind": "oracle",
               "sample": f"{n} sequence verifications of the same workload (its {w.B} sequences, repeated; "
                         f"{n * (w.N + 1)} verified rows) in {dt:.1f} s, float64 C oracle, one POSIX thread "
                         f"per core",
               "value_1core": rate1, "sample_1core": f"{n1} sequence verifications in {dt1:.1f} s on one core"}

    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": {"workload": workload_desc(w), "B": w.B, "N": w.N, "V": w.V,
                   "logit_bytes_per_step": w.logit_bytes,
                   "l2": ("L2 flushed before every timed call (256 MiB write + 256 MiB read); call times summed"
                          if flush else "inputs larger than L2 (129 MB); no flush between steps"),
                   "cluster_size": ctx.cluster_size(w.B, w.N), "parallelism": f"replicas x{world}"},
        "hbm_gbs": gbs,
        "roofline": {"bound": "hbm", "kernel": rows_kernel, "achieved": rows_gbs, "peak": peak,
                     "unit": "GB/s", "frac": rows_gbs / peak, "peak_kind": f"{peak_kind} (burst copy)",
                     "traffic": committed_traffic(w.name), "step_gbs": gbs, "step_frac": gbs / peak},
        "kernels": kernels,
        "acceptance": acc,
        "kv_commit": kv,
        "tree": tree,
        "fused_lm_head": fused,
        "e2e": e2e,
        "cpu_baseline": cpu,
        "gpu_launches": 3 * args.steps,  # rows, mass and pick kernels per verify call
        "clocks": clk.summary(),
        "check": check,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    # defaults: about a second of timed GPU work (long enough to sample clocks),
    # or a few oracle steps for the reference arm
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=None)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="headline")
    ap.add_argument("--batch", type=int, default=0, help="override B (profiling of a smaller case)")
    ap.add_argument("--cluster", type=int, default=0, help="cluster size override (0 = automatic)")
    ap.add_argument("--flush", action="store_true", help="flush L2 before every timed call, whatever the input size")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-check", action="store_true")
    ap.add_argument("--no-kv", action="store_true", help="skip the KV-cache commit measurement")
    ap.add_argument("--no-tree", action="store_true", help="skip the tree-verification measurement")
    ap.add_argument("--no-fused", action="store_true", help="skip the fused LM-head measurement")
    ap.add_argument("--fused-batch", type=int, default=0, help="override B of the fused LM-head measurement")
    ap.add_argument("--no-fused-sweep", action="store_true", help="skip the fused-vs-unfused batch sweep")
    ap.add_argument("--kv-max-len", type=int, default=KV_MAX_LEN,
                    help="cache positions of the KV-commit measurement (the copy does not depend on it)")
    ap.add_argument("--cpu-budget", type=float, default=10.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--ref-budget", type=float, default=8.0, help="seconds of oracle work per reference step")
    args = ap.parse_args()
    if args.steps is None:
        args.steps = 4000 if args.impl == "ours" else 5
    if args.warmup is None:
        args.warmup = 20 if args.impl == "ours" else 1
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
