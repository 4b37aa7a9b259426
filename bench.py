"""Benchmark of the attention forward hot path on GB300.

One step = the prefill workload "B=2, H=16, Sq=Sk=4096, d=128", run once
non-causal and once causal (two launches of the tcgen05 prefill kernel),
with inputs resident in HBM and L2 flushed between steps.  The JSON line's
``value`` is whole-job TFLOPS (4*B*H*S^2*d per non-causal pass, half for the
causal pass).  The same run also times the decode workload (B=64, Hq=64,
Hkv=8, d=128, key lengths ~U[1024, 16384] padded to 16384) in GB/s, and the
end-to-end path through the C ABI with host buffers (inputs copied in,
outputs copied back inside the timed region).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

``--impl reference`` times the fp64 CPU oracle (the test suite's reference
implementation) on a bounded sample of the same workload, on the host cores.
With N > 1 (launched by torchrun) every rank runs the same per-GPU workload
(weak scaling, no collective in the data path); times are the max over ranks.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "prefill fwd TFLOPS & % bf16 tensor peak; decode HBM GB/s & % peak (1×GB300)"
FLUSH_BYTES = 512 << 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# DRAM traffic per launch (dram__bytes_read.sum + dram__bytes_write.sum) from
# the ncu captures summarised under profiles/, keyed by the sha256 of the
# kernel sources at capture time.  A source change makes the entry stale, and
# stale entries are reported as null.
KERNEL_SOURCES = {
    "prefill": ["attention_forward_blackwell_gb300/csrc/prefill.cuh",
                "attention_forward_blackwell_gb300/csrc/ptx.cuh",
                "attention_forward_blackwell_gb300/csrc/common.cuh"],
    "decode": ["attention_forward_blackwell_gb300/csrc/decode.cu",
               "attention_forward_blackwell_gb300/csrc/ptx.cuh",
               "attention_forward_blackwell_gb300/csrc/common.cuh"],
}

CAPTURED_TRAFFIC = {
    # kernel: (sources sha256, bytes per launch, profile summary)
    "prefill": ("5f2090474e67d1d39c43c362dfd3b4ef62715398224c0f7bcd97a533a6de2de9",
                118664448, "profiles/prefill_kernel_d128_noncausal_b2_h16_s4096.md"),
    # captured at batch 16 (463.45 MB) and scaled to batch 64 by the
    # algorithmic bytes of the two batches
    "decode": ("6c42fe0c85c1b5e1ea69bf2dc9db9e431e10b54b837b8bdfa41a593ca1d3291a",
               2204452012, "profiles/decode_split_kernel_b16_hq64_hkv8_d128.md"),
}


def sources_hash(kernel):
    import hashlib
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def captured_traffic(kernel):
    entry = CAPTURED_TRAFFIC.get(kernel)
    if entry is None or entry[0] != sources_hash(kernel):
        return None
    return entry[1]


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=400)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-decode", action="store_true")
    p.add_argument("--decode-batch", type=int, default=None,
                   help="batch of the decode leg (default: the workload's 64); a "
                        "smaller batch keeps profiler captures small")
    p.add_argument("--cpu-seconds", type=float, default=10.0,
                   help="budget of the CPU (oracle) baseline sample")
    p.add_argument("--only", default=None, metavar="WORKLOAD",
                   help="time one named prefill workload alone (e.g. for a profiler "
                        "capture of its kernel) and print its median; not the bench line")
    return p.parse_args(argv)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained",
                                                     d["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS, source="fallback")


# ------------------------------------------------------------ distributed ----

class Dist:
    """Rank bookkeeping; N > 1 uses torch.distributed only for barriers and
    the max-over-ranks reduction of timings."""

    def __init__(self, gpus):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            backend = os.environ.get("BENCH_DIST_BACKEND", "nccl")
            dist.init_process_group(backend=backend)
            self.pg = dist
        if gpus != self.world and self.world > 1:
            print(f"warning: --gpus {gpus} but WORLD_SIZE {self.world}", file=sys.stderr)

    def barrier(self):
        if self.pg is not None:
            self.pg.barrier()

    def max(self, value: float) -> float:
        return reduce_max(self.pg, value)

    def close(self):
        if self.pg is not None:
            self.pg.destroy_process_group()


def reduce_max(pg, value: float) -> float:
    """Max of a float over all ranks (identity without a process group)."""
    if pg is None:
        return float(value)
    import torch
    backend = pg.get_backend()
    dev = torch.device("cuda") if backend == "nccl" else torch.device("cpu")
    t = torch.tensor([float(value)], dtype=torch.float64, device=dev)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def aggregate(per_rank_units: float, world: int, max_seconds: float) -> float:
    """Whole-job throughput: units processed by all ranks / slowest rank's time."""
    return per_rank_units * world / max_seconds


# ----------------------------------------------------------------- clocks ----

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index=0, period_ms=50):
        self.device_index = device_index
        self.period_ms = period_ms
        self.proc = None
        self.lines = []

    def start(self):
        try:
            import torch
            sel = []
            try:
                uuid = str(torch.cuda.get_device_properties(self.device_index).uuid)
                sel = ["-i", uuid if uuid.startswith("GPU-") else "GPU-" + uuid]
            except Exception:
                sel = []
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", str(self.period_ms)] + sel,
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.lines = [l for l in out.splitlines() if l.strip()]
        return self.summary()

    def summary(self):
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------- our arm ----

def _events(torch, n):
    return [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in range(n)]


def run_ours(args, dist):
    import torch
    from attention_forward_blackwell_gb300 import binding, build, inputs, workloads

    build.build()
    torch.cuda.set_device(dist.local_rank)
    dev = torch.device("cuda", dist.local_rank)
    peaks = load_peaks()
    W = workloads
    wn, wc = W.PREFILL_D128, W.PREFILL_D128_CAUSAL
    x = inputs.make_inputs(wn.B, wn.Hq, wn.Hkv, wn.Sq, wn.Sk, wn.d, tag=wn.tag, device=dev)
    o_n, o_c = torch.empty_like(x.q), torch.empty_like(x.q)
    l_n = torch.empty(wn.B, wn.Hq, wn.Sq, device=dev)
    l_c = torch.empty_like(l_n)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.int8, device=dev)
    f_n = W.prefill_flops(wn.B, wn.Hq, wn.Sq, wn.Sk, wn.d, False)
    f_c = W.prefill_flops(wc.B, wc.Hq, wc.Sq, wc.Sk, wc.d, True)

    def step_nc():
        binding.prefill(x.q, x.k, x.v, scale=wn.scale, causal=False, out=o_n, lse=l_n)

    def step_c():
        binding.prefill(x.q, x.k, x.v, scale=wc.scale, causal=True, out=o_c, lse=l_c)

    for _ in range(max(3, args.warmup)):
        flush.zero_()
        step_nc()
        step_c()
    torch.cuda.synchronize()
    assert binding.get_device_error() == binding.FA_OK

    K = args.steps
    ev_n, ev_c = _events(torch, K), _events(torch, K)
    clocks = ClockSampler(dist.local_rank).start()
    time.sleep(0.3)
    dist.barrier()
    torch.cuda.synchronize()
    for i in range(K):
        flush.zero_()                    # L2 flush, outside the timed events
        ev_n[i][0].record()
        step_nc()
        ev_n[i][1].record()
        ev_c[i][0].record()
        step_c()
        ev_c[i][1].record()
    torch.cuda.synchronize()
    dist.barrier()
    clk = clocks.stop()
    t_n = [a.elapsed_time(b) for a, b in ev_n]
    t_c = [a.elapsed_time(b) for a, b in ev_c]
    assert binding.get_device_error() == binding.FA_OK
    dev_seconds = (sum(t_n) + sum(t_c)) / 1e3
    max_seconds = dist.max(dev_seconds)
    value = aggregate((f_n + f_c) * K, dist.world, max_seconds) / 1e12
    ms_per_step = max_seconds * 1e3 / K
    avg_n, avg_c = sum(t_n) / K, sum(t_c) / K
    achieved = f_n / (avg_n * 1e-3) / 1e12
    result = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOPS",
        "n_gpus": dist.world, "steps": K, "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "prefill_mha_b2_h16_s4096_d128 non-causal + causal "
                               "(one launch each per step)",
                   "B": wn.B, "H": wn.Hq, "Sq": wn.Sq, "Sk": wn.Sk, "d": wn.d,
                   "scale": "1/sqrt(128)", "inputs": "bf16 N(0,1), seeded",
                   "l2": "flushed between steps (512 MiB write outside the timed events)",
                   "parallelism": f"replica x{dist.world}"},
        "breakdown": {
            "noncausal_ms": round(avg_n, 4),
            "noncausal_tflops": round(f_n / (avg_n * 1e-3) / 1e12, 2),
            "causal_ms": round(avg_c, 4),
            "causal_tflops": round(f_c / (avg_c * 1e-3) / 1e12, 2),
            "context_pages_sm120_noncausal_tflops": 258.7,
        },
        "roofline": {"kernel": "prefill_kernel<128,false> (non-causal launch)",
                     "bound": "tensor", "achieved": round(achieved, 2),
                     "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": round(achieved / peaks["bf16_tflops"], 4),
                     "peak_source": peaks["source"] + " (burst bf16 GEMM)",
                     "traffic": captured_traffic("prefill"),
                     "kernel_sources_sha256": sources_hash("prefill")[:16]},
        "gpu_launches": 2 * K,
        "clocks": clk,
    }
    del o_c, l_c
    if not args.no_e2e:
        result["e2e"] = run_e2e(args, torch, binding, x, wn, f_n, f_c, dist)
    if not args.no_decode:
        result["decode"] = run_decode(args, torch, binding, inputs, W, peaks, dev, dist)
    if dist.rank == 0:
        result["cpu_baseline"] = cpu_baseline(args, wn)
    return result


def run_e2e(args, torch, binding, x, w, f_n, f_c, dist):
    """Same two prefill passes through the public API, fed from pinned host
    buffers: every step copies its Q, K, V in and both passes' O and LSE out
    inside the timed region.  The steps are pipelined the way a serving loop
    streams batches: two device buffer sets; step i+1's inputs copy in on a
    copy stream while step i computes, and step i's outputs copy out on a
    second copy stream; events order each buffer set's reuse."""
    hq, hk, hv = (t.cpu().pin_memory() for t in (x.q, x.k, x.v))
    n_sets = 2
    din = [[torch.empty_like(t) for t in (x.q, x.k, x.v)] for _ in range(n_sets)]
    dout = [[torch.empty_like(x.q) for _ in range(2)] for _ in range(n_sets)]
    dlse = [[torch.empty(w.B, w.Hq, w.Sq, device=x.q.device) for _ in range(2)]
            for _ in range(n_sets)]
    hout = [[torch.empty(x.q.shape, dtype=x.q.dtype, pin_memory=True) for _ in range(2)]
            for _ in range(n_sets)]
    hlse = [[torch.empty(w.B, w.Hq, w.Sq, dtype=torch.float32, pin_memory=True)
             for _ in range(2)] for _ in range(n_sets)]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    s_comp = torch.cuda.current_stream()
    ev = lambda: torch.cuda.Event()
    in_done = [ev() for _ in range(n_sets)]
    comp_done = [ev() for _ in range(n_sets)]
    out_done = [ev() for _ in range(n_sets)]
    used = [False] * n_sets
    K = max(1, min(args.steps, 200))

    def step(i):
        j = i % n_sets
        dq, dk, dv = din[j]
        with torch.cuda.stream(s_in):
            if used[j]:
                s_in.wait_event(comp_done[j])      # the set's inputs are no longer read
            dq.copy_(hq, non_blocking=True)
            dk.copy_(hk, non_blocking=True)
            dv.copy_(hv, non_blocking=True)
            in_done[j].record(s_in)
        s_comp.wait_event(in_done[j])
        if used[j]:
            s_comp.wait_event(out_done[j])         # the set's outputs have been read back
        binding.prefill(dq, dk, dv, scale=w.scale, causal=False, out=dout[j][0],
                        lse=dlse[j][0], stream=s_comp)
        binding.prefill(dq, dk, dv, scale=w.scale, causal=True, out=dout[j][1],
                        lse=dlse[j][1], stream=s_comp)
        comp_done[j].record(s_comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(comp_done[j])
            for r in range(2):
                hout[j][r].copy_(dout[j][r], non_blocking=True)
                hlse[j][r].copy_(dlse[j][r], non_blocking=True)
            out_done[j].record(s_out)
        used[j] = True

    for i in range(3):
        step(i)
    torch.cuda.synchronize()
    dist.barrier()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(s_in)
    for i in range(K):
        step(i)
    s_out.wait_stream(s_in)
    s_out.wait_stream(s_comp)
    b.record(s_out)
    torch.cuda.synchronize()
    secs = dist.max(a.elapsed_time(b) / 1e3)
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv))
    d2h = sum(t.numel() * t.element_size() for t in hout[0] + hlse[0])
    return {"value": round(aggregate((f_n + f_c) * K, dist.world, secs) / 1e12, 2),
            "unit": "TFLOPS", "steps": K, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": round(secs * 1e3 / K, 4),
            "pipelined": "2 buffer sets; copy-in, compute and copy-out on 3 streams"}


def run_decode(args, torch, binding, inputs, W, peaks, dev, dist):
    w = W.DECODE
    if args.decode_batch is not None and args.decode_batch != w.B:
        import dataclasses
        w = dataclasses.replace(w, B=int(args.decode_batch), name=f"{w.name}_batch{args.decode_batch}")
    x = inputs.make_inputs(w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.d, tag=w.tag, device=dev,
                           lengths=w.lengths)
    lens = x.seqlens_k.cpu().tolist()
    nbytes = W.decode_bytes(w.Hkv, w.Hq, w.d, lens)
    o = torch.empty_like(x.q)
    lse = torch.empty(w.B, w.Hq, w.Sq, device=dev)

    def step():
        binding.decode(x.q, x.k, x.v, scale=w.scale, seqlens_k=x.seqlens_k, out=o, lse=lse)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    K = args.steps
    ev = _events(torch, K)
    dist.barrier()
    flush = torch.empty(FLUSH_BYTES, dtype=torch.int8, device=dev)
    for i in range(K):
        flush.zero_()           # L2 flush outside the timed events
        ev[i][0].record()
        step()
        ev[i][1].record()
    torch.cuda.synchronize()
    assert binding.get_device_error() == binding.FA_OK
    t = [a.elapsed_time(b) for a, b in ev]
    secs = dist.max(sum(t) / 1e3)
    gbs = aggregate(nbytes * K, dist.world, secs) / 1e9
    per_gpu = nbytes / (sum(t) / K * 1e-3) / 1e9
    return {"workload": w.name, "value": round(gbs, 1), "unit": "GB/s",
            "ms_per_step": round(secs * 1e3 / K, 4), "algorithmic_bytes": nbytes,
            "sum_lengths": int(sum(lens)),
            "roofline": {"bound": "hbm", "achieved": round(per_gpu, 1),
                         "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": round(per_gpu / peaks["hbm_gbs"], 4),
                         "peak_source": peaks["source"],
                         "traffic": captured_traffic("decode") if w.B == W.DECODE.B else None,
                         "kernel_sources_sha256": sources_hash("decode")[:16]},
            "gpu_launches": 2 * K,
            "l2": "flushed between steps (512 MiB write outside the timed events)"}


# -------------------------------------------------------- CPU baseline ----

def cpu_baseline(args, w, budget=None):
    """The fp64 oracle, as it stands, on a bounded sample of query rows of the
    non-causal prefill workload, over all host cores; scaled to TFLOPS."""
    import numpy as np
    import torch
    import oracle
    from attention_forward_blackwell_gb300 import inputs
    budget = args.cpu_seconds if budget is None else budget
    x = inputs.make_inputs(w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.d, tag=w.tag, device="cpu")
    qb, kb, vb = (inputs.bf16_bits(t) for t in (x.q, x.k, x.v))
    cores = os.cpu_count() or 1
    rng = np.random.default_rng(7)
    total = w.B * w.Hq * w.Sq
    per_row = 4.0 * w.Sk * w.d
    # calibrate on a few rows, then size the sample to the budget
    probe = rng.integers(0, total, size=cores * 2)
    t0 = time.perf_counter()
    oracle.attention_fwd(qb, kb, vb, scale=w.scale, rows=probe, threads=cores)
    dt = time.perf_counter() - t0
    n = int(max(cores, min(total, len(probe) * budget / max(dt, 1e-6))))
    rows = rng.integers(0, total, size=n)
    t0 = time.perf_counter()
    oracle.attention_fwd(qb, kb, vb, scale=w.scale, rows=rows, threads=cores)
    dt = time.perf_counter() - t0
    return {"value": round(per_row * n / dt / 1e12, 6), "unit": "TFLOPS", "cores": cores,
            "kind": "oracle", "seconds": round(dt, 2),
            "sample": f"{n} random query rows of {w.name} (non-causal, all {w.Sk} keys "
                      f"each), fp64 C oracle, one thread per core"}


# ---------------------------------------------------------- reference arm ----

def run_reference(args, dist):
    """The oracle on the host cores, per step a bounded sample of the same
    workload, with the same metric, unit and config as our arm."""
    if dist.rank != 0:
        return None
    import numpy as np
    import oracle
    from attention_forward_blackwell_gb300 import inputs, workloads
    wn = workloads.PREFILL_D128
    x = inputs.make_inputs(wn.B, wn.Hq, wn.Hkv, wn.Sq, wn.Sk, wn.d, tag=wn.tag, device="cpu")
    qb, kb, vb = (inputs.bf16_bits(t) for t in (x.q, x.k, x.v))
    cores = os.cpu_count() or 1
    total = wn.B * wn.Hq * wn.Sq
    rng = np.random.default_rng(11)
    # rows per step: sized so warmup + steps stay within ~2 minutes
    probe = rng.integers(0, total, size=cores)
    t0 = time.perf_counter()
    oracle.attention_fwd(qb, kb, vb, scale=wn.scale, rows=probe, threads=cores)
    per_row_s = (time.perf_counter() - t0) / len(probe)
    n_steps = args.warmup + args.steps
    rows_per_step = int(max(cores, min(total, 120.0 / n_steps / per_row_s)))
    # causal rows see on average half the keys: sample them too
    flops_nc = 4.0 * wn.Sk * wn.d
    for _ in range(args.warmup):
        oracle.attention_fwd(qb, kb, vb, scale=wn.scale, rows=rng.integers(0, total, rows_per_step),
                             threads=cores)
    flops = 0.0
    t0 = time.perf_counter()
    for i in range(args.steps):
        causal = bool(i % 2)
        rows = rng.integers(0, total, rows_per_step)
        oracle.attention_fwd(qb, kb, vb, scale=wn.scale, causal=causal, rows=rows, threads=cores)
        if causal:
            flops += float(np.sum(4.0 * ((rows % wn.Sq) + 1) * wn.d))
        else:
            flops += flops_nc * rows_per_step
    secs = time.perf_counter() - t0
    value = flops / secs / 1e12
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOPS",
        "n_gpus": dist.world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(secs * 1e3 / max(1, args.steps), 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "prefill_mha_b2_h16_s4096_d128 non-causal + causal",
                   "B": wn.B, "H": wn.Hq, "Sq": wn.Sq, "Sk": wn.Sk, "d": wn.d},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOPS", "cores": cores,
                         "kind": "oracle",
                         "sample": f"{rows_per_step} random query rows per step, "
                                   "alternating non-causal and causal steps"},
        "e2e": {"value": round(value, 6), "unit": "TFLOPS", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def run_only(args, dist):
    """One prefill workload (workloads.ALL by name), L2 flushed before each of
    `steps` timed launches after `warmup` untimed ones."""
    import torch
    from attention_forward_blackwell_gb300 import binding, build, inputs, workloads as W

    build.build()
    torch.cuda.set_device(dist.local_rank)
    dev = torch.device("cuda", dist.local_rank)
    w = {x.name: x for x in W.ALL}.get(args.only)
    if w is None or w.Sq != w.Sk:
        raise SystemExit(f"--only: not a prefill workload: {args.only}")
    x = inputs.make_inputs(w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.d, tag=w.tag, device=dev,
                           k_scale=w.k_scale)
    o = torch.empty_like(x.q)
    lse = torch.empty(w.B, w.Hq, w.Sq, device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.int8, device=dev)

    def step():
        binding.prefill(x.q, x.k, x.v, scale=w.scale, causal=w.causal, out=o, lse=lse)

    for _ in range(max(1, args.warmup)):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    ev = _events(torch, args.steps)
    for a, b in ev:
        flush.zero_()
        a.record()
        step()
        b.record()
    torch.cuda.synchronize()
    assert binding.get_device_error() == binding.FA_OK
    ms = sorted(a.elapsed_time(b) for a, b in ev)[len(ev) // 2]
    f = W.prefill_flops(w.B, w.Hq, w.Sq, w.Sk, w.d, w.causal)
    return {"only": w.name, "ms": round(ms, 4), "tflops": round(f / (ms * 1e-3) / 1e12, 2)}


def main(argv=None):
    args = parse_args(argv)
    dist = Dist(args.gpus)
    try:
        if args.only is not None:
            res = run_only(args, dist)
        elif args.impl == "reference":
            res = run_reference(args, dist)
        else:
            res = run_ours(args, dist)
        if dist.rank == 0 and res is not None:
            print(json.dumps(res), flush=True)
    finally:
        dist.close()


if __name__ == "__main__":
    main()
