"""Benchmark of the attention forward hot path on GB300.

One step runs every configuration of the hot path once per repetition: the
long prefill "B=1, H=16, Sq=Sk=8192, d=128" (the headline: the largest
prefill configuration, and the shape of the "fa4-sm120-research" throughput
table's first row), the prefill "B=2, H=16, S=4096, d=128" non-causal and
causal, its d=96 variant, the causal GQA "B=4, Hq=32, Hkv=4, S=2048, d=256"
(K scaled by 0.5), head_dim 64 at "B=4, H=32, S=2048" (the table's last
row), the tiny "B=1, H=1, S=128, d=64" (latency, in us) and the split-KV
decode "B=64, Hq=64, Hkv=8, d=128" with key lengths ~U[1024, 16384] (GB/s).
Every launch is timed on its own with CUDA events after an L2 flush
(a 512 MiB write outside the events); each configuration gets at least 50
timed launches (repetitions per step = ceil(50 / steps)) and reports the
median.  ``value`` is the headline configuration's TFLOPS (4*B*H*S^2*d over
its median time).  ``e2e`` is the headline configuration through the C ABI
fed from pinned host buffers (inputs copied in and outputs copied back inside
the timed region).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

``--impl reference`` times the fp64 CPU oracle (the test suite's reference
implementation) on a bounded sample of the headline configuration, on the
host cores.  With N > 1 (launched by torchrun) each configuration's
(batch entry, key/value head) pairs are dealt out over the ranks (shard_plan;
no collective in the data path) and times are the max over ranks.
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
MIN_REPS = 50
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# The pages' own forward figure for the headline shape (b=1, s=8192, h=16,
# d=128), measured on an RTX PRO 6000 (SM120): context, not a target.
PAGES_FWD_TFLOPS_B1_S8192_H16_D128 = 275.5

# DRAM traffic per launch (dram__bytes_read.sum + dram__bytes_write.sum) from
# one ncu capture of the named kernel, keyed by the sha256 of the kernel
# sources at capture time.  A source change makes the entry stale, and stale
# entries are reported as null.
KERNEL_SOURCES = {
    "prefill": ["attention_forward_blackwell_gb300/csrc/prefill.cuh",
                "attention_forward_blackwell_gb300/csrc/prefill_wide.cuh",
                "attention_forward_blackwell_gb300/csrc/ptx.cuh",
                "attention_forward_blackwell_gb300/csrc/common.cuh"],
    "decode": ["attention_forward_blackwell_gb300/csrc/decode.cu",
               "attention_forward_blackwell_gb300/csrc/ptx.cuh",
               "attention_forward_blackwell_gb300/csrc/common.cuh"],
}

CAPTURED_TRAFFIC = {
    # kernel: (sources sha256, workload, bytes per launch)
    "prefill": ("2c87fe4f574f485b478774c76ac76c261f8ae7a5bb32e1582f47bd86ef6e07af",
                "long_prefill_b1_h16_s8192_d128", 115617024),
    # captured at batch 16 (463.73 MB, 1.017 x its algorithmic bytes) and
    # scaled to batch 64 by the algorithmic bytes of the two batches
    "decode": ("4f0491259b04d4788454cb2e2704a1707995117770ea3398451eb287333e470e",
               "decode_gqa_b64_hq64_hkv8_d128", 2205759804),
}


def sources_hash(kernel):
    import hashlib
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def captured_traffic(kernel, workload):
    entry = CAPTURED_TRAFFIC.get(kernel)
    if entry is None or entry[0] != sources_hash(kernel) or entry[1] != workload:
        return None
    return entry[2]


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--decode-batch", type=int, default=None,
                   help="batch of the decode configuration (default: the workload's 64); a "
                        "smaller batch keeps profiler captures small")
    p.add_argument("--cpu-seconds", type=float, default=10.0,
                   help="budget of the CPU (oracle) baseline sample")
    p.add_argument("--only", default=None, metavar="WORKLOAD",
                   help="time one named workload alone (e.g. for a profiler capture of its "
                        "kernel) and print its median; not the bench line")
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


def shard_plan(B: int, Hkv: int, world: int, rank: int):
    """This rank's share of one problem's (batch entry, key/value head) pairs.

    The B * Hkv pairs, in (batch entry, kv head) order, are dealt out in
    contiguous ranges of equal size (within one pair); a rank's range is
    returned as rectangles (b0, b1, hk0, hk1) that are each one contiguous
    slice of the [B, H, S, d] tensors: whole batch entries, or a range of kv
    heads (with their query heads) of one batch entry.  Every pair belongs to
    exactly one rank, so the ranks together compute the whole problem once
    and exchange nothing.
    """
    n = B * Hkv
    p, p1 = n * rank // world, n * (rank + 1) // world
    segs = []
    while p < p1:
        b, hk = divmod(p, Hkv)
        if hk == 0 and p1 - p >= Hkv:
            nb = (p1 - p) // Hkv
            segs.append((b, b + nb, 0, Hkv))
            p += nb * Hkv
        else:
            e = min(p1, (b + 1) * Hkv)
            segs.append((b, b + 1, hk, e - b * Hkv))
            p = e
    return segs


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

def bench_workloads(decode_batch=None):
    """(key, workload) pairs of one step, the headline first."""
    from attention_forward_blackwell_gb300 import workloads as W
    dec = W.DECODE
    if decode_batch is not None and decode_batch != dec.B:
        import dataclasses
        dec = dataclasses.replace(dec, B=int(decode_batch), name=f"{dec.name}_batch{decode_batch}")
    return [("long_d128", W.LONG_D128), ("d128", W.PREFILL_D128),
            ("d128_causal", W.PREFILL_D128_CAUSAL), ("d96", W.LONG_D96),
            ("gqa_d256_causal", W.GQA_D256), ("d64", W.PREFILL_D64), ("tiny_d64", W.TINY),
            ("chunked_gqa", W.CHUNKED_GQA), ("decode", dec)]


class Case:
    """One workload's resident inputs and outputs on this rank, and the
    launches of this rank's shard of it (one per shard_plan rectangle)."""

    def __init__(self, w, dev, world, rank):
        import torch
        from attention_forward_blackwell_gb300 import inputs
        self.w = w
        self.x = inputs.make_inputs(w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.d, tag=w.tag, device=dev,
                                    k_scale=w.k_scale, lengths=w.lengths)
        self.o = torch.empty_like(self.x.q)
        self.lse = torch.empty(w.B, w.Hq, w.Sq, device=dev)
        self.segs = shard_plan(w.B, w.Hkv, world, rank)
        G = w.Hq // w.Hkv
        self.views = []
        for b0, b1, k0, k1 in self.segs:
            sl = None if self.x.seqlens_k is None else self.x.seqlens_k[b0:b1]
            self.views.append((self.x.q[b0:b1, k0 * G:k1 * G], self.x.k[b0:b1, k0:k1],
                               self.x.v[b0:b1, k0:k1], sl, self.o[b0:b1, k0 * G:k1 * G],
                               self.lse[b0:b1, k0 * G:k1 * G]))
        if w.decode:
            lens = self.x.seqlens_k.cpu().tolist()
            self.units = W_decode_bytes(w, lens)          # algorithmic bytes
            self.launches = 2 * len(self.segs)            # split + combine kernels
        else:
            self.units = W_prefill_flops(w)
            self.launches = len(self.segs)

    def run(self, stream=None):
        from attention_forward_blackwell_gb300 import binding
        w = self.w
        for q, k, v, sl, o, lse in self.views:
            if w.decode:
                binding.decode(q, k, v, scale=w.scale, causal=w.causal, seqlens_k=sl, out=o,
                               lse=lse, stream=stream)
            else:
                binding.prefill(q, k, v, scale=w.scale, causal=w.causal, seqlens_k=sl, out=o,
                                lse=lse, stream=stream)


def W_prefill_flops(w):
    from attention_forward_blackwell_gb300 import workloads as W
    return W.prefill_flops(w.B, w.Hq, w.Sq, w.Sk, w.d, w.causal)


def W_prefill_bytes(w):
    from attention_forward_blackwell_gb300 import workloads as W
    return W.prefill_bytes(w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.d)


def W_decode_bytes(w, lens):
    from attention_forward_blackwell_gb300 import workloads as W
    return W.decode_bytes(w.Hkv, w.Hq, w.d, lens)


def _median(xs):
    return statistics.median(xs)


def run_ours(args, dist):
    import torch
    from attention_forward_blackwell_gb300 import binding, build

    build.build()
    torch.cuda.set_device(dist.local_rank)
    dev = torch.device("cuda", dist.local_rank)
    peaks = load_peaks()
    cases = [(key, Case(w, dev, dist.world, dist.rank))
             for key, w in bench_workloads(args.decode_batch)]
    flush = torch.empty(FLUSH_BYTES, dtype=torch.int8, device=dev)
    K = args.steps
    W_ = max(3, args.warmup)
    reps = max(1, math.ceil(MIN_REPS / K))

    for _ in range(W_):
        for _, c in cases:
            flush.zero_()
            c.run()
    torch.cuda.synchronize()
    assert binding.get_device_error() == binding.FA_OK

    ev = {key: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                for _ in range(K * reps)] for key, _ in cases}
    clocks = ClockSampler(dist.local_rank).start()
    time.sleep(0.3)
    dist.barrier()
    torch.cuda.synchronize()
    for i in range(K):
        for key, c in cases:
            for r in range(reps):
                flush.zero_()                    # L2 flush, outside the timed events
                a, b = ev[key][i * reps + r]
                a.record()
                c.run()
                b.record()
    torch.cuda.synchronize()
    dist.barrier()
    clk = clocks.stop()
    assert binding.get_device_error() == binding.FA_OK

    times = {key: [a.elapsed_time(b) for a, b in ev[key]] for key, _ in cases}
    step_ms = dist.max(sum(sum(t) for t in times.values()) / K)
    breakdown = {}
    for key, c in cases:
        w = c.w
        med = dist.max(_median(times[key]))        # slowest rank's median, ms
        rate = aggregate(c.units / dist.world, dist.world, med * 1e-3)
        e = {"workload": w.name, "ms": round(med, 4), "reps": len(times[key]),
             "launches_per_rep": c.launches}
        if w.decode:
            gbs = rate / 1e9
            e.update({"GB_per_s": round(gbs, 1), "frac": round(gbs / peaks["hbm_gbs"], 4),
                      "algorithmic_bytes": c.units, "bound": "hbm",
                      "sum_lengths": int(c.x.seqlens_k.sum().item())})
        else:
            tf = rate / 1e12
            e.update({"TFLOPS": round(tf, 2), "frac": round(tf / peaks["bf16_tflops"], 4),
                      "flops": c.units, "causal": w.causal, "d": w.d, "bound": "tensor"})
            if key == "tiny_d64":
                e["us"] = round(med * 1e3, 2)
                e["note"] = "latency-bound (4.19 MFLOP): the roofline fraction does not apply"
            if key == "chunked_gqa":
                # 16 queries per sequence: 128 FLOP per K/V byte, HBM-bound;
                # the causal-halved FLOP count undercounts (the mask removes
                # almost nothing of 4,096 keys)
                nbytes = W_prefill_bytes(w)
                gbs = aggregate(nbytes / dist.world, dist.world, med * 1e-3) / 1e9
                e.update({"GB_per_s": round(gbs, 1), "frac": round(gbs / peaks["hbm_gbs"], 4),
                          "algorithmic_bytes": nbytes, "bound": "hbm",
                          "note": "GQA head packing: the 8 query heads of a kv group share "
                                  "one 128-row tile"})
        breakdown[key] = e

    head_key, head = cases[0]
    hw = head.w
    head_med = breakdown[head_key]["ms"]
    value = breakdown[head_key]["TFLOPS"]
    result = {
        "metric": METRIC, "value": value, "unit": "TFLOPS",
        "n_gpus": dist.world, "steps": K, "warmup": W_,
        "ms_per_step": round(step_ms, 4), "higher_is_better": True,
        "scaling": "strong" if dist.world > 1 else "weak",
        "vs_baseline": round(value / PAGES_FWD_TFLOPS_B1_S8192_H16_D128, 3),
        "vs_baseline_note": "value / 275.5 TFLOPS, the pages' forward figure for this shape on "
                            "an RTX PRO 6000 (SM120): context, not a target",
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{hw.name} (headline); every step also runs "
                               + ", ".join(c.w.name for _, c in cases[1:]),
                   "B": hw.B, "H": hw.Hq, "Sq": hw.Sq, "Sk": hw.Sk, "d": hw.d, "causal": False,
                   "scale": "1/sqrt(128)", "inputs": "bf16 N(0,1), seeded",
                   "timing": f"median of {K * reps} launches per configuration "
                             f"({reps} per step), CUDA events around each launch",
                   "l2": "flushed before every timed launch (512 MiB write outside the events)",
                   "parallelism": ("one GPU" if dist.world == 1 else
                                   f"(batch, kv head) pairs sharded over {dist.world} ranks")},
        "breakdown": breakdown,
        "roofline": {"kernel": "prefill_kernel_wide<128, non-causal> (persistent, 256-key "
                               "blocks; headline launch)",
                     "bound": "tensor", "achieved": value,
                     "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": round(value / peaks["bf16_tflops"], 4),
                     "peak_source": peaks["source"] + " (burst bf16 GEMM)",
                     "traffic": captured_traffic("prefill", hw.name),
                     "kernel_sources_sha256": sources_hash("prefill")[:16]},
        "gpu_launches": K * reps * sum(c.launches for _, c in cases),
        "clocks": clk,
    }
    dec = breakdown["decode"]
    dec["roofline"] = {"bound": "hbm", "achieved": dec["GB_per_s"], "peak": peaks["hbm_gbs"],
                       "unit": "GB/s", "frac": dec["frac"], "peak_source": peaks["source"],
                       "traffic": captured_traffic("decode", dict(cases)["decode"].w.name),
                       "kernel_sources_sha256": sources_hash("decode")[:16]}
    if not args.no_e2e:
        result["e2e"] = run_e2e(args, torch, head, dist)
    del cases
    torch.cuda.empty_cache()
    if dist.rank == 0:
        result["cpu_baseline"] = cpu_baseline(args, hw)
    return result


def run_e2e(args, torch, case, dist):
    """The headline configuration through the public API, fed from pinned
    host buffers: every step copies this rank's Q, K, V in and its O and LSE
    out inside the timed region.  Steps are pipelined the way a serving loop
    streams batches: two device buffer sets; step i+1's inputs copy in on a
    copy stream while step i computes, and step i's outputs copy out on a
    second copy stream; events order each buffer set's reuse."""
    from attention_forward_blackwell_gb300 import binding
    w = case.w
    views = case.views
    host_in = [[t.cpu().pin_memory() for t in v[:3]] for v in views]
    n_sets = 2
    dev_in = [[[torch.empty_like(t) for t in v[:3]] for v in views] for _ in range(n_sets)]
    dev_out = [[(torch.empty_like(v[4]), torch.empty_like(v[5])) for v in views]
               for _ in range(n_sets)]
    host_out = [[(torch.empty(v[4].shape, dtype=v[4].dtype, pin_memory=True),
                  torch.empty(v[5].shape, dtype=v[5].dtype, pin_memory=True)) for v in views]
                for _ in range(n_sets)]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    s_comp = torch.cuda.current_stream()
    in_done = [torch.cuda.Event() for _ in range(n_sets)]
    comp_done = [torch.cuda.Event() for _ in range(n_sets)]
    out_done = [torch.cuda.Event() for _ in range(n_sets)]
    used = [False] * n_sets
    K = max(20, min(args.steps, 200))

    def step(i):
        j = i % n_sets
        with torch.cuda.stream(s_in):
            if used[j]:
                s_in.wait_event(comp_done[j])      # the set's inputs are no longer read
            for hs, ds in zip(host_in, dev_in[j]):
                for h, d in zip(hs, ds):
                    d.copy_(h, non_blocking=True)
            in_done[j].record(s_in)
        s_comp.wait_event(in_done[j])
        if used[j]:
            s_comp.wait_event(out_done[j])         # the set's outputs have been read back
        for (q, k, v), (o, lse), view in zip(dev_in[j], dev_out[j], views):
            binding.prefill(q, k, v, scale=w.scale, causal=w.causal, seqlens_k=view[3], out=o,
                            lse=lse, stream=s_comp)
        comp_done[j].record(s_comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(comp_done[j])
            for (o, lse), (ho, hl) in zip(dev_out[j], host_out[j]):
                ho.copy_(o, non_blocking=True)
                hl.copy_(lse, non_blocking=True)
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
    h2d = sum(t.numel() * t.element_size() for hs in host_in for t in hs)
    d2h = sum(t.numel() * t.element_size() for hs in host_out[0] for t in hs)
    return {"value": round(aggregate(case.units / dist.world * K, dist.world, secs) / 1e12, 2),
            "unit": "TFLOPS", "workload": w.name, "steps": K, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": round(secs * 1e3 / K, 4),
            "pipelined": "2 buffer sets; copy-in, compute and copy-out on 3 streams"}


# -------------------------------------------------------- CPU baseline ----

def cpu_baseline(args, w, budget=None):
    """The fp64 oracle, as it stands, on a bounded sample of query rows of the
    headline prefill workload, over all host cores; scaled to TFLOPS."""
    import numpy as np
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
    """The oracle on the host cores, per step a bounded sample of the headline
    workload, with the same metric, unit and config as our arm."""
    if dist.rank != 0:
        return None
    import numpy as np
    import oracle
    from attention_forward_blackwell_gb300 import inputs, workloads
    w = workloads.LONG_D128
    x = inputs.make_inputs(w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.d, tag=w.tag, device="cpu")
    qb, kb, vb = (inputs.bf16_bits(t) for t in (x.q, x.k, x.v))
    cores = os.cpu_count() or 1
    total = w.B * w.Hq * w.Sq
    rng = np.random.default_rng(11)
    # rows per step: sized so warmup + steps stay within ~2 minutes
    probe = rng.integers(0, total, size=cores)
    t0 = time.perf_counter()
    oracle.attention_fwd(qb, kb, vb, scale=w.scale, rows=probe, threads=cores)
    per_row_s = (time.perf_counter() - t0) / len(probe)
    n_steps = args.warmup + args.steps
    rows_per_step = int(max(cores, min(total, 120.0 / n_steps / per_row_s)))
    flops_per_row = 4.0 * w.Sk * w.d
    for _ in range(args.warmup):
        oracle.attention_fwd(qb, kb, vb, scale=w.scale, rows=rng.integers(0, total, rows_per_step),
                             threads=cores)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.attention_fwd(qb, kb, vb, scale=w.scale, rows=rng.integers(0, total, rows_per_step),
                             threads=cores)
    secs = time.perf_counter() - t0
    value = flops_per_row * rows_per_step * args.steps / secs / 1e12
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOPS",
        "n_gpus": dist.world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(secs * 1e3 / max(1, args.steps), 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{w.name} (headline)", "B": w.B, "H": w.Hq, "Sq": w.Sq,
                   "Sk": w.Sk, "d": w.d, "causal": False},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOPS", "cores": cores,
                         "kind": "oracle",
                         "sample": f"{rows_per_step} random query rows per step "
                                   f"(all {w.Sk} keys each)"},
        "e2e": {"value": round(value, 6), "unit": "TFLOPS", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def run_only(args, dist):
    """One workload (workloads.ALL by name), L2 flushed before each of `steps`
    timed launches after `warmup` untimed ones."""
    import torch
    from attention_forward_blackwell_gb300 import binding, build, workloads as W

    build.build()
    torch.cuda.set_device(dist.local_rank)
    dev = torch.device("cuda", dist.local_rank)
    w = {x.name: x for x in W.ALL}.get(args.only)
    if w is None:
        raise SystemExit(f"--only: unknown workload: {args.only}")
    if w.decode and args.decode_batch is not None:
        import dataclasses
        w = dataclasses.replace(w, B=int(args.decode_batch))
    c = Case(w, dev, 1, 0)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.int8, device=dev)
    for _ in range(max(1, args.warmup)):
        flush.zero_()
        c.run()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    for a, b in ev:
        flush.zero_()
        a.record()
        c.run()
        b.record()
    torch.cuda.synchronize()
    assert binding.get_device_error() == binding.FA_OK
    ms = _median([a.elapsed_time(b) for a, b in ev])
    if w.decode:
        return {"only": w.name, "ms": round(ms, 4), "GB_per_s": round(c.units / (ms * 1e-3) / 1e9, 1)}
    return {"only": w.name, "ms": round(ms, 4), "tflops": round(c.units / (ms * 1e-3) / 1e12, 2)}


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
