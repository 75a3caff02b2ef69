"""Benchmark of the GB300 attention forward (prints one JSON line on rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Headline workload: the lecture demo's sequence-length sweep, non-causal MHA,
B=4, H=8, D=64, Lq=Lk in {64, ..., 8192}.  One step = one forward pass at every
length of the sweep.  `value` = total algorithmic FLOPs (4*B*H*Lq*Lk*D) of a
step / device time of the step, in TFLOPS, with the inputs resident in HBM;
L2 is flushed (a 256 MiB write) before every launch and the flush is not
timed.  `e2e` is the same metric through the host-buffer API (pinned host
tensors copied in, O and LSE copied back, inside the timed region).
`per_config` adds the causal prefill, long-context and single-query decode
workloads (device time, TFLOPS or GB/s, and the fraction of the measured
peak).  `--impl reference` times the fp64 CPU oracle on a bounded sample of
the same workload instead.

Multi-GPU (torchrun): every rank runs the same per-GPU workload on its own
GPU (heads are independent: weak scaling, no collective on the data path);
rank 0 reports the max step time over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
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

METRIC = "attention fwd TFLOPS (bf16) and % of GB300 BF16 peak; decode GB/s vs HBM peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FLUSH_BYTES = 256 << 20
# GB300's specified HBM3e bandwidth: the ceiling for a read-mostly stream,
# next to the measured copy rate (a copy's read+write mix runs below it)
NOMINAL_HBM_GBS = 7900.0
# GB300's specified dense bf16 tensor rate (at full clock; the measured burst
# peak above comes from a cuBLAS GEMM whose clock settled lower under the
# power cap, so a kernel running at full clock can read high against it)
NOMINAL_BF16_TFLOPS = 2250.0


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


_CSRC = "exact_attention_03_gb300/csrc/"
PREFILL_SOURCES = tuple(_CSRC + f for f in ("fa_prefill_d128_sm103.cu", "sm103_ptx.cuh", "fa_internal.h",
                                            "philox.cuh"))
PREFILL_D64_SOURCES = tuple(_CSRC + f for f in ("fa_prefill_d64x1_sm103.cu", "sm103_ptx.cuh", "fa_internal.h"))
DECODE_SOURCES = tuple(_CSRC + f for f in ("fa_decode_sm103.cu", "sm103_ptx.cuh", "fa_internal.h"))
BACKWARD_SOURCES = tuple(_CSRC + f for f in ("fa_backward_sm103.cu", "sm103_ptx.cuh", "fa_internal.h",
                                             "philox.cuh"))


def measured_traffic(key, sources):
    """DRAM bytes of a kernel unit from profiles/traffic.json (ncu counters),
    or None when the kernel sources changed since the counters were taken."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            entry = json.load(f)[key]
        h = hashlib.sha256()
        for src in sources:
            with open(os.path.join(ROOT, src), "rb") as f:
                h.update(f.read())
    except Exception:
        return None
    return entry["bytes"] if h.hexdigest() == entry["src_sha256"] else None


def max_over_ranks(x: float, world: int) -> float:
    """The largest value of x over all ranks (the job's step time)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(step_flops: float, step_ms: float, world: int) -> float:
    """Whole-job TFLOPS: every rank runs the same per-GPU step (weak scaling)."""
    return world * step_flops / (step_ms * 1e-3) / 1e12


def sweep_workloads():
    from exact_attention_03_gb300.inputs import SWEEP_LENGTHS, sweep
    return [sweep(L) for L in SWEEP_LENGTHS]


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples of the SM clock and the throttle reasons, every 10 ms,
    started before the timed region; `stop(t0, t1)` keeps the samples whose
    timestamps fall in the timed region's wall-clock window (+-20 ms; the
    nearest sample if none does)."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        import threading
        self.proc = None
        self.lines = []
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(device_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "10"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True, bufsize=1)
        except Exception:
            self.proc = None
            return
        self.reader = threading.Thread(target=self._read, daemon=True)
        self.reader.start()
        # let the sampler start producing before the timed region begins
        t_end = time.time() + 5.0
        while not self.lines and time.time() < t_end and self.proc.poll() is None:
            time.sleep(0.01)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line)

    @staticmethod
    def _epoch(stamp: str):
        import datetime
        for fmt in ("%Y/%m/%d %H:%M:%S.%f", "%Y/%m/%d %H:%M:%S"):
            try:
                return datetime.datetime.strptime(stamp.strip(), fmt).timestamp()
            except ValueError:
                continue
        return None

    def stop(self, t0: float, t1: float):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.reader.join(timeout=5)
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        rows = []
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((self._epoch(parts[0]), float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        rows = [r for r in rows if r[0] is not None]
        inside = [r for r in rows if t0 - 0.02 <= r[0] <= t1 + 0.02]
        if not inside and rows:
            mid = 0.5 * (t0 + t1)
            inside = [min(rows, key=lambda r: abs(r[0] - mid))]
        reasons = sorted({n for r in inside for n, v in zip(names, r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median([r[1] for r in inside]) if inside else None,
                "sm_max_mhz": max(r[2] for r in inside) if inside else None,
                "samples": len(inside), "samples_total": len(rows),
                "window_ms": round((t1 - t0) * 1e3, 1), "reasons": reasons}


# ---------------------------------------------------------------- our arm

def _time_launches(calls, flush, reps):
    """Device time (ms) of each call, L2 flushed before each (not timed)."""
    import torch
    s = torch.cuda.current_stream()
    evs = []
    for _ in range(reps):
        for fn in calls:
            flush.zero_()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(s)
            fn()
            e1.record(s)
            evs.append((e0, e1))
    s.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


def run_ours(args, rank, world):
    import torch
    import exact_attention_03_gb300 as fa
    from exact_attention_03_gb300 import build as fa_build
    from exact_attention_03_gb300.inputs import WORKLOADS, make_inputs

    fa_build.build()
    fa.load()
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    peaks, peak_src = load_peaks()
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def check():
        st, site = fa.last_device_error()
        if st != fa.FA_OK:
            raise RuntimeError(f"device wait gave up: {st} at site {site}")

    # ---- headline: the sweep, inputs resident in HBM
    ws = sweep_workloads()
    bufs = []
    for w in ws:
        q, k, v = make_inputs(w, dev)
        o = torch.empty_like(q)
        lse = torch.empty((w.B, w.H, w.Lq), dtype=torch.float32, device=dev)
        bufs.append((w, q, k, v, o, lse))
    calls = [(lambda w=w, q=q, k=k, v=v, o=o, lse=lse:
              fa.forward(q, k, v, causal=w.causal, out=o, lse=lse)) for (w, q, k, v, o, lse) in bufs]
    _time_launches(calls, flush, args.warmup)
    check()
    clocks = ClockSampler(dev.index)   # started (and producing) before the barrier
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    w0 = time.time()
    times = _time_launches(calls, flush, args.steps)
    wall = time.perf_counter() - t0
    clk = clocks.stop(w0, time.time())
    torch.cuda.synchronize()
    check()
    n = len(calls)
    step_ms = [sum(times[i * n:(i + 1) * n]) for i in range(args.steps)]
    mean_step = sum(step_ms) / len(step_ms)
    mean_step = max_over_ranks(mean_step, world)
    step_flops = sum(w.flops for w in ws)
    value = job_throughput(step_flops, mean_step, world)
    per_len = {}
    for i, w in enumerate(ws):
        ts = [times[s * n + i] for s in range(args.steps)]
        ms = statistics.median(ts)
        tf_l = w.flops / (ms * 1e-3) / 1e12
        per_len[str(w.Lq)] = {"ms": round(ms, 5), "tflops": round(tf_l, 2),
                              "frac_bf16": round(tf_l / peaks["bf16_tflops"], 4),
                              "frac_bf16_nominal": round(tf_l / NOMINAL_BF16_TFLOPS, 4),
                              "GB/s": round(w.bytes / (ms * 1e-3) / 1e9, 1)}

    # ---- e2e: the same sweep through the host-buffer API
    host = [(w, *(t.cpu().pin_memory() for t in (q, k, v)),
             torch.empty((w.B, w.H, w.Lq, w.D), dtype=torch.bfloat16, pin_memory=True),
             torch.empty((w.B, w.H, w.Lq), dtype=torch.float32, pin_memory=True))
            for (w, q, k, v, _, _) in bufs]
    for (w, qh, kh, vh, oh, lh) in host:
        fa.forward_host(qh, kh, vh, causal=w.causal, out=oh, lse=lh)
    torch.cuda.synchronize()
    e2e_ms = []
    for _ in range(args.steps):
        s = torch.cuda.current_stream()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        flush.zero_()
        # the host-buffer copies run on the library's own streams, which do
        # not wait for `s`: let the flush finish first, so that no copy of
        # the step starts before e0
        torch.cuda.synchronize()
        e0.record(s)
        # the step's problems are queued back to back (each one's copies
        # overlap the previous one's kernels); the outputs are on the host
        # when the stream reaches e1
        for (w, qh, kh, vh, oh, lh) in host:
            fa.forward_host(qh, kh, vh, causal=w.causal, out=oh, lse=lh, sync=False)
        e1.record(s)
        s.synchronize()
        e2e_ms.append(e0.elapsed_time(e1))
    check()
    h2d = sum(t.numel() * t.element_size() for (_, qh, kh, vh, _, _) in host for t in (qh, kh, vh))
    d2h = sum(w.B * w.H * w.Lq * (w.D * 2 + 4) for w in ws)
    e2e_value = job_throughput(step_flops, max_over_ranks(statistics.mean(e2e_ms), world), world)

    result = {
        "metric": METRIC, "value": round(value, 3), "unit": "TFLOPS", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(mean_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16 q, k, v)",
        "config": {"workload": "sweep_d64: non-causal MHA B=4 H=8 D=64, Lq=Lk in 64..8192 "
                               "(one forward per length per step)",
                   "global_batch": 4 * world, "seq_len": "64..8192",
                   "l2": "flushed before every launch (256 MiB write, untimed)",
                   "parallelism": f"replicas x{world} (heads independent)"},
        "per_length": per_len,
        "gpu_launches": n * args.steps,
        "clocks": clk,
        "e2e": {"value": round(e2e_value, 3), "unit": "TFLOPS", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
    }
    prefill_ms = mean_step  # every launch of the step is the prefill kernel
    achieved = step_flops / (prefill_ms * 1e-3) / 1e12
    result["roofline"] = {"kernel": "fa_prefill_d64x1_kernel", "bound": "tensor",
                          "achieved": round(achieved, 3), "peak": peaks["bf16_tflops"],
                          "unit": "TFLOP/s", "frac": round(achieved / peaks["bf16_tflops"], 4),
                          "frac_nominal": round(achieved / NOMINAL_BF16_TFLOPS, 4),
                          "peak_source": f"{peak_src} bf16 burst",
                          "per": "one step (one launch at each of the 8 sweep lengths)",
                          "algorithmic_bytes": sum(w.bytes for w in ws),
                          "traffic": measured_traffic("fa_prefill_d64x1_kernel/sweep_d64_step",
                                                      PREFILL_D64_SOURCES)}
    del bufs, calls, host

    if rank == 0 and world == 1 and not args.no_configs:
        result["per_config"] = per_config(args, fa, flush, dev, peaks, check)
    if rank == 0 and world == 1 and not args.no_cpu:
        result["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
        if args.oracle_configs:
            result["cpu_baseline"]["per_config"] = oracle_per_config()
    return result


def per_config(args, fa, flush, dev, peaks, check):
    import torch
    from exact_attention_03_gb300.inputs import WORKLOADS, make_inputs
    out = {}
    # median of >= 20 timed launches (>= 5 for the 22 ms long-context one), 3 warm-ups
    for name, reps in (("mha_l256_d64", 20), ("causal_l8k_d128", 20),
                       ("causal_l64k_d128", 5), ("decode_l128k_d128", 20)):
        w = WORKLOADS[name]
        q, k, v = make_inputs(w, dev)
        o = torch.empty((w.B, w.H, w.Lq, w.D), dtype=torch.bfloat16, device=dev)
        lse = torch.empty((w.B, w.H, w.Lq), dtype=torch.float32, device=dev)
        call = lambda: fa.forward(q, k, v, causal=w.causal, out=o, lse=lse)
        _time_launches([call], flush, 3)
        ts = _time_launches([call], flush, reps)
        check()
        ms = statistics.median(ts)
        entry = {"B": w.B, "H": w.H, "Lq": w.Lq, "Lk": w.Lk, "D": w.D, "causal": w.causal,
                 "ms": round(ms, 5)}
        if w.Lq == 1:
            gbs = w.bytes / (ms * 1e-3) / 1e9
            tr = measured_traffic("fa_decode_split_kernel<128>/decode_l128k_d128_b1", DECODE_SOURCES)
            entry.update({"GB/s": round(gbs, 1), "frac_hbm": round(gbs / peaks["hbm_gbs"], 4),
                          "frac_hbm_nominal": round(gbs / NOMINAL_HBM_GBS, 4),
                          "launches": 2, "algorithmic_bytes": w.bytes,
                          "traffic": None if tr is None else tr * w.B})
        else:
            tf = w.flops / (ms * 1e-3) / 1e12
            tr = (measured_traffic("fa_prefill_d128_kernel/causal_l8k_d128", PREFILL_SOURCES)
                  if name == "causal_l8k_d128" else None)
            entry.update({"TFLOPS": round(tf, 2), "frac_bf16": round(tf / peaks["bf16_tflops"], 4),
                          "frac_bf16_sustained": round(tf / peaks["bf16_tflops_sustained"], 4),
                          "frac_bf16_nominal": round(tf / NOMINAL_BF16_TFLOPS, 4),
                          "GB/s": round(w.bytes / (ms * 1e-3) / 1e9, 1),
                          "launches": 1, "algorithmic_bytes": w.bytes, "traffic": tr})
        out[name] = entry
        del q, k, v, o, lse
        torch.cuda.empty_cache()
    out.update(per_config_paged(fa, flush, dev, peaks, check))
    out.update(per_config_softmax(fa, flush, dev, peaks, check))
    out.update(per_config_backward(fa, flush, dev, peaks, check))
    out.update(per_config_dropout(fa, flush, dev, peaks, check))
    return out


def per_config_backward(fa, flush, dev, peaks, check):
    """The backward pass (fa_bwd: preparation + dK/dV + dQ kernels) on the
    causal 8K D128 workload.  TFLOPS count the five products a backward pass
    needs (2.5 x the forward's flops); the kernels compute seven (S and dP
    once for dK/dV and once for dQ)."""
    import torch
    from exact_attention_03_gb300.inputs import WORKLOADS, make_inputs
    out = {}
    w = WORKLOADS["causal_l8k_d128"]
    q, k, v = make_inputs(w, dev)
    g = torch.Generator(device=dev).manual_seed(11)
    do = torch.randn(q.shape, generator=g, device=dev).to(torch.bfloat16)
    o, lse = fa.forward(q, k, v, causal=True)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    call = lambda: fa.backward(q, k, v, o, lse, do, causal=True, dq=dq, dk=dk, dv=dv)
    _time_launches([call], flush, 2)
    ts = _time_launches([call], flush, 10)
    check()
    ms = statistics.median(ts)
    flops = 2.5 * w.flops
    tf = flops / (ms * 1e-3) / 1e12
    out["backward_causal_l8k_d128"] = {"B": w.B, "H": w.H, "L": w.Lq, "D": w.D, "causal": True,
                                       "ms": round(ms, 5), "TFLOPS": round(tf, 2),
                                       "frac_bf16": round(tf / peaks["bf16_tflops"], 4),
                                       "frac_bf16_nominal": round(tf / NOMINAL_BF16_TFLOPS, 4),
                                       "launches": 3, "flops_counted": flops,
                                       "traffic": measured_traffic("fa_bwd/causal_l8k_d128", BACKWARD_SOURCES)}
    # the backward of the dropout forward (fa_bwd_dropout, p = 0.1): the same
    # products, the keep bits drawn again in both kernels
    o, lse = fa.forward_dropout(q, k, v, 0.1, 1234, 0, causal=True)
    call = lambda: fa.backward_dropout(q, k, v, o, lse, do, 0.1, 1234, 0, causal=True, dq=dq, dk=dk, dv=dv)
    _time_launches([call], flush, 2)
    ts = _time_launches([call], flush, 10)
    check()
    ms_d = statistics.median(ts)
    tf = flops / (ms_d * 1e-3) / 1e12
    out["backward_dropout_causal_l8k_d128"] = {"B": w.B, "H": w.H, "L": w.Lq, "D": w.D, "causal": True,
                                               "p_drop": 0.1, "ms": round(ms_d, 5), "TFLOPS": round(tf, 2),
                                               "frac_bf16": round(tf / peaks["bf16_tflops"], 4),
                                               "frac_bf16_nominal": round(tf / NOMINAL_BF16_TFLOPS, 4),
                                               "vs_no_dropout": round(ms_d / ms, 3),
                                               "launches": 3, "flops_counted": flops,
                                               "traffic": measured_traffic("fa_bwd_dropout/causal_l8k_d128",
                                                                           BACKWARD_SOURCES)}
    del q, k, v, do, o, lse, dq, dk, dv
    torch.cuda.empty_cache()
    return out


def per_config_dropout(fa, flush, dev, peaks, check):
    """The forward with dropout on the weights (fa_fwd_dropout, p = 0.1) on
    the causal 8K D128 workload and the D64 sweep's 8K length, next to the
    plain forward on the same inputs: TFLOPS count the same products (the
    Philox bits are extra work, not extra flops)."""
    import torch
    from exact_attention_03_gb300.inputs import WORKLOADS, Workload, make_inputs
    out = {}
    for name, w in (("dropout_causal_l8k_d128", WORKLOADS["causal_l8k_d128"]),
                    ("dropout_l8k_d64", Workload("sweep_8192", 4, 8, 8192, 8192, 64, False, seed=1))):
        q, k, v = make_inputs(w, dev)
        o = torch.empty_like(q)
        lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
        call = lambda: fa.forward_dropout(q, k, v, 0.1, 1234, 0, causal=w.causal, out=o, lse=lse)
        plain = lambda: fa.forward(q, k, v, causal=w.causal, out=o, lse=lse)
        _time_launches([call, plain], flush, 2)
        ts = _time_launches([call, plain], flush, 10)
        check()
        ms = statistics.median(ts[0::2])
        ms_plain = statistics.median(ts[1::2])
        tf = w.flops / (ms * 1e-3) / 1e12
        out[name] = {"B": w.B, "H": w.H, "L": w.Lq, "D": w.D, "causal": w.causal, "p_drop": 0.1,
                     "ms": round(ms, 5), "TFLOPS": round(tf, 2), "frac_bf16": round(tf / peaks["bf16_tflops"], 4),
                     "frac_bf16_nominal": round(tf / NOMINAL_BF16_TFLOPS, 4),
                     "ms_without_dropout": round(ms_plain, 5), "launches": 1}
        del q, k, v, o, lse
        torch.cuda.empty_cache()
    return out


def per_config_softmax(fa, flush, dev, peaks, check):
    """The two-read row softmax (fa_softmax_rows) on a 1 GiB fp32 matrix: GB/s
    over the bytes every softmax must move (x read once, y written once); the
    second read of a row comes back from L2 right after the first."""
    import torch
    out = {}
    rows, cols = 32768, 8192
    g = torch.Generator(device=dev).manual_seed(10)
    x = torch.randn(rows, cols, generator=g, device=dev) * 4
    y = torch.empty_like(x)
    lse = torch.empty(rows, dtype=torch.float32, device=dev)
    call = lambda: fa.softmax_rows(x, out=y, lse=lse)
    _time_launches([call], flush, 3)
    ts = _time_launches([call], flush, 20)
    check()
    ms = statistics.median(ts)
    nbytes = rows * cols * 4 * 2 + rows * 4
    gbs = nbytes / (ms * 1e-3) / 1e9
    out["softmax_rows_32k_x_8k"] = {"rows": rows, "cols": cols, "ms": round(ms, 5),
                                    "GB/s": round(gbs, 1), "frac_hbm": round(gbs / peaks["hbm_gbs"], 4),
                                    "frac_hbm_nominal": round(gbs / NOMINAL_HBM_GBS, 4),
                                    "launches": 1, "algorithmic_bytes": nbytes}
    del x, y, lse
    torch.cuda.empty_cache()
    return out


def per_config_paged(fa, flush, dev, peaks, check):
    """Single-query attention against the paged cache (fa_fwd_decode_paged):
    GB/s over the algorithmic bytes (every cached K and V row of every
    sequence once, q once, O and LSE once)."""
    import torch
    from exact_attention_03_gb300.inputs import PAGED_WORKLOADS, make_paged_inputs
    out = {}
    for name, reps in (("decode_paged_128k_d128", 5),):
        w = PAGED_WORKLOADS[name]
        q, kc, vc, bt, lens = make_paged_inputs(w, dev)
        o = torch.empty((w.B, w.H, w.D), dtype=torch.bfloat16, device=dev)
        lse = torch.empty((w.B, w.H), dtype=torch.float32, device=dev)
        call = lambda: fa.decode_paged(q, kc, vc, bt, lens, out=o, lse=lse)
        _time_launches([call], flush, 2)
        ts = _time_launches([call], flush, reps)
        check()
        ms = statistics.median(ts)
        total = int(lens.sum().item())
        nbytes = total * w.H * w.D * 2 * 2 + w.B * w.H * (w.D * 2 * 2 + 4)
        gbs = nbytes / (ms * 1e-3) / 1e9
        out[name] = {"B": w.B, "H": w.H, "D": w.D, "page_size": w.page_size,
                     "max_len": w.max_len, "cached_positions": total, "ms": round(ms, 5),
                     "GB/s": round(gbs, 1), "frac_hbm": round(gbs / peaks["hbm_gbs"], 4),
                     "frac_hbm_nominal": round(gbs / NOMINAL_HBM_GBS, 4),
                     "launches": 2, "algorithmic_bytes": nbytes}
        del q, kc, vc, bt, lens, o, lse
        torch.cuda.empty_cache()
    return out


# ---------------------------------------------------------------- CPU oracle

def _oracle_sample(max_seconds, per_len_rows=None, max_rounds=None):
    """Runs the oracle on a bounded sample of the sweep: round r computes head r
    (b = r // H, h = r % H) at every length, until `max_seconds` of oracle time
    or `max_rounds` rounds.  Returns (flops, seconds, description)."""
    import numpy as np
    from exact_attention_03_gb300.inputs import make_inputs
    from oracle.naive import attention_head, to_f64

    ws = sweep_workloads()
    inputs = [make_inputs(w, "cpu") for w in ws]
    flops = 0.0
    spent = 0.0
    rounds = 0
    nheads = ws[0].B * ws[0].H
    while rounds < nheads:
        b, h = divmod(rounds, ws[0].H)
        for w, (q, k, v) in zip(ws, inputs):
            qh, kh, vh = to_f64(q[b, h]), to_f64(k[b, h]), to_f64(v[b, h])
            rows = w.Lq if per_len_rows is None else min(w.Lq, per_len_rows)
            t0 = time.perf_counter()
            attention_head(qh, kh, vh, w.scale, causal=w.causal, rows=np.arange(rows))
            spent += time.perf_counter() - t0
            flops += 4.0 * rows * w.Lk * w.D
        rounds += 1
        if spent > max_seconds or (max_rounds is not None and rounds >= max_rounds):
            break
    rows_desc = "all rows" if per_len_rows is None else f"first {per_len_rows} rows"
    return flops, spent, (f"{rounds} head(s) at every sweep length L=64..8192, {rows_desc}"
                          " per head (numpy fp64, BLAS threads = all host cores)")


def oracle_per_config(seconds_each=5.0):
    """The oracle's rate on bounded samples of the other workloads (on the
    host cores, after the GPU part), all from batch entry 0: the L = 256
    config's 8 heads; whole heads of the causal 8K config; the long-context
    config's sampled rows of its first heads; whole heads of the 128K decode
    config.  Each sample stops after
    about `seconds_each` of oracle time.  Rates are over the flops of the rows
    computed (causal: the visible keys only), or the K/V bytes for decode."""
    import numpy as np
    from exact_attention_03_gb300.inputs import WORKLOADS, make_inputs, sample_rows
    from oracle.naive import attention_head, to_f64

    out = {}
    for name in ("mha_l256_d64", "causal_l8k_d128", "causal_l64k_d128", "decode_l128k_d128"):
        w = WORKLOADS[name]
        q, k, v = make_inputs(w, "cpu", batches=range(1))   # batch 0 only (bounded host memory)
        picked = sample_rows(w) if name == "causal_l64k_d128" else None
        flops = nbytes = spent = 0.0
        heads = 0
        for h in range(w.H):
            qh, kh, vh = to_f64(q[0, h]), to_f64(k[0, h]), to_f64(v[0, h])
            rows = picked[h].numpy() if picked is not None else np.arange(w.Lq)
            t0 = time.perf_counter()
            attention_head(qh, kh, vh, w.scale, causal=w.causal, rows=rows)
            spent += time.perf_counter() - t0
            keys = (rows + 1) if w.causal else np.full(rows.shape, w.Lk)
            flops += 4.0 * float(keys.sum()) * w.D
            nbytes += 4.0 * w.Lk * w.D
            heads += 1
            if spent > seconds_each:
                break
        entry = {"heads": heads, "seconds": round(spent, 2), "GFLOP/s": round(flops / spent / 1e9, 3)}
        if w.Lq == 1:
            entry["GB/s"] = round(nbytes / spent / 1e9, 3)
        out[name] = entry
    return out


def cpu_model():
    """The host CPU's model as the OS reports it (x86: 'model name'; Arm:
    implementer and part numbers), else the machine type."""
    try:
        with open("/proc/cpuinfo") as f:
            info = f.read()
        for key in ("model name", "Model name"):
            for line in info.splitlines():
                if line.startswith(key):
                    return line.split(":", 1)[1].strip()
        impl = [l.split(":", 1)[1].strip() for l in info.splitlines() if l.startswith("CPU implementer")]
        part = [l.split(":", 1)[1].strip() for l in info.splitlines() if l.startswith("CPU part")]
        if impl and part:
            return f"Arm implementer {impl[0]} part {part[0]}"
    except OSError:
        pass
    import platform
    return platform.machine()


def _oracle_l256_rate():
    """The oracle over the whole L = 256 config (B4 H8 D64, non-causal, every
    row of every head) in this process, repeated until it has run ~1 s;
    returns its rate."""
    import numpy as np
    from exact_attention_03_gb300.inputs import WORKLOADS, make_inputs
    from oracle.naive import attention_head, to_f64

    w = WORKLOADS["mha_l256_d64"]
    q, k, v = make_inputs(w, "cpu")
    spent = 0.0
    rounds = 0
    while rounds == 0 or spent < 1.0:
        for b in range(w.B):
            for h in range(w.H):
                qh, kh, vh = to_f64(q[b, h]), to_f64(k[b, h]), to_f64(v[b, h])
                t0 = time.perf_counter()
                attention_head(qh, kh, vh, w.scale, causal=w.causal, rows=np.arange(w.Lq))
                spent += time.perf_counter() - t0
        rounds += 1
    return {"GFLOP/s": round(rounds * w.flops / spent / 1e9, 3), "seconds": round(spent, 3),
            "rounds": rounds}


def oracle_l256_one_core():
    """The same on ONE host core: a child process (spawned, not forked) that
    pins itself to one CPU, with the BLAS and OpenMP thread counts set to 1
    before numpy loads."""
    cpu = min(os.sched_getaffinity(0))
    code = (f"import os; os.sched_setaffinity(0, {{{cpu}}}); import json, bench; "
            "print(json.dumps(bench._oracle_l256_rate()))")
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1",
               BLIS_NUM_THREADS="1")
    try:
        out = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True,
                             text=True, timeout=600)
        res = json.loads(out.stdout.strip().splitlines()[-1])
    except (subprocess.SubprocessError, ValueError, IndexError) as e:
        return {"error": f"{type(e).__name__}: {e}"[:200]}
    res.update({"cores": 1, "workload": "mha_l256_d64 (B4 H8 L256 D64, all rows)"})
    return res


def cpu_baseline(seconds):
    flops, spent, desc = _oracle_sample(seconds)
    return {"value": round(flops / spent / 1e12, 6), "unit": "TFLOPS",
            "cores": len(os.sched_getaffinity(0)), "cpu": cpu_model(), "kind": "oracle",
            "sample": desc,
            "seconds": round(spent, 2),
            "one_core_l256": oracle_l256_one_core()}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    step = []
    for i in range(args.warmup + args.steps):
        flops, spent, desc = _oracle_sample(1e9, per_len_rows=256, max_rounds=1)
        if i >= args.warmup:
            step.append((flops, spent))
    flops = sum(f for f, _ in step)
    secs = sum(s for _, s in step)
    value = flops / secs / 1e12
    cores = len(os.sched_getaffinity(0))
    return {"metric": METRIC, "impl": "reference", "value": round(value, 6), "unit": "TFLOPS",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(secs / len(step) * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "sweep_d64: non-causal MHA B=4 H=8 D=64, Lq=Lk in 64..8192",
                       "sample": desc},
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOPS", "cores": cores,
                             "cpu": cpu_model(), "kind": "oracle", "sample": desc},
            "e2e": {"value": round(value, 6), "unit": "TFLOPS", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def run_profile_case(args):
    """Runs one workload `reps` times with no flush or timing: the command
    the ncu captures profile.  `--profile-op` picks the operation: the
    forward, the forward with dropout, the backward or the backward with
    dropout on a prefill workload,
    the paged decode on a paged workload, or the row softmax (an 8192 x 8192
    fp32 matrix; the case name is ignored)."""
    import dataclasses
    import torch
    import exact_attention_03_gb300 as fa
    from exact_attention_03_gb300 import build as fa_build
    from exact_attention_03_gb300.inputs import PAGED_WORKLOADS, WORKLOADS, make_inputs, make_paged_inputs

    fa_build.build()
    fa.load()
    name, B = args.profile_case, 0
    if args.profile_op == "softmax":
        g = torch.Generator(device="cuda").manual_seed(10)
        x = torch.randn(8192, 8192, generator=g, device="cuda") * 4
        call = lambda: fa.softmax_rows(x)
    elif args.profile_op == "paged":
        w = PAGED_WORKLOADS[args.profile_case]
        if args.profile_batch:
            w = dataclasses.replace(w, B=args.profile_batch)
        qp, kc, vc, bt, lens = make_paged_inputs(w, "cuda")
        call = lambda: fa.decode_paged(qp, kc, vc, bt, lens)
        B = w.B
    else:
        w = WORKLOADS[args.profile_case]
        if args.profile_batch:
            w = w.with_(B=args.profile_batch)
        B = w.B
        q, k, v = make_inputs(w, "cuda")
        if args.profile_op == "forward":
            call = lambda: fa.forward(q, k, v, causal=w.causal)
        elif args.profile_op == "dropout":
            call = lambda: fa.forward_dropout(q, k, v, 0.1, 1234, 0, causal=w.causal)
        elif args.profile_op == "backward_dropout":
            g = torch.Generator(device="cuda").manual_seed(11)
            do = torch.randn(q.shape, generator=g, device="cuda").to(torch.bfloat16)
            o, lse = fa.forward_dropout(q, k, v, 0.1, 1234, 0, causal=w.causal)
            call = lambda: fa.backward_dropout(q, k, v, o, lse, do, 0.1, 1234, 0, causal=w.causal)
        else:
            g = torch.Generator(device="cuda").manual_seed(11)
            do = torch.randn(q.shape, generator=g, device="cuda").to(torch.bfloat16)
            o, lse = fa.forward(q, k, v, causal=w.causal)
            call = lambda: fa.backward(q, k, v, o, lse, do, causal=w.causal)
    torch.cuda.synchronize()
    for _ in range(args.reps):
        call()
    st, site = fa.last_device_error()
    print(json.dumps({"profile_case": name, "op": args.profile_op, "B": B, "reps": args.reps, "status": st}))
    if st != fa.FA_OK:
        sys.exit(1)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-configs", action="store_true", help="skip the per-config section")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--oracle-configs", action="store_true",
                    help="also time the oracle on bounded samples of the other workloads (~20 s)")
    ap.add_argument("--profile-case", default=None, help="run one workload (for ncu captures)")
    ap.add_argument("--profile-batch", type=int, default=0, help="batch override for --profile-case")
    ap.add_argument("--profile-op", default="forward", choices=["forward", "dropout", "backward", "backward_dropout", "paged",
                                                        "softmax"],
                    help="operation run by --profile-case")
    ap.add_argument("--reps", type=int, default=3)
    args = ap.parse_args()
    if args.profile_case:
        run_profile_case(args)
        return
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        res = run_reference(args, rank, world)
        if res is not None:
            print(json.dumps(res), flush=True)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        dist.init_process_group("nccl")
    res = run_ours(args, rank, world)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
