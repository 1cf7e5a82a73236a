"""Benchmark: TFLOP/s of fwd + dX + dW on the bf16 tensor-core tier, 7B-class layer.

One step = the four projections of a 7B-class transformer layer at M = 8192
tokens (qkv 4096->12288, o 4096->4096, up 4096->11008, down 11008->4096), each
run through bi_forward, bi_backward_dx and bi_backward_dw (f32 dW) on the
tensor-core tier: 12 GEMM launches (plus one chunk-sum launch per dW whose
last wave of tiles is split), 7.73 TFLOP of algorithmic work.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Prints one JSON line (rank 0).  `value` is whole-job TFLOP/s with inputs
resident in HBM; `e2e` is the same metric with pinned host buffers copied in and
results copied out inside the timed region; `roofline` describes the dominant
kernel; `cpu_baseline` times the CPU oracle on a bounded sample of the same
workload.  `--impl reference` times that oracle alone as the reference arm.
Under torchrun (N > 1) every rank runs an independent replica (the passes have
no exchange step); the time is the max over ranks.
"""
from __future__ import annotations

import argparse
import datetime
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "TFLOP/s fwd+dX+dW (bf16 TC tier) and fraction of dense-bf16 roofline"
WORKLOAD = "7B-class layer bf16 tensor-core tier, M=8192: qkv 4096x12288, o 4096x4096, up 4096x11008, down 11008x4096; fwd+dX+dW (f32 dW)"
# Timed regions at least this long are compared with the sustained (power-capped)
# peak; shorter ones with the burst peak.
SUSTAINED_REGION_S = 2.0
# One bounded sample of the step for the oracle, used by both the reference
# arm and the cpu_baseline of our arm (the same rows, columns and seeds).
SAMPLE_ROWS, SAMPLE_COLS = 256, 64
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--only", default=None, help="restrict the step to one projection (profiling case)")
    ap.add_argument("--profile-case", default=None, choices=["grouped", "f16-edge", "gpt2"],
                    help="run one secondary workload's calls four times and exit (a case for profilers)")
    ap.add_argument("--oracle-sample", default=f"{SAMPLE_ROWS},{SAMPLE_COLS}",
                    help="rows,cols of the oracle's sample per projection (smaller for host-only checks)")
    return ap.parse_args()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return FALLBACK_PEAKS, "fallback"


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples (every 50 ms) with their timestamps; started before the
    warm-up so that it is producing when the timed region begins, and
    summarised over the samples inside the region's wall-clock window."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0=None, t1=None):
        """Median SM clock, max clock and throttle reasons over the samples whose
        timestamps lie in [t0, t1] (epoch seconds); without one there, the first
        sample after t0."""
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        rows = []
        for ln in list(self.lines):
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(parts[1]), float(parts[2]),
                             {nm for nm, v in zip(names, parts[5:9]) if v.lower().startswith("active")}))
            except ValueError:
                continue
        if not rows:
            return None
        inside = [r for r in rows if t0 is None or t0 <= r[0] <= t1]
        where = "inside the timed region"
        if not inside:
            after = [r for r in rows if r[0] >= t0]
            inside = after[:1] if after else rows[-1:]
            where = "first sample after the timed region began (none inside it)"
        reasons = set().union(*(r[3] for r in inside))
        return {"sm_mhz": statistics.median(r[1] for r in inside), "sm_max_mhz": inside[-1][2],
                "reasons": sorted(reasons), "samples": len(inside), "window": where}


# ---------------------------------------------------------------- workload

ONLY = None


def projections():
    from deterministic_invariant_gemm_fixed_gb300 import synth
    projs = [p for p in synth.SEVEN_B if ONLY is None or p[0] == ONLY]
    return projs, synth.SEVEN_B_M


def max_over_ranks(seconds, dist, device):
    """The slowest rank's time (all ranks get it); `dist` None on one process."""
    if dist is None:
        return seconds
    import torch
    t = torch.tensor([seconds], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(flops_per_step, steps, world, seconds):
    """Whole-job TFLOP/s: every rank runs its own replica of the step."""
    return world * flops_per_step * steps / seconds / 1e12


def step_flops():
    projs, m = projections()
    return sum(3 * 2.0 * m * k * n for _, k, n in projs)


def make_inputs(device):
    """Per projection: X [M,K], W [K,N], dY [M,N] (bf16) and outputs Y, dX, dW (f32)."""
    import torch
    from deterministic_invariant_gemm_fixed_gb300 import synth
    projs, m = projections()
    bufs = []
    for i, (name, k, n) in enumerate(projs):
        x, w, dy, _ = synth.dense_inputs(m, k, n, "bf16", x=("normal", 1.0), w=("normal", 0.02),
                                         dy=("normal", 1.0), b=None, seed_offset=10 * i)
        bufs.append(dict(name=name, k=k, n=n, x_h=x, w_h=w, dy_h=dy,
                         x=x.to(device), w=w.to(device), dy=dy.to(device),
                         y=torch.empty(m, n, dtype=torch.bfloat16, device=device),
                         dx=torch.empty(m, k, dtype=torch.bfloat16, device=device),
                         dw=torch.empty(k, n, dtype=torch.float32, device=device)))
    return bufs, m


def run_step(eng, bufs, m, stream, events=None):
    """Enqueue one step (12 calls).  events: list to append (pass, start, end)."""
    import torch
    for b in bufs:
        k, n = b["k"], b["n"]
        for pas in ("fwd", "dx", "dw"):
            if events is not None:
                e0 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
            if pas == "fwd":
                eng.forward(b["y"], b["x"], b["w"], None, m, k, n, "bf16", stream, 1)
                fl = 2.0 * m * k * n
            elif pas == "dx":
                eng.backward_dx(b["dx"], b["dy"], b["w"], m, k, n, "bf16", stream, 1)
                fl = 2.0 * m * k * n
            else:
                eng.backward_dw(b["dw"], 1, b["x"], b["dy"], m, k, n, "bf16", stream, 1)
                fl = 2.0 * m * k * n
            if events is not None:
                e1 = torch.cuda.Event(enable_timing=True)
                e1.record(stream)
                events.append((pas, b["name"], fl, e0, e1))


# ---------------------------------------------------------------- CPU oracle sample

_HOST_INPUTS = {}


def oracle_sample(rows=SAMPLE_ROWS, cols=SAMPLE_COLS, seed=0):
    """Time the oracle on a bounded sample of the step: `rows` rows of Y and dX
    and `cols` columns of dW per projection (each a complete set of outputs of
    the same definition).  Returns (seconds, algorithmic flops of the sample,
    threads used, description)."""
    import numpy as np
    import oracle
    from deterministic_invariant_gemm_fixed_gb300 import synth
    projs, m = projections()
    rng = np.random.default_rng(seed)
    total_fl, total_t = 0.0, 0.0
    for i, (name, k, n) in enumerate(projs):
        if name not in _HOST_INPUTS:
            x, w, dy, _ = synth.dense_inputs(m, k, n, "bf16", x=("normal", 1.0), w=("normal", 0.02),
                                             dy=("normal", 1.0), b=None, seed_offset=10 * i)
            _HOST_INPUTS[name] = (synth.to_np(x), synth.to_np(w), synth.to_np(dy))
        xn, wn, dyn = _HOST_INPUTS[name]
        r = np.sort(rng.choice(m, size=rows, replace=False))
        c = np.sort(rng.choice(n, size=cols, replace=False))
        t0 = time.perf_counter()
        oracle.forward(xn, wn, None, m, k, n, "bf16", rows=r)
        oracle.backward_dx(dyn, wn, m, k, n, "bf16", rows=r)
        oracle.backward_dw(xn, dyn, m, k, n, "bf16", dw_f32=True, cols=c)
        total_t += time.perf_counter() - t0
        total_fl += 2.0 * rows * k * n * 2 + 2.0 * m * k * cols
    desc = (f"per projection: {rows} rows of Y and dX and {cols} columns of dW (full M=8192 "
            f"reduction) of the same workload, rows and columns drawn per step; {total_fl / 1e9:.1f} GFLOP")
    return total_t, total_fl, oracle.num_threads(), desc


def cpu_entry(flops, seconds, sample):
    """A cpu_baseline record: the oracle as it stands on the host cores."""
    import oracle
    return {"value": flops / seconds / 1e12, "unit": "TFLOP/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": sample, "seconds": seconds}


def timed_oracle(fn):
    t0 = time.perf_counter()
    fn()
    return time.perf_counter() - t0


PAIR_BEGIN = "// ---------------------------------------------------------------- CTA-pair kernel"
PAIR_END = "// ---------------------------------------------------------------- dW chunk sum"


def pair_kernel_sha():
    """sha256 prefix of the CTA-pair kernel's source text (the dense passes)."""
    src = open(os.path.join(ROOT, "deterministic_invariant_gemm_fixed_gb300", "csrc", "tc.cu")).read()
    i, j = src.find(PAIR_BEGIN), src.find(PAIR_END)
    return hashlib.sha256(src[i:j].encode()).hexdigest()[:16]


def traffic_from_profiles(kernel_tag):
    """DRAM bytes per launch recorded by an ncu capture summary under profiles/,
    valid only while the kernel's source is unchanged (see pair_kernel_sha)."""
    sha = pair_kernel_sha()
    pdir = os.path.join(ROOT, "profiles")
    if not os.path.isdir(pdir):
        return None
    for fn in sorted(os.listdir(pdir)):
        if not fn.endswith((".md", ".txt")):
            continue
        for line in open(os.path.join(pdir, fn)):
            mo = re.match(r"^bench-traffic:\s*(\{.*\})\s*$", line.strip())
            if not mo:
                continue
            d = json.loads(mo.group(1))
            if d.get("kernel") == kernel_tag and d.get("pair_kernel_sha256_16") == sha:
                return float(d["bytes_per_launch"])
    return None


# ---------------------------------------------------------------- secondary figures

def library_peaks(n=8192, reps=10):
    """Dense library matmuls on this GPU, measured the way the bf16 denominator
    is (n^3 problems, best of `reps`, CUDA events): bf16, tf32 (f32 operands,
    TF32 tensor-core math) and fp8 e4m3 (scaled matmul, bf16 out).  These are
    the denominators of the 3xTF32 and FP8 fractions."""
    import torch
    out = {"how": f"torch {torch.__version__}: {n}^3 (2*n^3 flop), best of {reps}, CUDA events"}

    def best(fn):
        for _ in range(3):
            fn()
        ts = []
        for _ in range(reps):
            e0 = torch.cuda.Event(enable_timing=True); e1 = torch.cuda.Event(enable_timing=True)
            e0.record(); fn(); e1.record(); e1.synchronize()
            ts.append(e0.elapsed_time(e1) / 1e3)
        return 2.0 * n ** 3 / min(ts) / 1e12

    g = torch.Generator(device="cuda").manual_seed(7)
    a = torch.randn(n, n, device="cuda", generator=g)
    b = torch.randn(n, n, device="cuda", generator=g)
    a16, b16 = a.bfloat16(), b.bfloat16()
    out["bf16_tflops"] = best(lambda: torch.matmul(a16, b16))
    prev = torch.get_float32_matmul_precision()
    try:
        torch.set_float32_matmul_precision("high")  # TF32 tensor-core math for f32 operands
        out["tf32_tflops"] = best(lambda: torch.matmul(a, b))
    finally:
        torch.set_float32_matmul_precision(prev)
    try:
        a8 = (a * 0.5).to(torch.float8_e4m3fn)
        b8 = (b * 0.5).to(torch.float8_e4m3fn)  # row-major [n, n]; b8.t() is the column-major operand
        one = torch.ones((), device="cuda")
        out["fp8_tflops"] = best(lambda: torch._scaled_mm(a8, b8.t(), scale_a=one, scale_b=one,
                                                          out_dtype=torch.bfloat16))
    except (RuntimeError, AttributeError, TypeError) as exc:  # a torch build without the scaled matmul
        out["fp8_tflops"] = None
        out["fp8_error"] = str(exc)[:200]
    del a, b, a16, b16
    torch.cuda.empty_cache()
    return out


def timed_oracle_min(fn, min_s=0.3):
    """Seconds per call of fn, repeated until at least min_s has elapsed (tiny
    workloads would otherwise time the call overhead of one run)."""
    calls, t = 0, 0.0
    while t < min_s:
        t += timed_oracle(fn)
        calls += 1
    return t / calls


def secondary(eng, stream, cpu=True, reps=5):
    """The other named workloads, each timed on the GPU and, with cpu, beside
    the oracle timed on the host cores on the same workload (full size where
    that takes seconds, else a stated sample)."""
    import torch
    import numpy as np
    from deterministic_invariant_gemm_fixed_gb300 import synth
    if cpu:
        import oracle
    out = {}
    libpk = library_peaks()
    out["library_peaks"] = libpk

    def timeit(fn):
        for _ in range(2):
            fn()
        e0 = torch.cuda.Event(enable_timing=True); e1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / 1e3 / reps

    props = torch.cuda.get_device_properties(0)
    ffma_peak = props.multi_processor_count * 128 * 2 * 2070e6 / 1e12  # FP32 FMA lanes x 2 flop x max SM clock

    # linear f32 M=64 K=256 N=512 on the scalar tier (fwd with bias + dX + f32 dW)
    c = synth.LINEAR_F32
    m, k, n = c["m"], c["k"], c["n"]
    x, w, dy, b = synth.dense_inputs(m, k, n, "f32", x=c["x"], w=c["w"], dy=c["dy"], b=c["b"])
    X, W, DY, B = x.cuda(), w.cuda(), dy.cuda(), b.cuda()
    Y, DX, DW = torch.empty(m, n, device="cuda"), torch.empty(m, k, device="cuda"), torch.empty(k, n, device="cuda")

    def lin_step():
        eng.forward(Y, X, W, B, m, k, n, "f32", stream, 0)
        eng.backward_dx(DX, DY, W, m, k, n, "f32", stream, 0)
        eng.backward_dw(DW, 1, X, DY, m, k, n, "f32", stream, 0)
    fl = 3 * 2.0 * m * k * n
    t = timeit(lin_step)
    rec = {"workload": c["name"] + " fwd+dX+dW (scalar tier)", "tflops": fl / t / 1e12, "us": t * 1e6,
           "ffma_peak_tflops": ffma_peak, "frac_of_ffma_peak": fl / t / 1e12 / ffma_peak}
    if cpu:
        xn, wn, dyn, bn = (synth.to_np(v) for v in (x, w, dy, b))
        rec["cpu_baseline"] = cpu_entry(fl, timed_oracle_min(lambda: (
            oracle.forward(xn, wn, bn, m, k, n, "f32"), oracle.backward_dx(dyn, wn, m, k, n, "f32"),
            oracle.backward_dw(xn, dyn, m, k, n, "f32", dw_f32=True))), "the full workload")
    out["scalar_linear_f32"] = rec
    del X, W, DY, B, Y, DX, DW

    # grouped bf16 M=16384 K=2048 E=8 N=1408, tensor-core tier
    c = synth.GROUPED
    m, k, n, e = c["m"], c["k"], c["n"], c["e"]
    x, w, dy, ids = synth.grouped_inputs(m, k, n, e, "bf16", pad_frac=c["pad_frac"])
    ids_np = synth.to_np(ids)
    valid = int((ids_np < e).sum())
    X, W, DY = x.cuda(), w.cuda(), dy.cuda()
    I = torch.from_numpy(ids_np.astype(np.int32)).cuda()
    Y = torch.empty(m, n, dtype=torch.bfloat16, device="cuda")
    DX = torch.empty(m, k, dtype=torch.bfloat16, device="cuda")
    DWg = torch.empty(e, n, k, dtype=torch.float32, device="cuda")
    fl = 2.0 * valid * n * k
    t_f = timeit(lambda: eng.grouped_forward(Y, X, W, I, m, k, n, e, "bf16", stream, 1))
    t_b = timeit(lambda: eng.grouped_backward(DX, DWg, X, W, DY, I, m, k, n, e, "bf16", stream, 1))
    rec = {"workload": c["name"], "fwd_tflops": fl / t_f / 1e12, "bwd_tflops": 2 * fl / t_b / 1e12,
           "fwd_ms": t_f * 1e3, "bwd_ms": t_b * 1e3, "tflops": 3 * fl / (t_f + t_b) / 1e12}
    if cpu:
        xn, wn, dyn = (synth.to_np(v) for v in (x, w, dy))
        rec["cpu_baseline"] = cpu_entry(3 * fl, timed_oracle(lambda: (
            oracle.grouped_forward(xn, wn, ids_np, m, k, n, e, "bf16"),
            oracle.grouped_dinput(wn, dyn, ids_np, m, k, n, e, "bf16"),
            oracle.grouped_dweights(xn, dyn, ids_np, m, k, n, e, "bf16"))),
            "the full workload: forward, dinput and f32 dweights (value against the GPU's fwd+bwd "
            "'tflops')")
    out["grouped_tc"] = rec
    # the same rows already grouped by the caller (segmented entry points, tensor cores)
    order = np.argsort(np.minimum(ids_np, e), kind="stable")
    counts = np.bincount(np.minimum(ids_np, e), minlength=e + 1)[:e]
    offs = torch.from_numpy(np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)).cuda()
    Xs, DYs = X[torch.from_numpy(order).cuda()].contiguous(), DY[torch.from_numpy(order).cuda()].contiguous()
    t_sf = timeit(lambda: eng.grouped_forward_segmented(Y, Xs, W, offs, m, k, n, e, "bf16", stream, 1))
    t_sb = timeit(lambda: eng.grouped_backward_segmented(DX, DWg, Xs, W, DYs, offs, m, k, n, e, "bf16", stream, 1))
    out["grouped_segmented_tc"] = {"workload": c["name"] + " (rows pre-grouped)", "fwd_tflops": fl / t_sf / 1e12,
                                   "bwd_tflops": 2 * fl / t_sb / 1e12, "fwd_ms": t_sf * 1e3, "bwd_ms": t_sb * 1e3}
    del Xs, DYs
    del X, W, DY, Y, DX, DWg

    # GPT-2-small MLP up-projection bf16 4096x768x3072, both tiers
    g = synth.GPT2_UP
    m, k, n = g["m"], g["k"], g["n"]
    x, w, dy, b = synth.dense_inputs(m, k, n, "bf16", x=g["x"], w=g["w"], dy=g["dy"], b=g["b"])
    X, W, DY, B = x.cuda(), w.cuda(), dy.cuda(), b.cuda()
    Y = torch.empty(m, n, dtype=torch.bfloat16, device="cuda")
    DX = torch.empty(m, k, dtype=torch.bfloat16, device="cuda")
    DW = torch.empty(k, n, dtype=torch.float32, device="cuda")

    def scal(tc):
        eng.forward(Y, X, W, B, m, k, n, "bf16", stream, tc)
        eng.backward_dx(DX, DY, W, m, k, n, "bf16", stream, tc)
        eng.backward_dw(DW, 1, X, DY, m, k, n, "bf16", stream, tc)
    fl = 3 * 2.0 * m * k * n
    t_s = timeit(lambda: scal(0))
    t_t = timeit(lambda: scal(1))
    cpu_g = None
    if cpu:
        xn, wn, dyn, bn = (synth.to_np(v) for v in (x, w, dy, b))
        cpu_g = cpu_entry(fl, timed_oracle(lambda: (
            oracle.forward(xn, wn, bn, m, k, n, "bf16"), oracle.backward_dx(dyn, wn, m, k, n, "bf16"),
            oracle.backward_dw(xn, dyn, m, k, n, "bf16", dw_f32=True))), "the full workload")
    out["scalar_gpt2_up"] = {"workload": g["name"], "tflops": fl / t_s / 1e12, "us": t_s * 1e6,
                             "ffma_peak_tflops": ffma_peak, "frac_of_ffma_peak": fl / t_s / 1e12 / ffma_peak,
                             "cpu_baseline": cpu_g}
    pk, _ = peaks()
    burst = float(pk.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    out["tc_gpt2_up"] = {"workload": g["name"], "tflops": fl / t_t / 1e12, "us": t_t * 1e6,
                         "frac_of_bf16_burst": fl / t_t / 1e12 / burst, "cpu_baseline": cpu_g}
    del X, W, DY, B, Y, DX, DW

    # bias gradient of the qkv projection: column sums of dY [8192, 12288] bf16 (HBM-bound)
    gh = synth.normal((8192, 12288), 1.0, "bf16", 60)
    g = gh.cuda()
    db = torch.empty(12288, dtype=torch.bfloat16, device="cuda")
    t_bg = timeit(lambda: eng.bias_grad(db, 0, g, 8192, 12288, "bf16", stream))
    rec = {"workload": "bf16 dY 8192x12288 column sums", "gbs": (g.nbytes + db.nbytes) / t_bg / 1e9,
           "us": t_bg * 1e6, "frac_of_hbm": (g.nbytes + db.nbytes) / t_bg / 1e9 / float(pk.get("hbm_gbs", 6800.0))}
    if cpu:
        gn = synth.to_np(gh)
        ts = timed_oracle(lambda: oracle.bias_grad(gn, 8192, 12288, "bf16"))
        rec["cpu_baseline"] = {"value": (g.nbytes + db.nbytes) / ts / 1e9, "unit": "GB/s",
                               "cores": oracle.num_threads(), "kind": "oracle", "sample": "the full workload",
                               "seconds": ts}
    out["bias_grad"] = rec
    del g, gh

    # FP8 e4m3 per-tensor-scaled linear on the qkv projection, as one path: quantize
    # X, W (forward) and dY (backward) from bf16 with the caller's scales, then
    # the scaled forward, dX and dW (f32); the quantize launches are timed too
    m, k, n = synth.SEVEN_B_M, 4096, 12288
    xh, wh, gh, _ = synth.dense_inputs(m, k, n, "bf16", x=("normal", 1.0), w=("normal", 0.02),
                                       dy=("normal", 1.0), b=None, seed_offset=70)
    X8, W8, G8 = xh.cuda(), wh.cuda(), gh.cuda()
    xq = torch.empty(m, k, dtype=torch.uint8, device="cuda")
    wq = torch.empty(k, n, dtype=torch.uint8, device="cuda")
    gq = torch.empty(m, n, dtype=torch.uint8, device="cuda")
    amax = torch.empty(3, dtype=torch.float32, device="cuda")
    # per-tensor scales from the inputs' maxima (448 / amax), as a caller would hold them
    sc = torch.tensor([X8.abs().max().item(), W8.abs().max().item(), G8.abs().max().item()],
                      dtype=torch.float32) / 448.0
    scale = sc.cuda()
    scale_inv = (1.0 / sc).cuda()
    y8 = torch.empty(m, n, dtype=torch.bfloat16, device="cuda")
    dx8 = torch.empty(m, k, dtype=torch.bfloat16, device="cuda")
    dw8 = torch.empty(k, n, dtype=torch.float32, device="cuda")

    def fp8_step():
        eng.fp8_quantize(xq, amax[0:1], X8, scale_inv[0:1], m * k, "bf16", stream)
        eng.fp8_quantize(wq, amax[1:2], W8, scale_inv[1:2], k * n, "bf16", stream)
        eng.fp8_forward(y8, xq, wq, None, scale[0:1], scale[1:2], m, k, n, "bf16", stream)
        eng.fp8_quantize(gq, amax[2:3], G8, scale_inv[2:3], m * n, "bf16", stream)
        eng.fp8_backward_dx(dx8, gq, wq, scale[2:3], scale[1:2], m, k, n, "bf16", stream)
        eng.fp8_backward_dw(dw8, xq, gq, scale[0:1], scale[2:3], m, k, n, "f32", stream)
    t8 = timeit(fp8_step)
    fl = 3 * 2.0 * m * k * n
    fp8_peak = libpk.get("fp8_tflops")
    src = "measured (library_peaks.fp8_tflops)"
    if not fp8_peak:
        fp8_peak = 2.0 * burst
        src = "nominal fp8:bf16 ratio 2 x the measured bf16 burst peak (library fp8 matmul unavailable)"
    rec = {"workload": "e4m3 qkv 8192x4096x12288: quantize X, W, dY from bf16 + fwd + dX + f32 dW",
           "tflops": fl / t8 / 1e12, "ms": t8 * 1e3, "peak_tflops": fp8_peak, "peak_source": src,
           "frac": fl / t8 / 1e12 / fp8_peak}
    if cpu:
        rows = np.sort(np.random.default_rng(11).choice(m, size=SAMPLE_ROWS, replace=False))
        xn, wn, gn = synth.to_np(xh), synth.to_np(wh), synth.to_np(gh)
        sch = sc.numpy()

        def fp8_oracle():
            wq_o, _ = oracle.fp8_quantize(wn, "bf16", 1.0 / sch[1])
            xq_o, _ = oracle.fp8_quantize(np.ascontiguousarray(xn[rows]), "bf16", 1.0 / sch[0])
            gq_o, _ = oracle.fp8_quantize(np.ascontiguousarray(gn[rows]), "bf16", 1.0 / sch[2])
            oracle.fp8_forward(xq_o, wq_o, None, sch[0], sch[1], len(rows), k, n, "bf16")
            oracle.fp8_backward_dx(gq_o, wq_o, sch[2], sch[1], len(rows), k, n, "bf16")
        ts = timed_oracle(fp8_oracle)
        rec["cpu_baseline"] = cpu_entry(2 * 2.0 * len(rows) * k * n, ts,
                                        f"{len(rows)} rows of Y and dX, with the quantizing of W and of those "
                                        "rows of X and dY (no dW columns)")
    out["fp8_qkv"] = rec
    del X8, W8, G8, xq, wq, gq, y8, dx8, dw8

    # f32 operands on the tensor cores (3xTF32: split kernels + three tf32 MMAs per
    # contraction step), the o-projection shape 8192x4096x4096 in f32
    m, k, n = synth.SEVEN_B_M, 4096, 4096
    x, w, dy, _ = synth.dense_inputs(m, k, n, "f32", b=None)
    X, W, DY = x.cuda(), w.cuda(), dy.cuda()
    Yf = torch.empty(m, n, device="cuda")
    DXf = torch.empty(m, k, device="cuda")
    DWf = torch.empty(k, n, device="cuda")

    def tf32_step():
        eng.forward(Yf, X, W, None, m, k, n, "f32", stream, 1)
        eng.backward_dx(DXf, DY, W, m, k, n, "f32", stream, 1)
        eng.backward_dw(DWf, 1, X, DY, m, k, n, "f32", stream, 1)
    t32 = timeit(tf32_step)
    v32 = 3 * 2.0 * m * k * n / t32 / 1e12
    tf32_peak = libpk.get("tf32_tflops")
    rec = {"workload": "f32 o-projection 8192x4096x4096 fwd+dX+dW, 3xTF32", "tflops": v32, "ms": t32 * 1e3,
           "ceiling_tflops": tf32_peak / 3, "frac": v32 / (tf32_peak / 3),
           "ceiling_source": "measured library tf32 matmul (library_peaks.tf32_tflops) / 3 MMAs per product"}
    if cpu:
        xn, wn, dyn = (synth.to_np(v) for v in (x, w, dy))
        rg = np.random.default_rng(12)
        rows = np.sort(rg.choice(m, size=SAMPLE_ROWS, replace=False))
        cols = np.sort(rg.choice(n, size=SAMPLE_COLS, replace=False))
        ts = timed_oracle(lambda: (oracle.forward(xn, wn, None, m, k, n, "f32", rows=rows),
                                   oracle.backward_dx(dyn, wn, m, k, n, "f32", rows=rows),
                                   oracle.backward_dw(xn, dyn, m, k, n, "f32", dw_f32=True, cols=cols)))
        rec["cpu_baseline"] = cpu_entry(2 * 2.0 * len(rows) * k * n + 2.0 * m * k * len(cols), ts,
                                        f"{len(rows)} rows of Y and dX and {len(cols)} columns of dW")
    out["tf32x3_f32_o"] = rec
    del X, W, DY, Yf, DXf, DWf, x, w, dy

    # f16 edge shapes: N = 48 (the scalar fallback: an output dimension < 64) and
    # the ragged 1000^3 on the tensor-core tier; fwd + dX + dW (f32 dW) each
    for name, m, k, n in synth.F16_EDGE[:2]:
        x, w, dy, b = synth.dense_inputs(m, k, n, "f16", x=("uniform", 1.0), w=("uniform", 1.0),
                                         dy=("uniform", 1.0), b=("uniform", 1.0))
        X, W, DY, B = x.cuda(), w.cuda(), dy.cuda(), b.cuda()
        Y = torch.empty(m, n, dtype=torch.float16, device="cuda")
        DX = torch.empty(m, k, dtype=torch.float16, device="cuda")
        DW = torch.empty(k, n, dtype=torch.float32, device="cuda")
        tc = 0 if n < 64 else 1

        def edge_step():
            eng.forward(Y, X, W, B, m, k, n, "f16", stream, tc)
            eng.backward_dx(DX, DY, W, m, k, n, "f16", stream, tc)
            eng.backward_dw(DW, 1, X, DY, m, k, n, "f16", stream, tc)
        te = timeit(edge_step)
        fl = 3 * 2.0 * m * k * n
        moved = 2 * (X.nbytes + W.nbytes + DY.nbytes) + Y.nbytes + DX.nbytes + DW.nbytes  # each pass reads two operands
        rec = {"workload": f"f16 {m}x{k}x{n} fwd+dX+dW ({'scalar' if tc == 0 else 'tensor-core'} tier)",
               "tflops": fl / te / 1e12, "gbs": moved / te / 1e9, "us": te * 1e6}
        if tc == 0:
            rec["frac_of_ffma_peak"] = fl / te / 1e12 / ffma_peak
        else:
            rec["frac_of_bf16_burst"] = fl / te / 1e12 / burst
        if cpu:
            xn, wn, dyn, bn = (synth.to_np(v) for v in (x, w, dy, b))
            rec["cpu_baseline"] = cpu_entry(fl, timed_oracle_min(lambda: (
                oracle.forward(xn, wn, bn, m, k, n, "f16"), oracle.backward_dx(dyn, wn, m, k, n, "f16"),
                oracle.backward_dw(xn, dyn, m, k, n, "f16", dw_f32=True))), "the full workload")
        out["f16_" + name] = rec
        del X, W, DY, B, Y, DX, DW

    # GEMV f16 1x4096x4096 (HBM-bound): W rotated over 8 copies > L2
    k = n = 4096
    whs = [synth.uniform((k, n), -1, 1, "f16", 100 + i) for i in range(8)]
    ws = [v.cuda() for v in whs]
    xh = synth.uniform((1, k), -1, 1, "f16", 99)
    xv = xh.cuda()
    yv = torch.empty(1, n, dtype=torch.float16, device="cuda")
    state = {"i": 0}
    gemv_bytes = k * n * 2 + k * 2 + n * 2
    hbm = float(pk.get("hbm_gbs", 6800.0))
    cpu_v = None
    if cpu:
        xn, wn = synth.to_np(xh), synth.to_np(whs[0])
        ts = timed_oracle_min(lambda: oracle.forward(xn, wn, None, 1, k, n, "f16"))
        cpu_v = {"value": gemv_bytes / ts / 1e9, "unit": "GB/s", "cores": oracle.num_threads(), "kind": "oracle",
                 "sample": "the full workload", "seconds": ts}

    def gemv():
        eng.forward(yv, xv, ws[state["i"] % 8], None, 1, k, n, "f16", stream, 1)
        state["i"] += 1
    t_g = timeit(gemv)
    out["gemv_tc_f16"] = {"workload": "f16 1x4096x4096", "gbs": gemv_bytes / t_g / 1e9, "us": t_g * 1e6,
                          "frac_of_hbm": gemv_bytes / t_g / 1e9 / hbm, "cpu_baseline": cpu_v}

    # the same GEMV on the scalar tier (one lane per output column, bit-exact chains)
    def gemv_scalar():
        eng.forward(yv, xv, ws[state["i"] % 8], None, 1, k, n, "f16", stream, 0)
        state["i"] += 1
    t_gs = timeit(gemv_scalar)
    out["gemv_scalar_f16"] = {"workload": "f16 1x4096x4096 (scalar tier)", "gbs": gemv_bytes / t_gs / 1e9,
                              "us": t_gs * 1e6, "frac_of_hbm": gemv_bytes / t_gs / 1e9 / hbm,
                              "chain_bound_us": k * 4 / 2.07e3, "cpu_baseline": cpu_v}
    return out


def profile_case(name, reps=4):
    """The calls one secondary figure times, `reps` times each, on cuda:0."""
    import torch
    import numpy as np
    import deterministic_invariant_gemm_fixed_gb300 as bi
    from deterministic_invariant_gemm_fixed_gb300 import synth
    eng = bi.Engine(0)
    stream = torch.cuda.current_stream()
    if name == "grouped":
        c = synth.GROUPED
        m, k, n, e = c["m"], c["k"], c["n"], c["e"]
        x, w, dy, ids = synth.grouped_inputs(m, k, n, e, "bf16", pad_frac=c["pad_frac"])
        X, W, DY = x.cuda(), w.cuda(), dy.cuda()
        I = torch.from_numpy(synth.to_np(ids).astype(np.int32)).cuda()
        Y = torch.empty(m, n, dtype=torch.bfloat16, device="cuda")
        DX = torch.empty(m, k, dtype=torch.bfloat16, device="cuda")
        DW = torch.empty(e, n, k, dtype=torch.float32, device="cuda")
        for _ in range(reps):
            eng.grouped_forward(Y, X, W, I, m, k, n, e, "bf16", stream, 1)
            eng.grouped_backward(DX, DW, X, W, DY, I, m, k, n, e, "bf16", stream, 1)
    elif name == "gpt2":  # the GPT-2-small MLP up-projection on the tensor-core tier
        g = synth.GPT2_UP
        m, k, n = g["m"], g["k"], g["n"]
        x, w, dy, b = synth.dense_inputs(m, k, n, "bf16", x=g["x"], w=g["w"], dy=g["dy"], b=g["b"])
        X, W, DY, B = x.cuda(), w.cuda(), dy.cuda(), b.cuda()
        Y = torch.empty(m, n, dtype=torch.bfloat16, device="cuda")
        DX = torch.empty(m, k, dtype=torch.bfloat16, device="cuda")
        DW = torch.empty(k, n, dtype=torch.float32, device="cuda")
        for _ in range(reps):
            eng.forward(Y, X, W, B, m, k, n, "bf16", stream, 1)
            eng.backward_dx(DX, DY, W, m, k, n, "bf16", stream, 1)
            eng.backward_dw(DW, 1, X, DY, m, k, n, "bf16", stream, 1)
    else:  # the f16 edge shapes: N = 48 on the scalar tier, the ragged 1000^3 and the GEMV
        for nm, m, k, n in synth.F16_EDGE:
            x, w, dy, b = synth.dense_inputs(m, k, n, "f16", x=("uniform", 1.0), w=("uniform", 1.0),
                                             dy=("uniform", 1.0), b=("uniform", 1.0))
            X, W, DY, B = x.cuda(), w.cuda(), dy.cuda(), b.cuda()
            Y = torch.empty(m, n, dtype=torch.float16, device="cuda")
            DX = torch.empty(m, k, dtype=torch.float16, device="cuda")
            DW = torch.empty(k, n, dtype=torch.float32, device="cuda")
            for tc in ((0,) if n < 64 else ((1, 0) if m == 1 else (1,))):
                for _ in range(reps):
                    eng.forward(Y, X, W, B, m, k, n, "f16", stream, tc)
                    if m > 1:
                        eng.backward_dx(DX, DY, W, m, k, n, "f16", stream, tc)
                        eng.backward_dw(DW, 1, X, DY, m, k, n, "f16", stream, tc)
    torch.cuda.synchronize()
    eng.check(stream)
    eng.close()


# ---------------------------------------------------------------- arms

def reference_arm(args, rank, world):
    if rank != 0:
        return
    secs, fl, cores, desc = [], 0.0, 1, ""
    rows, cols = (int(v) for v in args.oracle_sample.split(","))
    for s in range(args.warmup + args.steps):
        t, f, cores, desc = oracle_sample(rows=rows, cols=cols, seed=s)
        if s >= args.warmup:
            secs.append(t)
            fl = f
    per = statistics.mean(secs)
    v = fl / per / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": per * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32-accumulate bf16",
            "data": "synthetic", "config": {"workload": WORKLOAD, "sample": desc},
            "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": desc},
            "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def our_arm(args, rank, world):
    import torch
    import deterministic_invariant_gemm_fixed_gb300 as bi
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    eng = bi.Engine(local)
    stream = torch.cuda.Stream()
    bufs, m = make_inputs("cuda")
    fl_step = step_flops()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:  # producing samples before the timed region begins
        with torch.cuda.stream(stream):
            for _ in range(max(3, args.warmup)):
                run_step(eng, bufs, m, stream)
        eng.check(stream)

        # ---- device-resident timing
        events = []
        launches0 = eng.launches()
        barrier()
        w0 = time.time()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for _ in range(args.steps):
            run_step(eng, bufs, m, stream, events)
        t1.record(stream)
        t1.synchronize()
        w1 = time.time()
        barrier()
        time.sleep(0.12)  # the sample that follows the region's end has been read
    clocks = clk.summary(w0, w1)
    launches = eng.launches() - launches0
    eng.check(stream)
    elapsed = max_over_ranks(t0.elapsed_time(t1) / 1e3, dist, "cuda")
    value = job_value(fl_step, args.steps, world, elapsed)

    # per-pass kernel times
    per = {}
    for pas, name, fl, e0, e1 in events:
        d = per.setdefault(pas, {"fl": 0.0, "t": 0.0, "n": 0, "by_proj": {}})
        dt = e0.elapsed_time(e1) / 1e3
        d["fl"] += fl; d["t"] += dt; d["n"] += 1
        bp = d["by_proj"].setdefault(name, [0.0, 0.0])
        bp[0] += fl; bp[1] += dt
    total_t = sum(d["t"] for d in per.values())
    dom = max(per, key=lambda p: per[p]["t"])
    pk, pk_kind = peaks()
    burst = float(pk.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    sustained = float(pk.get("bf16_tflops_sustained", burst))
    # The denominator is the burst figure (a library matmul timed alone)
    # unless the timed region is seconds long, like the sustained figure's
    # 4-second loop under the power cap; both fractions are reported.
    long_region = elapsed >= SUSTAINED_REGION_S
    peak = sustained if long_region else burst
    peak_source = (f"{pk_kind} bf16_tflops_sustained (timed region {elapsed:.3f} s: power-capped regime)"
                   if long_region else f"{pk_kind} bf16_tflops (burst; timed region {elapsed:.3f} s)")
    d = per[dom]
    achieved = d["fl"] / d["n"] / (d["t"] / d["n"]) / 1e12
    kernel_tag = {"fwd": "tc_gemm_pair_kernel fwd (A K-major, B MN-major)",
                  "dx": "tc_gemm_pair_kernel dX (A K-major, B K-major)",
                  "dw": "tc_gemm_pair_kernel dW (A MN-major, B MN-major, f32 out)"}[dom]
    traffic = traffic_from_profiles(dom)
    passes = {p: {"tflops": v["fl"] / v["t"] / 1e12, "share": v["t"] / total_t,
                  "by_projection_tflops": {nm: f / t / 1e12 for nm, (f, t) in v["by_proj"].items()}}
              for p, v in per.items()}

    # ---- end to end through host buffers (pinned), copies inside the timed region
    for b in bufs:
        b["x_p"] = b["x_h"].pin_memory(); b["w_p"] = b["w_h"].pin_memory(); b["dy_p"] = b["dy_h"].pin_memory()
        b["y_p"] = torch.empty(b["y"].shape, dtype=b["y"].dtype).pin_memory()
        b["dx_p"] = torch.empty(b["dx"].shape, dtype=b["dx"].dtype).pin_memory()
        b["dw_p"] = torch.empty(b["dw"].shape, dtype=b["dw"].dtype).pin_memory()
    h2d = sum(b["x_p"].nbytes + b["w_p"].nbytes + b["dy_p"].nbytes for b in bufs)
    d2h = sum(b["y_p"].nbytes + b["dx_p"].nbytes + b["dw_p"].nbytes for b in bufs)

    # The host link's floor for one step: every input copied in and every
    # result copied out, both directions at once, nothing else running; taken
    # with 1, 2 and 4 copy streams per direction (each tensor split into that
    # many contiguous chunks, one cudaMemcpyAsync each), the fastest reported.
    def chunk_copy(dst, src_t, streams):
        d, s = dst.view(-1), src_t.view(-1)
        per = (d.numel() + len(streams) - 1) // len(streams)
        for j, st in enumerate(streams):
            lo, hi = j * per, min(d.numel(), (j + 1) * per)
            if lo < hi:
                with torch.cuda.stream(st):
                    d[lo:hi].copy_(s[lo:hi], non_blocking=True)

    def copy_floor(nsd, reps=3):
        ins = [torch.cuda.Stream() for _ in range(nsd)]
        outs = [torch.cuda.Stream() for _ in range(nsd)]
        best = None
        for _ in range(reps):
            torch.cuda.synchronize()
            c0 = time.perf_counter()
            for b in bufs:
                for nm in ("x", "w", "dy"):
                    chunk_copy(b[nm], b[nm + "_p"], ins)
                for nm in ("y", "dx", "dw"):
                    chunk_copy(b[nm + "_p"], b[nm], outs)
            torch.cuda.synchronize()
            dt = time.perf_counter() - c0
            best = dt if best is None else min(best, dt)
        return best

    floors = {nsd: copy_floor(nsd) for nsd in (1, 2, 4)}
    floor_s = min(floors.values())

    # Copies run on their own streams (one per direction: the floor above is
    # lowest that way) and overlap the compute of other passes: the forward of
    # projection i waits for its X and W, dX for its dY, dW for both; each result
    # is copied out as soon as its pass ends; a pass waits for the copy-out of
    # its output from the previous step, and the copy-in of an input waits for
    # the last pass of the previous step that reads it.  The events are made
    # once and recorded again every step (a wait refers to the latest record),
    # so the host enqueues a step in well under its GPU time.
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    nb = len(bufs)
    ev = {(key, i): torch.cuda.Event() for i in range(nb)
          for key in ("in_xw", "in_dy", "y", "dx", "dw", "out_y", "out_dx", "out_dw")}
    started = {"first": True}

    def e2e_step():
        first = started["first"]
        with torch.cuda.stream(s_in):
            for i, b in enumerate(bufs):
                if not first:
                    s_in.wait_event(ev[("dw", i)])  # X, W, dY are read up to this projection's dW
                b["x"].copy_(b["x_p"], non_blocking=True)
                b["w"].copy_(b["w_p"], non_blocking=True)
                ev[("in_xw", i)].record(s_in)
                b["dy"].copy_(b["dy_p"], non_blocking=True)
                ev[("in_dy", i)].record(s_in)
        for i, b in enumerate(bufs):
            k, n = b["k"], b["n"]
            stream.wait_event(ev[("in_xw", i)])
            if not first:
                stream.wait_event(ev[("out_y", i)])
            eng.forward(b["y"], b["x"], b["w"], None, m, k, n, "bf16", stream, 1)
            ev[("y", i)].record(stream)
            stream.wait_event(ev[("in_dy", i)])
            if not first:
                stream.wait_event(ev[("out_dx", i)])
            eng.backward_dx(b["dx"], b["dy"], b["w"], m, k, n, "bf16", stream, 1)
            ev[("dx", i)].record(stream)
            if not first:
                stream.wait_event(ev[("out_dw", i)])
            eng.backward_dw(b["dw"], 1, b["x"], b["dy"], m, k, n, "bf16", stream, 1)
            ev[("dw", i)].record(stream)
        with torch.cuda.stream(s_out):
            for i, b in enumerate(bufs):
                for nm in ("y", "dx", "dw"):
                    s_out.wait_event(ev[(nm, i)])
                    b[nm + "_p"].copy_(b[nm], non_blocking=True)
                    ev[("out_" + nm, i)].record(s_out)
        started["first"] = False

    e2e_steps = max(3, min(10, args.steps))
    e2e_step()
    torch.cuda.synchronize()
    barrier()
    s0 = torch.cuda.Event(enable_timing=True); s1 = torch.cuda.Event(enable_timing=True)
    s0.record(stream)
    for st in (s_in, s_out):
        st.wait_event(s0)
    for _ in range(e2e_steps):
        e2e_step()
    for st in (s_in, s_out):
        e = torch.cuda.Event()
        e.record(st)
        stream.wait_event(e)
    s1.record(stream)
    s1.synchronize()
    torch.cuda.synchronize()
    barrier()
    e2e_t = max_over_ranks(s0.elapsed_time(s1) / 1e3, dist, "cuda")
    e2e_value = job_value(fl_step, e2e_steps, world, e2e_t)
    eng.check(stream)

    sec = None
    if rank == 0 and not args.no_secondary:
        sec = secondary(eng, stream, cpu=(world == 1 and not args.no_cpu))
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        # the reference arm's measurement: the same sample, averaged over three draws
        runs = [oracle_sample(seed=s) for s in range(3)]
        t = statistics.mean(r[0] for r in runs)
        f = runs[-1][1]
        cpu = {"value": f / t / 1e12, "unit": "TFLOP/s", "cores": runs[-1][2], "kind": "oracle",
               "sample": runs[-1][3] + "; mean of 3 draws (the reference arm's per-step sample)", "seconds": t}
        if ONLY is None:  # one pass of the step at full size: the o-projection forward
            import oracle
            xn, wn, _ = _HOST_INPUTS["o"]
            _, k, n = [p for p in projections()[0] if p[0] == "o"][0]
            ts = timed_oracle(lambda: oracle.forward(xn, wn, None, m, k, n, "bf16"))
            cpu["full_pass"] = {"value": 2.0 * m * k * n / ts / 1e12, "unit": "TFLOP/s", "seconds": ts,
                                "sample": f"the o-projection forward at full size ({m}x{k}x{n})"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": elapsed / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": WORKLOAD, "m": m, "projections": {nm: [k, n] for nm, k, n in projections()[0]},
                       "tier": "tensor-core (tcgen05)", "dw_dtype": "f32",
                       "l2": "inputs larger than L2 (2.7 GB working set per step, each pass > 129 MB)",
                       "parallelism": "replicas" if world > 1 else "single GPU"},
            "roofline": {"bound": "tensor", "kernel": kernel_tag, "achieved": achieved, "peak": peak,
                         "unit": "TFLOP/s", "frac": achieved / peak, "traffic": traffic,
                         "peak_source": peak_source,
                         "frac_of_burst": achieved / burst, "frac_of_sustained": achieved / sustained},
            "step_frac_of_peak": value / world / peak,
            "passes": passes,
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "steps": e2e_steps, "ms_per_step": e2e_t / e2e_steps * 1e3,
                    "copy_floor_ms": floor_s * 1e3, "copy_streams_per_direction": 1,
                    "copy_floor_ms_by_streams": {str(kk): vv * 1e3 for kk, vv in floors.items()},
                    "frac_of_copy_floor": floor_s / (e2e_t / e2e_steps)},
            "gpu_launches": launches,
            "clocks": clocks,
            "secondary": sec,
        }
        print(json.dumps(line), flush=True)
    eng.close()
    if dist is not None:
        dist.destroy_process_group()


def main():
    global ONLY
    args = parse()
    ONLY = args.only
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.profile_case:
        profile_case(args.profile_case)
    elif args.impl == "reference":
        reference_arm(args, rank, world)
    else:
        our_arm(args, rank, world)


if __name__ == "__main__":
    main()
