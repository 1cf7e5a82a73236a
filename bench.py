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
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "TFLOP/s fwd+dX+dW (bf16 TC tier) and fraction of dense-bf16 roofline"
WORKLOAD = "7B-class layer bf16 tensor-core tier, M=8192: qkv 4096x12288, o 4096x4096, up 4096x11008, down 11008x4096; fwd+dX+dW (f32 dW)"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--only", default=None, help="restrict the step to one projection (profiling case)")
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


def oracle_sample(rows=512, cols=128, seed=0):
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
            f"reduction) of the same workload; {total_fl / 1e9:.1f} GFLOP")
    return total_t, total_fl, oracle.num_threads(), desc


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

def secondary(eng, stream, reps=5):
    """Grouped tensor-core pass, scalar tier and GEMV on their own workloads."""
    import torch
    import numpy as np
    from deterministic_invariant_gemm_fixed_gb300 import synth
    out = {}

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

    # grouped bf16 M=16384 K=2048 E=8 N=1408, tensor-core tier
    c = synth.GROUPED
    m, k, n, e = c["m"], c["k"], c["n"], c["e"]
    x, w, dy, ids = synth.grouped_inputs(m, k, n, e, "bf16", pad_frac=c["pad_frac"])
    valid = int((synth.to_np(ids) < e).sum())
    X, W, DY = x.cuda(), w.cuda(), dy.cuda()
    I = torch.from_numpy(synth.to_np(ids).astype(np.int32)).cuda()
    Y = torch.empty(m, n, dtype=torch.bfloat16, device="cuda")
    DX = torch.empty(m, k, dtype=torch.bfloat16, device="cuda")
    DWg = torch.empty(e, n, k, dtype=torch.float32, device="cuda")
    fl = 2.0 * valid * n * k
    t_f = timeit(lambda: eng.grouped_forward(Y, X, W, I, m, k, n, e, "bf16", stream, 1))
    t_b = timeit(lambda: eng.grouped_backward(DX, DWg, X, W, DY, I, m, k, n, e, "bf16", stream, 1))
    out["grouped_tc"] = {"workload": c["name"], "fwd_tflops": fl / t_f / 1e12,
                         "bwd_tflops": 2 * fl / t_b / 1e12, "fwd_ms": t_f * 1e3, "bwd_ms": t_b * 1e3}
    # the same rows already grouped by the caller (segmented entry points, tensor cores)
    ids_np = synth.to_np(ids)
    order = np.argsort(np.minimum(ids_np, e), kind="stable")
    counts = np.bincount(np.minimum(ids_np, e), minlength=e + 1)[:e]
    offs = torch.from_numpy(np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)).cuda()
    Xs, DYs = X[torch.from_numpy(order).cuda()].contiguous(), DY[torch.from_numpy(order).cuda()].contiguous()
    t_sf = timeit(lambda: eng.grouped_forward_segmented(Y, Xs, W, offs, m, k, n, e, "bf16", stream, 1))
    t_sb = timeit(lambda: eng.grouped_backward_segmented(DX, DWg, Xs, W, DYs, offs, m, k, n, e, "bf16", stream, 1))
    out["grouped_segmented_tc"] = {"workload": c["name"] + " (rows pre-grouped)", "fwd_tflops": fl / t_sf / 1e12,
                                   "bwd_tflops": 2 * fl / t_sb / 1e12}
    del Xs, DYs
    del X, W, DY, Y, DX, DWg
    # scalar tier, GPT-2-small MLP up-projection bf16 4096x768x3072
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
    props = torch.cuda.get_device_properties(0)
    sms = props.multi_processor_count
    ffma_peak = sms * 128 * 2 * 2070e6 / 1e12  # FP32 FMA lanes x 2 flop x max SM clock
    t_s = timeit(lambda: scal(0))
    t_t = timeit(lambda: scal(1))
    out["scalar_gpt2_up"] = {"workload": g["name"], "tflops": fl / t_s / 1e12,
                             "ffma_peak_tflops": ffma_peak, "frac_of_ffma_peak": fl / t_s / 1e12 / ffma_peak}
    out["tc_gpt2_up"] = {"workload": g["name"], "tflops": fl / t_t / 1e12}
    del X, W, DY, B, Y, DX, DW
    # bias gradient of the qkv projection: column sums of dY [8192, 12288] bf16 (HBM-bound)
    g = synth.normal((8192, 12288), 1.0, "bf16", 60).cuda()
    db = torch.empty(12288, dtype=torch.bfloat16, device="cuda")
    t_bg = timeit(lambda: eng.bias_grad(db, 0, g, 8192, 12288, "bf16", stream))
    out["bias_grad"] = {"workload": "bf16 dY 8192x12288 column sums", "gbs": (g.nbytes + db.nbytes) / t_bg / 1e9,
                        "us": t_bg * 1e6}
    del g
    # FP8 e4m3 per-tensor-scaled passes on the qkv projection (pre-quantized operands)
    m, k, n = synth.SEVEN_B_M, 4096, 12288
    xq = torch.randint(0, 0x70, (m, k), dtype=torch.uint8, device="cuda")
    wq = torch.randint(0, 0x70, (k, n), dtype=torch.uint8, device="cuda")
    gq = torch.randint(0, 0x70, (m, n), dtype=torch.uint8, device="cuda")
    one = torch.ones(1, dtype=torch.float32, device="cuda")
    y8 = torch.empty(m, n, dtype=torch.bfloat16, device="cuda")
    dx8 = torch.empty(m, k, dtype=torch.bfloat16, device="cuda")
    dw8 = torch.empty(k, n, dtype=torch.float32, device="cuda")

    def fp8_step():
        eng.fp8_forward(y8, xq, wq, None, one, one, m, k, n, "bf16", stream)
        eng.fp8_backward_dx(dx8, gq, wq, one, one, m, k, n, "bf16", stream)
        eng.fp8_backward_dw(dw8, xq, gq, one, one, m, k, n, "f32", stream)
    t8 = timeit(fp8_step)
    pk, _ = peaks()
    fp8_peak = 2.0 * float(pk.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))  # nominal fp8:bf16 = 2:1
    out["fp8_qkv"] = {"workload": "e4m3 qkv 8192x4096x12288 fwd+dX+dW", "tflops": 3 * 2.0 * m * k * n / t8 / 1e12,
                      "peak_tflops": fp8_peak, "frac": 3 * 2.0 * m * k * n / t8 / 1e12 / fp8_peak}
    del xq, wq, gq, y8, dx8, dw8
    # f32 operands on the tensor cores (3xTF32: split kernels + three tf32 MMAs per
    # contraction step), the o-projection shape 8192x4096x4096 in f32
    m, k, n = synth.SEVEN_B_M, 4096, 4096
    x, w, dy, _ = synth.dense_inputs(m, k, n, "f32", b=None)
    X, W, DY = x.cuda(), w.cuda(), dy.cuda()
    del x, w, dy
    Yf = torch.empty(m, n, device="cuda")
    DXf = torch.empty(m, k, device="cuda")
    DWf = torch.empty(k, n, device="cuda")

    def tf32_step():
        eng.forward(Yf, X, W, None, m, k, n, "f32", stream, 1)
        eng.backward_dx(DXf, DY, W, m, k, n, "f32", stream, 1)
        eng.backward_dw(DWf, 1, X, DY, m, k, n, "f32", stream, 1)
    t32 = timeit(tf32_step)
    # ceiling: measured bf16 peak x the nominal tf32:bf16 ratio (1.1 : 2.25), over 3 MMAs per product
    tf32_ceiling = float(pk.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])) * (1.1 / 2.25) / 3
    v32 = 3 * 2.0 * m * k * n / t32 / 1e12
    out["tf32x3_f32_o"] = {"workload": "f32 o-projection 8192x4096x4096 fwd+dX+dW, 3xTF32", "tflops": v32,
                           "ceiling_tflops": tf32_ceiling, "frac": v32 / tf32_ceiling}
    del X, W, DY, Yf, DXf, DWf
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
        moved = 2 * (X.nbytes + W.nbytes + DY.nbytes) + Y.nbytes + DX.nbytes + DW.nbytes  # each pass reads two operands
        out["f16_" + name] = {"workload": f"f16 {m}x{k}x{n} fwd+dX+dW ({'scalar' if tc == 0 else 'tensor-core'} tier)",
                              "tflops": 3 * 2.0 * m * k * n / te / 1e12, "gbs": moved / te / 1e9, "us": te * 1e6}
        del X, W, DY, B, Y, DX, DW
    # GEMV f16 1x4096x4096, tensor-core tier (HBM-bound): W rotated over 8 copies > L2
    k = n = 4096
    ws = [synth.uniform((k, n), -1, 1, "f16", 100 + i).cuda() for i in range(8)]
    xv = synth.uniform((1, k), -1, 1, "f16", 99).cuda()
    yv = torch.empty(1, n, dtype=torch.float16, device="cuda")
    state = {"i": 0}

    def gemv():
        eng.forward(yv, xv, ws[state["i"] % 8], None, 1, k, n, "f16", stream, 1)
        state["i"] += 1
    t_g = timeit(gemv)
    out["gemv_tc_f16"] = {"workload": "f16 1x4096x4096", "gbs": (k * n * 2 + k * 2 + n * 2) / t_g / 1e9,
                          "us": t_g * 1e6}

    # the same GEMV on the scalar tier (one lane per output column, bit-exact chains)
    def gemv_scalar():
        eng.forward(yv, xv, ws[state["i"] % 8], None, 1, k, n, "f16", stream, 0)
        state["i"] += 1
    t_gs = timeit(gemv_scalar)
    out["gemv_scalar_f16"] = {"workload": "f16 1x4096x4096 (scalar tier)",
                              "gbs": (k * n * 2 + k * 2 + n * 2) / t_gs / 1e9, "us": t_gs * 1e6,
                              "chain_bound_us": k * 4 / 2.07e3}
    return out


# ---------------------------------------------------------------- arms

def reference_arm(args, rank, world):
    if rank != 0:
        return
    secs, fl, cores, desc = [], 0.0, 1, ""
    for s in range(args.warmup + args.steps):
        t, f, cores, desc = oracle_sample(rows=8, cols=2, seed=s)
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
    # The denominator follows the regime of the timed region: back-to-back dense
    # GEMMs reach the power cap within a fraction of a second (measured: 40
    # steps, 0.2 s, ran 6-7 % below 10 steps on one box, with sw_power_cap
    # active), so a region of 0.1 s or more is compared with the sustained
    # (power-capped) figure and a shorter one with the burst figure.
    long_region = elapsed >= 0.1
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

    # Copies run on their own streams and overlap the compute of other
    # projections: h2d of projection i (step s) waits for the compute of i in
    # step s-1; the compute of i waits for its h2d and for the d2h of i in step
    # s-1; the d2h of i waits for its compute.
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev = {(kind, i): torch.cuda.Event() for kind in ("in", "comp", "out") for i in range(len(bufs))}
    started = {"first": True}

    def e2e_step():
        for i, b in enumerate(bufs):
            if not started["first"]:
                s_in.wait_event(ev[("comp", i)])
            with torch.cuda.stream(s_in):
                b["x"].copy_(b["x_p"], non_blocking=True)
                b["w"].copy_(b["w_p"], non_blocking=True)
                b["dy"].copy_(b["dy_p"], non_blocking=True)
            ev[("in", i)].record(s_in)
            stream.wait_event(ev[("in", i)])
            if not started["first"]:
                stream.wait_event(ev[("out", i)])
            run_step(eng, [b], m, stream)
            ev[("comp", i)].record(stream)
            s_out.wait_event(ev[("comp", i)])
            with torch.cuda.stream(s_out):
                b["y_p"].copy_(b["y"], non_blocking=True)
                b["dx_p"].copy_(b["dx"], non_blocking=True)
                b["dw_p"].copy_(b["dw"], non_blocking=True)
            ev[("out", i)].record(s_out)
        started["first"] = False

    e2e_steps = max(3, min(10, args.steps))
    e2e_step()
    torch.cuda.synchronize()
    barrier()
    s0 = torch.cuda.Event(enable_timing=True); s1 = torch.cuda.Event(enable_timing=True)
    s0.record(s_in)
    stream.wait_event(s0)
    s_out.wait_event(s0)
    for _ in range(e2e_steps):
        e2e_step()
    s1.record(s_out)
    s1.synchronize()
    torch.cuda.synchronize()
    barrier()
    e2e_t = max_over_ranks(s0.elapsed_time(s1) / 1e3, dist, "cuda")
    e2e_value = job_value(fl_step, e2e_steps, world, e2e_t)

    sec = None
    if rank == 0 and not args.no_secondary:
        sec = secondary(eng, stream)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        t, f, cores, desc = oracle_sample()
        cpu = {"value": f / t / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": desc,
               "seconds": t}

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
                    "steps": e2e_steps, "ms_per_step": e2e_t / e2e_steps * 1e3},
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
    if args.impl == "reference":
        reference_arm(args, rank, world)
    else:
        our_arm(args, rank, world)


if __name__ == "__main__":
    main()
