"""Shared helpers for the GPU tests: device staging and the tensor-core tolerance.

Tolerance of the tensor-core tier (the published bound: 2e-6 relative for f32
results, 1 ulp of bf16/f16 after the downcast), read per element with the
oracle's f32 value r (before its rounding) and S = sum |a_i * b_i| (+ |bias|):

* f32 results:      |t - r| <= 2e-6 * S
* bf16/f16 results: ulp distance(t, rne(r)) <= 1, or, where cancellation makes
                    the rounded result smaller than the accumulated f32 error,
                    |t - r| <= 2e-6 * S + ulp(t) / 2

S is the scale against which any two f32 summation orders of the same terms
differ (their difference is bounded by a multiple of u * S, not of u * |r|);
elements with |r| far below S are where a literal relative test would fail for
every order change.  The strict element-wise figures are reported alongside:
with the environment variable BI_PARITY_LOG set to a file name, every check
appends one JSON line (the test, the output type, the element count, and the
literal figures: the share of f32 elements beyond 2e-6 relative error, or the
count of 16-bit elements more than 1 ulp away) to that file.
"""
from __future__ import annotations

import json
import os

import numpy as np
import torch

import oracle
from deterministic_invariant_gemm_fixed_gb300 import synth

TC_REL = 2e-6


def dev(t):
    return t.cuda() if t is not None else None


def out_np(t):
    torch.cuda.synchronize()
    return synth.to_np(t.cpu())


def f64(a, dtype):
    if dtype == "f32" or a.dtype == np.float32:
        return a.astype(np.float64)
    return synth.from_np(a, dtype).to(torch.float64).numpy()


def ulp_of(v64, dtype):
    """Spacing of the dtype's grid at |v| (subnormal spacing near zero)."""
    mant, emin = {"bf16": (8, -126), "f16": (11, -14), "f32": (24, -126)}[dtype]
    a = np.maximum(np.abs(v64), np.ldexp(1.0, emin))
    e = np.floor(np.log2(a))
    return np.ldexp(1.0, (e - (mant - 1)).astype(np.int64))


def ulp_distance(a_u16, b_u16):
    def key(h):
        h = h.astype(np.int64)
        return np.where(h & 0x8000, -(h & 0x7FFF), h)
    return np.abs(key(a_u16) - key(b_u16))


def _record(ok, dtype_out, stats):
    path = os.environ.get("BI_PARITY_LOG")
    if not path:
        return
    test = os.environ.get("PYTEST_CURRENT_TEST", "?").split(" (")[0]
    with open(path, "a") as f:
        f.write(json.dumps(dict(test=test, out=dtype_out, ok=ok, **stats)) + "\n")


def check_tc(t, r32, S, dtype_out):
    """t: GPU result (uint16 encodings or float32); r32: oracle f32 value before
    rounding; S: float64 magnitude sums.  Returns (all_ok, stats dict)."""
    r = r32.astype(np.float64)
    nan = np.isnan(r)
    fin = ~nan
    if dtype_out == "f32":
        tv = t.astype(np.float64)
        err = np.abs(tv - r)
        ok = (err <= TC_REL * S) | (nan & np.isnan(tv))
        rel = (err / np.maximum(np.abs(r), 1e-300))[fin]
        stats = dict(max_err_over_S=float(np.max((err / np.maximum(S, 1e-300))[fin])) if fin.any() else 0.0,
                     frac_rel_gt_2e6=float(np.mean(rel > TC_REL)) if rel.size else 0.0,
                     max_rel=float(np.max(rel)) if rel.size else 0.0, n=int(r.size))
        _record(bool(ok.all()), dtype_out, stats)
        return bool(ok.all()), stats
    want = oracle.rne(r32.astype(np.float32), dtype_out)
    d = ulp_distance(t, want)
    tv = f64(t, dtype_out)
    strict = d <= 1
    loose = np.abs(tv - r) <= TC_REL * S + 0.5 * ulp_of(tv, dtype_out)
    ok = strict | loose | (nan & np.isnan(tv))
    strict_fin = strict | ~fin
    stats = dict(max_ulp=int(d[fin].max()) if fin.any() else 0, n_over_1ulp=int((~strict_fin).sum()),
                 frac_over_1ulp=float(np.mean(~strict_fin)) if d.size else 0.0, n=int(d.size))
    _record(bool(ok.all()), dtype_out, stats)
    return bool(ok.all()), stats


def abs_sum(a64, b64, bias64=None):
    s = np.abs(a64) @ np.abs(b64)
    if bias64 is not None:
        s = s + np.abs(bias64)
    return s


def sample_rows(m, count, seed=0):
    rng = np.random.default_rng(seed)
    base = {0, m - 1, m // 2, min(m - 1, 127), min(m - 1, 128)}
    extra = rng.choice(m, size=min(m, count), replace=False)
    return np.array(sorted(base | set(int(v) for v in extra)), dtype=np.int64)
