"""CPU oracle for the deterministic, batch-invariant training matmul.

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's
CPU-baseline leg may import this package; the library itself never does.  It
shares no code with the CUDA path.

The arithmetic lives in ``bi_oracle.c`` (plain C, fmaf chains, IEEE-754 format
helpers written from the binary16/bfloat16 encodings).  This module only
compiles it with gcc and marshals numpy arrays into it.

Operand convention: f32 data travel as ``np.float32`` arrays; bf16 and f16 data
travel as ``np.uint16`` arrays holding the raw encodings.  ``dtype`` is one of
``"f32"``, ``"bf16"``, ``"f16"``.

What each function computes (the sources are the pages' own titles):

* ``forward``      - sgemm-bi 0.1.1.post2, "Use" and "Determinism contracts";
                     ViperLLM ffma.py, _FFMAAddmm.forward (bias in f32, one
                     downcast).  Y = rne(chain_k X W + b).
* ``backward_dx``  - ViperLLM ffma.py, _FFMAAddmm.backward: gx = gy W^T.
* ``backward_dw``  - ViperLLM ffma.py, _FFMAAddmm.backward: gW = x^T gy, with
                     the reduction over rows cut into chunks of ``chunk`` rows
                     and summed by the fixed pairwise tree.
* ``bias_grad``    - sgemm-bi 0.1.1.post2 (the bias gradient is an f32 column
                     sum, kept outside the engine there); here in fixed order.
* ``fp8_*``        - AstrAI csrc/kernels/fp8_mm.cu: quantize_kernel (codes and
                     amax), fp8_linear_forward_scaled / _backward_scaled (the
                     per-tensor scales applied to the f32 product).
* ``grouped_*``    - rublas 0.1.45 src/tensor_grouped/mod.rs: fn
                     grouped_matmul_nt (ids outside [0,E) give zero rows),
                     struct GroupedBackward (dweights always f32).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "bi_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD_DIR, "libbi_oracle.so")

DTYPES = {"f32": 0, "bf16": 1, "f16": 2}
# The dW chunk length of the scalar tier's published contract.
DW_CHUNK = 256

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile bi_oracle.c into a shared object with gcc (OpenMP if available)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(_SRC):
        return _SO
    base = ["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-ffp-contract=off",
            "-fno-fast-math", "-Wall", "-Wextra", "-Wno-unused-parameter"]
    tmp = _SO + ".tmp.%d" % os.getpid()
    err = ""
    for extra in (["-fopenmp"], []):
        cmd = base + extra + ["-o", tmp, _SRC, "-lm"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode == 0:
            os.replace(tmp, _SO)
            return _SO
        err = r.stderr
    raise RuntimeError("oracle build failed:\n" + err)


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            p, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
            sig = {
                "or_forward_rows": [p, p, p, p, p, i64, i64, i64, i64, i32, i32],
                "or_backward_dx_rows": [p, p, p, p, i64, i64, i64, i64, i32, i32],
                "or_backward_dw_cols": [p, p, p, p, i64, i64, i64, i64, i32, i64, i32],
                "or_grouped_segment": [p, i64, i64, p, p],
                "or_bias_grad": [p, p, i64, i64, i32, i64, i32],
                "or_fp8_forward_rows": [p, p, p, p, ctypes.c_float, ctypes.c_float, p, i64, i64, i64, i64, i32],
                "or_fp8_backward_dx_rows": [p, p, p, ctypes.c_float, ctypes.c_float, p, i64, i64, i64, i64, i32],
                "or_fp8_backward_dw": [p, p, p, ctypes.c_float, ctypes.c_float, i64, i64, i64, i32, i64],
                "or_grouped_forward_rows": [p, p, p, p, p, i64, i64, i64, i64, i64, i32, i32],
                "or_grouped_dinput_rows": [p, p, p, p, p, i64, i64, i64, i64, i64, i32, i32],
                "or_grouped_dweights_sel": [p, p, p, p, p, p, i64, i64, i64, i64, i64, i32, i64],
                "or_rne_array": [p, p, i64, i32],
                "or_rne_bits_range": [p, ctypes.c_uint64, i64, i32],
                "or_up_array": [p, p, i64, i32],
                "or_tree_sum": [p, i64],
                "or_num_threads": [],
                "or_set_num_threads": [i32],
            }
            for name, args in sig.items():
                fn = getattr(lib, name)
                fn.argtypes = args
                fn.restype = ctypes.c_int
            lib.or_tree_sum.restype = ctypes.c_float
            lib.or_fmaf.argtypes = [ctypes.c_float] * 3
            lib.or_fmaf.restype = ctypes.c_float
            for name in ("or_set_num_threads", "or_rne_array", "or_rne_bits_range", "or_up_array"):
                getattr(lib, name).restype = None
            lib.or_e4m3_bits_range.argtypes = [p, ctypes.c_uint64, i64]
            lib.or_e4m3_bits_range.restype = None
            lib.or_up_e4m3_array.argtypes = [p, p, i64]
            lib.or_up_e4m3_array.restype = None
            lib.or_fp8_quantize.argtypes = [p, p, p, i32, ctypes.c_float, i64]
            lib.or_fp8_quantize.restype = None
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _elem(dtype):
    return np.float32 if dtype == "f32" else np.uint16


def _check(a, dtype, count, name):
    if a.dtype != _elem(dtype):
        raise TypeError(f"{name}: expected {_elem(dtype).__name__} data for {dtype}")
    if not a.flags.c_contiguous:
        raise ValueError(f"{name}: must be C-contiguous")
    if a.size != count:
        raise ValueError(f"{name}: expected {count} elements, got {a.size}")


def _index_arg(idx, full):
    if idx is None:
        return None, full
    r = np.ascontiguousarray(np.asarray(idx, dtype=np.int64))
    return r, r.size


def num_threads() -> int:
    return _load().or_num_threads()


def set_num_threads(n: int) -> None:
    _load().or_set_num_threads(int(n))


def fmaf(a: float, b: float, c: float) -> float:
    return _load().or_fmaf(a, b, c)


def tree_sum(values) -> np.float32:
    v = np.ascontiguousarray(np.asarray(values, dtype=np.float32)).copy()
    return np.float32(_load().or_tree_sum(_ptr(v), v.size))


def rne(values_f32: np.ndarray, dtype: str) -> np.ndarray:
    """f32 -> bf16/f16 encodings, round to nearest even."""
    v = np.ascontiguousarray(values_f32, dtype=np.float32)
    out = np.empty(v.shape, dtype=np.uint16)
    _load().or_rne_array(_ptr(out), _ptr(v), v.size, DTYPES[dtype])
    return out


def rne_bits_range(first_bits: int, count: int, dtype: str, out=None) -> np.ndarray:
    if out is None:
        out = np.empty(count, dtype=np.uint16)
    _load().or_rne_bits_range(_ptr(out), first_bits, count, DTYPES[dtype])
    return out


def up(values_u16: np.ndarray, dtype: str) -> np.ndarray:
    """bf16/f16 encodings -> f32 values (exact widening)."""
    v = np.ascontiguousarray(values_u16, dtype=np.uint16)
    out = np.empty(v.shape, dtype=np.float32)
    _load().or_up_array(_ptr(out), _ptr(v), v.size, DTYPES[dtype])
    return out


def forward(x, w, bias, m, k, n, dtype, rows=None, out_f32=False):
    """Y[rows] (all rows when rows is None): [len(rows), N] in dtype (or f32)."""
    _check(x, dtype, m * k, "x"); _check(w, dtype, k * n, "w")
    if bias is not None:
        _check(bias, dtype, n, "bias")
    r, nr = _index_arg(rows, m)
    y = np.empty((nr, n), dtype=np.float32 if out_f32 else _elem(dtype))
    rc = _load().or_forward_rows(_ptr(y), _ptr(x), _ptr(w), _ptr(bias), _ptr(r), nr, m, k, n,
                                 DTYPES[dtype], int(out_f32))
    if rc:
        raise MemoryError("oracle forward failed")
    return y


def backward_dx(dy, w, m, k, n, dtype, rows=None, out_f32=False):
    """dX[rows]: [len(rows), K]."""
    _check(dy, dtype, m * n, "dy"); _check(w, dtype, k * n, "w")
    r, nr = _index_arg(rows, m)
    dx = np.empty((nr, k), dtype=np.float32 if out_f32 else _elem(dtype))
    rc = _load().or_backward_dx_rows(_ptr(dx), _ptr(dy), _ptr(w), _ptr(r), nr, m, k, n,
                                     DTYPES[dtype], int(out_f32))
    if rc:
        raise MemoryError("oracle dX failed")
    return dx


def backward_dw(x, dy, m, k, n, dtype, dw_f32=False, chunk=DW_CHUNK, cols=None):
    """dW[:, cols] (all columns when cols is None): [K, len(cols)]."""
    _check(x, dtype, m * k, "x"); _check(dy, dtype, m * n, "dy")
    c, nc = _index_arg(cols, n)
    dw = np.empty((k, nc), dtype=np.float32 if dw_f32 else _elem(dtype))
    rc = _load().or_backward_dw_cols(_ptr(dw), _ptr(x), _ptr(dy), _ptr(c), nc, m, k, n,
                                     DTYPES[dtype], int(chunk), int(dw_f32))
    if rc:
        raise MemoryError("oracle dW failed")
    return dw


def bias_grad(dy, m, n, dtype, out_f32=False, chunk=DW_CHUNK):
    """db[N]: the fixed-order column sum of dY (chunks of `chunk` rows, f32
    additions from +0 in row order, then the dW tree over chunk partials)."""
    _check(dy, dtype, m * n, "dy")
    db = np.empty(n, dtype=np.float32 if out_f32 else _elem(dtype))
    if _load().or_bias_grad(_ptr(db), _ptr(dy), m, n, DTYPES[dtype], int(chunk), int(out_f32)):
        raise MemoryError("oracle bias grad failed")
    return db


def e4m3_bits_range(first_bits: int, count: int) -> np.ndarray:
    """e4m3 encodings of the f32 patterns first_bits .. first_bits+count-1."""
    out = np.empty(count, dtype=np.uint8)
    _load().or_e4m3_bits_range(_ptr(out), first_bits, count)
    return out


def up_e4m3(q: np.ndarray) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.uint8)
    out = np.empty(q.shape, dtype=np.float32)
    _load().or_up_e4m3_array(_ptr(out), _ptr(q), q.size)
    return out


def fp8_quantize(src, dtype, scale_inv):
    """(e4m3 codes, amax) of src * scale_inv (AstrAI fp8_mm.cu quantize_kernel)."""
    src = np.ascontiguousarray(src)
    _check(src, dtype, src.size, "src")
    q = np.empty(src.shape, dtype=np.uint8)
    amax = np.zeros(1, dtype=np.float32)
    _load().or_fp8_quantize(_ptr(q), _ptr(amax), _ptr(src), DTYPES[dtype], float(scale_inv), src.size)
    return q, np.float32(amax[0])


def fp8_forward(xq, wq, bias, sx, sw, m, k, n, out_dtype, rows=None):
    r, nr = _index_arg(rows, m)
    y = np.empty((nr, n), dtype=_elem(out_dtype))
    _load().or_fp8_forward_rows(_ptr(y), _ptr(np.ascontiguousarray(xq)), _ptr(np.ascontiguousarray(wq)),
                                _ptr(bias), float(sx), float(sw), _ptr(r), nr, m, k, n, DTYPES[out_dtype])
    return y


def fp8_backward_dx(gq, wq, sg, sw, m, k, n, out_dtype, rows=None):
    r, nr = _index_arg(rows, m)
    dx = np.empty((nr, k), dtype=_elem(out_dtype))
    _load().or_fp8_backward_dx_rows(_ptr(dx), _ptr(np.ascontiguousarray(gq)), _ptr(np.ascontiguousarray(wq)),
                                    float(sg), float(sw), _ptr(r), nr, m, k, n, DTYPES[out_dtype])
    return dx


def fp8_backward_dw(xq, gq, sx, sg, m, k, n, out_dtype, chunk=DW_CHUNK):
    dw = np.empty((k, n), dtype=_elem(out_dtype))
    rc = _load().or_fp8_backward_dw(_ptr(dw), _ptr(np.ascontiguousarray(xq)), _ptr(np.ascontiguousarray(gq)),
                                    float(sx), float(sg), m, k, n, DTYPES[out_dtype], int(chunk))
    if rc:
        raise MemoryError("oracle fp8 dW failed")
    return dw


def grouped_segment(ids, m, e):
    """(perm [M] u32, offsets [E+2] u32): stable grouping by expert, padding last."""
    ids = np.ascontiguousarray(ids, dtype=np.uint32)
    perm = np.zeros(max(m, 1), dtype=np.uint32)
    offs = np.empty(e + 2, dtype=np.uint32)
    if _load().or_grouped_segment(_ptr(ids), m, e, _ptr(perm), _ptr(offs)):
        raise RuntimeError("segment mismatch")
    return perm[:m], offs


def grouped_forward(x, w, ids, m, k, n, e, dtype, rows=None, out_f32=False):
    _check(x, dtype, m * k, "x"); _check(w, dtype, e * n * k, "w")
    ids = np.ascontiguousarray(ids, dtype=np.uint32)
    r, nr = _index_arg(rows, m)
    y = np.empty((nr, n), dtype=np.float32 if out_f32 else _elem(dtype))
    _load().or_grouped_forward_rows(_ptr(y), _ptr(x), _ptr(w), _ptr(ids), _ptr(r), nr, m, k, n, e,
                                    DTYPES[dtype], int(out_f32))
    return y


def grouped_dinput(w, dy, ids, m, k, n, e, dtype, rows=None, out_f32=False):
    _check(dy, dtype, m * n, "dy"); _check(w, dtype, e * n * k, "w")
    ids = np.ascontiguousarray(ids, dtype=np.uint32)
    r, nr = _index_arg(rows, m)
    dx = np.empty((nr, k), dtype=np.float32 if out_f32 else _elem(dtype))
    _load().or_grouped_dinput_rows(_ptr(dx), _ptr(w), _ptr(dy), _ptr(ids), _ptr(r), nr, m, k, n, e,
                                   DTYPES[dtype], int(out_f32))
    return dx


def grouped_dweights(x, dy, ids, m, k, n, e, dtype, chunk=DW_CHUNK, sel=None):
    """dW[E,N,K] f32, or, with sel = (experts, ns), the rows dW[sel_e[i], sel_n[i], :]."""
    _check(x, dtype, m * k, "x"); _check(dy, dtype, m * n, "dy")
    ids = np.ascontiguousarray(ids, dtype=np.uint32)
    if sel is None:
        se = sn = None
        nsel = e * n
        shape = (e, n, k)
    else:
        se = np.ascontiguousarray(np.asarray(sel[0], dtype=np.int64))
        sn = np.ascontiguousarray(np.asarray(sel[1], dtype=np.int64))
        nsel = se.size
        shape = (nsel, k)
    dw = np.empty(shape, dtype=np.float32)
    rc = _load().or_grouped_dweights_sel(_ptr(dw), _ptr(x), _ptr(dy), _ptr(ids), _ptr(se), _ptr(sn),
                                         nsel, m, k, n, e, DTYPES[dtype], int(chunk))
    if rc:
        raise MemoryError("oracle grouped dweights failed")
    return dw
