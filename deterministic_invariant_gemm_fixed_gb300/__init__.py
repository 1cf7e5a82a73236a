"""Deterministic, batch-invariant training matmul for GB300 (sm_103a).

Thin ctypes binding over the C ABI in ``include/bi.h`` (libbi.so, built in-tree
by ``deterministic_invariant_gemm_fixed_gb300.build``).  The functions below
carry the C names and only marshal arguments: tensors become device pointers,
torch dtypes become ``bi_dtype`` values, streams become ``cudaStream_t``
handles.  Every step of the computation runs in the library's CUDA kernels.
There is no fallback: if libbi.so is missing, the first call raises.

Each ``bi_*`` function returns the C status code; ``Engine`` wraps the same
calls and raises ``BiError`` on a non-zero status.
"""
from __future__ import annotations

import ctypes
import os

from . import synth  # noqa: F401  (seeded inputs; holds no arithmetic)

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libbi.so")

BI_F32, BI_BF16, BI_F16 = 0, 1, 2
BI_OK, BI_ERR_INVALID_ARG, BI_ERR_MISALIGNED, BI_ERR_UNSUPPORTED = 0, 1, 2, 3
BI_ERR_CUDA, BI_ERR_OOM, BI_ERR_TIMEOUT = 4, 5, 6
STATUS_NAMES = {0: "BI_OK", 1: "BI_ERR_INVALID_ARG", 2: "BI_ERR_MISALIGNED", 3: "BI_ERR_UNSUPPORTED",
                4: "BI_ERR_CUDA", 5: "BI_ERR_OOM", 6: "BI_ERR_TIMEOUT"}
(BI_PASS_FORWARD, BI_PASS_DX, BI_PASS_DW, BI_PASS_GROUPED_FORWARD, BI_PASS_GROUPED_DINPUT,
 BI_PASS_GROUPED_DWEIGHTS) = range(6)
BI_DW_CHUNK = 256
BI_STRATEGY_SCALAR, BI_STRATEGY_TENSOR_CORE, BI_STRATEGY_AUTO = 0, 1, 2

# Every entry point declared in include/bi.h, with its ctypes signature.
_p, _i64, _i32, _u64 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_uint64
SIGNATURES = {
    "bi_engine_create": (_i32, [_i32, ctypes.POINTER(_p)]),
    "bi_engine_destroy": (None, [_p]),
    "bi_last_error": (ctypes.c_char_p, [_p]),
    "bi_engine_check": (_i32, [_p, _p]),
    "bi_forward": (_i32, [_p, _p, _p, _p, _p, _i64, _i64, _i64, _i32, _p, _i32]),
    "bi_backward_dx": (_i32, [_p, _p, _p, _p, _i64, _i64, _i64, _i32, _p, _i32]),
    "bi_backward_dw": (_i32, [_p, _p, _i32, _p, _p, _i64, _i64, _i64, _i32, _p, _i32]),
    "bi_bias_grad": (_i32, [_p, _p, _i32, _p, _i64, _i64, _i32, _p]),
    "bi_grouped_forward": (_i32, [_p, _p, _p, _p, _p, _i64, _i64, _i64, _i64, _i32, _p, _i32]),
    "bi_grouped_backward": (_i32, [_p, _p, _p, _p, _p, _p, _p, _i64, _i64, _i64, _i64, _i32, _p, _i32]),
    "bi_dispatch_tier": (_i32, [_i32, _i32, _i32, _i64, _i64]),
    "bi_launch_count": (_u64, [_p]),
    "bi_engine_set_wait_limit": (_i32, [_p, _u64]),
    "bi_engine_fail_allocations": (_i32, [_p, _i64]),
    "bi_engine_set_tile_cols": (_i32, [_p, _i32]),
    "bi_selftest_wait_timeout": (_i32, [_p, _p]),
    "bi_version": (ctypes.c_char_p, []),
    "bi_grouped_forward_segmented": (_i32, [_p, _p, _p, _p, _p, _i64, _i64, _i64, _i64, _i32, _p, _i32]),
    "bi_grouped_backward_segmented": (_i32, [_p, _p, _p, _p, _p, _p, _p, _i64, _i64, _i64, _i64, _i32, _p, _i32]),
    "bi_fp8_quantize": (_i32, [_p, _p, _p, _p, _p, _i64, _i32, _p]),
    "bi_fp8_forward": (_i32, [_p, _p, _p, _p, _p, _p, _p, _i64, _i64, _i64, _i32, _p]),
    "bi_fp8_backward_dx": (_i32, [_p, _p, _p, _p, _p, _p, _i64, _i64, _i64, _i32, _p]),
    "bi_fp8_backward_dw": (_i32, [_p, _p, _p, _p, _p, _p, _i64, _i64, _i64, _i32, _p]),
    "bi_grouped_forward_noalloc": (_i32, [_p, _p, _p, _p, _i64, _i64, _i64, _i64, _i32, _p]),
}


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it with "
            "`python -c 'import __graft_entry__ as g; g.build()'` (no CPU fallback exists)")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


class _LazyLib:
    """Loads libbi.so on first use (so the build module and the input generator
    can be imported before the library exists); raises if it is missing."""
    _h = None

    def __getattr__(self, name):
        if _LazyLib._h is None:
            _LazyLib._h = _load()
        return getattr(_LazyLib._h, name)


_lib = _LazyLib()


def library():
    """The loaded ctypes library (loads it now; raises ImportError if absent)."""
    _lib.bi_version  # noqa: B018
    return _LazyLib._h


class BiError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


def dtype_code(dtype) -> int:
    """bi_dtype from a torch dtype, a string ('f32', 'bf16', 'f16') or an int."""
    if isinstance(dtype, int):
        return dtype
    s = str(dtype).replace("torch.", "")
    table = {"float32": BI_F32, "f32": BI_F32, "bfloat16": BI_BF16, "bf16": BI_BF16,
             "float16": BI_F16, "f16": BI_F16, "half": BI_F16}
    if s not in table:
        raise ValueError(f"unsupported dtype {dtype!r}")
    return table[s]


def _ptr(t):
    """Device address of a tensor (or an int / None passed through).  The C ABI
    reads dense row-major device memory, so a tensor on the host or a strided
    view is refused here rather than handed to the kernels."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError("bi: tensors must be on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("bi: tensors must be contiguous (dense, row-major)")
    return t.data_ptr()


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


# ---- the C entry points, same names, argument marshalling only ----------------

def bi_engine_create(device: int = 0):
    h = ctypes.c_void_p()
    st = _lib.bi_engine_create(device, ctypes.byref(h))
    return st, h.value


def bi_engine_destroy(engine) -> None:
    _lib.bi_engine_destroy(engine)


def bi_last_error(engine=None) -> str:
    return (_lib.bi_last_error(engine) or b"").decode()


def bi_engine_check(engine, stream=None) -> int:
    return _lib.bi_engine_check(engine, _stream(stream))


def bi_forward(engine, y, x, w, bias, m, k, n, dtype, stream=None, tensor_cores=1) -> int:
    return _lib.bi_forward(engine, _ptr(y), _ptr(x), _ptr(w), _ptr(bias), m, k, n, dtype_code(dtype),
                           _stream(stream), int(tensor_cores))


def bi_backward_dx(engine, dx, dy, w, m, k, n, dtype, stream=None, tensor_cores=1) -> int:
    return _lib.bi_backward_dx(engine, _ptr(dx), _ptr(dy), _ptr(w), m, k, n, dtype_code(dtype),
                               _stream(stream), int(tensor_cores))


def bi_backward_dw(engine, dw, dw_f32, x, dy, m, k, n, dtype, stream=None, tensor_cores=1) -> int:
    return _lib.bi_backward_dw(engine, _ptr(dw), int(dw_f32), _ptr(x), _ptr(dy), m, k, n,
                               dtype_code(dtype), _stream(stream), int(tensor_cores))


def bi_bias_grad(engine, db, db_f32, dy, m, n, dtype, stream=None) -> int:
    return _lib.bi_bias_grad(engine, _ptr(db), int(db_f32), _ptr(dy), m, n, dtype_code(dtype), _stream(stream))


def bi_grouped_forward(engine, y, x, w, row_experts, m, k, n, e, dtype, stream=None, tensor_cores=1) -> int:
    return _lib.bi_grouped_forward(engine, _ptr(y), _ptr(x), _ptr(w), _ptr(row_experts), m, k, n, e,
                                   dtype_code(dtype), _stream(stream), int(tensor_cores))


def bi_grouped_backward(engine, dx, dw, x, w, dy, row_experts, m, k, n, e, dtype, stream=None,
                        tensor_cores=1) -> int:
    return _lib.bi_grouped_backward(engine, _ptr(dx), _ptr(dw), _ptr(x), _ptr(w), _ptr(dy),
                                    _ptr(row_experts), m, k, n, e, dtype_code(dtype), _stream(stream),
                                    int(tensor_cores))


def bi_grouped_forward_segmented(engine, y, x, w, offsets, m, k, n, e, dtype, stream=None,
                                 strategy=BI_STRATEGY_SCALAR) -> int:
    return _lib.bi_grouped_forward_segmented(engine, _ptr(y), _ptr(x), _ptr(w), _ptr(offsets), m, k, n, e,
                                             dtype_code(dtype), _stream(stream), int(strategy))


def bi_grouped_backward_segmented(engine, dx, dw, x, w, dy, offsets, m, k, n, e, dtype, stream=None,
                                  strategy=BI_STRATEGY_SCALAR) -> int:
    return _lib.bi_grouped_backward_segmented(engine, _ptr(dx), _ptr(dw), _ptr(x), _ptr(w), _ptr(dy),
                                              _ptr(offsets), m, k, n, e, dtype_code(dtype), _stream(stream),
                                              int(strategy))


def bi_fp8_quantize(engine, q, amax, src, scale_inv, count, src_dtype, stream=None) -> int:
    return _lib.bi_fp8_quantize(engine, _ptr(q), _ptr(amax), _ptr(src), _ptr(scale_inv), count,
                                dtype_code(src_dtype), _stream(stream))


def bi_fp8_forward(engine, y, xq, wq, bias, scale_x, scale_w, m, k, n, out_dtype, stream=None) -> int:
    return _lib.bi_fp8_forward(engine, _ptr(y), _ptr(xq), _ptr(wq), _ptr(bias), _ptr(scale_x), _ptr(scale_w),
                               m, k, n, dtype_code(out_dtype), _stream(stream))


def bi_fp8_backward_dx(engine, dx, gq, wq, scale_g, scale_w, m, k, n, out_dtype, stream=None) -> int:
    return _lib.bi_fp8_backward_dx(engine, _ptr(dx), _ptr(gq), _ptr(wq), _ptr(scale_g), _ptr(scale_w),
                                   m, k, n, dtype_code(out_dtype), _stream(stream))


def bi_fp8_backward_dw(engine, dw, xq, gq, scale_x, scale_g, m, k, n, out_dtype, stream=None) -> int:
    return _lib.bi_fp8_backward_dw(engine, _ptr(dw), _ptr(xq), _ptr(gq), _ptr(scale_x), _ptr(scale_g),
                                   m, k, n, dtype_code(out_dtype), _stream(stream))


def bi_grouped_forward_noalloc(y, x, w, row_experts, m, k, n, e, dtype, stream=None) -> int:
    """Scalar-tier grouped forward with no allocation (see include/bi.h); errors
    are read with bi_last_error(None)."""
    return _lib.bi_grouped_forward_noalloc(_ptr(y), _ptr(x), _ptr(w), _ptr(row_experts), m, k, n, e,
                                           dtype_code(dtype), _stream(stream))


def bi_dispatch_tier(pass_, dtype, tensor_cores, k, n) -> int:
    return _lib.bi_dispatch_tier(int(pass_), dtype_code(dtype), int(tensor_cores), k, n)


def bi_launch_count(engine) -> int:
    return _lib.bi_launch_count(engine)


def bi_engine_set_wait_limit(engine, nanoseconds: int) -> int:
    return _lib.bi_engine_set_wait_limit(engine, int(nanoseconds))


def bi_engine_fail_allocations(engine, count: int) -> int:
    return _lib.bi_engine_fail_allocations(engine, int(count))


def bi_engine_set_tile_cols(engine, cols: int) -> int:
    return _lib.bi_engine_set_tile_cols(engine, int(cols))


def bi_selftest_wait_timeout(engine, stream=None) -> int:
    return _lib.bi_selftest_wait_timeout(engine, _stream(stream))


def bi_version() -> str:
    return _lib.bi_version().decode()


# ---- convenience wrapper that raises ---------------------------------------------

class Engine:
    """Owns a bi_engine handle; methods mirror the C calls and raise BiError."""

    def __init__(self, device: int = 0):
        st, h = bi_engine_create(device)
        if st != BI_OK:
            raise BiError(st, bi_last_error(None))
        self.handle = h
        self.device = device

    def _ok(self, st):
        if st != BI_OK:
            raise BiError(st, bi_last_error(self.handle))

    def forward(self, y, x, w, bias, m, k, n, dtype, stream=None, tensor_cores=1):
        self._ok(bi_forward(self.handle, y, x, w, bias, m, k, n, dtype, stream, tensor_cores))

    def backward_dx(self, dx, dy, w, m, k, n, dtype, stream=None, tensor_cores=1):
        self._ok(bi_backward_dx(self.handle, dx, dy, w, m, k, n, dtype, stream, tensor_cores))

    def backward_dw(self, dw, dw_f32, x, dy, m, k, n, dtype, stream=None, tensor_cores=1):
        self._ok(bi_backward_dw(self.handle, dw, dw_f32, x, dy, m, k, n, dtype, stream, tensor_cores))

    def bias_grad(self, db, db_f32, dy, m, n, dtype, stream=None):
        self._ok(bi_bias_grad(self.handle, db, db_f32, dy, m, n, dtype, stream))

    def grouped_forward(self, y, x, w, ids, m, k, n, e, dtype, stream=None, tensor_cores=1):
        self._ok(bi_grouped_forward(self.handle, y, x, w, ids, m, k, n, e, dtype, stream, tensor_cores))

    def grouped_backward(self, dx, dw, x, w, dy, ids, m, k, n, e, dtype, stream=None, tensor_cores=1):
        self._ok(bi_grouped_backward(self.handle, dx, dw, x, w, dy, ids, m, k, n, e, dtype, stream,
                                     tensor_cores))

    def grouped_forward_segmented(self, y, x, w, offsets, m, k, n, e, dtype, stream=None,
                                  strategy=BI_STRATEGY_SCALAR):
        self._ok(bi_grouped_forward_segmented(self.handle, y, x, w, offsets, m, k, n, e, dtype, stream, strategy))

    def grouped_backward_segmented(self, dx, dw, x, w, dy, offsets, m, k, n, e, dtype, stream=None,
                                   strategy=BI_STRATEGY_SCALAR):
        self._ok(bi_grouped_backward_segmented(self.handle, dx, dw, x, w, dy, offsets, m, k, n, e, dtype,
                                               stream, strategy))

    def fp8_quantize(self, q, amax, src, scale_inv, count, src_dtype, stream=None):
        self._ok(bi_fp8_quantize(self.handle, q, amax, src, scale_inv, count, src_dtype, stream))

    def fp8_forward(self, y, xq, wq, bias, scale_x, scale_w, m, k, n, out_dtype, stream=None):
        self._ok(bi_fp8_forward(self.handle, y, xq, wq, bias, scale_x, scale_w, m, k, n, out_dtype, stream))

    def fp8_backward_dx(self, dx, gq, wq, scale_g, scale_w, m, k, n, out_dtype, stream=None):
        self._ok(bi_fp8_backward_dx(self.handle, dx, gq, wq, scale_g, scale_w, m, k, n, out_dtype, stream))

    def fp8_backward_dw(self, dw, xq, gq, scale_x, scale_g, m, k, n, out_dtype, stream=None):
        self._ok(bi_fp8_backward_dw(self.handle, dw, xq, gq, scale_x, scale_g, m, k, n, out_dtype, stream))

    def check(self, stream=None):
        self._ok(bi_engine_check(self.handle, stream))

    def launches(self) -> int:
        return bi_launch_count(self.handle)

    def close(self):
        if getattr(self, "handle", None):
            bi_engine_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
