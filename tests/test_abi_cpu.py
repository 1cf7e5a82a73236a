"""The C-ABI library on a machine without a GPU: it builds, loads, exports every
entry point declared in include/bi.h, and answers host-only calls (dispatch,
argument validation) without touching a device."""
import ctypes
import os
import re

import pytest

from conftest import ROOT


@pytest.fixture(scope="module")
def bi():
    from deterministic_invariant_gemm_fixed_gb300 import build as _b
    try:
        _b.build()
    except FileNotFoundError as e:
        pytest.skip(f"cannot build the library here: {e}")
    import deterministic_invariant_gemm_fixed_gb300 as m
    m.library()
    return m


def declared_entry_points():
    src = open(os.path.join(ROOT, "include", "bi.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(bi_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(bi):
    names = declared_entry_points()
    assert len(names) >= 14
    lib = ctypes.CDLL(bi.LIB_PATH)
    for name in names:
        assert hasattr(lib, name), name
    # and the binding covers every one of them under the same name
    assert set(names) == set(bi.SIGNATURES)
    for name in names:
        assert callable(getattr(bi, name))


def test_dispatch_is_shape_only(bi):
    P = bi
    # forward: the non-M output dim is N
    assert bi.bi_dispatch_tier(P.BI_PASS_FORWARD, "bf16", 1, 768, 3072) == 1
    assert bi.bi_dispatch_tier(P.BI_PASS_FORWARD, "f16", 1, 1024, 48) == 0
    assert bi.bi_dispatch_tier(P.BI_PASS_FORWARD, "f16", 1, 1024, 64) == 1
    # dX: the non-M output dim is K
    assert bi.bi_dispatch_tier(P.BI_PASS_DX, "f16", 1, 48, 1024) == 0
    assert bi.bi_dispatch_tier(P.BI_PASS_DX, "f16", 1, 1024, 48) == 1
    # dW: both output dims
    assert bi.bi_dispatch_tier(P.BI_PASS_DW, "f16", 1, 1024, 48) == 0
    assert bi.bi_dispatch_tier(P.BI_PASS_DW, "bf16", 1, 4096, 12288) == 1
    # tensor_cores=0 always takes the scalar tier; f32 operands reach the tensor
    # cores (3xTF32) on the dense passes only, with rows in 16-byte units
    for p in range(6):
        assert bi.bi_dispatch_tier(p, "bf16", 0, 4096, 4096) == 0
        assert bi.bi_dispatch_tier(p, "f32", 0, 4096, 4096) == 0
        assert bi.bi_dispatch_tier(p, "f32", 1, 4096, 4096) == (1 if p <= P.BI_PASS_DW else 0)
    assert bi.bi_dispatch_tier(P.BI_PASS_FORWARD, "f32", 1, 1002, 1000) == 0
    assert bi.bi_dispatch_tier(P.BI_PASS_FORWARD, "f32", 1, 1004, 1000) == 1
    # rows that are not whole 16-byte units cannot be fed by TMA
    assert bi.bi_dispatch_tier(P.BI_PASS_FORWARD, "bf16", 1, 1001, 1000) == 0
    assert bi.bi_dispatch_tier(P.BI_PASS_FORWARD, "bf16", 1, 1000, 1000) == 1


def test_null_engine_is_rejected_on_the_host(bi):
    assert bi.bi_forward(None, 16, 16, 16, None, 1, 1, 1, "bf16", 0, 1) == bi.BI_ERR_INVALID_ARG
    assert "NULL" in bi.bi_last_error(None)
    assert bi.bi_backward_dx(None, 16, 16, 16, 1, 1, 1, "bf16", 0, 1) == bi.BI_ERR_INVALID_ARG
    assert bi.bi_backward_dw(None, 16, 1, 16, 16, 1, 1, 1, "bf16", 0, 1) == bi.BI_ERR_INVALID_ARG
    assert bi.bi_grouped_forward(None, 16, 16, 16, 16, 1, 1, 1, 1, "bf16", 0, 1) == bi.BI_ERR_INVALID_ARG
    assert bi.bi_grouped_backward(None, 16, 16, 16, 16, 16, 16, 1, 1, 1, 1, "bf16", 0, 1) == bi.BI_ERR_INVALID_ARG
    assert bi.bi_engine_check(None, 0) == bi.BI_ERR_INVALID_ARG
    assert bi.bi_launch_count(None) == 0
    assert bi.bi_version().startswith("bi ")


def test_engine_creation_fails_cleanly_without_a_device(bi):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    st, h = bi.bi_engine_create(0)
    assert st == bi.BI_ERR_CUDA and h is None
    assert bi.bi_last_error(None)


def test_binding_rejects_unknown_dtypes(bi):
    with pytest.raises(ValueError):
        bi.dtype_code("int8")
    assert bi.dtype_code("bf16") == bi.BI_BF16


def test_binding_refuses_host_and_strided_tensors(bi):
    import torch
    with pytest.raises(ValueError):
        bi._ptr(torch.zeros(4, 4))  # a host tensor never reaches the kernels
    if torch.cuda.is_available():
        with pytest.raises(ValueError):
            bi._ptr(torch.zeros(4, 4, device="cuda").t())
    assert bi._ptr(None) is None and bi._ptr(1234) == 1234


def test_noalloc_applies_the_allocating_path_size_limits_on_the_host(bi):
    # The allocation-free grouped forward refuses exactly what bi_grouped_forward
    # refuses, before it looks for a device: k beyond 8388480 with tiny U32
    # element counts, too many experts, a zero expert count, a bad dtype.
    limit = 65535 * 128
    assert bi.bi_grouped_forward_noalloc(16, 16, 16, 16, 1, limit + 8, 1, 1, "bf16", 0) == bi.BI_ERR_UNSUPPORTED
    assert "8388480" in bi.bi_last_error(None)
    assert bi.bi_grouped_forward_noalloc(16, 16, 16, 16, 1, 8, 8, 65536, "bf16", 0) == bi.BI_ERR_UNSUPPORTED
    assert bi.bi_grouped_forward_noalloc(16, 16, 16, 16, 1, 8, 8, 0, "bf16", 0) == bi.BI_ERR_INVALID_ARG
    assert bi.bi_grouped_forward_noalloc(16, 16, 16, 16, 1, 8, 8, 2, 7, 0) == bi.BI_ERR_INVALID_ARG
    assert bi.bi_grouped_forward_noalloc(16, 16, 16, 16, 1 << 20, 1 << 12, 8, 2, "bf16", 0) == bi.BI_ERR_UNSUPPORTED
    # m = 0 is a no-op once the sizes pass
    assert bi.bi_grouped_forward_noalloc(None, None, None, None, 0, 8, 8, 2, "bf16", 0) == bi.BI_OK


def test_allocation_failure_setter_checks_its_engine(bi):
    assert bi.bi_engine_fail_allocations(None, 1) == bi.BI_ERR_INVALID_ARG
    assert "NULL" in bi.bi_last_error(None)
