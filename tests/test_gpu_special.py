"""Special values through the C ABI: NaN, infinities and subnormal operands,
results that overflow the output type, and a grouping whose rows are all
padding.

Scalar tier: bit-exact with the oracle, NaN compared as NaN (the NaN encoding
after rounding is not part of the contract).  Tensor-core tier: the NaN and
infinity pattern equals the oracle's (with no finite partial sum near
overflow, the pattern does not depend on the summation order), finite
results within the tolerance."""
import numpy as np
import pytest
import torch

import oracle
import deterministic_invariant_gemm_fixed_gb300 as bi
from deterministic_invariant_gemm_fixed_gb300 import synth
from helpers import abs_sum, check_tc, dev, f64, out_np

pytestmark = pytest.mark.gpu
TD = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}


@pytest.fixture(scope="module")
def eng():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    e = bi.Engine(0)
    yield e
    e.close()


def values(a, dtype):
    """Float64 view of oracle/GPU outputs (encodings for 16-bit types)."""
    return oracle.up(a, dtype).astype(np.float64) if dtype != "f32" else a.astype(np.float64)


def same_with_nan(got, want, dtype):
    g, w = values(got, dtype), values(want, dtype)
    gn, wn = np.isnan(g), np.isnan(w)
    return np.array_equal(gn, wn) and np.array_equal(got[~gn], want[~wn])


def plant(t, dtype, seed, subnormals):
    """Put NaN, +-Inf (and subnormals) at seeded positions of a CPU tensor."""
    rng = np.random.default_rng(seed)
    flat = t.view(-1)
    idx = rng.choice(flat.numel(), size=12, replace=False)
    specials = [float("nan"), float("inf"), float("-inf")] * 3
    if subnormals:
        tiny = {"bf16": 1e-40, "f16": 3e-6, "f32": 1e-40}[dtype]
        specials += [tiny, -tiny, tiny * 3]
    else:
        specials += [0.5, -0.5, 0.25]
    for i, v in zip(idx, specials):
        flat[int(i)] = v
    return t


def run(eng, x, w, dy, b, m, k, n, dtype, tc):
    X, W, DY, B = dev(x), dev(w), dev(dy), dev(b)
    td = TD[dtype]
    y = torch.empty(m, n, dtype=td, device="cuda")
    dx = torch.empty(m, k, dtype=td, device="cuda")
    dw = torch.empty(k, n, dtype=torch.float32, device="cuda")
    eng.forward(y, X, W, B, m, k, n, dtype, None, tc)
    eng.backward_dx(dx, DY, W, m, k, n, dtype, None, tc)
    eng.backward_dw(dw, 1, X, DY, m, k, n, dtype, None, tc)
    eng.check()
    return out_np(y), out_np(dx), out_np(dw)


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_scalar_special_values_bit_exact(eng, dtype):
    m, k, n = 96, 136, 200
    x, w, dy, b = synth.dense_inputs(m, k, n, dtype, w=("normal", 1.0))
    x, w, dy = plant(x, dtype, 1, True), plant(w, dtype, 2, True), plant(dy, dtype, 3, True)
    if dtype == "f16":  # columns whose sums overflow f16 after rounding
        x[:, 0] = 200.0
        w[0, :8] = 400.0
    y, dx, dw = run(eng, x, w, dy, b, m, k, n, dtype, tc=0)
    xn, wn, dyn, bn = (synth.to_np(t) for t in (x, w, dy, b))
    assert same_with_nan(y, oracle.forward(xn, wn, bn, m, k, n, dtype), dtype)
    assert same_with_nan(dx, oracle.backward_dx(dyn, wn, m, k, n, dtype), dtype)
    assert same_with_nan(dw, oracle.backward_dw(xn, dyn, m, k, n, dtype, dw_f32=True), "f32")
    assert np.isnan(values(y, dtype)).any() and np.isinf(values(y, dtype)).any()
    if dtype == "f16":
        assert np.isinf(values(y, dtype)[:, 0:8]).any()  # the overflow case was hit


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_tensor_core_special_values(eng, dtype):
    m, k, n = 260, 264, 272
    x, w, dy, b = synth.dense_inputs(m, k, n, dtype, w=("normal", 1.0))
    x, w, dy = plant(x, dtype, 4, False), plant(w, dtype, 5, False), plant(dy, dtype, 6, False)
    y, dx, dw = run(eng, x, w, dy, b, m, k, n, dtype, tc=1)
    xn, wn, dyn, bn = (synth.to_np(t) for t in (x, w, dy, b))
    x64, w64, dy64, b64 = (f64(a, dtype) for a in (xn, wn, dyn, bn))
    for got, want32, S, out in (
            (y, oracle.forward(xn, wn, bn, m, k, n, dtype, out_f32=True),
             abs_sum(np.nan_to_num(x64, posinf=0, neginf=0), np.nan_to_num(w64, posinf=0, neginf=0), b64), dtype),
            (dx, oracle.backward_dx(dyn, wn, m, k, n, dtype, out_f32=True),
             abs_sum(np.nan_to_num(dy64, posinf=0, neginf=0), np.nan_to_num(w64, posinf=0, neginf=0).T), dtype),
            (dw, oracle.backward_dw(xn, dyn, m, k, n, dtype, dw_f32=True),
             abs_sum(np.nan_to_num(x64, posinf=0, neginf=0).T, np.nan_to_num(dy64, posinf=0, neginf=0)), "f32")):
        g = values(got, out)
        r = want32.astype(np.float64)
        assert np.array_equal(np.isnan(g), np.isnan(r))
        assert np.array_equal(np.isposinf(g), np.isposinf(r)) and np.array_equal(np.isneginf(g), np.isneginf(r))
        fin = np.isfinite(r)
        assert fin.sum() > 0.5 * fin.size
        ok, st = check_tc(got[fin], want32[fin], S[fin], out)
        assert ok, st


@pytest.mark.parametrize("tc", [0, 1])
def test_grouped_all_rows_padding(eng, tc):
    m, k, n, e = 300, 128, 136, 4
    x, w, dy, _ = synth.grouped_inputs(m, k, n, e, "bf16")
    ids = torch.full((m,), e, dtype=torch.int32)
    ids[::7] = e + 100  # every id is padding (E itself and beyond)
    X, W, DY, I = dev(x), dev(w), dev(dy), ids.cuda()
    y = torch.full((m, n), 7.0, dtype=torch.bfloat16, device="cuda")
    dx = torch.full((m, k), 7.0, dtype=torch.bfloat16, device="cuda")
    dw = torch.full((e, n, k), 7.0, dtype=torch.float32, device="cuda")
    eng.grouped_forward(y, X, W, I, m, k, n, e, "bf16", None, tc)
    eng.grouped_backward(dx, dw, X, W, DY, I, m, k, n, e, "bf16", None, tc)
    eng.check()
    for t in (y, dx, dw):
        assert torch.equal(t.float().abs().sum(), torch.zeros((), device="cuda"))
        assert not torch.signbit(t.float()).any()  # +0, not -0
