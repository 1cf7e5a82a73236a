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
@pytest.mark.parametrize("m", [1, 3])
def test_skinny_rows_special_values_bit_exact(eng, dtype, m):
    """Batches of at most 4 rows (the matrix-vector kernel, forward and dX) on
    NaN, infinities and subnormal operands, planted in W so that each reaches
    only its own outputs; x and dY carry subnormals."""
    k, n = 264, 136
    x, w, dy, b = synth.dense_inputs(m, k, n, dtype, w=("normal", 1.0))
    tiny = {"bf16": 1e-40, "f16": 3e-6, "f32": 1e-40}[dtype]
    x.view(-1)[::17] = tiny
    dy.view(-1)[::13] = -tiny
    w = plant(w, dtype, 7, True)
    xn, wn, dyn, bn = (synth.to_np(t) for t in (x, w, dy, b))
    td = TD[dtype]
    y = torch.empty(m, n, dtype=td, device="cuda")
    dx = torch.empty(m, k, dtype=td, device="cuda")
    eng.forward(y, dev(x), dev(w), dev(b), m, k, n, dtype, None, 0)
    eng.backward_dx(dx, dev(dy), dev(w), m, k, n, dtype, None, 0)
    eng.check()
    y, dx = out_np(y), out_np(dx)
    assert same_with_nan(y, oracle.forward(xn, wn, bn, m, k, n, dtype), dtype)
    assert same_with_nan(dx, oracle.backward_dx(dyn, wn, m, k, n, dtype), dtype)
    assert np.isnan(values(y, dtype)).any() and np.isfinite(values(y, dtype)).any()


@pytest.mark.parametrize("m", [1, 4])
def test_skinny_rows_subnormal_chains_bit_exact(eng, m):
    """bf16 operands near 1e-20: every product is an f32 subnormal and so is
    every partial sum, so each step of the chain rounds in the subnormal range
    (f16 operands cannot get there: their smallest product is an f32 normal).
    The outputs, bf16 subnormals, must equal the oracle's bit for bit."""
    k, n, dtype = 1000, 264, "bf16"
    nrm = ("normal", 1.0)
    x, w, dy, _ = synth.dense_inputs(m, k, n, dtype, x=nrm, w=nrm, dy=nrm)
    x, w, dy = (t.float().mul(1e-20).to(torch.bfloat16) for t in (x, w, dy))
    xn, wn, dyn = (synth.to_np(t) for t in (x, w, dy))
    y = torch.empty(m, n, dtype=torch.bfloat16, device="cuda")
    dx = torch.empty(m, k, dtype=torch.bfloat16, device="cuda")
    eng.forward(y, dev(x), dev(w), None, m, k, n, dtype, None, 0)
    eng.backward_dx(dx, dev(dy), dev(w), m, k, n, dtype, None, 0)
    eng.check()
    y, dx = out_np(y), out_np(dx)
    want = oracle.forward(xn, wn, None, m, k, n, dtype)
    assert np.array_equal(y, want)
    assert np.array_equal(dx, oracle.backward_dx(dyn, wn, m, k, n, dtype))
    v = np.abs(values(want, dtype))
    assert ((v > 0) & (v < np.finfo(np.float32).tiny)).mean() > 0.9  # subnormal results


SIGNED_ZERO_SHAPES = [
    (3, 200, 136),     # matrix-vector kernel (Y, dX), narrow dW; contractions 200, 136, 3
    (333, 200, 48),    # narrow kernels for Y, dX and dW (two chunks, the last of 77 rows)
    (2004, 632, 648),  # tiled kernels (Y, dX: 632 and 648 steps), dW chunk kernel (last chunk 212 rows)
    (2001, 631, 647),  # the same kernels on rows that are not whole 16-byte units
]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("m,k,n", SIGNED_ZERO_SHAPES, ids=lambda v: str(v))
def test_scalar_chains_keep_a_negative_zero(eng, dtype, m, k, n):
    """Every product is a negative value far below the smallest subnormal
    (-1e-30 * 1e-20), so it rounds to -0, and a chain from +0 stays at -0 after
    its first step (+0 + -0 rounds to +0, but the fused product is rounded
    together with the sum: RN(-1e-50 + 0) = -0, then RN(-1e-50 + -0) = -0).
    Every output of Y, dX and dW is therefore -0, bit for bit, in the oracle and
    on the scalar tier.  The contractions are not whole multiples of any
    kernel's staged block, so padded steps must leave a chain at -0 unchanged."""
    td = TD[dtype]
    neg, pos = torch.full((1,), -1e-30).to(td), torch.full((1,), 1e-20).to(td)
    x = neg.expand(m, k).contiguous()
    w = pos.expand(k, n).contiguous()
    dy_dx = neg.expand(m, n).contiguous()          # dX = dY W^T: products -1e-30 * 1e-20
    dy_dw = (-neg).expand(m, n).contiguous()       # dW = X^T dY: products -1e-30 * 1e-30
    y = torch.empty(m, n, dtype=td, device="cuda")
    dx = torch.empty(m, k, dtype=td, device="cuda")
    dw = torch.empty(k, n, dtype=torch.float32, device="cuda")
    dwr = torch.empty(k, n, dtype=td, device="cuda")
    eng.forward(y, dev(x), dev(w), None, m, k, n, dtype, None, 0)
    eng.backward_dx(dx, dev(dy_dx), dev(w), m, k, n, dtype, None, 0)
    eng.backward_dw(dw, 1, dev(x), dev(dy_dw), m, k, n, dtype, None, 0)
    eng.backward_dw(dwr, 0, dev(x), dev(dy_dw), m, k, n, dtype, None, 0)
    eng.check()
    for name, t in (("y", y), ("dx", dx), ("dw", dw), ("dw rounded", dwr)):
        f = t.float()
        assert torch.equal(f, torch.zeros_like(f)), name
        assert bool(torch.signbit(f).all()), name  # -0 everywhere
    if m * k * n <= 200 * 136 * 3:  # the oracle agrees (small case only)
        xn, wn = synth.to_np(x), synth.to_np(w)
        want = oracle.forward(xn, wn, None, m, k, n, dtype, out_f32=True)
        assert np.all(want == 0) and np.all(np.signbit(want))
        want = oracle.backward_dw(xn, synth.to_np(dy_dw), m, k, n, dtype, dw_f32=True)
        assert np.all(want == 0) and np.all(np.signbit(want))


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
