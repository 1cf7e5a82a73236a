"""GPU parity of the dense passes (forward, dX, dW) through the C ABI.

Scalar tier: bit-exact against the oracle.  Tensor-core tier: within the
tolerance in helpers.py, and bit-exact on exact small-integer problems.  Both
tiers: bit-identical over 10 runs, and row m of Y / dX independent of M.
"""
import numpy as np
import pytest
import torch

import oracle
import deterministic_invariant_gemm_fixed_gb300 as bi
from deterministic_invariant_gemm_fixed_gb300 import synth
from helpers import abs_sum, check_tc, dev, f64, out_np, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def eng():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    e = bi.Engine(0)
    yield e
    e.close()


def run_dense(eng, x, w, dy, b, m, k, n, dtype, tc, dw_f32=True, passes=("y", "dx", "dw")):
    tdt = synth.TORCH_DTYPES[dtype]
    X, W, DY, B = dev(x), dev(w), dev(dy), dev(b)
    out = {}
    if "y" in passes:
        y = torch.empty(m, n, dtype=tdt, device="cuda")
        eng.forward(y, X, W, B, m, k, n, dtype, None, tc)
        out["y"] = y
    if "dx" in passes:
        dx = torch.empty(m, k, dtype=tdt, device="cuda")
        eng.backward_dx(dx, DY, W, m, k, n, dtype, None, tc)
        out["dx"] = dx
    if "dw" in passes:
        dw = torch.empty(k, n, dtype=torch.float32 if (dw_f32 or dtype == "f32") else tdt, device="cuda")
        eng.backward_dw(dw, int(dw_f32), X, DY, m, k, n, dtype, None, tc)
        out["dw"] = dw
    eng.check()
    return {kk: out_np(v) for kk, v in out.items()}


def np_in(*ts):
    return [synth.to_np(t) if t is not None else None for t in ts]


SCALAR_CASES = [
    # name, dtype, M, K, N, value spec
    ("linear_f32", "f32", 64, 256, 512, ("normal", 1.0)),
    ("ragged_f16", "f16", 300, 200, 130, ("uniform", 1.0)),
    ("odd_bf16", "bf16", 257, 77, 131, ("normal", 1.0)),     # unaligned rows: scalar loads
    ("n48_fallback_f16", "f16", 2048, 1024, 48, ("uniform", 1.0)),
    ("gemv_f16", "f16", 1, 4096, 4096, ("uniform", 1.0)),
    ("ragged_1000_f16", "f16", 1000, 1000, 1000, ("uniform", 1.0)),
    ("long_dw_chunks_bf16", "bf16", 1500, 64, 72, ("normal", 1.0)),  # 6 chunks, odd tree
    ("narrow_both_bf16", "bf16", 333, 40, 48, ("normal", 1.0)),  # narrow-output kernel for Y and dX
    ("tree32_f16", "f16", 8192, 64, 72, ("uniform", 1.0)),   # 32 dW chunks: the register tree
    ("tree33_bf16", "bf16", 8200, 64, 72, ("normal", 1.0)),  # 33 dW chunks: the counter form
]


@pytest.mark.parametrize("case", SCALAR_CASES, ids=lambda c: c[0])
def test_scalar_tier_bit_exact(eng, case):
    _, dtype, m, k, n, spec = case
    x, w, dy, b = synth.dense_inputs(m, k, n, dtype, x=spec, w=spec, dy=spec, b=("normal", 0.1))
    got = run_dense(eng, x, w, dy, b, m, k, n, dtype, tc=0)
    xn, wn, dyn, bn = np_in(x, w, dy, b)
    assert np.array_equal(got["y"], oracle.forward(xn, wn, bn, m, k, n, dtype))
    assert np.array_equal(got["dx"], oracle.backward_dx(dyn, wn, m, k, n, dtype))
    assert np.array_equal(got["dw"], oracle.backward_dw(xn, dyn, m, k, n, dtype, dw_f32=True))
    # rounded dW as well
    got2 = run_dense(eng, x, w, dy, b, m, k, n, dtype, tc=0, dw_f32=False, passes=("dw",))
    assert np.array_equal(got2["dw"], oracle.backward_dw(xn, dyn, m, k, n, dtype, dw_f32=False))


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("m", [1, 2, 3, 4])
def test_scalar_skinny_rows_bit_exact(eng, dtype, m):
    """Batches of at most 4 rows take one lane per output column (forward and
    dX): bit-exact with the oracle, with a ragged last column tile (136, 200
    columns), a contraction shorter than one 64-step stage, and one of 81
    stages that wraps the 16-stage ring."""
    for k, n in ((200, 136), (5184, 264), (32, 72)):
        x, w, dy, b = synth.dense_inputs(m, k, n, dtype)
        got = run_dense(eng, x, w, dy, b, m, k, n, dtype, tc=0, passes=("y", "dx"))
        xn, wn, dyn, bn = np_in(x, w, dy, b)
        assert np.array_equal(got["y"], oracle.forward(xn, wn, bn, m, k, n, dtype)), (k, n)
        assert np.array_equal(got["dx"], oracle.backward_dx(dyn, wn, m, k, n, dtype)), (k, n)


@pytest.mark.parametrize("case", SCALAR_CASES, ids=lambda c: c[0])
def test_tc_flag_on_scalar_shapes_is_scalar(eng, case):
    """With tensor_cores=1, passes whose shape the dispatcher keeps on the scalar
    tier (an output dim < 64, rows not whole 16-byte units) give the scalar
    results bit for bit."""
    _, dtype, m, k, n, spec = case
    x, w, dy, b = synth.dense_inputs(m, k, n, dtype, x=spec, w=spec, dy=spec, b=("normal", 0.1))
    a = run_dense(eng, x, w, dy, b, m, k, n, dtype, tc=0)
    t = run_dense(eng, x, w, dy, b, m, k, n, dtype, tc=1)
    for key, p in (("y", bi.BI_PASS_FORWARD), ("dx", bi.BI_PASS_DX), ("dw", bi.BI_PASS_DW)):
        if bi.bi_dispatch_tier(p, dtype, 1, k, n) == 0:
            assert np.array_equal(a[key], t[key]), key


def test_scalar_gpt2_up_sampled(eng):
    c = synth.GPT2_UP
    m, k, n, dtype = c["m"], c["k"], c["n"], c["dtype"]
    x, w, dy, b = synth.dense_inputs(m, k, n, dtype, x=c["x"], w=c["w"], dy=c["dy"], b=c["b"])
    got = run_dense(eng, x, w, dy, b, m, k, n, dtype, tc=0)
    xn, wn, dyn, bn = np_in(x, w, dy, b)
    rows = sample_rows(m, 96)
    cols = sample_rows(n, 24, seed=1)
    assert np.array_equal(got["y"][rows], oracle.forward(xn, wn, bn, m, k, n, dtype, rows=rows))
    assert np.array_equal(got["dx"][rows], oracle.backward_dx(dyn, wn, m, k, n, dtype, rows=rows))
    assert np.array_equal(got["dw"][:, cols], oracle.backward_dw(xn, dyn, m, k, n, dtype, dw_f32=True, cols=cols))


TC_CASES = [
    ("ragged_f32", "f32", 300, 200, 520),       # 3xTF32
    ("multi_tile_f32", "f32", 520, 1004, 776),  # 3xTF32, long contraction
    ("odd_m_f32", "f32", 301, 260, 132),        # 3xTF32: M not a multiple of 4, N not of 8
    ("ragged_bf16", "bf16", 300, 200, 520),
    ("multi_tile_bf16", "bf16", 520, 264, 776),
    ("ragged_1000_f16", "f16", 1000, 1000, 1000),
    ("gemv_f16", "f16", 1, 4096, 4096),
    ("small_k_f16", "f16", 130, 8, 72),
    ("ragged_tiles_bf16", "bf16", 700, 384, 1408),  # 5.5 and 1.5 column tiles; dW on 128-column tiles
    ("ragged_tiles_f16", "f16", 520, 640, 384),
]


@pytest.mark.parametrize("case", TC_CASES, ids=lambda c: c[0])
def test_tc_tier_within_tolerance(eng, case):
    _, dtype, m, k, n = case
    spec = ("uniform", 1.0) if dtype == "f16" else ("normal", 1.0)
    x, w, dy, b = synth.dense_inputs(m, k, n, dtype, x=spec, w=spec, dy=spec, b=("normal", 0.1))
    for p in (bi.BI_PASS_FORWARD, bi.BI_PASS_DX, bi.BI_PASS_DW):
        assert bi.bi_dispatch_tier(p, dtype, 1, k, n) == (0 if (p != bi.BI_PASS_FORWARD and k < 64) else 1)
    got = run_dense(eng, x, w, dy, b, m, k, n, dtype, tc=1)
    got_r = got if dtype == "f32" else run_dense(eng, x, w, dy, b, m, k, n, dtype, tc=1, dw_f32=False,
                                                  passes=("dw",))
    xn, wn, dyn, bn = np_in(x, w, dy, b)
    x64, w64, dy64, b64 = (f64(a, dtype) for a in (xn, wn, dyn, bn))
    r = oracle.forward(xn, wn, bn, m, k, n, dtype, out_f32=True)
    ok, st = check_tc(got["y"], r, abs_sum(x64, w64, b64), dtype)
    assert ok, ("y", st)
    r = oracle.backward_dx(dyn, wn, m, k, n, dtype, out_f32=True)
    ok, st = check_tc(got["dx"], r, abs_sum(dy64, w64.T), dtype)
    assert ok, ("dx", st)
    r = oracle.backward_dw(xn, dyn, m, k, n, dtype, dw_f32=True)
    S = abs_sum(x64.T, dy64)
    ok, st = check_tc(got["dw"], r, S, "f32")
    assert ok, ("dw f32", st)
    ok, st = check_tc(got_r["dw"], r, S, dtype)
    assert ok, ("dw rounded", st)


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_tc_tier_exact_on_small_integers(eng, dtype):
    """Integer operands in [-8, 8] (f16: [-16, 16]) make every partial sum exact in
    f32, so the tensor-core result must equal the oracle bit for bit, bias and
    the single rounding included."""
    m, k, n = 333, 320, 392
    hi = 16 if dtype == "f16" else 8
    x = synth.small_ints((m, k), -hi, hi, dtype, 11)
    w = synth.small_ints((k, n), -hi, hi, dtype, 12)
    dy = synth.small_ints((m, n), -hi, hi, dtype, 13)
    b = (synth.small_ints((n,), -128, 127, "f32", 14) / 2).to(synth.TORCH_DTYPES[dtype])
    got = run_dense(eng, x, w, dy, b, m, k, n, dtype, tc=1)
    got_r = got if dtype == "f32" else run_dense(eng, x, w, dy, b, m, k, n, dtype, tc=1, dw_f32=False,
                                                  passes=("dw",))
    xn, wn, dyn, bn = np_in(x, w, dy, b)
    assert np.array_equal(got["y"], oracle.forward(xn, wn, bn, m, k, n, dtype))
    assert np.array_equal(got["dx"], oracle.backward_dx(dyn, wn, m, k, n, dtype))
    assert np.array_equal(got["dw"], oracle.backward_dw(xn, dyn, m, k, n, dtype, dw_f32=True))
    assert np.array_equal(got_r["dw"], oracle.backward_dw(xn, dyn, m, k, n, dtype, dw_f32=False))


def test_tc_gpt2_up_sampled(eng):
    c = synth.GPT2_UP
    m, k, n, dtype = c["m"], c["k"], c["n"], c["dtype"]
    x, w, dy, b = synth.dense_inputs(m, k, n, dtype, x=c["x"], w=c["w"], dy=c["dy"], b=c["b"])
    got = run_dense(eng, x, w, dy, b, m, k, n, dtype, tc=1)
    xn, wn, dyn, bn = np_in(x, w, dy, b)
    x64, w64, dy64, b64 = (f64(a, dtype) for a in (xn, wn, dyn, bn))
    rows = sample_rows(m, 64)
    cols = sample_rows(n, 16, seed=1)
    r = oracle.forward(xn, wn, bn, m, k, n, dtype, rows=rows, out_f32=True)
    ok, st = check_tc(got["y"][rows], r, abs_sum(x64[rows], w64, b64), dtype)
    assert ok, st
    r = oracle.backward_dx(dyn, wn, m, k, n, dtype, rows=rows, out_f32=True)
    ok, st = check_tc(got["dx"][rows], r, abs_sum(dy64[rows], w64.T), dtype)
    assert ok, st
    r = oracle.backward_dw(xn, dyn, m, k, n, dtype, dw_f32=True, cols=cols)
    ok, st = check_tc(got["dw"][:, cols], r, abs_sum(x64.T, dy64[:, cols]), "f32")
    assert ok, st


@pytest.mark.parametrize("proj", synth.SEVEN_B, ids=lambda p: p[0])
def test_tc_7b_layer_sampled(eng, proj):
    name, k, n = proj
    m, dtype = synth.SEVEN_B_M, "bf16"
    x, w, dy, _ = synth.dense_inputs(m, k, n, dtype, x=("normal", 1.0), w=("normal", 0.02),
                                     dy=("normal", 1.0), b=None)
    got = run_dense(eng, x, w, dy, None, m, k, n, dtype, tc=1)
    xn, wn, dyn = np_in(x, w, dy)
    x64, w64, dy64 = (f64(a, dtype) for a in (xn, wn, dyn))
    rows = sample_rows(m, 6, seed=2)
    # dW: three sampled columns plus two of the last column tile, where the
    # tiles of the last, partial wave (contracted in chunks) lie
    cols = np.unique(np.concatenate([sample_rows(n, 3, seed=3), [n - 200, n - 1]]))
    r = oracle.forward(xn, wn, None, m, k, n, dtype, rows=rows, out_f32=True)
    ok, st = check_tc(got["y"][rows], r, abs_sum(x64[rows], w64), dtype)
    assert ok, st
    r = oracle.backward_dx(dyn, wn, m, k, n, dtype, rows=rows, out_f32=True)
    ok, st = check_tc(got["dx"][rows], r, abs_sum(dy64[rows], w64.T), dtype)
    assert ok, st
    r = oracle.backward_dw(xn, dyn, m, k, n, dtype, dw_f32=True, cols=cols)
    ok, st = check_tc(got["dw"][:, cols], r, abs_sum(x64.T, dy64[:, cols]), "f32")
    assert ok, st


def test_tc_f32_o_proj_sampled(eng):
    """3xTF32 at the f32 o-projection size 8192 x 4096 x 4096 (the bench's f32
    figure), sampled rows of Y / dX and columns of dW against the oracle."""
    m, k, n, dtype = synth.SEVEN_B_M, 4096, 4096, "f32"
    x, w, dy, b = synth.dense_inputs(m, k, n, dtype, b=("normal", 0.1))
    got = run_dense(eng, x, w, dy, b, m, k, n, dtype, tc=1)
    xn, wn, dyn, bn = np_in(x, w, dy, b)
    x64, w64, dy64, b64 = (f64(a, dtype) for a in (xn, wn, dyn, bn))
    rows = sample_rows(m, 6, seed=4)
    cols = sample_rows(n, 3, seed=5)
    r = oracle.forward(xn, wn, bn, m, k, n, dtype, rows=rows)
    ok, st = check_tc(got["y"][rows], r, abs_sum(x64[rows], w64, b64), dtype)
    assert ok, st
    r = oracle.backward_dx(dyn, wn, m, k, n, dtype, rows=rows)
    ok, st = check_tc(got["dx"][rows], r, abs_sum(dy64[rows], w64.T), dtype)
    assert ok, st
    r = oracle.backward_dw(xn, dyn, m, k, n, dtype, dw_f32=True, cols=cols)
    ok, st = check_tc(got["dw"][:, cols], r, abs_sum(x64.T, dy64[:, cols]), dtype)
    assert ok, st


@pytest.mark.parametrize("m,k,n", [(256, 13288, 264),   # forward: pieces 4096 x 3 + 1000
                                   (200, 136, 9000),    # dX: pieces 4096 x 2 + 808
                                   (8201, 132, 136)])   # dW: pieces 4096 x 2 + 9, padded ld
def test_tc_f32_long_contractions(eng, m, k, n):
    """3xTF32 over contractions longer than one 4096-element piece: every pass
    stays within the tolerance, and rows of Y / dX still do not depend on M."""
    dtype = "f32"
    x, w, dy, b = synth.dense_inputs(m, k, n, dtype, w=("normal", 1.0), b=("normal", 0.1))
    got = run_dense(eng, x, w, dy, b, m, k, n, dtype, tc=1)
    xn, wn, dyn, bn = np_in(x, w, dy, b)
    x64, w64, dy64, b64 = (f64(a, dtype) for a in (xn, wn, dyn, bn))
    rows = sample_rows(m, min(m, 24), seed=6)
    cols = sample_rows(n, min(n, 8), seed=7)
    r = oracle.forward(xn, wn, bn, m, k, n, dtype, rows=rows)
    ok, st = check_tc(got["y"][rows], r, abs_sum(x64[rows], w64, b64), dtype)
    assert ok, ("y", st)
    r = oracle.backward_dx(dyn, wn, m, k, n, dtype, rows=rows)
    ok, st = check_tc(got["dx"][rows], r, abs_sum(dy64[rows], w64.T), dtype)
    assert ok, ("dx", st)
    r = oracle.backward_dw(xn, dyn, m, k, n, dtype, dw_f32=True, cols=cols)
    ok, st = check_tc(got["dw"][:, cols], r, abs_sum(x64.T, dy64[:, cols]), dtype)
    assert ok, ("dw", st)
    mp = 3
    part = run_dense(eng, x[:mp].contiguous(), w, dy[:mp].contiguous(), b, mp, k, n, dtype, tc=1, passes=("y", "dx"))
    assert np.array_equal(part["y"], got["y"][:mp]) and np.array_equal(part["dx"], got["dx"][:mp])


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("tc", [0, 1])
def test_ten_runs_bit_identical(eng, tc, dtype):
    m, k, n = 1024, 768, 1536
    x, w, dy, b = synth.dense_inputs(m, k, n, dtype)
    first = run_dense(eng, x, w, dy, b, m, k, n, dtype, tc=tc)
    for _ in range(9):
        again = run_dense(eng, x, w, dy, b, m, k, n, dtype, tc=tc)
        for key in first:
            assert np.array_equal(first[key], again[key]), key


def test_batch_invariance_tc_7b_qkv(eng):
    """Rows of Y and dX on the tensor-core tier do not depend on M."""
    k, n, dtype = 4096, 12288, "bf16"
    M = synth.SEVEN_B_M
    x, w, dy, _ = synth.dense_inputs(M, k, n, dtype, b=None)
    full = run_dense(eng, x, w, dy, None, M, k, n, dtype, tc=1, passes=("y", "dx"))
    for mp in (1, 7, 64, 513):
        part = run_dense(eng, x[:mp].contiguous(), w, dy[:mp].contiguous(), None, mp, k, n, dtype, tc=1,
                         passes=("y", "dx"))
        assert np.array_equal(part["y"], full["y"][:mp]), mp
        assert np.array_equal(part["dx"], full["dx"][:mp]), mp


@pytest.mark.parametrize("dtype,tc", [("f32", 0), ("bf16", 0), ("f16", 1), ("bf16", 1), ("f32", 1)])
def test_batch_invariance_prefixes(eng, dtype, tc):
    m, k, n = 64, 256, 512
    x, w, dy, b = synth.dense_inputs(m, k, n, dtype, w=("normal", 1.0))
    full = run_dense(eng, x, w, dy, b, m, k, n, dtype, tc=tc, passes=("y", "dx"))
    for mp in (1, 17, 64):
        part = run_dense(eng, x[:mp].contiguous(), w, dy[:mp].contiguous(), b, mp, k, n, dtype, tc=tc,
                         passes=("y", "dx"))
        assert np.array_equal(part["y"], full["y"][:mp])
        assert np.array_equal(part["dx"], full["dx"][:mp])


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_batch_invariance_ragged_tiles(eng, dtype):
    """Rows of Y and dX do not depend on M where N and K end half-way through
    a column tile (N = 5.5 tiles, K = 1.5 tiles) and M is not a multiple of the
    256-row pair tile."""
    m, k, n = 700, 384, 1408
    x, w, dy, b = synth.dense_inputs(m, k, n, dtype)
    full = run_dense(eng, x, w, dy, b, m, k, n, dtype, tc=1, passes=("y", "dx"))
    for mp in (1, 7, 256, 300):
        part = run_dense(eng, x[:mp].contiguous(), w, dy[:mp].contiguous(), b, mp, k, n, dtype, tc=1,
                         passes=("y", "dx"))
        assert np.array_equal(part["y"], full["y"][:mp]), mp
        assert np.array_equal(part["dx"], full["dx"][:mp]), mp


# ------------------------------------------------------------------- edge cases and errors

def test_m_zero(eng):
    k, n = 128, 256
    y = torch.full((1, n), 7.0, dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(k, n, dtype=torch.bfloat16, device="cuda")
    x = torch.zeros(1, k, dtype=torch.bfloat16, device="cuda")
    for tc in (0, 1):
        eng.forward(y, x, w, None, 0, k, n, "bf16", None, tc)
        dw = torch.full((k, n), 5.0, dtype=torch.float32, device="cuda")
        eng.backward_dw(dw, 1, x, x, 0, k, n, "bf16", None, tc)
        eng.check()
        assert torch.all(y == 7.0)
        assert torch.all(dw == 0) and not torch.any(torch.signbit(dw))


DEGENERATE = [(1, 1, 1), (1, 1, 7), (3, 1, 5), (5, 7, 1), (300, 1, 200), (300, 200, 1), (1, 4096, 1),
              (2, 5, 3), (70, 3, 130), (4, 24, 1000)]


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_degenerate_shapes_bit_exact(eng, dtype):
    """Dimensions of 1 and a few: one-step chains (K = 1 forward, N = 1 dX,
    M = 1 dW), one-column and one-row outputs, through the matrix-vector,
    narrow and tiled kernels, bit-exact with the oracle."""
    for m, k, n in DEGENERATE:
        x, w, dy, b = synth.dense_inputs(m, k, n, dtype, w=("normal", 1.0))
        got = run_dense(eng, x, w, dy, b, m, k, n, dtype, tc=0)
        xn, wn, dyn, bn = np_in(x, w, dy, b)
        assert np.array_equal(got["y"], oracle.forward(xn, wn, bn, m, k, n, dtype)), (m, k, n)
        assert np.array_equal(got["dx"], oracle.backward_dx(dyn, wn, m, k, n, dtype)), (m, k, n)
        assert np.array_equal(got["dw"], oracle.backward_dw(xn, dyn, m, k, n, dtype, dw_f32=True)), (m, k, n)


def test_m_zero_dx_and_bias_grad(eng):
    """M = 0: dX (no rows) writes nothing; the bias gradient is +0."""
    k, n = 64, 136
    dx = torch.full((1, k), 7.0, dtype=torch.bfloat16, device="cuda")
    dy = torch.zeros(1, n, dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(k, n, dtype=torch.bfloat16, device="cuda")
    for tc in (0, 1):
        eng.backward_dx(dx, dy, w, 0, k, n, "bf16", None, tc)
        db = torch.full((n,), 5.0, dtype=torch.float32, device="cuda")
        eng.bias_grad(db, 1, dy, 0, n, "bf16")
        eng.check()
        assert torch.all(dx == 7.0)
        assert torch.all(db == 0) and not torch.any(torch.signbit(db))


def test_errors_are_reported(eng):
    h = eng.handle
    x = torch.zeros(16, 128, dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(128, 128, dtype=torch.bfloat16, device="cuda")
    y = torch.zeros(17, 128, dtype=torch.bfloat16, device="cuda")
    assert bi.bi_forward(h, y, x, w, None, 16, 0, 128, "bf16", None, 1) == bi.BI_ERR_INVALID_ARG
    assert bi.bi_forward(h, y, x, w, None, 16, 128, 128, 7, None, 1) == bi.BI_ERR_INVALID_ARG
    assert bi.bi_forward(h, None, x, w, None, 16, 128, 128, "bf16", None, 1) == bi.BI_ERR_INVALID_ARG
    assert bi.bi_forward(h, y, x, w, None, -1, 128, 128, "bf16", None, 1) == bi.BI_ERR_INVALID_ARG
    # misaligned output with the tensor-core tier selected
    st = bi.bi_forward(h, y.view(-1)[1:].data_ptr(), x, w, None, 16, 128, 128, "bf16", None, 1)
    assert st == bi.BI_ERR_MISALIGNED, bi.bi_last_error(h)
    assert "aligned" in bi.bi_last_error(h)
    # the scalar tier accepts the same misaligned pointer
    assert bi.bi_forward(h, y.view(-1)[1:].data_ptr(), x, w, None, 16, 128, 128, "bf16", None, 0) == bi.BI_OK
    eng.check()


def test_timeout_path_reports_and_recovers(eng):
    h = eng.handle
    assert bi.bi_engine_set_wait_limit(h, 20_000_000) == bi.BI_OK  # 20 ms
    assert bi.bi_selftest_wait_timeout(h, None) == bi.BI_OK
    assert bi.bi_engine_check(h, None) == bi.BI_ERR_TIMEOUT
    assert "self-test" in bi.bi_last_error(h)
    assert bi.bi_engine_set_wait_limit(h, 0) == bi.BI_OK
    # the context is still usable and the status word was cleared
    assert bi.bi_engine_check(h, None) == bi.BI_OK
    m, k, n = 128, 128, 256
    x, w, dy, b = synth.dense_inputs(m, k, n, "bf16")
    got = run_dense(eng, x, w, dy, b, m, k, n, "bf16", tc=1, passes=("y",))
    assert got["y"].shape == (m, n)


def test_launch_count_counts_kernels(eng):
    m, k, n = 128, 128, 256
    x, w, dy, b = synth.dense_inputs(m, k, n, "bf16")
    before = eng.launches()
    run_dense(eng, x, w, dy, b, m, k, n, "bf16", tc=1)
    assert eng.launches() - before == 3  # one tcgen05 kernel per pass
    before = eng.launches()
    run_dense(eng, x, w, dy, b, m, k, n, "bf16", tc=0, passes=("y", "dx"))
    assert eng.launches() - before == 2


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_tc_dw_tail_tiles_in_chunks(eng, dtype):
    """dW tiles of the last, partial wave run their contraction as chunks added
    by the dW tree.  1024 x 2048 x 2560: 80 tiles of 256 x 256, the last 4 (rows
    1024-2047, columns 2304-2559) in 2 chunks of 512 rows; checked there and on
    whole tiles, f32 and rounded, and run to run.  2048 x 256 x 2048: 16 tiles of
    256 x 128, each in 4 chunks of 512 rows, exact on small integers, and the
    chunk order: chunk results 2^24, 1, 1, -2^24 give (c0 + c1) + (c2 + c3) = 1
    by the pairwise tree (2^24 + 1 rounds to 2^24), where adding them one by
    one would give 0."""
    m, k, n = 1024, 2048, 2560
    x, _, dy, _ = synth.dense_inputs(m, k, n, dtype, b=None)
    got = run_dense(eng, x, None, dy, None, m, k, n, dtype, tc=1, passes=("dw",))
    got_r = run_dense(eng, x, None, dy, None, m, k, n, dtype, tc=1, dw_f32=False, passes=("dw",))
    xn, dyn = synth.to_np(x), synth.to_np(dy)
    x64, dy64 = f64(xn, dtype), f64(dyn, dtype)
    cols = np.concatenate([np.arange(2304, 2560), sample_rows(2304, 24, seed=4)])
    r = oracle.backward_dw(xn, dyn, m, k, n, dtype, dw_f32=True, cols=cols)
    S = abs_sum(x64.T, dy64[:, cols])
    ok, st = check_tc(got["dw"][:, cols], r, S, "f32")
    assert ok, st
    ok, st = check_tc(got_r["dw"][:, cols], r, S, dtype)
    assert ok, st
    again = run_dense(eng, x, None, dy, None, m, k, n, dtype, tc=1, passes=("dw",))
    assert np.array_equal(again["dw"], got["dw"])
    m, k, n = 2048, 256, 2048
    hi = 16 if dtype == "f16" else 8
    xi = synth.small_ints((m, k), -hi, hi, dtype, 97)
    gi = synth.small_ints((m, n), -2, 2, dtype, 98)  # every partial sum exact in f32
    got = run_dense(eng, xi, None, gi, None, m, k, n, dtype, tc=1, passes=("dw",))
    assert np.array_equal(got["dw"], oracle.backward_dw(synth.to_np(xi), synth.to_np(gi), m, k, n, dtype, dw_f32=True))
    k0, n0 = 5, 700
    xa, ga = np.zeros((m, k)), np.zeros((m, n))
    xa[:512, k0], ga[:512, n0] = 64.0, 512.0          # chunk 0: 512 * 2^15 = 2^24, every partial sum exact
    xa[600, k0], ga[600, n0] = 1.0, 1.0                # chunk 1: 1
    xa[1100, k0], ga[1100, n0] = 1.0, 1.0              # chunk 2: 1
    xa[1536:, k0], ga[1536:, n0] = 64.0, -512.0        # chunk 3: -2^24
    xt, gt = (torch.from_numpy(a).to(synth.TORCH_DTYPES[dtype]) for a in (xa, ga))  # all values exact
    got = run_dense(eng, xt, None, gt, None, m, k, n, dtype, tc=1, passes=("dw",))
    want = np.zeros((k, n), dtype=np.float32)
    want[k0, n0] = 1.0
    assert np.array_equal(got["dw"], want)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_tc_dw_f32_in_pieces(eng, dtype):
    """dW kept in f32 over more rows than one 8192-row piece (8192 + 8192 + 3616):
    exact on small integers, within the tolerance on random data, and the rounded
    dW (one launch over all rows) within 1 ulp."""
    m, k, n = 20000, 64, 136
    hi = 16 if dtype == "f16" else 8
    xi = synth.small_ints((m, k), -hi, hi, dtype, 95)
    gi = synth.small_ints((m, n), -2, 2, dtype, 96)  # keeps every partial sum exact in f32
    got = run_dense(eng, xi, None, gi, None, m, k, n, dtype, tc=1, passes=("dw",))
    assert np.array_equal(got["dw"], oracle.backward_dw(synth.to_np(xi), synth.to_np(gi), m, k, n, dtype, dw_f32=True))
    x, _, dy, _ = synth.dense_inputs(m, k, n, dtype, b=None)
    got = run_dense(eng, x, None, dy, None, m, k, n, dtype, tc=1, passes=("dw",))
    xn, dyn = synth.to_np(x), synth.to_np(dy)
    x64, dy64 = f64(xn, dtype), f64(dyn, dtype)
    r = oracle.backward_dw(xn, dyn, m, k, n, dtype, dw_f32=True)
    ok, st = check_tc(got["dw"], r, abs_sum(x64.T, dy64), "f32")
    assert ok, st
    got_r = run_dense(eng, x, None, dy, None, m, k, n, dtype, tc=1, dw_f32=False, passes=("dw",))
    ok, st = check_tc(got_r["dw"], r, abs_sum(x64.T, dy64), dtype)
    assert ok, st
