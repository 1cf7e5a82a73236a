"""Pins for the CPU oracle: checks against facts that do not come from the oracle.

* hand-derived fixtures under tests/golden (chain order, fused multiply-add,
  bias rounding, the dW chunk tree, IEEE rounding points);
* exhaustive agreement of the format code with torch's own conversions;
* exact small-integer problems, whose result is rne(exact integer matmul)
  whatever the summation order;
* the forward error bound of a recursive sum (gamma_L times the sum of |a*b|);
* finite differences of f = sum(Y * G), which fix the gradient formulas and
  operand layouts of dX, dW and the grouped passes;
* invariants (row-prefix invariance, grouped E=1 equals dense, padding rows);
* brute force on every shape up to 3 x 3 x 3: each fused multiply-add of the
  chain evaluated in exact rational arithmetic and rounded to nearest-even
  f32, then the bias add and the output rounding the same way.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from deterministic_invariant_gemm_fixed_gb300 import synth
from conftest import read_golden

DT = ["f32", "bf16", "f16"]


def enc(values, dtype):
    """Exact encodings of float values in the operand type (via torch)."""
    t = torch.tensor(np.asarray(values, dtype=np.float64)).to(synth.TORCH_DTYPES[dtype])
    return synth.to_np(t)


def dec(a, dtype):
    """Operand data -> float64 values."""
    if dtype == "f32":
        return a.astype(np.float64)
    return synth.from_np(a, dtype).to(torch.float64).numpy()


def as_f32_bits(a):
    return np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)


# --------------------------------------------------------------------------- golden fixtures

@pytest.mark.parametrize("dtype", DT)
def test_golden_chain_order(dtype):
    kv, _ = read_golden("chain_order.txt")
    x = enc([float(v) for v in kv["x"][0].split()], dtype)
    w = enc([float(v) for v in kv["w"][0].split()], dtype)
    y = oracle.forward(x, w, None, 1, 3, 1, dtype, out_f32=True)
    assert y[0, 0] == float(kv["y_ascending"][0])
    # the reverse order gives another value, so the fixture separates the two
    yr = oracle.forward(x[::-1].copy(), w[::-1].copy(), None, 1, 3, 1, dtype, out_f32=True)
    assert yr[0, 0] == float(kv["y_descending"][0])


def test_golden_fma_not_mul_add():
    kv, _ = read_golden("fma_vs_muladd.txt")
    x = np.array([int(v, 16) for v in kv["x"][0].split()], dtype=np.uint32).view(np.float32)
    w = np.array([int(v, 16) for v in kv["w"][0].split()], dtype=np.uint32).view(np.float32)
    y = oracle.forward(x.copy(), w.copy(), None, 1, 2, 1, "f32")
    assert as_f32_bits(y)[0, 0] == int(kv["y_fma"][0], 16)
    # the same data through a product-then-add chain gives the other value
    p = np.float32(x[0]) * np.float32(w[0])
    q = np.float32(x[1]) * np.float32(w[1])
    assert np.float32(np.float32(0) + p + q).view(np.uint32) == int(kv["y_mul_then_add"][0], 16)


def test_golden_bias_single_rounding():
    kv, _ = read_golden("bias_single_rounding.txt")
    x = enc([float(v) for v in kv["x"][0].split()], "bf16")
    w = enc([float(v) for v in kv["w"][0].split()], "bf16")
    b = enc([float(kv["b"][0])], "bf16")
    y = oracle.forward(x, w, b, 1, 2, 1, "bf16")
    assert y[0, 0] == int(kv["y_bits_single"][0], 16)
    assert int(kv["y_bits_single"][0], 16) != int(kv["y_bits_double"][0], 16)


@pytest.mark.parametrize("dtype", DT)
def test_golden_dw_tree(dtype):
    kv, _ = read_golden("dw_tree.txt")
    for case in kv["case"]:
        c, xs, dys, want = [s.strip() for s in case.split("|")]
        xv = [float(v) for v in xs.split()]
        dyv = [float(v) for v in dys.split()]
        m = len(xv)
        x, dy = enc(xv, dtype), enc(dyv, dtype)
        got = oracle.backward_dw(x, dy, m, 1, 1, dtype, dw_f32=True, chunk=int(c))
        assert got[0, 0] == float(want), (case, got[0, 0])
        got_t = oracle.backward_dw(x, dy, m, 1, 1, dtype, dw_f32=False, chunk=int(c))
        assert dec(got_t, dtype)[0, 0] == float(want)


def test_golden_tree_sum_values():
    # the same tree on raw partials (level pairing, odd last entry carried)
    t24 = 2.0 ** 24
    assert oracle.tree_sum([]) == 0.0
    assert oracle.tree_sum([5.0]) == 5.0
    assert oracle.tree_sum([1.0, t24, -t24]) == 0.0
    assert oracle.tree_sum([1.0, t24, -t24, 1.0, 1.0]) == 2.0
    assert oracle.tree_sum([t24, 1.0, 1.0, -t24, 1.0, 1.0]) == 3.0


def test_golden_rne_points():
    _, rows = read_golden("rne_points.txt")
    assert len(rows) > 20
    for dtype, fbits, want in rows:
        f = np.array([int(fbits, 16)], dtype=np.uint32).view(np.float32)
        got = oracle.rne(f, dtype)[0]
        assert got == int(want, 16), (dtype, fbits, hex(got), want)


# --------------------------------------------------------------------------- format code vs torch

@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_rne_exhaustive_vs_torch(dtype):
    """Every one of the 2^32 binary32 patterns rounds as torch rounds it
    (NaN inputs: both sides give a NaN; payloads are not compared)."""
    tdt = synth.TORCH_DTYPES[dtype]
    chunk = 1 << 25
    base = np.arange(chunk, dtype=np.uint32)
    buf = np.empty(chunk, dtype=np.uint16)
    for start in range(0, 1 << 32, chunk):
        bits = base + np.uint32(start)
        ours = oracle.rne_bits_range(start, chunk, dtype, out=buf)
        theirs = torch.from_numpy(bits.view(np.float32)).to(tdt).view(torch.int16).numpy().view(np.uint16)
        diff = ours != theirs
        if diff.any():
            f = bits.view(np.float32)[diff]
            assert np.isnan(f).all(), (dtype, hex(int(bits[diff][0])))
            o = ours[diff]
            expo = 0x7f80 if dtype == "bf16" else 0x7c00
            assert ((o & expo) == expo).all() and ((o & (0x7f if dtype == "bf16" else 0x3ff)) != 0).all()


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_up_exhaustive_vs_torch(dtype):
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ours = oracle.up(h, dtype)
    theirs = synth.from_np(h, dtype).to(torch.float32).numpy()
    nan = np.isnan(theirs)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan].view(np.uint32), theirs[~nan].view(np.uint32))
    # round trip: rne(up(h)) == h for every non-NaN encoding
    back = oracle.rne(ours, dtype)
    assert np.array_equal(back[~nan], h[~nan])


# --------------------------------------------------------------------------- exact integers

def int_problem(m, k, n, dtype, seed, lo=-8, hi=8):
    x = synth.small_ints((m, k), lo, hi, dtype, seed)
    w = synth.small_ints((k, n), lo, hi, dtype, seed + 1)
    dy = synth.small_ints((m, n), lo, hi, dtype, seed + 2)
    # bias in halves: rounding before vs after the add differs on many outputs
    b = (synth.small_ints((n,), -128, 127, "f32", seed + 3) / 2).to(synth.TORCH_DTYPES[dtype])
    return [synth.to_np(t) for t in (x, w, dy, b)]


def round_exact(v64, dtype):
    """Round exact (integer or half-integer, |v| < 2^24) values to the dtype via torch."""
    return synth.to_np(torch.from_numpy(np.ascontiguousarray(v64)).to(synth.TORCH_DTYPES[dtype]))


@pytest.mark.parametrize("dtype", DT)
def test_exact_integer_dense(dtype):
    m, k, n = 37, 300, 45
    # f16 holds every integer and half below 2048 exactly: use a wider range so
    # that the outputs reach the binades where rounding happens
    hi = 16 if dtype == "f16" else 8
    x, w, dy, b = int_problem(m, k, n, dtype, seed=11, lo=-hi, hi=hi)
    xi, wi, dyi, bf = dec(x, dtype), dec(w, dtype), dec(dy, dtype), dec(b, dtype)
    y = oracle.forward(x, w, b, m, k, n, dtype)
    assert np.array_equal(y, round_exact(xi @ wi + bf, dtype))
    dx = oracle.backward_dx(dy, w, m, k, n, dtype)
    assert np.array_equal(dx, round_exact(dyi @ wi.T, dtype))
    for chunk in (1, 7, 16, 256):
        dw = oracle.backward_dw(x, dy, m, k, n, dtype, dw_f32=False, chunk=chunk)
        assert np.array_equal(dw, round_exact(xi.T @ dyi, dtype))
        dwf = oracle.backward_dw(x, dy, m, k, n, dtype, dw_f32=True, chunk=chunk)
        assert np.array_equal(dwf, (xi.T @ dyi).astype(np.float32))
    if dtype != "f32":
        # rounding the accumulator before the bias would differ somewhere
        twice = round_exact(dec(round_exact(xi @ wi, dtype), dtype) + bf, dtype)
        assert not np.array_equal(y, twice)


@pytest.mark.parametrize("dtype", DT)
def test_exact_integer_grouped(dtype):
    m, k, n, e = 200, 96, 40, 5
    x = synth.to_np(synth.small_ints((m, k), -8, 8, dtype, 21))
    w = synth.to_np(synth.small_ints((e, n, k), -8, 8, dtype, 22))
    dy = synth.to_np(synth.small_ints((m, n), -8, 8, dtype, 23))
    ids = synth.to_np(synth.expert_ids(m, e, 0.1, 24))
    ids[3] = e + 7           # an id beyond E is padding too
    ids[ids == 2] = 0        # expert 2 has no rows
    xi, wi, dyi = dec(x, dtype), dec(w, dtype), dec(dy, dtype)
    valid = ids < e
    y_ref = np.zeros((m, n))
    dx_ref = np.zeros((m, k))
    dw_ref = np.zeros((e, n, k))
    for r in range(m):
        if valid[r]:
            y_ref[r] = wi[ids[r]] @ xi[r]
            dx_ref[r] = dyi[r] @ wi[ids[r]]
            dw_ref[ids[r]] += np.outer(dyi[r], xi[r])
    y = oracle.grouped_forward(x, w, ids, m, k, n, e, dtype)
    assert np.array_equal(y, round_exact(y_ref, dtype))
    dx = oracle.grouped_dinput(w, dy, ids, m, k, n, e, dtype)
    assert np.array_equal(dx, round_exact(dx_ref, dtype))
    for chunk in (1, 5, 256):
        dw = oracle.grouped_dweights(x, dy, ids, m, k, n, e, dtype, chunk=chunk)
        assert np.array_equal(dw, dw_ref.astype(np.float32))
    assert np.all(dw[2] == 0) and not np.signbit(dw[2]).any()
    # padding rows are +0 (all bits zero)
    assert np.all(y[~valid] == 0) and np.all(dx[~valid] == 0)
    assert not np.signbit(dec(y[~valid], dtype)).any()


# --------------------------------------------------------------------------- error bound

def gamma(L):
    u = 2.0 ** -24
    return L * u / (1 - L * u)


@pytest.mark.parametrize("dtype", DT)
def test_error_bound_dense(dtype):
    m, k, n = 24, 1000, 40
    x, w, dy, b = [synth.to_np(t) for t in synth.dense_inputs(m, k, n, dtype, w=("normal", 1.0))]
    xf, wf, dyf, bf = (dec(a, dtype) for a in (x, w, dy, b))
    y = oracle.forward(x, w, b, m, k, n, dtype, out_f32=True).astype(np.float64)
    ref = xf @ wf + bf
    s = np.abs(xf) @ np.abs(wf) + np.abs(bf)
    assert np.all(np.abs(y - ref) <= gamma(k + 1) * s)
    dx = oracle.backward_dx(dy, w, m, k, n, dtype, out_f32=True).astype(np.float64)
    assert np.all(np.abs(dx - dyf @ wf.T) <= gamma(n) * (np.abs(dyf) @ np.abs(wf).T))
    for chunk in (4, 256):
        dw = oracle.backward_dw(x, dy, m, k, n, dtype, dw_f32=True, chunk=chunk).astype(np.float64)
        depth = min(chunk, m) + math.ceil(math.log2(max(1, -(-m // chunk))))
        assert np.all(np.abs(dw - xf.T @ dyf) <= gamma(depth) * (np.abs(xf).T @ np.abs(dyf)))


def test_error_bound_is_not_vacuous():
    # a plausible slip (dropping the last term of every chain) breaks the bound
    m, k, n = 8, 64, 8
    x, w, _, _ = [synth.to_np(t) for t in synth.dense_inputs(m, k, n, "f32", w=("normal", 1.0))]
    y = oracle.forward(x[:, :-1].copy(), w[:-1].copy(), None, m, k - 1, n, "f32", out_f32=True)
    ref = x.astype(np.float64) @ w.astype(np.float64)
    s = np.abs(x.astype(np.float64)) @ np.abs(w.astype(np.float64))
    assert not np.all(np.abs(y - ref) <= gamma(k) * s)


# --------------------------------------------------------------------------- finite differences

def f_sum(y, g):
    return float(np.sum(y.astype(np.float64) * g.astype(np.float64)))


def test_finite_differences_dense():
    m, k, n = 6, 50, 9
    x, w, g, _ = [synth.to_np(t) for t in synth.dense_inputs(m, k, n, "f32", w=("normal", 1.0))]
    dx = oracle.backward_dx(g, w, m, k, n, "f32")
    dw = oracle.backward_dw(x, g, m, k, n, "f32", dw_f32=True)
    h = np.float32(0.5)  # Y is linear in X and W: no truncation error
    rng = np.random.default_rng(0)
    for _ in range(12):
        i, j = rng.integers(m), rng.integers(k)
        xp, xm = x.copy(), x.copy()
        xp[i, j] += h; xm[i, j] -= h
        fd = (f_sum(oracle.forward(xp, w, None, m, k, n, "f32"), g)
              - f_sum(oracle.forward(xm, w, None, m, k, n, "f32"), g)) / (2 * h)
        assert abs(fd - dx[i, j]) <= 1e-4 * (1 + abs(dx[i, j])), (i, j, fd, dx[i, j])
        i, j = rng.integers(k), rng.integers(n)
        wp, wm = w.copy(), w.copy()
        wp[i, j] += h; wm[i, j] -= h
        fd = (f_sum(oracle.forward(x, wp, None, m, k, n, "f32"), g)
              - f_sum(oracle.forward(x, wm, None, m, k, n, "f32"), g)) / (2 * h)
        assert abs(fd - dw[i, j]) <= 1e-4 * (1 + abs(dw[i, j])), (i, j, fd, dw[i, j])


def test_finite_differences_grouped():
    m, k, n, e = 30, 20, 7, 3
    x, w, g, ids = synth.grouped_inputs(m, k, n, e, "f32", pad_frac=0.1, w=("normal", 1.0))
    x, w, g, ids = synth.to_np(x), synth.to_np(w), synth.to_np(g), synth.to_np(ids)
    dx = oracle.grouped_dinput(w, g, ids, m, k, n, e, "f32")
    dw = oracle.grouped_dweights(x, g, ids, m, k, n, e, "f32")
    h = np.float32(0.5)
    rng = np.random.default_rng(1)

    def f(xx, ww):
        return f_sum(oracle.grouped_forward(xx, ww, ids, m, k, n, e, "f32"), g)

    for _ in range(12):
        i, j = rng.integers(m), rng.integers(k)
        xp, xm = x.copy(), x.copy()
        xp[i, j] += h; xm[i, j] -= h
        fd = (f(xp, w) - f(xm, w)) / (2 * h)
        assert abs(fd - dx[i, j]) <= 1e-4 * (1 + abs(dx[i, j]))
        a, b_, c = rng.integers(e), rng.integers(n), rng.integers(k)
        wp, wm = w.copy(), w.copy()
        wp[a, b_, c] += h; wm[a, b_, c] -= h
        fd = (f(x, wp) - f(x, wm)) / (2 * h)
        assert abs(fd - dw[a, b_, c]) <= 1e-4 * (1 + abs(dw[a, b_, c]))


# --------------------------------------------------------------------------- invariants

@pytest.mark.parametrize("dtype", DT)
def test_row_prefix_invariance(dtype):
    m, k, n = 64, 256, 512
    x, w, dy, b = [synth.to_np(t) for t in synth.dense_inputs(m, k, n, dtype)]
    y = oracle.forward(x, w, b, m, k, n, dtype)
    dx = oracle.backward_dx(dy, w, m, k, n, dtype)
    for mp in (1, 17, 64):
        assert np.array_equal(oracle.forward(x[:mp].copy(), w, b, mp, k, n, dtype), y[:mp])
        assert np.array_equal(oracle.backward_dx(dy[:mp].copy(), w, mp, k, n, dtype), dx[:mp])
    rows = [5, 63, 0]
    assert np.array_equal(oracle.forward(x, w, b, m, k, n, dtype, rows=rows), y[rows])


@pytest.mark.parametrize("dtype", DT)
def test_scalar_contract_is_upcast_f32_then_rne(dtype):
    """bf16/f16 results equal torch's round-to-nearest of the f32 computation on
    exactly widened operands (sgemm-bi, "Determinism contracts", first row)."""
    if dtype == "f32":
        pytest.skip("f32 is the f32 computation itself")
    m, k, n = 16, 128, 64
    x, w, dy, b = [synth.to_np(t) for t in synth.dense_inputs(m, k, n, dtype)]
    up = {a_name: oracle.up(a, dtype) for a_name, a in (("x", x), ("w", w), ("dy", dy), ("b", b))}
    tdt = synth.TORCH_DTYPES[dtype]

    def torch_rne(a32):
        return synth.to_np(torch.from_numpy(a32).to(tdt))

    y32 = oracle.forward(up["x"], up["w"], up["b"], m, k, n, "f32")
    assert np.array_equal(oracle.forward(x, w, b, m, k, n, dtype), torch_rne(y32))
    dx32 = oracle.backward_dx(up["dy"], up["w"], m, k, n, "f32")
    assert np.array_equal(oracle.backward_dx(dy, w, m, k, n, dtype), torch_rne(dx32))
    dw32 = oracle.backward_dw(up["x"], up["dy"], m, k, n, "f32", dw_f32=True)
    assert np.array_equal(oracle.backward_dw(x, dy, m, k, n, dtype), torch_rne(dw32))


def test_k1_is_one_rounded_product():
    """With K=1 the chain is fmaf(x, w, +0) = the correctly rounded product,
    i.e. numpy's float32 multiply; the bias is one more float32 add."""
    m, n = 50, 60
    x, w, _, b = [synth.to_np(t) for t in synth.dense_inputs(m, 1, n, "f32", w=("normal", 1.0))]
    y = oracle.forward(x, w, b, m, 1, n, "f32")
    ref = (x.reshape(m, 1) * w.reshape(1, n)).astype(np.float32) + b.reshape(1, n)
    assert np.array_equal(y.view(np.uint32), ref.astype(np.float32).view(np.uint32))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_chains_keep_a_negative_zero(dtype):
    """Signed zeros through the chain.  Every product -1e-30 * 1e-20 lies far
    below the smallest f32 subnormal, so round to nearest gives -0 for the
    first fused multiply-add, RN(-1e-50 + +0) = -0, and for every later one,
    RN(-1e-50 + -0) = -0: each output of Y, dX and dW (every chunk and every
    tree sum, -0 + -0 = -0) is -0.  A product that is an exact zero instead
    gives RN(-0 + +0) = +0, so the all-zero contraction is +0."""
    m, k, n = 5, 37, 6  # dW over 5 rows; also a dW tree over chunks of 2 rows
    neg, pos = enc([-1e-30], dtype)[0], enc([1e-20], dtype)[0]
    x = np.full(m * k, neg, dtype=neg.dtype)
    w = np.full(k * n, pos, dtype=pos.dtype)
    dy_dx = np.full(m * n, neg, dtype=neg.dtype)
    dy_dw = np.full(m * n, enc([1e-30], dtype)[0], dtype=neg.dtype)
    outs = [oracle.forward(x, w, None, m, k, n, dtype, out_f32=True),
            oracle.backward_dx(dy_dx, w, m, k, n, dtype, out_f32=True),
            oracle.backward_dw(x, dy_dw, m, k, n, dtype, dw_f32=True),
            oracle.backward_dw(x, dy_dw, m, k, n, dtype, dw_f32=True, chunk=2)]
    for o in outs:
        assert np.all(o == 0) and np.all(np.signbit(o))
    zx = np.full(m * k, enc([-0.0], dtype)[0], dtype=neg.dtype)  # -0 * w: exact zero products
    y0 = oracle.forward(zx, w, None, m, k, n, dtype, out_f32=True)
    assert np.all(y0 == 0) and not np.any(np.signbit(y0))


@pytest.mark.parametrize("dtype", DT)
def test_dw_large_chunk_is_plain_chain(dtype):
    m, k, n = 40, 24, 31
    x, _, dy, _ = [synth.to_np(t) for t in synth.dense_inputs(m, k, n, dtype)]
    dw = oracle.backward_dw(x, dy, m, k, n, dtype, dw_f32=True, chunk=m)
    # dW = X^T dY as a forward over the transposed X: the same chain over rows
    xt = np.ascontiguousarray(x.reshape(m, k).T)
    assert np.array_equal(dw, oracle.forward(xt, dy, None, k, m, n, dtype, out_f32=True))
    cols = [30, 0, 7]
    assert np.array_equal(oracle.backward_dw(x, dy, m, k, n, dtype, dw_f32=True, chunk=m, cols=cols),
                          dw[:, cols])


def test_dw_zero_row_of_dy_changes_nothing():
    m, k, n = 600, 8, 8
    x, _, dy, _ = [synth.to_np(t) for t in synth.dense_inputs(m, k, n, "bf16")]
    dw = oracle.backward_dw(x, dy, m, k, n, "bf16", dw_f32=True)
    dy2 = dy.copy()
    dy2[300] = 0
    x2 = x.copy()
    x2[300] = enc(np.full(k, 3.0), "bf16")
    base = oracle.backward_dw(x2, dy2, m, k, n, "bf16", dw_f32=True)
    x3 = x.copy()
    x3[300] = enc(np.full(k, -5.0), "bf16")
    assert np.array_equal(base, oracle.backward_dw(x3, dy2, m, k, n, "bf16", dw_f32=True))
    assert not np.array_equal(dw, base)


@pytest.mark.parametrize("dtype", DT)
def test_grouped_single_expert_equals_dense(dtype):
    m, k, n = 300, 48, 40
    x, w, dy, _ = synth.grouped_inputs(m, k, n, 1, dtype, pad_frac=0.0)
    x, w, dy = synth.to_np(x), synth.to_np(w), synth.to_np(dy)
    ids = np.zeros(m, dtype=np.uint32)
    wd = np.ascontiguousarray(w.reshape(n, k).T)  # dense W[K,N] = W[0]^T
    assert np.array_equal(oracle.grouped_forward(x, w, ids, m, k, n, 1, dtype),
                          oracle.forward(x, wd, None, m, k, n, dtype))
    assert np.array_equal(oracle.grouped_dinput(w, dy, ids, m, k, n, 1, dtype),
                          oracle.backward_dx(dy, wd, m, k, n, dtype))
    dwg = oracle.grouped_dweights(x, dy, ids, m, k, n, 1, dtype)
    dwd = oracle.backward_dw(x, dy, m, k, n, dtype, dw_f32=True)
    assert np.array_equal(dwg[0], dwd.T)


def test_grouped_padding_rows_do_not_touch_dweights():
    m, k, n, e = 700, 16, 12, 4
    x, w, dy, ids = synth.grouped_inputs(m, k, n, e, "bf16", pad_frac=0.2)
    x, w, dy, ids = synth.to_np(x), synth.to_np(w), synth.to_np(dy), synth.to_np(ids)
    keep = ids < e
    full = oracle.grouped_dweights(x, dy, ids, m, k, n, e, "bf16")
    mk = int(keep.sum())
    kept = oracle.grouped_dweights(x[keep].copy(), dy[keep].copy(), ids[keep].copy(), mk, k, n, e, "bf16")
    assert np.array_equal(full, kept)
    sel = ([0, 3, 1], [11, 0, 5])
    assert np.array_equal(oracle.grouped_dweights(x, dy, ids, m, k, n, e, "bf16", sel=sel),
                          full[sel[0], sel[1]])


def test_row_permutation_permutes_outputs():
    m, k, n = 33, 64, 20
    x, w, _, b = [synth.to_np(t) for t in synth.dense_inputs(m, k, n, "bf16")]
    p = np.random.default_rng(3).permutation(m)
    y = oracle.forward(x, w, b, m, k, n, "bf16")
    assert np.array_equal(oracle.forward(x[p].copy(), w, b, m, k, n, "bf16"), y[p])


def test_segment_matches_stable_argsort():
    m, e = 5000, 9
    ids = synth.to_np(synth.expert_ids(m, e, 0.05, 7))
    ids[10] = 1 << 31
    perm, offs = oracle.grouped_segment(ids, m, e)
    bucket = np.minimum(ids.astype(np.int64), e)
    assert np.array_equal(perm, np.argsort(bucket, kind="stable"))
    counts = np.bincount(bucket, minlength=e + 1)
    assert np.array_equal(offs, np.concatenate([[0], np.cumsum(counts)]).astype(np.uint32))


# --------------------------------------------------------------------------- bias gradient

@pytest.mark.parametrize("dtype", DT)
def test_bias_grad_exact_integers_and_dw_identity(dtype):
    m, n = 700, 37
    dy = synth.to_np(synth.small_ints((m, n), -8, 8, dtype, 41))
    want = dec(dy, dtype).sum(axis=0)
    for chunk in (1, 7, 256):
        assert np.array_equal(oracle.bias_grad(dy, m, n, dtype, out_f32=True, chunk=chunk),
                              want.astype(np.float32))
    # on any data it is dW with a column of ones for X (fmaf(1, g, acc) = acc + g)
    g = synth.to_np(synth.normal((m, n), 1.0, dtype, 42))
    ones = enc(np.ones(m), dtype)
    for chunk in (5, 256):
        dw = oracle.backward_dw(ones, g, m, 1, n, dtype, dw_f32=True, chunk=chunk)[0]
        assert np.array_equal(oracle.bias_grad(g, m, n, dtype, out_f32=True, chunk=chunk), dw)
    assert np.array_equal(oracle.bias_grad(g, m, n, dtype),
                          oracle.backward_dw(ones, g, m, 1, n, dtype)[0])


def test_bias_grad_golden_tree():
    kv, _ = read_golden("dw_tree.txt")
    for case in kv["case"]:
        c, xs, dys, want = [s_.strip() for s_ in case.split("|")]
        prod = [float(a) * float(b) for a, b in zip(xs.split(), dys.split())]
        g = np.array(prod, dtype=np.float32)
        got = oracle.bias_grad(g, g.size, 1, "f32", out_f32=True, chunk=int(c))
        assert got[0] == float(want), case


def test_bias_grad_empty_is_zero():
    assert np.array_equal(oracle.bias_grad(np.zeros(0, np.float32), 0, 3, "f32"), np.zeros(3, np.float32))


# --------------------------------------------------------------------------- FP8 e4m3

def test_golden_e4m3_points():
    _, rows = read_golden("e4m3_points.txt")
    assert len(rows) > 15
    for fbits, want in rows:
        got = oracle.e4m3_bits_range(int(fbits, 16), 1)[0]
        assert got == int(want, 16), (fbits, hex(got), want)


def test_e4m3_exhaustive_vs_torch():
    """Every binary32 pattern: for exponents 2^-11 .. 2^9 (where e4m3 has distinct
    codes) the result equals torch's float8_e4m3fn rounding wherever |v| <= 464;
    beyond 464 (where torch gives NaN) this format saturates to +-448, the
    saturating cast of the FP8 design; below 2^-11 everything rounds to +-0;
    NaN stays NaN."""
    frac = np.arange(1 << 23, dtype=np.uint32)
    for sign in (0, 1):
        for ef in range(256):
            start = (sign << 31) | (ef << 23)
            bits = frac | np.uint32(start)
            ours = oracle.e4m3_bits_range(start, 1 << 23)
            if ef == 255:  # inf (frac 0) saturates, NaN stays NaN
                assert ours[0] == (0xfe if sign else 0x7e)
                assert np.all((ours[1:] & 0x7f) == 0x7f)
            elif ef < 116:  # |v| < 2^-11: below half the smallest subnormal
                assert np.all(ours == (0x80 if sign else 0))
            elif ef > 136:  # |v| >= 2^10 > 464
                assert np.all(ours == (0xfe if sign else 0x7e))
            else:
                f = bits.view(np.float32)
                theirs = torch.from_numpy(f).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
                inrange = np.abs(f) <= 464
                assert np.array_equal(ours[inrange], theirs[inrange]), (sign, ef)
                assert np.all((ours[~inrange] & 0x7f) == 0x7e)


def test_up_e4m3_exhaustive_vs_torch():
    q = np.arange(256, dtype=np.uint8)
    ours = oracle.up_e4m3(q)
    theirs = torch.from_numpy(q).view(torch.float8_e4m3fn).to(torch.float32).numpy()
    nan = np.isnan(theirs)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan].view(np.uint32), theirs[~nan].view(np.uint32))


def test_fp8_quantize_and_amax():
    x = synth.normal((1000,), 3.0, "bf16", 70)
    xn = synth.to_np(x)
    q, amax = oracle.fp8_quantize(xn, "bf16", 0.5)
    v = dec(xn, "bf16")
    assert amax == np.float32(np.max(np.abs(v)))
    # scale_inv a power of two: v * 0.5 is exact, so q is torch's e4m3 of v/2
    want = torch.from_numpy((v * 0.5).astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(q, want)


@pytest.mark.parametrize("out", ["bf16", "f32"])
def test_fp8_matmuls_exact_on_small_integers(out):
    # integers in [-16, 16] are exact in e4m3; scales are powers of two, so every
    # step is exact and the result is the rounded exact integer matmul times s
    m, k, n = 40, 96, 56
    rng = np.random.default_rng(71)
    xi = rng.integers(-16, 17, size=(m, k)).astype(np.float64)
    wi = rng.integers(-16, 17, size=(k, n)).astype(np.float64)
    gi = rng.integers(-16, 17, size=(m, n)).astype(np.float64)
    e8 = lambda a: torch.from_numpy(a.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    xq, wq, gq = e8(xi), e8(wi), e8(gi)
    sx, sw, sg = 0.25, 2.0, 0.5
    b = (rng.integers(-64, 64, size=n) / 4).astype(np.float64)
    bias = enc(b, out)
    y = oracle.fp8_forward(xq, wq, bias, sx, sw, m, k, n, out)
    assert np.array_equal(y, round_exact((xi @ wi) * sx * sw + b, out))
    dx = oracle.fp8_backward_dx(gq, wq, sg, sw, m, k, n, out)
    assert np.array_equal(dx, round_exact((gi @ wi.T) * sg * sw, out))
    for chunk in (7, 256):
        dw = oracle.fp8_backward_dw(xq, gq, sx, sg, m, k, n, out, chunk=chunk)
        assert np.array_equal(dw, round_exact((xi.T @ gi) * sx * sg, out))
    rows = [3, 0, 39]
    assert np.array_equal(oracle.fp8_forward(xq, wq, bias, sx, sw, m, k, n, out, rows=rows), y[rows])


# --------------------------------------------------------------------------- brute force, tiny shapes

from fractions import Fraction  # noqa: E402

_FMT = {"f32": (24, -126), "bf16": (8, -126), "f16": (11, -14)}  # significand bits, least normal exponent


def round_ne(q, dtype):
    """Exact rational q rounded to the nearest value of the format, ties to
    even (subnormals included; no overflow at these sizes)."""
    if q == 0:
        return Fraction(0)
    p, emin = _FMT[dtype]
    a = abs(q)
    e = a.numerator.bit_length() - a.denominator.bit_length()  # 2^e <= a < 2^(e+2)
    if Fraction(2) ** e > a:
        e -= 1
    if Fraction(2) ** (e + 1) <= a:
        e += 1
    ulp = Fraction(2) ** (max(e, emin) - (p - 1))
    t = a / ulp
    n = t.numerator // t.denominator
    r = t - n
    if r > Fraction(1, 2) or (r == Fraction(1, 2) and n % 2 == 1):
        n += 1
    return (n * ulp) if q > 0 else -(n * ulp)


def test_round_ne_matches_numpy_conversions():
    """The exact rounding helper agrees with numpy's own f32 and f16
    conversions (round to nearest even), normals and subnormals."""
    rng = np.random.default_rng(7)
    vals = np.concatenate([rng.normal(size=2000) * np.exp2(rng.integers(-30, 30, size=2000)),
                           rng.normal(size=500) * 2.0 ** -140, rng.normal(size=500) * 2.0 ** -20])
    for v in vals:
        assert round_ne(Fraction(float(v)), "f32") == Fraction(float(np.float32(v)))
        if abs(v) < 60000:
            assert round_ne(Fraction(float(v)), "f16") == Fraction(float(np.float16(v)))


def chain_exact(avals, bvals):
    """acc = +0; acc = round_f32(a_l * b_l + acc) for l ascending."""
    acc = Fraction(0)
    for a, b in zip(avals, bvals):
        acc = round_ne(Fraction(a) * Fraction(b) + acc, "f32")
    return acc


def out_bits(v, dtype):
    """Encoding of an exactly representable value in the output type."""
    return enc([float(v)], dtype)[0] if dtype != "f32" else np.float32(float(v))


@pytest.mark.parametrize("dtype", DT)
def test_brute_force_tiny_shapes(dtype):
    rng = np.random.default_rng(2024)
    for m in (1, 2, 3):
        for k in (1, 2, 3):
            for n in (1, 2, 3):
                x = enc(rng.normal(size=(m, k)), dtype)
                w = enc(rng.normal(size=(k, n)), dtype)
                dy = enc(rng.normal(size=(m, n)), dtype)
                b = enc(rng.normal(scale=0.5, size=n), dtype)
                xv, wv, dyv, bv = dec(x, dtype), dec(w, dtype), dec(dy, dtype), dec(b, dtype)
                y = oracle.forward(x, w, b, m, k, n, dtype)
                dx = oracle.backward_dx(dy, w, m, k, n, dtype)
                dw32 = oracle.backward_dw(x, dy, m, k, n, dtype, dw_f32=True)
                dwr = oracle.backward_dw(x, dy, m, k, n, dtype, dw_f32=False)
                for i in range(m):
                    for j in range(n):
                        acc = chain_exact(xv[i, :], wv[:, j])
                        want = round_ne(round_ne(acc + Fraction(bv[j]), "f32"), dtype)
                        assert y[i, j] == out_bits(want, dtype), ("y", m, k, n, i, j)
                    for j in range(k):
                        acc = chain_exact(dyv[i, :], wv[j, :])
                        assert dx[i, j] == out_bits(round_ne(acc, dtype), dtype), ("dx", m, k, n, i, j)
                for i in range(k):
                    for j in range(n):
                        acc = chain_exact(xv[:, i], dyv[:, j])  # one chunk: the plain chain over rows
                        assert dw32[i, j] == np.float32(float(acc)), ("dw", m, k, n, i, j)
                        assert dwr[i, j] == out_bits(round_ne(acc, dtype), dtype), ("dw rounded", m, k, n, i, j)


@pytest.mark.parametrize("dtype", DT)
def test_brute_force_tiny_grouped_forward(dtype):
    rng = np.random.default_rng(2025)
    e = 2
    for m in (1, 2, 3):
        for k in (1, 2, 3):
            for n in (1, 2, 3):
                x = enc(rng.normal(size=(m, k)), dtype)
                w = enc(rng.normal(size=(e * n * k,)), dtype)  # [E, N, K]
                ids = rng.integers(0, e + 1, size=m).astype(np.uint32)  # id e: a padding row
                xv, wv = dec(x, dtype), dec(w, dtype).reshape(e, n, k)
                y = oracle.grouped_forward(x, w, ids, m, k, n, e, dtype)
                for i in range(m):
                    for j in range(n):
                        if ids[i] >= e:
                            want = Fraction(0)
                        else:
                            want = round_ne(chain_exact(xv[i, :], wv[ids[i], j, :]), dtype)
                        assert y[i, j] == out_bits(want, dtype), (m, k, n, i, j, int(ids[i]))


@pytest.mark.parametrize("dtype", DT)
def test_brute_force_tiny_grouped_backward(dtype):
    """dinput chains over n with W[e(m)]; dweights chains over the expert's rows
    in ascending original index (one chunk at these sizes); padding rows give a
    zero dinput row and touch no dweights; an expert without rows gets zeros."""
    rng = np.random.default_rng(2026)
    e = 2
    for m in (1, 2, 3):
        for k in (1, 2, 3):
            for n in (1, 2, 3):
                x = enc(rng.normal(size=(m, k)), dtype)
                w = enc(rng.normal(size=(e * n * k,)), dtype)  # [E, N, K]
                dy = enc(rng.normal(size=(m, n)), dtype)
                ids = rng.integers(0, e + 1, size=m).astype(np.uint32)
                xv, wv, dyv = dec(x, dtype), dec(w, dtype).reshape(e, n, k), dec(dy, dtype)
                dx = oracle.grouped_dinput(w, dy, ids, m, k, n, e, dtype)
                dw = oracle.grouped_dweights(x, dy, ids, m, k, n, e, dtype)
                for i in range(m):
                    for j in range(k):
                        want = Fraction(0) if ids[i] >= e else round_ne(chain_exact(dyv[i, :], wv[ids[i], :, j]), dtype)
                        assert dx[i, j] == out_bits(want, dtype), ("dx", m, k, n, i, j)
                dw = dw.reshape(e, n, k)
                for g in range(e):
                    rows = [i for i in range(m) if ids[i] == g]
                    for j in range(n):
                        for l in range(k):
                            acc = chain_exact([dyv[i, j] for i in rows], [xv[i, l] for i in rows])
                            assert dw[g, j, l] == np.float32(float(acc)), ("dw", m, k, n, g, j, l)


def e4m3_exact(code):
    """Value of an e4m3 (fn) code from its fields: sign, 4-bit exponent (bias
    7), 3-bit mantissa; exponent 0 is subnormal (m * 2^-9)."""
    code = int(code)
    sign = -1 if code & 0x80 else 1
    ex, mant = (code >> 3) & 0xF, code & 0x7
    if ex == 0:
        return sign * Fraction(mant, 512)
    return sign * (1 + Fraction(mant, 8)) * Fraction(2) ** (ex - 7)


@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_brute_force_tiny_fp8_forward(out):
    """y = rne(round_f32(round_f32(chain * round_f32(sx * sw)) + bias)) with the
    chain over exactly decoded e4m3 values; every shape up to 3 x 3 x 3."""
    rng = np.random.default_rng(2027)
    finite = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    sx, sw = 0.375, 1.25
    s32 = round_ne(Fraction(sx) * Fraction(sw), "f32")
    for m in (1, 2, 3):
        for k in (1, 2, 3):
            for n in (1, 2, 3):
                xq = rng.choice(finite, size=(m, k)).astype(np.uint8)
                wq = rng.choice(finite, size=(k, n)).astype(np.uint8)
                bias = enc(rng.normal(size=n), out) if out != "f32" else None
                y = oracle.fp8_forward(xq, wq, bias, sx, sw, m, k, n, out)
                bv = dec(bias, out) if bias is not None else None
                for i in range(m):
                    for j in range(n):
                        acc = chain_exact([e4m3_exact(c) for c in xq[i, :]], [e4m3_exact(c) for c in wq[:, j]])
                        v = round_ne(acc * s32, "f32")
                        if bv is not None:
                            v = round_ne(v + Fraction(bv[j]), "f32")
                        assert y[i, j] == out_bits(round_ne(v, out), out), (m, k, n, i, j)


@pytest.mark.parametrize("dtype", DT)
def test_brute_force_tiny_bias_grad(dtype):
    """db[n] = ((+0 + dY[0,n]) + dY[1,n]) + ... with f32 additions (one chunk at
    these sizes), then one rounding unless kept in f32."""
    rng = np.random.default_rng(2028)
    for m in (1, 2, 3):
        for n in (1, 2, 3):
            dy = enc(rng.normal(size=(m, n)), dtype)
            dyv = dec(dy, dtype)
            db32 = oracle.bias_grad(dy, m, n, dtype, out_f32=True)
            dbr = oracle.bias_grad(dy, m, n, dtype)
            for j in range(n):
                acc = Fraction(0)
                for i in range(m):
                    acc = round_ne(acc + Fraction(dyv[i, j]), "f32")
                assert db32[j] == np.float32(float(acc))
                assert dbr[j] == out_bits(round_ne(acc, dtype), dtype)

