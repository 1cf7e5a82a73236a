"""GPU parity of the grouped per-row-expert passes through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
import deterministic_invariant_gemm_fixed_gb300 as bi
from deterministic_invariant_gemm_fixed_gb300 import synth
from helpers import check_tc, dev, f64, out_np, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def eng():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    e = bi.Engine(0)
    yield e
    e.close()


def ids_dev(ids):
    return torch.from_numpy(synth.to_np(ids).astype(np.int32)).cuda()  # u32 bit patterns


def run_grouped(eng, x, w, dy, ids, m, k, n, e, dtype, tc, with_dx=True):
    tdt = synth.TORCH_DTYPES[dtype]
    X, W, DY, I = dev(x), dev(w), dev(dy), ids_dev(ids)
    y = torch.empty(m, n, dtype=tdt, device="cuda")
    dx = torch.empty(m, k, dtype=tdt, device="cuda") if with_dx else None
    dw = torch.empty(e, n, k, dtype=torch.float32, device="cuda")
    eng.grouped_forward(y, X, W, I, m, k, n, e, dtype, None, tc)
    eng.grouped_backward(dx, dw, X, W, DY, I, m, k, n, e, dtype, None, tc)
    eng.check()
    return out_np(y), (out_np(dx) if with_dx else None), out_np(dw)


def small_case(dtype, m=700, k=96, n=136, e=5, seed=0):
    x, w, dy, ids = synth.grouped_inputs(m, k, n, e, dtype, pad_frac=0.06, seed_offset=seed,
                                         x=("normal", 1.0), w=("normal", 1.0), dy=("normal", 1.0))
    ids = ids.clone()
    ids[ids == 2] = 0          # expert 2 gets no rows
    ids[5] = e + 1000          # an id far beyond E is padding
    return x, w, dy, ids


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_grouped_scalar_bit_exact(eng, dtype):
    m, k, n, e = 700, 96, 136, 5
    x, w, dy, ids = small_case(dtype)
    y, dx, dw = run_grouped(eng, x, w, dy, ids, m, k, n, e, dtype, tc=0)
    xn, wn, dyn, idn = (synth.to_np(t) for t in (x, w, dy, ids))
    assert np.array_equal(y, oracle.grouped_forward(xn, wn, idn, m, k, n, e, dtype))
    assert np.array_equal(dx, oracle.grouped_dinput(wn, dyn, idn, m, k, n, e, dtype))
    assert np.array_equal(dw, oracle.grouped_dweights(xn, dyn, idn, m, k, n, e, dtype))
    assert np.all(dw[2] == 0)


@pytest.mark.parametrize("k,n", [(96, 136), (384, 640)])  # (384, 640): half-used last column tiles
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_grouped_tc_within_tolerance(eng, dtype, k, n):
    m, e = 700, 5
    x, w, dy, ids = small_case(dtype, k=k, n=n)
    y, dx, dw = run_grouped(eng, x, w, dy, ids, m, k, n, e, dtype, tc=1)
    xn, wn, dyn, idn = (synth.to_np(t) for t in (x, w, dy, ids))
    x64, w64, dy64 = f64(xn, dtype), f64(wn, dtype).reshape(e, n, k), f64(dyn, dtype)
    valid = idn < e
    S_y = np.zeros((m, n)); S_dx = np.zeros((m, k)); S_dw = np.zeros((e, n, k))
    for g in range(e):
        rows = np.nonzero(idn == g)[0]
        S_y[rows] = np.abs(x64[rows]) @ np.abs(w64[g]).T
        S_dx[rows] = np.abs(dy64[rows]) @ np.abs(w64[g])
        S_dw[g] = np.abs(dy64[rows]).T @ np.abs(x64[rows])
    r = oracle.grouped_forward(xn, wn, idn, m, k, n, e, dtype, out_f32=True)
    ok, st = check_tc(y, r, S_y, dtype)
    assert ok, st
    r = oracle.grouped_dinput(wn, dyn, idn, m, k, n, e, dtype, out_f32=True)
    ok, st = check_tc(dx, r, S_dx, dtype)
    assert ok, st
    r = oracle.grouped_dweights(xn, dyn, idn, m, k, n, e, dtype)
    ok, st = check_tc(dw, r, S_dw, "f32")
    assert ok, st
    assert np.all(y[~valid] == 0) and np.all(dx[~valid] == 0)
    assert np.all(dw[2] == 0)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_grouped_tc_exact_on_small_integers(eng, dtype):
    m, k, n, e = 640, 128, 200, 4
    x = synth.small_ints((m, k), -8, 8, dtype, 31)
    w = synth.small_ints((e, n, k), -8, 8, dtype, 32)
    dy = synth.small_ints((m, n), -8, 8, dtype, 33)
    ids = synth.expert_ids(m, e, 0.05, 34)
    y, dx, dw = run_grouped(eng, x, w, dy, ids, m, k, n, e, dtype, tc=1)
    xn, wn, dyn, idn = (synth.to_np(t) for t in (x, w, dy, ids))
    assert np.array_equal(y, oracle.grouped_forward(xn, wn, idn, m, k, n, e, dtype))
    assert np.array_equal(dx, oracle.grouped_dinput(wn, dyn, idn, m, k, n, e, dtype))
    assert np.array_equal(dw, oracle.grouped_dweights(xn, dyn, idn, m, k, n, e, dtype))


@pytest.mark.parametrize("tc", [0, 1])
def test_grouped_full_config_sampled(eng, tc):
    c = synth.GROUPED
    m, k, n, e, dtype = c["m"], c["k"], c["n"], c["e"], c["dtype"]
    x, w, dy, ids = synth.grouped_inputs(m, k, n, e, dtype, pad_frac=c["pad_frac"])
    y, dx, dw = run_grouped(eng, x, w, dy, ids, m, k, n, e, dtype, tc=tc)
    xn, wn, dyn, idn = (synth.to_np(t) for t in (x, w, dy, ids))
    assert int((idn >= e).sum()) == round(0.05 * m)
    rows = sample_rows(m, 24, seed=5)
    rows = np.unique(np.concatenate([rows, np.nonzero(idn >= e)[0][:3]]))
    rng = np.random.default_rng(6)
    sel = (rng.integers(0, e, size=6), rng.integers(0, n, size=6))
    if tc == 0:
        assert np.array_equal(y[rows], oracle.grouped_forward(xn, wn, idn, m, k, n, e, dtype, rows=rows))
        assert np.array_equal(dx[rows], oracle.grouped_dinput(wn, dyn, idn, m, k, n, e, dtype, rows=rows))
        assert np.array_equal(dw[sel[0], sel[1]], oracle.grouped_dweights(xn, dyn, idn, m, k, n, e, dtype, sel=sel))
        return
    x64, dy64 = f64(xn, dtype), f64(dyn, dtype)
    w64 = f64(wn, dtype).reshape(e, n, k)
    S_y = np.zeros((rows.size, n)); S_dx = np.zeros((rows.size, k))
    for i, r_ in enumerate(rows):
        if idn[r_] < e:
            S_y[i] = np.abs(w64[idn[r_]]) @ np.abs(x64[r_])
            S_dx[i] = np.abs(dy64[r_]) @ np.abs(w64[idn[r_]])
    r = oracle.grouped_forward(xn, wn, idn, m, k, n, e, dtype, rows=rows, out_f32=True)
    ok, st = check_tc(y[rows], r, S_y, dtype)
    assert ok, st
    r = oracle.grouped_dinput(wn, dyn, idn, m, k, n, e, dtype, rows=rows, out_f32=True)
    ok, st = check_tc(dx[rows], r, S_dx, dtype)
    assert ok, st
    S_dw = np.stack([np.abs(dy64[idn == g_, j]) @ np.abs(x64[idn == g_]) for g_, j in zip(*sel)])
    r = oracle.grouped_dweights(xn, dyn, idn, m, k, n, e, dtype, sel=sel)
    ok, st = check_tc(dw[sel[0], sel[1]], r, S_dw, "f32")
    assert ok, st


@pytest.mark.parametrize("tc", [0, 1])
def test_grouped_ten_runs_and_prefix_invariance(eng, tc):
    m, k, n, e, dtype = 1100, 128, 256, 6, "bf16"
    x, w, dy, ids = synth.grouped_inputs(m, k, n, e, dtype)
    first = run_grouped(eng, x, w, dy, ids, m, k, n, e, dtype, tc=tc)
    for _ in range(9):
        again = run_grouped(eng, x, w, dy, ids, m, k, n, e, dtype, tc=tc)
        for a, b in zip(first, again):
            assert np.array_equal(a, b)
    for mp in (1, 129, 513):
        part = run_grouped(eng, x[:mp].contiguous(), w, dy[:mp].contiguous(), ids[:mp].contiguous(),
                           mp, k, n, e, dtype, tc=tc)
        assert np.array_equal(part[0], first[0][:mp])
        assert np.array_equal(part[1], first[1][:mp])


def test_grouped_single_expert_matches_dense_scalar(eng):
    m, k, n, dtype = 300, 96, 80, "bf16"
    x, w, dy, _ = synth.grouped_inputs(m, k, n, 1, dtype, pad_frac=0.0)
    ids = torch.zeros(m, dtype=torch.int64)
    y, dx, dw = run_grouped(eng, x, w, dy, ids, m, k, n, 1, dtype, tc=0)
    wd = w.reshape(n, k).t().contiguous()
    Y = torch.empty(m, n, dtype=torch.bfloat16, device="cuda")
    DX = torch.empty(m, k, dtype=torch.bfloat16, device="cuda")
    DW = torch.empty(k, n, dtype=torch.float32, device="cuda")
    eng.forward(Y, dev(x), dev(wd), None, m, k, n, dtype, None, 0)
    eng.backward_dx(DX, dev(dy), dev(wd), m, k, n, dtype, None, 0)
    eng.backward_dw(DW, 1, dev(x), dev(dy), m, k, n, dtype, None, 0)
    assert np.array_equal(y, out_np(Y))
    assert np.array_equal(dx, out_np(DX))
    assert np.array_equal(dw[0], out_np(DW).T)


def test_grouped_m_zero_zeroes_dw(eng):
    k, n, e = 64, 64, 3
    dw = torch.full((e, n, k), 3.0, dtype=torch.float32, device="cuda")
    z = torch.zeros(1, 64, dtype=torch.bfloat16, device="cuda")
    ids = torch.zeros(1, dtype=torch.int32, device="cuda")
    eng.grouped_backward(None, dw, z, z, z, ids, 0, k, n, e, "bf16", None, 1)
    eng.check()
    assert torch.all(dw == 0)
    h = eng.handle
    assert bi.bi_grouped_forward(h, z, z, z, ids, 1, k, n, 0, "bf16", None, 1) == bi.BI_ERR_INVALID_ARG


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_grouped_tc_tile_edges_exact(eng, dtype):
    """Expert row counts on the tensor-core tiling's edges (0, 1, 63/64/65 around
    the 64-row contraction block, 255/256/257 around the 256-row tile, more than
    two tiles), rows shuffled (id path) and grouped (segmented path), with
    padding rows: small integers, so every pass must equal the oracle bit for bit."""
    counts = np.array([0, 1, 63, 64, 65, 255, 256, 257, 577, 130])
    e, npad, k, n = len(counts), 37, 136, 200
    m = int(counts.sum()) + npad
    rng = np.random.default_rng(71)
    grouped_ids = np.concatenate([np.repeat(np.arange(e), counts), np.full(npad, e + 3)]).astype(np.uint32)
    shuffled_ids = grouped_ids[rng.permutation(m)]
    x = synth.small_ints((m, k), -8, 8, dtype, 72)
    w = synth.small_ints((e, n, k), -8, 8, dtype, 73)
    dy = synth.small_ints((m, n), -8, 8, dtype, 74)
    xn, wn, dyn = (synth.to_np(t) for t in (x, w, dy))
    tdt = synth.TORCH_DTYPES[dtype]
    for idn in (shuffled_ids, grouped_ids):
        y, dx, dw = run_grouped(eng, x, w, dy, torch.from_numpy(idn.astype(np.int64)), m, k, n, e, dtype, tc=1)
        assert np.array_equal(y, oracle.grouped_forward(xn, wn, idn, m, k, n, e, dtype))
        assert np.array_equal(dx, oracle.grouped_dinput(wn, dyn, idn, m, k, n, e, dtype))
        assert np.array_equal(dw, oracle.grouped_dweights(xn, dyn, idn, m, k, n, e, dtype))
        assert np.all(dw[0] == 0)
    # the segmented entry points on the grouped rows
    offs = torch.from_numpy(np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)).cuda()
    X, W, DY = dev(x), dev(w), dev(dy)
    Y = torch.empty(m, n, dtype=tdt, device="cuda")
    DX = torch.empty(m, k, dtype=tdt, device="cuda")
    DW = torch.empty(e, n, k, dtype=torch.float32, device="cuda")
    eng.grouped_forward_segmented(Y, X, W, offs, m, k, n, e, dtype, None, bi.BI_STRATEGY_TENSOR_CORE)
    eng.grouped_backward_segmented(DX, DW, X, W, DY, offs, m, k, n, e, dtype, None, bi.BI_STRATEGY_TENSOR_CORE)
    eng.check()
    assert np.array_equal(out_np(Y), oracle.grouped_forward(xn, wn, grouped_ids, m, k, n, e, dtype))
    assert np.array_equal(out_np(DX), oracle.grouped_dinput(wn, dyn, grouped_ids, m, k, n, e, dtype))
    assert np.array_equal(out_np(DW), oracle.grouped_dweights(xn, dyn, grouped_ids, m, k, n, e, dtype))


@pytest.mark.parametrize("e", [64, 300, 1500])  # 1500: more buckets than the two-launch grouping takes
@pytest.mark.parametrize("tc", [0, 1])
def test_grouped_many_experts_exact(eng, e, tc):
    """Many experts, most of them small and some empty (ids drawn from a skewed
    distribution): exact small-integer problems, both tiers, ids and the
    segmented entry points, equal to the oracle bit for bit."""
    m, k, n, dtype = 3000, 128, 136, "bf16"
    rng = np.random.default_rng(90 + e)
    raw = np.minimum((rng.pareto(1.2, size=m) * e / 8).astype(np.int64), e + 5)  # skewed, some >= E
    ids = raw.astype(np.uint32)
    x = synth.small_ints((m, k), -8, 8, dtype, 91)
    w = synth.small_ints((e, n, k), -8, 8, dtype, 92)
    dy = synth.small_ints((m, n), -8, 8, dtype, 93)
    xn, wn, dyn = (synth.to_np(t) for t in (x, w, dy))
    want = (oracle.grouped_forward(xn, wn, ids, m, k, n, e, dtype),
            oracle.grouped_dinput(wn, dyn, ids, m, k, n, e, dtype),
            oracle.grouped_dweights(xn, dyn, ids, m, k, n, e, dtype))
    assert (np.bincount(np.minimum(ids, e), minlength=e + 1)[:e] == 0).any()  # empty experts
    got = run_grouped(eng, x, w, dy, torch.from_numpy(ids.astype(np.int64)), m, k, n, e, dtype, tc=tc)
    for g_, w_ in zip(got, want):
        assert np.array_equal(g_, w_)
    # the same rows grouped by the caller
    order = np.argsort(np.minimum(ids, e), kind="stable")
    gids = ids[order]
    xs, dys = x[torch.from_numpy(order)], dy[torch.from_numpy(order)]
    counts = np.bincount(np.minimum(gids, e), minlength=e + 1)[:e]
    offs = torch.from_numpy(np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)).cuda()
    tdt = synth.TORCH_DTYPES[dtype]
    Y = torch.empty(m, n, dtype=tdt, device="cuda")
    DX = torch.empty(m, k, dtype=tdt, device="cuda")
    DW = torch.empty(e, n, k, dtype=torch.float32, device="cuda")
    strat = bi.BI_STRATEGY_TENSOR_CORE if tc else bi.BI_STRATEGY_SCALAR
    eng.grouped_forward_segmented(Y, dev(xs), dev(w), offs, m, k, n, e, dtype, None, strat)
    eng.grouped_backward_segmented(DX, DW, dev(xs), dev(w), dev(dys), offs, m, k, n, e, dtype, None, strat)
    eng.check()
    assert np.array_equal(out_np(Y), want[0][order])
    assert np.array_equal(out_np(DX), want[1][order])
    assert np.array_equal(out_np(DW), want[2])


@pytest.mark.parametrize("tc", [0, 1])
def test_grouped_long_expert_in_pieces(eng, tc):
    """One expert with more rows than an 8192-row piece (17000), one small, one
    empty, plus padding: dweights bit-exact on small integers (the tensor-core
    tier sums the expert's pieces in order), ids and caller-grouped rows."""
    counts = np.array([17000, 2000, 0])
    e, npad, k, n = 3, 1000, 64, 72
    m = int(counts.sum()) + npad
    rng = np.random.default_rng(97)
    grouped_ids = np.concatenate([np.repeat(np.arange(e), counts), np.full(npad, e)]).astype(np.uint32)
    ids = grouped_ids[rng.permutation(m)]
    x = synth.small_ints((m, k), -4, 4, "bf16", 98)
    w = synth.small_ints((e, n, k), -4, 4, "bf16", 99)
    dy = synth.small_ints((m, n), -2, 2, "bf16", 100)
    xn, wn, dyn = (synth.to_np(t) for t in (x, w, dy))
    want = oracle.grouped_dweights(xn, dyn, ids, m, k, n, e, "bf16")
    _, _, dw = run_grouped(eng, x, w, dy, torch.from_numpy(ids.astype(np.int64)), m, k, n, e, "bf16", tc=tc,
                           with_dx=False)
    assert np.array_equal(dw, want) and np.all(dw[2] == 0)
    order = np.argsort(np.minimum(ids, e), kind="stable")
    offs = torch.from_numpy(np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)).cuda()
    DW = torch.empty(e, n, k, dtype=torch.float32, device="cuda")
    strat = bi.BI_STRATEGY_TENSOR_CORE if tc else bi.BI_STRATEGY_SCALAR
    eng.grouped_backward_segmented(None, DW, dev(x[torch.from_numpy(order)]), dev(w),
                                   dev(dy[torch.from_numpy(order)]), offs, m, k, n, e, "bf16", None, strat)
    eng.check()
    assert np.array_equal(out_np(DW), want)


def test_grouped_dweights_last_wave_in_chunks(eng):
    """Grouped dweights whose last, partial wave of units contracts in chunks
    added by the dW tree: 4 experts x 2 column tiles = 8 units on 76 CTA pairs,
    about 31 blocks per expert, so each unit runs as 3 chunks (one expert has no
    rows, so all of its chunks are empty).  Within tolerance of the oracle on
    random data, bit-identical over runs, exact on small integers, and equal
    to the scalar tier on them."""
    m, k, n, e, dtype = 8000, 264, 136, 4, "bf16"
    rng = np.random.default_rng(404)
    ids = rng.integers(0, e, size=m).astype(np.uint32)
    ids[ids == 1] = 0            # expert 1 gets no rows
    ids[rng.choice(m, 300, replace=False)] = e  # padding
    x, w, dy, _ = synth.grouped_inputs(m, k, n, e, dtype)
    I = torch.from_numpy(ids.astype(np.int64))
    _, _, dw = run_grouped(eng, x, w, dy, I, m, k, n, e, dtype, tc=1, with_dx=False)
    for _ in range(2):
        _, _, dw2 = run_grouped(eng, x, w, dy, I, m, k, n, e, dtype, tc=1, with_dx=False)
        assert np.array_equal(dw.view(np.uint32), dw2.view(np.uint32))
    xn, dyn = synth.to_np(x), synth.to_np(dy)
    x64, dy64 = f64(xn, dtype), f64(dyn, dtype)
    S = np.zeros((e, n, k))
    for g in range(e):
        rows = np.nonzero(ids == g)[0]
        S[g] = np.abs(dy64[rows]).T @ np.abs(x64[rows])
    ok, st = check_tc(dw, oracle.grouped_dweights(xn, dyn, ids, m, k, n, e, dtype), S, "f32")
    assert ok, st
    assert np.all(dw[1] == 0) and not np.signbit(dw[1]).any()
    xi = synth.small_ints((m, k), -4, 4, dtype, 405)
    wi = synth.small_ints((e, n, k), -4, 4, dtype, 406)
    dyi = synth.small_ints((m, n), -4, 4, dtype, 407)
    _, _, dwt = run_grouped(eng, xi, wi, dyi, I, m, k, n, e, dtype, tc=1, with_dx=False)
    _, _, dws = run_grouped(eng, xi, wi, dyi, I, m, k, n, e, dtype, tc=0, with_dx=False)
    want = oracle.grouped_dweights(synth.to_np(xi), synth.to_np(dyi), ids, m, k, n, e, dtype)
    assert np.array_equal(dwt, want) and np.array_equal(dws, want)
