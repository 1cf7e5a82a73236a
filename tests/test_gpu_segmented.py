"""GPU tests of the caller-segmented grouped API and its strategy enum."""
import numpy as np
import pytest
import torch

import oracle
import deterministic_invariant_gemm_fixed_gb300 as bi
from deterministic_invariant_gemm_fixed_gb300 import synth
from helpers import out_np

pytestmark = pytest.mark.gpu
S = bi.BI_STRATEGY_SCALAR, bi.BI_STRATEGY_TENSOR_CORE, bi.BI_STRATEGY_AUTO


@pytest.fixture(scope="module")
def eng():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    e = bi.Engine(0)
    yield e
    e.close()


def grouped_case(m, k, n, e, dtype, npad, seed=0):
    """Rows grouped by expert (expert 2 empty), npad padding rows at the end."""
    rng = np.random.default_rng(seed)
    counts = rng.multinomial(m - npad, np.ones(e) / e)
    if e > 2:  # expert 2 gets no rows
        counts[0] += counts[2]
        counts[2] = 0
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.uint32)
    ids = np.full(m, e + 3, dtype=np.uint32)
    for g in range(e):
        ids[offs[g]:offs[g + 1]] = g
    x, w, dy, _ = synth.grouped_inputs(m, k, n, e, dtype, pad_frac=0.0, seed_offset=seed,
                                       w=("normal", 0.5))
    return x, w, dy, ids, offs


def run(eng, x, w, dy, ids, offs, m, k, n, e, dtype, strategy=None, tc=None):
    tdt = synth.TORCH_DTYPES[dtype]
    X, W, DY = x.cuda(), w.cuda(), dy.cuda()
    y = torch.full((m, n), float("nan"), dtype=tdt, device="cuda")
    dx = torch.full((m, k), float("nan"), dtype=tdt, device="cuda")
    dw = torch.full((e, n, k), float("nan"), dtype=torch.float32, device="cuda")
    if strategy is not None:
        O = torch.from_numpy(offs.astype(np.int32)).cuda()
        eng.grouped_forward_segmented(y, X, W, O, m, k, n, e, dtype, None, strategy)
        eng.grouped_backward_segmented(dx, dw, X, W, DY, O, m, k, n, e, dtype, None, strategy)
    else:
        I = torch.from_numpy(ids.astype(np.int32)).cuda()
        eng.grouped_forward(y, X, W, I, m, k, n, e, dtype, None, tc)
        eng.grouped_backward(dx, dw, X, W, DY, I, m, k, n, e, dtype, None, tc)
    eng.check()
    return out_np(y), out_np(dx), out_np(dw)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_segmented_equals_id_based_on_both_tiers(eng, dtype):
    m, k, n, e = 900, 128, 200, 5
    x, w, dy, ids, offs = grouped_case(m, k, n, e, dtype, npad=40)
    for strategy, tc in ((S[0], 0), (S[1], 1), (S[2], 1)):
        a = run(eng, x, w, dy, ids, offs, m, k, n, e, dtype, strategy=strategy)
        b = run(eng, x, w, dy, ids, offs, m, k, n, e, dtype, tc=tc)
        for u, v in zip(a, b):
            assert np.array_equal(u, v), strategy
    # the scalar strategy is the oracle's definition
    y, dx, dw = run(eng, x, w, dy, ids, offs, m, k, n, e, dtype, strategy=S[0])
    xn, wn, dyn = (synth.to_np(t) for t in (x, w, dy))
    assert np.array_equal(y, oracle.grouped_forward(xn, wn, ids, m, k, n, e, dtype))
    assert np.array_equal(dx, oracle.grouped_dinput(wn, dyn, ids, m, k, n, e, dtype))
    assert np.array_equal(dw, oracle.grouped_dweights(xn, dyn, ids, m, k, n, e, dtype))
    assert np.all(y[offs[e]:] == 0) and np.all(dx[offs[e]:] == 0)


def test_tensor_core_request_that_cannot_be_met_is_an_error(eng):
    h = eng.handle
    z = torch.zeros(64, 64, dtype=torch.float32, device="cuda")
    o = torch.zeros(3, dtype=torch.int32, device="cuda")
    # f32 operands have no tensor-core path
    st = bi.bi_grouped_forward_segmented(h, z, z, z, o, 64, 64, 64, 2, "f32", None, S[1])
    assert st == bi.BI_ERR_UNSUPPORTED, bi.bi_last_error(h)
    # K = 48 rules out the tensor-core dinput and dweights
    zb = torch.zeros(64, 64, dtype=torch.bfloat16, device="cuda")
    dw = torch.zeros(2, 64, 48, dtype=torch.float32, device="cuda")
    st = bi.bi_grouped_backward_segmented(h, zb, dw, zb, zb, zb, o, 64, 48, 64, 2, "bf16", None, S[1])
    assert st == bi.BI_ERR_UNSUPPORTED
    # Auto takes the scalar tier there instead, and Scalar always works
    assert bi.bi_grouped_backward_segmented(h, zb, dw, zb, zb, zb, o, 64, 48, 64, 2, "bf16", None, S[2]) == bi.BI_OK
    assert bi.bi_grouped_forward_segmented(h, z, z, z, o, 64, 64, 64, 2, "f32", None, S[0]) == bi.BI_OK
    assert bi.bi_grouped_forward_segmented(h, z, z, z, o, 64, 64, 64, 2, "f32", None, 9) == bi.BI_ERR_INVALID_ARG
    eng.check()


def test_bad_offsets_are_clamped_and_reported(eng):
    m, k, n, e, dtype = 300, 64, 72, 3, "bf16"
    x, w, dy, ids, offs = grouped_case(m, k, n, e, dtype, npad=0, seed=3)
    bad = np.array([0, 250, 100, 10_000], dtype=np.uint32)  # decreasing, then beyond m
    O = torch.from_numpy(bad.astype(np.int32)).cuda()
    y = torch.empty(m, n, dtype=torch.bfloat16, device="cuda")
    eng.grouped_forward_segmented(y, x.cuda(), w.cuda(), O, m, k, n, e, dtype, None, S[0])
    st = bi.bi_engine_check(eng.handle, None)
    assert st == bi.BI_ERR_INVALID_ARG
    assert "clamped" in bi.bi_last_error(eng.handle)
    # clamped to [0, 250, 250, 300]: expert 0 rows 0..249, expert 2 rows 250..299
    ids2 = np.zeros(m, dtype=np.uint32)
    ids2[250:] = 2
    want = oracle.grouped_forward(synth.to_np(x), synth.to_np(w), ids2, m, k, n, e, dtype)
    assert np.array_equal(out_np(y), want)
    assert bi.bi_engine_check(eng.handle, None) == bi.BI_OK
