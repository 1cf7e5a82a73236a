"""Failure handling and memory discipline of every entry point, on the GPU.

* Allocation failure: with bi_engine_fail_allocations, every call that takes
  scratch from the engine's pool returns BI_ERR_OOM, launches nothing, leaves
  its outputs as they were, and the engine keeps working (the next call gives
  the same bits as before).  The failure is made on the host; no GPU memory is
  exhausted.
* Guard bands: each output sits in a larger buffer whose bytes before and after
  it hold a poison pattern; after the call (ragged shapes, both tiers, every
  pass: dense, bias gradient, grouped by ids and by offsets, FP8, 3xTF32) the
  poison must be intact, i.e. no kernel wrote outside its output.
"""
import numpy as np
import pytest
import torch

import deterministic_invariant_gemm_fixed_gb300 as bi
from deterministic_invariant_gemm_fixed_gb300 import synth

pytestmark = pytest.mark.gpu

GUARD = 64  # elements on each side; 64 x element size keeps 16-byte alignment
POISON = {1: 0xA5, 2: 0x7DEF, 4: 0x7F8ABCDE}
INT_VIEW = {1: torch.uint8, 2: torch.int16, 4: torch.int32}


@pytest.fixture(scope="module")
def eng():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    e = bi.Engine(0)
    yield e
    e.close()


class Guarded:
    """An output tensor of `shape` inside a poisoned buffer."""

    def __init__(self, shape, dtype):
        self.numel = int(np.prod(shape))
        self.buf = torch.empty(self.numel + 2 * GUARD, dtype=dtype, device="cuda")
        self.es = self.buf.element_size()
        self.iv = self.buf.view(INT_VIEW[self.es])
        pv = POISON[self.es]
        if self.es == 2 and pv > 0x7FFF:
            pv -= 1 << 16
        self.iv.fill_(pv)
        self.t = self.buf[GUARD:GUARD + self.numel].view(shape)
        self.pv = pv

    def intact(self):
        torch.cuda.synchronize()
        return bool((self.iv[:GUARD] == self.pv).all() and (self.iv[GUARD + self.numel:] == self.pv).all())


def _dense(m, k, n, dtype, seed=0):
    x, w, dy, b = synth.dense_inputs(m, k, n, dtype, w=("normal", 0.1), seed_offset=seed)
    return x.cuda(), w.cuda(), dy.cuda(), b.cuda()


def _grouped(m, k, n, e, dtype):
    x, w, dy, ids = synth.grouped_inputs(m, k, n, e, dtype, pad_frac=0.1)
    idn = synth.to_np(ids)
    I = torch.from_numpy(idn.astype(np.int32)).cuda()
    order = np.argsort(np.minimum(idn, e), kind="stable")
    counts = np.bincount(np.minimum(idn, e), minlength=e + 1)[:e]
    offs = torch.from_numpy(np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)).cuda()
    oi = torch.from_numpy(order).cuda()
    X, W, DY = x.cuda(), w.cuda(), dy.cuda()
    return X, W, DY, I, offs, X[oi].contiguous(), DY[oi].contiguous()


# ---------------------------------------------------------------- guard bands

@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("tc", [0, 1])
def test_dense_passes_write_only_their_outputs(eng, dtype, tc):
    m, k, n = 300, 200, 136  # several tiles and a ragged tail; multiples of 8 for the tensor cores
    X, W, DY, B = _dense(m, k, n, dtype)
    td = synth.TORCH_DTYPES[dtype]
    y, dx = Guarded((m, n), td), Guarded((m, k), td)
    dw32, dw16, db = Guarded((k, n), torch.float32), Guarded((k, n), td), Guarded((n,), td)
    eng.forward(y.t, X, W, B, m, k, n, dtype, None, tc)
    eng.backward_dx(dx.t, DY, W, m, k, n, dtype, None, tc)
    eng.backward_dw(dw32.t, 1, X, DY, m, k, n, dtype, None, tc)
    eng.backward_dw(dw16.t, 0, X, DY, m, k, n, dtype, None, tc)
    eng.bias_grad(db.t, 0, DY, m, n, dtype, None)
    eng.check()
    for name, g in (("y", y), ("dx", dx), ("dw f32", dw32), ("dw", dw16), ("db", db)):
        assert g.intact(), (name, dtype, tc)
        assert not torch.isnan(g.t.float()).any(), (name, dtype, tc)  # every element was written


def test_tensor_core_dw_with_chunked_last_wave_writes_only_its_output(eng):
    # 1024 rows, one 256 x 256 tile: the tile's contraction runs as chunks added
    # by the chunk-sum kernel, which must stay inside dW too
    m, k, n = 1024, 264, 136
    X, _, DY, _ = _dense(m, k, n, "bf16")
    for f32 in (1, 0):
        dw = Guarded((k, n), torch.float32 if f32 else torch.bfloat16)
        eng.backward_dw(dw.t, f32, X, DY, m, k, n, "bf16", None, 1)
        eng.check()
        assert dw.intact() and not torch.isnan(dw.t.float()).any()


@pytest.mark.parametrize("tc", [0, 1])
def test_grouped_passes_write_only_their_outputs(eng, tc):
    m, k, n, e = 300, 136, 72, 5
    X, W, DY, I, offs, Xs, DYs = _grouped(m, k, n, e, "bf16")
    y, dx, dw = Guarded((m, n), torch.bfloat16), Guarded((m, k), torch.bfloat16), Guarded((e, n, k), torch.float32)
    eng.grouped_forward(y.t, X, W, I, m, k, n, e, "bf16", None, tc)
    eng.grouped_backward(dx.t, dw.t, X, W, DY, I, m, k, n, e, "bf16", None, tc)
    eng.check()
    for name, g in (("y", y), ("dx", dx), ("dw", dw)):
        assert g.intact(), (name, tc)
        assert not torch.isnan(g.t.float()).any(), (name, tc)
    strat = bi.BI_STRATEGY_TENSOR_CORE if tc else bi.BI_STRATEGY_SCALAR
    y2, dx2, dw2 = Guarded((m, n), torch.bfloat16), Guarded((m, k), torch.bfloat16), Guarded((e, n, k), torch.float32)
    eng.grouped_forward_segmented(y2.t, Xs, W, offs, m, k, n, e, "bf16", None, strat)
    eng.grouped_backward_segmented(dx2.t, dw2.t, Xs, W, DYs, offs, m, k, n, e, "bf16", None, strat)
    eng.check()
    for name, g in (("y seg", y2), ("dx seg", dx2), ("dw seg", dw2)):
        assert g.intact(), (name, tc)
        assert not torch.isnan(g.t.float()).any(), (name, tc)


def test_fp8_passes_write_only_their_outputs(eng):
    m, k, n = 300, 208, 144  # multiples of 16 for the 8-bit rows
    X, W, DY, B = _dense(m, k, n, "bf16")
    inv = torch.full((1,), 4.0, device="cuda")
    sc = torch.full((1,), 0.25, device="cuda")
    xq, wq, gq = Guarded((m, k), torch.uint8), Guarded((k, n), torch.uint8), Guarded((m, n), torch.uint8)
    amax = Guarded((3,), torch.float32)
    eng.fp8_quantize(xq.t, amax.t[0:1], X, inv, m * k, "bf16")
    eng.fp8_quantize(wq.t, amax.t[1:2], W, inv, k * n, "bf16")
    eng.fp8_quantize(gq.t, amax.t[2:3], DY, inv, m * n, "bf16")
    y, dx = Guarded((m, n), torch.bfloat16), Guarded((m, k), torch.bfloat16)
    dw, dw16 = Guarded((k, n), torch.float32), Guarded((k, n), torch.bfloat16)
    eng.fp8_forward(y.t, xq.t, wq.t, B, sc, sc, m, k, n, "bf16")
    eng.fp8_backward_dx(dx.t, gq.t, wq.t, sc, sc, m, k, n, "bf16")
    eng.fp8_backward_dw(dw.t, xq.t, gq.t, sc, sc, m, k, n, "f32")
    eng.fp8_backward_dw(dw16.t, xq.t, gq.t, sc, sc, m, k, n, "bf16")
    eng.check()
    for name, g in (("xq", xq), ("wq", wq), ("gq", gq), ("amax", amax), ("y", y), ("dx", dx), ("dw", dw),
                    ("dw16", dw16)):
        assert g.intact(), name


# ---------------------------------------------------------------- allocation failure

def _scratch_calls(eng):
    """(name, output tensor, call) for calls that take scratch from the pool."""
    calls = []
    m, k, n = 600, 64, 72  # 3 dW chunks: the scalar dW keeps chunk partials
    X, W, DY, B = _dense(m, k, n, "bf16", seed=5)
    dw = torch.zeros(k, n, device="cuda")
    calls.append(("scalar dW", dw, lambda: bi.bi_backward_dw(eng.handle, dw, 1, X, DY, m, k, n, "bf16", None, 0)))
    db = torch.zeros(n, device="cuda")
    calls.append(("bias grad", db, lambda: bi.bi_bias_grad(eng.handle, db, 1, DY, m, n, "bf16", None)))
    m2, k2, n2 = 1024, 256, 256  # one tile contracted in chunks: chunk scratch
    X2, _, DY2, _ = _dense(m2, k2, n2, "bf16", seed=6)
    dw2 = torch.zeros(k2, n2, device="cuda")
    calls.append(("tensor-core dW", dw2,
                  lambda: bi.bi_backward_dw(eng.handle, dw2, 1, X2, DY2, m2, k2, n2, "bf16", None, 1)))
    Xf, Wf, _, Bf = _dense(96, 128, 64, "f32", seed=7)
    yf = torch.zeros(96, 64, device="cuda")
    calls.append(("3xTF32 forward", yf,
                  lambda: bi.bi_forward(eng.handle, yf, Xf, Wf, Bf, 96, 128, 64, "f32", None, 1)))
    mg, kg, ng, eg = 300, 136, 72, 5
    Xg, Wg, DYg, I, offs, Xs, _ = _grouped(mg, kg, ng, eg, "bf16")
    for tc in (0, 1):
        yg = torch.zeros(mg, ng, dtype=torch.bfloat16, device="cuda")
        calls.append((f"grouped forward tc={tc}", yg,
                      lambda yg=yg, tc=tc: bi.bi_grouped_forward(eng.handle, yg, Xg, Wg, I, mg, kg, ng, eg, "bf16",
                                                                 None, tc)))
        dwg = torch.zeros(eg, ng, kg, device="cuda")
        calls.append((f"grouped backward tc={tc}", dwg,
                      lambda dwg=dwg, tc=tc: bi.bi_grouped_backward(eng.handle, None, dwg, Xg, Wg, DYg, I, mg, kg,
                                                                    ng, eg, "bf16", None, tc)))
    ys = torch.zeros(mg, ng, dtype=torch.bfloat16, device="cuda")
    calls.append(("segmented forward", ys,
                  lambda: bi.bi_grouped_forward_segmented(eng.handle, ys, Xs, Wg, offs, mg, kg, ng, eg, "bf16", None,
                                                          bi.BI_STRATEGY_TENSOR_CORE)))
    m8, k8, n8 = 2048, 256, 256  # FP8 dW with its tile in chunks
    xq = torch.randint(0, 0x60, (m8, k8), dtype=torch.uint8, device="cuda")
    gq = torch.randint(0, 0x60, (m8, n8), dtype=torch.uint8, device="cuda")
    one = torch.ones(1, device="cuda")
    dw8 = torch.zeros(k8, n8, device="cuda")
    calls.append(("FP8 dW", dw8,
                  lambda: bi.bi_fp8_backward_dw(eng.handle, dw8, xq, gq, one, one, m8, k8, n8, "f32", None)))
    return calls


def test_allocation_failure_returns_oom_and_enqueues_nothing(eng):
    for name, out, call in _scratch_calls(eng):
        assert call() == bi.BI_OK, (name, bi.bi_last_error(eng.handle))
        eng.check()
        want = out.clone()
        out.view(INT_VIEW[out.element_size()]).fill_(0x55)
        poisoned = out.clone()
        launches = eng.launches()
        assert bi.bi_engine_fail_allocations(eng.handle, 1) == bi.BI_OK
        assert call() == bi.BI_ERR_OOM, name
        assert "scratch" in bi.bi_last_error(eng.handle).lower() or "memory" in bi.bi_last_error(eng.handle).lower()
        assert eng.launches() == launches, name  # nothing was launched
        torch.cuda.synchronize()
        assert torch.equal(out, poisoned), name  # nothing was written
        # the one injected failure is used up: the engine works again, same bits
        assert call() == bi.BI_OK, (name, bi.bi_last_error(eng.handle))
        eng.check()
        assert torch.equal(out.view(INT_VIEW[out.element_size()]), want.view(INT_VIEW[out.element_size()])), name


def test_persistent_allocation_failure_spares_calls_without_scratch(eng):
    m, k, n = 64, 64, 72
    X, W, DY, B = _dense(m, k, n, "bf16", seed=8)
    y = torch.empty(m, n, dtype=torch.bfloat16, device="cuda")
    dw = torch.empty(k, n, device="cuda")
    assert bi.bi_engine_fail_allocations(eng.handle, -1) == bi.BI_OK
    try:
        # the forward and a single-chunk scalar dW need no scratch
        assert bi.bi_forward(eng.handle, y, X, W, B, m, k, n, "bf16", None, 1) == bi.BI_OK
        assert bi.bi_backward_dw(eng.handle, dw, 1, X, DY, m, k, n, "bf16", None, 0) == bi.BI_OK
        m3 = 600
        X3, _, DY3, _ = _dense(m3, k, n, "bf16", seed=9)
        for _ in range(2):  # every scratch allocation fails until the setting changes
            assert bi.bi_backward_dw(eng.handle, dw, 1, X3, DY3, m3, k, n, "bf16", None, 0) == bi.BI_ERR_OOM
    finally:
        assert bi.bi_engine_fail_allocations(eng.handle, 0) == bi.BI_OK
    assert bi.bi_backward_dw(eng.handle, dw, 1, X3, DY3, m3, k, n, "bf16", None, 0) == bi.BI_OK
    eng.check()
