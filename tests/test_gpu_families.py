"""Tile families of the tensor-core tier give bit-identical results.

The sgemm-bi page ("Determinism contracts") runs its tensor-core tier in two
tile families and states that they agree bit for bit.  Here the families are
the output-tile widths of the CTA-pair kernel (256 and 128 columns for every
16-bit dense and grouped pass, 176 and 192 as well for the grouped forward;
bi_engine_set_tile_cols forces one).  A tile's width only decides which outputs
share a work unit; each output is the same ascending chain of 64-wide
contraction blocks, so Y, dX and dW must be equal for every width, including
the automatic choice (256 columns, or 128 for a 16-bit dW whose 256-column
tiling gives few work units).
"""
import numpy as np
import pytest
import torch

import deterministic_invariant_gemm_fixed_gb300 as bi
from deterministic_invariant_gemm_fixed_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture()
def eng():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    e = bi.Engine(0)
    yield e
    bi.bi_engine_set_tile_cols(e.handle, 0)
    e.close()


def _bits(t):
    torch.cuda.synchronize()
    return t.view(torch.int32 if t.element_size() == 4 else torch.int16).cpu().numpy()


def _dense_all(eng, X, W, DY, B, m, k, n, dtype):
    tdt = synth.TORCH_DTYPES[dtype]
    Y = torch.empty(m, n, dtype=tdt, device="cuda")
    DX = torch.empty(m, k, dtype=tdt, device="cuda")
    DW = torch.empty(k, n, dtype=torch.float32, device="cuda")
    DWr = torch.empty(k, n, dtype=tdt, device="cuda")
    eng.forward(Y, X, W, B, m, k, n, dtype, None, 1)
    eng.backward_dx(DX, DY, W, m, k, n, dtype, None, 1)
    eng.backward_dw(DW, 1, X, DY, m, k, n, dtype, None, 1)
    eng.backward_dw(DWr, 0, X, DY, m, k, n, dtype, None, 1)
    eng.check()
    return [_bits(t) for t in (Y, DX, DW, DWr)]


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("m,k,n", [(700, 520, 392), (1024, 4096, 1024), (9000, 264, 136)])
def test_dense_families_are_bit_identical(eng, dtype, m, k, n):
    x, w, dy, b = synth.dense_inputs(m, k, n, dtype, w=("normal", 0.05))
    X, W, DY, B = x.cuda(), w.cuda(), dy.cuda(), b.cuda()
    ref = _dense_all(eng, X, W, DY, B, m, k, n, dtype)  # automatic widths
    for cols in (256, 128):
        assert bi.bi_engine_set_tile_cols(eng.handle, cols) == bi.BI_OK
        got = _dense_all(eng, X, W, DY, B, m, k, n, dtype)
        for name, g_, r_ in zip(("y", "dx", "dw f32", "dw"), got, ref):
            assert np.array_equal(g_, r_), (name, cols, m, k, n, dtype)


@pytest.mark.parametrize("n", [1408, 392])
def test_grouped_families_are_bit_identical(eng, n):
    m, k, e, dtype = 3000, 136, 6, "bf16"
    x, w, dy, ids = synth.grouped_inputs(m, k, n, e, dtype, pad_frac=0.05)
    X, W, DY = x.cuda(), w.cuda(), dy.cuda()
    I = torch.from_numpy(synth.to_np(ids).astype(np.int32)).cuda()

    def run():
        Y = torch.empty(m, n, dtype=torch.bfloat16, device="cuda")
        DX = torch.empty(m, k, dtype=torch.bfloat16, device="cuda")
        DW = torch.empty(e, n, k, dtype=torch.float32, device="cuda")
        eng.grouped_forward(Y, X, W, I, m, k, n, e, dtype, None, 1)
        eng.grouped_backward(DX, DW, X, W, DY, I, m, k, n, e, dtype, None, 1)
        eng.check()
        return [_bits(t) for t in (Y, DX, DW)]
    ref = run()
    for cols in (256, 192, 176, 128):
        assert bi.bi_engine_set_tile_cols(eng.handle, cols) == bi.BI_OK
        got = run()
        for name, g_, r_ in zip(("y", "dx", "dw"), got, ref):
            assert np.array_equal(g_, r_), (name, cols, n)


def test_tile_cols_setting_is_checked(eng):
    assert bi.bi_engine_set_tile_cols(eng.handle, 64) == bi.BI_ERR_INVALID_ARG
    assert bi.bi_engine_set_tile_cols(eng.handle, 0) == bi.BI_OK
    assert bi.bi_engine_set_tile_cols(None, 128) == bi.BI_ERR_INVALID_ARG
