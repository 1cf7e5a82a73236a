"""GPU parity of the FP8 e4m3 per-tensor-scaled linear through the C ABI.

Quantize: codes and amax bit-exact against the oracle.  Matmuls: bit-exact on
exact small-integer problems, within the tensor-core tolerance on random data,
run-to-run identical and batch-invariant.
"""
import numpy as np
import pytest
import torch

import oracle
import deterministic_invariant_gemm_fixed_gb300 as bi
from deterministic_invariant_gemm_fixed_gb300 import synth
from helpers import check_tc, out_np

pytestmark = pytest.mark.gpu
TD = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}


@pytest.fixture(scope="module")
def eng():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    e = bi.Engine(0)
    yield e
    e.close()


def u8(t):
    """e4m3 codes of a device tensor as a numpy uint8 array."""
    torch.cuda.synchronize()
    return t.cpu().numpy()


def scal(v):
    return torch.tensor([v], dtype=torch.float32, device="cuda")


def quantize(eng, t, scale_inv):
    q = torch.empty(t.shape, dtype=torch.uint8, device="cuda")
    amax = torch.full((1,), 7.0, dtype=torch.float32, device="cuda")
    dt = {torch.bfloat16: "bf16", torch.float16: "f16", torch.float32: "f32"}[t.dtype]
    eng.fp8_quantize(q, amax, t, scal(scale_inv), t.numel(), dt)
    return q, amax


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("scale_inv", [1.0, 0.37, 64.0])  # 64 drives many values past 448
def test_quantize_bit_exact(eng, dtype, scale_inv):
    x = synth.normal((3, 1001), 3.0, dtype, 80)
    q, amax = quantize(eng, x.cuda(), scale_inv)
    eng.check()
    want_q, want_amax = oracle.fp8_quantize(synth.to_np(x), dtype, scale_inv)
    assert np.array_equal(u8(q), want_q)
    assert out_np(amax)[0] == want_amax
    if scale_inv == 64.0:
        assert ((want_q & 0x7f) == 0x7e).sum() > 20  # saturation was exercised


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("offset", [0, 1, 3])  # 16-byte steps, and element by element from a misaligned start
def test_quantize_vector_and_element_paths_agree(eng, dtype, offset):
    count = 200003  # many 16-byte steps and a ragged tail
    x = synth.normal((count + 8,), 2.0, dtype, 81)
    src = x.cuda()[offset:offset + count]
    q = torch.empty(count + 16, dtype=torch.uint8, device="cuda")[offset:offset + count]
    amax = torch.zeros(1, device="cuda")
    eng.fp8_quantize(q, amax, src, scal(3.0), count, dtype)
    eng.check()
    want_q, want_amax = oracle.fp8_quantize(synth.to_np(x)[offset:offset + count], dtype, 3.0)
    assert np.array_equal(u8(q), want_q)
    assert out_np(amax)[0] == want_amax


def run_fp8(eng, xq, wq, gq, bias, sx, sw, sg, m, k, n, out):
    td = TD[out]
    y = torch.empty(m, n, dtype=td, device="cuda")
    dx = torch.empty(m, k, dtype=td, device="cuda")
    dw = torch.empty(k, n, dtype=td, device="cuda")
    eng.fp8_forward(y, xq, wq, bias, scal(sx), scal(sw), m, k, n, out)
    eng.fp8_backward_dx(dx, gq, wq, scal(sg), scal(sw), m, k, n, out)
    eng.fp8_backward_dw(dw, xq, gq, scal(sx), scal(sg), m, k, n, out)
    eng.check()
    return out_np(y), out_np(dx), out_np(dw)


def e4m3(a64):
    return torch.from_numpy(np.ascontiguousarray(a64, dtype=np.float32)).to(torch.float8_e4m3fn).view(torch.uint8)


@pytest.mark.parametrize("out", ["bf16", "f32"])
def test_fp8_exact_on_small_integers(eng, out):
    m, k, n = 300, 384, 272
    rng = np.random.default_rng(81)
    xi = rng.integers(-16, 17, size=(m, k))
    wi = rng.integers(-16, 17, size=(k, n))
    gi = rng.integers(-16, 17, size=(m, n))
    xq, wq, gq = e4m3(xi), e4m3(wi), e4m3(gi)
    sx, sw, sg = 0.25, 2.0, 0.5
    b = (rng.integers(-64, 64, size=n) / 4).astype(np.float64)
    bias = torch.from_numpy(b).to(TD[out]).cuda() if out != "f32" else None
    y, dx, dw = run_fp8(eng, xq.cuda(), wq.cuda(), gq.cuda(), bias, sx, sw, sg, m, k, n, out)
    bn = synth.to_np(bias.cpu()) if bias is not None else None
    assert np.array_equal(y, oracle.fp8_forward(xq.numpy(), wq.numpy(), bn, sx, sw, m, k, n, out))
    assert np.array_equal(dx, oracle.fp8_backward_dx(gq.numpy(), wq.numpy(), sg, sw, m, k, n, out))
    assert np.array_equal(dw, oracle.fp8_backward_dw(xq.numpy(), gq.numpy(), sx, sg, m, k, n, out))


def test_fp8_random_within_tolerance_and_invariant(eng):
    m, k, n, out = 640, 512, 768, "bf16"
    x = synth.normal((m, k), 1.0, "bf16", 82).cuda()
    w = synth.normal((k, n), 0.02, "bf16", 83).cuda()
    g = synth.normal((m, n), 1.0, "bf16", 84).cuda()
    si_x, si_w, si_g = 64.0, 4096.0, 64.0  # quantize with 1/scale; the matmuls take the scales
    xq, _ = quantize(eng, x, si_x)
    wq, _ = quantize(eng, w, si_w)
    gq, _ = quantize(eng, g, si_g)
    sx, sw, sg = 1 / si_x, 1 / si_w, 1 / si_g
    y, dx, dw = run_fp8(eng, xq, wq, gq, None, sx, sw, sg, m, k, n, out)
    xqn, wqn, gqn = u8(xq), u8(wq), u8(gq)
    xv, wv, gv = (oracle.up_e4m3(a).astype(np.float64) for a in (xqn, wqn, gqn))
    r = oracle.fp8_forward(xqn, wqn, None, sx, sw, m, k, n, "f32")
    ok, st = check_tc(y, r, (np.abs(xv) @ np.abs(wv)) * (np.float32(sx) * np.float32(sw)), out)
    assert ok, st
    r = oracle.fp8_backward_dx(gqn, wqn, sg, sw, m, k, n, "f32")
    ok, st = check_tc(dx, r, (np.abs(gv) @ np.abs(wv).T) * (np.float32(sg) * np.float32(sw)), out)
    assert ok, st
    r = oracle.fp8_backward_dw(xqn, gqn, sx, sg, m, k, n, "f32")
    ok, st = check_tc(dw, r, (np.abs(xv).T @ np.abs(gv)) * (np.float32(sx) * np.float32(sg)), out)
    assert ok, st
    # run to run and for a prefix of the batch
    for _ in range(2):
        again = run_fp8(eng, xq, wq, gq, None, sx, sw, sg, m, k, n, out)
        for a, b_ in zip((y, dx, dw), again):
            assert np.array_equal(a, b_)
    mp = 129
    part = run_fp8(eng, xq[:mp].contiguous(), wq, gq[:mp].contiguous(), None, sx, sw, sg, mp, k, n, out)
    assert np.array_equal(part[0], y[:mp]) and np.array_equal(part[1], dx[:mp])


def test_fp8_argument_checks(eng):
    h = eng.handle
    z8 = torch.zeros(64, 64, dtype=torch.uint8, device="cuda")
    y = torch.zeros(64, 64, dtype=torch.bfloat16, device="cuda")
    s = scal(1.0)
    assert bi.bi_fp8_forward(h, y, z8, z8, None, s, s, 64, 40, 64, "bf16", None) == bi.BI_ERR_UNSUPPORTED
    yf = torch.zeros(64, 64, dtype=torch.float32, device="cuda")
    assert bi.bi_fp8_forward(h, yf, z8, z8, y[0], s, s, 64, 64, 64, "f32", None) == bi.BI_ERR_UNSUPPORTED
    assert bi.bi_fp8_forward(h, y, z8, z8, None, None, s, 64, 64, 64, "bf16", None) == bi.BI_ERR_INVALID_ARG
    assert bi.bi_fp8_forward(h, y, z8, z8, None, s, s, 64, 64, 64, "bf16", None) == bi.BI_OK
    eng.check()


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
def test_quantize_special_values(eng, dtype):
    """NaN quantizes to the e4m3 NaN code, infinities saturate to +-448, and
    amax ignores NaN (an infinite input makes amax infinite)."""
    x = synth.normal((2, 500), 1.0, dtype, 85)
    flat = x.view(-1)
    flat[3] = float("nan")
    flat[10] = float("inf")
    flat[20] = float("-inf")
    flat[30] = float("nan")
    q, amax = quantize(eng, x.cuda(), 1.0)
    eng.check()
    want_q, want_amax = oracle.fp8_quantize(synth.to_np(x), dtype, 1.0)
    got = u8(q).reshape(-1)
    assert np.array_equal(got, want_q.reshape(-1))
    assert (got[3] & 0x7F) == 0x7F and (got[30] & 0x7F) == 0x7F
    assert got[10] == 0x7E and got[20] == 0xFE
    assert out_np(amax)[0] == want_amax and np.isinf(want_amax)
    # without the infinities, the NaN inputs leave the maximum finite
    flat[10] = 0.5
    flat[20] = -0.5
    q, amax = quantize(eng, x.cuda(), 1.0)
    eng.check()
    want_q, want_amax = oracle.fp8_quantize(synth.to_np(x), dtype, 1.0)
    assert out_np(amax)[0] == want_amax and np.isfinite(want_amax)


def test_fp8_dw_f32_in_pieces(eng):
    """The FP8 dW kept in f32 over 20000 rows (pieces of 8192): exact on small integers."""
    m, k, n = 20000, 128, 144
    rng = np.random.default_rng(86)
    xq = e4m3(rng.integers(-8, 9, size=(m, k)))
    gq = e4m3(rng.integers(-2, 3, size=(m, n)))
    dw = torch.empty(k, n, dtype=torch.float32, device="cuda")
    eng.fp8_backward_dw(dw, xq.cuda(), gq.cuda(), scal(0.5), scal(0.25), m, k, n, "f32")
    eng.check()
    assert np.array_equal(out_np(dw), oracle.fp8_backward_dw(xq.numpy(), gq.numpy(), 0.5, 0.25, m, k, n, "f32"))


@pytest.mark.parametrize("out", ["bf16", "f32"])
def test_fp8_dw_tail_chunks(eng, out):
    """2048 x 256 x 1024: 4 dW tiles, each contracting as 2 chunks of 1024 rows
    added by the dW tree, then scaled: within the tolerance, and run to run."""
    m, k, n = 2048, 256, 1024
    x = synth.normal((m, k), 1.0, "bf16", 87).cuda()
    g = synth.normal((m, n), 1.0, "bf16", 88).cuda()
    xq, _ = quantize(eng, x, 64.0)
    gq, _ = quantize(eng, g, 64.0)
    sx = sg = 1 / 64.0
    dw = torch.empty(k, n, dtype=TD[out], device="cuda")
    eng.fp8_backward_dw(dw, xq, gq, scal(sx), scal(sg), m, k, n, out)
    eng.check()
    got = out_np(dw)
    xqn, gqn = u8(xq), u8(gq)
    xv, gv = (oracle.up_e4m3(a).astype(np.float64) for a in (xqn, gqn))
    r = oracle.fp8_backward_dw(xqn, gqn, sx, sg, m, k, n, "f32")
    ok, st = check_tc(got, r, (np.abs(xv).T @ np.abs(gv)) * (np.float32(sx) * np.float32(sg)), out)
    assert ok, st
    eng.fp8_backward_dw(dw, xq, gq, scal(sx), scal(sg), m, k, n, out)
    assert np.array_equal(out_np(dw), got)

