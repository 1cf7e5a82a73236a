"""GPU tests of the bias gradient and the PyTorch layer built on the C ABI.

The training check follows the sgemm-bi page's example (train twice from one
seed, compare the weights bit for bit, then check batch invariance).
"""
import numpy as np
import pytest
import torch

import oracle
import deterministic_invariant_gemm_fixed_gb300 as bi
from deterministic_invariant_gemm_fixed_gb300 import synth
from deterministic_invariant_gemm_fixed_gb300.nn import Linear, deterministic_linear
from helpers import out_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def eng():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    e = bi.Engine(0)
    yield e
    e.close()


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("m", [1, 255, 256, 257, 3000])
@pytest.mark.parametrize("n", [1000, 1001])  # 16-byte rows (vector path) and not
def test_bias_grad_bit_exact(eng, dtype, m, n):
    dy = synth.normal((m, n), 1.0, dtype, 50 + m)
    dyn = synth.to_np(dy)
    D = dy.cuda()
    for f32 in (1, 0):
        db = torch.empty(n, dtype=torch.float32 if (f32 or dtype == "f32") else synth.TORCH_DTYPES[dtype],
                         device="cuda")
        eng.bias_grad(db, f32, D, m, n, dtype)
        eng.check()
        assert np.array_equal(out_np(db), oracle.bias_grad(dyn, m, n, dtype, out_f32=bool(f32)))


def test_bias_grad_empty_batch(eng):
    db = torch.full((64,), 3.0, device="cuda")
    eng.bias_grad(db, 1, torch.zeros(1, 64, device="cuda"), 0, 64, "f32")
    eng.check()
    assert torch.all(db == 0)


@pytest.mark.parametrize("tc", [False, True])
def test_deterministic_linear_matches_the_oracle(eng, tc):
    m, k, n, dtype = 96, 128, 192, "bf16"
    x, w, g, b = synth.dense_inputs(m, k, n, dtype, w=("normal", 0.1))
    X = x.cuda().requires_grad_(True)
    W = w.cuda().requires_grad_(True)
    B = b.cuda().requires_grad_(True)
    y = deterministic_linear(X.reshape(4, 24, k), W, B, tensor_cores=tc)
    assert y.shape == (4, 24, n)
    y.backward(g.cuda().reshape(4, 24, n))
    xn, wn, gn, bn = (synth.to_np(t) for t in (x, w, g, b))
    got_y = out_np(y.detach().reshape(m, n))
    got = {"dx": out_np(X.grad), "dw": out_np(W.grad), "db": out_np(B.grad)}
    assert np.array_equal(got["db"], oracle.bias_grad(gn, m, n, dtype))
    if not tc:
        assert np.array_equal(got_y, oracle.forward(xn, wn, bn, m, k, n, dtype))
        assert np.array_equal(got["dx"], oracle.backward_dx(gn, wn, m, k, n, dtype))
        assert np.array_equal(got["dw"], oracle.backward_dw(xn, gn, m, k, n, dtype))
    else:
        # the layer passes exactly what the C ABI computes for the same call
        Y = torch.empty(m, n, dtype=torch.bfloat16, device="cuda")
        DX = torch.empty(m, k, dtype=torch.bfloat16, device="cuda")
        DW = torch.empty(k, n, dtype=torch.bfloat16, device="cuda")
        eng.forward(Y, x.cuda(), w.cuda(), b.cuda(), m, k, n, dtype, None, 1)
        eng.backward_dx(DX, g.cuda(), w.cuda(), m, k, n, dtype, None, 1)
        eng.backward_dw(DW, 0, x.cuda(), g.cuda(), m, k, n, dtype, None, 1)
        assert np.array_equal(got_y, out_np(Y))
        assert np.array_equal(got["dx"], out_np(DX))
        assert np.array_equal(got["dw"], out_np(DW))


def _mlp(tc, dtype, seed):
    torch.manual_seed(seed)
    return torch.nn.Sequential(
        Linear(64, 256, device="cuda", dtype=dtype, tensor_cores=tc), torch.nn.GELU(),
        Linear(256, 128, device="cuda", dtype=dtype, tensor_cores=tc), torch.nn.GELU(),
        Linear(128, 64, device="cuda", dtype=dtype, tensor_cores=tc))


def _train(tc, dtype, steps=15):
    model = _mlp(tc, dtype, seed=1234)
    opt = torch.optim.SGD(model.parameters(), lr=0.05)
    xs = synth.normal((steps, 256, 64), 1.0, "f32", 7).to(dtype).cuda()
    ts = synth.normal((steps, 256, 64), 1.0, "f32", 8).to(dtype).cuda()
    for i in range(steps):
        opt.zero_grad(set_to_none=True)
        loss = torch.nn.functional.mse_loss(model(xs[i]).float(), ts[i].float())
        loss.backward()
        opt.step()
    return model


@pytest.mark.parametrize("tc", [False, True])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_training_twice_gives_identical_weights(eng, tc, dtype):
    a = _train(tc, dtype)
    b = _train(tc, dtype)
    for (na, pa), (nb, pb) in zip(a.named_parameters(), b.named_parameters()):
        assert na == nb
        assert torch.equal(pa.detach().view(torch.uint8), pb.detach().view(torch.uint8)), na
    # the model is batch-invariant: any row computed alone equals its row in a batch
    x = synth.normal((64, 64), 1.0, "f32", 9).to(dtype).cuda()
    with torch.no_grad():
        full = a(x)
        for r in (0, 17, 63):
            assert torch.equal(a(x[r:r + 1]).view(torch.uint8), full[r:r + 1].view(torch.uint8))
        assert torch.equal(a(x[:7]).view(torch.uint8), full[:7].view(torch.uint8))


def test_from_torch_keeps_the_function(eng):
    torch.manual_seed(0)
    ref = torch.nn.Linear(96, 80, device="cuda", dtype=torch.float32)
    lay = Linear.from_torch(ref, tensor_cores=False)
    assert lay.weight.shape == (96, 80)
    x = torch.randn(33, 96, device="cuda")
    want = (x.double() @ ref.weight.double().t() + ref.bias.double()).float()
    got = lay(x)
    assert torch.allclose(got, want, rtol=1e-5, atol=1e-5)


@pytest.mark.parametrize("scales", [(1.0, 1.0, 1.0), (0.5, 2.0, 0.25)])
def test_fp8_route_matches_the_oracle_on_exact_integers(eng, scales):
    # Small integers and power-of-two scales: every e4m3 code, product and sum is
    # exact, so the layer's forward, dX, dW and bias gradient must equal the
    # oracle's FP8 definitions (quantize, scaled matmul, one rounding) bit for bit.
    from deterministic_invariant_gemm_fixed_gb300.nn import Fp8Scales
    m, k, n, dtype = 96, 64, 48, "bf16"
    sx, sw, sg = scales
    x = synth.small_ints((m, k), -8, 8, dtype, 31) * sx
    w = synth.small_ints((k, n), -8, 8, dtype, 32) * sw
    g = synth.small_ints((m, n), -8, 8, dtype, 33) * sg
    b = synth.small_ints((n,), -8, 8, dtype, 34) * 0.5
    X = x.cuda().requires_grad_(True)
    W = w.cuda().requires_grad_(True)
    B = b.cuda().requires_grad_(True)
    amax = torch.zeros(3, device="cuda")
    fp8 = Fp8Scales(sx, torch.tensor([sw], device="cuda"), sg, amax=amax)
    y = deterministic_linear(X.reshape(4, 24, k), W, B, fp8=fp8)
    y.backward(g.cuda().reshape(4, 24, n))
    xn, wn, gn, bn = (synth.to_np(t) for t in (x, w, g, b))
    xq, ax = oracle.fp8_quantize(xn, dtype, np.float32(1.0) / np.float32(sx))
    wq, aw = oracle.fp8_quantize(wn, dtype, np.float32(1.0) / np.float32(sw))
    gq, ag = oracle.fp8_quantize(gn, dtype, np.float32(1.0) / np.float32(sg))
    torch.cuda.synchronize()
    assert np.array_equal(out_np(amax), np.array([ax, aw, ag], dtype=np.float32))
    assert np.array_equal(out_np(y.detach().reshape(m, n)), oracle.fp8_forward(xq, wq, bn, sx, sw, m, k, n, dtype))
    assert np.array_equal(out_np(X.grad), oracle.fp8_backward_dx(gq, wq, sg, sw, m, k, n, dtype))
    assert np.array_equal(out_np(W.grad), oracle.fp8_backward_dw(xq, gq, sx, sg, m, k, n, dtype))
    assert np.array_equal(out_np(B.grad), oracle.bias_grad(gn, m, n, dtype))


def test_fp8_route_trains_bit_identically_twice(eng):
    from deterministic_invariant_gemm_fixed_gb300.nn import Fp8Scales

    def train():
        torch.manual_seed(99)
        lay = Linear(128, 96, device="cuda", dtype=torch.bfloat16)
        opt = torch.optim.SGD(lay.parameters(), lr=0.05)
        xs = synth.normal((6, 160, 128), 1.0, "bf16", 41).cuda()
        ts = synth.normal((6, 160, 96), 1.0, "bf16", 42).cuda()
        for i in range(6):
            opt.zero_grad(set_to_none=True)
            out = deterministic_linear(xs[i], lay.weight, lay.bias, fp8=Fp8Scales(1 / 64, 1 / 2048, 1 / 8192))
            torch.nn.functional.mse_loss(out.float(), ts[i].float()).backward()
            opt.step()
        return lay
    a, b = train(), train()
    for pa, pb in zip(a.parameters(), b.parameters()):
        assert torch.equal(pa.detach().view(torch.int16), pb.detach().view(torch.int16))
