"""PyTorch layer over the C ABI: a linear layer whose three matmuls and bias
gradient run in libbi's deterministic kernels.

Sources: sgemm-bi 0.1.1.post2, "Use" -- a drop-in `Linear(in, out, ...,
tensor_cores=...)` whose weight is stored [in, out], `Linear.from_torch` for
converting existing layers, and the functional `deterministic_linear(x,
weight, bias, tensor_cores)`; ViperLLM ffma.py, `_FFMAAddmm` -- an autograd
function that saves the original x and W and returns gx = gy W^T, gW = x^T gy
and gb = column sums of gy.

Everything numeric happens in the library: this module only reshapes tensors,
allocates outputs with torch and passes pointers and the current stream.  The
bias gradient comes from bi_bias_grad (fixed-order column sum) instead of
torch's reduction, so a whole training step is bit-reproducible.

FP8 route (AstrAI csrc/kernels/fp8_mm.cu, fp8_linear_forward_scaled and
fp8_linear_backward_scaled): with `fp8=Fp8Scales(...)`, the forward quantizes
x and the weight to e4m3 with the caller's per-tensor scales (codes =
e4m3(value / scale)), multiplies the codes on the tensor cores and scales the
f32 product by scale_x * scale_w, then adds the bias and rounds once; the
backward quantizes the output gradient with scale_g and computes dX and dW from
the saved codes the same way.  The bias gradient is the fixed-order column sum
of the unquantized output gradient.
"""
from __future__ import annotations

import dataclasses
import math
import threading

import torch

from . import Engine

_engines: dict[int, Engine] = {}
_engines_lock = threading.Lock()


def engine_for(device: torch.device) -> Engine:
    """One engine per CUDA device, created on first use."""
    idx = device.index if device.index is not None else torch.cuda.current_device()
    with _engines_lock:
        eng = _engines.get(idx)
        if eng is None:
            eng = Engine(idx)
            _engines[idx] = eng
        return eng


def _check(x: torch.Tensor, weight: torch.Tensor, bias):
    if not (x.is_cuda and weight.is_cuda):
        raise ValueError("deterministic_linear needs CUDA tensors")
    if x.dtype != weight.dtype or (bias is not None and bias.dtype != x.dtype):
        raise TypeError("x, weight and bias must share one dtype (float32, bfloat16 or float16)")
    if weight.dim() != 2 or x.shape[-1] != weight.shape[0]:
        raise ValueError(f"weight must be [in, out] with in = x.shape[-1]; got {tuple(weight.shape)}")
    if bias is not None and bias.shape != (weight.shape[1],):
        raise ValueError("bias must be [out]")


class _DeterministicLinear(torch.autograd.Function):
    @staticmethod
    def forward(ctx, x, weight, bias, tensor_cores):
        _check(x, weight, bias)
        k, n = weight.shape
        x2 = x.reshape(-1, k).contiguous()
        w = weight.contiguous()
        b = bias.contiguous() if bias is not None else None
        m = x2.shape[0]
        y = torch.empty(m, n, dtype=x.dtype, device=x.device)
        eng = engine_for(x.device)
        eng.forward(y, x2, w, b, m, k, n, x.dtype, torch.cuda.current_stream(x.device), int(tensor_cores))
        ctx.save_for_backward(x2, w)
        ctx.has_bias = bias is not None
        ctx.tensor_cores = int(tensor_cores)
        ctx.x_shape = x.shape
        return y.reshape(*x.shape[:-1], n)

    @staticmethod
    def backward(ctx, gy):
        x2, w = ctx.saved_tensors
        k, n = w.shape
        gy2 = gy.reshape(-1, n).to(w.dtype).contiguous()
        m = gy2.shape[0]
        eng = engine_for(w.device)
        stream = torch.cuda.current_stream(w.device)
        tc = ctx.tensor_cores
        gx = gw = gb = None
        if ctx.needs_input_grad[0]:
            gx = torch.empty(m, k, dtype=w.dtype, device=w.device)
            eng.backward_dx(gx, gy2, w, m, k, n, w.dtype, stream, tc)
            gx = gx.reshape(ctx.x_shape)
        if ctx.needs_input_grad[1]:
            gw = torch.empty(k, n, dtype=w.dtype, device=w.device)
            eng.backward_dw(gw, int(w.dtype == torch.float32), x2, gy2, m, k, n, w.dtype, stream, tc)
        if ctx.has_bias and ctx.needs_input_grad[2]:
            gb = torch.empty(n, dtype=w.dtype, device=w.device)
            eng.bias_grad(gb, int(w.dtype == torch.float32), gy2, m, n, w.dtype, stream)
        return gx, gw, gb, None


@dataclasses.dataclass
class Fp8Scales:
    """Per-tensor scales of the FP8 route: a value v is stored as the e4m3 code
    of v / scale.  Each scale is a float or a one-element float32 CUDA tensor.
    `amax`, if given, is a float32 CUDA tensor of 3 elements that receives the
    maximum |value| of x and of the weight (forward) and of the output gradient
    (backward), for a caller that derives the next step's scales from them."""
    scale_x: float | torch.Tensor
    scale_w: float | torch.Tensor
    scale_g: float | torch.Tensor
    amax: torch.Tensor | None = None


def _scale_pair(s, device):
    """(scale, 1 / scale) as one-element f32 tensors on device (the reciprocal is
    taken by torch on the device; power-of-two scales have exact reciprocals)."""
    t = (s if isinstance(s, torch.Tensor) else torch.tensor([float(s)])).to(device=device, dtype=torch.float32)
    t = t.reshape(1).contiguous()
    return t, torch.reciprocal(t)


def _amax_slot(amax, i, device):
    if amax is None:
        return torch.empty(1, dtype=torch.float32, device=device)
    if not (amax.is_cuda and amax.dtype == torch.float32 and amax.numel() == 3 and amax.is_contiguous()):
        raise ValueError("Fp8Scales.amax must be a contiguous float32 CUDA tensor of 3 elements")
    return amax[i:i + 1]


class _DeterministicLinearFp8(torch.autograd.Function):
    @staticmethod
    def forward(ctx, x, weight, bias, fp8):
        _check(x, weight, bias)
        if x.dtype not in (torch.bfloat16, torch.float16):
            raise TypeError("the FP8 route takes bfloat16 or float16 x and weight")
        k, n = weight.shape
        x2 = x.reshape(-1, k).contiguous()
        w = weight.contiguous()
        b = bias.contiguous() if bias is not None else None
        m = x2.shape[0]
        dev = x.device
        eng = engine_for(dev)
        stream = torch.cuda.current_stream(dev)
        sx, sx_inv = _scale_pair(fp8.scale_x, dev)
        sw, sw_inv = _scale_pair(fp8.scale_w, dev)
        xq = torch.empty(m, k, dtype=torch.uint8, device=dev)
        wq = torch.empty(k, n, dtype=torch.uint8, device=dev)
        eng.fp8_quantize(xq, _amax_slot(fp8.amax, 0, dev), x2, sx_inv, m * k, x.dtype, stream)
        eng.fp8_quantize(wq, _amax_slot(fp8.amax, 1, dev), w, sw_inv, k * n, x.dtype, stream)
        y = torch.empty(m, n, dtype=x.dtype, device=dev)
        eng.fp8_forward(y, xq, wq, b, sx, sw, m, k, n, x.dtype, stream)
        ctx.save_for_backward(xq, wq, sx, sw)
        ctx.fp8 = fp8
        ctx.dtype = x.dtype
        ctx.has_bias = bias is not None
        ctx.x_shape = x.shape
        return y.reshape(*x.shape[:-1], n)

    @staticmethod
    def backward(ctx, gy):
        xq, wq, sx, sw = ctx.saved_tensors
        k, n = wq.shape
        dt = ctx.dtype
        gy2 = gy.reshape(-1, n).to(dt).contiguous()
        m = gy2.shape[0]
        dev = wq.device
        eng = engine_for(dev)
        stream = torch.cuda.current_stream(dev)
        sg, sg_inv = _scale_pair(ctx.fp8.scale_g, dev)
        gq = torch.empty(m, n, dtype=torch.uint8, device=dev)
        eng.fp8_quantize(gq, _amax_slot(ctx.fp8.amax, 2, dev), gy2, sg_inv, m * n, dt, stream)
        gx = gw = gb = None
        if ctx.needs_input_grad[0]:
            gx = torch.empty(m, k, dtype=dt, device=dev)
            eng.fp8_backward_dx(gx, gq, wq, sg, sw, m, k, n, dt, stream)
            gx = gx.reshape(ctx.x_shape)
        if ctx.needs_input_grad[1]:
            gw = torch.empty(k, n, dtype=dt, device=dev)
            eng.fp8_backward_dw(gw, xq, gq, sx, sg, m, k, n, dt, stream)
        if ctx.has_bias and ctx.needs_input_grad[2]:
            gb = torch.empty(n, dtype=dt, device=dev)
            eng.bias_grad(gb, 0, gy2, m, n, dt, stream)
        return gx, gw, gb, None


def deterministic_linear(x: torch.Tensor, weight: torch.Tensor, bias: torch.Tensor | None = None,
                         tensor_cores: bool = True, fp8: Fp8Scales | None = None) -> torch.Tensor:
    """y = x @ weight (+ bias) with weight [in, out]; bit-reproducible forward and
    backward (scalar tier with tensor_cores=False, tcgen05 tier otherwise).
    With fp8 (Fp8Scales), the three matmuls run on e4m3 codes of x, the weight
    and the output gradient, quantized with the given per-tensor scales, on the
    tensor cores (tensor_cores is then ignored)."""
    if fp8 is not None:
        return _DeterministicLinearFp8.apply(x, weight, bias, fp8)
    return _DeterministicLinear.apply(x, weight, bias, tensor_cores)


class Linear(torch.nn.Module):
    """Linear layer with the weight stored [in, out] (the layout the library's
    matmuls read without a transpose)."""

    def __init__(self, in_features: int, out_features: int, bias: bool = True, device=None,
                 dtype=None, tensor_cores: bool = True):
        super().__init__()
        self.in_features, self.out_features = in_features, out_features
        self.tensor_cores = tensor_cores
        self.weight = torch.nn.Parameter(torch.empty(in_features, out_features, device=device, dtype=dtype))
        self.bias = torch.nn.Parameter(torch.empty(out_features, device=device, dtype=dtype)) if bias else None
        self.reset_parameters()

    def reset_parameters(self):
        # the usual uniform(-1/sqrt(in), 1/sqrt(in)) initialisation of a linear layer
        bound = 1.0 / math.sqrt(self.in_features)
        with torch.no_grad():
            self.weight.uniform_(-bound, bound)
            if self.bias is not None:
                self.bias.uniform_(-bound, bound)

    @classmethod
    def from_torch(cls, layer: torch.nn.Linear, tensor_cores: bool = True) -> "Linear":
        """Convert a torch.nn.Linear (weight [out, in]) into this layout."""
        new = cls(layer.in_features, layer.out_features, bias=layer.bias is not None,
                  device=layer.weight.device, dtype=layer.weight.dtype, tensor_cores=tensor_cores)
        with torch.no_grad():
            new.weight.copy_(layer.weight.t())
            if layer.bias is not None:
                new.bias.copy_(layer.bias)
        return new

    def forward(self, x: torch.Tensor) -> torch.Tensor:
        return deterministic_linear(x, self.weight, self.bias, self.tensor_cores)

    def extra_repr(self) -> str:
        return (f"in_features={self.in_features}, out_features={self.out_features}, "
                f"bias={self.bias is not None}, tensor_cores={self.tensor_cores}")
