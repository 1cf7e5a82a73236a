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
"""
from __future__ import annotations

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


def deterministic_linear(x: torch.Tensor, weight: torch.Tensor, bias: torch.Tensor | None = None,
                         tensor_cores: bool = True) -> torch.Tensor:
    """y = x @ weight (+ bias) with weight [in, out]; bit-reproducible forward and
    backward (scalar tier with tensor_cores=False, tcgen05 tier otherwise)."""
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
