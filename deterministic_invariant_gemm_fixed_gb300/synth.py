"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module holds none of the method's arithmetic: it only draws numbers.
Values are drawn in float64 by numpy's PCG64 generator (platform independent),
then converted to the operand type by torch's own conversion, so the same seed
gives the same tensors on any host.  Every function returns CPU torch tensors;
callers move them to the device themselves.

Recipes (the workloads the library is exercised on):

* linear f32, M=64 K=256 N=512: X, W, dY ~ N(0,1), bias ~ N(0,0.1)
* GPT-2-small MLP up-projection bf16, M=4096 K=768 N=3072:
  X ~ N(0,1), W ~ N(0,0.02), dY ~ N(0,1e-3), bias ~ N(0,0.1)
* 7B-class layer bf16, M=8192: qkv 4096->12288, o 4096->4096,
  up 4096->11008, down 11008->4096; X ~ N(0,1), W ~ N(0,0.02), dY ~ N(0,1)
* f16 edge shapes (2048x1024x48, 1000^3, GEMV 1x4096x4096): X, W, dY ~ U(-1,1)
* grouped bf16, M=16384 K=2048 E=8 N=1408: W ~ N(0,0.02), X, dY ~ N(0,1),
  row ids uniform in [0,8) with exactly round(0.05*M) rows set to 8 (padding)

Seeds by role: X 1, W 2, dY 3, bias 4, ids 5 (a test may offset them).
"""
from __future__ import annotations

import numpy as np
import torch

SEED_X, SEED_W, SEED_DY, SEED_B, SEED_IDS = 1, 2, 3, 4, 5

TORCH_DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}


def _to(a64: np.ndarray, dtype: str) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a64)).to(TORCH_DTYPES[dtype])


def normal(shape, std: float, dtype: str, seed: int) -> torch.Tensor:
    rng = np.random.default_rng(seed)
    return _to(rng.standard_normal(size=shape) * std, dtype)


def uniform(shape, lo: float, hi: float, dtype: str, seed: int) -> torch.Tensor:
    rng = np.random.default_rng(seed)
    return _to(rng.uniform(lo, hi, size=shape), dtype)


def small_ints(shape, lo: int, hi: int, dtype: str, seed: int) -> torch.Tensor:
    """Integers uniform in [lo, hi], stored exactly in the operand type."""
    rng = np.random.default_rng(seed)
    return _to(rng.integers(lo, hi + 1, size=shape).astype(np.float64), dtype)


def expert_ids(m: int, e: int, pad_frac: float, seed: int, pad_id: int | None = None) -> torch.Tensor:
    """Row ids uniform in [0, e) with exactly round(pad_frac*m) rows set to
    pad_id (default e), chosen without replacement.  Returned as int64 holding
    the u32 values (torch lacks uint32 arithmetic on some versions)."""
    rng = np.random.default_rng(seed)
    ids = rng.integers(0, e, size=m).astype(np.int64)
    npad = int(round(pad_frac * m))
    if npad:
        rows = rng.choice(m, size=npad, replace=False)
        ids[rows] = e if pad_id is None else pad_id
    return torch.from_numpy(ids)


def to_np(t: torch.Tensor) -> np.ndarray:
    """Raw data of a tensor as numpy: float32 stays float32, bf16/f16 become the
    uint16 encodings, integer ids become uint32."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.float32:
        return t.numpy()
    if t.dtype in (torch.bfloat16, torch.float16):
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy().astype(np.uint32)


def from_np(a: np.ndarray, dtype: str) -> torch.Tensor:
    """Inverse of to_np for operand data."""
    if dtype == "f32":
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint16).view(np.int16)).view(TORCH_DTYPES[dtype])


# Named workloads ---------------------------------------------------------------

LINEAR_F32 = dict(name="linear_f32_64x256x512", dtype="f32", m=64, k=256, n=512,
                  x=("normal", 1.0), w=("normal", 1.0), dy=("normal", 1.0), b=("normal", 0.1))
GPT2_UP = dict(name="gpt2_small_mlp_up_bf16_4096x768x3072", dtype="bf16", m=4096, k=768, n=3072,
               x=("normal", 1.0), w=("normal", 0.02), dy=("normal", 1e-3), b=("normal", 0.1))
SEVEN_B = [  # (projection, K, N) of the 7B-class layer at M=8192
    ("qkv", 4096, 12288), ("o", 4096, 4096), ("up", 4096, 11008), ("down", 11008, 4096)]
SEVEN_B_M = 8192
F16_EDGE = [  # (name, M, K, N)
    ("n48_fallback", 2048, 1024, 48), ("ragged_1000", 1000, 1000, 1000), ("gemv", 1, 4096, 4096)]
GROUPED = dict(name="grouped_bf16_16384x2048_e8_n1408", dtype="bf16", m=16384, k=2048, n=1408, e=8,
               pad_frac=0.05)


def draw(spec, shape, dtype, seed):
    kind, p = spec
    if kind == "normal":
        return normal(shape, p, dtype, seed)
    if kind == "uniform":
        return uniform(shape, -p, p, dtype, seed)
    if kind == "ints":
        return small_ints(shape, -p, p, dtype, seed)
    raise ValueError(kind)


def dense_inputs(m, k, n, dtype, x=("normal", 1.0), w=("normal", 0.02), dy=("normal", 1.0),
                 b=("normal", 0.1), seed_offset=0):
    """X [M,K], W [K,N], dY [M,N], bias [N] (or None) on the CPU."""
    return (draw(x, (m, k), dtype, SEED_X + seed_offset),
            draw(w, (k, n), dtype, SEED_W + seed_offset),
            draw(dy, (m, n), dtype, SEED_DY + seed_offset),
            draw(b, (n,), dtype, SEED_B + seed_offset) if b is not None else None)


def grouped_inputs(m, k, n, e, dtype, pad_frac=0.05, x=("normal", 1.0), w=("normal", 0.02),
                   dy=("normal", 1.0), seed_offset=0):
    """X [M,K], W [E,N,K], dY [M,N], row ids [M] on the CPU."""
    return (draw(x, (m, k), dtype, SEED_X + seed_offset),
            draw(w, (e, n, k), dtype, SEED_W + seed_offset),
            draw(dy, (m, n), dtype, SEED_DY + seed_offset),
            expert_ids(m, e, pad_frac, SEED_IDS + seed_offset))
