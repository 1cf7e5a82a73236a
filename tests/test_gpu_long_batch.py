"""A batch long enough that dW has more row chunks than one grid dimension
holds (65535).

The rublas page ("Determinism" / dW reduction) cuts the batch rows of dW into
fixed chunks and adds the chunk results by a fixed tree; nothing there bounds
the number of chunks.  At M = 65535 * 256 + 612 rows there are 65538 chunks of
256, so the chunk kernels run in two slices of the grid and the tree reads
partials written by both.

The inputs are small integers, so every partial sum in any order is an exact
f32 integer and the expected result is exact whatever the tier: with
X[m, r] = 1 + (m + r) mod 2 and dY[m, c] = 1 for the last L_c rows (else 0),
dW[r, c] is the sum of X[m, r] over those rows and the bias gradient is L_c.
L_c = 37 + 300 c reaches back about 84 chunks, across the boundary between the
two slices.  The expected values are this closed form, computed in numpy over
the last rows only.
"""
import numpy as np
import pytest
import torch

import deterministic_invariant_gemm_fixed_gb300 as bi

pytestmark = pytest.mark.gpu

M = 65535 * 256 + 612
assert (M + 255) // 256 == 65538


@pytest.fixture(scope="module")
def eng():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    e = bi.Engine(0)
    yield e
    e.close()


def lengths(n):
    return 37 + 300 * np.arange(n, dtype=np.int64)


def inputs(k, n):
    L = torch.from_numpy(lengths(n)).cuda()
    mi = torch.arange(M, device="cuda", dtype=torch.int64)
    x = ((mi[:, None] + torch.arange(k, device="cuda")[None, :]) % 2 + 1).to(torch.bfloat16)
    dy = (mi[:, None] >= (M - L)[None, :]).to(torch.bfloat16)
    del mi
    return x, dy


def expected_dw(k, n):
    L = lengths(n)
    ms = np.arange(M - L.max(), M, dtype=np.int64)
    out = np.empty((k, n), dtype=np.float64)
    for r in range(k):
        xv = 1 + (ms + r) % 2
        for c in range(n):
            out[r, c] = xv[ms >= M - L[c]].sum()
    return out.astype(np.float32)


@pytest.mark.parametrize("k,n,tc", [(8, 48, 0), (8, 72, 0), (64, 64, 1)],
                         ids=["narrow-kernel", "chunk-kernel", "tensor-core"])
def test_dw_with_more_chunks_than_a_grid_dimension(eng, k, n, tc):
    x, dy = inputs(k, n)
    assert bi.bi_dispatch_tier(bi.BI_PASS_DW, "bf16", tc, k, n) == tc
    dw = torch.full((k, n), float("nan"), dtype=torch.float32, device="cuda")
    eng.backward_dw(dw, 1, x, dy, M, k, n, "bf16", None, tc)
    eng.check()
    assert np.array_equal(dw.cpu().numpy(), expected_dw(k, n))
    if tc == 0:
        db = torch.full((n,), float("nan"), dtype=torch.float32, device="cuda")
        eng.bias_grad(db, 1, dy, M, n, "bf16")
        eng.check()
        assert np.array_equal(db.cpu().numpy(), lengths(n).astype(np.float32))
    del x, dy
    torch.cuda.empty_cache()


def test_grouped_dweights_with_more_chunks_than_a_grid_dimension(eng):
    k, n, e = 8, 72, 1
    x, dy = inputs(k, n)
    w = torch.ones(e, n, k, dtype=torch.bfloat16, device="cuda")
    ids = torch.zeros(M, dtype=torch.int32, device="cuda")
    dx = torch.empty(M, k, dtype=torch.bfloat16, device="cuda")
    dw = torch.full((e, n, k), float("nan"), dtype=torch.float32, device="cuda")
    eng.grouped_backward(dx, dw, x, w, dy, ids, M, k, n, e, "bf16", None, 0)
    eng.check()
    assert np.array_equal(dw[0].cpu().numpy(), expected_dw(k, n).T)
    # dX[m, :] = sum over c of dY[m, c] (W all ones): the number of L_c reaching row m
    tail = dx[-int(lengths(n).max()) - 5:].float().cpu().numpy()
    ms = np.arange(M - tail.shape[0], M)
    want = (ms[:, None] >= M - lengths(n)[None, :]).sum(axis=1).astype(np.float32)
    assert np.array_equal(tail, np.repeat(want[:, None], k, axis=1))
    del x, dy, dx
    torch.cuda.empty_cache()
