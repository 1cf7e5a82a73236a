"""The grouped forward that allocates nothing (bi_grouped_forward_noalloc).

It serves callers that cannot allocate GPU memory when they run it: its
grouping scratch is a fixed array inside the library instead of memory taken
from a pool.  This test calls it through the C ABI twice in a row, on different
inputs, and checks each result against the allocating entry point
(bi_grouped_forward on the scalar tier), bit for bit -- the scalar tier's
tolerance.  The second call also shows that nothing left in the shared array by
the first call leaks into the next one.  It is collected last so that a failing
run stopping at the first failure has already run everything else, and it
creates everything it needs, so it also passes alone in a fresh process.
"""
import numpy as np
import pytest
import torch

import deterministic_invariant_gemm_fixed_gb300 as bi
from deterministic_invariant_gemm_fixed_gb300 import synth

pytestmark = pytest.mark.gpu


def _inputs(m, k, n, e, dtype, seed):
    x, w, dy, ids = synth.grouped_inputs(m, k, n, e, dtype, pad_frac=0.05, seed_offset=seed)
    return x.cuda(), w.cuda(), torch.from_numpy(synth.to_np(ids).astype(np.int32)).cuda()


def _bits(t):
    return t.view(torch.int32 if t.element_size() == 4 else torch.int16)


def test_noalloc_grouped_forward_matches_the_allocating_entry_point():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    eng = bi.Engine(0)
    stream = torch.cuda.current_stream()
    cases = [  # calls in a row; each has more rows or experts than the one before
        (700, 96, 136, 5, "bf16", 1),
        (3000, 64, 200, 9, "f16", 2),
        (3100, 40, 24, 11, "f32", 3),
    ]
    for m, k, n, e, dtype, seed in cases:
        x, w, ids = _inputs(m, k, n, e, dtype, seed)
        tdt = synth.TORCH_DTYPES[dtype]
        want = torch.empty(m, n, dtype=tdt, device="cuda")
        eng.grouped_forward(want, x, w, ids, m, k, n, e, dtype, stream, 0)
        for repeat in range(2):
            got = torch.full((m, n), float("nan"), dtype=tdt, device="cuda")
            torch.cuda.synchronize()
            free0, torch0 = torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated()
            st = bi.bi_grouped_forward_noalloc(got, x, w, ids, m, k, n, e, dtype, stream)
            assert st == bi.BI_OK, bi.bi_last_error(None)
            torch.cuda.synchronize()
            if repeat:  # the first call of a dtype may load its kernels; a repeat allocates nothing at all
                assert torch.cuda.mem_get_info()[0] == free0, (m, k, n, e, dtype)
                assert torch.cuda.memory_allocated() == torch0
            assert torch.equal(_bits(got), _bits(want)), (m, k, n, e, dtype, repeat)
    # a call needing more scratch than the fixed array holds is refused up front
    x, w, ids = _inputs(64, 64, 64, 4, "bf16", 3)
    y = torch.empty(64, 64, dtype=torch.bfloat16, device="cuda")
    st = bi.bi_grouped_forward_noalloc(y, x, w, ids, 4 << 20, 64, 64, 4, "bf16", stream)
    assert st == bi.BI_ERR_UNSUPPORTED
    assert "scratch" in bi.bi_last_error(None)
    eng.close()
