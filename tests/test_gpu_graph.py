"""The C ABI under CUDA graph capture: every pass enqueues only stream-ordered
work (pool scratch, kernels, event fork/join), so a captured graph replays
the same bits as eager calls, on new data written into the captured buffers."""
import numpy as np
import pytest
import torch

import deterministic_invariant_gemm_fixed_gb300 as bi
from deterministic_invariant_gemm_fixed_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def eng():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    e = bi.Engine(0)
    yield e
    e.close()


def _dense(eng, bufs, stream, tc):
    m, k, n = bufs["shape"]
    h = stream.cuda_stream
    eng.forward(bufs["y"], bufs["x"], bufs["w"], bufs["b"], m, k, n, "bf16", h, tc)
    eng.backward_dx(bufs["dx"], bufs["dy"], bufs["w"], m, k, n, "bf16", h, tc)
    eng.backward_dw(bufs["dw"], 1, bufs["x"], bufs["dy"], m, k, n, "bf16", h, tc)


def _grouped(eng, g, stream):
    m, k, n, e = g["shape"]
    h = stream.cuda_stream
    eng.grouped_forward(g["y"], g["x"], g["w"], g["ids"], m, k, n, e, "bf16", h, 1)
    eng.grouped_backward(g["dx"], g["dw"], g["x"], g["w"], g["dy"], g["ids"], m, k, n, e, "bf16", h, 1)


def _snap(d, keys):
    torch.cuda.synchronize()
    return {key: d[key].detach().cpu().clone() for key in keys}


def test_graph_replay_equals_eager(eng):
    m, k, n = 520, 264, 776
    x, w, dy, b = synth.dense_inputs(m, k, n, "bf16")
    dense = {"shape": (m, k, n), "x": x.cuda(), "w": w.cuda(), "dy": dy.cuda(), "b": b.cuda(),
             "y": torch.empty(m, n, dtype=torch.bfloat16, device="cuda"),
             "dx": torch.empty(m, k, dtype=torch.bfloat16, device="cuda"),
             "dw": torch.empty(k, n, dtype=torch.float32, device="cuda")}
    gm, gk, gn, ge = 1500, 192, 264, 6
    gx, gw, gdy, gids = synth.grouped_inputs(gm, gk, gn, ge, "bf16", pad_frac=0.05)
    grp = {"shape": (gm, gk, gn, ge), "x": gx.cuda(), "w": gw.cuda(), "dy": gdy.cuda(),
           "ids": torch.from_numpy(synth.to_np(gids).astype(np.int32)).cuda(),
           "y": torch.empty(gm, gn, dtype=torch.bfloat16, device="cuda"),
           "dx": torch.empty(gm, gk, dtype=torch.bfloat16, device="cuda"),
           "dw": torch.empty(ge, gn, gk, dtype=torch.float32, device="cuda")}
    outs = ("y", "dx", "dw")
    s = torch.cuda.Stream()
    # eager warm-up (first calls configure the kernels), then reference results
    with torch.cuda.stream(s):
        for tc in (0, 1):
            _dense(eng, dense, s, tc)
        _grouped(eng, grp, s)
    eng.check()

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        _dense(eng, dense, s, 1)
        _grouped(eng, grp, s)

    for seed in (11, 12):  # new inputs in the captured buffers
        x2, w2, dy2, b2 = synth.dense_inputs(m, k, n, "bf16", seed_offset=seed)
        for key, t in (("x", x2), ("w", w2), ("dy", dy2), ("b", b2)):
            dense[key].copy_(t)
        gx2, gw2, gdy2, gids2 = synth.grouped_inputs(gm, gk, gn, ge, "bf16", pad_frac=0.05, seed_offset=seed)
        for key, t in (("x", gx2), ("w", gw2), ("dy", gdy2)):
            grp[key].copy_(t)
        grp["ids"].copy_(torch.from_numpy(synth.to_np(gids2).astype(np.int32)))
        torch.cuda.synchronize()
        g.replay()
        got_d, got_g = _snap(dense, outs), _snap(grp, outs)
        with torch.cuda.stream(s):
            _dense(eng, dense, s, 1)
            _grouped(eng, grp, s)
        eng.check()
        want_d, want_g = _snap(dense, outs), _snap(grp, outs)
        for key in outs:
            assert torch.equal(got_d[key].view(torch.uint8), want_d[key].view(torch.uint8)), key
            assert torch.equal(got_g[key].view(torch.uint8), want_g[key].view(torch.uint8)), key
