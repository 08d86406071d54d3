"""Forward + backward with a caller workspace captured into a CUDA graph and
replayed: the replay reproduces the eager results bit for bit (the kernels
are deterministic), on new inputs copied into the captured buffers too."""
import numpy as np
import pytest
import torch

from chunked_lm_head_gb300 import _lib
from chunked_lm_head_gb300 import workloads as WL

from gpu_util import upload

pytestmark = pytest.mark.gpu


def test_forward_backward_graph_replay_matches_eager():
    wl = WL.custom("graph", 700, 256, 3000, 256, w_std=0.05, targets="zipf", ignore_frac=0.05, seed=801)
    inp = WL.make_inputs(wl)
    h, W, t, w = upload(inp)
    N, H, V, cr = wl.N, wl.H, wl.V, 256
    ws_bytes = _lib.flce_workspace_bytes(N, H, V, cr)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    bufs = dict(logp=torch.empty(N, device="cuda"), lse=torch.empty(N, device="cuda"),
                loss=torch.empty(1, device="cuda"), nv=torch.empty(1, dtype=torch.int64, device="cuda"),
                dH=torch.empty_like(h), dW=torch.empty((V, H), device="cuda"))
    g = 1.0 / int((inp.targets != -100).sum())

    def step():
        s1 = _lib.flce_forward(h, W, t, None, N, H, V, cr, -100, bufs["logp"], bufs["lse"],
                               bufs["loss"], bufs["nv"], ws, ws_bytes)
        s2 = _lib.flce_backward(h, W, t, None, bufs["lse"], g, bufs["dH"], bufs["dW"], N, H, V, cr,
                                -100, ws, ws_bytes)
        return s1, s2

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        assert step() == (0, 0)  # eager warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    eager = {k: v.clone() for k, v in bufs.items()}
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        assert step() == (0, 0)
    for v in bufs.values():
        v.zero_()
    graph.replay()
    torch.cuda.synchronize()
    for k in bufs:
        assert torch.equal(bufs[k], eager[k]), k
    # new inputs in the captured buffers: the replay follows them
    h2 = torch.from_numpy(WL.normal_bf16(99, 1, N * H, 1.0).view(np.int16)).cuda().view(torch.bfloat16)
    h.copy_(h2.view(N, H))
    graph.replay()
    torch.cuda.synchronize()
    ref_lse = bufs["lse"].clone()
    with torch.cuda.stream(side):
        assert step() == (0, 0)
    torch.cuda.synchronize()
    assert torch.equal(bufs["lse"], ref_lse)
    assert _lib.flce_device_status() == 0


def test_one_call_forward_backward_graph_replay_matches_eager():
    """flce_forward_backward (no logits recompute) with a caller workspace:
    captured, replayed, bit for bit the eager results."""
    wl = WL.custom("graph1", 700, 256, 3000, 768, w_std=0.05, targets="zipf", ignore_frac=0.05, seed=802)
    inp = WL.make_inputs(wl)
    h, W, t, w = upload(inp)
    N, H, V, cr = wl.N, wl.H, wl.V, 768
    ws_bytes = _lib.flce_forward_backward_workspace_bytes(N, H, V, cr)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    bufs = dict(logp=torch.empty(N, device="cuda"), lse=torch.empty(N, device="cuda"),
                loss=torch.empty(1, device="cuda"), nv=torch.empty(1, dtype=torch.int64, device="cuda"),
                dH=torch.empty_like(h), dW=torch.empty((V, H), device="cuda"))

    def step():
        return _lib.flce_forward_backward(h, W, t, None, N, H, V, cr, -100, None, 1.0, bufs["logp"],
                                          bufs["lse"], bufs["loss"], bufs["nv"], bufs["dH"], bufs["dW"],
                                          ws, ws_bytes)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        assert step() == 0
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    eager = {k: v.clone() for k, v in bufs.items()}
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        assert step() == 0
    for v in bufs.values():
        v.zero_()
    graph.replay()
    torch.cuda.synchronize()
    for k in bufs:
        assert torch.equal(bufs[k], eager[k]), k
    assert _lib.flce_device_status() == 0
