"""Concurrent use: forward + backward steps of two problems issued on two CUDA
streams at once (persistent GEMM grids of both streams share the SMs, each
stream's GEMMs chained by programmatic dependent launch) give bit for bit the
results of the same calls run one after the other."""
import numpy as np
import pytest
import torch

from chunked_lm_head_gb300 import _lib
from chunked_lm_head_gb300 import workloads as WL

from gpu_util import upload

pytestmark = pytest.mark.gpu


def _step(h, W, t, w, chunk, ws, stream):
    N, H = h.shape
    V = W.shape[0]
    dev = h.device
    logp = torch.empty(N, dtype=torch.float32, device=dev)
    lse = torch.empty(N, dtype=torch.float32, device=dev)
    loss = torch.empty(1, dtype=torch.float32, device=dev)
    nv = torch.empty(1, dtype=torch.int64, device=dev)
    dH = torch.empty_like(h)
    dW = torch.empty((V, H), dtype=torch.float32, device=dev)
    n = ws.numel()
    with torch.cuda.stream(stream):
        assert _lib.flce_forward(h, W, t, w, N, H, V, chunk, -100, logp, lse, loss, nv, ws, n, stream) == 0
        # g on the device would need a sync; a fixed scale keeps the two streams independent
        assert _lib.flce_backward(h, W, t, w, lse, 1e-3, dH, dW, N, H, V, chunk, -100, ws, n, stream) == 0
    return logp, lse, loss, dH, dW


def test_two_streams_at_once_match_the_serial_results():
    cases = [WL.custom("s1", 3000, 512, 20000, 1024, w_std=0.04, targets="zipf", ignore_frac=0.05, seed=601),
             WL.custom("s2", 2200, 384, 30011, 256, w_std=0.05, targets="zipf", ignore_frac=0.1, seed=602)]
    data = [upload(WL.make_inputs(wl)) for wl in cases]
    wss = [torch.empty(_lib.flce_workspace_bytes(d[0].shape[0], d[0].shape[1], d[1].shape[0], wl.chunk_rows),
                       dtype=torch.uint8, device="cuda") for d, wl in zip(data, cases)]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    serial = []
    for (h, W, t, w), wl, ws, s in zip(data, cases, wss, streams):
        serial.append(_step(h, W, t, w, wl.chunk_rows, ws, s))
        torch.cuda.synchronize()
    for _ in range(3):  # issue both problems back to back, then wait for both
        both = [_step(h, W, t, w, wl.chunk_rows, ws, s)
                for (h, W, t, w), wl, ws, s in zip(data, cases, wss, streams)]
        torch.cuda.synchronize()
        assert _lib.flce_device_status() == 0
        for a, b in zip(serial, both):
            for x, y in zip(a, b):
                assert torch.equal(x, y)
