"""The torch-facing API (chunked_lm_head_gb300.api): autograd wrapper against
the oracle, and the extra device memory of a forward+backward."""
import numpy as np
import pytest
import torch

import chunked_lm_head_gb300 as flce
from chunked_lm_head_gb300 import workloads as WL
from oracle import flce_oracle as O

from gpu_util import LOSS_RTOL, assert_grad_close, assert_logp_close, np64, upload

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("recompute", [True, False])
@pytest.mark.parametrize("transform", [None, {"softcap": 15.0, "temperature": 0.9}])
def test_autograd_matches_oracle(transform, recompute):
    wl = WL.custom("api", 400, 256, 2500, 128, w_std=0.05, targets="zipf", ignore_frac=0.05, seed=401)
    inp = WL.make_inputs(wl)
    inp.weights = np.random.default_rng(8).uniform(0.2, 2.0, wl.N).astype(np.float32)
    h, W, t, w = upload(inp)
    h.requires_grad_(True)
    W.requires_grad_(True)
    loss, logp, n_valid = flce.linear_cross_entropy(h, W, t, w, chunk_rows=128 if recompute else 512,
                                                    transform=transform, recompute=recompute)
    (3.0 * loss).backward()
    tf = None if transform is None else O.LogitTransform(**transform)
    ref = O.forward(inp.h, inp.W, inp.targets, inp.weights, tf=tf)
    refb = O.backward(inp.h, inp.W, inp.targets, inp.weights, g=3.0 / ref.n_valid, tf=tf)
    assert int(n_valid) == ref.n_valid
    assert float(loss.detach()) == pytest.approx(ref.loss, rel=LOSS_RTOL)
    assert_logp_close(np64(logp), ref.logp, "logp")
    assert h.grad.dtype == torch.bfloat16 and W.grad.shape == W.shape
    assert_grad_close(np64(h.grad), refb.dH, "dH")
    assert_grad_close(np64(W.grad), refb.dW, "dW")


def test_extra_memory_is_the_chunk_workspace():
    N, H, V, chunk = 4096, 512, 32768, 512
    wl = WL.custom("mem", N, H, V, chunk, seed=402)
    inp = WL.make_inputs(wl)
    h, W, t, w = upload(inp)
    ws_bytes = flce.workspace_bytes(N, H, V, chunk)
    # at most a [chunk, V] bf16 dlogits block plus dH partials and gathered
    # rows no larger than it; the forward's split partials are O(N), not O(N*V)
    assert ws_bytes <= 2 * chunk * V * 2 + N * 8 * 256 + (1 << 20)
    assert ws_bytes < N * V * 2 / 2
    torch.cuda.synchronize()
    torch.cuda.reset_peak_memory_stats()
    base = torch.cuda.memory_allocated()
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    out = flce.forward(h, W, t, None, chunk, workspace=ws)
    dH, dW = flce.backward(h, W, t, None, out["lse"], 1.0 / int(out["n_valid"]), chunk, workspace=ws)
    torch.cuda.synchronize()
    outputs = N * 4 * 2 + 16 + N * H * 2 + V * H * 4
    extra = torch.cuda.max_memory_allocated() - base
    assert extra <= ws_bytes + outputs + (4 << 20), (extra, ws_bytes, outputs)
    assert flce._lib.flce_device_status() == 0
