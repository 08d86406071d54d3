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


@pytest.mark.parametrize("beta", [None, 0.3])
def test_distill_loss_autograd_matches_oracle(beta):
    """distill_loss (KL, or Jensen-Shannon at beta 0.3) through autograd:
    loss and the student's gradients against the oracle, with a mask, weights,
    a temperature and an upstream gradient of 2."""
    from gpu_util import to_dev_bf16
    si = WL.make_inputs(WL.custom("dl_s", 300, 192, 2100, 128, w_std=0.05, seed=421))
    ti = WL.make_inputs(WL.custom("dl_t", 300, 256, 2100, 128, w_std=0.065, seed=422))
    targets = np.random.default_rng(3).integers(0, 2100, 300).astype(np.int64)
    targets[np.random.default_rng(4).permutation(300)[:30]] = WL.IGNORE_INDEX
    weights = np.random.default_rng(5).uniform(0.3, 1.7, 300).astype(np.float32)
    tfd = {"temperature": 2.0}
    tf = O.LogitTransform(**tfd)
    hs, Ws, ht, Wt = (to_dev_bf16(x) for x in (si.h, si.W, ti.h, ti.W))
    hs.requires_grad_(True)
    Ws.requires_grad_(True)
    tg = torch.from_numpy(targets).cuda()
    w = torch.from_numpy(weights).cuda()
    loss = flce.distill_loss(hs, Ws, ht, Wt, tg, w, beta=beta, chunk_rows=128, transform=tfd)
    (2.0 * loss).backward()
    if beta is None:
        ref = O.kd_forward(si.h, si.W, ti.h, ti.W, targets, weights, tf=tf)
        refb = O.kd_backward(si.h, si.W, ti.h, ti.W, targets, weights, g=2.0 / ref.n_valid, tf=tf)
    else:
        ref = O.jsd_forward(si.h, si.W, ti.h, ti.W, beta, targets, weights, tf=tf)
        refb = O.jsd_backward(si.h, si.W, ti.h, ti.W, beta, targets, weights, g=2.0 / ref.n_valid, tf=tf)
    assert float(loss.detach()) == pytest.approx(ref.loss, rel=LOSS_RTOL, abs=1e-6)
    assert_grad_close(np64(hs.grad), refb.dH, "dH_s")
    assert_grad_close(np64(Ws.grad), refb.dW, "dW_s")
    assert ht.grad is None and Wt.grad is None


@pytest.mark.parametrize("transform", [None, {"softcap": 10.0, "temperature": 0.7}])
def test_selective_log_softmax_autograd_matches_oracle(transform):
    """logp through autograd with an arbitrary upstream gradient u:
    d(sum u logp) / d(h, W) is the oracle's weighted backward with w = -u, g = 1."""
    wl = WL.custom("sls", 700, 256, 3000, 128, w_std=0.05, targets="zipf", ignore_frac=0.1, seed=431)
    inp = WL.make_inputs(wl)
    h, W, t, _ = upload(inp)
    h.requires_grad_(True)
    W.requires_grad_(True)
    logp = flce.selective_log_softmax(h, W, t, chunk_rows=128, transform=transform)
    u = np.random.default_rng(9).normal(size=wl.N).astype(np.float32)
    (logp * torch.from_numpy(u).cuda()).sum().backward()
    tf = None if transform is None else O.LogitTransform(**transform)
    ref = O.forward(inp.h, inp.W, inp.targets, None, tf=tf)
    refb = O.backward(inp.h, inp.W, inp.targets, -u, g=1.0, tf=tf)
    assert_logp_close(np64(logp), ref.logp, "logp")
    assert_grad_close(np64(h.grad), refb.dH, "dH")
    assert_grad_close(np64(W.grad), refb.dW, "dW")
    if transform is not None:  # the same transform through the page's keyword names
        logp2 = flce.selective_log_softmax(h.detach(), W.detach(), t, chunk_rows=128,
                                           logit_softcapping=transform["softcap"],
                                           temperature=transform["temperature"])
        assert torch.equal(logp2, logp.detach())


def test_loss_module_matches_the_function():
    wl = WL.custom("mod", 500, 256, 2500, 128, w_std=0.05, targets="zipf", ignore_frac=0.05, seed=441)
    inp = WL.make_inputs(wl)
    h, W, t, _ = upload(inp)
    grads = []
    for use_module in (True, False):
        hh, WW = h.clone().requires_grad_(True), W.clone().requires_grad_(True)
        if use_module:
            loss = flce.LinearCrossEntropyLoss(chunk_rows=128)(hh, WW, t)
        else:
            loss = flce.linear_cross_entropy(hh, WW, t, None, 128)[0]
        loss.backward()
        grads.append((float(loss.detach()), hh.grad, WW.grad))
    assert grads[0][0] == grads[1][0]
    assert torch.equal(grads[0][1], grads[1][1]) and torch.equal(grads[0][2], grads[1][2])
