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


def test_autograd_backwards_do_not_synchronise_the_host():
    """The incoming gradient of the loss and the token count reach the
    kernels as device pointers: no backward of the autograd wrappers reads a
    value back to the host (torch's sync debug mode raises if one does)."""
    from gpu_util import to_dev_bf16
    wl = WL.custom("nosync", 600, 256, 3000, 128, w_std=0.05, targets="zipf", grpo_seqs=2,
                   prompt_len=60, seed=451)
    inp = WL.make_inputs(wl)
    h, W, t, _ = upload(inp)
    adv = torch.from_numpy(np.random.default_rng(2).standard_normal(wl.N).astype(np.float32)).cuda()
    ti = WL.make_inputs(WL.custom("nosync_t", 600, 128, 3000, 128, w_std=0.06, seed=452))
    ht, Wt = to_dev_bf16(ti.h), to_dev_bf16(ti.W)
    cases = [
        lambda a, b: flce.linear_cross_entropy(a, b, t, None, 128)[0],
        lambda a, b: flce.linear_cross_entropy(a, b, t, None, 2048, recompute=False)[0],
        lambda a, b: flce.grpo_loss(a, b, t, adv, chunk_rows=128)[0],
        lambda a, b: flce.grpo_loss(a, b, t, adv, chunk_rows=2048, recompute=False)[0],
        lambda a, b: flce.distill_loss(a, b, ht, Wt, t, None, beta=None, chunk_rows=128),
        lambda a, b: flce.distill_loss(a, b, ht, Wt, t, None, beta=0.5, chunk_rows=128),
    ]
    for k, f in enumerate(cases):
        a, b = h.clone().requires_grad_(True), W.clone().requires_grad_(True)
        loss = f(a, b)
        torch.cuda.synchronize()
        torch.cuda.set_sync_debug_mode("error")
        try:
            (0.5 * loss).backward()
        finally:
            torch.cuda.set_sync_debug_mode("default")
        torch.cuda.synchronize()
        assert a.grad is not None and b.grad is not None, k
        assert torch.isfinite(a.grad.float()).all() and torch.isfinite(b.grad).all(), k
        assert flce._lib.flce_device_status() == 0


def test_device_side_scale_equals_the_host_scale():
    """flce_backward_ex2 with grad_scale * scale / max(count, 1) read on the
    device against flce_backward_ex with the same factor from the host; and
    flce_scale_grads (a scale of 1 moves nothing, 0.25 scales exactly)."""
    from chunked_lm_head_gb300 import _lib
    wl = WL.custom("dscale", 500, 192, 2600, 128, w_std=0.05, targets="zipf", ignore_frac=0.1, seed=453)
    inp = WL.make_inputs(wl)
    h, W, t, _ = upload(inp)
    out = flce.forward(h, W, t, None, 128)
    nv = out["n_valid"]
    s = torch.tensor([0.75], device="cuda")
    dH1, dW1 = flce.backward(h, W, t, None, out["lse"], 2.0, 128, scale=s, count=nv)
    dH0, dW0 = flce.backward(h, W, t, None, out["lse"], 2.0 * 0.75 / int(nv), 128)
    assert rel_fro_t(dH1, dH0) <= 1e-6 and rel_fro_t(dW1, dW0) <= 1e-6
    ref = O.backward(inp.h, inp.W, inp.targets, None, g=1.5 / int(nv))
    assert_grad_close(np64(dH1), ref.dH, "dH")
    assert_grad_close(np64(dW1), ref.dW, "dW")
    # a zero count divides by 1
    zero = torch.zeros(1, dtype=torch.int64, device="cuda")
    _, dWz = flce.backward(h, W, t, None, out["lse"], 2.0, 128, need_dH=False, scale=s, count=zero)
    _, dWh = flce.backward(h, W, t, None, out["lse"], 1.5, 128, need_dH=False)
    assert rel_fro_t(dWz, dWh) <= 1e-6
    # in-place scaling by a device scalar
    a, b = dH1.clone(), dW1.clone()
    flce.scale_grads(a, b, torch.ones(1, device="cuda"))
    assert torch.equal(a, dH1) and torch.equal(b, dW1)
    flce.scale_grads(a, b, torch.full((1,), 0.25, device="cuda"))
    assert torch.equal(a, (dH1.float() * 0.25).to(torch.bfloat16)) and torch.equal(b, dW1 * 0.25)
    odd = torch.randn(1001, device="cuda")  # a scalar tail past the 16-byte vectors
    o2 = odd.clone()
    flce.scale_grads(None, o2, torch.full((1,), -3.0, device="cuda"))
    assert torch.equal(o2, odd * -3.0)
    assert _lib.flce_device_status() == 0


def rel_fro_t(a, b):
    a, b = a.double(), b.double()
    return float((a - b).norm() / b.norm().clamp_min(1e-300))


def test_data_parallel_step_on_one_rank_matches_oracle():
    """The data-parallel step with libflce as the per-rank compute and no
    process group (one rank): the count reaches the backward as a device
    scalar; loss, dH and dW against the oracle."""
    from chunked_lm_head_gb300 import dp
    wl = WL.custom("dp1", 700, 256, 5003, 256, w_std=0.05, targets="zipf", ignore_frac=0.1, seed=171)
    inp = WL.make_inputs(wl)
    inp.weights = np.random.default_rng(17).uniform(0.3, 1.7, wl.N).astype(np.float32)
    h, W, t, w = upload(inp)
    out = dp.data_parallel_step(h, W, t, w, grad=0.5, local=dp.LibflceStep(chunk_rows=256))
    ref = O.forward(inp.h, inp.W, inp.targets, inp.weights)
    refb = O.backward(inp.h, inp.W, inp.targets, inp.weights, g=0.5 / ref.n_valid)
    assert int(out["n_valid"]) == ref.n_valid
    assert float(out["loss"]) == pytest.approx(ref.loss, rel=LOSS_RTOL)
    assert_logp_close(np64(out["logp"]), ref.logp, "logp")
    assert_grad_close(np64(out["dH"]), refb.dH, "dH")
    assert_grad_close(np64(out["dW"]), refb.dW, "dW")
