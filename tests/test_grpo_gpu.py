"""GRPO per-token objective (clipped ratio, k3 KL to a reference policy) on
the GPU: the token kernel and the whole LM-head path against the fp64 oracle.

Old-policy log-probs sit a fixed set of offsets away from the current ones,
so every probability ratio is at least 0.09 away from the clip edges: the
clip decision, a comparison in floating point, is then the same in the
kernel's fp32 and the oracle's fp64."""
import numpy as np
import pytest
import torch

import chunked_lm_head_gb300 as flce
from chunked_lm_head_gb300 import workloads as WL
from oracle import flce_oracle as O

from gpu_util import LOSS_RTOL, assert_grad_close, assert_logp_close, np64, upload

pytestmark = pytest.mark.gpu

OFFSETS = [-0.5, -0.1, 0.0, 0.1, 0.5, 1.0]


def _cuda32(x):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).cuda()


@pytest.mark.parametrize("eps_low,eps_high,beta", [(0.2, 0.2, 0.0), (0.2, 0.28, 0.04), (0.1, 0.3, 0.5)])
def test_grpo_token_kernel_matches_oracle(eps_low, eps_high, beta):
    r = np.random.default_rng(21)
    N = 5000
    lp = (-r.uniform(0.05, 8.0, N)).astype(np.float32)
    old = (lp + r.choice(OFFSETS, N)).astype(np.float32)
    ref = (lp + r.uniform(-1.0, 1.0, N)).astype(np.float32)
    A = r.standard_normal(N).astype(np.float32)
    t = r.integers(0, 1000, N)
    t[r.uniform(size=N) < 0.12] = WL.IGNORE_INDEX
    out = flce.grpo_token_loss(_cuda32(lp), _cuda32(A), torch.from_numpy(t).cuda(), _cuda32(old),
                               _cuda32(ref), eps_low, eps_high, beta)
    o = O.grpo_token_loss(lp, A, t != WL.IGNORE_INDEX, old, ref, eps_low, eps_high, beta)
    assert int(out["n_valid"]) == o.n_valid
    assert np.allclose(np64(out["token_loss"]), o.token_loss, rtol=2e-6, atol=2e-6)
    assert np.allclose(np64(out["weights"]), o.weights, rtol=2e-6, atol=2e-6)
    assert float(out["loss"]) == pytest.approx(o.loss, rel=1e-5)


def test_grpo_on_policy_weights_are_the_advantages():
    r = np.random.default_rng(22)
    N = 3000
    lp = (-r.uniform(0.05, 8.0, N)).astype(np.float32)
    A = r.standard_normal(N).astype(np.float32)
    t = r.integers(0, 1000, N)
    t[:200] = WL.IGNORE_INDEX
    out = flce.grpo_token_loss(_cuda32(lp), _cuda32(A), torch.from_numpy(t).cuda())
    m = t != WL.IGNORE_INDEX
    assert np.array_equal(np64(out["weights"]), np.where(m, A, 0.0).astype(np.float32).astype(np.float64))
    assert float(out["loss"]) == pytest.approx(-float(A[m].astype(np.float64).sum()) / m.sum(), rel=1e-6)


@pytest.mark.parametrize("path", ["recompute", "one_call", "one_call_fallback", "one_call_in_row_order"])
@pytest.mark.parametrize("transform", [None, {"temperature": 0.8}])
def test_grpo_loss_through_the_head_matches_oracle(transform, path, flce_opts):
    """4 sequences x 150 tokens, 40-token prompts masked, one advantage per
    sequence; old-policy and reference log-probs near the current ones.  The
    recomputing autograd path, and the one-call path (flce_grpo_forward_backward)
    on one 640-row block (with and without the row permutation) and on the
    forward + tiled backward of a 128-row budget."""
    if path == "one_call_in_row_order":
        flce_opts.set("compact", "0")
    chunk = 1024 if path in ("one_call", "one_call_in_row_order") else 128
    wl = WL.custom("grpo_api", 600, 256, 3000, 128, w_std=0.05, targets="zipf", grpo_seqs=4,
                   prompt_len=40, seed=411)
    inp = WL.make_inputs(wl)
    tf = None if transform is None else O.LogitTransform(**transform)
    ref_fwd = O.forward(inp.h, inp.W, inp.targets, None, tf=tf)
    r = np.random.default_rng(23)
    A = np.repeat(r.standard_normal(4), 150).astype(np.float32)
    old = (ref_fwd.logp + r.choice(OFFSETS, 600)).astype(np.float32)
    refp = (ref_fwd.logp + r.uniform(-0.5, 0.5, 600)).astype(np.float32)
    h, W, t, _ = upload(inp)
    h.requires_grad_(True)
    W.requires_grad_(True)
    loss, logp = flce.grpo_loss(h, W, t, _cuda32(A), _cuda32(old), _cuda32(refp), 0.2, 0.28, 0.04,
                                chunk_rows=chunk, transform=transform, recompute=path == "recompute")
    (2.0 * loss).backward()
    m = inp.targets != WL.IGNORE_INDEX
    o = O.grpo_token_loss(ref_fwd.logp, A, m, old, refp, 0.2, 0.28, 0.04)
    refb = O.backward(inp.h, inp.W, inp.targets, o.weights, g=2.0 / o.n_valid, tf=tf)
    assert_logp_close(np64(logp), ref_fwd.logp, "logp")
    assert float(loss.detach()) == pytest.approx(o.loss, rel=LOSS_RTOL, abs=1e-6)
    assert_grad_close(np64(h.grad), refb.dH, "dH")
    assert_grad_close(np64(W.grad), refb.dW, "dW")


def test_grpo_one_call_on_policy_gradients_equal_the_weighted_cross_entropy():
    """With no old-policy log-probs (ratio 1) and beta 0, the GRPO weights
    are the advantages: flce_grpo_forward_backward gives bit for bit the
    gradients of flce_forward_backward with weights = advantages.  With every
    row ignored, loss and gradients are zero."""
    from chunked_lm_head_gb300 import _lib
    wl = WL.custom("grpo_pol", 2400, 256, 3000, 2048, w_std=0.05, targets="zipf", grpo_seqs=4,
                   prompt_len=100, seed=412)
    inp = WL.make_inputs(wl)
    h, W, t, A = upload(inp)
    N, H, V = wl.N, wl.H, wl.V

    def bufs():
        return (torch.empty(N, device="cuda"), torch.empty(1, device="cuda"),
                torch.empty(1, dtype=torch.int64, device="cuda"), torch.empty_like(h),
                torch.empty((V, H), device="cuda"))

    lp1, loss1, nv1, dH1, dW1 = bufs()
    assert _lib.flce_grpo_forward_backward(h, W, t, A, None, None, 0.2, 0.2, 0.0, N, H, V, 2048, -100, None, 1.0,
                                           lp1, None, loss1, nv1, dH1, dW1) == 0
    lp2, loss2, nv2, dH2, dW2 = bufs()
    assert _lib.flce_forward_backward(h, W, t, A, N, H, V, 2048, -100, None, 1.0, lp2, None, loss2, nv2,
                                      dH2, dW2) == 0
    assert _lib.flce_device_status() == 0
    m = inp.targets != WL.IGNORE_INDEX
    assert int(nv1.item()) == int(nv2.item()) == int(m.sum())
    assert torch.equal(lp1, lp2) and torch.equal(dH1, dH2) and torch.equal(dW1, dW2)
    # the GRPO loss is sum(-A) / n here (its value, unlike its gradient, has no logp)
    assert float(loss1.item()) == pytest.approx(-float(inp.weights[m].astype(np.float64).sum()) / m.sum(),
                                                rel=1e-5)
    t.fill_(-100)
    assert _lib.flce_grpo_forward_backward(h, W, t, A, None, None, 0.2, 0.2, 0.0, N, H, V, 2048, -100, None, 1.0,
                                           lp1, None, loss1, nv1, dH1, dW1) == 0
    assert int(nv1.item()) == 0 and float(loss1.item()) == 0.0
    assert float(dH1.float().abs().max()) == 0.0 and float(dW1.abs().max()) == 0.0
