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
def test_grpo_loss_through_the_head_matches_oracle(transform, path, monkeypatch):
    """4 sequences x 150 tokens, 40-token prompts masked, one advantage per
    sequence; old-policy and reference log-probs near the current ones.  The
    recomputing autograd path, and the one-call path (flce_grpo_forward_backward)
    on one 640-row block (with and without the row permutation) and on the
    forward + tiled backward of a 128-row budget."""
    if path == "one_call_in_row_order":
        monkeypatch.setenv("FLCE_COMPACT", "0")
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
