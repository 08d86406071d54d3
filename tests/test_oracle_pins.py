"""Pins of the fp64 oracle against closed forms, invariants, finite differences,
a library routine (torch cross_entropy + autograd in fp64) and the numbers the
pages print.  CPU only."""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import flce_oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _rand(N, H, V, seed=0, ignore=(), scale_w=0.3, weights=False):
    r = np.random.default_rng(seed)
    h = r.standard_normal((N, H))
    W = r.standard_normal((V, H)) * scale_w
    t = r.integers(0, V, N)
    for i in ignore:
        t[i] = O.IGNORE_INDEX
    w = r.standard_normal(N) if weights else None
    return h, W, t, w


# ---------------------------------------------------------------- closed forms

def test_zero_weight_matrix_closed_form():
    N, H, V = 9, 6, 11
    h, _, t, w = _rand(N, H, V, seed=1, ignore=(2, 5), weights=True)
    W = np.zeros((V, H))
    g = 0.37
    f = O.forward(h, W, t, w)
    m = t != O.IGNORE_INDEX
    assert np.allclose(f.lse, math.log(V), atol=1e-14)
    assert np.allclose(f.logp[m], -math.log(V), atol=1e-14)
    assert np.all(f.logp[~m] == 0)
    assert f.n_valid == 7
    assert f.loss == pytest.approx(-np.sum(w[m]) * (-math.log(V)) / 7, rel=1e-13)
    b = O.backward(h, W, t, w, g=g)
    assert np.all(b.dH == 0)
    # dW[v,:] = sum_i (1/V - [v == t_i]) m_i w_i g h_i, by explicit loops
    ref = np.zeros((V, H))
    for i in range(N):
        if not m[i]:
            continue
        for v in range(V):
            ref[v] += (1.0 / V - (1.0 if v == t[i] else 0.0)) * w[i] * g * h[i]
    assert np.allclose(b.dW, ref, atol=1e-13)


def test_single_word_vocab():
    h, W, t, _ = _rand(5, 4, 1, seed=2)
    f = O.forward(h, W, t)
    assert np.allclose(f.logp, 0, atol=1e-14)
    assert np.allclose(f.lse, (h @ W.T)[:, 0], atol=1e-13)
    b = O.backward(h, W, t, g=1.0)
    assert np.allclose(b.dH, 0, atol=1e-14) and np.allclose(b.dW, 0, atol=1e-14)


def test_two_word_vocab_is_softplus():
    h, W, t, _ = _rand(40, 7, 2, seed=3, scale_w=2.0)
    f = O.forward(h, W, t)
    z = h @ W.T
    rows = np.arange(40)
    other = z[rows, 1 - t] - z[rows, t]
    assert np.allclose(f.logp, -np.logaddexp(0.0, other), atol=1e-13)


def test_row_constant_shift_leaves_logp():
    h, W, t, _ = _rand(12, 5, 17, seed=4)
    f = O.forward(h, W, t)
    for c in (3.0, 1000.0):  # 1000 also checks the max shift (exp(1000) overflows)
        h2 = np.concatenate([h, np.ones((12, 1))], axis=1)
        W2 = np.concatenate([W, np.full((17, 1), c)], axis=1)
        f2 = O.forward(h2, W2, t)
        assert np.all(np.isfinite(f2.lse))
        assert np.allclose(f2.logp, f.logp, atol=1e-10)
        assert np.allclose(f2.lse, f.lse + c, atol=1e-10)


# ------------------------------------------------------------------ invariants

def test_softmax_rows_sum_to_one_and_dlogits_rows_to_zero():
    h, W, t, w = _rand(20, 8, 31, seed=5, ignore=(3,), weights=True)
    z = O.logits(h, W)
    lse = O.logsumexp_rows(z)
    assert np.allclose(O.probs(z, lse).sum(axis=1), 1.0, atol=1e-12)
    D = O.dlogits(z, lse, np.where(t == O.IGNORE_INDEX, 0, t), t != O.IGNORE_INDEX, w, 0.5)
    assert np.allclose(D.sum(axis=1), 0.0, atol=1e-12)
    assert np.all(D[3] == 0)


def test_ignored_rows_have_no_influence():
    ign = (0, 4, 9)
    h, W, t, w = _rand(12, 6, 13, seed=6, ignore=ign, weights=True)
    f = O.forward(h, W, t, w)
    b = O.backward(h, W, t, w, g=0.25)
    h2 = h.copy()
    h2[list(ign)] += np.random.default_rng(7).standard_normal((3, 6)) * 5
    f2 = O.forward(h2, W, t, w)
    b2 = O.backward(h2, W, t, w, g=0.25)
    keep = np.setdiff1d(np.arange(12), ign)
    assert np.allclose(f2.lse[keep], f.lse[keep], atol=1e-13)
    assert not np.allclose(f2.lse[list(ign)], f.lse[list(ign)])
    assert np.all(f2.logp[list(ign)] == 0)
    assert f2.loss == pytest.approx(f.loss, rel=1e-13)
    assert np.allclose(b2.dH, b.dH, atol=1e-13) and np.all(b2.dH[list(ign)] == 0)
    assert np.allclose(b2.dW, b.dW, atol=1e-13)


@pytest.mark.parametrize("chunk", [1, 16, 64, None])
def test_chunk_size_independence(chunk):
    h, W, t, w = _rand(64, 16, 50, seed=8, ignore=(1, 30, 63), weights=True)
    f0 = O.forward(h, W, t, w)
    b0 = O.backward(h, W, t, w, g=1 / f0.n_valid)
    f = O.forward(h, W, t, w, chunk_rows=chunk)
    b = O.backward(h, W, t, w, g=1 / f0.n_valid, chunk_rows=chunk)
    assert np.allclose(f.lse, f0.lse, atol=1e-12) and np.allclose(f.logp, f0.logp, atol=1e-12)
    assert f.loss == pytest.approx(f0.loss, rel=1e-12, abs=1e-15)
    assert np.allclose(b.dH, b0.dH, atol=1e-12) and np.allclose(b.dW, b0.dW, atol=1e-12)


def test_row_and_vocab_permutation_equivariance():
    h, W, t, w = _rand(15, 6, 19, seed=9, ignore=(2,), weights=True)
    f = O.forward(h, W, t, w)
    b = O.backward(h, W, t, w, g=0.3)
    r = np.random.default_rng(10)
    pr = r.permutation(15)
    fr = O.forward(h[pr], W, t[pr], w[pr])
    br = O.backward(h[pr], W, t[pr], w[pr], g=0.3)
    assert np.allclose(fr.logp, f.logp[pr], atol=1e-13) and np.allclose(br.dH, b.dH[pr], atol=1e-13)
    assert np.allclose(br.dW, b.dW, atol=1e-12)
    pv = r.permutation(19)  # new vocab index j holds old word pv[j]
    inv = np.argsort(pv)
    t2 = np.where(t == O.IGNORE_INDEX, t, inv[np.where(t == O.IGNORE_INDEX, 0, t)])
    fv = O.forward(h, W[pv], t2, w)
    bv = O.backward(h, W[pv], t2, w, g=0.3)
    assert np.allclose(fv.logp, f.logp, atol=1e-13) and np.allclose(fv.lse, f.lse, atol=1e-13)
    assert np.allclose(bv.dW, b.dW[pv], atol=1e-13) and np.allclose(bv.dH, b.dH, atol=1e-13)


def test_gradients_linear_in_grad_scale():
    h, W, t, w = _rand(10, 5, 9, seed=11, weights=True)
    b1 = O.backward(h, W, t, w, g=1.0)
    b3 = O.backward(h, W, t, w, g=-2.5)
    assert np.allclose(b3.dH, -2.5 * b1.dH, atol=1e-13) and np.allclose(b3.dW, -2.5 * b1.dW, atol=1e-13)


def test_n_valid_exact_and_empty_batch():
    h, W, t, _ = _rand(33, 4, 8, seed=12, ignore=range(0, 33, 4))
    assert O.forward(h, W, t).n_valid == 33 - 9
    t_all = np.full(33, O.IGNORE_INDEX)
    f = O.forward(h, W, t_all)
    assert f.n_valid == 0 and f.loss == 0.0 and np.all(f.logp == 0)
    b = O.backward(h, W, t_all, g=1.0)
    assert np.all(b.dH == 0) and np.all(b.dW == 0)


def test_bad_target_is_an_error():
    h, W, t, _ = _rand(4, 3, 5, seed=13)
    t[1] = 5
    with pytest.raises(ValueError):
        O.forward(h, W, t)


# ---------------------------------------------------------- finite differences

def test_central_finite_differences():
    N, H, V = 3, 5, 7
    h, W, t, w = _rand(N, H, V, seed=14, weights=True)
    f = O.forward(h, W, t, w)
    b = O.backward(h, W, t, w, g=1.0 / f.n_valid)
    eps = 1e-6

    def loss(hh, WW):
        return O.forward(hh, WW, t, w).loss

    num_dH = np.zeros_like(h)
    for i in range(N):
        for k in range(H):
            e = np.zeros_like(h)
            e[i, k] = eps
            num_dH[i, k] = (loss(h + e, W) - loss(h - e, W)) / (2 * eps)
    num_dW = np.zeros_like(W)
    for v in range(V):
        for k in range(H):
            e = np.zeros_like(W)
            e[v, k] = eps
            num_dW[v, k] = (loss(h, W + e) - loss(h, W - e)) / (2 * eps)
    assert np.linalg.norm(num_dH - b.dH) <= 1e-7 * np.linalg.norm(b.dH)
    assert np.linalg.norm(num_dW - b.dW) <= 1e-7 * np.linalg.norm(b.dW)


# ------------------------------------------------------------- library routine

def _torch_ref(h, W, t, w, ignore_index=O.IGNORE_INDEX):
    """torch fp64 cross_entropy (per token) and autograd for the weighted loss."""
    ht = torch.tensor(O.widen(h), requires_grad=True)
    Wt = torch.tensor(O.widen(W), requires_grad=True)
    tt = torch.tensor(np.asarray(t, dtype=np.int64))
    ce = torch.nn.functional.cross_entropy(ht @ Wt.T, tt, ignore_index=ignore_index, reduction="none")
    n_valid = int((tt != ignore_index).sum())
    wt = torch.ones_like(ce) if w is None else torch.tensor(np.asarray(w, dtype=np.float64))
    loss = (wt * ce).sum() / max(n_valid, 1)
    loss.backward()
    return -ce.detach().numpy(), float(loss.detach()), ht.grad.numpy(), Wt.grad.numpy(), n_valid


def test_matches_torch_cross_entropy_on_tiny_workload():
    from chunked_lm_head_gb300 import workloads as WL
    inp = WL.make_inputs("tiny")
    logp_t, loss_t, dH_t, dW_t, nv = _torch_ref(inp.h, inp.W, inp.targets, None)
    f = O.forward(inp.h, inp.W, inp.targets, chunk_rows=16)
    b = O.backward(inp.h, inp.W, inp.targets, g=1.0 / f.n_valid, chunk_rows=16)
    assert f.n_valid == nv == 61
    assert np.allclose(f.logp, logp_t, atol=1e-12)
    assert f.loss == pytest.approx(loss_t, rel=1e-12)
    # mean reduction of the library equals the oracle's loss with w = 1
    ce_mean = torch.nn.functional.cross_entropy(
        torch.tensor(O.logits(inp.h, inp.W)), torch.tensor(inp.targets), ignore_index=-100)
    assert f.loss == pytest.approx(float(ce_mean), rel=1e-12)
    assert np.allclose(b.dH, dH_t, atol=1e-12) and np.allclose(b.dW, dW_t, atol=1e-12)


def test_matches_torch_on_weighted_grpo_shape():
    from chunked_lm_head_gb300 import workloads as WL
    wl = WL.custom("grpo_small", 4 * 96, 128, 3000, 64, w_std=0.02, targets="zipf",
                   grpo_seqs=4, prompt_len=16, seed=77)
    inp = WL.make_inputs(wl)
    assert inp.weights is not None and inp.n_ignored == 64
    logp_t, loss_t, dH_t, dW_t, nv = _torch_ref(inp.h, inp.W, inp.targets, inp.weights)
    f = O.forward(inp.h, inp.W, inp.targets, inp.weights, chunk_rows=64)
    b = O.backward(inp.h, inp.W, inp.targets, inp.weights, g=1.0 / f.n_valid, chunk_rows=64)
    assert f.n_valid == nv
    assert np.allclose(f.logp, logp_t, atol=1e-12)
    assert f.loss == pytest.approx(loss_t, rel=1e-11)
    # per-sequence form: sum_s a_s * (summed CE over the sequence) / n_valid
    z = torch.tensor(O.logits(inp.h, inp.W))
    tt = torch.tensor(inp.targets)
    seg = 0.0
    L = wl.N // 4
    for s in range(4):
        ce_s = torch.nn.functional.cross_entropy(z[s * L:(s + 1) * L], tt[s * L:(s + 1) * L],
                                                 ignore_index=-100, reduction="sum")
        seg += float(inp.weights[s * L]) * float(ce_s)
    assert f.loss == pytest.approx(seg / f.n_valid, rel=1e-11)
    assert np.allclose(b.dH, dH_t, atol=1e-12) and np.allclose(b.dW, dW_t, atol=1e-12)


def test_sampled_row_functions_match_full():
    h, W, t, w = _rand(40, 9, 23, seed=15, ignore=(5, 6), weights=True)
    f = O.forward(h, W, t, w)
    b = O.backward(h, W, t, w, g=0.1)
    rows = np.array([0, 5, 17, 39])
    lse, logp = O.rows_forward(h, W, t, rows)
    assert np.allclose(lse, f.lse[rows], atol=1e-13) and np.allclose(logp, f.logp[rows], atol=1e-13)
    dH, dWp = O.rows_backward(h, W, t, np.arange(40), w, g=0.1, vocab_rows=[1, 22])
    assert np.allclose(dH, b.dH, atol=1e-13) and np.allclose(dWp, b.dW[[1, 22]], atol=1e-13)
    lse2, logp2, dH2, dWp2 = O.rows_all(h, W, t, rows, w, g=0.1, vocab_rows=[1, 22])
    assert np.allclose(lse2, f.lse[rows], atol=1e-13) and np.allclose(logp2, f.logp[rows], atol=1e-13)
    assert np.allclose(dH2, b.dH[rows], atol=1e-13)
    w_rows = np.zeros(40)
    w_rows[rows] = w[rows]
    assert np.allclose(dWp2, O.backward(h, W, t, w_rows, g=0.1).dW[[1, 22]], atol=1e-13)
    # dW columns from every row's lse
    vr = [0, 7, 22]
    assert np.allclose(O.vocab_rows_dW(h, W, t, f.lse, vr, w, g=0.1, block_rows=16), b.dW[vr], atol=1e-13)
    # linearity in the per-row weights: weights zero outside a row subset keep
    # only those rows' dW contribution
    w0 = np.zeros(40)
    w0[rows] = w[rows]
    b0 = O.backward(h, W, t, w0, g=0.1)
    _, part = O.rows_backward(h, W, t, rows, w, g=0.1)
    assert np.allclose(b0.dW, part, atol=1e-13)


# --------------------------------------------------------- the pages' numbers

def test_logit_memory_equations():
    g = json.load(open(os.path.join(GOLD, "logit_memory.json")))
    ex = g["example"]
    B, L, V = ex["batch_size"], ex["context_length"], ex["vocab_dim"]
    eq1 = O.logit_memory_gb(L, V, batch_size=B)
    eq2 = O.logit_memory_gb(L, V)
    mult = O.default_chunk_multiplier(L)
    assert mult == ex["multiplier"] == 4
    eq3 = O.logit_memory_gb(L, V, multiplier=mult)
    assert eq1 == pytest.approx(3.906, abs=1e-3)
    assert eq2 == pytest.approx(0.977, abs=1e-3)
    assert eq3 == pytest.approx(0.244, abs=1e-3)
    p = g["printed_gb"]
    # the printed values keep the formula's x4 steps ...
    assert eq1 / eq2 == pytest.approx(4.0) and eq2 / eq3 == pytest.approx(4.0)
    assert p["eq1_whole_batch"] / p["eq2_one_sample"] == pytest.approx(4.0, rel=0.01)
    assert p["eq2_one_sample"] / p["eq3_sequence_chunked"] == pytest.approx(4.0, rel=0.01)
    # ... but not its values: 3.3 / 0.83 / 0.207 sit ~15% under the formula
    assert p["eq1_whole_batch"] / eq1 == pytest.approx(0.845, abs=0.01)
    hs = g["hidden_states_example"]
    hs_all = O.logit_memory_gb(hs["context_length"], hs["hidden_states_dim"], batch_size=hs["batch_size"])
    hs_one = O.logit_memory_gb(hs["context_length"], hs["hidden_states_dim"])
    assert hs_all == pytest.approx(g["hidden_states_printed_gb"]["whole_batch"], rel=0.03)
    assert hs_one == pytest.approx(g["hidden_states_printed_gb"]["per_sample"], abs=5e-4)
    # long-context workload: full bf16 logits would be ~40 GB (never allocated)
    assert 131072 * 151936 * 2 / 1e9 == pytest.approx(39.83, abs=0.01)


def test_fp32_weight_copy_bytes():
    g = json.load(open(os.path.join(GOLD, "trl_fp32_copy.json")))
    assert g["vocab"] * g["hidden"] * g["bytes_per_element"] / 1e9 == pytest.approx(g["printed_gb"], abs=0.005)


# ------------------------------------------------------------ logit transforms

def test_identity_transform_is_no_transform():
    h, W, t, w = _rand(20, 6, 15, seed=30, ignore=(3,), weights=True)
    tf = O.LogitTransform()
    f0, f1 = O.forward(h, W, t, w), O.forward(h, W, t, w, tf=tf)
    b0, b1 = O.backward(h, W, t, w, g=0.2), O.backward(h, W, t, w, g=0.2, tf=tf)
    assert np.array_equal(f0.logp, f1.logp) and np.array_equal(b0.dH, b1.dH) and np.array_equal(b0.dW, b1.dW)


def test_linear_transforms_equal_a_scaled_head():
    # multiply / divide / temperature are one scale a on the logits: the same
    # as using the weight matrix a*W (forward), with dH picking up a and dW
    # (w.r.t. the original W) picking up a as well
    h, W, t, w = _rand(25, 7, 19, seed=31, ignore=(0,), weights=True)
    tf = O.LogitTransform(scale_multiply=3.0, scale_divide=2.0, temperature=0.5)
    a = 3.0 / 2.0 / 0.5
    f = O.forward(h, W, t, w, tf=tf)
    fa = O.forward(h, a * W, t, w)
    assert np.allclose(f.logp, fa.logp, atol=1e-12) and np.allclose(f.lse, fa.lse, atol=1e-12)
    b = O.backward(h, W, t, w, g=0.3, tf=tf)
    ba = O.backward(h, a * W, t, w, g=0.3)
    assert np.allclose(b.dH, ba.dH, atol=1e-12) and np.allclose(b.dW, a * ba.dW, atol=1e-12)


def test_softcap_bounds_logits_and_vanishes_for_large_cap():
    h, W, t, _ = _rand(10, 6, 13, seed=32, scale_w=3.0)
    z = O.logits(h, W)
    y = O.LogitTransform(softcap=5.0).apply(z)
    assert np.all(np.abs(y) < 5.0) and np.max(np.abs(z)) > 5.0
    big = O.LogitTransform(softcap=1e7)
    assert np.allclose(O.forward(h, W, t, tf=big).logp, O.forward(h, W, t).logp, atol=1e-9)


def test_transform_gradients_by_finite_differences():
    N, H, V = 3, 5, 7
    h, W, t, w = _rand(N, H, V, seed=33, weights=True, scale_w=2.0)
    tf = O.LogitTransform(scale_multiply=1.7, scale_divide=1.3, softcap=2.5, temperature=0.8)
    f = O.forward(h, W, t, w, tf=tf)
    b = O.backward(h, W, t, w, g=1.0 / f.n_valid, tf=tf)
    eps = 1e-6

    def loss(hh, WW):
        return O.forward(hh, WW, t, w, tf=tf).loss

    num_dH = np.zeros_like(h)
    for i in range(N):
        for k in range(H):
            e = np.zeros_like(h)
            e[i, k] = eps
            num_dH[i, k] = (loss(h + e, W) - loss(h - e, W)) / (2 * eps)
    num_dW = np.zeros_like(W)
    for v in range(V):
        for k in range(H):
            e = np.zeros_like(W)
            e[v, k] = eps
            num_dW[v, k] = (loss(h, W + e) - loss(h, W - e)) / (2 * eps)
    assert np.linalg.norm(num_dH - b.dH) <= 1e-7 * np.linalg.norm(b.dH)
    assert np.linalg.norm(num_dW - b.dW) <= 1e-7 * np.linalg.norm(b.dW)


def test_transform_matches_torch_autograd():
    h, W, t, w = _rand(30, 8, 40, seed=34, ignore=(2, 9), weights=True, scale_w=1.5)
    tf = O.LogitTransform(scale_multiply=0.9, softcap=4.0, temperature=1.3)
    ht = torch.tensor(h, requires_grad=True)
    Wt = torch.tensor(W, requires_grad=True)
    z = ht @ Wt.T * 0.9
    z = 4.0 * torch.tanh(z / 4.0) / 1.3
    ce = torch.nn.functional.cross_entropy(z, torch.tensor(t), ignore_index=-100, reduction="none")
    nv = int((t != -100).sum())
    loss = (torch.tensor(w) * ce).sum() / nv
    loss.backward()
    f = O.forward(h, W, t, w, tf=tf)
    b = O.backward(h, W, t, w, g=1.0 / nv, tf=tf)
    assert f.loss == pytest.approx(float(loss.detach()), rel=1e-12)
    assert np.allclose(f.logp, -ce.detach().numpy(), atol=1e-12)
    assert np.allclose(b.dH, ht.grad.numpy(), atol=1e-12) and np.allclose(b.dW, Wt.grad.numpy(), atol=1e-12)
    lse, logp = O.rows_forward(h, W, t, [1, 5], tf=tf)
    assert np.allclose(logp, f.logp[[1, 5]], atol=1e-13)
    _, lp2, dH2, _ = O.rows_all(h, W, t, [1, 5], w, g=1.0 / nv, tf=tf)
    assert np.allclose(dH2, b.dH[[1, 5]], atol=1e-13)


# ------------------------------------------------------------------ distillation

def _kd_rand(N, Hs, Ht, V, seed):
    r = np.random.default_rng(seed)
    return (r.standard_normal((N, Hs)), r.standard_normal((V, Hs)) * 0.4,
            r.standard_normal((N, Ht)), r.standard_normal((V, Ht)) * 0.4)


def test_kd_is_zero_for_identical_heads_and_nonnegative():
    hs, Ws, _, _ = _kd_rand(12, 6, 6, 17, 40)
    f = O.kd_forward(hs, Ws, hs, Ws)
    assert np.allclose(f.kl, 0.0, atol=1e-13) and f.loss == pytest.approx(0.0, abs=1e-13)
    b = O.kd_backward(hs, Ws, hs, Ws, g=1.0)
    assert np.allclose(b.dH, 0, atol=1e-13) and np.allclose(b.dW, 0, atol=1e-13)
    hs, Ws, ht, Wt = _kd_rand(20, 6, 9, 17, 41)
    f = O.kd_forward(hs, Ws, ht, Wt)
    assert np.all(f.kl > 0)


def test_kd_matches_torch_kl_div_and_autograd():
    hs, Ws, ht, Wt = _kd_rand(25, 7, 5, 31, 42)
    t = np.random.default_rng(1).integers(0, 31, 25)
    t[[3, 8]] = O.IGNORE_INDEX
    w = np.random.default_rng(2).uniform(0.5, 2, 25)
    tf = O.LogitTransform(temperature=2.0)
    hst = torch.tensor(hs, requires_grad=True)
    Wst = torch.tensor(Ws, requires_grad=True)
    zs = (hst @ Wst.T) / 2.0
    zt = torch.tensor(ht @ Wt.T) / 2.0
    kl = torch.nn.functional.kl_div(torch.log_softmax(zs, -1), torch.log_softmax(zt, -1),
                                    log_target=True, reduction="none").sum(-1)
    m = torch.tensor(t != O.IGNORE_INDEX, dtype=torch.float64)
    loss = (m * torch.tensor(w) * kl).sum() / m.sum()
    loss.backward()
    f = O.kd_forward(hs, Ws, ht, Wt, t, w, tf=tf)
    b = O.kd_backward(hs, Ws, ht, Wt, t, w, g=1.0 / f.n_valid, tf=tf)
    assert f.n_valid == 23
    assert np.allclose(f.kl, (m * kl).detach().numpy(), atol=1e-12)
    assert f.loss == pytest.approx(float(loss.detach()), rel=1e-12)
    assert np.allclose(b.dH, hst.grad.numpy(), atol=1e-12) and np.allclose(b.dW, Wst.grad.numpy(), atol=1e-12)
    # chunking does not change anything
    fc = O.kd_forward(hs, Ws, ht, Wt, t, w, tf=tf, chunk_rows=4)
    bc = O.kd_backward(hs, Ws, ht, Wt, t, w, g=1.0 / f.n_valid, tf=tf, chunk_rows=4)
    assert np.allclose(fc.kl, f.kl, atol=1e-13) and np.allclose(bc.dW, b.dW, atol=1e-13)


def test_kd_gradients_by_finite_differences():
    hs, Ws, ht, Wt = _kd_rand(3, 4, 5, 6, 43)
    tf = O.LogitTransform(softcap=3.0, temperature=1.5)
    f = O.kd_forward(hs, Ws, ht, Wt, tf=tf)
    b = O.kd_backward(hs, Ws, ht, Wt, g=1.0 / f.n_valid, tf=tf)
    eps = 1e-6
    num = np.zeros_like(Ws)
    for v in range(Ws.shape[0]):
        for k in range(Ws.shape[1]):
            e = np.zeros_like(Ws)
            e[v, k] = eps
            num[v, k] = (O.kd_forward(hs, Ws + e, ht, Wt, tf=tf).loss -
                         O.kd_forward(hs, Ws - e, ht, Wt, tf=tf).loss) / (2 * eps)
    assert np.linalg.norm(num - b.dW) <= 1e-7 * np.linalg.norm(b.dW)
    numh = np.zeros_like(hs)
    for i in range(hs.shape[0]):
        for k in range(hs.shape[1]):
            e = np.zeros_like(hs)
            e[i, k] = eps
            numh[i, k] = (O.kd_forward(hs + e, Ws, ht, Wt, tf=tf).loss -
                          O.kd_forward(hs - e, Ws, ht, Wt, tf=tf).loss) / (2 * eps)
    assert np.linalg.norm(numh - b.dH) <= 1e-7 * np.linalg.norm(b.dH)


def _torch_jsd(zs, zt, beta):
    """Generalised JSD written with torch's kl_div on a log-sum-exp mixture."""
    log_ps, log_pt = torch.log_softmax(zs, -1), torch.log_softmax(zt, -1)
    log_m = torch.logsumexp(torch.stack([log_pt + np.log(beta), log_ps + np.log(1 - beta)]), 0)
    kl_t = torch.nn.functional.kl_div(log_m, log_pt, log_target=True, reduction="none").sum(-1)
    kl_s = torch.nn.functional.kl_div(log_m, log_ps, log_target=True, reduction="none").sum(-1)
    return beta * kl_t + (1 - beta) * kl_s, kl_s


@pytest.mark.parametrize("beta", [0.5, 0.1, 0.9])
def test_jsd_matches_torch_mixture_kl_divs_and_autograd(beta):
    hs, Ws, ht, Wt = _kd_rand(25, 7, 5, 31, 44)
    t = np.random.default_rng(3).integers(0, 31, 25)
    t[[2, 9, 17]] = O.IGNORE_INDEX
    w = np.random.default_rng(4).uniform(0.5, 2, 25)
    tf = O.LogitTransform(softcap=4.0, temperature=1.5)
    hst = torch.tensor(hs, requires_grad=True)
    Wst = torch.tensor(Ws, requires_grad=True)
    zs = 4.0 * torch.tanh((hst @ Wst.T) / 4.0) / 1.5
    zt = 4.0 * torch.tanh(torch.tensor(ht @ Wt.T) / 4.0) / 1.5
    jsd, kl_s = _torch_jsd(zs, zt, beta)
    m = torch.tensor(t != O.IGNORE_INDEX, dtype=torch.float64)
    loss = (m * torch.tensor(w) * jsd).sum() / m.sum()
    loss.backward()
    f = O.jsd_forward(hs, Ws, ht, Wt, beta, t, w, tf=tf)
    b = O.jsd_backward(hs, Ws, ht, Wt, beta, t, w, g=1.0 / f.n_valid, tf=tf)
    assert f.n_valid == 22
    assert np.allclose(f.jsd, (m * jsd).detach().numpy(), atol=1e-12)
    assert np.allclose(f.kl_sm, kl_s.detach().numpy(), atol=1e-12)
    assert f.loss == pytest.approx(float(loss.detach()), rel=1e-12)
    assert np.allclose(b.dH, hst.grad.numpy(), atol=1e-12) and np.allclose(b.dW, Wst.grad.numpy(), atol=1e-12)
    # chunking does not change anything
    fc = O.jsd_forward(hs, Ws, ht, Wt, beta, t, w, tf=tf, chunk_rows=4)
    bc = O.jsd_backward(hs, Ws, ht, Wt, beta, t, w, g=1.0 / f.n_valid, tf=tf, chunk_rows=4)
    assert np.allclose(fc.jsd, f.jsd, atol=1e-13) and np.allclose(bc.dW, b.dW, atol=1e-13)


def test_jsd_identical_heads_symmetry_and_bounds():
    hs, Ws, ht, Wt = _kd_rand(16, 6, 9, 23, 45)
    f = O.jsd_forward(hs, Ws, hs, Ws, 0.3)
    assert np.allclose(f.jsd, 0.0, atol=1e-13)
    b = O.jsd_backward(hs, Ws, hs, Ws, 0.3, g=1.0)
    assert np.allclose(b.dH, 0, atol=1e-13) and np.allclose(b.dW, 0, atol=1e-13)
    # the textbook JSD (beta = 1/2) is symmetric in its two distributions
    a = O.jsd_forward(hs, Ws, ht, Wt, 0.5)
    c = O.jsd_forward(ht, Wt, hs, Ws, 0.5)
    assert np.allclose(a.jsd, c.jsd, atol=1e-13) and np.all(a.jsd > 0)
    # 0 <= JSD_beta <= the entropy of the mixing weight, reached by disjoint
    # supports (huge opposite logits)
    for beta in (0.5, 0.2):
        hb = -beta * np.log(beta) - (1 - beta) * np.log(1 - beta)
        assert np.all(O.jsd_forward(hs, Ws, ht, Wt, beta).jsd <= hb + 1e-12)
        Wd = np.zeros((4, 1))
        Wd[0, 0], Wd[1, 0] = 400.0, -400.0
        far = O.jsd_forward(np.ones((1, 1)), Wd, np.ones((1, 1)), -Wd, beta)
        assert far.jsd[0] == pytest.approx(hb, abs=1e-12)


def test_jsd_limits_are_the_two_kl_divergences():
    # beta -> 0: JSD_beta / beta -> KL(p_t || p_s) (the forward KL of the
    # distillation oracle); beta -> 1: JSD_beta / (1 - beta) -> KL(p_s || p_t)
    hs, Ws, ht, Wt = _kd_rand(10, 5, 7, 19, 46)
    kl_ts = O.kd_forward(hs, Ws, ht, Wt).kl
    kl_st = O.kd_forward(ht, Wt, hs, Ws).kl
    eps = 1e-6
    assert np.allclose(O.jsd_forward(hs, Ws, ht, Wt, eps).jsd / eps, kl_ts, rtol=1e-4)
    assert np.allclose(O.jsd_forward(hs, Ws, ht, Wt, 1 - eps).jsd / eps, kl_st, rtol=1e-4)


def test_jsd_gradients_by_finite_differences():
    hs, Ws, ht, Wt = _kd_rand(3, 4, 5, 6, 47)
    tf = O.LogitTransform(softcap=3.0, temperature=1.5)
    beta = 0.3
    f = O.jsd_forward(hs, Ws, ht, Wt, beta, tf=tf)
    b = O.jsd_backward(hs, Ws, ht, Wt, beta, g=1.0 / f.n_valid, tf=tf)
    eps = 1e-6
    num = np.zeros_like(Ws)
    for v in range(Ws.shape[0]):
        for k in range(Ws.shape[1]):
            e = np.zeros_like(Ws)
            e[v, k] = eps
            num[v, k] = (O.jsd_forward(hs, Ws + e, ht, Wt, beta, tf=tf).loss -
                         O.jsd_forward(hs, Ws - e, ht, Wt, beta, tf=tf).loss) / (2 * eps)
    assert np.linalg.norm(num - b.dW) <= 1e-7 * np.linalg.norm(b.dW)
    numh = np.zeros_like(hs)
    for i in range(hs.shape[0]):
        for k in range(hs.shape[1]):
            e = np.zeros_like(hs)
            e[i, k] = eps
            numh[i, k] = (O.jsd_forward(hs + e, Ws, ht, Wt, beta, tf=tf).loss -
                          O.jsd_forward(hs - e, Ws, ht, Wt, beta, tf=tf).loss) / (2 * eps)
    assert np.linalg.norm(numh - b.dH) <= 1e-7 * np.linalg.norm(b.dH)


def test_jsd_rejects_beta_outside_the_open_interval():
    hs, Ws, ht, Wt = _kd_rand(2, 3, 3, 4, 48)
    for beta in (0.0, 1.0, -0.5, 1.5, float("nan")):
        with pytest.raises(ValueError):
            O.jsd_forward(hs, Ws, ht, Wt, beta)


# ------------------------------------------------------------------------ GRPO

def _grpo_rand(N, seed):
    r = np.random.default_rng(seed)
    lp = -r.uniform(0.1, 6.0, N)
    # ratios exp(-delta) kept >= 0.09 away from the clip edges 0.8 / 1.2
    delta = r.choice([-0.5, -0.1, 0.0, 0.1, 0.5, 1.0], N)
    A = r.standard_normal(N)
    ref = lp + r.uniform(-1.0, 1.0, N)
    mask = r.uniform(size=N) > 0.15
    return lp, lp + delta, ref, A, mask


def test_grpo_token_loss_matches_torch_autograd():
    lp, old, ref, A, mask = _grpo_rand(200, 50)
    for eps_low, eps_high, beta in ((0.2, 0.2, 0.0), (0.2, 0.28, 0.04), (0.1, 0.3, 0.5)):
        t = torch.tensor(lp, requires_grad=True)
        r = torch.exp(t - torch.tensor(old))
        At = torch.tensor(A)
        obj = torch.minimum(r * At, torch.clamp(r, 1 - eps_low, 1 + eps_high) * At)
        d = torch.tensor(ref) - t
        kl = torch.exp(d) - d - 1
        m = torch.tensor(mask, dtype=torch.float64)
        loss = (m * (beta * kl - obj)).sum() / m.sum()
        loss.backward()
        o = O.grpo_token_loss(lp, A, mask, old, ref, eps_low, eps_high, beta)
        assert o.n_valid == int(mask.sum())
        assert o.loss == pytest.approx(float(loss.detach()), rel=1e-13)
        # weights = -n_valid * dloss/dlogp
        assert np.allclose(o.weights, -o.n_valid * t.grad.numpy(), atol=1e-12)


def test_grpo_on_policy_is_the_advantage_weighted_nll_gradient():
    # old = logp (r = 1), no KL: the gradient is that of -sum(m A logp) / n_valid,
    # the GRPO-style loss of the per-token-weight path with w = A
    lp, _, _, A, mask = _grpo_rand(100, 51)
    o = O.grpo_token_loss(lp, A, mask)
    assert np.array_equal(o.weights, np.where(mask, A, 0.0))
    assert o.loss == pytest.approx(-float(np.sum(mask * A)) / int(mask.sum()), rel=1e-13)


def test_grpo_clip_region_has_no_gradient_and_kl_vanishes_at_the_reference():
    lp = np.log(np.array([0.5, 0.5, 0.5, 0.5]))
    old = lp - np.log(np.array([1.5, 0.5, 1.5, 0.5]))  # ratios 1.5, 0.5, 1.5, 0.5
    A = np.array([1.0, -1.0, -1.0, 1.0])
    o = O.grpo_token_loss(lp, A, np.ones(4, bool), old, eps_low=0.2, eps_high=0.2)
    # r > 1 + eps with A > 0 and r < 1 - eps with A < 0: clipped, no gradient;
    # the other two sit on the unclipped (smaller) branch
    assert o.weights[0] == 0.0 and o.weights[1] == 0.0
    assert o.weights[2] == pytest.approx(-1.5) and o.weights[3] == pytest.approx(0.5)
    assert o.token_loss[0] == pytest.approx(-1.2) and o.token_loss[1] == pytest.approx(0.8)
    k = O.grpo_token_loss(lp, np.zeros(4), np.ones(4, bool), ref_logp=lp, beta=0.7)
    assert np.all(k.token_loss == 0.0) and np.all(k.weights == 0.0)
    lp2, _, ref2, _, m2 = _grpo_rand(50, 52)
    k2 = O.grpo_token_loss(lp2, np.zeros(50), m2, ref_logp=ref2, beta=1.0)
    assert np.all(k2.token_loss >= 0.0)  # the k3 estimate is never negative


def test_grpo_full_path_matches_torch_autograd_through_the_head():
    hs, Ws, _, _ = _kd_rand(30, 6, 6, 23, 53)
    t = np.random.default_rng(9).integers(0, 23, 30)
    t[[4, 11]] = O.IGNORE_INDEX
    r = np.random.default_rng(10)
    A = r.standard_normal(30)
    f = O.forward(hs, Ws, t)
    m = t != O.IGNORE_INDEX
    old = f.logp + r.choice([-0.5, 0.0, 0.5], 30)
    ref = f.logp + r.uniform(-0.5, 0.5, 30)
    o = O.grpo_token_loss(f.logp, A, m, old, ref, 0.2, 0.28, 0.05)
    b = O.backward(hs, Ws, t, o.weights, g=1.0 / o.n_valid)
    ht = torch.tensor(hs, requires_grad=True)
    Wt = torch.tensor(Ws, requires_grad=True)
    logp = torch.log_softmax(ht @ Wt.T, -1)[torch.arange(30), torch.tensor(np.where(m, t, 0))]
    ratio = torch.exp(logp - torch.tensor(old))
    At = torch.tensor(A)
    obj = torch.minimum(ratio * At, torch.clamp(ratio, 0.8, 1.28) * At)
    d = torch.tensor(ref) - logp
    mt = torch.tensor(m, dtype=torch.float64)
    loss = (mt * (0.05 * (torch.exp(d) - d - 1) - obj)).sum() / mt.sum()
    loss.backward()
    assert o.loss == pytest.approx(float(loss.detach()), rel=1e-12)
    assert np.allclose(b.dH, ht.grad.numpy(), atol=1e-12) and np.allclose(b.dW, Wt.grad.numpy(), atol=1e-12)


# ------------------------------------------------------------------------ fp8

def test_e4m3_decode_matches_torch_for_every_code():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = O.e4m3_to_f64(codes)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(got[~np.isnan(got)], ref[~np.isnan(ref)])


def test_e4m3_rounding_matches_torch_saturating_conversion():
    r = np.random.default_rng(3)
    y = np.concatenate([r.standard_normal(20000).astype(np.float32) * s for s in (1e-4, 0.01, 1, 50, 400)]
                       + [np.array([0.0, -0.0, 448.0, 449.0, 1e6, -1e6, 2.0 ** -10, 3 * 2.0 ** -10,
                                    464.0, 240.0, 248.0, 232.0], dtype=np.float32)])
    ref = torch.from_numpy(np.clip(y, -448, 448)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = O.f32_to_e4m3(y)
    # -0.0 and 0.0 both decode to zero; compare values, and codes away from zero
    assert np.array_equal(O.e4m3_to_f64(got), O.e4m3_to_f64(ref))
    nz = y != 0
    assert np.array_equal(got[nz], ref[nz])


def test_row_quantiser_bounds_and_dequantised_forward():
    r = np.random.default_rng(4)
    x = r.standard_normal((50, 64)).astype(np.float32) * np.exp(r.standard_normal((50, 1)))
    x[7] = 0.0
    q, s = O.quantize_e4m3_rows(x)
    assert q.dtype == np.uint8 and s.dtype == np.float32 and s[7] == 1.0
    back = O.dequantize_e4m3_rows(q, s)
    # e4m3 keeps 3 mantissa bits: relative error <= 2^-4 for normals, row max exact-ish
    big = np.abs(x) > np.max(np.abs(x), axis=1, keepdims=True) * 2.0 ** -5
    assert np.all(np.abs(back - x)[big] <= np.abs(x)[big] * 2.0 ** -4 + 1e-12)
    assert np.allclose(np.max(np.abs(back), axis=1)[s != 1.0], np.max(np.abs(x), axis=1)[s != 1.0],
                       rtol=2.0 ** -4)
    h8, hs = O.quantize_e4m3_rows(r.standard_normal((20, 64)))
    W8, Ws = O.quantize_e4m3_rows(r.standard_normal((30, 64)) * 0.1)
    t = r.integers(0, 30, 20)
    f8 = O.forward_fp8(h8, hs, W8, Ws, t)
    f = O.forward(O.dequantize_e4m3_rows(h8, hs), O.dequantize_e4m3_rows(W8, Ws), t)
    assert np.array_equal(f8.logp, f.logp)
