"""fp64 CPU oracle for the chunked LM-head cross-entropy -- TEST INFRASTRUCTURE.

Only the tests, the smoke check and the benchmark's CPU-baseline leg may call
this module.  The CUDA library never imports it, and it imports nothing from
the library: the two share no code.  It is written to be read against the
pages, not to be fast; numpy's matmul is the only library primitive used for
the contractions.

What it computes (one row i of the flattened batch x context tokens, vocab
index v, hidden index k; bf16 inputs widened exactly to fp64):

    z[i,v]  = sum_k h[i,k] * W[v,k]                 logits, "hidden_states @ lm_head"
    lse[i]  = log sum_v exp(z[i,v])                 (max-shifted)
    m[i]    = [t_i != ignore_index]
    logp[i] = m[i] * (z[i,t_i] - lse[i])            selective log-softmax
    n_valid = sum_i m[i]
    loss    = -sum_i m[i] w[i] logp[i] / n_valid    (0 when n_valid == 0)
    D[i,v]  = (exp(z[i,v] - lse[i]) - [v == t_i]) * m[i] * w[i] * g
    dH      = D @ W        dW = D^T @ h

Sources:
  * Unsloth, "Reinforcement Learning GRPO with 7x longer context",
    section "Flattened sequence-length chunking": rows are the flattened
    (batch x context) tokens, processed in chunks; each chunk's logits are
    ``hidden_states_chunk @ lm_head``, upcast to float32 for accuracy (fp64
    here), followed by a log-softmax and a gather of the completion token.
    Equations 1-3 of the same section give the logit-memory estimates
    reproduced in ``logit_memory_gb``.
  * Same page, section "Offloading activations for log-softmax": the
    backward recomputes the chunk's logits and back-propagates through them;
    the gradient is the textbook softmax-minus-one-hot.
  * TRL v1.13 release article ("Training Beyond 1M Tokens"), section on the
    four hurdles: the loss is computed 256 rows at a time and the chunk
    losses are summed (loss_type="chunked_nll").
  * Per-token weights and the GRPO-style loss -sum(w*logp)/sum(mask) are the
    weighted form of the same masked mean; with w = 1 it is the mean NLL.

Readings where the pages are silent: ignored rows have logp = 0, a zero
dlogits row and no influence on anything but their own lse; n_valid = 0 gives
loss 0; the denominator counts unmasked rows, not the sum of weights; a
target outside [0, V) that is not ignore_index is an error here.
"""
from __future__ import annotations

import dataclasses

import numpy as np

IGNORE_INDEX = -100


def widen(x: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> exact fp64; float arrays -> fp64."""
    x = np.asarray(x)
    if x.dtype == np.uint16:
        return (x.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    return x.astype(np.float64)


def logits(h: np.ndarray, W: np.ndarray) -> np.ndarray:
    """z = h @ W^T in fp64 (one chunk's "hidden_states @ lm_head")."""
    return widen(h) @ widen(W).T


def logsumexp_rows(z: np.ndarray) -> np.ndarray:
    """log sum_v exp(z[i,v]) per row, shifted by the row max."""
    m = z.max(axis=1, keepdims=True)
    return (m + np.log(np.exp(z - m).sum(axis=1, keepdims=True)))[:, 0]


@dataclasses.dataclass(frozen=True)
class LogitTransform:
    """Elementwise logit transforms applied before the log-softmax.

    Unsloth GRPO page, section "Flattened sequence-length chunking": the
    chunked selective log-softmax takes logit_scale_multiply,
    logit_scale_divide, logit_softcapping and temperature.  Reading taken
    (the page prints neither order nor defaults): applied in that order, 0
    disables the first three, temperature 1 is the identity; soft-capping is
    y -> c * tanh(y / c).
    """

    scale_multiply: float = 0.0
    scale_divide: float = 0.0
    softcap: float = 0.0
    temperature: float = 1.0

    def apply(self, z: np.ndarray) -> np.ndarray:
        y = z
        if self.scale_multiply != 0.0:
            y = y * self.scale_multiply
        if self.scale_divide != 0.0:
            y = y / self.scale_divide
        if self.softcap != 0.0:
            y = self.softcap * np.tanh(y / self.softcap)
        if self.temperature != 1.0:
            y = y / self.temperature
        return y

    def grad(self, z: np.ndarray) -> np.ndarray:
        """dy/dz of apply(), elementwise (chain rule of the steps above)."""
        d = np.ones_like(z)
        y = z
        if self.scale_multiply != 0.0:
            y = y * self.scale_multiply
            d = d * self.scale_multiply
        if self.scale_divide != 0.0:
            y = y / self.scale_divide
            d = d / self.scale_divide
        if self.softcap != 0.0:
            d = d * (1.0 - np.tanh(y / self.softcap) ** 2)
            y = self.softcap * np.tanh(y / self.softcap)
        if self.temperature != 1.0:
            d = d / self.temperature
        return d


def _tf(z: np.ndarray, tf: "LogitTransform | None") -> np.ndarray:
    return z if tf is None else tf.apply(z)


def _mask(targets: np.ndarray, V: int, ignore_index: int) -> np.ndarray:
    t = np.asarray(targets, dtype=np.int64)
    m = t != ignore_index
    bad = m & ((t < 0) | (t >= V))
    if bad.any():
        raise ValueError(f"{int(bad.sum())} targets outside [0, V) and != ignore_index")
    return m


def _weights(weights, N: int) -> np.ndarray:
    if weights is None:
        return np.ones(N, dtype=np.float64)
    return np.asarray(weights, dtype=np.float64)


@dataclasses.dataclass
class Forward:
    lse: np.ndarray  # [N] fp64
    logp: np.ndarray  # [N] fp64, 0 on ignored rows
    n_valid: int
    loss: float


def selective_log_softmax(z: np.ndarray, targets: np.ndarray, mask: np.ndarray):
    """Per-row (lse, logp) of a logits block: log_softmax, then gather t_i."""
    lse = logsumexp_rows(z)
    rows = np.arange(z.shape[0])
    t = np.where(mask, targets, 0)
    logp = np.where(mask, z[rows, t] - lse, 0.0)
    return lse, logp


def forward(h, W, targets, weights=None, ignore_index: int = IGNORE_INDEX,
            chunk_rows: int | None = None, tf: LogitTransform | None = None) -> Forward:
    """Chunked selective log-softmax and masked (weighted) mean NLL.

    Rows are taken ``chunk_rows`` at a time (all at once when None); each
    chunk's logits are formed in full, log-softmaxed, the target column is
    gathered, and the chunk's loss terms are summed into the total.
    """
    hf, Wf = widen(h), widen(W)
    N, V = hf.shape[0], Wf.shape[0]
    t = np.asarray(targets, dtype=np.int64)
    m = _mask(t, V, ignore_index)
    w = _weights(weights, N)
    step = N if chunk_rows is None else max(1, int(chunk_rows))
    lse = np.zeros(N)
    logp = np.zeros(N)
    total = 0.0
    for r0 in range(0, N, step):
        r1 = min(N, r0 + step)
        z = _tf(hf[r0:r1] @ Wf.T, tf)
        lse[r0:r1], logp[r0:r1] = selective_log_softmax(z, t[r0:r1], m[r0:r1])
        total += float(np.sum(m[r0:r1] * w[r0:r1] * logp[r0:r1]))
    n_valid = int(m.sum())
    loss = -total / n_valid if n_valid > 0 else 0.0
    return Forward(lse, logp, n_valid, loss)


def probs(z: np.ndarray, lse: np.ndarray) -> np.ndarray:
    """Softmax rows p[i,v] = exp(z[i,v] - lse[i])."""
    return np.exp(z - lse[:, None])


def dlogits(z, lse, targets, mask, w, g: float) -> np.ndarray:
    """D = (softmax - onehot(t)) * m * w * g for a block of rows."""
    D = probs(z, lse)
    rows = np.nonzero(mask)[0]
    D[rows, np.asarray(targets)[rows]] -= 1.0
    return D * (mask * w * g)[:, None]


@dataclasses.dataclass
class Backward:
    dH: np.ndarray  # [N,H] fp64
    dW: np.ndarray  # [V,H] fp64


def backward(h, W, targets, weights=None, g: float = 1.0,
             ignore_index: int = IGNORE_INDEX, chunk_rows: int | None = None,
             lse: np.ndarray | None = None, tf: LogitTransform | None = None) -> Backward:
    """dH = D W and dW = D^T h, recomputing each chunk's logits.

    ``lse`` defaults to the oracle's own forward.  g multiplies D literally
    (g = 1/n_valid gives the gradient of the mean loss).  With a logit
    transform y = f(z), D is taken with respect to z: (softmax(y) - onehot)
    times f'(z).
    """
    hf, Wf = widen(h), widen(W)
    N, V = hf.shape[0], Wf.shape[0]
    t = np.asarray(targets, dtype=np.int64)
    m = _mask(t, V, ignore_index)
    w = _weights(weights, N)
    step = N if chunk_rows is None else max(1, int(chunk_rows))
    dH = np.zeros_like(hf)
    dW = np.zeros_like(Wf)
    for r0 in range(0, N, step):
        r1 = min(N, r0 + step)
        z = hf[r0:r1] @ Wf.T
        y = _tf(z, tf)
        l = logsumexp_rows(y) if lse is None else np.asarray(lse[r0:r1], dtype=np.float64)
        D = dlogits(y, l, t[r0:r1], m[r0:r1], w[r0:r1], g)
        if tf is not None:
            D *= tf.grad(z)
        dH[r0:r1] = D @ Wf
        dW += D.T @ hf[r0:r1]
    return Backward(dH, dW)


def rows_forward(h, W, targets, rows, ignore_index: int = IGNORE_INDEX,
                 tf: LogitTransform | None = None):
    """(lse, logp) of the selected rows only; the same formulas as forward()."""
    rows = np.asarray(rows, dtype=np.int64)
    Wf = widen(W)
    t = np.asarray(targets, dtype=np.int64)[rows]
    m = _mask(t, Wf.shape[0], ignore_index)
    z = _tf(widen(np.asarray(h)[rows]) @ Wf.T, tf)
    return selective_log_softmax(z, t, m)


def rows_backward(h, W, targets, rows, weights=None, g: float = 1.0,
                  ignore_index: int = IGNORE_INDEX, vocab_rows=None,
                  tf: LogitTransform | None = None):
    """dH of the selected rows and those rows' contribution to dW.

    Returns (dH[rows], dW_part) where dW_part = D[rows]^T h[rows], restricted
    to ``vocab_rows`` when given.  Each row's lse is the oracle's own.
    """
    rows = np.asarray(rows, dtype=np.int64)
    hf = widen(np.asarray(h)[rows])
    Wf = widen(W)
    t = np.asarray(targets, dtype=np.int64)[rows]
    m = _mask(t, Wf.shape[0], ignore_index)
    w = _weights(None if weights is None else np.asarray(weights)[rows], len(rows))
    z = hf @ Wf.T
    y = _tf(z, tf)
    D = dlogits(y, logsumexp_rows(y), t, m, w, g)
    if tf is not None:
        D *= tf.grad(z)
    del y
    dH = D @ Wf
    if vocab_rows is not None:
        D = D[:, np.asarray(vocab_rows, dtype=np.int64)]
    return dH, D.T @ hf


def rows_all(h, W, targets, rows, weights=None, g: float = 1.0,
             ignore_index: int = IGNORE_INDEX, vocab_rows=None,
             tf: LogitTransform | None = None):
    """rows_forward and rows_backward of the same rows from one logits block.

    Returns (lse, logp, dH[rows], dW_part) with dW_part = D[rows]^T h[rows]
    (restricted to ``vocab_rows`` when given).
    """
    rows = np.asarray(rows, dtype=np.int64)
    hf = widen(np.asarray(h)[rows])
    Wf = widen(W)
    t = np.asarray(targets, dtype=np.int64)[rows]
    m = _mask(t, Wf.shape[0], ignore_index)
    w = _weights(None if weights is None else np.asarray(weights)[rows], len(rows))
    z = hf @ Wf.T
    y = _tf(z, tf)
    lse, logp = selective_log_softmax(y, t, m)
    D = dlogits(y, lse, t, m, w, g)
    del y
    if tf is not None:
        D *= tf.grad(z)
    del z
    dH = D @ Wf
    if vocab_rows is not None:
        D = D[:, np.asarray(vocab_rows, dtype=np.int64)]
    return lse, logp, dH, D.T @ hf


def vocab_rows_dW(h, W, targets, lse, vocab_rows, weights=None, g: float = 1.0,
                  ignore_index: int = IGNORE_INDEX, block_rows: int = 4096):
    """dW restricted to the given vocabulary rows: D[:, vocab_rows]^T h.

    Needs every row's lse (the oracle's own full forward); the columns of D
    are formed from z[:, vocab_rows] = h W[vocab_rows]^T only.
    """
    vr = np.asarray(vocab_rows, dtype=np.int64)
    Wv = widen(np.asarray(W)[vr])
    hN = np.asarray(h)
    N = hN.shape[0]
    t = np.asarray(targets, dtype=np.int64)
    m = _mask(t, np.asarray(W).shape[0], ignore_index)
    w = _weights(weights, N)
    out = np.zeros((len(vr), hN.shape[1]))
    for r0 in range(0, N, block_rows):
        r1 = min(N, r0 + block_rows)
        hf = widen(hN[r0:r1])
        Dv = np.exp(hf @ Wv.T - np.asarray(lse[r0:r1], dtype=np.float64)[:, None])
        hit = (t[r0:r1][:, None] == vr[None, :]) & m[r0:r1][:, None]
        Dv -= hit
        Dv *= (m[r0:r1] * w[r0:r1] * g)[:, None]
        out += Dv.T @ hf
    return out


@dataclasses.dataclass
class KDForward:
    kl: np.ndarray  # [N] fp64, 0 on ignored rows
    lse_s: np.ndarray  # [N] student log-sum-exp
    lse_t: np.ndarray  # [N] teacher log-sum-exp
    n_valid: int
    loss: float


def _kd_mask(targets, N: int, ignore_index: int) -> np.ndarray:
    if targets is None:
        return np.ones(N, dtype=bool)
    return np.asarray(targets, dtype=np.int64) != ignore_index


def kd_forward(hs, Ws, ht, Wt, targets=None, weights=None, ignore_index: int = IGNORE_INDEX,
               tf: LogitTransform | None = None, chunk_rows: int | None = None) -> KDForward:
    """Distillation of a teacher head into a student head, chunk by chunk.

    TRL v1.13 article, speed & memory section: the distillation trainer
    computes every chunk twice, once with the student's head and once with
    the teacher's.  Reading taken (the page names no formula): the per-token
    loss is KL(p_teacher || p_student) over the vocabulary, masked by
    ignore_index rows of ``targets`` (all rows count when None) and weighted
    like the cross-entropy; loss = sum(m w kl) / sum(m).  Both heads' logits
    pass through the same transform (e.g. a distillation temperature).
    """
    hsf, Wsf, htf, Wtf = widen(hs), widen(Ws), widen(ht), widen(Wt)
    N = hsf.shape[0]
    m = _kd_mask(targets, N, ignore_index)
    w = _weights(weights, N)
    step = N if chunk_rows is None else max(1, int(chunk_rows))
    kl = np.zeros(N)
    lse_s = np.zeros(N)
    lse_t = np.zeros(N)
    for r0 in range(0, N, step):
        r1 = min(N, r0 + step)
        zs = _tf(hsf[r0:r1] @ Wsf.T, tf)
        zt = _tf(htf[r0:r1] @ Wtf.T, tf)
        ls, lt = logsumexp_rows(zs), logsumexp_rows(zt)
        log_ps, log_pt = zs - ls[:, None], zt - lt[:, None]
        kl[r0:r1] = np.where(m[r0:r1], np.sum(np.exp(log_pt) * (log_pt - log_ps), axis=1), 0.0)
        lse_s[r0:r1], lse_t[r0:r1] = ls, lt
    n_valid = int(m.sum())
    loss = float(np.sum(m * w * kl)) / n_valid if n_valid > 0 else 0.0
    return KDForward(kl, lse_s, lse_t, n_valid, loss)


def kd_backward(hs, Ws, ht, Wt, targets=None, weights=None, g: float = 1.0,
                ignore_index: int = IGNORE_INDEX, tf: LogitTransform | None = None,
                chunk_rows: int | None = None) -> Backward:
    """Student gradients of the distillation loss (teacher frozen):
    D = (p_student - p_teacher) * m * w * g * f'(z_student); dH = D Ws, dW = D^T hs."""
    hsf, Wsf, htf, Wtf = widen(hs), widen(Ws), widen(ht), widen(Wt)
    N = hsf.shape[0]
    m = _kd_mask(targets, N, ignore_index)
    w = _weights(weights, N)
    step = N if chunk_rows is None else max(1, int(chunk_rows))
    dH = np.zeros_like(hsf)
    dW = np.zeros_like(Wsf)
    for r0 in range(0, N, step):
        r1 = min(N, r0 + step)
        z = hsf[r0:r1] @ Wsf.T
        zs = _tf(z, tf)
        zt = _tf(htf[r0:r1] @ Wtf.T, tf)
        D = probs(zs, logsumexp_rows(zs)) - probs(zt, logsumexp_rows(zt))
        D *= (m[r0:r1] * w[r0:r1] * g)[:, None]
        if tf is not None:
            D *= tf.grad(z)
        dH[r0:r1] = D @ Wsf
        dW += D.T @ hsf[r0:r1]
    return Backward(dH, dW)


@dataclasses.dataclass
class JSDForward:
    jsd: np.ndarray     # [N] m * JSD_beta(p_teacher, p_student)
    lse_s: np.ndarray   # [N]
    lse_t: np.ndarray   # [N]
    kl_sm: np.ndarray   # [N] KL(p_student || mixture) of every row (mask not applied)
    n_valid: int
    loss: float


def _jsd_rows(zs: np.ndarray, zt: np.ndarray, beta: float):
    """Per-row generalised Jensen-Shannon divergence of two logit blocks.

    With p_s = softmax(zs), p_t = softmax(zt) and the mixture
    M = beta * p_t + (1 - beta) * p_s:
        JSD_beta = beta * KL(p_t || M) + (1 - beta) * KL(p_s || M),
    terms with a zero probability contribute 0 (x log x -> 0).  Returns
    (jsd, KL(p_s || M), lse_s, lse_t, p_s, M)."""
    ls, lt = logsumexp_rows(zs), logsumexp_rows(zt)
    log_ps, log_pt = zs - ls[:, None], zt - lt[:, None]
    ps, pt = np.exp(log_ps), np.exp(log_pt)
    mix = beta * pt + (1.0 - beta) * ps
    with np.errstate(divide="ignore", invalid="ignore"):
        log_mix = np.log(mix)
        kl_t = np.sum(np.where(pt > 0, pt * (log_pt - log_mix), 0.0), axis=1)
        kl_s = np.sum(np.where(ps > 0, ps * (log_ps - log_mix), 0.0), axis=1)
    return beta * kl_t + (1.0 - beta) * kl_s, kl_s, ls, lt, ps, log_mix


def _check_beta(beta: float) -> float:
    beta = float(beta)
    if not (0.0 < beta < 1.0):
        raise ValueError("beta must lie strictly between 0 and 1")
    return beta


def jsd_forward(hs, Ws, ht, Wt, beta: float = 0.5, targets=None, weights=None,
                ignore_index: int = IGNORE_INDEX, tf: LogitTransform | None = None,
                chunk_rows: int | None = None) -> JSDForward:
    """Jensen-Shannon distillation of a teacher head into a student head.

    TRL v1.13 article, section "Other changes in v1.13": TRL's fused linear
    losses include a JSD loss next to DPO, KTO and GRPO; the page gives no
    formula.  Reading taken: the generalised Jensen-Shannon divergence with
    mixture weight beta in (0, 1) (beta = 1/2 is the textbook JSD), per
    token, masked by ignore_index rows of ``targets`` (all rows when None),
    weighted and averaged like the cross-entropy; loss = sum(m w jsd) /
    sum(m).  Both heads pass through the same logit transform.
    """
    beta = _check_beta(beta)
    hsf, Wsf, htf, Wtf = widen(hs), widen(Ws), widen(ht), widen(Wt)
    N = hsf.shape[0]
    m = _kd_mask(targets, N, ignore_index)
    w = _weights(weights, N)
    step = N if chunk_rows is None else max(1, int(chunk_rows))
    jsd, kl_sm, lse_s, lse_t = np.zeros(N), np.zeros(N), np.zeros(N), np.zeros(N)
    for r0 in range(0, N, step):
        r1 = min(N, r0 + step)
        zs = _tf(hsf[r0:r1] @ Wsf.T, tf)
        zt = _tf(htf[r0:r1] @ Wtf.T, tf)
        j, ksm, ls, lt, _, _ = _jsd_rows(zs, zt, beta)
        jsd[r0:r1] = np.where(m[r0:r1], j, 0.0)
        kl_sm[r0:r1], lse_s[r0:r1], lse_t[r0:r1] = ksm, ls, lt
    n_valid = int(m.sum())
    loss = float(np.sum(m * w * jsd)) / n_valid if n_valid > 0 else 0.0
    return JSDForward(jsd, lse_s, lse_t, kl_sm, n_valid, loss)


def jsd_backward(hs, Ws, ht, Wt, beta: float = 0.5, targets=None, weights=None, g: float = 1.0,
                 ignore_index: int = IGNORE_INDEX, tf: LogitTransform | None = None,
                 chunk_rows: int | None = None) -> Backward:
    """Student gradients of the JSD distillation loss (teacher frozen).

    JSD_beta = beta sum p_t log p_t + (1 - beta) sum p_s log p_s - sum M log M,
    so dJSD/dp_s[v] = (1 - beta) log(p_s[v] / M[v]); through the softmax,
        D[v] = (1 - beta) p_s[v] (log(p_s[v] / M[v]) - KL(p_s || M)) * m w g * f'(z_s[v]),
    then dH = D Ws and dW = D^T hs."""
    beta = _check_beta(beta)
    hsf, Wsf, htf, Wtf = widen(hs), widen(Ws), widen(ht), widen(Wt)
    N = hsf.shape[0]
    m = _kd_mask(targets, N, ignore_index)
    w = _weights(weights, N)
    step = N if chunk_rows is None else max(1, int(chunk_rows))
    dH = np.zeros_like(hsf)
    dW = np.zeros_like(Wsf)
    for r0 in range(0, N, step):
        r1 = min(N, r0 + step)
        z = hsf[r0:r1] @ Wsf.T
        zs = _tf(z, tf)
        zt = _tf(htf[r0:r1] @ Wtf.T, tf)
        _, kl_s, ls, _, ps, log_mix = _jsd_rows(zs, zt, beta)
        with np.errstate(divide="ignore", invalid="ignore"):
            g_s = np.where(ps > 0, (zs - ls[:, None]) - log_mix, 0.0)
        D = (1.0 - beta) * ps * (g_s - kl_s[:, None])
        D *= (m[r0:r1] * w[r0:r1] * g)[:, None]
        if tf is not None:
            D *= tf.grad(z)
        dH[r0:r1] = D @ Wsf
        dW += D.T @ hsf[r0:r1]
    return Backward(dH, dW)


# ------------------------------------------------------------------ GRPO token loss

@dataclasses.dataclass
class GRPOTokens:
    token_loss: np.ndarray  # [N] m * per-token loss
    weights: np.ndarray     # [N] -m * d(token loss)/d(logp): per-token weights for backward()
    n_valid: int
    loss: float             # sum(token_loss) / n_valid (0 when n_valid == 0)


def grpo_token_loss(logp, advantages, mask, old_logp=None, ref_logp=None, eps_low: float = 0.2,
                    eps_high: float = 0.2, beta: float = 0.0) -> GRPOTokens:
    """Per-token GRPO objective on the log-probs of the sampled tokens.

    TRL v1.13 article, section "Other changes in v1.13": TRL's fused linear
    losses include a GRPO loss; the page gives no formula.  Reading taken
    (the GRPO objective with a clipped probability ratio and the k3 estimate
    of the KL divergence to a reference policy), per token with the mask m:
        r     = exp(logp - old_logp)              (old_logp = logp when absent: r = 1)
        obj   = min(r A, clip(r, 1 - eps_low, 1 + eps_high) A)
        kl    = exp(ref - logp) - (ref - logp) - 1  (0 when ref_logp is absent)
        token = m (beta kl - obj),   loss = sum(token) / sum(m)
    old_logp and ref_logp are constants (no gradient).  The derivative of the
    token loss by logp is  m (beta (1 - exp(ref - logp)) - A r [the unclipped
    term is the minimum]); weights = -that derivative, so that
    backward(..., weights, g = 1 / n_valid) gives the loss's dH and dW."""
    lp = np.asarray(logp, dtype=np.float64)
    A = np.asarray(advantages, dtype=np.float64)
    m = np.asarray(mask, dtype=bool)
    old = lp if old_logp is None else np.asarray(old_logp, dtype=np.float64)
    r = np.exp(lp - old)
    unclipped = r * A
    clipped = np.clip(r, 1.0 - eps_low, 1.0 + eps_high) * A
    obj = np.minimum(unclipped, clipped)
    d_obj = np.where(unclipped <= clipped, unclipped, 0.0)  # d obj / d logp
    if ref_logp is None or beta == 0.0:
        kl = np.zeros_like(lp)
        d_kl = np.zeros_like(lp)
    else:
        diff = np.asarray(ref_logp, dtype=np.float64) - lp
        kl = np.exp(diff) - diff - 1.0
        d_kl = 1.0 - np.exp(diff)
    token = np.where(m, beta * kl - obj, 0.0)
    weights = np.where(m, -(beta * d_kl - d_obj), 0.0)
    n_valid = int(m.sum())
    loss = float(token.sum()) / n_valid if n_valid > 0 else 0.0
    return GRPOTokens(token, weights, n_valid, loss)


# ------------------------------------------------------------------ fp8 (e4m3)

E4M3_MAX = 448.0


def e4m3_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact value of e4m3 bytes (sign, 4 exponent bits with bias 7, 3 mantissa
    bits; exponent 0 is subnormal; S.1111.111 is NaN; no infinities)."""
    b = np.asarray(bits, dtype=np.uint8).astype(np.int64)
    sign = np.where(b & 0x80, -1.0, 1.0)
    e = (b >> 3) & 0xF
    m = b & 0x7
    val = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    val = np.where((e == 15) & (m == 7), np.nan, val)
    return sign * val


def f32_to_e4m3(y: np.ndarray) -> np.ndarray:
    """Round fp32 values to e4m3 bytes: nearest, ties to even, saturating at
    +-448 (finite inputs)."""
    y = np.asarray(y, dtype=np.float32).astype(np.float64)
    a = np.minimum(np.abs(y), E4M3_MAX)
    _, ex = np.frexp(np.where(a > 0, a, 1.0))  # a = f * 2^ex, f in [0.5, 1)
    e = np.maximum(ex - 1, -6)  # unbiased exponent, subnormals share 2^-6
    quantum = np.exp2(e - 3.0)
    r = np.rint(a / quantum) * quantum  # exact: powers of two
    r = np.minimum(r, E4M3_MAX)
    # encode
    _, ex2 = np.frexp(np.where(r > 0, r, 1.0))
    e2 = ex2 - 1
    normal = r >= 2.0 ** -6
    mant = np.where(normal, np.rint((r / np.exp2(e2) - 1.0) * 8.0), np.rint(r / 2.0 ** -9))
    code = np.where(normal, ((e2 + 7) << 3) | mant.astype(np.int64), mant.astype(np.int64))
    code = np.where(r == 0, 0, code)
    return (code | np.where(y < 0, 0x80, 0)).astype(np.uint8)


def quantize_e4m3_rows(x) -> tuple[np.ndarray, np.ndarray]:
    """Per-row e4m3 quantisation: scale = max|x_row| / 448 (fp32; 1 for an
    all-zero row), q = e4m3(x / scale) with the division in fp32.  Returns
    (q bytes [rows, cols], scale fp32 [rows])."""
    xf = widen(x).astype(np.float32)
    amax = np.max(np.abs(xf), axis=1)
    scale = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
    return f32_to_e4m3(xf / scale[:, None]), scale


def dequantize_e4m3_rows(q, scale) -> np.ndarray:
    return e4m3_to_f64(q) * np.asarray(scale, dtype=np.float64)[:, None]


def forward_fp8(h8, h_scale, W8, W_scale, targets, weights=None, ignore_index: int = IGNORE_INDEX,
                tf: LogitTransform | None = None, chunk_rows: int | None = None) -> Forward:
    """The forward of the e4m3-quantised operands: exactly forward() on the
    dequantised values (logits = (q_h s_h)(q_W s_W)^T)."""
    return forward(dequantize_e4m3_rows(h8, h_scale), dequantize_e4m3_rows(W8, W_scale), targets,
                   weights, ignore_index, chunk_rows, tf)


def logit_memory_gb(context_length: int, vocab_dim: int, batch_size: int = 1,
                    multiplier: int = 1) -> float:
    """Unsloth GRPO page, flattened-chunking section, Equations 1-3.

    Eq.1 (whole batch): batch x context x vocab / 1024^3;
    Eq.2 (one sample at a time): context x vocab / 1024^3;
    Eq.3 (sequence chunked): (context / multiplier) x vocab / 1024^3.
    The formula counts elements; multiply by the element size for bytes.
    """
    return batch_size * (context_length / multiplier) * vocab_dim / 1024 ** 3


def default_chunk_multiplier(context_length: int) -> int:
    """Same section: the default sequence-chunk multiplier max(4, L // 4096)."""
    return max(4, context_length // 4096)
