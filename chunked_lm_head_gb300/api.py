"""PyTorch-facing calls of libflce (device memory and streams from torch).

Every arithmetic step runs in libflce's CUDA kernels; this module only checks
tensor properties, allocates outputs and passes pointers.
"""
from __future__ import annotations

import torch

from . import _lib

IGNORE_INDEX = -100


def _check(h: torch.Tensor, W: torch.Tensor, targets: torch.Tensor, weights):
    if not (h.is_cuda and W.is_cuda and targets.is_cuda):
        raise ValueError("h, W and targets must be CUDA tensors")
    if h.dtype != torch.bfloat16 or W.dtype != torch.bfloat16:
        raise ValueError("h and W must be bfloat16")
    if targets.dtype != torch.int64:
        raise ValueError("targets must be int64")
    if h.dim() != 2 or W.dim() != 2 or h.shape[1] != W.shape[1] or targets.shape != (h.shape[0],):
        raise ValueError("expected h[N,H], W[V,H], targets[N]")
    if not (h.is_contiguous() and W.is_contiguous() and targets.is_contiguous()):
        raise ValueError("h, W and targets must be contiguous")
    if weights is not None:
        if weights.dtype != torch.float32 or weights.shape != (h.shape[0],) or not weights.is_contiguous():
            raise ValueError("weights must be a contiguous float32 [N] tensor")


def workspace_bytes(N: int, H: int, V: int, chunk_rows: int) -> int:
    return _lib.flce_workspace_bytes(N, H, V, chunk_rows)


def forward(h, W, targets, weights=None, chunk_rows: int = 256, ignore_index: int = IGNORE_INDEX,
            workspace: torch.Tensor | None = None, stream=None, transform=None,
            skip_ignored: bool = False):
    """Returns dict(logp[N] f32, lse[N] f32, loss[] f32, n_valid[] i64), on device.

    ``transform``: None, or a dict with scale_multiply / scale_divide /
    softcap / temperature (flce_logit_transform).  ``skip_ignored``: the GEMM
    skips the ignored rows, whose lse is then NaN (the backward never reads
    it)."""
    _check(h, W, targets, weights)
    N, H = h.shape
    V = W.shape[0]
    dev = h.device
    logp = torch.empty(N, dtype=torch.float32, device=dev)
    lse = torch.empty(N, dtype=torch.float32, device=dev)
    loss = torch.empty((), dtype=torch.float32, device=dev)
    n_valid = torch.empty((), dtype=torch.int64, device=dev)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    flags = _lib.FORWARD_SKIP_IGNORED if skip_ignored else 0
    st = _lib.flce_forward_ex2(h, W, targets, weights, N, H, V, chunk_rows, ignore_index, transform,
                               flags, logp, lse, loss, n_valid, workspace, ws_bytes, stream)
    _lib.check("flce_forward_ex2", st)
    return {"logp": logp, "lse": lse, "loss": loss, "n_valid": n_valid}


def _device_scalar(x, dtype, dev):
    """A one-element device tensor of x (a tensor already there stays there: no
    host synchronisation), or None."""
    if x is None:
        return None
    return torch.as_tensor(x).to(device=dev, dtype=dtype).reshape(1).contiguous()


def backward(h, W, targets, weights, lse, grad_scale: float, chunk_rows: int = 256,
             ignore_index: int = IGNORE_INDEX, need_dH: bool = True, need_dW: bool = True,
             workspace: torch.Tensor | None = None, stream=None, transform=None,
             scale=None, count=None):
    """Returns (dH[N,H] bf16 or None, dW[V,H] f32 or None).

    scale / count (optional, one-element device tensors, e.g. the incoming
    gradient of the loss and the forward's n_valid) multiply grad_scale by
    scale / max(count, 1) on the device."""
    _check(h, W, targets, weights)
    N, H = h.shape
    V = W.shape[0]
    dH = torch.empty_like(h) if need_dH else None
    dW = torch.empty((V, H), dtype=torch.float32, device=h.device) if need_dW else None
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    scale = _device_scalar(scale, torch.float32, h.device)
    count = _device_scalar(count, torch.int64, h.device)
    if scale is None and count is None:
        st = _lib.flce_backward_ex(h, W, targets, weights, lse, grad_scale, dH, dW, N, H, V, chunk_rows,
                                   ignore_index, transform, workspace, ws_bytes, stream)
        _lib.check("flce_backward_ex", st)
    else:
        st = _lib.flce_backward_ex2(h, W, targets, weights, lse, grad_scale, scale, count, dH, dW, N, H,
                                    V, chunk_rows, ignore_index, transform, workspace, ws_bytes, stream)
        _lib.check("flce_backward_ex2", st)
    return dH, dW


def scale_grads(dH, dW, scale, stream=None):
    """dH, dW *= scale in place (scale: a one-element device tensor; a scale of
    exactly 1 moves no data).  Returns (dH, dW)."""
    dev = (dH if dH is not None else dW).device
    s = _device_scalar(scale, torch.float32, dev)
    st = _lib.flce_scale_grads(dH, 0 if dH is None else dH.numel(), dW, 0 if dW is None else dW.numel(), s,
                               stream)
    _lib.check("flce_scale_grads", st)
    return dH, dW


def forward_backward(h, W, targets, weights=None, chunk_rows: int = 4096,
                     ignore_index: int = IGNORE_INDEX, grad_scale: float = 1.0, need_dH: bool = True,
                     need_dW: bool = True, workspace: torch.Tensor | None = None, stream=None,
                     transform=None, need_lse: bool = True):
    """Loss and its gradients in one call without the logits recompute
    (flce_forward_backward): dict(logp, lse, loss, n_valid, dH, dW).
    need_lse=False returns lse None and lets the call skip the ignored rows'
    forward."""
    _check(h, W, targets, weights)
    N, H = h.shape
    V = W.shape[0]
    dev = h.device
    logp = torch.empty(N, dtype=torch.float32, device=dev)
    lse = torch.empty(N, dtype=torch.float32, device=dev) if need_lse else None
    loss = torch.empty((), dtype=torch.float32, device=dev)
    n_valid = torch.empty((), dtype=torch.int64, device=dev)
    dH = torch.empty_like(h) if need_dH else None
    dW = torch.empty((V, H), dtype=torch.float32, device=dev) if need_dW else None
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = _lib.flce_forward_backward(h, W, targets, weights, N, H, V, chunk_rows, ignore_index,
                                    transform, grad_scale, logp, lse, loss, n_valid, dH, dW,
                                    workspace, ws_bytes, stream)
    _lib.check("flce_forward_backward", st)
    return {"logp": logp, "lse": lse, "loss": loss, "n_valid": n_valid, "dH": dH, "dW": dW}


class LinearCrossEntropy(torch.autograd.Function):
    """loss = -sum(w * logp) / n_valid with logits recomputed in backward.

    The forward keeps no logits; the backward recomputes them chunk by chunk
    (the recompute-in-backward of Unsloth's offloaded log-softmax function).
    """

    @staticmethod
    def forward(ctx, h, W, targets, weights, chunk_rows, ignore_index, transform=None):
        # the backward reads lse of the non-ignored rows only
        out = forward(h, W, targets, weights, chunk_rows, ignore_index, transform=transform,
                      skip_ignored=True)
        ctx.transform = transform
        ctx.save_for_backward(h, W, targets, weights if weights is not None else torch.empty(0),
                              out["lse"], out["n_valid"])
        ctx.has_weights = weights is not None
        ctx.chunk_rows = chunk_rows
        ctx.ignore_index = ignore_index
        ctx.mark_non_differentiable(out["logp"], out["n_valid"])
        return out["loss"], out["logp"], out["n_valid"]

    @staticmethod
    def backward(ctx, grad_loss, grad_logp, grad_n):
        h, W, targets, weights, lse, n_valid = ctx.saved_tensors
        weights = weights if ctx.has_weights else None
        # grad_loss / n_valid is applied on the device: no host synchronisation
        dH, dW = backward(h, W, targets, weights, lse, 1.0, ctx.chunk_rows, ctx.ignore_index,
                          need_dH=ctx.needs_input_grad[0], need_dW=ctx.needs_input_grad[1],
                          transform=ctx.transform, scale=grad_loss, count=n_valid)
        return dH, dW, None, None, None, None, None


class LinearCrossEntropyOneCall(torch.autograd.Function):
    """The same loss with its gradients computed in the forward call
    (flce_forward_backward, no logits recompute); the backward only scales
    them by the incoming gradient of the loss."""

    @staticmethod
    def forward(ctx, h, W, targets, weights, chunk_rows, ignore_index, transform=None):
        out = forward_backward(h, W, targets, weights, chunk_rows, ignore_index,
                               need_dH=ctx.needs_input_grad[0], need_dW=ctx.needs_input_grad[1],
                               transform=transform, need_lse=False)
        ctx.grads = (out["dH"], out["dW"])
        ctx.mark_non_differentiable(out["logp"], out["n_valid"])
        return out["loss"], out["logp"], out["n_valid"]

    @staticmethod
    def backward(ctx, grad_loss, grad_logp, grad_n):
        dH, dW = ctx.grads
        ctx.grads = None
        # e.g. a loss scale or a weighted sum of losses; read on the device
        # (no host synchronisation; a gradient of exactly 1 moves no data)
        if dH is not None or dW is not None:
            scale_grads(dH, dW, grad_loss)
        return dH, dW, None, None, None, None, None


def linear_cross_entropy(h, W, targets, weights=None, chunk_rows: int = 256,
                         ignore_index: int = IGNORE_INDEX, transform=None, recompute: bool = True):
    """Differentiable masked (weighted) mean NLL of softmax(f(h W^T)); returns (loss, logp, n_valid).

    recompute=False computes the gradients in the forward call without the
    logits recompute (faster when chunk_rows >= 2,048; dH and dW are held
    from the forward to the backward)."""
    if not recompute:
        return LinearCrossEntropyOneCall.apply(h, W, targets, weights, chunk_rows, ignore_index,
                                               transform)
    return LinearCrossEntropy.apply(h, W, targets, weights, chunk_rows, ignore_index, transform)


class LinearCrossEntropyLoss(torch.nn.Module):
    """Module form of linear_cross_entropy: forward(h, W, targets, weights=None)
    returns the masked (weighted) mean NLL of the LM head."""

    def __init__(self, chunk_rows: int = 256, ignore_index: int = IGNORE_INDEX, transform=None,
                 recompute: bool = True):
        super().__init__()
        self.chunk_rows, self.ignore_index = chunk_rows, ignore_index
        self.transform, self.recompute = transform, recompute

    def forward(self, h, W, targets, weights=None):
        loss, _, _ = linear_cross_entropy(h, W, targets, weights, self.chunk_rows, self.ignore_index,
                                          self.transform, self.recompute)
        return loss


class SelectiveLogSoftmax(torch.autograd.Function):
    """Per-token log-probabilities of the targets, log softmax(f(h W^T))[i, t_i]
    (0 on ignored rows), differentiable in h and W for any downstream use: the
    chunked selective log-softmax of the Unsloth GRPO page ("Flattened
    sequence-length chunking").  The backward is the weighted backward with
    w_i = -dL/dlogp_i and g = 1, recomputing the logits."""

    @staticmethod
    def forward(ctx, h, W, targets, chunk_rows, ignore_index, transform=None):
        # the backward reads lse of the non-ignored rows only
        out = forward(h, W, targets, None, chunk_rows, ignore_index, transform=transform, skip_ignored=True)
        ctx.save_for_backward(h, W, targets, out["lse"])
        ctx.chunk_rows, ctx.ignore_index, ctx.transform = chunk_rows, ignore_index, transform
        return out["logp"]

    @staticmethod
    def backward(ctx, grad_logp):
        h, W, targets, lse = ctx.saved_tensors
        w = (-grad_logp).to(torch.float32).contiguous()
        dH, dW = backward(h, W, targets, w, lse, 1.0, ctx.chunk_rows, ctx.ignore_index,
                          need_dH=ctx.needs_input_grad[0], need_dW=ctx.needs_input_grad[1],
                          transform=ctx.transform)
        return dH, dW, None, None, None, None


def selective_log_softmax(h, W, targets, chunk_rows: int = 256, ignore_index: int = IGNORE_INDEX,
                          transform=None, logit_scale_multiply: float = 0.0, logit_scale_divide: float = 0.0,
                          logit_softcapping: float = 0.0, temperature: float = 1.0):
    """logp[N] fp32 of each row's target (0 on ignored rows), differentiable in
    h and W (SelectiveLogSoftmax).  The logit transform is `transform` (a
    dict or LogitTransform), or the four keyword arguments of the Unsloth
    page's chunked selective log-softmax (0 disables the first three)."""
    if transform is None and (logit_scale_multiply or logit_scale_divide or logit_softcapping
                              or temperature != 1.0):
        transform = {"scale_multiply": logit_scale_multiply, "scale_divide": logit_scale_divide,
                     "softcap": logit_softcapping, "temperature": temperature}
    return SelectiveLogSoftmax.apply(h, W, targets, chunk_rows, ignore_index, transform)


def _f32_vec(x, N, name):
    if x is None:
        return None
    if not x.is_cuda or x.dtype != torch.float32 or x.shape != (N,) or not x.is_contiguous():
        raise ValueError(f"{name} must be a contiguous float32 [N] CUDA tensor")
    return x


def grpo_token_loss(logp, advantages, targets=None, old_logp=None, ref_logp=None,
                    eps_low: float = 0.2, eps_high: float = 0.2, beta: float = 0.0,
                    ignore_index: int = IGNORE_INDEX, stream=None):
    """GRPO per-token objective on log-probs (flce_grpo_token_loss):
    dict(token_loss[N], weights[N], loss[], n_valid[]) on device."""
    N = logp.shape[0]
    for x, name in ((logp, "logp"), (advantages, "advantages"), (old_logp, "old_logp"),
                    (ref_logp, "ref_logp")):
        _f32_vec(x, N, name)
    dev = logp.device
    tok = torch.empty(N, dtype=torch.float32, device=dev)
    wts = torch.empty(N, dtype=torch.float32, device=dev)
    loss = torch.empty((), dtype=torch.float32, device=dev)
    n_valid = torch.empty((), dtype=torch.int64, device=dev)
    st = _lib.flce_grpo_token_loss(logp, old_logp, ref_logp, advantages, targets, N, ignore_index,
                                   eps_low, eps_high, beta, tok, wts, loss, n_valid, None, 0, stream)
    _lib.check("flce_grpo_token_loss", st)
    return {"token_loss": tok, "weights": wts, "loss": loss, "n_valid": n_valid}


class GRPOLoss(torch.autograd.Function):
    """GRPO loss of the LM head: forward log-probs, the per-token objective,
    and a backward whose per-token weights are -d(token loss)/d(logp)."""

    @staticmethod
    def forward(ctx, h, W, targets, advantages, old_logp, ref_logp, eps_low, eps_high, beta,
                chunk_rows, ignore_index, transform=None):
        out = forward(h, W, targets, None, chunk_rows, ignore_index, transform=transform,
                      skip_ignored=True)
        tok = grpo_token_loss(out["logp"], advantages, targets, old_logp, ref_logp, eps_low, eps_high,
                              beta, ignore_index)
        ctx.save_for_backward(h, W, targets, out["lse"], tok["weights"], tok["n_valid"])
        ctx.chunk_rows = chunk_rows
        ctx.ignore_index = ignore_index
        ctx.transform = transform
        ctx.mark_non_differentiable(out["logp"])
        return tok["loss"], out["logp"]

    @staticmethod
    def backward(ctx, grad_loss, grad_logp):
        h, W, targets, lse, weights, n_valid = ctx.saved_tensors
        dH, dW = backward(h, W, targets, weights, lse, 1.0, ctx.chunk_rows, ctx.ignore_index,
                          need_dH=ctx.needs_input_grad[0], need_dW=ctx.needs_input_grad[1],
                          transform=ctx.transform, scale=grad_loss, count=n_valid)
        return dH, dW, None, None, None, None, None, None, None, None, None, None


class GRPOLossOneCall(torch.autograd.Function):
    """The GRPO loss with its gradients computed in the forward call
    (flce_grpo_forward_backward, no logits recompute); the backward only
    scales them by the incoming gradient of the loss."""

    @staticmethod
    def forward(ctx, h, W, targets, advantages, old_logp, ref_logp, eps_low, eps_high, beta, chunk_rows,
                ignore_index, transform=None):
        _check(h, W, targets, None)
        N, H = h.shape
        V = W.shape[0]
        for x, name in ((advantages, "advantages"), (old_logp, "old_logp"), (ref_logp, "ref_logp")):
            _f32_vec(x, N, name)
        dev = h.device
        logp = torch.empty(N, dtype=torch.float32, device=dev)
        loss = torch.empty((), dtype=torch.float32, device=dev)
        n_valid = torch.empty((), dtype=torch.int64, device=dev)
        need_dW = ctx.needs_input_grad[1]
        dH = torch.empty_like(h) if (ctx.needs_input_grad[0] or not need_dW) else None
        dW = torch.empty((V, H), dtype=torch.float32, device=dev) if need_dW else None
        st = _lib.flce_grpo_forward_backward(h, W, targets, advantages, old_logp, ref_logp, eps_low, eps_high,
                                             beta, N, H, V, chunk_rows, ignore_index, transform, 1.0, logp,
                                             None, loss, n_valid, dH, dW)
        _lib.check("flce_grpo_forward_backward", st)
        ctx.grads = (dH if ctx.needs_input_grad[0] else None, dW)
        ctx.mark_non_differentiable(logp)
        return loss, logp

    @staticmethod
    def backward(ctx, grad_loss, grad_logp):
        dH, dW = ctx.grads
        ctx.grads = None
        if dH is not None or dW is not None:  # scaled on the device, no host synchronisation
            scale_grads(dH, dW, grad_loss)
        return dH, dW, None, None, None, None, None, None, None, None, None, None


def grpo_loss(h, W, targets, advantages, old_logp=None, ref_logp=None, eps_low: float = 0.2,
              eps_high: float = 0.2, beta: float = 0.0, chunk_rows: int = 256,
              ignore_index: int = IGNORE_INDEX, transform=None, recompute: bool = True):
    """Differentiable GRPO loss of softmax(f(h W^T)) on the target tokens;
    returns (loss, logp).  advantages, old_logp, ref_logp: float32 [N].
    recompute=False computes the gradients in the forward call without the
    logits recompute (flce_grpo_forward_backward; faster when chunk_rows >=
    2,048)."""
    if not recompute:
        return GRPOLossOneCall.apply(h, W, targets, advantages, old_logp, ref_logp, eps_low, eps_high, beta,
                                     chunk_rows, ignore_index, transform)
    return GRPOLoss.apply(h, W, targets, advantages, old_logp, ref_logp, eps_low, eps_high, beta,
                          chunk_rows, ignore_index, transform)


def kd_forward(h_s, W_s, h_t, W_t, targets=None, weights=None, chunk_rows: int = 256,
               ignore_index: int = IGNORE_INDEX, transform=None,
               workspace: torch.Tensor | None = None, stream=None, skip_ignored: bool = False):
    """Distillation forward: dict(kl[N], lse_s[N], lse_t[N], loss[], n_valid[]) on device.
    skip_ignored: both heads skip the ignored rows (their lse become NaN)."""
    for x in (h_s, W_s, h_t, W_t):
        if not x.is_cuda or x.dtype != torch.bfloat16 or not x.is_contiguous() or x.dim() != 2:
            raise ValueError("h_s, W_s, h_t, W_t must be contiguous 2-D bfloat16 CUDA tensors")
    N, H_s = h_s.shape
    H_t = h_t.shape[1]
    V = W_s.shape[0]
    if W_s.shape != (V, H_s) or W_t.shape != (V, H_t) or h_t.shape[0] != N:
        raise ValueError("expected h_s[N,H_s], W_s[V,H_s], h_t[N,H_t], W_t[V,H_t]")
    dev = h_s.device
    kl = torch.empty(N, dtype=torch.float32, device=dev)
    lse_s = torch.empty(N, dtype=torch.float32, device=dev)
    lse_t = torch.empty(N, dtype=torch.float32, device=dev)
    loss = torch.empty((), dtype=torch.float32, device=dev)
    n_valid = torch.empty((), dtype=torch.int64, device=dev)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    flags = _lib.FORWARD_SKIP_IGNORED if skip_ignored else 0
    st = _lib.flce_kd_forward_ex2(h_s, W_s, H_s, h_t, W_t, H_t, targets, weights, N, V, chunk_rows,
                                  ignore_index, transform, flags, kl, lse_s, lse_t, loss, n_valid, workspace,
                                  ws_bytes, stream)
    _lib.check("flce_kd_forward_ex2", st)
    return {"kl": kl, "lse_s": lse_s, "lse_t": lse_t, "loss": loss, "n_valid": n_valid}


def _check_heads(h_s, W_s, h_t, W_t):
    for x in (h_s, W_s, h_t, W_t):
        if not x.is_cuda or x.dtype != torch.bfloat16 or not x.is_contiguous() or x.dim() != 2:
            raise ValueError("h_s, W_s, h_t, W_t must be contiguous 2-D bfloat16 CUDA tensors")
    N, H_s = h_s.shape
    V = W_s.shape[0]
    if W_s.shape != (V, H_s) or W_t.shape != (V, h_t.shape[1]) or h_t.shape[0] != N:
        raise ValueError("expected h_s[N,H_s], W_s[V,H_s], h_t[N,H_t], W_t[V,H_t]")
    return N, H_s, h_t.shape[1], V


def jsd_forward(h_s, W_s, h_t, W_t, beta: float = 0.5, targets=None, weights=None,
                chunk_rows: int = 256, ignore_index: int = IGNORE_INDEX, transform=None,
                workspace: torch.Tensor | None = None, stream=None, skip_ignored: bool = False):
    """Jensen-Shannon distillation forward:
    dict(jsd[N], lse_s[N], lse_t[N], kl_sm[N], loss[], n_valid[]) on device.
    skip_ignored: both heads skip the ignored rows (their lse and kl_sm
    become NaN)."""
    N, H_s, H_t, V = _check_heads(h_s, W_s, h_t, W_t)
    dev = h_s.device
    jsd = torch.empty(N, dtype=torch.float32, device=dev)
    lse_s = torch.empty(N, dtype=torch.float32, device=dev)
    lse_t = torch.empty(N, dtype=torch.float32, device=dev)
    kl_sm = torch.empty(N, dtype=torch.float32, device=dev)
    loss = torch.empty((), dtype=torch.float32, device=dev)
    n_valid = torch.empty((), dtype=torch.int64, device=dev)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    flags = _lib.FORWARD_SKIP_IGNORED if skip_ignored else 0
    st = _lib.flce_jsd_forward_ex2(h_s, W_s, H_s, h_t, W_t, H_t, targets, weights, N, V, chunk_rows,
                                   ignore_index, beta, transform, flags, jsd, lse_s, lse_t, kl_sm, loss, n_valid,
                                   workspace, ws_bytes, stream)
    _lib.check("flce_jsd_forward_ex2", st)
    return {"jsd": jsd, "lse_s": lse_s, "lse_t": lse_t, "kl_sm": kl_sm, "loss": loss,
            "n_valid": n_valid}


def jsd_backward(h_s, W_s, h_t, W_t, lse_s, lse_t, kl_sm, grad_scale: float, beta: float = 0.5,
                 targets=None, weights=None, chunk_rows: int = 256,
                 ignore_index: int = IGNORE_INDEX, transform=None, need_dH: bool = True,
                 need_dW: bool = True, workspace: torch.Tensor | None = None, stream=None,
                 scale=None, count=None):
    """Jensen-Shannon distillation backward: (dH_s bf16 or None, dW_s f32 or None).
    scale / count: device-side factors of grad_scale, as in backward()."""
    N, H_s, H_t, V = _check_heads(h_s, W_s, h_t, W_t)
    dH = torch.empty_like(h_s) if need_dH else None
    dW = torch.empty((V, H_s), dtype=torch.float32, device=h_s.device) if need_dW else None
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    scale = _device_scalar(scale, torch.float32, h_s.device)
    count = _device_scalar(count, torch.int64, h_s.device)
    st = _lib.flce_jsd_backward_ex2(h_s, W_s, H_s, h_t, W_t, H_t, targets, weights, lse_s, lse_t, kl_sm,
                                    beta, grad_scale, scale, count, dH, dW, N, V, chunk_rows, ignore_index,
                                    transform, workspace, ws_bytes, stream)
    _lib.check("flce_jsd_backward_ex2", st)
    return dH, dW


def kd_backward(h_s, W_s, h_t, W_t, lse_s, lse_t, grad_scale: float, targets=None, weights=None,
                chunk_rows: int = 256, ignore_index: int = IGNORE_INDEX, transform=None,
                need_dH: bool = True, need_dW: bool = True, workspace: torch.Tensor | None = None,
                stream=None, scale=None, count=None):
    """Distillation backward: (dH_s bf16 or None, dW_s f32 or None).
    scale / count: device-side factors of grad_scale, as in backward()."""
    N, H_s = h_s.shape
    H_t = h_t.shape[1]
    V = W_s.shape[0]
    dH = torch.empty_like(h_s) if need_dH else None
    dW = torch.empty((V, H_s), dtype=torch.float32, device=h_s.device) if need_dW else None
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    scale = _device_scalar(scale, torch.float32, h_s.device)
    count = _device_scalar(count, torch.int64, h_s.device)
    st = _lib.flce_kd_backward_ex2(h_s, W_s, H_s, h_t, W_t, H_t, targets, weights, lse_s, lse_t,
                                   grad_scale, scale, count, dH, dW, N, V, chunk_rows, ignore_index,
                                   transform, workspace, ws_bytes, stream)
    _lib.check("flce_kd_backward_ex2", st)
    return dH, dW


class DistillLoss(torch.autograd.Function):
    """Distillation loss of a student head against a frozen teacher head:
    KL(p_teacher || p_student) (beta None) or the generalised Jensen-Shannon
    divergence with mixture weight beta, masked by ignored targets (all rows
    when targets is None), weighted and averaged over the counted rows.  The
    gradients go to h_s and W_s; the backward recomputes both heads' logits."""

    @staticmethod
    def forward(ctx, h_s, W_s, h_t, W_t, targets, weights, beta, chunk_rows, ignore_index, transform=None):
        # the backward reads lse (and kl_sm) of the non-ignored rows only
        if beta is None:
            out = kd_forward(h_s, W_s, h_t, W_t, targets, weights, chunk_rows, ignore_index, transform,
                             skip_ignored=True)
            kl_sm = torch.empty(0, device=h_s.device)
        else:
            out = jsd_forward(h_s, W_s, h_t, W_t, beta, targets, weights, chunk_rows, ignore_index,
                              transform, skip_ignored=True)
            kl_sm = out["kl_sm"]
        empty = torch.empty(0, device=h_s.device)
        ctx.save_for_backward(h_s, W_s, h_t, W_t, targets if targets is not None else empty,
                              weights if weights is not None else empty, out["lse_s"], out["lse_t"], kl_sm,
                              out["n_valid"])
        ctx.has_targets, ctx.has_weights = targets is not None, weights is not None
        ctx.beta, ctx.chunk_rows, ctx.ignore_index, ctx.transform = beta, chunk_rows, ignore_index, transform
        return out["loss"]

    @staticmethod
    def backward(ctx, grad_loss):
        h_s, W_s, h_t, W_t, targets, weights, lse_s, lse_t, kl_sm, n_valid = ctx.saved_tensors
        targets = targets if ctx.has_targets else None
        weights = weights if ctx.has_weights else None
        # grad_loss / n_valid is applied on the device: no host synchronisation
        need = dict(need_dH=ctx.needs_input_grad[0], need_dW=ctx.needs_input_grad[1],
                    scale=grad_loss, count=n_valid)
        if ctx.beta is None:
            dH, dW = kd_backward(h_s, W_s, h_t, W_t, lse_s, lse_t, 1.0, targets, weights, ctx.chunk_rows,
                                 ctx.ignore_index, ctx.transform, **need)
        else:
            dH, dW = jsd_backward(h_s, W_s, h_t, W_t, lse_s, lse_t, kl_sm, 1.0, ctx.beta, targets, weights,
                                  ctx.chunk_rows, ctx.ignore_index, ctx.transform, **need)
        return dH, dW, None, None, None, None, None, None, None, None


def distill_loss(h_s, W_s, h_t, W_t, targets=None, weights=None, beta: float | None = None,
                 chunk_rows: int = 256, ignore_index: int = IGNORE_INDEX, transform=None):
    """Autograd distillation loss (DistillLoss): KL(p_teacher || p_student)
    with beta None, else the Jensen-Shannon divergence with mixture weight
    beta in (0, 1).  Returns the scalar loss; h_s and W_s receive gradients."""
    return DistillLoss.apply(h_s, W_s, h_t, W_t, targets, weights, beta, chunk_rows, ignore_index, transform)

