"""Data-parallel token split of the chunked LM-head loss (one process per GPU).

Each rank holds a slice of the tokens (rows of h, their targets and weights)
and a full copy of the lm_head weight W.  The pages describe the chunked loss
on one GPU; across ranks this module takes the plain data-parallel reading of
the mean NLL over every rank's tokens:

    loss  = -sum_ranks sum_i m_i w_i logp_i / sum_ranks n_valid
    D_i   = (softmax_i - onehot_i) m_i w_i g / n_valid_global      (each rank, its rows)
    dH    = D W                                                     (rows stay on their rank)
    dW    = sum_ranks D_r^T h_r                                     (one all-reduce of [V, H] fp32)

So the ranks exchange, besides dW, two scalars before the loss and the
gradient scale: the valid-token count (int64, exact) and the loss numerator
(fp64).  The count stays on the device and reaches the backward kernels as a
device scalar (flce_backward_ex2's count), so no rank synchronises its host.

The per-rank compute is a ``LocalStep``: by default libflce through
``chunked_lm_head_gb300.api`` (``LibflceStep``).  Collectives go through
torch.distributed on the default group (or ``group``); without an initialised
process group the step is the single-rank step.
"""
from __future__ import annotations

import torch
import torch.distributed as dist

from . import api


class LibflceStep:
    """The per-rank forward and backward of the step, in libflce's kernels."""

    def __init__(self, chunk_rows: int = 4096, ignore_index: int = api.IGNORE_INDEX, transform=None):
        self.chunk_rows = chunk_rows
        self.ignore_index = ignore_index
        self.transform = transform

    def forward(self, h, W, targets, weights):
        """dict(logp, lse, loss, n_valid): loss is this rank's mean NLL."""
        return api.forward(h, W, targets, weights, self.chunk_rows, self.ignore_index,
                           transform=self.transform)

    def backward(self, h, W, targets, weights, lse, grad, count):
        """(dH, dW) with D scaled by grad / max(count, 1), count a device int64 scalar."""
        return api.backward(h, W, targets, weights, lse, grad, self.chunk_rows, self.ignore_index,
                            transform=self.transform, count=count)


def _world(group) -> int:
    return dist.get_world_size(group) if dist.is_available() and dist.is_initialized() else 1


def data_parallel_step(h, W, targets, weights=None, grad: float = 1.0, local=None, group=None):
    """One data-parallel step of the mean NLL over all ranks' tokens.

    Returns dict(loss: the global mean NLL (fp64 scalar tensor), n_valid: the
    global count (int64 scalar tensor), logp: this rank's per-token log-probs,
    dH: this rank's rows, dW: the gradient summed over the ranks), on this
    rank's device.  ``grad`` is the upstream gradient of the loss."""
    local = local if local is not None else LibflceStep()
    f = local.forward(h, W, targets, weights)
    n_local = f["n_valid"].reshape(1).to(torch.int64)
    # the loss numerator of this rank (-sum m w logp = loss * n_valid) and
    # the count, summed over the ranks
    stats = torch.stack([f["loss"].reshape(()).to(torch.float64) * n_local[0].to(torch.float64),
                         n_local[0].to(torch.float64)])
    count = n_local.clone()
    if _world(group) > 1:
        dist.all_reduce(stats, group=group)
        dist.all_reduce(count, group=group)
    loss = stats[0] / torch.clamp(stats[1], min=1.0)
    dH, dW = local.backward(h, W, targets, weights, f["lse"], grad, count)
    if dW is not None and _world(group) > 1:
        dist.all_reduce(dW, group=group)
    return {"loss": loss, "n_valid": count[0], "logp": f["logp"], "dH": dH, "dW": dW}
