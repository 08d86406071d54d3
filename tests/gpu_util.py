"""Helpers shared by the GPU tests: upload seeded inputs, run libflce through
its C ABI, and compare with the oracle under the stated tolerances."""
from __future__ import annotations

import importlib.util
import os

import numpy as np
import torch

from chunked_lm_head_gb300 import _lib

# Tolerances of the parity bar (per-token log-prob absolute + relative; mean
# loss relative; gradients relative Frobenius; ignored-token count exact).
LOGP_ATOL, LOGP_RTOL = 5e-3, 1e-3
LOSS_RTOL = 1e-4
GRAD_RTOL = 1e-2


def to_dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def upload(inp):
    h = to_dev_bf16(inp.h)
    W = to_dev_bf16(inp.W)
    t = torch.from_numpy(np.ascontiguousarray(inp.targets)).cuda()
    w = None if inp.weights is None else torch.from_numpy(np.ascontiguousarray(inp.weights)).cuda()
    return h, W, t, w


def run_forward(h, W, t, w, chunk_rows, ignore_index=-100, workspace=None, transform=None):
    N, H = h.shape
    V = W.shape[0]
    logp = torch.full((N,), float("nan"), dtype=torch.float32, device="cuda")
    lse = torch.full((N,), float("nan"), dtype=torch.float32, device="cuda")
    loss = torch.full((1,), float("nan"), dtype=torch.float32, device="cuda")
    nv = torch.full((1,), -1, dtype=torch.int64, device="cuda")
    ws_bytes = 0 if workspace is None else workspace.numel()
    if transform is None:
        st = _lib.flce_forward(h, W, t, w, N, H, V, chunk_rows, ignore_index, logp, lse, loss, nv,
                               workspace, ws_bytes)
    else:
        st = _lib.flce_forward_ex(h, W, t, w, N, H, V, chunk_rows, ignore_index, transform, logp, lse,
                                  loss, nv, workspace, ws_bytes)
    assert st == 0, _lib.STATUS_NAMES.get(st)
    assert _lib.flce_device_status() == 0
    return logp, lse, float(loss.item()), int(nv.item())


def run_backward(h, W, t, w, lse, g, chunk_rows, ignore_index=-100, need_dH=True, need_dW=True,
                 workspace=None, transform=None):
    N, H = h.shape
    V = W.shape[0]
    dH = torch.full((N, H), float("nan"), dtype=torch.bfloat16, device="cuda") if need_dH else None
    dW = torch.full((V, H), float("nan"), dtype=torch.float32, device="cuda") if need_dW else None
    ws_bytes = 0 if workspace is None else workspace.numel()
    if transform is None:
        st = _lib.flce_backward(h, W, t, w, lse, g, dH, dW, N, H, V, chunk_rows, ignore_index,
                                workspace, ws_bytes)
    else:
        st = _lib.flce_backward_ex(h, W, t, w, lse, g, dH, dW, N, H, V, chunk_rows, ignore_index,
                                   transform, workspace, ws_bytes)
    assert st == 0, _lib.STATUS_NAMES.get(st)
    assert _lib.flce_device_status() == 0
    return dH, dW


def np64(x: torch.Tensor) -> np.ndarray:
    return x.detach().float().cpu().numpy().astype(np.float64)


def assert_logp_close(got: np.ndarray, ref: np.ndarray, what: str = "logp"):
    err = np.abs(got - ref)
    bound = LOGP_ATOL + LOGP_RTOL * np.abs(ref)
    bad = ~(err <= bound)
    assert not bad.any(), (f"{what}: {int(bad.sum())}/{bad.size} outside tolerance; "
                           f"worst |d|={float(np.nanmax(err)):.3e} at {int(np.nanargmax(err))}")


def rel_fro(got: np.ndarray, ref: np.ndarray) -> float:
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(got - ref) / (den if den > 0 else 1.0))


def assert_grad_close(got: np.ndarray, ref: np.ndarray, what: str):
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    e = rel_fro(got, ref)
    assert e <= GRAD_RTOL, f"{what}: relative Frobenius error {e:.3e}"


def _golden_module():
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                        "make_full_forward_golden.py")
    spec = importlib.util.spec_from_file_location("flce_full_forward_golden", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def load_golden(name: str) -> dict:
    """The oracle's stored full forward of a workload (tests/golden/)."""
    return _golden_module().load(name)


def input_digest(inp) -> str:
    """SHA-256 of a workload's generated inputs, as the golden files record it."""
    return _golden_module().input_digest(inp)
