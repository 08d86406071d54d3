"""ctypes binding of libflce's C ABI (include/flce.h).

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind these calls.  torch tensors are accepted for convenience and
turned into raw device pointers; torch supplies device memory and streams.
There is no fallback: if the library cannot be loaded the call raises.
"""
from __future__ import annotations

import ctypes
import os
import re

from . import build as _build

FLCE_OK = 0
STATUS_NAMES = {
    0: "FLCE_OK", 1: "FLCE_ERR_INVALID_ARG", 2: "FLCE_ERR_BAD_TARGET",
    3: "FLCE_ERR_UNSUPPORTED", 4: "FLCE_ERR_OOM", 5: "FLCE_ERR_CUDA", 6: "FLCE_ERR_TIMEOUT",
}

_c_i64 = ctypes.c_int64
_c_vp = ctypes.c_void_p

# name -> (restype, argtypes); mirrors include/flce.h
SIGNATURES = {
    "flce_forward": (ctypes.c_int, [_c_vp, _c_vp, _c_vp, _c_vp, _c_i64, _c_i64, _c_i64, _c_i64,
                                    _c_i64, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, ctypes.c_size_t, _c_vp]),
    "flce_backward": (ctypes.c_int, [_c_vp, _c_vp, _c_vp, _c_vp, _c_vp, ctypes.c_float, _c_vp, _c_vp,
                                     _c_i64, _c_i64, _c_i64, _c_i64, _c_i64, _c_vp, ctypes.c_size_t,
                                     _c_vp]),
    "flce_forward_ex": (ctypes.c_int, [_c_vp, _c_vp, _c_vp, _c_vp, _c_i64, _c_i64, _c_i64, _c_i64,
                                       _c_i64, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp,
                                       ctypes.c_size_t, _c_vp]),
    "flce_grpo_forward_backward": (ctypes.c_int, [_c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, ctypes.c_float,
                                                  ctypes.c_float, ctypes.c_float, _c_i64, _c_i64, _c_i64,
                                                  _c_i64, _c_i64, _c_vp, ctypes.c_float, _c_vp, _c_vp,
                                                  _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, ctypes.c_size_t,
                                                  _c_vp]),
    "flce_forward_ex2": (ctypes.c_int, [_c_vp, _c_vp, _c_vp, _c_vp, _c_i64, _c_i64, _c_i64, _c_i64,
                                        _c_i64, _c_vp, ctypes.c_uint32, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp,
                                        ctypes.c_size_t, _c_vp]),
    "flce_backward_ex": (ctypes.c_int, [_c_vp, _c_vp, _c_vp, _c_vp, _c_vp, ctypes.c_float, _c_vp,
                                        _c_vp, _c_i64, _c_i64, _c_i64, _c_i64, _c_i64, _c_vp, _c_vp,
                                        ctypes.c_size_t, _c_vp]),
    "flce_kd_forward": (ctypes.c_int, [_c_vp, _c_vp, _c_i64, _c_vp, _c_vp, _c_i64, _c_vp, _c_vp,
                                       _c_i64, _c_i64, _c_i64, _c_i64, _c_vp, _c_vp, _c_vp, _c_vp,
                                       _c_vp, _c_vp, _c_vp, ctypes.c_size_t, _c_vp]),
    "flce_kd_forward_ex2": (ctypes.c_int, [_c_vp, _c_vp, _c_i64, _c_vp, _c_vp, _c_i64, _c_vp, _c_vp,
                                           _c_i64, _c_i64, _c_i64, _c_i64, _c_vp, ctypes.c_uint32, _c_vp,
                                           _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, ctypes.c_size_t, _c_vp]),
    "flce_jsd_forward_ex2": (ctypes.c_int, [_c_vp, _c_vp, _c_i64, _c_vp, _c_vp, _c_i64, _c_vp, _c_vp,
                                            _c_i64, _c_i64, _c_i64, _c_i64, ctypes.c_float, _c_vp,
                                            ctypes.c_uint32, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp,
                                            _c_vp, ctypes.c_size_t, _c_vp]),
    "flce_kd_backward": (ctypes.c_int, [_c_vp, _c_vp, _c_i64, _c_vp, _c_vp, _c_i64, _c_vp, _c_vp,
                                        _c_vp, _c_vp, ctypes.c_float, _c_vp, _c_vp, _c_i64, _c_i64,
                                        _c_i64, _c_i64, _c_vp, _c_vp, ctypes.c_size_t, _c_vp]),
    "flce_kd_workspace_bytes": (ctypes.c_size_t, [_c_i64, _c_i64, _c_i64, _c_i64, _c_i64]),
    "flce_grpo_token_loss": (ctypes.c_int, [_c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_i64, _c_i64,
                                            ctypes.c_float, ctypes.c_float, ctypes.c_float, _c_vp,
                                            _c_vp, _c_vp, _c_vp, _c_vp, ctypes.c_size_t, _c_vp]),
    "flce_grpo_workspace_bytes": (ctypes.c_size_t, [_c_i64]),
    "flce_jsd_forward": (ctypes.c_int, [_c_vp, _c_vp, _c_i64, _c_vp, _c_vp, _c_i64, _c_vp, _c_vp,
                                        _c_i64, _c_i64, _c_i64, _c_i64, ctypes.c_float, _c_vp, _c_vp,
                                        _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, ctypes.c_size_t,
                                        _c_vp]),
    "flce_jsd_backward": (ctypes.c_int, [_c_vp, _c_vp, _c_i64, _c_vp, _c_vp, _c_i64, _c_vp, _c_vp,
                                         _c_vp, _c_vp, _c_vp, ctypes.c_float, ctypes.c_float, _c_vp,
                                         _c_vp, _c_i64, _c_i64, _c_i64, _c_i64, _c_vp, _c_vp,
                                         ctypes.c_size_t, _c_vp]),
    "flce_quantize_e4m3_rows": (ctypes.c_int, [_c_vp, _c_i64, _c_i64, _c_vp, _c_vp, _c_vp]),
    "flce_forward_e4m3": (ctypes.c_int, [_c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_i64, _c_i64,
                                         _c_i64, _c_i64, _c_i64, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp,
                                         _c_vp, ctypes.c_size_t, _c_vp]),
    "flce_forward_static_scratch": (ctypes.c_int, [_c_vp, _c_vp, _c_vp, _c_vp, _c_i64, _c_i64, _c_i64,
                                                   _c_i64, _c_i64, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp]),
    "flce_workspace_bytes": (ctypes.c_size_t, [_c_i64, _c_i64, _c_i64, _c_i64]),
    "flce_forward_backward": (ctypes.c_int, [_c_vp, _c_vp, _c_vp, _c_vp, _c_i64, _c_i64, _c_i64,
                                             _c_i64, _c_i64, _c_vp, ctypes.c_float, _c_vp, _c_vp,
                                             _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, ctypes.c_size_t,
                                             _c_vp]),
    "flce_forward_backward_workspace_bytes": (ctypes.c_size_t, [_c_i64, _c_i64, _c_i64, _c_i64]),
    "flce_backward_plan": (ctypes.c_int, [_c_i64, _c_i64, _c_i64, _c_i64, ctypes.c_int32,
                                          ctypes.c_int32, _c_vp]),
    "flce_backward_ex2": (ctypes.c_int, [_c_vp, _c_vp, _c_vp, _c_vp, _c_vp, ctypes.c_float, _c_vp, _c_vp,
                                         _c_vp, _c_i64, _c_i64, _c_i64, _c_i64, _c_i64, _c_vp, _c_vp,
                                         ctypes.c_size_t, _c_vp]),
    "flce_kd_backward_ex2": (ctypes.c_int, [_c_vp, _c_vp, _c_i64, _c_vp, _c_vp, _c_i64, _c_vp, _c_vp,
                                            _c_vp, _c_vp, ctypes.c_float, _c_vp, _c_vp, _c_vp, _c_i64,
                                            _c_i64, _c_i64, _c_i64, _c_vp, _c_vp, ctypes.c_size_t, _c_vp]),
    "flce_jsd_backward_ex2": (ctypes.c_int, [_c_vp, _c_vp, _c_i64, _c_vp, _c_vp, _c_i64, _c_vp, _c_vp,
                                             _c_vp, _c_vp, _c_vp, ctypes.c_float, ctypes.c_float, _c_vp,
                                             _c_vp, _c_vp, _c_i64, _c_i64, _c_i64, _c_i64, _c_vp, _c_vp,
                                             ctypes.c_size_t, _c_vp]),
    "flce_scale_grads": (ctypes.c_int, [_c_vp, _c_i64, _c_vp, _c_i64, _c_vp, _c_vp]),
    "flce_set_option": (ctypes.c_int, [ctypes.c_int, _c_i64]),
    "flce_get_option": (ctypes.c_int, [ctypes.c_int, ctypes.POINTER(ctypes.c_int64)]),
    "flce_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "flce_device_status": (ctypes.c_int, [_c_vp]),
    "flce_selftest_wait_timeout": (ctypes.c_int, [_c_i64, _c_vp]),
    "flce_profile_enable": (ctypes.c_int, [ctypes.c_int]),
    "flce_profile_num_kinds": (ctypes.c_int, []),
    "flce_profile_kind_name": (ctypes.c_char_p, [ctypes.c_int]),
    "flce_profile_read": (ctypes.c_int, [ctypes.c_int, ctypes.POINTER(ctypes.c_double),
                                         ctypes.POINTER(ctypes.c_int64)]),
}

class LogitTransform(ctypes.Structure):
    """flce_logit_transform: multiply, divide, soft-cap, temperature (0/0/0/1 = identity)."""

    _fields_ = [("scale_multiply", ctypes.c_float), ("scale_divide", ctypes.c_float),
                ("softcap", ctypes.c_float), ("temperature", ctypes.c_float)]


class DeviceScale(ctypes.Structure):
    """flce_device_scale: a device fp32 scale and a device int64 count (each may be NULL)."""

    _fields_ = [("scale", ctypes.c_void_p), ("count", ctypes.c_void_p)]


def _dscale_ptr(scale, count):
    """(pointer to a DeviceScale or None, the struct to keep alive)."""
    if scale is None and count is None:
        return None, None
    d = DeviceScale(_ptr(scale), _ptr(count))
    return ctypes.addressof(d), d


def make_transform(tf) -> "LogitTransform | None":
    """None, a LogitTransform, or a dict with any of its four field names."""
    if tf is None or isinstance(tf, LogitTransform):
        return tf
    d = {"scale_multiply": 0.0, "scale_divide": 0.0, "softcap": 0.0, "temperature": 1.0}
    d.update(tf)
    return LogitTransform(**d)


_LIB = None


class FlceError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: {STATUS_NAMES.get(status, status)}")
        self.status = status


def header_symbols() -> list[str]:
    """Function names declared in include/flce.h."""
    src = open(os.path.join(_build.INCLUDE, "flce.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return re.findall(r"\b(flce_[a-z0-9_]+)\s*\(", src)


def load(path: str | None = None, build_if_missing: bool = True) -> ctypes.CDLL:
    """Load libflce.so (building it in-tree first when it is absent).

    FLCE_LIB_PATH in the environment selects another build of the library."""
    global _LIB
    if _LIB is not None and path is None:
        return _LIB
    p = path or os.environ.get("FLCE_LIB_PATH") or _build.LIB_PATH
    if not os.path.exists(p):
        if not build_if_missing:
            raise FileNotFoundError(p)
        _build.build()
    lib = ctypes.CDLL(p)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path is None:
        _LIB = lib
    return lib


def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream_handle(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def check(fn: str, status: int) -> None:
    if status != FLCE_OK:
        raise FlceError(fn, status)


def flce_forward(h, W, targets, weights, N, H, V, chunk_rows, ignore_index, out_logp, out_lse,
                 out_loss, out_n_valid, workspace=None, workspace_bytes=0, stream=None) -> int:
    """Raw C call; tensors or integer device pointers.  Returns the status."""
    lib = load()
    return lib.flce_forward(_ptr(h), _ptr(W), _ptr(targets), _ptr(weights), N, H, V, chunk_rows,
                            ignore_index, _ptr(out_logp), _ptr(out_lse), _ptr(out_loss),
                            _ptr(out_n_valid), _ptr(workspace), workspace_bytes,
                            _stream_handle(stream))


def flce_backward(h, W, targets, weights, lse, grad_scale, dH, dW, N, H, V, chunk_rows,
                  ignore_index, workspace=None, workspace_bytes=0, stream=None) -> int:
    """Raw C call; tensors or integer device pointers.  Returns the status."""
    lib = load()
    return lib.flce_backward(_ptr(h), _ptr(W), _ptr(targets), _ptr(weights), _ptr(lse),
                             float(grad_scale), _ptr(dH), _ptr(dW), N, H, V, chunk_rows,
                             ignore_index, _ptr(workspace), workspace_bytes, _stream_handle(stream))


def _tf_ptr(tf):
    t = make_transform(tf)
    return None if t is None else ctypes.addressof(t), t


def flce_forward_ex(h, W, targets, weights, N, H, V, chunk_rows, ignore_index, transform, out_logp,
                    out_lse, out_loss, out_n_valid, workspace=None, workspace_bytes=0,
                    stream=None) -> int:
    """Raw C call with a logit transform (None / dict / LogitTransform)."""
    lib = load()
    tp, keep = _tf_ptr(transform)
    return lib.flce_forward_ex(_ptr(h), _ptr(W), _ptr(targets), _ptr(weights), N, H, V, chunk_rows,
                               ignore_index, tp, _ptr(out_logp), _ptr(out_lse), _ptr(out_loss),
                               _ptr(out_n_valid), _ptr(workspace), workspace_bytes,
                               _stream_handle(stream))


FORWARD_SKIP_IGNORED = 1


def flce_grpo_forward_backward(h, W, targets, advantages, old_logp, ref_logp, eps_low, eps_high, beta, N, H,
                               V, chunk_rows, ignore_index, transform, grad_scale, out_logp, out_token_loss,
                               out_loss, out_n_valid, dH, dW, workspace=None, workspace_bytes=0,
                               stream=None) -> int:
    """Raw C call of the GRPO loss and gradients in one call."""
    lib = load()
    tp, keep = _tf_ptr(transform)
    return lib.flce_grpo_forward_backward(_ptr(h), _ptr(W), _ptr(targets), _ptr(advantages), _ptr(old_logp),
                                          _ptr(ref_logp), float(eps_low), float(eps_high), float(beta), N, H, V,
                                          chunk_rows, ignore_index, tp, float(grad_scale), _ptr(out_logp),
                                          _ptr(out_token_loss), _ptr(out_loss), _ptr(out_n_valid), _ptr(dH),
                                          _ptr(dW), _ptr(workspace), workspace_bytes, _stream_handle(stream))


def flce_forward_ex2(h, W, targets, weights, N, H, V, chunk_rows, ignore_index, transform, flags,
                     out_logp, out_lse, out_loss, out_n_valid, workspace=None, workspace_bytes=0,
                     stream=None) -> int:
    """Raw C call with a logit transform and flags (FORWARD_SKIP_IGNORED)."""
    lib = load()
    tp, keep = _tf_ptr(transform)
    return lib.flce_forward_ex2(_ptr(h), _ptr(W), _ptr(targets), _ptr(weights), N, H, V, chunk_rows,
                                ignore_index, tp, int(flags), _ptr(out_logp), _ptr(out_lse),
                                _ptr(out_loss), _ptr(out_n_valid), _ptr(workspace), workspace_bytes,
                                _stream_handle(stream))


def flce_backward_ex(h, W, targets, weights, lse, grad_scale, dH, dW, N, H, V, chunk_rows,
                     ignore_index, transform, workspace=None, workspace_bytes=0, stream=None) -> int:
    """Raw C call with a logit transform (None / dict / LogitTransform)."""
    lib = load()
    tp, keep = _tf_ptr(transform)
    return lib.flce_backward_ex(_ptr(h), _ptr(W), _ptr(targets), _ptr(weights), _ptr(lse),
                                float(grad_scale), _ptr(dH), _ptr(dW), N, H, V, chunk_rows,
                                ignore_index, tp, _ptr(workspace), workspace_bytes,
                                _stream_handle(stream))


def flce_backward_ex2(h, W, targets, weights, lse, grad_scale, scale, count, dH, dW, N, H, V,
                      chunk_rows, ignore_index, transform, workspace=None, workspace_bytes=0,
                      stream=None) -> int:
    """Raw C call with a device-side scale (scale: [1] fp32, count: [1] int64; each may be None)."""
    lib = load()
    tp, keep = _tf_ptr(transform)
    dp, keep_d = _dscale_ptr(scale, count)
    return lib.flce_backward_ex2(_ptr(h), _ptr(W), _ptr(targets), _ptr(weights), _ptr(lse),
                                 float(grad_scale), dp, _ptr(dH), _ptr(dW), N, H, V, chunk_rows,
                                 ignore_index, tp, _ptr(workspace), workspace_bytes,
                                 _stream_handle(stream))


def flce_kd_backward_ex2(h_s, W_s, H_s, h_t, W_t, H_t, targets, weights, lse_s, lse_t, grad_scale,
                         scale, count, dH_s, dW_s, N, V, chunk_rows, ignore_index, transform,
                         workspace=None, workspace_bytes=0, stream=None) -> int:
    """Raw C call of the distillation backward with a device-side scale."""
    lib = load()
    tp, keep = _tf_ptr(transform)
    dp, keep_d = _dscale_ptr(scale, count)
    return lib.flce_kd_backward_ex2(_ptr(h_s), _ptr(W_s), H_s, _ptr(h_t), _ptr(W_t), H_t, _ptr(targets),
                                    _ptr(weights), _ptr(lse_s), _ptr(lse_t), float(grad_scale), dp,
                                    _ptr(dH_s), _ptr(dW_s), N, V, chunk_rows, ignore_index, tp,
                                    _ptr(workspace), workspace_bytes, _stream_handle(stream))


def flce_jsd_backward_ex2(h_s, W_s, H_s, h_t, W_t, H_t, targets, weights, lse_s, lse_t, kl_sm, beta,
                          grad_scale, scale, count, dH_s, dW_s, N, V, chunk_rows, ignore_index,
                          transform, workspace=None, workspace_bytes=0, stream=None) -> int:
    """Raw C call of the Jensen-Shannon backward with a device-side scale."""
    lib = load()
    tp, keep = _tf_ptr(transform)
    dp, keep_d = _dscale_ptr(scale, count)
    return lib.flce_jsd_backward_ex2(_ptr(h_s), _ptr(W_s), H_s, _ptr(h_t), _ptr(W_t), H_t, _ptr(targets),
                                     _ptr(weights), _ptr(lse_s), _ptr(lse_t), _ptr(kl_sm), float(beta),
                                     float(grad_scale), dp, _ptr(dH_s), _ptr(dW_s), N, V, chunk_rows,
                                     ignore_index, tp, _ptr(workspace), workspace_bytes,
                                     _stream_handle(stream))


def flce_scale_grads(dH, n_dH, dW, n_dW, scale, stream=None) -> int:
    """Raw C call: dH, dW *= *scale in place (scale a [1] fp32 device tensor)."""
    return load().flce_scale_grads(_ptr(dH), n_dH, _ptr(dW), n_dW, _ptr(scale), _stream_handle(stream))


def flce_kd_forward(h_s, W_s, H_s, h_t, W_t, H_t, targets, weights, N, V, chunk_rows, ignore_index,
                    transform, out_kl, out_lse_s, out_lse_t, out_loss, out_n_valid, workspace=None,
                    workspace_bytes=0, stream=None) -> int:
    """Raw C call of the distillation forward."""
    lib = load()
    tp, keep = _tf_ptr(transform)
    return lib.flce_kd_forward(_ptr(h_s), _ptr(W_s), H_s, _ptr(h_t), _ptr(W_t), H_t, _ptr(targets),
                               _ptr(weights), N, V, chunk_rows, ignore_index, tp, _ptr(out_kl),
                               _ptr(out_lse_s), _ptr(out_lse_t), _ptr(out_loss), _ptr(out_n_valid),
                               _ptr(workspace), workspace_bytes, _stream_handle(stream))


def flce_kd_backward(h_s, W_s, H_s, h_t, W_t, H_t, targets, weights, lse_s, lse_t, grad_scale, dH_s,
                     dW_s, N, V, chunk_rows, ignore_index, transform, workspace=None,
                     workspace_bytes=0, stream=None) -> int:
    """Raw C call of the distillation backward (student gradients)."""
    lib = load()
    tp, keep = _tf_ptr(transform)
    return lib.flce_kd_backward(_ptr(h_s), _ptr(W_s), H_s, _ptr(h_t), _ptr(W_t), H_t, _ptr(targets),
                                _ptr(weights), _ptr(lse_s), _ptr(lse_t), float(grad_scale),
                                _ptr(dH_s), _ptr(dW_s), N, V, chunk_rows, ignore_index, tp,
                                _ptr(workspace), workspace_bytes, _stream_handle(stream))


def flce_kd_forward_ex2(h_s, W_s, H_s, h_t, W_t, H_t, targets, weights, N, V, chunk_rows, ignore_index,
                        transform, flags, out_kl, out_lse_s, out_lse_t, out_loss, out_n_valid, workspace=None,
                        workspace_bytes=0, stream=None) -> int:
    """Raw C call of the distillation forward with flags (FORWARD_SKIP_IGNORED)."""
    lib = load()
    tp, keep = _tf_ptr(transform)
    return lib.flce_kd_forward_ex2(_ptr(h_s), _ptr(W_s), H_s, _ptr(h_t), _ptr(W_t), H_t, _ptr(targets),
                                   _ptr(weights), N, V, chunk_rows, ignore_index, tp, int(flags), _ptr(out_kl),
                                   _ptr(out_lse_s), _ptr(out_lse_t), _ptr(out_loss), _ptr(out_n_valid),
                                   _ptr(workspace), workspace_bytes, _stream_handle(stream))


def flce_jsd_forward_ex2(h_s, W_s, H_s, h_t, W_t, H_t, targets, weights, N, V, chunk_rows, ignore_index,
                         beta, transform, flags, out_jsd, out_lse_s, out_lse_t, out_kl_sm, out_loss,
                         out_n_valid, workspace=None, workspace_bytes=0, stream=None) -> int:
    """Raw C call of the Jensen-Shannon distillation forward with flags."""
    lib = load()
    tp, keep = _tf_ptr(transform)
    return lib.flce_jsd_forward_ex2(_ptr(h_s), _ptr(W_s), H_s, _ptr(h_t), _ptr(W_t), H_t, _ptr(targets),
                                    _ptr(weights), N, V, chunk_rows, ignore_index, float(beta), tp, int(flags),
                                    _ptr(out_jsd), _ptr(out_lse_s), _ptr(out_lse_t), _ptr(out_kl_sm),
                                    _ptr(out_loss), _ptr(out_n_valid), _ptr(workspace), workspace_bytes,
                                    _stream_handle(stream))


def flce_jsd_forward(h_s, W_s, H_s, h_t, W_t, H_t, targets, weights, N, V, chunk_rows, ignore_index,
                     beta, transform, out_jsd, out_lse_s, out_lse_t, out_kl_sm, out_loss,
                     out_n_valid, workspace=None, workspace_bytes=0, stream=None) -> int:
    """Raw C call of the Jensen-Shannon distillation forward."""
    lib = load()
    tp, keep = _tf_ptr(transform)
    return lib.flce_jsd_forward(_ptr(h_s), _ptr(W_s), H_s, _ptr(h_t), _ptr(W_t), H_t, _ptr(targets),
                                _ptr(weights), N, V, chunk_rows, ignore_index, float(beta), tp,
                                _ptr(out_jsd), _ptr(out_lse_s), _ptr(out_lse_t), _ptr(out_kl_sm),
                                _ptr(out_loss), _ptr(out_n_valid), _ptr(workspace), workspace_bytes,
                                _stream_handle(stream))


def flce_jsd_backward(h_s, W_s, H_s, h_t, W_t, H_t, targets, weights, lse_s, lse_t, kl_sm, beta,
                      grad_scale, dH_s, dW_s, N, V, chunk_rows, ignore_index, transform,
                      workspace=None, workspace_bytes=0, stream=None) -> int:
    """Raw C call of the Jensen-Shannon distillation backward (student gradients)."""
    lib = load()
    tp, keep = _tf_ptr(transform)
    return lib.flce_jsd_backward(_ptr(h_s), _ptr(W_s), H_s, _ptr(h_t), _ptr(W_t), H_t, _ptr(targets),
                                 _ptr(weights), _ptr(lse_s), _ptr(lse_t), _ptr(kl_sm), float(beta),
                                 float(grad_scale), _ptr(dH_s), _ptr(dW_s), N, V, chunk_rows,
                                 ignore_index, tp, _ptr(workspace), workspace_bytes,
                                 _stream_handle(stream))


def flce_grpo_token_loss(logp, old_logp, ref_logp, advantages, targets, N, ignore_index, eps_low,
                         eps_high, beta, out_token_loss, out_weights, out_loss, out_n_valid,
                         workspace=None, workspace_bytes=0, stream=None) -> int:
    """Raw C call of the GRPO per-token objective."""
    return load().flce_grpo_token_loss(_ptr(logp), _ptr(old_logp), _ptr(ref_logp), _ptr(advantages),
                                       _ptr(targets), N, ignore_index, float(eps_low), float(eps_high),
                                       float(beta), _ptr(out_token_loss), _ptr(out_weights),
                                       _ptr(out_loss), _ptr(out_n_valid), _ptr(workspace),
                                       workspace_bytes, _stream_handle(stream))


def flce_forward_backward(h, W, targets, weights, N, H, V, chunk_rows, ignore_index, transform,
                          grad_scale, out_logp, out_lse, out_loss, out_n_valid, dH, dW,
                          workspace=None, workspace_bytes=0, stream=None) -> int:
    """Raw C call of the forward + backward without the logits recompute."""
    lib = load()
    tp, keep = _tf_ptr(transform)
    return lib.flce_forward_backward(_ptr(h), _ptr(W), _ptr(targets), _ptr(weights), N, H, V,
                                     chunk_rows, ignore_index, tp, float(grad_scale), _ptr(out_logp),
                                     _ptr(out_lse), _ptr(out_loss), _ptr(out_n_valid), _ptr(dH),
                                     _ptr(dW), _ptr(workspace), workspace_bytes,
                                     _stream_handle(stream))


def flce_quantize_e4m3_rows(x, rows, cols, q, scale, stream=None) -> int:
    """Raw C call: per-row e4m3 quantisation."""
    return load().flce_quantize_e4m3_rows(_ptr(x), rows, cols, _ptr(q), _ptr(scale),
                                          _stream_handle(stream))


def flce_forward_e4m3(h8, h_scale, W8, W_scale, targets, weights, N, H, V, chunk_rows, ignore_index,
                      transform, out_logp, out_lse, out_loss, out_n_valid, workspace=None,
                      workspace_bytes=0, stream=None) -> int:
    """Raw C call of the e4m3 forward."""
    lib = load()
    tp, keep = _tf_ptr(transform)
    return lib.flce_forward_e4m3(_ptr(h8), _ptr(h_scale), _ptr(W8), _ptr(W_scale), _ptr(targets),
                                 _ptr(weights), N, H, V, chunk_rows, ignore_index, tp, _ptr(out_logp),
                                 _ptr(out_lse), _ptr(out_loss), _ptr(out_n_valid), _ptr(workspace),
                                 workspace_bytes, _stream_handle(stream))


def flce_forward_static_scratch(h, W, targets, weights, N, H, V, chunk_rows, ignore_index, out_logp,
                                out_lse, out_loss, out_n_valid, stream=None) -> int:
    """Raw C call of the allocation-free forward (library-owned scratch)."""
    lib = load()
    return lib.flce_forward_static_scratch(_ptr(h), _ptr(W), _ptr(targets), _ptr(weights), N, H, V,
                                           chunk_rows, ignore_index, _ptr(out_logp), _ptr(out_lse),
                                           _ptr(out_loss), _ptr(out_n_valid), _stream_handle(stream))


def flce_workspace_bytes(N, H, V, chunk_rows) -> int:
    return int(load().flce_workspace_bytes(N, H, V, chunk_rows))


def flce_forward_backward_workspace_bytes(N, H, V, chunk_rows) -> int:
    return int(load().flce_forward_backward_workspace_bytes(N, H, V, chunk_rows))


class BackwardPlanInfo(ctypes.Structure):
    """flce_backward_plan_info."""
    _fields_ = [("rows_per_block", ctypes.c_int64), ("vocab_per_slab", ctypes.c_int64),
                ("row_blocks", ctypes.c_int64), ("vocab_slabs", ctypes.c_int64),
                ("dh_splits", ctypes.c_int64), ("dlogits_bytes", ctypes.c_int64),
                ("workspace_bytes", ctypes.c_int64), ("dlogits_buffers", ctypes.c_int64),
                ("dh_wide", ctypes.c_int64)]


def flce_backward_plan(N, H, V, chunk_rows, workers=0, cta_group=0) -> dict:
    """The backward's tiling (row block, vocabulary slab, dH splits, bytes)."""
    info = BackwardPlanInfo()
    st = load().flce_backward_plan(N, H, V, chunk_rows, workers, cta_group, ctypes.addressof(info))
    check("flce_backward_plan", st)
    return {name: int(getattr(info, name)) for name, _ in BackwardPlanInfo._fields_}


# flce_option values (include/flce.h), by lower-case name without the prefix
OPTIONS = {
    "cta_group": 0, "compact": 1, "validate": 2, "pdl": 3, "d_tma": 4, "wide_epilogue": 5,
    "bwd_rows": 6, "fwd_splits": 7, "dh_splits": 8, "dh_group": 9, "fwd_block_rows": 10,
    "skip_min_rows": 11, "fuse_dh_dw": 12,
    "dw_epilogue_warps": 13, "pipeline": 14, "dh_wide": 15, "grid_workers": 16,
}


def flce_set_option(name: str, value: int) -> None:
    """Set a run-time option (e.g. "cta_group", "compact") for later calls."""
    check("flce_set_option", load().flce_set_option(OPTIONS[name], int(value)))


def flce_get_option(name: str) -> int:
    v = ctypes.c_int64(0)
    check("flce_get_option", load().flce_get_option(OPTIONS[name], ctypes.byref(v)))
    return int(v.value)


class options:
    """Context manager: set options for a block, restore the previous values."""

    def __init__(self, **values):
        self.values = values
        self.saved = {}

    def __enter__(self):
        for k, v in self.values.items():
            self.saved[k] = flce_get_option(k)
            flce_set_option(k, v)
        return self

    def __exit__(self, *exc):
        for k, v in self.saved.items():
            flce_set_option(k, v)
        return False


def flce_kd_workspace_bytes(N, H_s, H_t, V, chunk_rows) -> int:
    return int(load().flce_kd_workspace_bytes(N, H_s, H_t, V, chunk_rows))


def flce_status_string(status: int) -> str:
    return load().flce_status_string(status).decode()


def flce_device_status(stream=None) -> int:
    return load().flce_device_status(_stream_handle(stream))


def profile_enable(on: bool) -> None:
    check("flce_profile_enable", load().flce_profile_enable(1 if on else 0))


def profile_read() -> dict:
    """{kernel kind: (total_ms, launches)} accumulated since profile_enable."""
    lib = load()
    out = {}
    for k in range(lib.flce_profile_num_kinds()):
        ms = ctypes.c_double()
        n = ctypes.c_int64()
        check("flce_profile_read", lib.flce_profile_read(k, ctypes.byref(ms), ctypes.byref(n)))
        out[lib.flce_profile_kind_name(k).decode()] = (ms.value, n.value)
    return out
