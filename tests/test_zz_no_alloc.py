"""The allocation-free forward against the regular forward.

flce_forward_static_scratch is for callers that may not allocate device
memory (work recorded during CUDA graph capture, runtimes that own all device
memory through a fixed pool): it runs the forward on a scratch array the
library keeps in device memory instead of a caller-provided or stream-allocated
workspace.  Here it must reproduce flce_forward, call after call, even though
each call finds the previous call's leftovers in that shared scratch.

This file is named so that pytest collects it last."""
import numpy as np
import pytest
import torch

from chunked_lm_head_gb300 import _lib
from chunked_lm_head_gb300 import workloads as WL

from gpu_util import LOSS_RTOL, assert_logp_close, np64, run_forward, upload

pytestmark = pytest.mark.gpu


def _forward_static(h, W, t, w, chunk_rows):
    N, H = h.shape
    V = W.shape[0]
    logp = torch.full((N,), float("nan"), dtype=torch.float32, device="cuda")
    lse = torch.full((N,), float("nan"), dtype=torch.float32, device="cuda")
    loss = torch.full((1,), float("nan"), dtype=torch.float32, device="cuda")
    nv = torch.full((1,), -1, dtype=torch.int64, device="cuda")
    st = _lib.flce_forward_static_scratch(h, W, t, w, N, H, V, chunk_rows, -100, logp, lse, loss, nv)
    assert st == 0, _lib.STATUS_NAMES.get(st)
    assert _lib.flce_device_status() == 0
    return logp, lse, float(loss.item()), int(nv.item())


def test_static_scratch_forward_matches_regular_forward_on_consecutive_calls():
    cases = [
        WL.custom("noalloc_a", 3000, 512, 20000, 256, w_std=0.04, targets="zipf", ignore_frac=0.05,
                  seed=201),
        WL.custom("noalloc_b", 777, 256, 9000, 256, w_std=0.04, ignore_frac=0.1, seed=202),
    ]
    for k, wl in enumerate(cases):
        inp = WL.make_inputs(wl)
        if k == 1:
            inp.weights = np.random.default_rng(3).standard_normal(wl.N).astype(np.float32)
        h, W, t, w = upload(inp)
        ref_logp, ref_lse, ref_loss, ref_nv = run_forward(h, W, t, w, wl.chunk_rows)
        logp, lse, loss, nv = _forward_static(h, W, t, w, wl.chunk_rows)
        assert nv == ref_nv
        assert_logp_close(np64(logp), np64(ref_logp), "logp")
        assert_logp_close(np64(lse), np64(ref_lse), "lse")
        assert loss == pytest.approx(ref_loss, rel=LOSS_RTOL)


def test_static_scratch_forward_at_the_16k_sft_shape():
    """16,384 x 4,096 x 151,936: the regular plan's split partials (26 MB)
    exceed the 16 MiB array, so this call runs fewer vocabulary splits; the
    results still equal the regular forward's up to fp32 combine rounding."""
    inp = WL.make_inputs("sft_16k")
    h, W, t, w = upload(inp)
    ref_logp, ref_lse, ref_loss, ref_nv = run_forward(h, W, t, w, 4096)
    logp, lse, loss, nv = _forward_static(h, W, t, w, 4096)
    assert nv == ref_nv == 16380
    assert torch.allclose(lse, ref_lse, atol=2e-5, rtol=0)
    assert torch.allclose(logp, ref_logp, atol=2e-5, rtol=0)
    assert loss == pytest.approx(ref_loss, rel=1e-6)


def test_static_scratch_forward_rejects_problems_beyond_its_scratch():
    p = 256  # never dereferenced: the size check comes before any launch
    st = _lib.flce_forward_static_scratch(p, p, p, None, 1 << 21, 64, 151936, 256, -100, p, None,
                                          None, None, 0)
    assert st == 3  # FLCE_ERR_UNSUPPORTED
