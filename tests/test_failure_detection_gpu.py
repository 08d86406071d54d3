"""Failure detection without a GPU fault: a bounded wait that nothing ever
satisfies gives up, the kernel returns, the host reads FLCE_ERR_TIMEOUT from
the device error word, and the context keeps computing correct results."""
import numpy as np
import pytest

from chunked_lm_head_gb300 import _lib
from chunked_lm_head_gb300 import workloads as WL
from oracle import flce_oracle as O

from gpu_util import assert_logp_close, np64, run_forward, upload

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_context_survives():
    import torch
    lib = _lib.load()
    assert _lib.flce_device_status() == 0
    st = lib.flce_selftest_wait_timeout(20_000_000, torch.cuda.current_stream().cuda_stream)
    assert st == 0  # the wait gave up and the kernel returned
    assert _lib.flce_device_status() == 6  # FLCE_ERR_TIMEOUT, then cleared
    assert _lib.flce_device_status() == 0
    wl = WL.custom("after_timeout", 200, 64, 900, 64, seed=501)
    inp = WL.make_inputs(wl)
    h, W, t, w = upload(inp)
    logp, lse, loss, nv = run_forward(h, W, t, w, 64)
    ref = O.forward(inp.h, inp.W, inp.targets)
    assert nv == ref.n_valid
    assert_logp_close(np64(logp), ref.logp)


def test_selftest_rejects_bad_limits():
    lib = _lib.load()
    assert lib.flce_selftest_wait_timeout(0, None) == 1
    assert lib.flce_selftest_wait_timeout(10**12, None) == 1
