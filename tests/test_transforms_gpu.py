"""Logit transforms (multiply, divide, soft-cap, temperature) on the GPU
against the fp64 oracle, plus host-side rejection of invalid transforms."""
import numpy as np
import pytest
import torch

from chunked_lm_head_gb300 import _lib
from chunked_lm_head_gb300 import workloads as WL
from oracle import flce_oracle as O

from gpu_util import (LOSS_RTOL, assert_grad_close, assert_logp_close, np64, run_backward,
                      run_forward, upload)

CASES = {
    "softcap_temp": dict(scale_multiply=0.0, scale_divide=0.0, softcap=30.0, temperature=0.7),
    "tight_softcap": dict(scale_multiply=1.5, scale_divide=0.0, softcap=3.0, temperature=1.0),
    "linear": dict(scale_multiply=2.0, scale_divide=4.0, softcap=0.0, temperature=1.5),
    "temperature": dict(scale_multiply=0.0, scale_divide=0.0, softcap=0.0, temperature=0.25),
}


@pytest.mark.gpu
@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("cg", ["1", "2"])
def test_transform_parity(name, cg, flce_opts):
    flce_opts.set("cta_group", cg)
    tfd = CASES[name]
    tf = O.LogitTransform(**tfd)
    wl = WL.custom(f"tf_{name}", 520, 192, 3100, 256, w_std=0.25, targets="zipf", ignore_frac=0.05,
                   seed=301)
    inp = WL.make_inputs(wl)
    inp.weights = np.random.default_rng(4).uniform(-1, 1, wl.N).astype(np.float32)
    h, W, t, w = upload(inp)
    logp, lse, loss, nv = run_forward(h, W, t, w, 256, transform=tfd)
    ref = O.forward(inp.h, inp.W, inp.targets, inp.weights, tf=tf)
    assert nv == ref.n_valid
    assert_logp_close(np64(logp), ref.logp, "logp")
    assert_logp_close(np64(lse), ref.lse, "lse")
    assert loss == pytest.approx(ref.loss, rel=LOSS_RTOL, abs=1e-6)
    g = 1.0 / nv
    dH, dW = run_backward(h, W, t, w, lse, g, 256, transform=tfd)
    refb = O.backward(inp.h, inp.W, inp.targets, inp.weights, g=g, tf=tf)
    assert_grad_close(np64(dH), refb.dH, "dH")
    assert_grad_close(np64(dW), refb.dW, "dW")


@pytest.mark.gpu
@pytest.mark.parametrize("cg", ["1", "2"])
def test_transform_parity_row_blocks_and_vocabulary_slabs(cg, flce_opts):
    """Soft-cap + temperature through the backward's 512-row blocks x
    1,280-column vocabulary slabs (128-row dlogits budget; last slab 880
    columns, last block 76 rows)."""
    flce_opts.set("cta_group", cg)
    flce_opts.set("bwd_rows", "512")
    flce_opts.set("pipeline", "0")  # the per-slab launches (the pipelined blocks: test_parity_gpu)
    tfd = CASES["softcap_temp"]
    tf = O.LogitTransform(**tfd)
    N, H, V = 1100, 192, 6000
    plan = _lib.flce_backward_plan(N, H, V, 128)
    assert (plan["row_blocks"], plan["vocab_slabs"], plan["vocab_per_slab"]) == (3, 5, 1280)
    wl = WL.custom("tf_slabs", N, H, V, 128, w_std=0.25, targets="zipf", ignore_frac=0.05, seed=303)
    inp = WL.make_inputs(wl)
    h, W, t, w = upload(inp)
    logp, lse, loss, nv = run_forward(h, W, t, w, 128, transform=tfd)
    g = 1.0 / nv
    dH, dW = run_backward(h, W, t, w, lse, g, 128, transform=tfd)
    refb = O.backward(inp.h, inp.W, inp.targets, None, g=g, tf=tf)
    assert_grad_close(np64(dH), refb.dH, "dH")
    assert_grad_close(np64(dW), refb.dW, "dW")


@pytest.mark.gpu
def test_identity_transform_is_bitwise_the_plain_path():
    wl = WL.custom("tf_id", 300, 128, 1500, 128, seed=302)
    inp = WL.make_inputs(wl)
    h, W, t, w = upload(inp)
    a = run_forward(h, W, t, w, 128)
    b = run_forward(h, W, t, w, 128, transform={})
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1]) and a[2] == b[2]


def test_invalid_transforms_rejected_on_host():
    lib = _lib.load()
    p = 256  # never dereferenced: the transform check comes before any launch
    for bad in (dict(temperature=0.0), dict(temperature=-1.0), dict(softcap=-2.0),
                dict(scale_multiply=-1.0), dict(scale_divide=float("inf")),
                dict(temperature=float("nan"))):
        st = _lib.flce_forward_ex(p, p, p, None, 8, 64, 100, 16, -100, bad, p, None, None, None,
                                  None, 0, 0)
        assert st == 1, bad
        st = _lib.flce_backward_ex(p, p, p, None, p, 1.0, p, p, 8, 64, 100, 16, -100, bad, None, 0, 0)
        assert st == 1, bad
