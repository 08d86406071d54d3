"""Distillation (student head learning a frozen teacher head's distribution)
on the GPU against the fp64 oracle."""
import numpy as np
import pytest
import torch

import chunked_lm_head_gb300 as flce
from chunked_lm_head_gb300 import workloads as WL
from oracle import flce_oracle as O

from gpu_util import LOSS_RTOL, assert_grad_close, assert_logp_close, np64, to_dev_bf16

pytestmark = pytest.mark.gpu


def _heads(N, Hs, Ht, V, seed, w_std=0.05):
    s = WL.custom("kd_s", N, Hs, V, 256, w_std=w_std, seed=seed)
    t = WL.custom("kd_t", N, Ht, V, 256, w_std=w_std * 1.3, seed=seed + 1000)
    return WL.make_inputs(s), WL.make_inputs(t)


CASES = [
    # N, H_s, H_t, V, chunk, transform, masked
    (300, 192, 320, 2100, 128, None, True),
    (520, 256, 128, 3000, 256, {"temperature": 2.0}, False),
    (130, 64, 64, 777, 64, {"softcap": 5.0, "temperature": 1.5}, True),
]


@pytest.mark.parametrize("case", CASES)
@pytest.mark.parametrize("cg", ["1", "2"])
def test_kd_parity(case, cg, flce_opts):
    flce_opts.set("cta_group", cg)
    _kd_check(case)


@pytest.mark.parametrize("cg", ["1", "2"])
def test_kd_parity_row_blocks_and_vocabulary_slabs(cg, flce_opts):
    """Distillation backward over 512-row blocks x 1,280-column vocabulary
    slabs (3 blocks, the last 76 rows; 5 slabs, the last 880 columns) inside a
    128-row dlogits budget."""
    flce_opts.set("cta_group", cg)
    flce_opts.set("bwd_rows", "512")
    flce_opts.set("pipeline", "0")  # the distillation backward's plan: one dlogits buffer
    case = (1100, 256, 384, 6000, 128, {"temperature": 1.3}, True)
    plan = flce._lib.flce_backward_plan(case[0], case[1], case[3], case[4])
    assert (plan["row_blocks"], plan["vocab_slabs"], plan["vocab_per_slab"]) == (3, 5, 1280)
    _kd_check(case)


def _kd_check(case):
    N, Hs, Ht, V, chunk, tfd, masked = case
    si, ti = _heads(N, Hs, Ht, V, seed=601 + N)
    targets = None
    if masked:
        targets = np.random.default_rng(5).integers(0, V, N).astype(np.int64)
        targets[np.random.default_rng(6).permutation(N)[: N // 10]] = WL.IGNORE_INDEX
    weights = np.random.default_rng(7).uniform(0.3, 1.7, N).astype(np.float32)
    tf = None if tfd is None else O.LogitTransform(**tfd)
    hs, Ws, ht, Wt = (to_dev_bf16(x) for x in (si.h, si.W, ti.h, ti.W))
    tg = None if targets is None else torch.from_numpy(targets).cuda()
    w = torch.from_numpy(weights).cuda()
    out = flce.kd_forward(hs, Ws, ht, Wt, tg, w, chunk, transform=tfd)
    ref = O.kd_forward(si.h, si.W, ti.h, ti.W, targets, weights, tf=tf)
    assert int(out["n_valid"]) == ref.n_valid
    assert_logp_close(np64(out["lse_s"]), ref.lse_s, "lse_s")
    assert_logp_close(np64(out["lse_t"]), ref.lse_t, "lse_t")
    assert_logp_close(np64(out["kl"]), ref.kl, "kl")
    assert float(out["loss"]) == pytest.approx(ref.loss, rel=LOSS_RTOL, abs=1e-6)
    g = 1.0 / ref.n_valid
    dH, dW = flce.kd_backward(hs, Ws, ht, Wt, out["lse_s"], out["lse_t"], g, tg, w, chunk,
                              transform=tfd)
    refb = O.kd_backward(si.h, si.W, ti.h, ti.W, targets, weights, g=g, tf=tf)
    assert_grad_close(np64(dH), refb.dH, "dH_s")
    assert_grad_close(np64(dW), refb.dW, "dW_s")
    assert flce._lib.flce_device_status() == 0


def test_kd_of_identical_heads_is_zero():
    si, _ = _heads(200, 128, 128, 1500, seed=650)
    hs, Ws = to_dev_bf16(si.h), to_dev_bf16(si.W)
    out = flce.kd_forward(hs, Ws, hs, Ws, None, None, 128)
    assert np.max(np.abs(np64(out["kl"]))) < 1e-4
    dH, dW = flce.kd_backward(hs, Ws, hs, Ws, out["lse_s"], out["lse_t"], 1.0 / 200)
    assert float(dH.float().abs().max()) < 1e-6 and float(dW.abs().max()) < 1e-6
