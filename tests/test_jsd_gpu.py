"""Jensen-Shannon distillation (student head, frozen teacher head) on the GPU
against the fp64 oracle."""
import numpy as np
import pytest
import torch

import chunked_lm_head_gb300 as flce
from chunked_lm_head_gb300 import workloads as WL
from oracle import flce_oracle as O

from gpu_util import LOSS_RTOL, assert_grad_close, assert_logp_close, np64, to_dev_bf16

pytestmark = pytest.mark.gpu


def _heads(N, Hs, Ht, V, seed, w_std=0.05):
    s = WL.custom("jsd_s", N, Hs, V, 256, w_std=w_std, seed=seed)
    t = WL.custom("jsd_t", N, Ht, V, 256, w_std=w_std * 1.3, seed=seed + 1000)
    return WL.make_inputs(s), WL.make_inputs(t)


CASES = [
    # N, H_s, H_t, V, chunk, beta, transform, masked
    (300, 192, 320, 2100, 128, 0.5, None, True),
    (520, 256, 128, 3000, 256, 0.1, {"temperature": 2.0}, False),
    (130, 64, 64, 777, 64, 0.9, {"softcap": 5.0, "temperature": 1.5}, True),
]


def _jsd_check(case):
    N, Hs, Ht, V, chunk, beta, tfd, masked = case
    si, ti = _heads(N, Hs, Ht, V, seed=701 + N)
    targets = None
    if masked:
        targets = np.random.default_rng(5).integers(0, V, N).astype(np.int64)
        targets[np.random.default_rng(6).permutation(N)[: N // 10]] = WL.IGNORE_INDEX
    weights = np.random.default_rng(7).uniform(0.3, 1.7, N).astype(np.float32)
    tf = None if tfd is None else O.LogitTransform(**tfd)
    hs, Ws, ht, Wt = (to_dev_bf16(x) for x in (si.h, si.W, ti.h, ti.W))
    tg = None if targets is None else torch.from_numpy(targets).cuda()
    w = torch.from_numpy(weights).cuda()
    out = flce.jsd_forward(hs, Ws, ht, Wt, beta, tg, w, chunk, transform=tfd)
    ref = O.jsd_forward(si.h, si.W, ti.h, ti.W, beta, targets, weights, tf=tf)
    assert int(out["n_valid"]) == ref.n_valid
    assert_logp_close(np64(out["lse_s"]), ref.lse_s, "lse_s")
    assert_logp_close(np64(out["lse_t"]), ref.lse_t, "lse_t")
    assert_logp_close(np64(out["jsd"]), ref.jsd, "jsd")
    assert_logp_close(np64(out["kl_sm"]), ref.kl_sm, "kl_sm")
    assert float(out["loss"]) == pytest.approx(ref.loss, rel=LOSS_RTOL, abs=1e-6)
    g = 1.0 / ref.n_valid
    dH, dW = flce.jsd_backward(hs, Ws, ht, Wt, out["lse_s"], out["lse_t"], out["kl_sm"], g, beta, tg, w,
                               chunk, transform=tfd)
    refb = O.jsd_backward(si.h, si.W, ti.h, ti.W, beta, targets, weights, g=g, tf=tf)
    assert_grad_close(np64(dH), refb.dH, "dH_s")
    assert_grad_close(np64(dW), refb.dW, "dW_s")
    assert flce._lib.flce_device_status() == 0


@pytest.mark.parametrize("case", CASES)
@pytest.mark.parametrize("cg", ["1", "2"])
def test_jsd_parity(case, cg, flce_opts):
    flce_opts.set("cta_group", cg)
    _jsd_check(case)


@pytest.mark.parametrize("cg", ["1", "2"])
def test_jsd_parity_row_blocks_and_vocabulary_slabs(cg, flce_opts):
    """The JSD backward over 512-row blocks x 1,280-column vocabulary slabs
    (3 blocks, the last 76 rows; 5 slabs, the last 880 columns) inside a
    128-row dlogits budget."""
    flce_opts.set("cta_group", cg)
    flce_opts.set("bwd_rows", "512")
    flce_opts.set("pipeline", "0")  # the distillation backward's plan: one dlogits buffer
    case = (1100, 256, 384, 6000, 128, 0.3, {"temperature": 1.3}, True)
    plan = flce._lib.flce_backward_plan(case[0], case[1], case[3], case[4])
    assert (plan["row_blocks"], plan["vocab_slabs"], plan["vocab_per_slab"]) == (3, 5, 1280)
    _jsd_check(case)


def test_jsd_of_identical_heads_is_zero_and_symmetric_at_one_half():
    si, ti = _heads(400, 128, 192, 2500, seed=720)
    hs, Ws, ht, Wt = (to_dev_bf16(x) for x in (si.h, si.W, ti.h, ti.W))
    same = flce.jsd_forward(hs, Ws, hs, Ws, 0.4)
    assert float(same["jsd"].abs().max()) <= 1e-5
    dH, dW = flce.jsd_backward(hs, Ws, hs, Ws, same["lse_s"], same["lse_t"], same["kl_sm"], 1.0, 0.4)
    assert float(dH.float().abs().max()) <= 1e-5 and float(dW.abs().max()) <= 1e-4
    # the textbook JSD (beta = 1/2) does not depend on which head is the teacher
    a = flce.jsd_forward(hs, Ws, ht, Wt, 0.5)
    b = flce.jsd_forward(ht, Wt, hs, Ws, 0.5)
    assert torch.allclose(a["jsd"], b["jsd"], atol=2e-5, rtol=1e-4)
    assert float(a["jsd"].min()) > 0 and float(a["jsd"].max()) <= float(np.log(2)) + 1e-6


@pytest.mark.parametrize("beta", [None, 0.4])
@pytest.mark.parametrize("cg", ["1", "2"])
def test_distillation_forward_skipping_ignored_rows(beta, cg, flce_opts):
    """flce_kd_forward_ex2 / flce_jsd_forward_ex2 with FLCE_FORWARD_SKIP_IGNORED
    over 4 launches of 256 rows (the last holding fewer non-ignored rows, or
    none): KL or Jensen-Shannon values, loss and the counted rows' lse against
    the oracle, NaN lse on ignored rows, and the backwards from those lse
    (compacted and over every row) against the oracle."""
    flce_opts.set("cta_group", cg)
    flce_opts.set("skip_min_rows", "0")
    flce_opts.set("fwd_block_rows", "256")
    N, Hs, Ht, V = 900, 192, 256, 2100
    si, ti = _heads(N, Hs, Ht, V, seed=733)
    targets = np.random.default_rng(8).integers(0, V, N).astype(np.int64)
    targets[np.random.default_rng(9).permutation(N)[: N // 3]] = WL.IGNORE_INDEX
    weights = np.random.default_rng(10).uniform(0.3, 1.7, N).astype(np.float32)
    m = targets != WL.IGNORE_INDEX
    tfd = {"temperature": 1.5}
    tf = O.LogitTransform(**tfd)
    hs, Ws, ht, Wt = (to_dev_bf16(x) for x in (si.h, si.W, ti.h, ti.W))
    tg = torch.from_numpy(targets).cuda()
    w = torch.from_numpy(weights).cuda()
    if beta is None:
        out = flce.kd_forward(hs, Ws, ht, Wt, tg, w, 256, transform=tfd, skip_ignored=True)
        ref = O.kd_forward(si.h, si.W, ti.h, ti.W, targets, weights, tf=tf)
        assert_logp_close(np64(out["kl"]), ref.kl, "kl")
    else:
        out = flce.jsd_forward(hs, Ws, ht, Wt, beta, tg, w, 256, transform=tfd, skip_ignored=True)
        ref = O.jsd_forward(si.h, si.W, ti.h, ti.W, beta, targets, weights, tf=tf)
        assert_logp_close(np64(out["jsd"]), ref.jsd, "jsd")
        assert_logp_close(np64(out["kl_sm"])[m], ref.kl_sm[m], "kl_sm")
        assert np.all(np.isnan(np64(out["kl_sm"])[~m]))
    assert int(out["n_valid"]) == ref.n_valid == int(m.sum())
    assert float(out["loss"]) == pytest.approx(ref.loss, rel=LOSS_RTOL, abs=1e-6)
    for k, r in (("lse_s", ref.lse_s), ("lse_t", ref.lse_t)):
        assert_logp_close(np64(out[k])[m], r[m], k)
        assert np.all(np.isnan(np64(out[k])[~m]))
    g = 1.0 / ref.n_valid
    if beta is None:
        refb = O.kd_backward(si.h, si.W, ti.h, ti.W, targets, weights, g=g, tf=tf)
    else:
        refb = O.jsd_backward(si.h, si.W, ti.h, ti.W, beta, targets, weights, g=g, tf=tf)
    for compact in ("1", "0"):
        flce_opts.set("compact", compact)
        if beta is None:
            dH, dW = flce.kd_backward(hs, Ws, ht, Wt, out["lse_s"], out["lse_t"], g, tg, w, 256, transform=tfd)
        else:
            dH, dW = flce.jsd_backward(hs, Ws, ht, Wt, out["lse_s"], out["lse_t"], out["kl_sm"], g, beta, tg, w,
                                       256, transform=tfd)
        assert_grad_close(np64(dH), refb.dH, f"dH_s (compact {compact})")
        assert_grad_close(np64(dW), refb.dW, f"dW_s (compact {compact})")
    assert flce._lib.flce_device_status() == 0
