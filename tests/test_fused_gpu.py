"""Forward + backward in one call without the logits recompute
(flce_forward_backward) against the fp64 oracle and against the separate
forward and (recomputing) backward."""
import numpy as np
import pytest
import torch

from chunked_lm_head_gb300 import _lib
from chunked_lm_head_gb300 import workloads as WL
from oracle import flce_oracle as O

from gpu_util import (LOSS_RTOL, assert_grad_close, assert_logp_close, np64, rel_fro, run_backward,
                      run_forward, upload)

pytestmark = pytest.mark.gpu


def run_fused(h, W, t, w, chunk_rows, grad_scale=1.0, transform=None):
    N, H = h.shape
    V = W.shape[0]
    logp = torch.full((N,), float("nan"), dtype=torch.float32, device="cuda")
    lse = torch.full((N,), float("nan"), dtype=torch.float32, device="cuda")
    loss = torch.full((1,), float("nan"), dtype=torch.float32, device="cuda")
    nv = torch.full((1,), -1, dtype=torch.int64, device="cuda")
    dH = torch.full((N, H), float("nan"), dtype=torch.bfloat16, device="cuda")
    dW = torch.full((V, H), float("nan"), dtype=torch.float32, device="cuda")
    st = _lib.flce_forward_backward(h, W, t, w, N, H, V, chunk_rows, -100, transform, grad_scale, logp,
                                    lse, loss, nv, dH, dW)
    assert st == 0, _lib.STATUS_NAMES.get(st)
    assert _lib.flce_device_status() == 0
    return logp, lse, float(loss.item()), int(nv.item()), dH, dW


def _check(inp, chunk_rows, grad_scale=1.0, transform=None):
    h, W, t, w = upload(inp)
    logp, lse, loss, nv, dH, dW = run_fused(h, W, t, w, chunk_rows, grad_scale, transform)
    tf = None if transform is None else O.LogitTransform(**transform)
    ref = O.forward(inp.h, inp.W, inp.targets, inp.weights, tf=tf)
    assert nv == ref.n_valid
    assert_logp_close(np64(logp), ref.logp, "logp")
    assert_logp_close(np64(lse), ref.lse, "lse")
    if ref.n_valid:
        assert loss == pytest.approx(ref.loss, rel=LOSS_RTOL, abs=1e-6)
        g = grad_scale / ref.n_valid
        refb = O.backward(inp.h, inp.W, inp.targets, inp.weights, g=g, tf=tf)
        assert_grad_close(np64(dH), refb.dH, "dH")
        assert_grad_close(np64(dW), refb.dW, "dW")
    else:
        assert loss == 0.0
        assert float(dH.float().abs().max()) == 0.0 and float(dW.abs().max()) == 0.0
    return dH, dW


@pytest.mark.parametrize("cg", ["1", "2"])
def test_fused_single_block(cg, flce_opts):
    flce_opts.set("cta_group", cg)
    wl = WL.custom("fused1", 600, 256, 3000, 768, w_std=0.05, targets="zipf", ignore_frac=0.06, seed=501)
    inp = WL.make_inputs(wl)
    inp.weights = np.random.default_rng(31).uniform(0.3, 1.8, wl.N).astype(np.float32)
    _check(inp, 768, grad_scale=2.5)


@pytest.mark.parametrize("cg", ["1", "2"])
def test_fused_row_blocks_ragged(cg, flce_opts):
    """Two 2,048-row blocks (the last 952 rows) over V = 20,000."""
    flce_opts.set("cta_group", cg)
    wl = WL.custom("fused2", 3000, 512, 20000, 2048, w_std=0.04, targets="zipf", ignore_frac=0.05, seed=502)
    _check(WL.make_inputs(wl), 2048)


@pytest.mark.parametrize("transform", [{"softcap": 12.0, "temperature": 0.8},
                                       {"scale_multiply": 1.7, "temperature": 1.3}])
def test_fused_logit_transforms(transform):
    wl = WL.custom("fused_tf", 700, 192, 4000, 1024, w_std=0.2, targets="zipf", ignore_frac=0.05, seed=503)
    _check(WL.make_inputs(wl), 1024, transform=transform)


def test_fused_confident_rows_keep_the_target_gradient():
    """h aligned with its target's W row: p_t is about 0.99, so D_t = p_t - 1
    is about -0.01.  The call forms it from the exact target logit; the bf16
    exponentials alone (2^-9 relative rounding of p_t, about 0.002) would put
    a 20 % error on it.  The recomputing backward passes the same check."""
    r = np.random.default_rng(32)
    N, H, V = 512, 128, 700
    W = r.standard_normal((V, H)) * 0.3
    t = r.integers(0, V, N)
    h = 3.5 * W[t] / np.linalg.norm(W[t], axis=1, keepdims=True) + 0.05 * r.standard_normal((N, H))
    inp = WL.Inputs(WL.custom("conf", N, H, V, 512), WL.f32_to_bf16_bits(h.astype(np.float32)),
                    WL.f32_to_bf16_bits(W.astype(np.float32)), t.astype(np.int64), None,
                    np.array([0], dtype=np.int64))
    ref = O.forward(inp.h, inp.W, inp.targets)
    assert np.median(np.exp(ref.logp)) > 0.985
    _check(inp, 512)
    hd, Wd, td, _ = upload(inp)
    _, lse0, _, nv0 = run_forward(hd, Wd, td, None, 512)
    dH0, dW0 = run_backward(hd, Wd, td, None, lse0, 1.0 / nv0, 512)
    refb = O.backward(inp.h, inp.W, inp.targets, None, g=1.0 / nv0)
    assert_grad_close(np64(dH0), refb.dH, "dH (recomputing backward)")


def test_fused_all_rows_ignored_and_fallback_path():
    wl = WL.custom("fused_ign", 300, 128, 1500, 512, seed=504)
    inp = WL.make_inputs(wl)
    inp.targets[:] = WL.IGNORE_INDEX
    _check(inp, 512)
    # a chunk budget below 2,048 rows (and below N): forward + tiled backward,
    # the mean's 1 / n_valid applied on the device
    wl = WL.custom("fused_fb", 3000, 256, 5000, 256, w_std=0.05, targets="zipf", ignore_frac=0.1, seed=505)
    _check(WL.make_inputs(wl), 256, grad_scale=0.5)


@pytest.mark.parametrize("cg", ["1", "2"])
def test_fused_row_compaction_matches_the_full_rows(cg, flce_opts):
    """GRPO-style prompts (an ignored prefix of 690 rows in each of 4
    sequences of 1,500) over 2,048-row blocks.  Compacted, the blocks run over
    the non-ignored rows first: the second block mixes 1,192 of them with
    ignored rows, the ragged third holds ignored rows only.  Both the compacted
    and the full-row call match the oracle and each other."""
    flce_opts.set("cta_group", cg)
    wl = WL.custom("fused_cmp", 6000, 256, 9000, 2048, w_std=0.05, targets="zipf", grpo_seqs=4,
                   prompt_len=690, seed=506)
    inp = WL.make_inputs(wl)
    assert int((inp.targets != WL.IGNORE_INDEX).sum()) == 3240
    dH, dW = _check(inp, 2048, grad_scale=1.5)
    ign = torch.from_numpy(inp.targets == WL.IGNORE_INDEX).cuda()
    assert float(dH[ign].float().abs().max()) == 0.0
    flce_opts.set("compact", "0")
    h, W, t, w = upload(inp)
    logp0, lse0, loss0, nv0, dH0, dW0 = run_fused(h, W, t, w, 2048, grad_scale=1.5)
    flce_opts.set("compact", 1)
    logp1, lse1, loss1, nv1, _, _ = run_fused(h, W, t, w, 2048, grad_scale=1.5)
    assert nv0 == nv1 == 3240
    assert torch.allclose(lse1, lse0, atol=2e-5, rtol=0) and torch.allclose(logp1, logp0, atol=2e-5, rtol=0)
    assert loss1 == pytest.approx(loss0, rel=1e-6)
    assert rel_fro(np64(dH), np64(dH0)) <= 1e-3
    assert rel_fro(np64(dW), np64(dW0)) <= 1e-3


def test_fused_without_lse_skips_the_ignored_rows_forward():
    """out_lse = NULL: the compacted forward covers only the non-ignored rows
    (their lse is never observed).  Loss, logp and gradients match the oracle
    and the call that returns lse."""
    wl = WL.custom("fused_nolse", 6000, 256, 9000, 2048, w_std=0.05, targets="zipf", grpo_seqs=4,
                   prompt_len=690, seed=507)
    inp = WL.make_inputs(wl)
    h, W, t, w = upload(inp)
    N, H, V = wl.N, wl.H, wl.V
    logp = torch.full((N,), float("nan"), device="cuda")
    loss = torch.full((1,), float("nan"), device="cuda")
    nv = torch.full((1,), -1, dtype=torch.int64, device="cuda")
    dH = torch.full((N, H), float("nan"), dtype=torch.bfloat16, device="cuda")
    dW = torch.full((V, H), float("nan"), device="cuda")
    assert _lib.flce_forward_backward(h, W, t, w, N, H, V, 2048, -100, None, 1.0, logp, None, loss, nv,
                                      dH, dW) == 0
    assert _lib.flce_device_status() == 0
    ref = O.forward(inp.h, inp.W, inp.targets, inp.weights)
    refb = O.backward(inp.h, inp.W, inp.targets, inp.weights, g=1.0 / ref.n_valid)
    assert int(nv.item()) == ref.n_valid == 3240
    assert_logp_close(np64(logp), ref.logp, "logp")
    assert float(loss.item()) == pytest.approx(ref.loss, rel=LOSS_RTOL)
    assert_grad_close(np64(dH), refb.dH, "dH")
    assert_grad_close(np64(dW), refb.dW, "dW")
    logp1, _, loss1, _, dH1, dW1 = run_fused(h, W, t, w, 2048)
    assert torch.allclose(logp, logp1, atol=2e-5, rtol=0) and float(loss.item()) == pytest.approx(loss1, rel=1e-6)
    assert rel_fro(np64(dH), np64(dH1)) <= 1e-3 and rel_fro(np64(dW), np64(dW1)) <= 1e-3
    # every row ignored: no forward rows at all, zero loss and gradients
    t.fill_(-100)
    assert _lib.flce_forward_backward(h, W, t, w, N, H, V, 2048, -100, None, 1.0, logp, None, loss, nv,
                                      dH, dW) == 0
    assert _lib.flce_device_status() == 0
    assert int(nv.item()) == 0 and float(loss.item()) == 0.0 and float(logp.abs().max()) == 0.0
    assert float(dH.float().abs().max()) == 0.0 and float(dW.abs().max()) == 0.0


@pytest.mark.slow
def test_fused_grpo_32k_row_compaction(flce_opts):
    """32,768 x 4,096 x 128,000 at 4,096-row blocks, 12.5 % of the rows in
    ignored prompts: the compacted call (the eighth block all ignored rows)
    against the full-row call."""
    inp = WL.make_inputs("grpo_32k")
    h, W, t, w = upload(inp)
    logp, lse, loss, nv, dH, dW = run_fused(h, W, t, w, 4096)
    ign = torch.from_numpy(inp.targets == WL.IGNORE_INDEX).cuda()
    assert nv == 28672 and float(dH[ign].float().abs().max()) == 0.0
    flce_opts.set("compact", "0")
    logp0, lse0, loss0, nv0, dH0, dW0 = run_fused(h, W, t, w, 4096)
    assert nv0 == nv
    assert torch.allclose(lse, lse0, atol=2e-5, rtol=0) and torch.allclose(logp, logp0, atol=2e-5, rtol=0)
    assert loss == pytest.approx(loss0, rel=1e-6)
    assert rel_fro(np64(dH), np64(dH0)) <= 1e-3
    assert rel_fro(np64(dW), np64(dW0)) <= 1e-3


@pytest.mark.slow
def test_fused_sft_16k_matches_the_recomputing_path():
    """16,384 x 4,096 x 151,936 at 4,096-row blocks: the same loss and lse as
    the separate forward, gradients within the parity tolerance of the
    recomputing backward's."""
    inp = WL.make_inputs("sft_16k")
    h, W, t, w = upload(inp)
    logp, lse, loss, nv, dH, dW = run_fused(h, W, t, w, 4096)
    logp0, lse0, loss0, nv0 = run_forward(h, W, t, w, 4096)
    dH0, dW0 = run_backward(h, W, t, w, lse0, 1.0 / nv0, 4096)
    assert nv == nv0 == 16380
    assert torch.allclose(lse, lse0, atol=2e-5, rtol=0) and torch.allclose(logp, logp0, atol=2e-5, rtol=0)
    assert loss == pytest.approx(loss0, rel=1e-6)
    assert rel_fro(np64(dH), np64(dH0)) <= 1e-2
    assert rel_fro(np64(dW), np64(dW0)) <= 1e-2


@pytest.mark.slow
def test_fused_long_131k_sampled_int64_indexing():
    """131,072 x 2,560 x 151,936 with 4,096-row blocks (N V >= 2^31: the int64
    kernels): logp / lse and dH on seeded sampled rows, dW on sampled
    vocabulary rows through its linearity in the per-row weights."""
    inp = WL.make_inputs("long_131k")
    wl = inp.wl
    h, W, t, w = upload(inp)
    logp, lse, loss, nv, dH, dW = run_fused(h, W, t, w, 4096)
    m = inp.targets != WL.IGNORE_INDEX
    assert nv == int(m.sum())
    g = 1.0 / nv
    rows = WL.sample_rows(wl.N, 2048, seed=wl.seed)
    vrows = WL.sample_rows(wl.V, 256, seed=wl.seed + 1)
    ref_lse, ref_logp, ref_dH, ref_dWpart = O.rows_all(inp.h, inp.W, inp.targets, rows, inp.weights,
                                                       g=g, vocab_rows=vrows)
    assert_logp_close(np64(logp)[rows], ref_logp, "logp (sampled rows)")
    assert_logp_close(np64(lse)[rows], ref_lse, "lse (sampled rows)")
    assert_grad_close(np64(dH[torch.from_numpy(rows).cuda()]), ref_dH, "dH (sampled rows)")
    # dW: weights zero outside the sampled rows; grad_scale nv * g / (rows' n_valid) undoes
    # the call's own 1 / n_valid so that the scale is the same g as the oracle's
    w0 = np.zeros(wl.N, dtype=np.float32)
    w0[rows] = 1.0
    _, _, _, nv0, _, dW0 = run_fused(h, W, t, torch.from_numpy(w0).cuda(), 4096, grad_scale=nv * g)
    assert nv0 == nv
    vsel = torch.from_numpy(vrows).cuda()
    assert_grad_close(np64(dW0[vsel]), ref_dWpart, "dW (sampled rows x sampled vocabulary)")
