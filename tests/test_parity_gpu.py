"""GPU parity: libflce (through its C ABI) against the fp64 oracle on the same
seeded inputs.  Small cases and the 16,384-token SFT step are compared element
by element in full.  The GRPO and long-context workloads compare every row's
forward outputs with the oracle's stored full forward, dH on seeded sampled
rows and dW on seeded sampled vocabulary rows."""
import numpy as np
import pytest
import torch

from chunked_lm_head_gb300 import _lib
from chunked_lm_head_gb300 import workloads as WL
from oracle import flce_oracle as O

from gpu_util import (GRAD_RTOL, LOSS_RTOL, assert_grad_close, assert_logp_close, input_digest,
                      load_golden, np64, run_backward, run_forward, upload)

pytestmark = pytest.mark.gpu


def _full_check(inp, chunk_rows, g_scale=None):
    """Forward + backward of a small workload, every output against the oracle."""
    wl = inp.wl
    h, W, t, w = upload(inp)
    logp, lse, loss, nv = run_forward(h, W, t, w, chunk_rows)
    ref = O.forward(inp.h, inp.W, inp.targets, inp.weights, chunk_rows=chunk_rows)
    assert nv == ref.n_valid
    assert_logp_close(np64(logp), ref.logp, "logp")
    assert_logp_close(np64(lse), ref.lse, "lse")
    if ref.n_valid > 0:
        assert loss == pytest.approx(ref.loss, rel=LOSS_RTOL, abs=1e-6)
    else:
        assert loss == 0.0
    g = (1.0 / ref.n_valid if ref.n_valid else 1.0) if g_scale is None else g_scale
    dH, dW = run_backward(h, W, t, w, lse, g, chunk_rows)
    refb = O.backward(inp.h, inp.W, inp.targets, inp.weights, g=g, chunk_rows=chunk_rows)
    # an exactly-zero reference (V = 1, all rows ignored) admits only fp32
    # rounding noise of p - 1 in the kernels
    if np.linalg.norm(refb.dH) == 0:
        assert np.max(np.abs(np64(dH))) <= 1e-6 * max(abs(g), 1e-30) * 100
    else:
        assert_grad_close(np64(dH), refb.dH, "dH")
    if np.linalg.norm(refb.dW) == 0:
        assert np.max(np.abs(np64(dW))) <= 1e-6 * max(abs(g), 1e-30) * 100
    else:
        assert_grad_close(np64(dW), refb.dW, "dW")
    return logp, lse, loss, dH, dW


def test_tiny_workload_full():
    _full_check(WL.make_inputs("tiny"), 16)


def test_ragged_multi_tile_multi_chunk_weighted():
    # 3 row tiles (last 44 rows), K = 200 (ragged 64-blocks), 5 vocabulary
    # tiles (last 76 columns), 3 backward chunks, GRPO-style weights
    wl = WL.custom("ragged", 300, 200, 1100, 128, w_std=0.05, ignore_frac=0.1, seed=101)
    inp = WL.make_inputs(wl)
    inp.weights = np.random.default_rng(5).standard_normal(300).astype(np.float32)
    _full_check(inp, 128)


def test_multi_tile_zipf():
    wl = WL.custom("multi", 1000, 512, 5000, 256, w_std=0.04, targets="zipf", ignore_frac=0.03, seed=102)
    _full_check(WL.make_inputs(wl), 256)


def test_wide_hidden_ragged():
    # H = 1032: five 256-wide dH tiles (last one 8 wide), 17 K-blocks
    wl = WL.custom("wide", 130, 1032, 777, 64, w_std=0.03, seed=103)
    _full_check(WL.make_inputs(wl), 64)


@pytest.mark.parametrize("V", [1, 2, 8, 257])
def test_small_vocabularies(V):
    wl = WL.custom(f"v{V}", 40, 64, V, 32, w_std=0.5, seed=104 + V)
    _full_check(WL.make_inputs(wl), 32)


def test_empty_batch():
    wl = WL.custom("empty", 0, 64, 300, 16, seed=105)
    inp = WL.make_inputs(wl)
    h, W, t, w = upload(inp)
    h = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")
    t = torch.empty((0,), dtype=torch.int64, device="cuda")
    logp, lse, loss, nv = run_forward(h, W, t, None, 16)
    assert nv == 0 and loss == 0.0
    dH, dW = run_backward(h, W, t, None, lse, 1.0, 16)
    assert torch.all(dW == 0)


def test_all_rows_ignored():
    wl = WL.custom("allign", 150, 64, 500, 64, seed=106)
    inp = WL.make_inputs(wl)
    inp.targets[:] = WL.IGNORE_INDEX
    _, _, loss, dH, dW = _full_check(inp, 64, g_scale=1.0)
    assert loss == 0.0
    assert torch.all(dH == 0) and torch.all(dW == 0)


@pytest.mark.parametrize("compact", ["0", "1"])
def test_pipelined_row_blocks_all_rows_ignored(compact, flce_opts):
    """Pipelined row blocks (2 x 4 blocks, several slabs) where every row is
    ignored: without compaction the dlogits units write zero rows, with it
    the blocks have no rows and only the first writes dW's zeros; dH and dW
    are zero either way."""
    flce_opts.set("compact", compact)
    flce_opts.set("bwd_rows", 256)
    N, H, V, cr = 1000, 128, 4000, 128
    assert _lib.flce_backward_plan(N, H, V, cr)["dlogits_buffers"] == 2
    wl = WL.custom(f"pipeign{compact}", N, H, V, cr, w_std=0.05, seed=120)
    inp = WL.make_inputs(wl)
    inp.targets[:] = WL.IGNORE_INDEX
    h, W, t, w = upload(inp)
    logp, lse, loss, nv = run_forward(h, W, t, w, cr)
    assert nv == 0 and loss == 0.0
    dH, dW = run_backward(h, W, t, w, lse, 1.0, cr)
    _lib.check("flce_device_status", _lib.flce_device_status())
    assert torch.all(dH == 0) and torch.all(dW == 0)


def test_results_do_not_depend_on_chunk_rows_and_are_deterministic():
    wl = WL.custom("chunks", 700, 256, 3000, 128, w_std=0.05, targets="zipf", seed=107)
    inp = WL.make_inputs(wl)
    h, W, t, w = upload(inp)
    outs = []
    for cr in (128, 256, 700, 128):
        logp, lse, loss, nv = run_forward(h, W, t, w, cr)
        dH, dW = run_backward(h, W, t, w, lse, 1.0 / nv, cr)
        outs.append((logp, lse, loss, dH, dW))
    # forward never depends on chunk_rows: bitwise equal
    for o in outs[1:]:
        assert torch.equal(o[0], outs[0][0]) and torch.equal(o[1], outs[0][1]) and o[2] == outs[0][2]
    # same chunking twice: bitwise equal (no atomics in any reduction)
    assert torch.equal(outs[3][3], outs[0][3]) and torch.equal(outs[3][4], outs[0][4])
    # other chunkings: only the fp32 summation order of dW across chunks changes
    ref = O.backward(inp.h, inp.W, inp.targets, None, g=1.0 / int((inp.targets != -100).sum()))
    for o in outs:
        assert_grad_close(np64(o[3]), ref.dH, "dH")
        assert_grad_close(np64(o[4]), ref.dW, "dW")


def test_out_of_range_target():
    wl = WL.custom("bad", 64, 64, 300, 64, seed=108)
    inp = WL.make_inputs(wl)
    inp.targets[5] = 300  # == V: out of range
    h, W, t, w = upload(inp)
    logp, lse, loss, nv = run_forward(h, W, t, w, 64)
    assert np.isnan(np64(logp)[5]) and np.isnan(loss)
    ok = np.arange(64) != 5
    ref_lse = O.logsumexp_rows(O.logits(inp.h, inp.W))
    assert_logp_close(np64(lse), ref_lse, "lse")
    # validation mode rejects the call before any GEMM
    with _lib.options(validate=1):
        N, H, V = 64, 64, 300
        out = torch.empty(N, dtype=torch.float32, device="cuda")
        st = _lib.flce_forward(h, W, t, None, N, H, V, 64, -100, out, None, None, None, None, 0)
        assert st == 2
        dH = torch.empty_like(h)
        st = _lib.flce_backward(h, W, t, None, lse, 1.0, dH, None, N, H, V, 64, -100, None, 0)
        assert st == 2
        t[5] = 7
        assert _lib.flce_forward(h, W, t, None, N, H, V, 64, -100, out, None, None, None, None, 0) == 0
    assert _lib.flce_device_status() == 0
    assert ok.sum() == 63


def test_frozen_head_and_caller_workspace():
    wl = WL.custom("ws", 260, 128, 900, 128, seed=109)
    inp = WL.make_inputs(wl)
    h, W, t, w = upload(inp)
    nbytes = _lib.flce_workspace_bytes(260, 128, 900, 128)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    logp, lse, loss, nv = run_forward(h, W, t, w, 128, workspace=ws)
    dH, dW = run_backward(h, W, t, w, lse, 1.0 / nv, 128, need_dW=False, workspace=ws)
    assert dW is None
    ref = O.backward(inp.h, inp.W, inp.targets, None, g=1.0 / nv)
    assert_grad_close(np64(dH), ref.dH, "dH")
    # a workspace that is too small is refused before any launch
    small = ws[:256]
    st = _lib.flce_forward(h, W, t, None, 260, 128, 900, 128, -100, logp, None, None, None,
                           small, small.numel())
    assert st == 1
    st = _lib.flce_backward(h, W, t, None, lse, 1.0, dH, None, 260, 128, 900, 128, -100,
                            small, small.numel())
    assert st == 1


def test_single_chunk_workload_full():
    """256 x 248,320 x 2,048: the TRL single-chunk benchmark shape, in full."""
    _full_check(WL.make_inputs("single_chunk"), 256)


def _sft_16k_oracle_in_full(inp, g, block_rows=2048):
    """The oracle's forward and backward of every row, one logits block at a
    time: lse, logp, dH rows and each block's contribution to dW (summed)."""
    wl = inp.wl
    lse = np.empty(wl.N)
    logp = np.empty(wl.N)
    dH = np.empty((wl.N, wl.H))
    dW = np.zeros((wl.V, wl.H))
    for r0 in range(0, wl.N, block_rows):
        rows = np.arange(r0, min(wl.N, r0 + block_rows))
        lse[rows], logp[rows], dH[rows], part = O.rows_all(inp.h, inp.W, inp.targets, rows,
                                                            inp.weights, g=g)
        dW += part
    return lse, logp, dH, dW


def _fro_rows(got_dev, ref, what, block=8192):
    """Relative Frobenius error of a device matrix against an fp64 reference,
    copied back a block of rows at a time."""
    num = den = 0.0
    for r0 in range(0, ref.shape[0], block):
        a = np64(got_dev[r0:r0 + block])
        assert np.all(np.isfinite(a)), f"{what}: non-finite values in rows {r0}.."
        b = ref[r0:r0 + block]
        num += float(np.sum((a - b) ** 2))
        den += float(np.sum(b * b))
    e = (num / den) ** 0.5
    assert e <= GRAD_RTOL, f"{what}: relative Frobenius error {e:.3e}"


def _large_check(name, n_rows, n_vocab):
    """Full-size workload in the launch configuration the benchmark times.

    The 16,384-token SFT step is compared in full: every row's logp and lse,
    the loss, every row of dH and every vocabulary row of dW.  The GRPO and
    long-context workloads take the oracle's full forward from
    tests/golden/ (written by tests/golden/make_full_forward_golden.py, which
    calls only the oracle): every row's logp and lse, the loss and the
    ignored-token count against it; dH on seeded sampled rows; and the
    call's own dW on seeded sampled vocabulary rows, formed by the oracle from
    its stored lse of every row.
    """
    inp = WL.make_inputs(name)
    wl = inp.wl
    h, W, t, w = upload(inp)
    logp, lse, loss, nv = run_forward(h, W, t, w, wl.chunk_rows)
    m = inp.targets != WL.IGNORE_INDEX
    assert nv == int(m.sum())
    g = 1.0 / nv
    dH, dW = run_backward(h, W, t, w, lse, g, wl.chunk_rows)
    lp, ls = np64(logp), np64(lse)
    if name == "sft_16k":
        ref_lse, ref_logp, ref_dH, ref_dW = _sft_16k_oracle_in_full(inp, g)
        ref_loss = -float(np.sum(np.where(m, ref_logp, 0.0))) / nv
        assert_logp_close(lp, ref_logp, "logp (all rows)")
        assert_logp_close(ls, ref_lse, "lse (all rows)")
        assert loss == pytest.approx(ref_loss, rel=LOSS_RTOL)
        _fro_rows(dH, ref_dH, "dH (all rows)")
        _fro_rows(dW, ref_dW, "dW (all vocabulary rows)")
        return
    gold = load_golden(name)
    assert gold["meta"]["input_sha256"] == input_digest(inp), (
        "this machine drew other inputs than the ones the stored oracle forward was computed on")
    assert nv == gold["n_valid"]
    assert_logp_close(lp, gold["logp"], "logp (all rows)")
    assert_logp_close(ls, gold["lse"], "lse (all rows)")
    assert loss == pytest.approx(gold["loss"], rel=LOSS_RTOL)
    rows = WL.sample_rows(wl.N, n_rows, seed=wl.seed)
    vrows = WL.sample_rows(wl.V, n_vocab, seed=wl.seed + 1)
    ref_lse, ref_logp, ref_dH, _ = O.rows_all(inp.h, inp.W, inp.targets, rows, inp.weights, g=g,
                                              vocab_rows=vrows[:1])
    assert_logp_close(ls[rows], ref_lse, "lse (sampled rows, recomputed)")
    assert_grad_close(np64(dH[torch.from_numpy(rows).cuda()]), ref_dH, "dH (sampled rows)")
    ref_dWv = O.vocab_rows_dW(inp.h, inp.W, inp.targets, gold["lse"], vrows, inp.weights, g=g)
    assert_grad_close(np64(dW[torch.from_numpy(vrows).cuda()]), ref_dWv, "dW (sampled vocabulary rows)")


@pytest.mark.slow
def test_sft_16k_in_full():
    _large_check("sft_16k", 0, 0)


@pytest.mark.slow
def test_grpo_32k_full_forward_sampled_backward():
    _large_check("grpo_32k", 4096, 512)


@pytest.mark.slow
def test_long_131k_full_forward_sampled_backward():
    _large_check("long_131k", 4096, 512)


@pytest.mark.parametrize("cg", ["1", "2"])
def test_both_cta_group_paths(cg, flce_opts):
    """Single-CTA tiles (FLCE_CTA_GROUP=1) and SM-pair tiles (the default) both
    match the oracle on a ragged multi-tile, multi-chunk case."""
    flce_opts.set("cta_group", cg)
    wl = WL.custom(f"cg{cg}", 600, 264, 2100, 256, w_std=0.05, targets="zipf", ignore_frac=0.05,
                   seed=110)
    inp = WL.make_inputs(wl)
    inp.weights = np.random.default_rng(11).uniform(0.5, 1.5, wl.N).astype(np.float32)
    _full_check(inp, 256)


def test_row_compaction_matches_full_rows(flce_opts):
    """The backward on non-ignored rows only (default) against the backward
    over every row (FLCE_COMPACT=0) and the oracle, with a GRPO-like mask
    (prompt prefixes ignored) spanning several chunks and an empty last chunk."""
    wl = WL.custom("compact", 4 * 160, 192, 2500, 128, w_std=0.05, targets="zipf", grpo_seqs=4,
                   prompt_len=70, seed=111)
    inp = WL.make_inputs(wl)
    h, W, t, w = upload(inp)
    logp, lse, loss, nv = run_forward(h, W, t, w, 128)
    assert nv == 4 * 90
    g = 1.0 / nv
    dH_c, dW_c = run_backward(h, W, t, w, lse, g, 128)
    flce_opts.set("compact", "0")
    dH_f, dW_f = run_backward(h, W, t, w, lse, g, 128)
    ref = O.backward(inp.h, inp.W, inp.targets, inp.weights, g=g)
    for name, got in (("dH compact", dH_c), ("dH full", dH_f)):
        assert_grad_close(np64(got), ref.dH, name)
    for name, got in (("dW compact", dW_c), ("dW full", dW_f)):
        assert_grad_close(np64(got), ref.dW, name)
    ign = torch.from_numpy(inp.targets == WL.IGNORE_INDEX).cuda()
    assert torch.all(dH_c[ign] == 0)


@pytest.mark.parametrize("cg", ["1", "2"])
def test_forward_skipping_ignored_rows(cg, flce_opts):
    """flce_forward_ex2 with FLCE_FORWARD_SKIP_IGNORED: 5 forward launches of
    512 rows over the non-ignored rows (the third holds 256, the last two
    none), against the oracle.  Ignored rows get lse NaN and logp 0; the
    backward from that lse (compacted and over every row) matches the
    oracle."""
    flce_opts.set("cta_group", cg)
    flce_opts.set("fwd_block_rows", "512")
    wl = WL.custom("fskip", 2400, 192, 3100, 256, w_std=0.05, targets="zipf", grpo_seqs=4,
                   prompt_len=280, seed=112)
    inp = WL.make_inputs(wl)
    inp.weights = np.random.default_rng(5).uniform(0.2, 2.0, wl.N).astype(np.float32)
    h, W, t, w = upload(inp)
    N, H, V = wl.N, wl.H, wl.V
    logp = torch.full((N,), 7.0, device="cuda")
    lse = torch.full((N,), 7.0, device="cuda")
    loss = torch.full((1,), float("nan"), device="cuda")
    nv = torch.full((1,), -1, dtype=torch.int64, device="cuda")
    assert _lib.flce_forward_ex2(h, W, t, w, N, H, V, 256, -100, None, _lib.FORWARD_SKIP_IGNORED, logp, lse,
                                 loss, nv) == 0
    assert _lib.flce_device_status() == 0
    ref = O.forward(inp.h, inp.W, inp.targets, inp.weights)
    m = inp.targets != WL.IGNORE_INDEX
    assert int(nv.item()) == ref.n_valid == 2400 - 4 * 280
    assert float(loss.item()) == pytest.approx(ref.loss, rel=LOSS_RTOL)
    assert_logp_close(np64(logp), ref.logp, "logp")
    assert_logp_close(np64(lse)[m], ref.lse[m], "lse (non-ignored rows)")
    assert np.all(np.isnan(np64(lse)[~m])) and np.all(np64(logp)[~m] == 0.0)
    g = 1.0 / ref.n_valid
    refb = O.backward(inp.h, inp.W, inp.targets, inp.weights, g=g)
    for compact in ("1", "0"):
        flce_opts.set("compact", compact)
        dH, dW = run_backward(h, W, t, w, lse, g, 256)
        assert_grad_close(np64(dH), refb.dH, f"dH (compact {compact})")
        assert_grad_close(np64(dW), refb.dW, f"dW (compact {compact})")
    # FLCE_COMPACT=0 turns the skipping off, and so do calls under 2,048 rows:
    # every row gets its lse
    assert _lib.flce_forward_ex2(h, W, t, w, N, H, V, 256, -100, None, _lib.FORWARD_SKIP_IGNORED, logp, lse,
                                 loss, nv) == 0
    assert_logp_close(np64(lse), ref.lse, "lse (skipping off)")
    flce_opts.set("compact", "1")
    n = 2000
    assert _lib.flce_forward_ex2(h[:n], W, t[:n], w[:n], n, H, V, 256, -100, None, _lib.FORWARD_SKIP_IGNORED,
                                 logp[:n], lse[:n], loss, nv) == 0
    assert_logp_close(np64(lse[:n]), O.forward(inp.h[:n], inp.W, inp.targets[:n], inp.weights[:n]).lse,
                      "lse (2,000 rows)")


@pytest.mark.parametrize("splits", ["1", "3", "7"])
def test_forward_independent_of_vocabulary_splits(splits, flce_opts):
    """The split-V combine against a single split (and odd split counts):
    lse / logp agree to fp32 rounding and the loss to the loss tolerance."""
    wl = WL.custom("splits", 900, 192, 5000, 256, w_std=0.05, targets="zipf", ignore_frac=0.05, seed=112)
    inp = WL.make_inputs(wl)
    h, W, t, w = upload(inp)
    logp0, lse0, loss0, nv0 = run_forward(h, W, t, w, 256)
    flce_opts.set("fwd_splits", splits)
    logp1, lse1, loss1, nv1 = run_forward(h, W, t, w, 256)
    assert nv1 == nv0
    assert torch.allclose(lse1, lse0, atol=2e-5, rtol=0) and torch.allclose(logp1, logp0, atol=2e-5, rtol=0)
    assert loss1 == pytest.approx(loss0, rel=1e-6)
    ref = O.forward(inp.h, inp.W, inp.targets)
    assert_logp_close(np64(logp1), ref.logp, "logp")


@pytest.mark.parametrize("compact", ["0", "1"])
@pytest.mark.parametrize("cg", ["1", "2"])
def test_backward_row_blocks_and_vocabulary_slabs(cg, compact, flce_opts):
    """A 256-row dlogits budget walked as 768-row blocks x 5,120-column
    vocabulary slabs: 4 row blocks (the last 696 rows) x 4 slabs (the last
    4,640 columns), dH summed over the slabs in fp32 partials, dW
    read-modified-written once per row block; with and without row compaction,
    on both CTA-group paths."""
    flce_opts.set("cta_group", cg)
    flce_opts.set("compact", compact)
    flce_opts.set("bwd_rows", "768")
    flce_opts.set("pipeline", "0")  # the per-slab launches (the pipelined blocks: test_pipelined_row_blocks)
    N, H, V, cr = 3000, 512, 20000, 256
    plan = _lib.flce_backward_plan(N, H, V, cr)
    assert (plan["rows_per_block"], plan["vocab_per_slab"]) == (768, 5120)
    assert (plan["row_blocks"], plan["vocab_slabs"]) == (4, 4)
    assert plan["dlogits_bytes"] <= 256 * V * 2
    wl = WL.custom(f"slabs{cg}{compact}", N, H, V, cr, w_std=0.04, targets="zipf", ignore_frac=0.08,
                   seed=113)
    inp = WL.make_inputs(wl)
    inp.weights = np.random.default_rng(12).standard_normal(N).astype(np.float32)
    _full_check(inp, cr)


@pytest.mark.parametrize("compact", ["0", "1"])
@pytest.mark.parametrize("cg", ["1", "2"])
def test_one_launch_per_slab_for_dh_and_dw_is_bitwise_the_two_launches(cg, compact, flce_opts):
    """A slab's dH and dW units in one launch (the default) against two
    launches: every output element is accumulated by the same unit in the same
    order, so the results are bitwise equal; over 4 row blocks x 4 slabs, one
    slab (the default plan of a large chunk) and the one-call path."""
    flce_opts.set("cta_group", cg)
    flce_opts.set("compact", compact)
    flce_opts.set("pipeline", 0)  # the per-slab launches (the pipelined block has its own test)
    N, H, V = 3000, 512, 20000
    wl = WL.custom(f"fuse{cg}{compact}", N, H, V, 256, w_std=0.04, targets="zipf", ignore_frac=0.08,
                   seed=115)
    inp = WL.make_inputs(wl)
    inp.weights = np.random.default_rng(13).standard_normal(N).astype(np.float32)
    h, W, t, w = upload(inp)
    logp, lse, loss, nv = run_forward(h, W, t, w, 256)
    import chunked_lm_head_gb300 as flce
    for rows, chunk in ((768, 256), (0, 4096)):
        flce_opts.set("bwd_rows", rows)
        out = []
        for fuse in (1, 0):
            flce_opts.set("fuse_dh_dw", fuse)
            out.append(run_backward(h, W, t, w, lse, 1.0 / nv, chunk))
            out.append(tuple(flce.forward_backward(h, W, t, w, chunk)[k] for k in ("dH", "dW")))
        assert torch.equal(out[0][0], out[2][0]) and torch.equal(out[0][1], out[2][1]), rows
        assert torch.equal(out[1][0], out[3][0]) and torch.equal(out[1][1], out[3][1]), rows
    ref = O.backward(inp.h, inp.W, inp.targets, inp.weights, g=1.0 / nv)
    assert_grad_close(np64(out[0][0]), ref.dH, "dH")
    assert_grad_close(np64(out[0][1]), ref.dW, "dW")


# (N, H, V, chunk_rows, row block, logit transform): 4 row blocks (the last
# partial) x 4 slabs; an odd vocabulary with a narrow last slab, a ragged
# hidden tile and a soft-capped, tempered logit
PIPE_CASES = {
    "blocks4_slabs4": (3000, 512, 20000, 256, 768, None),
    "odd_v_softcap": (1000, 264, 7777, 128, 512, {"softcap": 20.0, "temperature": 0.8}),
}


@pytest.mark.parametrize("case", list(PIPE_CASES))
@pytest.mark.parametrize("compact", ["0", "1"])
@pytest.mark.parametrize("cg", ["1", "2"])
def test_pipelined_row_blocks(case, cg, compact, flce_opts):
    """A row block's dlogits, dH and dW units of every slab in one launch over
    two dlogits buffers, ordered by device-side counters (the default with
    several slabs): against the oracle and bitwise repeatable (every output
    element is summed by the same unit in the same order, the dH partials
    slab after slab); and the launch-per-slab path (one buffer of twice the
    slab) against the oracle."""
    N, H, V, chunk, rows, tfd = PIPE_CASES[case]
    flce_opts.set("cta_group", cg)
    flce_opts.set("compact", compact)
    flce_opts.set("bwd_rows", rows)
    plan = _lib.flce_backward_plan(N, H, V, chunk)
    assert plan["dlogits_buffers"] == 2 and plan["vocab_slabs"] > 1 and plan["row_blocks"] > 1, plan
    wl = WL.custom(f"pipe{case}{cg}{compact}", N, H, V, chunk, w_std=0.04, targets="zipf", ignore_frac=0.08,
                   seed=118)
    inp = WL.make_inputs(wl)
    inp.weights = np.random.default_rng(15).standard_normal(N).astype(np.float32)
    h, W, t, w = upload(inp)
    logp, lse, loss, nv = run_forward(h, W, t, w, chunk, transform=tfd)
    out = []
    for _ in range(3):
        out.append(run_backward(h, W, t, w, lse, 1.0 / nv, chunk, transform=tfd))
    flce_opts.set("pipeline", 0)
    assert _lib.flce_backward_plan(N, H, V, chunk)["dlogits_buffers"] == 1
    slabs = run_backward(h, W, t, w, lse, 1.0 / nv, chunk, transform=tfd)
    _lib.check("flce_device_status", _lib.flce_device_status())
    for k in (0, 1):
        for j in (1, 2):
            assert torch.equal(out[0][k], out[j][k]), (("dH", "dW")[k], j)
    tf = None if tfd is None else O.LogitTransform(**tfd)
    ref = O.backward(inp.h, inp.W, inp.targets, inp.weights, g=1.0 / nv, tf=tf)
    for name, got in (("pipelined", out[0]), ("per slab", slabs)):
        assert_grad_close(np64(got[0]), ref.dH, f"dH ({name})")
        assert_grad_close(np64(got[1]), ref.dW, f"dW ({name})")


@pytest.mark.parametrize("grid", ["few", "queued"])
@pytest.mark.parametrize("cg", ["1", "2"])
def test_pipelined_row_blocks_any_grid(grid, cg, flce_opts):
    """The pipelined launch on 3 workers, and on three times as many as the
    device holds at once (the extra ones start only as resident ones
    retire).  Workers draw units from a counter in an order in which every
    wait points back, so the launch completes either way; the plan is the
    device's and no summation order depends on the worker that runs a unit,
    so the gradients are bitwise those of the default grid."""
    N, H, V, chunk, rows, _ = PIPE_CASES["blocks4_slabs4"]
    flce_opts.set("cta_group", cg)
    flce_opts.set("bwd_rows", rows)
    plan = _lib.flce_backward_plan(N, H, V, chunk)
    assert plan["dlogits_buffers"] == 2 and plan["vocab_slabs"] > 1 and plan["row_blocks"] > 1, plan
    wl = WL.custom(f"pipegrid{cg}", N, H, V, chunk, w_std=0.04, targets="zipf", ignore_frac=0.08, seed=121)
    inp = WL.make_inputs(wl)
    h, W, t, w = upload(inp)
    logp, lse, loss, nv = run_forward(h, W, t, w, chunk)
    dflt = run_backward(h, W, t, w, lse, 1.0 / nv, chunk)
    resident = torch.cuda.get_device_properties(0).multi_processor_count // int(cg)
    flce_opts.set("grid_workers", 3 if grid == "few" else 3 * resident)
    got = run_backward(h, W, t, w, lse, 1.0 / nv, chunk)
    _lib.check("flce_device_status", _lib.flce_device_status())
    assert torch.equal(got[0], dflt[0]) and torch.equal(got[1], dflt[1])
    ref = O.backward(inp.h, inp.W, inp.targets, inp.weights, g=1.0 / nv)
    assert_grad_close(np64(got[0]), ref.dH, "dH")
    assert_grad_close(np64(got[1]), ref.dW, "dW")


@pytest.mark.parametrize("grid", [5, 600])
def test_one_slab_step_on_any_grid(grid, flce_opts):
    """Forward and one-slab backward with the GEMMs on 5 workers, and on 600
    (more than the device holds at once): bitwise the default grid's
    results."""
    wl = WL.custom("anygrid", 1500, 512, 5000, 256, w_std=0.05, targets="zipf", ignore_frac=0.05, seed=122)
    inp = WL.make_inputs(wl)
    h, W, t, w = upload(inp)

    def step():
        logp, lse, loss, nv = run_forward(h, W, t, w, 256)
        dH, dW = run_backward(h, W, t, w, lse, 1.0 / nv, 256)
        return logp, lse, torch.tensor([loss]), dH, dW

    dflt = step()
    flce_opts.set("grid_workers", grid)
    got = step()
    _lib.check("flce_device_status", _lib.flce_device_status())
    for name, a, b in zip(("logp", "lse", "loss", "dH", "dW"), got, dflt):
        assert torch.equal(a, b), name


@pytest.mark.parametrize("H", [4104, 4608])
@pytest.mark.parametrize("compact", ["0", "1"])
def test_wide_dh_tiles(H, compact, flce_opts):
    """dH over 256 x 512 tiles on SM pairs (the default for one slab with at
    least two waves of 256 x 256 tiles: 10 row tiles x 17 or 18 column tiles
    here): two 256-column tiles share each A stage, the last pair's second
    tile wholly past H when H = 4,104; against 256 x 256 tiles and the
    oracle, through the two-call backward and the one-call path."""
    import chunked_lm_head_gb300 as flce
    flce_opts.set("cta_group", 2)
    flce_opts.set("compact", compact)
    N, V, chunk = 2560, 3001, 2560
    wl = WL.custom(f"dh2_{H}{compact}", N, H, V, chunk, w_std=0.05, targets="zipf", ignore_frac=0.07,
                   seed=119 + H)
    inp = WL.make_inputs(wl)
    inp.weights = np.random.default_rng(16).uniform(0.2, 1.8, N).astype(np.float32)
    h, W, t, w = upload(inp)
    logp, lse, loss, nv = run_forward(h, W, t, w, chunk)
    out = {}
    for wide in (1, 0):
        flce_opts.set("dh_wide", wide)
        plan = _lib.flce_backward_plan(N, H, V, chunk)
        assert plan["vocab_slabs"] == 1 and plan["dh_wide"] == wide, plan
        out[wide] = (run_backward(h, W, t, w, lse, 1.0 / nv, chunk),
                     tuple(flce.forward_backward(h, W, t, w, chunk)[k] for k in ("dH", "dW")))
    _lib.check("flce_device_status", _lib.flce_device_status())
    ref = O.backward(inp.h, inp.W, inp.targets, inp.weights, g=1.0 / nv)
    for wide in (1, 0):
        for path in (0, 1):
            assert_grad_close(np64(out[wide][path][0]), ref.dH, f"dH (wide {wide}, path {path})")
        # dW does not depend on the dH tiling
        assert torch.equal(out[wide][0][1], out[0][0][1])


@pytest.mark.parametrize("cg", ["1", "2"])
def test_schedule_options_leave_the_gradients_bitwise_unchanged(cg, flce_opts):
    """An option that only changes the schedule: the dW epilogue with 16
    warps at short K (the default) against 8.  Every output element is summed
    by the same unit in the same order either way."""
    flce_opts.set("cta_group", cg)
    import chunked_lm_head_gb300 as flce
    # short K: 500 rows (8 K blocks) -> 8 or 16 dW epilogue warps
    wl = WL.custom(f"ew16{cg}", 500, 512, 30011, 512, w_std=0.04, targets="zipf", ignore_frac=0.06,
                   seed=116)
    inp = WL.make_inputs(wl)
    inp.weights = np.random.default_rng(14).uniform(0.3, 1.7, wl.N).astype(np.float32)
    h, W, t, w = upload(inp)
    logp, lse, loss, nv = run_forward(h, W, t, w, 512)
    outs = []
    for ew in (8, 16):
        flce_opts.set("dw_epilogue_warps", ew)
        outs.append(run_backward(h, W, t, w, lse, 1.0 / nv, 512))
        outs.append(tuple(flce.forward_backward(h, W, t, w, 512)[k] for k in ("dH", "dW")))
    assert torch.equal(outs[0][1], outs[2][1]) and torch.equal(outs[1][1], outs[3][1])
    ref = O.backward(inp.h, inp.W, inp.targets, inp.weights, g=1.0 / nv)
    assert_grad_close(np64(outs[2][1]), ref.dW, "dW (16 epilogue warps)")
    assert_grad_close(np64(outs[3][0]), ref.dH, "dH (one call, 16 epilogue warps)")


def test_backward_default_plan_odd_vocabulary():
    """The planner's own choice for a small chunk budget and an odd V (row
    pitch of D a multiple of 256, W rows of odd count) against the oracle,
    and bitwise repeatable."""
    N, H, V, cr = 2000, 256, 30011, 128
    plan = _lib.flce_backward_plan(N, H, V, cr)
    assert plan["dlogits_bytes"] <= 128 * (V + 5) * 2
    assert plan["row_blocks"] * plan["rows_per_block"] >= N
    assert plan["vocab_slabs"] * plan["vocab_per_slab"] >= V
    wl = WL.custom("oddv", N, H, V, cr, w_std=0.04, targets="zipf", ignore_frac=0.05, seed=114)
    inp = WL.make_inputs(wl)
    h, W, t, w = upload(inp)
    logp, lse, loss, nv = run_forward(h, W, t, w, cr)
    dH, dW = run_backward(h, W, t, w, lse, 1.0 / nv, cr)
    dH2, dW2 = run_backward(h, W, t, w, lse, 1.0 / nv, cr)
    assert torch.equal(dH, dH2) and torch.equal(dW, dW2)
    ref = O.backward(inp.h, inp.W, inp.targets, None, g=1.0 / nv)
    assert_grad_close(np64(dH), ref.dH, "dH")
    assert_grad_close(np64(dW), ref.dW, "dW")
