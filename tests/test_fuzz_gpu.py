"""Seeded random small problems (ragged N, H down to 8, V down to 1, chunk
sizes from 1 row up, masks, weights, transforms, both CTA-group paths, row
compaction on and off, forced backward row blocks, the one-call path, the
forward that skips ignored rows) against the fp64 oracle."""
import numpy as np
import pytest
import torch

from chunked_lm_head_gb300 import _lib
from chunked_lm_head_gb300 import workloads as WL
from oracle import flce_oracle as O

from gpu_util import LOSS_RTOL, assert_grad_close, assert_logp_close, np64, run_backward, run_forward, upload

pytestmark = pytest.mark.gpu

TRANSFORMS = [None, {"softcap": 8.0, "temperature": 1.2}, {"scale_multiply": 0.7, "temperature": 0.6}]


def _cases(n, seed=900):
    r = np.random.default_rng(seed)
    fixed = [dict(N=1, H=8, V=1, chunk=1), dict(N=3, H=8, V=5, chunk=1), dict(N=700, H=8, V=3001, chunk=128),
             dict(N=257, H=520, V=2, chunk=300), dict(N=129, H=64, V=4099, chunk=129)]
    out = []
    for k in range(n):
        c = fixed[k] if k < len(fixed) else dict(
            N=int(r.integers(1, 1200)), H=int(8 * r.integers(1, 80)), V=int(r.integers(1, 6000)),
            chunk=int(r.choice([1, 16, 100, 128, 256, 777, 2048])))
        c.update(cg=str(r.choice(["1", "2"])), compact=str(r.choice(["0", "1"])),
                 ignore=float(r.choice([0.0, 0.1, 0.5, 1.0], p=[0.35, 0.35, 0.2, 0.1])),
                 weights=bool(r.uniform() < 0.5), tf=int(r.integers(0, 3)),
                 rows=int(r.choice([0, 0, 256, 512])), fused=bool(r.uniform() < 0.3), seed=1000 + k)
        out.append(c)
    return out


@pytest.mark.parametrize("c", _cases(64), ids=lambda c: f"N{c['N']}H{c['H']}V{c['V']}c{c['chunk']}")
def test_random_problem_matches_oracle(c, flce_opts):
    flce_opts.set("cta_group", c["cg"])
    flce_opts.set("compact", c["compact"])
    if c["rows"]:
        flce_opts.set("bwd_rows", str(c["rows"]))
    wl = WL.custom("fuzz", c["N"], c["H"], c["V"], c["chunk"], w_std=0.1, ignore_frac=0.0, seed=c["seed"])
    inp = WL.make_inputs(wl)
    r = np.random.default_rng(c["seed"])
    inp.targets[r.uniform(size=c["N"]) < c["ignore"]] = WL.IGNORE_INDEX
    if c["weights"]:
        inp.weights = r.uniform(-1.0, 2.0, c["N"]).astype(np.float32)
    tfd = TRANSFORMS[c["tf"]]
    tf = None if tfd is None else O.LogitTransform(**tfd)
    ref = O.forward(inp.h, inp.W, inp.targets, inp.weights, tf=tf)
    g = 1.0 / ref.n_valid if ref.n_valid else 1.0
    refb = O.backward(inp.h, inp.W, inp.targets, inp.weights, g=g, tf=tf)
    h, W, t, w = upload(inp)
    N, H = h.shape
    V = W.shape[0]
    if c["fused"]:
        logp = torch.empty(N, dtype=torch.float32, device="cuda")
        lse = torch.empty(N, dtype=torch.float32, device="cuda")
        loss_t = torch.empty(1, dtype=torch.float32, device="cuda")
        nv_t = torch.empty(1, dtype=torch.int64, device="cuda")
        dH = torch.empty_like(h)
        dW = torch.empty((V, H), dtype=torch.float32, device="cuda")
        # grad_scale g * n_valid: the call divides by n_valid itself
        assert _lib.flce_forward_backward(h, W, t, w, N, H, V, c["chunk"], -100, tfd,
                                          g * max(ref.n_valid, 1), logp, lse, loss_t, nv_t, dH, dW) == 0
        assert _lib.flce_device_status() == 0
        loss, nv = float(loss_t.item()), int(nv_t.item())
    elif c["seed"] % 2 == 0:  # the forward that skips ignored rows (their lse is NaN)
        flce_opts.set("skip_min_rows", "0")  # at every size
        logp = torch.empty(N, dtype=torch.float32, device="cuda")
        lse = torch.empty(N, dtype=torch.float32, device="cuda")
        loss_t = torch.empty(1, dtype=torch.float32, device="cuda")
        nv_t = torch.empty(1, dtype=torch.int64, device="cuda")
        assert _lib.flce_forward_ex2(h, W, t, w, N, H, V, c["chunk"], -100, tfd, _lib.FORWARD_SKIP_IGNORED,
                                     logp, lse, loss_t, nv_t) == 0
        assert _lib.flce_device_status() == 0
        loss, nv = float(loss_t.item()), int(nv_t.item())
        dH, dW = run_backward(h, W, t, w, lse, g, c["chunk"], transform=tfd)
        m = inp.targets != WL.IGNORE_INDEX
        if c["compact"] == "1":
            assert np.all(np.isnan(np64(lse)[~m]))
            lse = torch.from_numpy(np.where(m, np64(lse), ref.lse))  # compared on the counted rows
    else:
        logp, lse, loss, nv = run_forward(h, W, t, w, c["chunk"], transform=tfd)
        dH, dW = run_backward(h, W, t, w, lse, g, c["chunk"], transform=tfd)
    assert nv == ref.n_valid
    assert_logp_close(np64(logp), ref.logp, "logp")
    assert_logp_close(np64(lse), ref.lse, "lse")
    assert loss == pytest.approx(ref.loss, rel=LOSS_RTOL, abs=1e-6)
    for name, got, want in (("dH", np64(dH), refb.dH), ("dW", np64(dW), refb.dW)):
        scale = np.linalg.norm(want)
        if scale < 1e-6:  # no valid row, V = 1, or all-zero weights: fp32 noise only
            assert np.max(np.abs(got)) <= 1e-5, name
        else:
            assert_grad_close(got, want, name)


def _kd_cases(n, seed=950):
    r = np.random.default_rng(seed)
    out = []
    for k in range(n):
        out.append(dict(N=int(r.integers(1, 700)), Hs=int(8 * r.integers(1, 48)), Ht=int(8 * r.integers(1, 48)),
                        V=int(r.integers(2, 4000)), chunk=int(r.choice([1, 64, 128, 300, 1024])),
                        cg=str(r.choice(["1", "2"])), masked=bool(r.uniform() < 0.6),
                        jsd=float(r.choice([0.0, 0.5, 0.2, 0.85])), tf=int(r.integers(0, 3)), seed=2000 + k,
                        compact="0" if k % 4 == 3 else "1", wide="0" if k % 4 == 1 else "1"))
    return out


@pytest.mark.parametrize("c", _kd_cases(24), ids=lambda c: f"N{c['N']}Hs{c['Hs']}Ht{c['Ht']}V{c['V']}b{c['jsd']}")
def test_random_distillation_matches_oracle(c, flce_opts):
    import chunked_lm_head_gb300 as flce
    from gpu_util import to_dev_bf16
    flce_opts.set("cta_group", c["cg"])
    flce_opts.set("compact", c["compact"])  # masked backward: compacted rows or every row
    flce_opts.set("wide_epilogue", c["wide"])  # dlogits epilogue: 8 warps or 4
    s = WL.make_inputs(WL.custom("kfs", c["N"], c["Hs"], c["V"], 256, w_std=0.1, seed=c["seed"]))
    t_ = WL.make_inputs(WL.custom("kft", c["N"], c["Ht"], c["V"], 256, w_std=0.12, seed=c["seed"] + 500))
    r = np.random.default_rng(c["seed"])
    targets = None
    if c["masked"]:
        targets = r.integers(0, c["V"], c["N"]).astype(np.int64)
        targets[r.uniform(size=c["N"]) < 0.2] = WL.IGNORE_INDEX
    weights = r.uniform(0.2, 1.8, c["N"]).astype(np.float32)
    tfd = TRANSFORMS[c["tf"]]
    tf = None if tfd is None else O.LogitTransform(**tfd)
    hs, Ws, ht, Wt = (to_dev_bf16(x) for x in (s.h, s.W, t_.h, t_.W))
    tg = None if targets is None else torch.from_numpy(targets).cuda()
    w = torch.from_numpy(weights).cuda()
    if c["jsd"]:
        out = flce.jsd_forward(hs, Ws, ht, Wt, c["jsd"], tg, w, c["chunk"], transform=tfd)
        ref = O.jsd_forward(s.h, s.W, t_.h, t_.W, c["jsd"], targets, weights, tf=tf)
        assert_logp_close(np64(out["jsd"]), ref.jsd, "jsd")
    else:
        out = flce.kd_forward(hs, Ws, ht, Wt, tg, w, c["chunk"], transform=tfd)
        ref = O.kd_forward(s.h, s.W, t_.h, t_.W, targets, weights, tf=tf)
        assert_logp_close(np64(out["kl"]), ref.kl, "kl")
    assert int(out["n_valid"]) == ref.n_valid
    assert_logp_close(np64(out["lse_s"]), ref.lse_s, "lse_s")
    assert float(out["loss"]) == pytest.approx(ref.loss, rel=LOSS_RTOL, abs=1e-6)
    g = 1.0 / ref.n_valid if ref.n_valid else 1.0
    if c["jsd"]:
        dH, dW = flce.jsd_backward(hs, Ws, ht, Wt, out["lse_s"], out["lse_t"], out["kl_sm"], g, c["jsd"], tg, w,
                                   c["chunk"], transform=tfd)
        refb = O.jsd_backward(s.h, s.W, t_.h, t_.W, c["jsd"], targets, weights, g=g, tf=tf)
    else:
        dH, dW = flce.kd_backward(hs, Ws, ht, Wt, out["lse_s"], out["lse_t"], g, tg, w, c["chunk"], transform=tfd)
        refb = O.kd_backward(s.h, s.W, t_.h, t_.W, targets, weights, g=g, tf=tf)
    assert _lib.flce_device_status() == 0
    for name, got, want in (("dH", np64(dH), refb.dH), ("dW", np64(dW), refb.dW)):
        if np.linalg.norm(want) < 1e-6:
            assert np.max(np.abs(got)) <= 1e-5, name
        else:
            assert_grad_close(got, want, name)
