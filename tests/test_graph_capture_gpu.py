"""Forward + backward with a caller workspace captured into a CUDA graph and
replayed: the replay reproduces the eager results bit for bit (the kernels
are deterministic), on new inputs copied into the captured buffers too."""
import numpy as np
import pytest
import torch

from chunked_lm_head_gb300 import _lib
from chunked_lm_head_gb300 import workloads as WL

from gpu_util import upload

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("rows", [0, 512], ids=["one_slab", "pipelined"])
def test_forward_backward_graph_replay_matches_eager(rows, flce_opts):
    """rows = 512: 512-row blocks x vocabulary slabs, run as pipelined row
    blocks (the dependency counters are zeroed in the captured work)."""
    wl = WL.custom("graph", 700, 256, 3000, 256, w_std=0.05, targets="zipf", ignore_frac=0.05, seed=801)
    inp = WL.make_inputs(wl)
    h, W, t, w = upload(inp)
    N, H, V, cr = wl.N, wl.H, wl.V, 256
    flce_opts.set("bwd_rows", rows)
    plan = _lib.flce_backward_plan(N, H, V, cr)
    assert plan["dlogits_buffers"] == (2 if rows else 1), plan
    ws_bytes = _lib.flce_workspace_bytes(N, H, V, cr)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    bufs = dict(logp=torch.empty(N, device="cuda"), lse=torch.empty(N, device="cuda"),
                loss=torch.empty(1, device="cuda"), nv=torch.empty(1, dtype=torch.int64, device="cuda"),
                dH=torch.empty_like(h), dW=torch.empty((V, H), device="cuda"))
    g = 1.0 / int((inp.targets != -100).sum())

    def step():
        s1 = _lib.flce_forward(h, W, t, None, N, H, V, cr, -100, bufs["logp"], bufs["lse"],
                               bufs["loss"], bufs["nv"], ws, ws_bytes)
        s2 = _lib.flce_backward(h, W, t, None, bufs["lse"], g, bufs["dH"], bufs["dW"], N, H, V, cr,
                                -100, ws, ws_bytes)
        return s1, s2

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        assert step() == (0, 0)  # eager warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    eager = {k: v.clone() for k, v in bufs.items()}
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        assert step() == (0, 0)
    for v in bufs.values():
        v.zero_()
    graph.replay()
    torch.cuda.synchronize()
    for k in bufs:
        assert torch.equal(bufs[k], eager[k]), k
    graph.replay()  # a second replay: the same again
    torch.cuda.synchronize()
    for k in bufs:
        assert torch.equal(bufs[k], eager[k]), k
    # new inputs in the captured buffers: the replay follows them
    h2 = torch.from_numpy(WL.normal_bf16(99, 1, N * H, 1.0).view(np.int16)).cuda().view(torch.bfloat16)
    h.copy_(h2.view(N, H))
    graph.replay()
    torch.cuda.synchronize()
    ref_lse = bufs["lse"].clone()
    with torch.cuda.stream(side):
        assert step() == (0, 0)
    torch.cuda.synchronize()
    assert torch.equal(bufs["lse"], ref_lse)
    assert _lib.flce_device_status() == 0


def test_one_call_forward_backward_graph_replay_matches_eager():
    """flce_forward_backward (no logits recompute) with a caller workspace:
    captured, replayed, bit for bit the eager results."""
    wl = WL.custom("graph1", 700, 256, 3000, 768, w_std=0.05, targets="zipf", ignore_frac=0.05, seed=802)
    inp = WL.make_inputs(wl)
    h, W, t, w = upload(inp)
    N, H, V, cr = wl.N, wl.H, wl.V, 768
    ws_bytes = _lib.flce_forward_backward_workspace_bytes(N, H, V, cr)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    bufs = dict(logp=torch.empty(N, device="cuda"), lse=torch.empty(N, device="cuda"),
                loss=torch.empty(1, device="cuda"), nv=torch.empty(1, dtype=torch.int64, device="cuda"),
                dH=torch.empty_like(h), dW=torch.empty((V, H), device="cuda"))

    def step():
        return _lib.flce_forward_backward(h, W, t, None, N, H, V, cr, -100, None, 1.0, bufs["logp"],
                                          bufs["lse"], bufs["loss"], bufs["nv"], bufs["dH"], bufs["dW"],
                                          ws, ws_bytes)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        assert step() == 0
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    eager = {k: v.clone() for k, v in bufs.items()}
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        assert step() == 0
    for v in bufs.values():
        v.zero_()
    graph.replay()
    torch.cuda.synchronize()
    for k in bufs:
        assert torch.equal(bufs[k], eager[k]), k
    assert _lib.flce_device_status() == 0


def _capture_and_compare(step, bufs, nan_equal=False):
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        assert step() == 0
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    eager = {k: v.clone() for k, v in bufs.items()}
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        assert step() == 0
    for v in bufs.values():
        v.zero_()
    graph.replay()
    torch.cuda.synchronize()
    for k in bufs:
        if nan_equal:  # rows whose lse the forward skipped hold NaN in both runs
            assert torch.equal(torch.nan_to_num(bufs[k], nan=-7.0), torch.nan_to_num(eager[k], nan=-7.0)), k
        else:
            assert torch.equal(bufs[k], eager[k]), k
    assert _lib.flce_device_status() == 0


def test_distillation_graph_replay_matches_eager():
    """KL and Jensen-Shannon distillation forward + backward, captured."""
    s = WL.make_inputs(WL.custom("gkd_s", 600, 192, 2500, 256, w_std=0.05, seed=803))
    tt = WL.make_inputs(WL.custom("gkd_t", 600, 256, 2500, 256, w_std=0.06, seed=804))
    hs, Ws, _, _ = upload(s)
    ht, Wt, _, _ = upload(tt)
    N, Hs, Ht, V, cr = 600, 192, 256, 2500, 256
    ws_bytes = _lib.flce_kd_workspace_bytes(N, Hs, Ht, V, cr)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    bufs = dict(out=torch.empty(N, device="cuda"), lse_s=torch.empty(N, device="cuda"),
                lse_t=torch.empty(N, device="cuda"), klsm=torch.empty(N, device="cuda"),
                loss=torch.empty(1, device="cuda"), nv=torch.empty(1, dtype=torch.int64, device="cuda"),
                dH=torch.empty_like(hs), dW=torch.empty((V, Hs), device="cuda"))

    def kl_step():
        a = _lib.flce_kd_forward(hs, Ws, Hs, ht, Wt, Ht, None, None, N, V, cr, -100, None, bufs["out"],
                                 bufs["lse_s"], bufs["lse_t"], bufs["loss"], bufs["nv"], ws, ws_bytes)
        b = _lib.flce_kd_backward(hs, Ws, Hs, ht, Wt, Ht, None, None, bufs["lse_s"], bufs["lse_t"], 1.0 / N,
                                  bufs["dH"], bufs["dW"], N, V, cr, -100, None, ws, ws_bytes)
        return a | b

    def jsd_step():
        a = _lib.flce_jsd_forward(hs, Ws, Hs, ht, Wt, Ht, None, None, N, V, cr, -100, 0.5, None, bufs["out"],
                                  bufs["lse_s"], bufs["lse_t"], bufs["klsm"], bufs["loss"], bufs["nv"], ws,
                                  ws_bytes)
        b = _lib.flce_jsd_backward(hs, Ws, Hs, ht, Wt, Ht, None, None, bufs["lse_s"], bufs["lse_t"],
                                   bufs["klsm"], 0.5, 1.0 / N, bufs["dH"], bufs["dW"], N, V, cr, -100, None,
                                   ws, ws_bytes)
        return a | b

    _capture_and_compare(kl_step, {k: v for k, v in bufs.items() if k != "klsm"})  # KL writes no kl_sm
    _capture_and_compare(jsd_step, bufs)


def test_masked_distillation_graph_replay_matches_eager():
    """KL and Jensen-Shannon distillation with ignored rows, captured: the
    forwards skip them (rows listed and both heads gathered on the device)
    and the backwards run over the compacted rows."""
    N, Hs, Ht, V, cr = 2600, 192, 256, 2500, 512
    s = WL.make_inputs(WL.custom("gmk_s", N, Hs, V, cr, w_std=0.05, targets="zipf", grpo_seqs=4, prompt_len=200,
                                 seed=807))
    tt = WL.make_inputs(WL.custom("gmk_t", N, Ht, V, cr, w_std=0.06, seed=808))
    hs, Ws, t, w = upload(s)
    ht, Wt, _, _ = upload(tt)
    g = 1.0 / (N - 4 * 200)
    ws_bytes = _lib.flce_kd_workspace_bytes(N, Hs, Ht, V, cr)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    bufs = dict(out=torch.empty(N, device="cuda"), lse_s=torch.empty(N, device="cuda"),
                lse_t=torch.empty(N, device="cuda"), klsm=torch.empty(N, device="cuda"),
                loss=torch.empty(1, device="cuda"), nv=torch.empty(1, dtype=torch.int64, device="cuda"),
                dH=torch.empty_like(hs), dW=torch.empty((V, Hs), device="cuda"))
    skip = _lib.FORWARD_SKIP_IGNORED

    def kl_step():
        a = _lib.flce_kd_forward_ex2(hs, Ws, Hs, ht, Wt, Ht, t, w, N, V, cr, -100, None, skip, bufs["out"],
                                     bufs["lse_s"], bufs["lse_t"], bufs["loss"], bufs["nv"], ws, ws_bytes)
        b = _lib.flce_kd_backward(hs, Ws, Hs, ht, Wt, Ht, t, w, bufs["lse_s"], bufs["lse_t"], g, bufs["dH"],
                                  bufs["dW"], N, V, cr, -100, None, ws, ws_bytes)
        return a | b

    def jsd_step():
        a = _lib.flce_jsd_forward_ex2(hs, Ws, Hs, ht, Wt, Ht, t, w, N, V, cr, -100, 0.3, None, skip, bufs["out"],
                                      bufs["lse_s"], bufs["lse_t"], bufs["klsm"], bufs["loss"], bufs["nv"], ws,
                                      ws_bytes)
        b = _lib.flce_jsd_backward(hs, Ws, Hs, ht, Wt, Ht, t, w, bufs["lse_s"], bufs["lse_t"], bufs["klsm"], 0.3,
                                   g, bufs["dH"], bufs["dW"], N, V, cr, -100, None, ws, ws_bytes)
        return a | b

    _capture_and_compare(kl_step, {k: v for k, v in bufs.items() if k != "klsm"}, nan_equal=True)
    _capture_and_compare(jsd_step, bufs, nan_equal=True)
    assert int(bufs["nv"]) == N - 4 * 200
    assert bool(torch.isnan(bufs["lse_s"]).any())  # the forward did skip rows


def test_e4m3_forward_graph_replay_matches_eager():
    """Per-row e4m3 quantisation of h and the e4m3 forward, captured."""
    inp = WL.make_inputs(WL.custom("g8", 700, 256, 3000, 256, w_std=0.05, seed=805))
    h, W, t, _ = upload(inp)
    N, H, V = 700, 256, 3000
    W8 = torch.empty((V, H), dtype=torch.uint8, device="cuda")
    Wsc = torch.empty(V, device="cuda")
    assert _lib.flce_quantize_e4m3_rows(W, V, H, W8, Wsc) == 0
    ws_bytes = _lib.flce_workspace_bytes(N, H, V, 256)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    bufs = dict(h8=torch.empty((N, H), dtype=torch.uint8, device="cuda"), hsc=torch.empty(N, device="cuda"),
                logp=torch.empty(N, device="cuda"), lse=torch.empty(N, device="cuda"),
                loss=torch.empty(1, device="cuda"), nv=torch.empty(1, dtype=torch.int64, device="cuda"))

    def step():
        a = _lib.flce_quantize_e4m3_rows(h, N, H, bufs["h8"], bufs["hsc"])
        b = _lib.flce_forward_e4m3(bufs["h8"], bufs["hsc"], W8, Wsc, t, None, N, H, V, 256, -100, None,
                                   bufs["logp"], bufs["lse"], bufs["loss"], bufs["nv"], ws, ws_bytes)
        return a | b

    _capture_and_compare(step, bufs)


def test_row_skipping_forward_graph_replay_matches_eager():
    """flce_forward_ex2 with FLCE_FORWARD_SKIP_IGNORED (rows listed and
    gathered on the device) and the backward from its lse, captured."""
    wl = WL.custom("gskip", 2600, 256, 3000, 512, w_std=0.05, targets="zipf", grpo_seqs=4, prompt_len=200,
                   seed=806)
    inp = WL.make_inputs(wl)
    h, W, t, w = upload(inp)
    N, H, V, cr = wl.N, wl.H, wl.V, 512
    ws_bytes = _lib.flce_workspace_bytes(N, H, V, cr)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    bufs = dict(logp=torch.empty(N, device="cuda"), lse=torch.empty(N, device="cuda"),
                loss=torch.empty(1, device="cuda"), nv=torch.empty(1, dtype=torch.int64, device="cuda"),
                dH=torch.empty_like(h), dW=torch.empty((V, H), device="cuda"))

    def step():
        a = _lib.flce_forward_ex2(h, W, t, w, N, H, V, cr, -100, None, _lib.FORWARD_SKIP_IGNORED, bufs["logp"],
                                  bufs["lse"], bufs["loss"], bufs["nv"], ws, ws_bytes)
        b = _lib.flce_backward(h, W, t, w, bufs["lse"], 1.0 / (N - 4 * 200), bufs["dH"], bufs["dW"], N, H, V, cr,
                               -100, ws, ws_bytes)
        return a | b

    # lse of the ignored rows is NaN in both runs: compare with NaNs equal
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        assert step() == 0
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    eager = {k: v.clone() for k, v in bufs.items()}
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        assert step() == 0
    for v in bufs.values():
        v.zero_()
    graph.replay()
    torch.cuda.synchronize()
    for k in bufs:
        assert torch.equal(torch.nan_to_num(bufs[k], nan=-7.0), torch.nan_to_num(eager[k], nan=-7.0)), k
    assert int(torch.isnan(bufs["lse"]).sum()) == 4 * 200
    assert _lib.flce_device_status() == 0
