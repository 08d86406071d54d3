"""The allocation-free forward against the regular forward.

flce_forward_static_scratch is for callers that may not allocate device
memory (runtimes that own all device memory through a fixed pool of their own,
services that must keep a constant footprint): it runs the forward on a scratch
array the library keeps in device memory instead of a caller-provided or
stream-allocated workspace.  Here it must reproduce flce_forward, call after
call, even though each call finds the previous call's leftovers in that shared
scratch, and it must leave the stream-ordered memory pool's high-water mark
and torch's allocator where they were.

This file is named so that pytest collects it last."""
import ctypes

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


# CUmemPool_attribute values (cuda.h): bytes in use, and its high-water mark
_POOL_USED_MEM_CURRENT, _POOL_USED_MEM_HIGH = 7, 8


class _StreamPool:
    """The current device's stream-ordered memory pool (the one cudaMallocAsync
    draws from), through the driver API."""

    def __init__(self):
        self.cu = ctypes.CDLL("libcuda.so.1")
        self.pool = ctypes.c_void_p()
        dev = torch.cuda.current_device()
        assert self.cu.cuDeviceGetMemPool(ctypes.byref(self.pool), ctypes.c_int(dev)) == 0

    def get(self, attr):
        v = ctypes.c_uint64(0)
        assert self.cu.cuMemPoolGetAttribute(self.pool, ctypes.c_int(attr), ctypes.byref(v)) == 0
        return v.value

    def reset_high(self):
        v = ctypes.c_uint64(0)  # the high-water mark can only be reset, to zero
        assert self.cu.cuMemPoolSetAttribute(self.pool, ctypes.c_int(_POOL_USED_MEM_HIGH),
                                             ctypes.byref(v)) == 0


def test_static_scratch_forward_allocates_nothing():
    """The regular forward without a workspace raises the pool's high-water
    mark (it allocates on the stream); the allocation-free forward, from its
    second call on, leaves it and torch's allocator untouched."""
    wl = WL.custom("noalloc_c", 2000, 256, 12000, 256, w_std=0.04, targets="zipf", ignore_frac=0.05,
                   seed=203)
    inp = WL.make_inputs(wl)
    h, W, t, w = upload(inp)
    ref = run_forward(h, W, t, w, wl.chunk_rows)
    _forward_static(h, W, t, w, wl.chunk_rows)  # first call on the device: address set-up
    torch.cuda.synchronize()
    pool = _StreamPool()
    pool.reset_high()
    used0 = pool.get(_POOL_USED_MEM_CURRENT)
    assert pool.get(_POOL_USED_MEM_HIGH) <= used0
    run_forward(h, W, t, w, wl.chunk_rows)
    torch.cuda.synchronize()
    assert pool.get(_POOL_USED_MEM_HIGH) > used0  # the check sees a stream allocation
    # the outputs are the caller's: allocated before the measured call
    N, H, V = wl.N, wl.H, wl.V
    logp = torch.full((N,), float("nan"), dtype=torch.float32, device="cuda")
    lse = torch.full((N,), float("nan"), dtype=torch.float32, device="cuda")
    loss = torch.full((1,), float("nan"), dtype=torch.float32, device="cuda")
    nv = torch.full((1,), -1, dtype=torch.int64, device="cuda")
    torch.cuda.synchronize()
    pool.reset_high()
    used0 = pool.get(_POOL_USED_MEM_CURRENT)
    alloc0, reserved0 = torch.cuda.memory_allocated(), torch.cuda.memory_reserved()
    st = _lib.flce_forward_static_scratch(h, W, t, w, N, H, V, wl.chunk_rows, -100, logp, lse, loss, nv)
    torch.cuda.synchronize()
    assert st == 0, _lib.STATUS_NAMES.get(st)
    assert pool.get(_POOL_USED_MEM_HIGH) <= used0  # no allocation at any point of the call
    assert pool.get(_POOL_USED_MEM_CURRENT) == used0
    assert torch.cuda.memory_reserved() == reserved0
    assert torch.cuda.memory_allocated() == alloc0
    assert _lib.flce_device_status() == 0
    assert int(nv.item()) == ref[3]
    assert_logp_close(np64(logp), np64(ref[0]), "logp")
    assert float(loss.item()) == pytest.approx(ref[2], rel=LOSS_RTOL)


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


def test_static_scratch_forward_graph_replay():
    """After one eager call on the device, the allocation-free forward is
    captured into a CUDA graph; each replay reproduces the eager call bit for
    bit, and follows new inputs copied into the captured buffers."""
    wl = WL.custom("noalloc_g", 1200, 256, 9000, 256, w_std=0.04, targets="zipf", ignore_frac=0.05,
                   seed=204)
    inp = WL.make_inputs(wl)
    h, W, t, w = upload(inp)
    N, H, V = wl.N, wl.H, wl.V
    out = dict(logp=torch.empty(N, device="cuda"), lse=torch.empty(N, device="cuda"),
               loss=torch.empty(1, device="cuda"), nv=torch.empty(1, dtype=torch.int64, device="cuda"))

    def call(stream):
        return _lib.flce_forward_static_scratch(h, W, t, w, N, H, V, wl.chunk_rows, -100, out["logp"],
                                                out["lse"], out["loss"], out["nv"], stream)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        assert call(side.cuda_stream) == 0  # eager: the scratch address is looked up here
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    eager = {k: v.clone() for k, v in out.items()}
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        assert call(torch.cuda.current_stream().cuda_stream) == 0
    for _ in range(2):
        for v in out.values():
            v.zero_()
        graph.replay()
        torch.cuda.synchronize()
        for k in out:
            assert torch.equal(out[k], eager[k]), k
    # the regular forward on the same inputs: the same results
    ref = run_forward(h, W, t, w, wl.chunk_rows)
    assert int(out["nv"].item()) == ref[3]
    assert_logp_close(np64(out["logp"]), np64(ref[0]), "logp")
    # new inputs in the captured buffers: the replay follows them
    h.copy_(torch.flip(h, dims=[0]))
    graph.replay()
    torch.cuda.synchronize()
    replayed = out["lse"].clone()
    with torch.cuda.stream(side):
        assert call(side.cuda_stream) == 0
    torch.cuda.synchronize()
    assert torch.equal(out["lse"], replayed)
    assert _lib.flce_device_status() == 0
