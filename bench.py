"""Benchmark of the fused LM-head cross-entropy forward+backward (libflce).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload sft_16k] [--impl gb300|reference]

One step = flce_forward + flce_backward (dH and dW) over one batch of the
workload, through the C ABI, inputs resident in HBM.  Prints ONE JSON line.
Under torchrun (N > 1) every rank runs an independent replica of the workload
on its own GPU (weak scaling, no collective on the data path); rank 0 prints.
`--impl reference` times the fp64 CPU oracle on a bounded sample of the same
workload (the only reference this method has).
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from chunked_lm_head_gb300 import workloads as WL  # noqa: E402

METRIC = "fused LM-head+CE fwd+bwd tokens/s; % of GB300 BF16 tensor peak (1 GPU)"
UNIT = "tokens/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                  "source": "fallback"}
# DRAM bytes (read + write) per launch of each GEMM kind on the 16K SFT
# workload at 4,096-row chunks: ncu's one-pass dram__bytes_read/write
# counters at full size, mean over one step's launches (dW: one store launch,
# three fp32 reduce-add launches), current kernels.
NCU_TRAFFIC_BYTES_PER_LAUNCH: dict[str, float | None] = {
    "bwd_dH": 5.17e9, "bwd_dW": 6.73e9}
NCU_TRAFFIC_WORKLOAD = "sft_16k"


def load_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        d["source"] = "measured"
        return d
    return dict(FALLBACK_PEAKS)


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_max(x: float, device=None) -> float:
    """Max of a per-rank scalar over all ranks (identity without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def algorithmic_bytes_step(N: int, nv: int, H: int, V: int, chunk_rows: int,
                           forward_rows: int) -> dict[str, float]:
    """Bytes each GEMM kind must move per step (bf16 operands, fp32 outputs)
    under the library's launch decomposition, for the forward + recomputing
    backward: forward launches of 4,096 rows, backward row blocks x
    vocabulary slabs from flce_backward_plan, over the non-ignored rows.
    Re-reads beyond one pass per launch are what ncu's DRAM counters add."""
    from chunked_lm_head_gb300 import _lib
    plan = _lib.flce_backward_plan(N, H, V, chunk_rows)
    R, S, splits = plan["rows_per_block"], plan["vocab_slabs"], plan["dh_splits"]
    B = max(1, -(-nv // R))  # row blocks with rows (compacted)
    Lf = max(1, -(-forward_rows // 4096))
    W, hb, Db = V * H * 2.0, H * 2.0, V * 2.0
    dh_out = nv * H * 2.0 if (splits == 1 and S == 1) else nv * H * 4.0 * splits * (2 * S - 1)
    out = {
        "fwd_logits_lse": Lf * W + forward_rows * hb,
        "bwd_dlogits": B * W + S * nv * hb + nv * Db,
        "bwd_dH": nv * Db + B * W + dh_out,
        "bwd_dW": nv * Db + S * nv * hb + B * V * H * 4.0 + (B - 1) * V * H * 4.0,
    }
    # a slab's dH and dW units in one launch, and a row block's dlogits, dH
    # and dW units in one launch (the library's defaults with several slabs)
    out["bwd_dH_dW"] = out["bwd_dH"] + out["bwd_dW"]
    out["bwd_pipeline"] = out["bwd_dlogits"] + out["bwd_dH_dW"]
    return out


def whole_job_rate(rows_per_rank: int, world: int, ms_per_step: float) -> float:
    """Tokens/s of the whole job: every rank's rows over the slowest rank's step time."""
    return world * rows_per_rank / (ms_per_step / 1e3)


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""

    FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None):
        self.uuid = uuid
        self.proc = None
        self.tmp = None

    def start(self):
        try:
            self.tmp = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=self.tmp, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.tmp.flush()
        self.tmp.seek(0)
        rows = [r.split(",") for r in self.tmp.read().strip().splitlines() if r.strip()]
        os.unlink(self.tmp.name)
        rows = [[c.strip() for c in r] for r in rows if len(r) >= 9]
        if self.uuid:
            mine = [r for r in rows if self.uuid in r[0]]
            rows = mine or rows
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except ValueError:
                continue
            for n, v in zip(names, r[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------ CPU baseline
def cpu_oracle_rate(inp, target_s: float = 12.0, max_rows: int = 4096) -> dict:
    """Time the fp64 oracle (fwd + bwd contributions) on a bounded row sample."""
    from oracle import flce_oracle as O  # test/benchmark-only use of the oracle
    wl = inp.wl
    nvalid = int((inp.targets != WL.IGNORE_INDEX).sum())
    g = 1.0 / max(nvalid, 1)

    def run(k):
        rows = WL.sample_rows(wl.N, k, seed=wl.seed + 7)
        t0 = time.perf_counter()
        O.rows_forward(inp.h, inp.W, inp.targets, rows)
        O.rows_backward(inp.h, inp.W, inp.targets, rows, inp.weights, g=g)
        return time.perf_counter() - t0

    k = 16
    dt = run(k)
    for _ in range(3):  # grow the sample until it is about target_s of work
        if dt >= target_s / 2 or k >= min(max_rows, wl.N):
            break
        k = int(min(max_rows, wl.N, max(2 * k, k * target_s / max(dt, 1e-3))))
        dt = run(k)
    try:
        cores = len(os.sched_getaffinity(0))
    except AttributeError:
        cores = os.cpu_count()
    return {"value": k / dt, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{k} of {wl.N} rows of {wl.name} (full V={wl.V}, H={wl.H}): fp64 logits, "
                      f"log-softmax, dlogits, dH rows and the rows' dW contribution; {dt:.1f} s",
            "seconds": dt, "rows": k}


def reference_arm(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    inp = WL.make_inputs(args.workload)
    vals, secs, rows = [], [], []
    info = None
    for i in range(args.warmup + args.steps):
        info = cpu_oracle_rate(inp, target_s=args.ref_step_s, max_rows=4096)
        if i >= args.warmup:
            vals.append(info["value"])
            secs.append(info["seconds"])
            rows.append(info["rows"])
    v = statistics.median(vals)
    wl = inp.wl
    # one step of this arm is a bounded sample of the workload's rows, so its
    # ms_per_step is the measured time of that sample (rows_per_step rows),
    # not a time for all N rows
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": statistics.median(secs) * 1e3,
            "rows_per_step": int(statistics.median(rows)),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": wl.name, "N": wl.N, "H": wl.H, "V": wl.V,
                       "chunk_rows": args.chunk_rows or wl.chunk_rows},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": info["cores"], "kind": "oracle",
                             "sample": info["sample"]},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU arm
GEMM_KINDS = ("fwd_logits_lse", "bwd_dlogits", "bwd_dH", "bwd_dW", "bwd_dH_dW", "bwd_pipeline", "kd_fwd_logits",
              "kd_bwd_dlogits", "jsd_fwd_terms", "jsd_bwd_dlogits")
# launch kinds that run the units of several kinds above (counted once in the step's FLOPs)
COMPOSITE_KINDS = ("bwd_dH_dW", "bwd_pipeline")


def gpu_arm(args):
    import torch
    from chunked_lm_head_gb300 import _lib

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    lib = _lib.load()
    wl = WL.WORKLOADS[args.workload]
    if args.shape:
        import dataclasses
        n_, h_, v_ = (int(x) for x in args.shape.split(","))
        wl = dataclasses.replace(wl, name=f"{wl.name}@{n_}x{h_}x{v_}", N=n_, H=h_, V=v_,
                                 packed_seqs=min(wl.packed_seqs, n_), grpo_seqs=0, prompt_len=0)
    chunk_rows = args.chunk_rows or wl.chunk_rows
    inp = WL.make_inputs(wl)
    N, H, V = wl.N, wl.H, wl.V
    dev = torch.device("cuda", local)

    def up(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)

    h = up(inp.h)
    W = up(inp.W)
    t = torch.from_numpy(inp.targets).to(dev)
    w = None if inp.weights is None else torch.from_numpy(inp.weights).to(dev)
    n_valid_host = int((inp.targets != WL.IGNORE_INDEX).sum())
    g = 1.0 / max(n_valid_host, 1)
    logp = torch.empty(N, dtype=torch.float32, device=dev)
    lse = torch.empty(N, dtype=torch.float32, device=dev)
    loss = torch.empty(1, dtype=torch.float32, device=dev)
    nv = torch.empty(1, dtype=torch.int64, device=dev)
    dH = torch.empty((N, H), dtype=torch.bfloat16, device=dev)
    dW = torch.empty((V, H), dtype=torch.float32, device=dev)
    ws_bytes = _lib.flce_workspace_bytes(N, H, V, chunk_rows)
    if args.fused:
        ws_bytes = max(ws_bytes, _lib.flce_forward_backward_workspace_bytes(N, H, V, chunk_rows))
    mem0 = torch.cuda.memory_allocated(dev)
    workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(dev)
    sh = stream.cuda_stream

    tf = None
    if args.transform:
        tf = _lib.make_transform({k: float(v) for k, v in
                                  (kv.split("=") for kv in args.transform.split(","))})
    tf_ptr = None if tf is None else ctypes.addressof(tf)
    Ht = args.kd_teacher_hidden
    if Ht:
        import dataclasses
        twl = dataclasses.replace(wl, name=wl.name + "_teacher", H=Ht, w_std=wl.w_std * 1.2,
                                  seed=wl.seed + 777)
        tinp = WL.make_inputs(twl)
        ht = up(tinp.h)
        Wt = up(tinp.W)
        lse_t = torch.empty(N, dtype=torch.float32, device=dev)
        kl_sm = torch.empty(N, dtype=torch.float32, device=dev)
        ws_bytes = max(ws_bytes, _lib.flce_kd_workspace_bytes(N, H, Ht, V, chunk_rows))
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)

    def check(name, s):
        if s != 0:
            raise RuntimeError(f"{name}: {_lib.STATUS_NAMES.get(s, s)}")

    if args.e4m3:
        if not args.forward_only or Ht:
            raise SystemExit("--e4m3 needs --forward-only (the backward is bf16)")
        h8 = torch.empty((N, H), dtype=torch.uint8, device=dev)
        hsc = torch.empty(N, dtype=torch.float32, device=dev)
        W8 = torch.empty((V, H), dtype=torch.uint8, device=dev)
        Wsc = torch.empty(V, dtype=torch.float32, device=dev)
        check("flce_quantize_e4m3_rows", lib.flce_quantize_e4m3_rows(
            W.data_ptr(), V, H, W8.data_ptr(), Wsc.data_ptr(), sh))  # frozen head: once

    def step():
        wp = None if w is None else w.data_ptr()
        if args.forward_only:
            if args.e4m3:
                check("flce_quantize_e4m3_rows", lib.flce_quantize_e4m3_rows(
                    h.data_ptr(), N, H, h8.data_ptr(), hsc.data_ptr(), sh))
                check("flce_forward_e4m3", lib.flce_forward_e4m3(
                    h8.data_ptr(), hsc.data_ptr(), W8.data_ptr(), Wsc.data_ptr(), t.data_ptr(), wp, N,
                    H, V, chunk_rows, -100, tf_ptr, logp.data_ptr(), lse.data_ptr(), loss.data_ptr(),
                    nv.data_ptr(), workspace.data_ptr(), ws_bytes, sh))
            else:
                check("flce_forward_ex", lib.flce_forward_ex(
                    h.data_ptr(), W.data_ptr(), t.data_ptr(), wp, N, H, V, chunk_rows, -100, tf_ptr,
                    logp.data_ptr(), lse.data_ptr(), loss.data_ptr(), nv.data_ptr(),
                    workspace.data_ptr(), ws_bytes, sh))
            return
        if Ht and args.jsd_beta:
            # a training step reads no lse of ignored rows: both heads skip them
            check("flce_jsd_forward_ex2", lib.flce_jsd_forward_ex2(
                h.data_ptr(), W.data_ptr(), H, ht.data_ptr(), Wt.data_ptr(), Ht, t.data_ptr(), wp, N,
                V, chunk_rows, -100, args.jsd_beta, tf_ptr, _lib.FORWARD_SKIP_IGNORED,
                logp.data_ptr(), lse.data_ptr(), lse_t.data_ptr(), kl_sm.data_ptr(), loss.data_ptr(),
                nv.data_ptr(), workspace.data_ptr(), ws_bytes, sh))
            check("flce_jsd_backward", lib.flce_jsd_backward(
                h.data_ptr(), W.data_ptr(), H, ht.data_ptr(), Wt.data_ptr(), Ht, t.data_ptr(), wp,
                lse.data_ptr(), lse_t.data_ptr(), kl_sm.data_ptr(), args.jsd_beta, g, dH.data_ptr(),
                dW.data_ptr(), N, V, chunk_rows, -100, tf_ptr, workspace.data_ptr(), ws_bytes, sh))
            return
        if Ht:
            check("flce_kd_forward_ex2", lib.flce_kd_forward_ex2(
                h.data_ptr(), W.data_ptr(), H, ht.data_ptr(), Wt.data_ptr(), Ht, t.data_ptr(), wp, N,
                V, chunk_rows, -100, tf_ptr, _lib.FORWARD_SKIP_IGNORED, logp.data_ptr(), lse.data_ptr(),
                lse_t.data_ptr(), loss.data_ptr(), nv.data_ptr(), workspace.data_ptr(), ws_bytes, sh))
            check("flce_kd_backward", lib.flce_kd_backward(
                h.data_ptr(), W.data_ptr(), H, ht.data_ptr(), Wt.data_ptr(), Ht, t.data_ptr(), wp,
                lse.data_ptr(), lse_t.data_ptr(), g, dH.data_ptr(), dW.data_ptr(), N, V, chunk_rows,
                -100, tf_ptr, workspace.data_ptr(), ws_bytes, sh))
            return
        if args.fused:
            # a training step needs no lse: without it the forward skips ignored rows
            check("flce_forward_backward", lib.flce_forward_backward(
                h.data_ptr(), W.data_ptr(), t.data_ptr(), wp, N, H, V, chunk_rows, -100, tf_ptr, 1.0,
                logp.data_ptr(), None, loss.data_ptr(), nv.data_ptr(), dH.data_ptr(),
                dW.data_ptr(), workspace.data_ptr(), ws_bytes, sh))
            return
        # the training step's forward (as the autograd wrapper runs it): the
        # backward reads lse of the non-ignored rows only, so the GEMM skips
        # the ignored ones
        check("flce_forward_ex2", lib.flce_forward_ex2(
            h.data_ptr(), W.data_ptr(), t.data_ptr(), wp, N, H, V, chunk_rows, -100, tf_ptr,
            _lib.FORWARD_SKIP_IGNORED, logp.data_ptr(), lse.data_ptr(), loss.data_ptr(), nv.data_ptr(),
            workspace.data_ptr(), ws_bytes, sh))
        check("flce_backward_ex", lib.flce_backward_ex(
            h.data_ptr(), W.data_ptr(), t.data_ptr(), wp, lse.data_ptr(), g, dH.data_ptr(),
            dW.data_ptr(), N, H, V, chunk_rows, -100, tf_ptr, workspace.data_ptr(), ws_bytes, sh))

    def barrier():
        if ws > 1:
            torch.distributed.barrier()

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    torch.cuda.synchronize(dev)
    st = _lib.flce_device_status(sh)
    if st != 0:
        raise RuntimeError(f"device status after warm-up: {_lib.STATUS_NAMES.get(st)}")
    extra_mem = torch.cuda.max_memory_allocated(dev) - mem0

    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    sampler = ClockSampler(uuid)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize(dev)
    sampler.start()
    time.sleep(0.3)  # let the sampler start before the timed region
    # per-launch CUDA events in a second pass of the same steps right after
    # the timed region (default), or inside it (--kernel-events timed)
    events_in_timed = args.kernel_events == "timed"
    _lib.profile_enable(events_in_timed)
    e0.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(args.steps):
            step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    clocks = sampler.stop()
    if not events_in_timed:
        _lib.profile_enable(True)
        with torch.cuda.stream(stream):
            for _ in range(args.steps):
                step()
        torch.cuda.synchronize(dev)
    prof = _lib.profile_read()
    _lib.profile_enable(False)
    st = _lib.flce_device_status(sh)
    if st != 0:
        raise RuntimeError(f"device status after timed steps: {_lib.STATUS_NAMES.get(st)}")
    ms = reduce_max(e0.elapsed_time(e1), device=dev)
    ms_step = ms / args.steps
    value = whole_job_rate(N, ws, ms_step)

    # ---- end to end through the public API with pinned host buffers
    from chunked_lm_head_gb300 import api
    h_host = torch.from_numpy(inp.h.view(np.int16)).pin_memory()
    t_host = torch.from_numpy(inp.targets).pin_memory()
    w_host = None if inp.weights is None else torch.from_numpy(inp.weights).pin_memory()
    loss_host = torch.empty(1, dtype=torch.float32).pin_memory()
    logp_host = torch.empty(N, dtype=torch.float32).pin_memory()
    # two device copies of the inputs: step i + 1's upload (copy stream) runs
    # while step i computes; step i's results are read back on the copy stream
    ins = [(torch.empty((N, H), dtype=torch.int16, device=dev), torch.empty(N, dtype=torch.int64, device=dev),
            None if w_host is None else torch.empty(N, dtype=torch.float32, device=dev)) for _ in range(2)]
    copy_stream = torch.cuda.Stream(device=dev)
    uploaded = [torch.cuda.Event() for _ in range(2)]
    consumed = [torch.cuda.Event() for _ in range(2)]

    def e2e_upload(i):
        h_e, t_e, w_e = ins[i % 2]
        with torch.cuda.stream(copy_stream):
            copy_stream.wait_event(consumed[i % 2])  # step i - 2 is done with this copy
            h_e.copy_(h_host, non_blocking=True)
            t_e.copy_(t_host, non_blocking=True)
            if w_e is not None:
                w_e.copy_(w_host, non_blocking=True)
            uploaded[i % 2].record(copy_stream)

    def e2e_compute(i):
        h_e, t_e, w_e = ins[i % 2]
        stream.wait_event(uploaded[i % 2])
        hb = h_e.view(torch.bfloat16)
        out = api.forward(hb, W, t_e, w_e, chunk_rows, workspace=workspace, skip_ignored=True)
        api.backward(hb, W, t_e, w_e, out["lse"], g, chunk_rows, workspace=workspace)
        consumed[i % 2].record(stream)
        with torch.cuda.stream(copy_stream):
            copy_stream.wait_event(consumed[i % 2])
            for x in (out["loss"], out["logp"]):
                x.record_stream(copy_stream)
            loss_host.copy_(out["loss"].view(1), non_blocking=True)
            logp_host.copy_(out["logp"], non_blocking=True)

    def e2e_run(n):
        e2e_upload(0)
        for i in range(n):
            if i + 1 < n:
                e2e_upload(i + 1)
            e2e_compute(i)
        stream.wait_stream(copy_stream)  # the last read-back is inside the region

    e2e_steps = max(3, min(args.steps, 10))
    if Ht or tf is not None or args.forward_only or args.fused:
        e2e_steps = 0
    e2e_ms = None
    if e2e_steps:
        with torch.cuda.stream(stream):
            e2e_run(2)
            torch.cuda.synchronize(dev)
            e2 = torch.cuda.Event(enable_timing=True)
            e3 = torch.cuda.Event(enable_timing=True)
            e2.record(stream)
            copy_stream.wait_event(e2)
            e2e_run(e2e_steps)
            e3.record(stream)
        torch.cuda.synchronize(dev)
        e2e_ms = reduce_max(e2.elapsed_time(e3), device=dev) / e2e_steps
    # ---- the same step through flce_forward_backward (no logits recompute),
    # timed after the headline with a workspace of its own
    fused_line = None
    if not (Ht or tf is not None or args.forward_only or args.fused or args.e4m3):
        fws = _lib.flce_forward_backward_workspace_bytes(N, H, V, chunk_rows)
        fwork = torch.empty(fws, dtype=torch.uint8, device=dev)

        def fstep():
            wp = None if w is None else w.data_ptr()
            check("flce_forward_backward", lib.flce_forward_backward(
                h.data_ptr(), W.data_ptr(), t.data_ptr(), wp, N, H, V, chunk_rows, -100, None, 1.0,
                logp.data_ptr(), None, loss.data_ptr(), nv.data_ptr(), dH.data_ptr(),
                dW.data_ptr(), fwork.data_ptr(), fws, sh))

        with torch.cuda.stream(stream):
            for _ in range(args.warmup):
                fstep()
            torch.cuda.synchronize(dev)
            f0 = torch.cuda.Event(enable_timing=True)
            f1 = torch.cuda.Event(enable_timing=True)
            f0.record(stream)
            for _ in range(args.steps):
                fstep()
            f1.record(stream)
        torch.cuda.synchronize(dev)
        f_ms = reduce_max(f0.elapsed_time(f1), device=dev) / args.steps
        fused_line = {"call": "flce_forward_backward", "value": whole_job_rate(N, ws, f_ms), "unit": UNIT,
                      "ms_per_step": f_ms,
                      "tflops_executed": 6.0 * n_valid_host * V * H / (f_ms / 1e3) / 1e12,
                      "note": "same loss, logp and gradients without the backward's logits recompute "
                              "(6 N V H tensor FLOPs instead of 8 N V H; no lse requested, so "
                              "ignored rows are skipped in every GEMM)"}
        del fwork
        st = _lib.flce_device_status(sh)
        if st != 0:
            raise RuntimeError(f"device status after the fused steps: {_lib.STATUS_NAMES.get(st)}")

    h2d = N * H * 2 + N * 8 + (0 if w_host is None else N * 4)
    d2h = 4 + N * 4

    # ---- roofline of the dominant kernel (algorithmic FLOPs / live event time)
    peaks = load_peaks()
    # algorithmic FLOPs: every GEMM of the training step covers the
    # non-ignored rows only (the backward needs no ignored row's lse, and
    # ignored rows have zero dlogits); so do the distillation steps, whose
    # targets mask rows the same way.  --forward-only covers every row.
    nv = n_valid_host
    flops_step = {"fwd_logits_lse": 2.0 * nv * V * H, "bwd_dlogits": 2.0 * nv * V * H,
                  "bwd_dH": 2.0 * nv * V * H, "bwd_dW": 2.0 * nv * V * H}
    if args.forward_only:
        flops_step = {"fwd_logits_lse": 2.0 * N * V * H}
    if args.fused:  # no recompute, no lse: the forward GEMM, dH and dW over the non-ignored
        # rows (bwd_dlogits is elementwise)
        flops_step = {"fwd_logits_lse": 2.0 * nv * V * H, "bwd_dH": 2.0 * nv * V * H,
                      "bwd_dW": 2.0 * nv * V * H}
    if Ht and args.jsd_beta:  # both heads twice in the forward (lse, then mixture terms)
        flops_step = {"kd_fwd_logits": 2.0 * nv * V * (H + Ht), "jsd_fwd_terms": 2.0 * nv * V * (H + Ht),
                      "jsd_bwd_dlogits": 2.0 * nv * V * (H + Ht),
                      "bwd_dH": 2.0 * nv * V * H, "bwd_dW": 2.0 * nv * V * H}
    elif Ht:  # distillation: both heads in the forward and the dlogits recompute
        flops_step = {"kd_fwd_logits": 2.0 * nv * V * (H + Ht), "kd_bwd_dlogits": 2.0 * nv * V * (H + Ht),
                      "bwd_dH": 2.0 * nv * V * H, "bwd_dW": 2.0 * nv * V * H}
    if "bwd_dH" in flops_step and "bwd_dW" in flops_step:  # one launch per slab for both
        flops_step["bwd_dH_dW"] = flops_step["bwd_dH"] + flops_step["bwd_dW"]
    if all(k in flops_step for k in ("bwd_dlogits", "bwd_dH", "bwd_dW")):  # one launch per row block
        flops_step["bwd_pipeline"] = flops_step["bwd_dlogits"] + flops_step["bwd_dH"] + flops_step["bwd_dW"]
    kern = {}
    for k, (tot_ms, n) in prof.items():
        if n:
            kern[k] = {"ms_per_step": tot_ms / args.steps, "launches_per_step": n / args.steps,
                       "share": None}
    tot = sum(v["ms_per_step"] for v in kern.values())
    for k in kern:
        kern[k]["share"] = kern[k]["ms_per_step"] / tot if tot else None
        if k in flops_step:
            kern[k]["tflops"] = flops_step[k] / (kern[k]["ms_per_step"] / 1e3) / 1e12
    dom = max((k for k in kern if k in GEMM_KINDS and k in flops_step), key=lambda k: kern[k]["ms_per_step"])
    peak_tf = peaks.get("bf16_tflops_sustained", peaks.get("bf16_tflops"))
    peak_note = "measured bf16_tflops_sustained (kernel timed inside a long step)"
    if args.e4m3:  # e4m3 dense rate = 2x bf16 (nominal 4.5 vs 2.25 PFLOP/s)
        peak_tf = 2.0 * peak_tf
        peak_note = "2 x measured bf16_tflops_sustained (e4m3 / bf16 nominal ratio)"
    launches_dom = kern[dom]["launches_per_step"]
    achieved = kern[dom]["tflops"]
    traffic = NCU_TRAFFIC_BYTES_PER_LAUNCH.get(dom) if (wl.name == NCU_TRAFFIC_WORKLOAD
                                                         and chunk_rows == 4096 and not Ht
                                                         and not args.fused
                                                         and tf is None and not args.forward_only
                                                         ) else None
    launch_s = kern[dom]["ms_per_step"] / launches_dom / 1e3
    bytes_launch = None
    if not (Ht or args.fused or args.forward_only or args.e4m3):
        bytes_launch = algorithmic_bytes_step(N, nv, H, V, chunk_rows, nv)[dom] / launches_dom
    roofline = {"bound": "tensor", "kernel": dom, "achieved": achieved, "peak": peak_tf,
                "unit": "TFLOP/s", "frac": achieved / peak_tf, "traffic": traffic,
                "peak_source": f"{peaks['source']}: {peak_note}",
                "flops_per_launch": flops_step[dom] / launches_dom,
                "algorithmic_bytes_per_launch": bytes_launch,
                "launch_ms": launch_s * 1e3}
    if bytes_launch is not None and bytes_launch / (peaks["hbm_gbs"] * 1e9) > \
            flops_step[dom] / launches_dom / (peak_tf * 1e12):
        # the kernel's bytes take longer at the copy bandwidth than its FLOPs
        # at the tensor rate: HBM-bound (e.g. the fp32 dW write at 256 rows)
        gbs = bytes_launch / launch_s / 1e9
        roofline.update({"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": gbs / peaks["hbm_gbs"],
                         "peak_source": f"{peaks['source']}: measured hbm_gbs (copy bandwidth)"})
    # the metric counts 8 N V H per step (forward, recompute, dH, dW over every
    # row); the GEMMs execute the FLOPs of flops_step (non-ignored rows)
    exec_tflops = sum(v for k, v in flops_step.items() if k not in COMPOSITE_KINDS) / (ms_step / 1e3) / 1e12
    step_tflops = exec_tflops
    if not (Ht or args.forward_only or args.fused):
        step_tflops = 8.0 * N * V * H / (ms_step / 1e3) / 1e12
    gpu_launches = int(round(sum(n for _, n in prof.values())))

    if rank == 0:
        cpu = None
        if (not args.no_cpu_baseline and ws == 1 and not args.shape and not Ht and tf is None
                and not args.forward_only):
            cpu = cpu_oracle_rate(inp, target_s=args.cpu_s)
            cpu.pop("seconds", None)
            cpu.pop("rows", None)
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "e4m3" if args.e4m3 else "bf16",
            "data": "synthetic",
            "config": {"workload": wl.name + (f"+kd_teacher_H{Ht}" if Ht else "")
                       + (f"+jsd_beta{args.jsd_beta:g}" if Ht and args.jsd_beta else "")
                       + (f"+transform({args.transform})" if args.transform else "")
                       + ("+forward_only" if args.forward_only else "") + ("+e4m3" if args.e4m3 else "")
                       + ("+fused_no_recompute(6NVH)" if args.fused else ""),
                       "N": N, "H": H, "V": V, "chunk_rows": chunk_rows,
                       "targets": wl.targets, "l2": "inputs larger than L2 (W alone "
                       f"{V * H * 2 / 1e9:.2f} GB > 129 MB); no flush",
                       "parallelism": "replicas" if ws > 1 else "single GPU"},
            "tflops": step_tflops,
            "tflops_executed": exec_tflops,
            "tensor_frac_of_peak": {"measured_burst": step_tflops / peaks["bf16_tflops"],
                                    "measured_sustained": step_tflops / peak_tf,
                                    "nominal_2250": step_tflops / 2250.0},
            "roofline": roofline,
            "kernels": kern,
            "cpu_baseline": cpu,
            "clocks": clocks,
            "e2e": None if e2e_ms is None else {
                "value": whole_job_rate(N, ws, e2e_ms), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms, "steps": e2e_steps,
                "boundary": "each step copies h, targets and weights from pinned host memory and "
                            "reads loss and logp back (on a copy stream, the next step's upload "
                            "overlapping this step's kernels; two device copies of the inputs); "
                            "W stays resident (a model parameter) and dH, dW stay on the device "
                            "(they feed the model's backward and the optimizer); no per-launch "
                            "profiling events in this region"},
            "gpu_launches": gpu_launches,
            "fused_no_recompute": fused_line,
            "kernel_events": args.kernel_events,
            "peak_extra_mem_bytes": int(extra_mem),
            "workspace_bytes": ws_bytes,
        }
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="sft_16k", choices=WL.WORKLOAD_ORDER)
    ap.add_argument("--chunk-rows", type=int, default=0)
    ap.add_argument("--shape", default="", help="N,H,V override of the workload's sizes (profiling small cases)")
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--cpu-s", type=float, default=12.0, help="target seconds of the CPU-oracle sample")
    ap.add_argument("--ref-step-s", type=float, default=8.0, help="reference arm: seconds per step")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--kernel-events", default="separate", choices=["timed", "separate"],
                    help="per-launch CUDA events in a second pass of the same K steps, right after "
                         "the timed steps, so that the timed steps run as a user's would (separate, "
                         "default: events between launches would serialise the GEMMs' programmatic "
                         "dependent launches); or inside the timed steps (timed)")
    ap.add_argument("--transform", default="",
                    help="logit transform, e.g. softcap=30,temperature=0.7 (flce_*_ex path)")
    ap.add_argument("--forward-only", action="store_true",
                    help="time the log-prob forward alone (e.g. reference / old-policy log-probs)")
    ap.add_argument("--e4m3", action="store_true",
                    help="with --forward-only: e4m3 operands (h quantised every step, W once)")
    ap.add_argument("--kd-teacher-hidden", type=int, default=0,
                    help="time the distillation step instead: the workload's head is the student, "
                         "a teacher head of this hidden size is added")
    ap.add_argument("--fused", action="store_true",
                    help="time flce_forward_backward (no logits recompute: 6 N V H tensor FLOPs) "
                         "instead of flce_forward + flce_backward")
    ap.add_argument("--jsd-beta", type=float, default=0.0,
                    help="with --kd-teacher-hidden: Jensen-Shannon distillation with this mixture "
                         "weight in (0, 1) instead of KL(teacher || student)")
    args = ap.parse_args()
    if args.jsd_beta and not (0.0 < args.jsd_beta < 1.0 and args.kd_teacher_hidden):
        ap.error("--jsd-beta needs --kd-teacher-hidden and a value in (0, 1)")
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        reference_arm(args)
    else:
        gpu_arm(args)


if __name__ == "__main__":
    main()
