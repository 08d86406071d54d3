"""The pipelined backward's unit schedule, checked on the host.

A pipelined row block runs as one launch whose SM pairs draw units in index
order and wait on dependency counters.  tests/pipe_schedule_check.cu decodes
every unit of the planner's launches for the library's workloads and of a
seeded sweep of plans, with the library's own decoding and counter helpers
compiled for the host, and checks that every wait's target is the number of
units adding to its counter, that all of them come earlier in the order (so
the launch completes on however many pairs are resident), that every counter
lies inside the launch's counter words, that each slab's units are decoded
exactly once, and that the hazards on the dlogits buffers and dH partials
(enumerated from the tiles each unit reads and writes) are all ordered.  For
the planner's plans over a sweep of problem sizes it checks the backward's
workspace layout (regions aligned and disjoint, inside the reported size, the
dlogits inside the O(chunk_rows x V) budget, a dH partial set for every
k-split) and the forward's (vocabulary splits covering every tile once,
regions aligned and disjoint).  It also checks the raster decoding every GEMM launch uses, over a
sweep of grid shapes and raster groups.  Needs nvcc, no GPU."""
import os
import subprocess

from chunked_lm_head_gb300 import build as B

HERE = os.path.dirname(os.path.abspath(__file__))


def test_pipelined_schedule_waits_only_on_earlier_units(tmp_path):
    exe = str(tmp_path / "pipe_schedule_check")
    src = os.path.join(HERE, "pipe_schedule_check.cu")
    cmd = [B.nvcc_path(), *B.ARCH_FLAGS, "-std=c++17", "-O1", "-I", B.INCLUDE, "-I", B.CSRC, src, "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, " ".join(cmd) + "\n" + r.stdout + r.stderr
    # the planner's defaults: no FLCE_* overrides from the environment
    env = {k: v for k, v in os.environ.items() if not k.startswith("FLCE_")}
    r = subprocess.run([exe], capture_output=True, text=True, timeout=600, env=env)
    assert r.returncode == 0 and r.stdout.startswith("ok:"), r.stdout + r.stderr
