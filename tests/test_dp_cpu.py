"""The data-parallel token split (chunked_lm_head_gb300.dp) on CPU with gloo,
2 ranks: the host logic (the count and loss-numerator all-reduces before the
gradient scale, the dW sum) checked against the unsharded oracle.  The
per-rank forward and backward here are the fp64 oracle (test infrastructure),
standing in for libflce, which needs a GPU."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from chunked_lm_head_gb300 import workloads as WL

# (N, H, V, rows of rank 0, ignored rows): uneven shards; in the second case
# every row of rank 1 is ignored
CASES = [(37, 24, 53, 20, [3, 11, 30]), (29, 16, 41, 21, list(range(21, 29)))]


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


class OracleStep:
    """Per-rank forward / backward from the oracle, on CPU tensors."""

    def forward(self, h, W, targets, weights):
        from oracle import flce_oracle as O
        f = O.forward(h.numpy(), W.numpy(), targets.numpy(), None if weights is None else weights.numpy())
        return {"logp": torch.from_numpy(f.logp), "lse": torch.from_numpy(f.lse),
                "loss": torch.tensor(f.loss, dtype=torch.float32), "n_valid": torch.tensor(f.n_valid)}

    def backward(self, h, W, targets, weights, lse, grad, count):
        from oracle import flce_oracle as O
        g = grad / max(int(count.reshape(-1)[0]), 1)
        b = O.backward(h.numpy(), W.numpy(), targets.numpy(), None if weights is None else weights.numpy(),
                       g=g)
        return torch.from_numpy(b.dH), torch.from_numpy(b.dW)


def _inputs(case):
    N, H, V, n0, ignored = case
    inp = WL.make_inputs(WL.custom("dp", N, H, V, 16, w_std=0.2, seed=77 + N))
    t = inp.targets.copy()
    t[ignored] = WL.IGNORE_INDEX
    w = np.random.default_rng(N).uniform(0.2, 1.8, N).astype(np.float32)
    return inp.h, inp.W, t, w


def _worker(rank, world, port, case, grad, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from chunked_lm_head_gb300 import dp
        h, W, t, w = _inputs(case)
        n0 = case[3]
        rows = slice(0, n0) if rank == 0 else slice(n0, None)
        out = dp.data_parallel_step(torch.from_numpy(h[rows]), torch.from_numpy(W), torch.from_numpy(t[rows]),
                                    torch.from_numpy(w[rows]), grad=grad, local=OracleStep())
        q.put((rank, float(out["loss"]), int(out["n_valid"]), out["dH"].numpy(), out["dW"].numpy()))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("case", CASES, ids=["uneven", "rank1_all_ignored"])
def test_two_rank_step_equals_the_unsharded_oracle(case):
    from oracle import flce_oracle as O
    grad = 0.75
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, case, grad, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted((q.get(timeout=120) for _ in range(2)), key=lambda x: x[0])
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    h, W, t, w = _inputs(case)
    ref = O.forward(h, W, t, w)
    refb = O.backward(h, W, t, w, g=grad / ref.n_valid)
    for rank, loss, nv, dH, dW in res:
        assert nv == ref.n_valid  # the global count, exact
        assert loss == pytest.approx(ref.loss, rel=1e-6)  # fp32 per-rank losses times their counts
        np.testing.assert_allclose(dW, refb.dW, rtol=1e-12, atol=1e-15)  # summed over the ranks
    dH = np.concatenate([res[0][3], res[1][3]])
    np.testing.assert_allclose(dH, refb.dH, rtol=1e-12, atol=1e-15)


def test_single_rank_step_is_the_local_step():
    """Without a process group the step is the rank's own forward and backward."""
    from chunked_lm_head_gb300 import dp
    from oracle import flce_oracle as O
    h, W, t, w = _inputs(CASES[0])
    out = dp.data_parallel_step(torch.from_numpy(h), torch.from_numpy(W), torch.from_numpy(t),
                                torch.from_numpy(w), grad=2.0, local=OracleStep())
    ref = O.forward(h, W, t, w)
    refb = O.backward(h, W, t, w, g=2.0 / ref.n_valid)
    assert int(out["n_valid"]) == ref.n_valid
    assert float(out["loss"]) == pytest.approx(ref.loss, rel=1e-6)
    np.testing.assert_allclose(out["dW"].numpy(), refb.dW, rtol=1e-12, atol=1e-15)
