"""The stored oracle forwards of the GRPO and long-context workloads
(tests/golden/*_full_forward.npz) against the oracle itself and the
workload recipe, on the CPU: the recipe and the input digest match what this
machine draws, the count and the loss follow from the stored log-probs, and
the oracle recomputes the stored lse and logp of seeded sampled rows."""
import numpy as np
import pytest

from chunked_lm_head_gb300 import workloads as WL
from oracle import flce_oracle as O

from gpu_util import input_digest, load_golden


@pytest.mark.slow
@pytest.mark.parametrize("name", ["grpo_32k", "long_131k"])
def test_stored_full_forward_is_the_oracles(name):
    gold = load_golden(name)
    wl = WL.WORKLOADS[name]
    for k, v in gold["meta"]["workload"].items():
        assert getattr(wl, k) == v, k
    inp = WL.make_inputs(wl)
    assert gold["meta"]["input_sha256"] == input_digest(inp)
    m = inp.targets != WL.IGNORE_INDEX
    w = np.ones(wl.N) if inp.weights is None else inp.weights.astype(np.float64)
    assert gold["n_valid"] == int(m.sum())
    assert gold["lse"].shape == gold["logp"].shape == (wl.N,)
    assert np.all(gold["logp"][~m] == 0.0) and np.all(gold["logp"][m] < 0.0)
    assert np.all(np.isfinite(gold["lse"]))
    loss = -float(np.sum(m * w * gold["logp"])) / gold["n_valid"]
    assert loss == pytest.approx(gold["loss"], rel=1e-12)
    rows = WL.sample_rows(wl.N, 24, seed=wl.seed + 3)
    lse, logp = O.rows_forward(inp.h, inp.W, inp.targets, rows)
    np.testing.assert_allclose(gold["lse"][rows], lse, rtol=1e-13, atol=1e-12)
    np.testing.assert_allclose(gold["logp"][rows], logp, rtol=1e-13, atol=1e-12)
