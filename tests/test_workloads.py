"""The seeded input generators: determinism, masks, distributions, rounding."""
import numpy as np
import pytest
import torch

from chunked_lm_head_gb300 import workloads as WL


def test_bf16_rounding_matches_torch():
    r = np.random.default_rng(0)
    x = np.concatenate([r.standard_normal(100000).astype(np.float32) * s for s in (1e-3, 0.02, 1.0, 300.0)])
    # ties: values exactly half-way between two bf16 numbers
    base = (r.integers(0, 1 << 15, 2000).astype(np.uint32) << 16) | np.uint32(0x8000)
    x = np.concatenate([x, base.view(np.float32)[np.isfinite(base.view(np.float32))]])
    ours = WL.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    assert np.array_equal(WL.bf16_bits_to_f32(ours), torch.from_numpy(ours.view(np.int16)).view(torch.bfloat16).float().numpy())


def test_normal_generator_is_deterministic_and_blocked():
    a = WL.normal_bf16(5, 1, (1 << 22) + 12345, 0.02)
    b = WL.normal_bf16(5, 1, (1 << 22) + 12345, 0.02)
    c = WL.normal_bf16(6, 1, 1000, 0.02)
    assert np.array_equal(a, b) and not np.array_equal(a[:1000], c)
    x = WL.bf16_bits_to_f32(a).astype(np.float64)
    assert abs(x.mean()) < 1e-4 and x.std() == pytest.approx(0.02, rel=1e-2)


def test_tiny_workload_masks_three_rows():
    inp = WL.make_inputs("tiny")
    assert inp.h.shape == (64, 64) and inp.W.shape == (1000, 64)
    assert inp.n_ignored == 3 and inp.weights is None
    v = inp.targets[inp.targets != WL.IGNORE_INDEX]
    assert v.min() >= 0 and v.max() < 1000


def test_sft_workload_packing():
    wl = WL.WORKLOADS["sft_16k"]
    t, w, starts = WL.make_targets(wl)
    assert len(starts) == 4 and starts[0] == 0
    lens = np.diff(np.concatenate([starts, [wl.N]]))
    assert lens.sum() == 16384 and np.all(lens > 0)
    assert np.all(t[starts] == WL.IGNORE_INDEX)
    assert int((t != WL.IGNORE_INDEX).sum()) == 16380
    assert w is None


def test_grpo_workload_prompt_mask_and_advantages():
    wl = WL.WORKLOADS["grpo_32k"]
    t, w, starts = WL.make_targets(wl)
    assert int((t != WL.IGNORE_INDEX).sum()) == 28672
    assert w.dtype == np.float32 and len(np.unique(w)) == 4
    for s in starts:
        assert np.all(t[s:s + 1024] == WL.IGNORE_INDEX) and np.all(t[s + 1024:s + 8192] >= 0)
        assert np.all(w[s:s + 8192] == w[s])


def test_zipf_targets_follow_power_law():
    rng = np.random.Generator(np.random.PCG64(3))
    V = 151936
    ids = WL.zipf_ids(rng, 2_000_000, V)
    Hn = np.sum(np.arange(1, V + 1, dtype=np.float64) ** -1.1)
    for r in (1, 2, 10):
        expect = r ** -1.1 / Hn
        got = np.mean(ids == r - 1)
        assert got == pytest.approx(expect, rel=0.05)
    assert ids.min() >= 0 and ids.max() < V


def test_long_context_workload_has_no_mask():
    wl = WL.WORKLOADS["long_131k"]
    t, w, _ = WL.make_targets(wl)
    assert len(t) == 131072 and np.all(t >= 0) and w is None


def test_sample_rows_distinct_sorted():
    r = WL.sample_rows(1000, 100)
    assert len(np.unique(r)) == 100 and np.all(np.diff(r) > 0)
