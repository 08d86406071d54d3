"""Seeded synthetic inputs for the chunked LM-head cross-entropy.

This module only draws inputs: hidden states ``h[N,H]`` and the LM-head weight
``W[V,H]`` as bf16 bit patterns, int64 targets (with ``ignore_index`` rows) and
fp32 per-token weights.  It holds none of the method's arithmetic (no logits,
no softmax, no loss), so the fp64 oracle and the CUDA library can both be fed
from it without sharing any of the computation they are compared on.

Workload shapes follow the pages:
  * TRL v1.13 "Training Beyond 1M Tokens" guide, speed & memory section: one
    256-row chunk of a 248,320-word vocabulary at hidden size 2,048.
  * Unsloth "GRPO with 7x longer context", flattened sequence chunking: rows
    are the flattened (batch x context) tokens, completion tokens are the
    targets, prompt tokens carry no loss.
Synthetic stand-ins replace the datasets the pages train on (PG-19 books,
GRPO rollouts): only the shapes, the value distributions and the masking
structure are reproduced.

Random numbers: numpy's PCG64 bit generator, one independent stream per
block of ``_BLOCK`` elements (``SeedSequence([seed, stream, block])``), so the
same seed gives the same bits whatever the thread count.
"""
from __future__ import annotations

import dataclasses
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

IGNORE_INDEX = -100
_BLOCK = 1 << 22
_SEED_BASE = 0xF1CE0000

# stream ids (distinct RNG streams per tensor of one workload)
_S_H, _S_W, _S_T, _S_MASK, _S_LEN, _S_ADV = 1, 2, 3, 4, 5, 6


@dataclasses.dataclass(frozen=True)
class Workload:
    """Shape and input recipe of one synthetic workload."""

    name: str
    N: int
    H: int
    V: int
    chunk_rows: int
    h_std: float = 1.0
    w_std: float = 0.02
    targets: str = "uniform"  # "uniform" | "zipf"
    ignore_frac: float = 0.0  # fraction of rows (random) set to ignore_index
    packed_seqs: int = 0  # >0: packed sequences, first token of each ignored
    grpo_seqs: int = 0  # >0: equal sequences, per-sequence advantage weights
    prompt_len: int = 0  # GRPO: prompt prefix of each sequence ignored
    seed: int = _SEED_BASE

    @property
    def flops(self) -> int:
        """8*N*V*H: forward, backward recompute, dH and dW contractions."""
        return 8 * self.N * self.V * self.H


# The five workloads the pages' measurements and the method's use cases map
# to (tiny; TRL single chunk; packed SFT step; GRPO; long context).
WORKLOADS = {
    "tiny": Workload("tiny", 64, 64, 1000, 16, 1.0, 0.02, "uniform",
                     ignore_frac=0.05, seed=_SEED_BASE + 0),
    "single_chunk": Workload("single_chunk", 256, 2048, 248320, 256, 1.0, 0.02,
                             "uniform", seed=_SEED_BASE + 1),
    "sft_16k": Workload("sft_16k", 16384, 4096, 151936, 4096, 1.0, 0.015,
                        "zipf", packed_seqs=4, seed=_SEED_BASE + 2),
    "grpo_32k": Workload("grpo_32k", 32768, 4096, 128000, 4096, 1.0, 0.02,
                         "zipf", grpo_seqs=4, prompt_len=1024,
                         seed=_SEED_BASE + 3),
    "long_131k": Workload("long_131k", 131072, 2560, 151936, 256, 1.0, 0.02,
                          "zipf", seed=_SEED_BASE + 4),
}
WORKLOAD_ORDER = ["tiny", "single_chunk", "sft_16k", "grpo_32k", "long_131k"]


def _rng(seed: int, stream: int, block: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, stream, block])))


def _threads() -> int:
    try:
        n = len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        n = os.cpu_count() or 1
    return max(1, min(n, 32))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round finite fp32 values to bf16 (round to nearest, ties to even).

    Returns the uint16 bit patterns.  Inputs here are finite normals, so no
    NaN handling is needed.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = u + (np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1)))
    return (r >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp32."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal_bf16(seed: int, stream: int, count: int, std: float) -> np.ndarray:
    """``count`` draws of N(0, std^2), rounded fp32 -> bf16; uint16 bits."""
    out = np.empty(count, dtype=np.uint16)
    nblk = (count + _BLOCK - 1) // _BLOCK

    def fill(b: int) -> None:
        lo = b * _BLOCK
        hi = min(count, lo + _BLOCK)
        x = _rng(seed, stream, b).standard_normal(hi - lo, dtype=np.float32)
        x *= np.float32(std)
        out[lo:hi] = f32_to_bf16_bits(x)

    if nblk == 1:
        fill(0)
    else:
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(fill, range(nblk)))
    return out


def zipf_ids(rng: np.random.Generator, n: int, V: int, s: float = 1.1) -> np.ndarray:
    """Token ids with P(id = r-1) proportional to r^-s, r = 1..V (inverse CDF)."""
    ranks = np.arange(1, V + 1, dtype=np.float64)
    cdf = np.cumsum(ranks ** (-s))
    cdf /= cdf[-1]
    u = rng.random(n)
    ids = np.searchsorted(cdf, u, side="right")
    return np.minimum(ids, V - 1).astype(np.int64)


def packed_lengths(rng: np.random.Generator, nseq: int, total: int,
                   lo: int = 512, hi: int = 8192) -> np.ndarray:
    """Sequence lengths drawn uniformly from [lo, hi], rescaled to sum to total.

    Each length is scaled by total/sum and floored; the residue goes to the
    last sequence.
    """
    raw = rng.integers(lo, hi + 1, size=nseq).astype(np.int64)
    scaled = (raw * total) // int(raw.sum())
    scaled[-1] += total - int(scaled.sum())
    return scaled


@dataclasses.dataclass
class Inputs:
    """One workload's inputs, host-side (bf16 as uint16 bit patterns)."""

    wl: Workload
    h: np.ndarray  # [N,H] uint16 (bf16 bits)
    W: np.ndarray  # [V,H] uint16 (bf16 bits)
    targets: np.ndarray  # [N] int64
    weights: np.ndarray | None  # [N] float32 or None (all ones)
    seq_starts: np.ndarray  # first row of each sequence

    @property
    def n_ignored(self) -> int:
        return int((self.targets == IGNORE_INDEX).sum())


def make_targets(wl: Workload, N: int | None = None):
    """Targets, weights and sequence starts of a workload (no h or W)."""
    N = wl.N if N is None else N
    rng_t = _rng(wl.seed, _S_T)
    if wl.targets == "uniform":
        t = rng_t.integers(0, wl.V, size=N).astype(np.int64)
    elif wl.targets == "zipf":
        t = zipf_ids(rng_t, N, wl.V)
    else:
        raise ValueError(wl.targets)
    weights = None
    starts = np.array([0], dtype=np.int64)
    if wl.ignore_frac > 0:
        k = int(round(wl.ignore_frac * N))
        idx = _rng(wl.seed, _S_MASK).permutation(N)[:k]
        t[idx] = IGNORE_INDEX
    if wl.packed_seqs > 0:
        lens = packed_lengths(_rng(wl.seed, _S_LEN), wl.packed_seqs, N)
        starts = np.concatenate([[0], np.cumsum(lens)[:-1]]).astype(np.int64)
        t[starts] = IGNORE_INDEX
    if wl.grpo_seqs > 0:
        L = N // wl.grpo_seqs
        assert L * wl.grpo_seqs == N
        starts = np.arange(wl.grpo_seqs, dtype=np.int64) * L
        adv = _rng(wl.seed, _S_ADV).standard_normal(wl.grpo_seqs).astype(np.float32)
        weights = np.repeat(adv, L).astype(np.float32)
        for s in starts:
            t[s:s + wl.prompt_len] = IGNORE_INDEX
    return t, weights, starts


def make_inputs(wl: Workload | str) -> Inputs:
    """Draw all inputs of a workload (deterministic in ``wl.seed``)."""
    if isinstance(wl, str):
        wl = WORKLOADS[wl]
    h = normal_bf16(wl.seed, _S_H, wl.N * wl.H, wl.h_std).reshape(wl.N, wl.H)
    W = normal_bf16(wl.seed, _S_W, wl.V * wl.H, wl.w_std).reshape(wl.V, wl.H)
    t, weights, starts = make_targets(wl)
    return Inputs(wl, h, W, t, weights, starts)


def custom(name: str, N: int, H: int, V: int, chunk_rows: int = 256, *,
           seed: int = 12345, **kw) -> Workload:
    """A workload of arbitrary shape (tests use these for ragged tiles)."""
    return Workload(name, N, H, V, chunk_rows, seed=seed, **kw)


def sample_rows(N: int, k: int, seed: int = 0x5A11) -> np.ndarray:
    """k distinct row indices in [0,N), sorted (seeded)."""
    k = min(k, N)
    return np.sort(_rng(seed, 99).choice(N, size=k, replace=False)).astype(np.int64)
