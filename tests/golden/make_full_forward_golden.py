"""Write the oracle's full forward of the two largest workloads to tests/golden/.

The GRPO workload (32,768 x 4,096 x 128,000) and the long-context workload
(131,072 x 2,560 x 151,936) need 3.4e13 and 1.0e14 fp64 multiply-adds for
their forward alone, minutes of CPU time, so their per-row log-sum-exp and
log-probs, the masked (weighted) mean loss and the ignored-token count are
computed once here and stored.  The GPU parity tests read them back to check
every row's logp and lse, the loss, and the vocabulary-row slices of dW (which
need every row's lse).

Only the oracle and the seeded input generator are called: no value comes
from the CUDA library.  Each file records the workload recipe and a SHA-256
digest of the generated input bytes, so a test can tell whether the machine it
runs on drew the same inputs.

    python tests/golden/make_full_forward_golden.py grpo_32k long_131k
"""
from __future__ import annotations

import hashlib
import json
import os
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from chunked_lm_head_gb300 import workloads as WL  # noqa: E402  (seeded inputs only)
from oracle import flce_oracle as O  # noqa: E402

HERE = os.path.dirname(os.path.abspath(__file__))


def input_digest(inp) -> str:
    """SHA-256 over h, W, targets and weights as generated (little-endian bytes)."""
    d = hashlib.sha256()
    for a in (inp.h, inp.W, inp.targets):
        d.update(np.ascontiguousarray(a).tobytes())
    if inp.weights is not None:
        d.update(np.ascontiguousarray(inp.weights).tobytes())
    return d.hexdigest()


def golden_path(name: str) -> str:
    return os.path.join(HERE, f"{name}_full_forward.npz")


def write(name: str, chunk_rows: int = 2048) -> None:
    wl = WL.WORKLOADS[name]
    t0 = time.time()
    inp = WL.make_inputs(wl)
    digest = input_digest(inp)
    ref = O.forward(inp.h, inp.W, inp.targets, inp.weights, chunk_rows=chunk_rows)
    meta = {
        "what": "oracle (fp64 numpy) full forward: lse and logp of every row, loss, n_valid",
        "workload": {k: getattr(wl, k) for k in ("name", "N", "H", "V", "chunk_rows", "h_std",
                                                  "w_std", "targets", "ignore_frac", "packed_seqs",
                                                  "grpo_seqs", "prompt_len", "seed")},
        "input_sha256": digest,
        "oracle_chunk_rows": chunk_rows,
        "command": "python tests/golden/make_full_forward_golden.py " + name,
    }
    np.savez_compressed(golden_path(name), lse=ref.lse, logp=ref.logp,
                        n_valid=np.int64(ref.n_valid), loss=np.float64(ref.loss),
                        meta=np.array(json.dumps(meta)))
    print(f"{name}: n_valid {ref.n_valid}, loss {ref.loss:.12g}, {time.time() - t0:.0f} s",
          flush=True)


def load(name: str) -> dict:
    """The stored arrays and the recipe (``meta`` parsed from JSON)."""
    with np.load(golden_path(name)) as z:
        out = {k: z[k] for k in z.files}
    out["meta"] = json.loads(str(out["meta"]))
    out["n_valid"] = int(out["n_valid"])
    out["loss"] = float(out["loss"])
    return out


if __name__ == "__main__":
    for n in sys.argv[1:] or ["grpo_32k", "long_131k"]:
        write(n)
