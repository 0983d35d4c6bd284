"""Writes oracle_regression.json: digests of the oracle's packed bytes and
fp64 outputs for small seeded cases.  Calls only the oracle and the seeded
input generators, never the CUDA library.  Re-run it only when a change to
the oracle's arithmetic is intended, and name the passage that justifies
the change in the commit message."""
import hashlib
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import synth  # noqa: E402

CASES = [  # (seed, rows, cols, n_keep, group, m)
    (1, 19, 512, 2, 128, 1),
    (2, 7, 768, 1, 256, 3),
    (3, 33, 256, 2, 64, 2),
    (4, 5, 1024, 1, 64, 1),
]


def digest(a: np.ndarray) -> str:
    return hashlib.sha256(np.ascontiguousarray(a).tobytes()).hexdigest()


def run_case(seed, rows, cols, n_keep, group, m):
    W = synth.weight_outliers(seed, rows, cols)
    x = synth.activations(seed + 100, m, cols)
    p = oracle.pack(W, n_keep, group)
    y = oracle.matvec(p, x)
    return {"vals": digest(p.vals), "idx": digest(p.idx),
            "scale": digest(p.scale), "zero": digest(p.zero),
            "y": y.ravel().tolist()}


def main():
    out = {"cases": []}
    for c in CASES:
        out["cases"].append({"args": list(c), "expect": run_case(*c)})
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)),
                        "oracle_regression.json")
    with open(path, "w") as f:
        json.dump(out, f, indent=1)
    print("wrote", path)


if __name__ == "__main__":
    main()
