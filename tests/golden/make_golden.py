"""Writes tests/golden/oracle_small_cases.json: inputs and float64 oracle outputs of
two small seeded cases (one with a ragged length).  It calls only ``oracle`` and
numpy; no value in the file comes from the CUDA path.  Re-run it only when the
oracle's arithmetic is changed on purpose, and name the reason in the commit."""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)
import oracle  # noqa: E402


def case(seed, B, T, H, K, V):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, T, H, K))
    k = rng.standard_normal((B, T, H, K))
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, T, H, V))
    alpha = np.exp(-np.logaddexp(0.0, rng.standard_normal((B, T, H))))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((B, T, H))))
    s0 = 0.1 * rng.standard_normal((B, H, V, K))
    do = rng.standard_normal((B, T, H, V))
    dsT = 0.01 * rng.standard_normal((B, H, V, K))
    o, sT = oracle.gated_delta_fwd(q, k, v, alpha, beta, s0)
    g = oracle.gated_delta_bwd(q, k, v, alpha, beta, s0, do, dsT)
    arrs = dict(q=q, k=k, v=v, alpha=alpha, beta=beta, initial_state=s0, d_o=do,
                d_final_state=dsT, o=o, final_state=sT, **g)
    return {n: {"shape": list(a.shape), "data": [float(x) for x in a.ravel()]}
            for n, a in arrs.items()}


def main():
    out = {
        "note": "inputs and float64 oracle outputs; written by make_golden.py",
        "cases": {
            "B1_T8_H1_K4_V4": case(100, 1, 8, 1, 4, 4),
            "B1_T19_H2_K4_V6": case(101, 1, 19, 2, 4, 6),
        },
    }
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_small_cases.json")
    with open(path, "w") as f:
        json.dump(out, f, indent=0)
    print("wrote", path)


if __name__ == "__main__":
    main()
