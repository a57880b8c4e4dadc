"""Writes oracle_regression_tiny.json: the FP64 oracle's outputs on one tiny
seeded problem, so that a later change to the oracle's arithmetic shows up
as a failing test.  Calls only oracle/ and the seeded input generator.

Run from the repository root:  python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import lce_inputs as L  # noqa: E402
import oracle  # noqa: E402

CASE = {"N": 20, "H": 64, "V": 100, "seed": 123, "w_sigma": 0.25, "b_sigma": 0.1,
        "ignore_rows": [3, 11, 12], "grad_scale": 0.5, "grad_output": 2.0}


def inputs(case=CASE):
    N, H, V, seed = case["N"], case["H"], case["V"], case["seed"]
    X = L.normal_bf16(seed, L.TID_X, 0, N * H, 1.0).reshape(N, H)
    W = L.normal_bf16(seed, L.TID_W, 0, V * H, case["w_sigma"]).reshape(V, H)
    b = L.normal_bf16(seed, L.TID_B, 0, V, case["b_sigma"])
    y = L.zipf_labels(seed, N, V)
    y[case["ignore_rows"]] = L.IGNORE_INDEX
    return X, W, b, y


def main():
    X, W, b, y = inputs()
    out = oracle.fused(X, W, b, y, grad_scale=CASE["grad_scale"], grad_output=CASE["grad_output"])
    rec = {
        "what": "FP64 oracle outputs on a tiny seeded problem (regression fixture, written by make_golden.py)",
        "case": CASE,
        "labels": y.tolist(),
        "loss": out["loss"],
        "n_valid": out["n_valid"],
        "lse": out["lse"].tolist(),
        "grad_X_row0": out["grad_X"][0].tolist(),
        "grad_W_col5": out["grad_W"][:, 5].tolist(),
        "grad_b": out["grad_b"].tolist(),
    }
    with open(os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_regression_tiny.json"), "w") as f:
        json.dump(rec, f, indent=1)


if __name__ == "__main__":
    main()
