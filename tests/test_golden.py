"""The oracle against its stored regression fixture (CPU only)."""
import json
import os

import numpy as np

import oracle
from tests.golden import make_golden

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def test_oracle_regression_tiny():
    rec = json.load(open(os.path.join(HERE, "oracle_regression_tiny.json")))
    X, W, b, y = make_golden.inputs(rec["case"])
    assert y.tolist() == rec["labels"]
    out = oracle.fused(X, W, b, y, grad_scale=rec["case"]["grad_scale"], grad_output=rec["case"]["grad_output"])
    assert out["n_valid"] == rec["n_valid"]
    assert abs(out["loss"] - rec["loss"]) <= 1e-12 * abs(rec["loss"])
    np.testing.assert_allclose(out["lse"], rec["lse"], rtol=1e-12)
    np.testing.assert_allclose(out["grad_X"][0], rec["grad_X_row0"], rtol=1e-10, atol=1e-15)
    np.testing.assert_allclose(out["grad_W"][:, 5], rec["grad_W_col5"], rtol=1e-10, atol=1e-15)
    np.testing.assert_allclose(out["grad_b"], rec["grad_b"], rtol=1e-10, atol=1e-15)
