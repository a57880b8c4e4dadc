"""Seeded random shapes in both GEMM forms against the FP64 oracle: N, H, V,
the chunk size, the ignored fraction and the bias drawn at random (V from 1
to about 5000 with every residue mod 8, chunks from 1 row to more than N),
so that tile edges, ragged chunks, compaction and split-K grad_X meet in
combinations the hand-picked cases do not cover."""
import numpy as np
import pytest

import lm_head_linear_chunked_gb300 as lce
from tests.gpu_util import check_against_oracle
from tests.test_gpu_parity import oracle_of, random_problem, run_fused

pytestmark = pytest.mark.gpu


def _cases(n=16, seed=2024):
    r = np.random.default_rng(seed)
    out = []
    for k in range(n):
        N = int(r.integers(1, 3000))
        H = int(r.choice([64, 128, 192, 320, 512]))
        V = int(r.integers(1, 5200))
        chunk = int(r.choice([0, 1, int(r.integers(1, N + 1)), int(r.integers(1, 1100)), 4096]))
        bias = bool(r.integers(0, 2))
        ignore = float(r.choice([0.0, 0.1, 0.5, 0.97]))
        out.append((k, N, H, V, chunk, bias, ignore))
    return out


@pytest.mark.parametrize("form", ["pair", "single"])
@pytest.mark.parametrize("case", _cases(), ids=lambda c: f"{c[0]}-N{c[1]}-H{c[2]}-V{c[3]}-c{c[4]}-b{int(c[5])}")
def test_random_shape(form, case):
    k, N, H, V, chunk, bias, ignore = case
    prev = lce.lce_set_gemm_form(form)
    try:
        X, W, b, y = random_problem(7000 + k, N, H, V, bias=bias, ignore_frac=ignore)
        out = run_fused(X, W, b, y, chunk)
    finally:
        lce.lce_set_gemm_form(prev)
    assert out["status"] == 0
    ref = oracle_of(X, W, b, y)
    check_against_oracle(out, ref, has_bias=bias)
