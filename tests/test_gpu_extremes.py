"""Shapes at the edges of the supported range against the FP64 oracle: a
vocabulary above 2^18 (more than a thousand 256-column vocab tiles, odd V),
a 8192-wide hidden state, and chunks of one row next to chunks of all rows."""
import pytest

import lm_head_linear_chunked_gb300 as lce
from tests.gpu_util import check_against_oracle
from tests.test_gpu_parity import oracle_of, random_problem, run_fused

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("N,H,V,bias,chunk", [
    (1536, 128, 262147, False, 0),     # V > 2^18, V % 8 == 3
    (1200, 128, 200003, True, 512),    # the same with a bias and three chunks
    (640, 8192, 2048, False, 256),     # wide hidden state: 128 K slices per logits tile
    (5000, 64, 1000, False, 5000),     # one chunk of all rows (4096 or more: overlap planning, one chunk)
    (9, 64, 4104, True, 1),            # one-row chunks
])
def test_extreme_shape(N, H, V, bias, chunk):
    X, W, b, y = random_problem(8000 + N, N, H, V, bias=bias, ignore_frac=0.15)
    out = run_fused(X, W, b, y, chunk)
    assert out["status"] == 0
    ref = oracle_of(X, W, b, y)
    check_against_oracle(out, ref, has_bias=bias)
