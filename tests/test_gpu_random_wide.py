"""Seeded random shapes with hidden sizes of 1024-2560 against the FP64
oracle, in the pair form: chunks large enough that grad_X is not split over K
as a whole, so its tiles are 512 columns wide (H a multiple of 512) or 256
(otherwise), its last partial round of tiles is split over the vocabulary
when that pays, and grad_W's chunks between the first and the last read and
write the FP32 accumulator through TMA.  V takes every residue mod 8; the
ignored fraction, the bias and the chunk size are drawn too."""
import numpy as np
import pytest

import lce_inputs as L
import lm_head_linear_chunked_gb300 as lce
from tests.gpu_util import check_against_oracle
from tests.test_gpu_parity import oracle_of, random_problem, run_fused

pytestmark = pytest.mark.gpu


def _cases(n=10, seed=77):
    r = np.random.default_rng(seed)
    out = []
    for k in range(n):
        H = int(r.choice([1024, 1280, 1536, 2048, 2304, 2560]))
        cmin = -(-152 // (-(-H // 256))) * 128  # smallest chunk whose grad_X has a full round of tiles
        N = int(r.integers(cmin, 3 * cmin + 1))
        V = int(r.integers(1024, 6001))
        chunk = int(r.choice([0, int(r.integers(cmin, N + 1))]))
        bias = bool(r.integers(0, 2))
        ignore = float(r.choice([0.0, 0.1, 0.5]))
        out.append((k, N, H, V, chunk, bias, ignore))
    return out


def _plans(N, H, V, chunk, y, slots):
    """The tail plan of each chunk's grad_X launch: (tile columns, plan)."""
    C = lce.lce_chunk_rows(N, H, V, chunk)
    cols = 512 if H % 512 == 0 else 256
    out = []
    for r0 in range(0, N, C):
        rows = min(C, N - r0)
        valid = int((y[r0:r0 + rows] != L.IGNORE_INDEX).sum())
        grid = min(slots, -(-rows // 256) * -(-H // cols) * 8)
        out.append((cols, lce.lce_debug_gradx_tail_plan(-(-valid // 256) * -(-H // cols), grid, -(-V // 64), cols)))
    return out


def test_cases_reach_the_wide_tiles_and_the_tail_split():
    """On a 76-pair device, the drawn cases include split tails with both tile widths."""
    if lce.lce_gemm_pair_slots() != 76:
        pytest.skip("case coverage is computed for 76 pairs")
    seen = set()
    for k, N, H, V, chunk, bias, ignore in _cases():
        _, _, _, y = random_problem(9500 + k, N, 64, 8, bias=False, ignore_frac=ignore)
        for cols, plan in _plans(N, H, V, chunk, y, 76):
            if plan[1] > 0:
                seen.add(cols)
    assert seen == {256, 512}, seen


@pytest.mark.parametrize("case", _cases(), ids=lambda c: f"{c[0]}-N{c[1]}-H{c[2]}-V{c[3]}-c{c[4]}-b{int(c[5])}")
def test_random_wide_shape(case):
    k, N, H, V, chunk, bias, ignore = case
    prev = lce.lce_set_gemm_form("pair")
    try:
        X, W, b, y = random_problem(9500 + k, N, H, V, bias=bias, ignore_frac=ignore)
        out = run_fused(X, W, b, y, chunk)
    finally:
        lce.lce_set_gemm_form(prev)
    assert out["status"] == 0
    check_against_oracle(out, oracle_of(X, W, b, y), has_bias=bias)
