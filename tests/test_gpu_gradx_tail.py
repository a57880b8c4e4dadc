"""grad_X of the pair form with its last partial round of tiles split over
the vocabulary (K), against the FP64 oracle.

Each grad_X tile of 256 rows x 256 columns (x 512 where H is a multiple of
512) runs the whole vocabulary as its K loop, so a launch whose tile count
leaves the last round of pairs partly idle splits the tiles of that round
into K slices and adds their partial sums in slice order.  The valid-row
counts of these cases are fixed (exact ignore counts), so the split each
chunk takes is known from the plan function the kernels use
(lce_debug_gradx_tail_plan); the cases cover, for both tile widths, a split
after whole rounds and a chunk that is all tail, and a ragged last chunk of
the overlapped schedule."""
import numpy as np
import pytest

import lce_inputs as L
import lm_head_linear_chunked_gb300 as lce
from tests.gpu_util import check_against_oracle
from tests.test_gpu_parity import oracle_of, run_fused

pytestmark = pytest.mark.gpu


def plans(N, H, V, chunk, y):
    """The tail plan of each chunk's grad_X launch (pair form)."""
    C = lce.lce_chunk_rows(N, H, V, chunk)
    slots = lce.lce_gemm_pair_slots()
    out = []
    for r0 in range(0, N, C):
        rows = min(C, N - r0)
        valid = int((y[r0:r0 + rows] != L.IGNORE_INDEX).sum())
        cols = 512 if H % 512 == 0 else 256  # the library's tile width
        tiles = -(-valid // 256) * -(-H // cols)
        grid = min(slots, -(-rows // 256) * -(-H // cols) * 8)
        out.append(lce.lce_debug_gradx_tail_plan(tiles, grid, -(-V // 64), cols))
    return out


def problem(seed, N, H, V, ignored):
    X = L.normal_bf16(seed, L.TID_X, 0, N * H, 1.0).reshape(N, H)
    W = L.normal_bf16(seed, L.TID_W, 0, V * H, 2.0 / np.sqrt(H)).reshape(V, H)
    y = L.zipf_labels(seed, N, V)
    y[L.random_ignore_positions(seed, N, ignored / N)] = L.IGNORE_INDEX
    return X, W, y


# (N, H, V, chunk rows, ignored rows, the plans on a 76-pair device: (whole tiles, split tiles, slices, k-blocks))
CASES = [
    # 512-column tiles; 5530 valid rows: 22 x 4 = 88 tiles, one whole round of 76, 12 tiles in 4 slices
    (6144, 2048, 4096, 0, 614, [(76, 12, 4, 16)]),
    # 512-column tiles; 1280 valid rows: 20 tiles, all split (7 slices of 19 k-blocks; the last of 14)
    (2560, 2048, 8192, 0, 1280, [(0, 20, 7, 19)]),
    # 256-column tiles (H = 2304); 2868 valid rows: 12 x 9 = 108 tiles, 76 whole, 32 in 2 slices
    (4096, 2304, 4096, 0, 1228, [(76, 32, 2, 32)]),
    # 256-column tiles; 1280 valid rows: 45 tiles, all split in 3 slices
    (2560, 2304, 4096, 0, 1280, [(0, 45, 3, 22)]),
    # 4096-row chunks (overlapped schedule), 512-column tiles, and a ragged last chunk of 1000 rows
    (9192, 2048, 4096, 4096, 919, None),
    # one column of 512-wide tiles (H = 512) in one 10240-row chunk: 36 tiles, all split in 2 slices
    (10240, 512, 4096, 10240, 1024, [(0, 36, 2, 32)]),
]


@pytest.mark.parametrize("N,H,V,chunk,ignored,want", CASES)
def test_gradx_tail_split_matches_oracle(N, H, V, chunk, ignored, want):
    X, W, y = problem(9100 + N + H, N, H, V, ignored)
    got_plans = plans(N, H, V, chunk, y)
    if lce.lce_gemm_pair_slots() == 76:
        if want is not None:
            assert got_plans == want
        assert any(p[1] > 0 for p in got_plans), got_plans
    prev = lce.lce_set_gemm_form("pair")
    try:
        out = run_fused(X, W, None, y, chunk)
    finally:
        lce.lce_set_gemm_form(prev)
    assert out["status"] == 0
    check_against_oracle(out, oracle_of(X, W, None, y), has_bias=False)


def test_gradx_tail_split_is_deterministic():
    X, W, y = problem(9177, 2560, 2048, 8192, 1280)
    prev = lce.lce_set_gemm_form("pair")
    try:
        a = run_fused(X, W, None, y, 0)
        b = run_fused(X, W, None, y, 0)
    finally:
        lce.lce_set_gemm_form(prev)
    assert a["status"] == 0 and b["status"] == 0
    for k in ("grad_X", "grad_W_acc", "lse"):
        assert bool((a[k] == b[k]).all().item()), k
