"""bench.py's algorithmic bytes per GEMM role (the HBM side of the roofline)
on hand-computed cases, and which peak bounds each role at the pages'
256-row chunks and at the library's 8192-row chunks."""
import bench

H, V = 64, 1000


def test_single_chunk():
    b = bench.role_bytes(H, V, rows=[100], valid=[80], overlapped=False)
    assert b["logits_lse"] == 2 * 100 * H + 2 * V * H + 2 * 80 * V
    assert b["grad_x"] == 2 * 80 * V + 2 * V * H + 2 * 80 * H
    # first and last chunk at once: accumulator stored (4 VH) and its bf16 cast written (2 VH)
    assert b["grad_w"] == 2 * 80 * V + 2 * 80 * H + 6 * V * H


def test_chunks_with_and_without_valid_rows():
    rows, valid = [100, 100, 100, 50], [90, 0, 70, 0]
    b = bench.role_bytes(H, V, rows, valid, overlapped=True)
    fwd = sum(2 * r * H + 2 * V * H + 2 * v * V for r, v in zip(rows, valid)) + 4 * V * (90 + 0 + 70)
    assert b["logits_lse"] == fwd
    assert b["grad_x"] == (2 * 90 * V + 2 * V * H + 2 * 90 * H) + (2 * 70 * V + 2 * V * H + 2 * 70 * H)
    # chunk 0 stores, chunk 1 (no valid rows, in the middle) adds nothing, chunk 2 reads and writes,
    # chunk 3 (last, no valid rows) still reads, writes and casts
    gw = (2 * 90 * V + 2 * 90 * H + 4 * V * H) + (2 * 70 * V + 2 * 70 * H + 8 * V * H) + (8 + 2) * V * H
    assert b["grad_w"] == gw
    assert bench.role_bytes(H, V, rows, valid, overlapped=False)["logits_lse"] == fwd - 4 * V * (90 + 70)


def _bound(H, V, C, N, valid_frac):
    rows = [min(C, N - r0) for r0 in range(0, N, C)]
    valid = [int(r * valid_frac) for r in rows]
    b = bench.role_bytes(H, V, rows, valid, overlapped=True)
    t_tensor = 2.0 * N * H * V / (1693.4e12)
    return {k: ("hbm" if v / 6689.5e9 > t_tensor else "tensor") for k, v in b.items()}


def test_bounds_follow_the_chunk_size():
    # Qwen3-0.6B head at 256-row chunks: the FP32 accumulator's traffic makes grad_W bandwidth-bound
    assert _bound(1024, 151936, 256, 16384, 0.7)["grad_w"] == "hbm"
    # Qwen3-8B head at 8192-row chunks: all three products are bound by the tensor cores
    assert set(_bound(4096, 151936, 8192, 131072, 0.95).values()) == {"tensor"}
