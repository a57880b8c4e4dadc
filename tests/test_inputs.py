"""The seeded input generator (CPU only): the C twin against the numpy
definition, and the workload recipe's label and mask statistics."""
import math

import numpy as np
import pytest

import lce_inputs as L


@pytest.mark.parametrize("start,count", [(0, 1), (0, 1000), (1, 999), (12345, 77777), (2**33 + 5, 4097)])
def test_c_twin_matches_numpy_definition(start, count):
    for sigma in (1.0, 0.03125, 0.1):
        a = L.normal_bf16_reference(11, L.TID_W, start, count, sigma)
        b = L.normal_bf16(11, L.TID_W, start, count, sigma)
        assert np.array_equal(a, b)


def test_ranges_compose():
    whole = L.normal_bf16(5, L.TID_X, 0, 10001, 1.0)
    parts = np.concatenate([L.normal_bf16(5, L.TID_X, 0, 4567, 1.0),
                            L.normal_bf16(5, L.TID_X, 4567, 10001 - 4567, 1.0, threads=3)])
    assert np.array_equal(whole, parts)


def test_normal_moments():
    x = L.bf16_bits_to_f64(L.normal_bf16(3, L.TID_X, 0, 1 << 20, 1.0))
    assert abs(x.mean()) < 5e-3 and abs(x.std() - 1.0) < 5e-3
    w = L.bf16_bits_to_f64(L.normal_bf16(3, L.TID_W, 0, 1 << 20, 0.0625))
    assert abs(w.std() / 0.0625 - 1.0) < 5e-3


def test_streams_differ():
    a = L.normal_bf16(3, L.TID_X, 0, 4096, 1.0)
    b = L.normal_bf16(3, L.TID_W, 0, 4096, 1.0)
    c = L.normal_bf16(4, L.TID_X, 0, 4096, 1.0)
    assert (a != b).mean() > 0.9 and (a != c).mean() > 0.9


def test_bf16_rounding_is_nearest_even():
    f = np.array([1.0, 1.0 + 2**-8, 1.0 + 3 * 2**-8, 1.0 + 2**-9, -2.5, 0.0], dtype=np.float32)
    got = L.bf16_bits_to_f64(L.f32_to_bf16_bits(f))
    assert list(got) == [1.0, 1.0, 1.0 + 4 * 2**-8, 1.0, -2.5, 0.0]


def test_zipf_head_probability():
    V = 151936
    y = L.zipf_labels(0, 200000, V)
    h = sum(k ** -1.1 for k in range(1, V + 1))
    p0 = 1.0 / h
    assert abs(p0 - 0.132) < 2e-3
    sd = math.sqrt(p0 * (1 - p0) / len(y))
    assert abs((y == 0).mean() - p0) < 5 * sd
    assert abs((y == 1).mean() - 2 ** -1.1 * p0) < 5 * sd
    assert y.min() >= 0 and y.max() < V


@pytest.mark.parametrize("w", L.WORKLOADS, ids=lambda w: w.name)
def test_workload_masks(w):
    y = L.labels(w)
    n_ign = int((y == L.IGNORE_INDEX).sum())
    if w.mask == "random":
        assert n_ign == round(w.mask_frac * w.N)
    else:
        k = math.floor(w.mask_frac * w.seq_len)
        assert n_ign == k * w.seqs
        for s in range(w.seqs):
            seg = y[s * w.seq_len:(s + 1) * w.seq_len]
            assert np.all(seg[:k] == L.IGNORE_INDEX) and np.all(seg[k:] >= 0)
    assert np.all((y == L.IGNORE_INDEX) | ((y >= 0) & (y < w.V)))


def test_workload_shapes():
    names = [w.name for w in L.WORKLOADS]
    assert len(set(names)) == 5
    w3 = L.BY_NAME["qwen3-8b-head-N131072-H4096-V151936"]
    assert (w3.N, w3.H, w3.V, w3.chunk_rows, w3.seed) == (131072, 4096, 151936, 0, 3)
    assert abs(w3.w_sigma - 0.03125) < 1e-15
    assert w3.flops_fused() == 8.0 * 131072 * 4096 * 151936


def test_x_rows_match_whole_tensor():
    w = L.WORKLOADS[0]
    X = np.empty((w.N, w.H), dtype=np.uint16)
    L.x_into(w, X.ctypes.data)
    rows = np.array([0, 3, 511, 100])
    assert np.array_equal(L.x_rows(w, rows), X[rows])
