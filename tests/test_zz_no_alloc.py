"""lce_forward_static_ws, the forward entry point for callers that cannot
allocate device memory (it uses the library's own fixed scratch array), is
checked through the C ABI against the FP64 oracle and against lce_forward on
the same inputs, on two calls in a row; on a problem whose forward workspace
at the default chunk size exceeds the array, so that the entry point picks
a smaller chunk itself; and with a bad label, which its status query and a
NaN loss must report.  This file is named to be collected last."""
import numpy as np
import pytest

import lce_inputs as L
import lm_head_linear_chunked_gb300 as lce
import oracle
from tests.gpu_util import LOSS_RTOL, LSE_ATOL, dev_bf16, dev_i64, host_f64

pytestmark = pytest.mark.gpu


def _problem(w):
    P = L.problem(w)
    return P, dev_bf16(P["X"]), dev_bf16(P["W"]), dev_bf16(P["b"]), dev_i64(P["y"])


def _forward_with_workspace(w, X, W, b, y, chunk_rows):
    import torch
    out = lce.forward(X, W, b, y, chunk_rows=chunk_rows)
    assert lce.lce_check_status(out["ws"], torch.cuda.current_stream()) == 0
    return out


def _forward_static(N, H, V, X, W, b, y, chunk_rows):
    import torch
    loss = torch.full((1,), float("nan"), device="cuda")
    lse = torch.full((N,), float("nan"), device="cuda")
    n_valid = torch.full((1,), -1, dtype=torch.int64, device="cuda")
    s = torch.cuda.current_stream()
    lce.lce_forward_static_ws(N, H, V, X, W, b, y, -100, chunk_rows, loss, lse, n_valid, s)
    status = lce.lce_static_ws_check_status(s)
    return {"loss": loss, "lse": lse, "n_valid": n_valid, "status": status}


def _against_oracle(got, ref):
    loss = float(got["loss"].item())
    assert abs(loss - ref["loss"]) <= LOSS_RTOL * abs(ref["loss"]), (loss, ref["loss"])
    assert np.abs(host_f64(got["lse"]) - ref["lse"]).max() <= LSE_ATOL
    assert int(got["n_valid"].item()) == ref["n_valid"]


def _same_bits(a, b):
    # lse and loss do not depend on the chunk size, bit for bit
    assert float(a["loss"].item()) == float(b["loss"].item())
    assert bool((a["lse"] == b["lse"]).all().item())
    assert int(a["n_valid"].item()) == int(b["n_valid"].item())


def test_two_calls_in_a_row_match_the_oracle_and_lce_forward():
    # first call: the bias workload with the library choosing the chunk size;
    # second call, right after: the tiny workload with its own 256-row chunks
    for w, chunk in ((L.WORKLOADS[1], 0), (L.WORKLOADS[0], 256)):
        P, X, W, b, y = _problem(w)
        got = _forward_static(w.N, w.H, w.V, X, W, b, y, chunk)
        assert got["status"] == 0
        _against_oracle(got, oracle.forward(P["X"], P["W"], P["b"], P["y"]))
        _same_bits(got, _forward_with_workspace(w, X, W, b, y, w.chunk_rows))


def test_chunk_search_when_the_default_chunk_does_not_fit():
    """Qwen3-0.6B head shape (N = 16384, V = 151936): the forward workspace
    at the default chunk is above the 32 MiB array, so chunk_rows = 0 makes
    the entry point search for the largest chunk that fits."""
    w = L.BY_NAME["qwen3-0.6b-head-N16384-H1024-V151936"]
    assert lce.lce_workspace_size(w.N, w.H, w.V, 0, w.has_bias, lce.WS_FORWARD) > lce.STATIC_SCRATCH_BYTES
    P, X, W, b, y = _problem(w)
    got = _forward_static(w.N, w.H, w.V, X, W, b, y, 0)
    assert got["status"] == 0
    _same_bits(got, _forward_with_workspace(w, X, W, b, y, 0))
    rows = np.sort(np.random.default_rng(2000).choice(w.N, 512, replace=False))
    ref = oracle.rows_forward(P["X"][rows], P["W"], P["b"], P["y"][rows])
    assert np.abs(host_f64(got["lse"])[rows] - ref["lse"]).max() <= LSE_ATOL
    assert int(got["n_valid"].item()) == int((P["y"] != L.IGNORE_INDEX).sum())


def test_bad_label_is_reported_then_cleared():
    w = L.WORKLOADS[0]
    P, X, W, b, y = _problem(w)
    ok = _forward_static(w.N, w.H, w.V, X, W, b, y, 256)
    assert ok["status"] == 0 and np.isfinite(float(ok["loss"].item()))
    bad_y = y.clone()
    bad_y[7] = w.V  # one label past the vocabulary
    bad = _forward_static(w.N, w.H, w.V, X, W, b, bad_y, 256)
    assert bad["status"] == 4  # LCE_ERR_LABEL_RANGE
    assert np.isnan(float(bad["loss"].item()))
    again = _forward_static(w.N, w.H, w.V, X, W, b, y, 256)
    assert again["status"] == 0
    _same_bits(again, ok)


def test_too_large_is_rejected_before_any_work():
    with pytest.raises(lce.LCEError) as e:
        lce.lce_forward_static_ws(1 << 30, 64, 1024, 1 << 20, 1 << 20, None, 1 << 20, -100, 0,
                                  1 << 20, 1 << 20, None, None)
    assert e.value.status == 3  # LCE_ERR_WORKSPACE
    with pytest.raises(lce.LCEError) as e:
        lce.lce_forward_static_ws(131072, 4096, 151936, 1 << 20, 1 << 20, None, 1 << 20, -100, 8192,
                                  1 << 20, 1 << 20, None, None)
    assert e.value.status == 3
