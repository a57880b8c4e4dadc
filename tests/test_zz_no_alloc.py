"""lce_forward_static_ws, the forward entry point for callers that cannot
allocate device memory (it uses the library's own fixed scratch array), is
checked through the C ABI against lce_forward on the same inputs, on two
calls in a row.  This file is named to be collected last."""
import numpy as np
import pytest

import lce_inputs as L
import lm_head_linear_chunked_gb300 as lce
from tests.gpu_util import LOSS_RTOL, LSE_ATOL, dev_bf16, dev_i64

pytestmark = pytest.mark.gpu


def _problem(w):
    P = L.problem(w)
    return dev_bf16(P["X"]), dev_bf16(P["W"]), dev_bf16(P["b"]), dev_i64(P["y"])


def _forward_with_workspace(w, X, W, b, y):
    import torch
    out = lce.forward(X, W, b, y, chunk_rows=w.chunk_rows)
    assert lce.lce_check_status(out["ws"], torch.cuda.current_stream()) == 0
    return out


def _forward_static(w, X, W, b, y, chunk_rows):
    import torch
    loss = torch.full((1,), float("nan"), device="cuda")
    lse = torch.full((w.N,), float("nan"), device="cuda")
    n_valid = torch.full((1,), -1, dtype=torch.int64, device="cuda")
    s = torch.cuda.current_stream()
    lce.lce_forward_static_ws(w.N, w.H, w.V, X, W, b, y, -100, chunk_rows, loss, lse, n_valid, s)
    torch.cuda.synchronize()
    return {"loss": loss, "lse": lse, "n_valid": n_valid}


def _same(a, b):
    la, lb = float(a["loss"].item()), float(b["loss"].item())
    assert abs(la - lb) <= LOSS_RTOL * abs(lb), (la, lb)
    assert float((a["lse"] - b["lse"]).abs().max().item()) <= LSE_ATOL
    assert int(a["n_valid"].item()) == int(b["n_valid"].item())


def test_two_calls_in_a_row_match_lce_forward():
    # first call: the bias workload with the library choosing the chunk size;
    # second call, right after: the tiny workload with its own 256-row chunks
    for w, chunk in ((L.WORKLOADS[1], 0), (L.WORKLOADS[0], 256)):
        X, W, b, y = _problem(w)
        ref = _forward_with_workspace(w, X, W, b, y)
        got = _forward_static(w, X, W, b, y, chunk)
        _same(got, ref)


def test_too_large_is_rejected_before_any_work():
    with pytest.raises(lce.LCEError) as e:
        lce.lce_forward_static_ws(1 << 30, 64, 1024, 1 << 20, 1 << 20, None, 1 << 20, -100, 0,
                                  1 << 20, 1 << 20, None, None)
    assert e.value.status == 3  # LCE_ERR_WORKSPACE
    with pytest.raises(lce.LCEError) as e:
        lce.lce_forward_static_ws(131072, 4096, 151936, 1 << 20, 1 << 20, None, 1 << 20, -100, 8192,
                                  1 << 20, 1 << 20, None, None)
    assert e.value.status == 3
