"""The FP32 grad_W accumulation over many chunks against the FP64 oracle on
ALL rows of a large problem: a seeded 64-column slice of grad_W (every
vocabulary row), as the pages' FP32 accumulation across chunks requires
(LlamaFactory PR #10762 analysis page, section 4: grad_weight accumulated
in FP32 over the chunks, then cast to the weight dtype).

* Qwen3-0.6B head shape (N = 16384, H = 1024, V = 151936) at its 256-row
  chunks: 64 chunks, each adding its tile products into the accumulator
  through the TMA add; through the fused call and through lce_forward then
  lce_backward (which recomputes the logits).
* The first 12288 rows of the Qwen3-8B head shape (H = 4096, V = 151936) in
  three chunks of 4096 rows: the fused call's overlapped schedule, where each
  chunk's forward turns the previous chunk's kept exponentials into the
  softmax, with its two alternating buffers.

The oracle computes the slice from the full logits one row block at a time
(oracle.grad_W_columns), with lse and the loss of all rows on the way."""
import gc

import numpy as np
import pytest

import lce_inputs as L
import lm_head_linear_chunked_gb300 as lce
import oracle
from tests import gpu_util
from tests.gpu_util import BF16_GRAD_TOL, F32_ACC_TOL, LOSS_RTOL, LSE_ATOL, assert_grad, dev_bf16, dev_i64, \
    host_f64

pytestmark = pytest.mark.gpu

COLS = 64


def _inputs(w, rows):
    X = np.empty((rows, w.H), dtype=np.uint16)
    L.x_into(w, X.ctypes.data, 0, rows)
    Wb = np.empty((w.V, w.H), dtype=np.uint16)
    L.w_into(w, Wb.ctypes.data)
    y = L.labels(w)[:rows].copy()
    return X, Wb, y


def _check(out, ref, h0, what):
    import torch
    s = torch.cuda.current_stream()
    assert lce.lce_check_status(out["ws"], s) == 0
    if "loss" in out:
        loss = float(out["loss"].item())
        gpu_util._record(f"{what}: loss (relative)", abs(loss - ref["loss"]) / abs(ref["loss"]), LOSS_RTOL)
        assert abs(loss - ref["loss"]) <= LOSS_RTOL * abs(ref["loss"]), (loss, ref["loss"])
        err = np.abs(host_f64(out["lse"]) - ref["lse"]).max()
        gpu_util._record(f"{what}: lse of all rows (absolute)", err, LSE_ATOL)
        assert err <= LSE_ATOL
    assert_grad(host_f64(out["grad_W_acc"][:, h0:h0 + COLS]), ref["grad_W_cols"], F32_ACC_TOL,
                f"{what}: grad_W_acc columns {h0}:{h0 + COLS}, all rows (fp32)")
    assert_grad(host_f64(out["grad_W"][:, h0:h0 + COLS]), ref["grad_W_cols"], BF16_GRAD_TOL,
                f"{what}: grad_W columns {h0}:{h0 + COLS}, all rows (bf16)")


def test_qwen3_06b_head_256_row_chunks_full_rows_slice():
    import torch
    w = L.BY_NAME["qwen3-0.6b-head-N16384-H1024-V151936"]
    X, Wb, y = _inputs(w, w.N)
    h0 = int(np.random.default_rng(3000 + w.seed).integers(0, w.H - COLS + 1))
    ref = oracle.grad_W_columns(X, Wb, None, y, h0, h0 + COLS, block_rows=256, threads=4)
    Xd, Wd, yd = dev_bf16(X), dev_bf16(Wb), dev_i64(y)
    assert lce.lce_chunk_rows(w.N, w.H, w.V, w.chunk_rows) == 256
    out = lce.fused(Xd, Wd, None, yd, chunk_rows=w.chunk_rows)
    _check(out, ref, h0, "Qwen3-0.6B head fused")
    del out
    f = lce.forward(Xd, Wd, None, yd, chunk_rows=w.chunk_rows)
    g = lce.backward(Xd, Wd, None, yd, f["lse"], chunk_rows=w.chunk_rows)
    _check(g, ref, h0, "Qwen3-0.6B head backward (recompute)")
    del f, g
    gc.collect()
    torch.cuda.empty_cache()


def test_qwen3_8b_head_prefix_three_overlapped_chunks_full_rows_slice():
    import torch
    w = L.BY_NAME["qwen3-8b-head-N131072-H4096-V151936"]
    rows, chunk = 3 * 4096, 4096
    X, Wb, y = _inputs(w, rows)
    h0 = int(np.random.default_rng(3000 + w.seed).integers(0, w.H - COLS + 1))
    ref = oracle.grad_W_columns(X, Wb, None, y, h0, h0 + COLS, block_rows=128, threads=4)
    Xd, Wd, yd = dev_bf16(X), dev_bf16(Wb), dev_i64(y)
    # the fused call's default workspace holds two chunks of kept exponentials:
    # the overlapped schedule
    assert lce.lce_workspace_size(rows, w.H, w.V, chunk, False, lce.WS_FUSED) > \
        lce.lce_workspace_size(rows, w.H, w.V, chunk, False, lce.WS_FUSED_MIN)
    out = lce.fused(Xd, Wd, None, yd, chunk_rows=chunk)
    _check(out, ref, h0, "Qwen3-8B head, 3 x 4096 rows, overlapped")
    del out
    gc.collect()
    torch.cuda.empty_cache()
