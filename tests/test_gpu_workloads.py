"""GPU path against the FP64 oracle on the three large head-shape workloads,
at full size and in the launch configuration bench.py times:

* 512 seeded rows: lse, target logit and grad_X of each row are computed by
  the oracle one row at a time (row-local work) and compared element by
  element;
* n_valid exactly, from the labels;
* the loss, through an identity that holds at any size: loss * n_valid =
  sum over valid rows of (lse_i - z[i, y_i]), with z[i, y_i] from the oracle
  for every row (N*H work) and lse_i the library's own, itself checked on
  the sampled rows; for the Qwen3-0.6B-head workload the oracle also runs
  the whole forward and the loss is compared directly;
* grad_W and grad_b: the 512 sampled rows are run as a problem of their own
  (through lce_fused_fwd_bwd, and through lce_forward then lce_backward)
  and every output, including the full fp32 grad_W accumulator over all V
  rows, is compared with the oracle's;
* the full-size accumulation over chunks: the rows split in two halves,
  each run with grad_scale = n_valid(half) / n_valid(all) so that it uses the
  whole problem's 1/n_valid, must add up to the whole run's grad_W
  accumulator (additivity, a property of the sum over rows).
"""
import gc

import numpy as np
import pytest

import lce_inputs as L
import lm_head_linear_chunked_gb300 as lce
import oracle
from tests import gpu_util
from tests.gpu_util import BF16_GRAD_TOL, F32_ACC_TOL, LOSS_RTOL, LSE_ATOL, assert_grad, check_against_oracle, \
    host_f64

pytestmark = pytest.mark.gpu

BIG = [w for w in L.WORKLOADS if w.N >= 16384]
SAMPLE = 512


class Problem:
    """Host copies (bf16 bit patterns) and device tensors of one workload."""

    def __init__(self, w):
        import torch
        self.w = w
        self.Xh = torch.empty((w.N, w.H), dtype=torch.bfloat16, pin_memory=True)
        self.Wh = torch.empty((w.V, w.H), dtype=torch.bfloat16, pin_memory=True)
        L.x_into(w, self.Xh.data_ptr())
        L.w_into(w, self.Wh.data_ptr())
        self.y = L.labels(w)
        self.bh = None
        if w.has_bias:
            self.bh = torch.empty(w.V, dtype=torch.bfloat16)
            L.b_into(w, self.bh.data_ptr())
        self.X = self.Xh.cuda()
        self.W = self.Wh.cuda()
        self.b = self.bh.cuda() if self.bh is not None else None
        self.yd = torch.from_numpy(self.y).cuda()

    def bits(self, t):
        return t.view(__import__("torch").int16).numpy().view(np.uint16)


def _fused(X, W, b, y, chunk_rows, grad_scale=1.0):
    import torch
    out = lce.fused(X, W, b, y, chunk_rows=chunk_rows, grad_scale=grad_scale)
    assert lce.lce_check_status(out["ws"], torch.cuda.current_stream()) == 0
    del out["ws"]
    return out


@pytest.fixture(scope="module", params=BIG, ids=lambda w: w.name)
def problem(request):
    import torch
    p = Problem(request.param)
    yield p
    del p
    gc.collect()
    torch.cuda.empty_cache()


def test_sampled_rows_and_loss(problem):
    import torch
    w = problem.w
    out = _fused(problem.X, problem.W, problem.b, problem.yd, w.chunk_rows)
    Wb = problem.bits(problem.Wh)
    bb = problem.bits(problem.bh) if problem.bh is not None else None
    y = problem.y
    n_valid = int((y != L.IGNORE_INDEX).sum())
    assert int(out["n_valid"].item()) == n_valid
    s = 1.0 / n_valid

    rows = np.sort(np.random.default_rng(1000 + w.seed).choice(w.N, SAMPLE, replace=False))
    Xr = problem.bits(problem.Xh)[rows]
    ref = oracle.rows_forward(Xr, Wb, bb, y[rows])
    lse = host_f64(out["lse"])
    err = np.abs(lse[rows] - ref["lse"]).max()
    gpu_util._record("lse on 512 sampled rows (absolute)", err, LSE_ATOL)
    assert err <= LSE_ATOL, f"lse on sampled rows: max abs err {err}"
    gx_ref = oracle.rows_grad_X(Xr, Wb, bb, y[rows], ref["lse"], s)
    gx = host_f64(out["grad_X"][torch.from_numpy(rows).cuda()])
    assert_grad(gx, gx_ref, BF16_GRAD_TOL, "grad_X on sampled rows")

    # loss identity over all rows, with the oracle's target logits
    zt = oracle.target_logits(problem.bits(problem.Xh), Wb, bb, y)
    ok = y != L.IGNORE_INDEX
    expect = (lse[ok].sum() - zt[ok].sum()) / n_valid
    loss = float(out["loss"].item())
    gpu_util._record("loss identity over all rows (relative)", abs(loss - expect) / abs(expect), LOSS_RTOL)
    assert abs(loss - expect) <= LOSS_RTOL * abs(expect), (loss, expect)
    if w.N <= 16384:
        full = oracle.forward(problem.bits(problem.Xh), Wb, bb, y, block_rows=512, threads=1)
        assert abs(loss - full["loss"]) <= LOSS_RTOL * abs(full["loss"]), (loss, full["loss"])
        assert np.abs(lse - full["lse"]).max() <= LSE_ATOL


def test_sub_batch_all_outputs(problem):
    """The 512 sampled rows as their own problem: every output against the oracle."""
    import torch
    w = problem.w
    rows = np.sort(np.random.default_rng(1000 + w.seed).choice(w.N, SAMPLE, replace=False))
    idx = torch.from_numpy(rows).cuda()
    Xs = problem.X[idx].contiguous()
    ys = problem.yd[idx].contiguous()
    out = _fused(Xs, problem.W, problem.b, ys, w.chunk_rows)
    Wb = problem.bits(problem.Wh)
    bb = problem.bits(problem.bh) if problem.bh is not None else None
    ref = oracle.fused(problem.bits(problem.Xh)[rows], Wb, bb, problem.y[rows], block_rows=512, threads=1)
    check_against_oracle(out, ref, has_bias=w.has_bias)
    del out
    # the same rows through lce_forward, then lce_backward (which recomputes the logits)
    f = lce.forward(Xs, problem.W, problem.b, ys, chunk_rows=w.chunk_rows)
    assert lce.lce_check_status(f["ws"], torch.cuda.current_stream()) == 0
    check_against_oracle(f, ref, has_bias=w.has_bias, bwd=False)
    g = lce.backward(Xs, problem.W, problem.b, ys, f["lse"], chunk_rows=w.chunk_rows)
    assert lce.lce_check_status(g["ws"], torch.cuda.current_stream()) == 0
    check_against_oracle(g, ref, has_bias=w.has_bias, fwd=False)


def test_full_size_accumulation_is_additive(problem):
    w = problem.w
    y = problem.y
    n_all = int((y != L.IGNORE_INDEX).sum())
    whole = _fused(problem.X, problem.W, problem.b, problem.yd, w.chunk_rows)
    acc_whole = whole["grad_W_acc"]
    gb_whole = whole.get("grad_b_acc")
    del whole
    half = w.N // 2
    parts = []
    for r0, r1 in ((0, half), (half, w.N)):
        n_part = int((y[r0:r1] != L.IGNORE_INDEX).sum())
        o = _fused(problem.X[r0:r1], problem.W, problem.b, problem.yd[r0:r1], w.chunk_rows,
                   grad_scale=n_part / n_all)
        parts.append((o["grad_W_acc"], o.get("grad_b_acc")))
        del o
    tot = parts[0][0].double() + parts[1][0].double()
    ref = acc_whole.double()
    err = float((tot - ref).abs().max().item())
    scale = float(ref.abs().max().item())
    gpu_util._record("grad_W_acc additivity over row halves", err, F32_ACC_TOL * scale)
    assert err <= F32_ACC_TOL * scale, f"grad_W_acc additivity: {err} > 1e-4 * {scale}"
    if gb_whole is not None:
        tb = parts[0][1].double() + parts[1][1].double()
        assert float((tb - gb_whole.double()).abs().max().item()) <= F32_ACC_TOL * float(gb_whole.abs().max().item())
