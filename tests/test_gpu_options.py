"""The option flags of the _ex entry points on the GPU, against the FP64
oracle: reduction "sum" (loss = sum over valid rows, gradient scale without
the division by n_valid) and accumulation of the FP32 gradient accumulators
across calls (gradient accumulation over micro-batches)."""
import pytest

import lm_head_linear_chunked_gb300 as lce
import oracle
from tests.gpu_util import F32_ACC_TOL, assert_grad, check_against_oracle, dev_bf16, dev_i64
from tests.test_gpu_parity import random_problem

pytestmark = pytest.mark.gpu


def _dev(X, W, b, y):
    return dev_bf16(X), dev_bf16(W), dev_bf16(b), dev_i64(y)


def _ok(out):
    import torch
    assert lce.lce_check_status(out["ws"], torch.cuda.current_stream()) == 0


@pytest.mark.parametrize("N,H,V,bias,chunk", [(300, 128, 1000, True, 128), (1024, 256, 8192, False, 0)])
def test_sum_reduction_fused(N, H, V, bias, chunk):
    X, W, b, y = random_problem(50 + N, N, H, V, bias, ignore_frac=0.25)
    Xd, Wd, bd, yd = _dev(X, W, b, y)
    out = lce.fused(Xd, Wd, bd, yd, chunk_rows=chunk, grad_scale=0.5, reduction="sum")
    _ok(out)
    ref = oracle.fused(X, W, b, y, grad_scale=0.5, reduction="sum")
    check_against_oracle(out, ref, has_bias=bias)


def test_sum_reduction_forward_and_backward():
    X, W, b, y = random_problem(61, 700, 192, 4100, True, ignore_frac=0.3)
    Xd, Wd, bd, yd = _dev(X, W, b, y)
    f = lce.forward(Xd, Wd, bd, yd, chunk_rows=256, reduction="sum")
    _ok(f)
    ref = oracle.fused(X, W, b, y, reduction="sum")
    check_against_oracle(f, ref, has_bias=True, bwd=False)
    g = lce.backward(Xd, Wd, bd, yd, f["lse"], chunk_rows=256, reduction="sum")
    _ok(g)
    check_against_oracle(g, ref, has_bias=True, fwd=False)


@pytest.mark.parametrize("entry", ["fused", "backward"])
@pytest.mark.parametrize("reduction", ["mean", "sum"])
def test_accumulate_over_micro_batches(entry, reduction):
    """Three micro-batches, the first written and the others added: the FP32
    accumulators end at the whole batch's gradient.  With the mean, each
    micro-batch passes grad_scale = its share of the valid rows, as a trainer
    normalising by the global count does."""
    import torch
    X, W, b, y = random_problem(71, 900, 128, 3000, True, ignore_frac=0.3)
    n_all = int((y != -100).sum())
    Xd, Wd, bd, yd = _dev(X, W, b, y)
    cuts = [0, 250, 600, 900]
    acc_W = acc_b = None
    for k in range(3):
        r0, r1 = cuts[k], cuts[k + 1]
        n_k = int((y[r0:r1] != -100).sum())
        gs = n_k / n_all if reduction == "mean" else 1.0
        xs, ys = Xd[r0:r1].contiguous(), yd[r0:r1].contiguous()
        kw = dict(chunk_rows=128, grad_scale=gs, reduction=reduction, accumulate=k > 0, grad_W_acc=acc_W,
                  grad_b_acc=acc_b)
        if entry == "fused":
            out = lce.fused(xs, Wd, bd, ys, **kw)
        else:
            f = lce.forward(xs, Wd, bd, ys, chunk_rows=128)
            _ok(f)
            out = lce.backward(xs, Wd, bd, ys, f["lse"], **kw)
        _ok(out)
        acc_W, acc_b = out["grad_W_acc"], out["grad_b_acc"]
    ref = oracle.fused(X, W, b, y, reduction=reduction)
    s = 1.0 / n_all if reduction == "mean" else 1.0
    assert_grad(acc_W, ref["grad_W"], F32_ACC_TOL, "accumulated grad_W_acc")
    assert_grad(acc_b, ref["grad_b"], F32_ACC_TOL, "accumulated grad_b_acc")
    # the bf16 outputs of the last call are the cast of the totals
    assert torch.equal(out["grad_W"], acc_W.to(torch.bfloat16))
    assert torch.equal(out["grad_b"], acc_b.to(torch.bfloat16))


def test_accumulate_adds_to_existing_values():
    """An accumulator that starts at A ends at A + this call's gradient."""
    import torch
    X, W, b, y = random_problem(81, 256, 64, 512, False)
    Xd, Wd, bd, yd = _dev(X, W, b, y)
    base = lce.fused(Xd, Wd, None, yd, chunk_rows=100)
    _ok(base)
    start = torch.randn(W.shape, dtype=torch.float32, device="cuda")
    acc = start.clone()
    out = lce.fused(Xd, Wd, None, yd, chunk_rows=100, accumulate=True, grad_W_acc=acc)
    _ok(out)
    err = float((acc.double() - (start.double() + base["grad_W_acc"].double())).abs().max().item())
    assert err <= 1e-6 * float(start.abs().max().item()), err


def test_accumulate_needs_the_accumulators():
    X, W, b, y = random_problem(82, 64, 64, 128, True)
    Xd, Wd, bd, yd = _dev(X, W, b, y)
    with pytest.raises(ValueError):
        lce.fused(Xd, Wd, bd, yd, accumulate=True)


def test_autograd_sum_reduction():
    """linear_cross_entropy(reduction="sum") against torch float32 autograd of
    the materialised logits."""
    import torch
    from lm_head_linear_chunked_gb300.chunk_loss import linear_cross_entropy
    torch.manual_seed(5)
    N, H, V = 320, 128, 2000
    hidden = torch.randn(N, H, device="cuda").to(torch.bfloat16).requires_grad_()
    head = torch.nn.Linear(H, V, bias=True, device="cuda").to(torch.bfloat16)
    labels = torch.randint(0, V, (N,), device="cuda")
    labels[::7] = -100
    loss = linear_cross_entropy(hidden, head.weight, labels, head.bias, chunk_rows=128, reduction="sum")
    loss.backward()
    h32 = hidden.detach().float().requires_grad_()
    w32 = head.weight.detach().float().requires_grad_()
    b32 = head.bias.detach().float().requires_grad_()
    ref = torch.nn.functional.cross_entropy(h32 @ w32.T + b32, labels, reduction="sum")
    ref.backward()
    assert abs(loss.item() - ref.item()) <= 1e-4 * abs(ref.item())
    for got, want in ((hidden.grad, h32.grad), (head.weight.grad, w32.grad), (head.bias.grad, b32.grad)):
        err = (got.float() - want).abs().max().item()
        assert err <= 1e-2 * want.abs().max().item(), err
