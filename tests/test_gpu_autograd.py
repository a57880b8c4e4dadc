"""The autograd front end (chunk_loss.py) on the GPU: its gradients against
the oracle, against torch's own cross_entropy autograd in float32, and with
a grad_output other than 1."""
import numpy as np
import pytest

import oracle
from tests.gpu_util import LOSS_RTOL, assert_grad, dev_bf16, dev_i64, host_f64
from tests.test_gpu_parity import random_problem

pytestmark = pytest.mark.gpu


def _setup(seed, N, H, V, bias):
    import torch
    X, W, b, y = random_problem(seed, N, H, V, bias=bias)
    Xd = dev_bf16(X).requires_grad_(True)
    Wd = dev_bf16(W).requires_grad_(True)
    bd = dev_bf16(b).requires_grad_(True) if b is not None else None
    return (X, W, b, y), (Xd, Wd, bd, dev_i64(y)), torch


@pytest.mark.parametrize("bias", [False, True])
def test_autograd_matches_oracle(bias):
    from lm_head_linear_chunked_gb300.chunk_loss import linear_cross_entropy
    (X, W, b, y), (Xd, Wd, bd, yd), torch = _setup(31, 384, 128, 2048, bias)
    loss = linear_cross_entropy(Xd.view(3, 128, 128), Wd, yd.view(3, 128), bias=bd, chunk_rows=128, check=True)
    (loss * 2.5).backward()
    ref = oracle.fused(X, W, b, y, grad_output=2.5)
    assert abs(float(loss.item()) - ref["loss"]) <= LOSS_RTOL * abs(ref["loss"])
    assert Xd.grad.shape == Xd.shape
    assert_grad(Xd.grad, ref["grad_X"], 1e-2, "grad_X")
    assert_grad(Wd.grad, ref["grad_W"], 1e-2, "grad_W")
    if bias:
        assert_grad(bd.grad, ref["grad_b"], 1e-2, "grad_b")


def test_autograd_matches_torch_float32():
    from lm_head_linear_chunked_gb300.chunk_loss import ChunkLoss
    (X, W, b, y), (Xd, Wd, bd, yd), torch = _setup(32, 256, 256, 4096, True)
    head = torch.nn.Linear(256, 4096, bias=True, device="cuda", dtype=torch.bfloat16)
    with torch.no_grad():
        head.weight.copy_(Wd)
        head.bias.copy_(bd)
    loss = ChunkLoss(head, chunk_rows=64)(Xd, yd)
    loss.backward()
    Xf = Xd.detach().float().requires_grad_(True)
    Wf = Wd.detach().float().requires_grad_(True)
    bf = bd.detach().float().requires_grad_(True)
    ref = torch.nn.functional.cross_entropy(Xf @ Wf.T + bf, yd, ignore_index=-100)
    ref.backward()
    assert abs(loss.item() - ref.item()) <= 1e-4 * abs(ref.item())
    for got, want in ((Xd.grad, Xf.grad), (head.weight.grad, Wf.grad), (head.bias.grad, bf.grad)):
        err = (got.float() - want).abs().max().item()
        assert err <= 1e-2 * want.abs().max().item()


def test_no_grad_forward_only():
    import torch
    from lm_head_linear_chunked_gb300.chunk_loss import linear_cross_entropy
    (X, W, b, y), (Xd, Wd, bd, yd), torch = _setup(33, 200, 64, 1024, False)
    with torch.no_grad():
        loss, lse = linear_cross_entropy(Xd, Wd, yd, return_lse=True, check=True)
    ref = oracle.forward(X, W, None, y)
    assert abs(float(loss.item()) - ref["loss"]) <= LOSS_RTOL * abs(ref["loss"])
    assert np.abs(host_f64(lse) - ref["lse"]).max() <= 1e-3


def test_autograd_overlap_option_same_bits():
    """overlap=True (the larger workspace: each chunk's forward rescales the
    previous chunk's softmax) gives the same loss and gradients, bit for bit,
    as the default minimum workspace."""
    from lm_head_linear_chunked_gb300.chunk_loss import linear_cross_entropy
    (X, W, b, y), (Xd, Wd, bd, yd), torch = _setup(33, 9000, 128, 2048, False)
    grads = []
    for overlap in (False, True):
        Xd.grad = None
        Wd.grad = None
        loss = linear_cross_entropy(Xd, Wd, yd, chunk_rows=4096, check=True, overlap=overlap)
        loss.backward()
        grads.append((loss.detach().clone(), Xd.grad.clone(), Wd.grad.clone()))
    for a, b_ in zip(*grads):
        assert torch.equal(a, b_)
