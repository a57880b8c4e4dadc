"""PyTorch autograd front end over the C ABI: the LM-head loss as one call.

This is the shape in which the chunk-loss plugin of LlamaFactory PR #10762
(analysis page, section 4) offers the method: a torch.autograd.Function
whose forward computes the per-chunk loss and, at the same time, the
gradients of the head weight, bias and hidden states (accumulated in FP32
and cast), and whose backward only scales those saved gradients by the
incoming grad_output; and a module that replaces an nn.Linear head's
forward with the loss.

Here the forward is one lce_fused_fwd_bwd_ex call and the backward one
lce_scale_grads call; all arithmetic runs in the library's kernels (torch
only allocates the outputs).  With torch.is_grad_enabled() false, or when
nothing needs a gradient, the forward is a plain lce_forward_ex.
"""
from __future__ import annotations

from typing import Optional

import torch

from . import IGNORE_INDEX, WS_FORWARD, WS_FUSED, WS_FUSED_MIN, _flags, lce_check_status, lce_forward_ex, \
    lce_fused_fwd_bwd_ex, lce_scale_grads, lce_workspace_size


def _flat_contiguous(t: torch.Tensor) -> torch.Tensor:
    t = t.reshape(-1, t.shape[-1])
    return t if t.is_contiguous() else t.contiguous()


class ChunkedLinearCrossEntropy(torch.autograd.Function):
    """loss = mean (or sum) over valid rows of cross_entropy(hidden @ weight.T + bias, labels)."""

    @staticmethod
    def forward(ctx, hidden, weight, bias, labels, ignore_index: int, chunk_rows: int, check: bool,
                grad_wanted: bool, reduction: str = "mean", overlap: bool = False):
        X = _flat_contiguous(hidden)
        y = labels.reshape(-1).to(torch.int64).contiguous()
        N, H = X.shape
        V = weight.shape[0]
        dev = X.device
        stream = torch.cuda.current_stream(dev)
        # (forward runs with autograd off; the caller says whether a graph is built)
        want_grads = grad_wanted and any(ctx.needs_input_grad[:3])
        flags = _flags(reduction, False)
        loss = torch.empty(1, dtype=torch.float32, device=dev)
        lse = torch.empty(N, dtype=torch.float32, device=dev)
        n_valid = torch.empty(1, dtype=torch.int64, device=dev)
        if not want_grads:
            nws = lce_workspace_size(N, H, V, chunk_rows, bias is not None, WS_FORWARD)
            ws = torch.empty(nws, dtype=torch.uint8, device=dev)
            lce_forward_ex(N, H, V, X, weight, bias, y, ignore_index, chunk_rows, loss, lse, n_valid, ws, nws, stream,
                           flags)
        else:
            nws = lce_workspace_size(N, H, V, chunk_rows, bias is not None, WS_FUSED if overlap else WS_FUSED_MIN)
            ws = torch.empty(nws, dtype=torch.uint8, device=dev)
            grad_X = torch.empty_like(X)
            grad_W_acc = torch.empty((V, H), dtype=torch.float32, device=dev)
            grad_b_acc = torch.empty(V, dtype=torch.float32, device=dev) if bias is not None else None
            lce_fused_fwd_bwd_ex(N, H, V, X, weight, bias, y, ignore_index, chunk_rows, 1.0, None, loss, lse,
                                 n_valid, grad_X, None, None, grad_W_acc, grad_b_acc, ws, nws, stream, flags)
            ctx.save_for_backward(grad_X, grad_W_acc, grad_b_acc)
            ctx.shape = (tuple(hidden.shape), N, H, V)
            ctx.dtypes = (weight.dtype, bias.dtype if bias is not None else None)
        if check:
            st = lce_check_status(ws, stream)
            if st != 0:
                from . import LCEError
                raise LCEError(st, "chunked linear cross-entropy")
        ctx.mark_non_differentiable(lse)
        return loss.reshape(()), lse

    @staticmethod
    def backward(ctx, grad_loss, _grad_lse):
        grad_X, grad_W_acc, grad_b_acc = ctx.saved_tensors
        shape, N, H, V = ctx.shape
        g = grad_loss.reshape(1).to(torch.float32).contiguous()
        grad_W = torch.empty((V, H), dtype=ctx.dtypes[0], device=grad_X.device) if ctx.needs_input_grad[1] else None
        grad_b = (torch.empty(V, dtype=ctx.dtypes[1], device=grad_X.device)
                  if grad_b_acc is not None and ctx.needs_input_grad[2] else None)
        lce_scale_grads(N, H, V, g, grad_X if ctx.needs_input_grad[0] else None,
                        grad_W_acc if grad_W is not None else None, grad_W,
                        grad_b_acc if grad_b is not None else None, grad_b,
                        torch.cuda.current_stream(grad_X.device))
        gx = grad_X.reshape(shape) if ctx.needs_input_grad[0] else None
        return gx, grad_W, grad_b, None, None, None, None, None, None, None


def linear_cross_entropy(hidden: torch.Tensor, weight: torch.Tensor, labels: torch.Tensor,
                         bias: Optional[torch.Tensor] = None, ignore_index: int = IGNORE_INDEX,
                         chunk_rows: int = 0, check: bool = False, return_lse: bool = False,
                         reduction: str = "mean", overlap: bool = False):
    """Chunked linear cross-entropy with autograd.

    hidden [..., H] bf16, weight [V, H] bf16 (nn.Linear layout), labels [...]
    with ignore_index for ignored positions, bias [V] or None.  Returns the
    mean (reduction="mean") or sum (reduction="sum") of the loss over valid
    positions (0 if none), and the per-row logsumexp if return_lse.
    chunk_rows = 0 lets the library choose.  check=True synchronises and
    raises on a device-side error (bad label).  overlap=True gives the fused
    call the larger workspace (one more chunk of fp16 exponentials) with
    which each chunk's forward also rescales the previous chunk's softmax:
    a little faster, the same results; the default keeps the minimum."""
    if chunk_rows < 0:
        raise ValueError("chunk_rows must not be negative")
    _flags(reduction, False)  # validates reduction
    grad_wanted = torch.is_grad_enabled() and any(
        t is not None and t.requires_grad for t in (hidden, weight, bias))
    loss, lse = ChunkedLinearCrossEntropy.apply(hidden, weight, bias, labels, ignore_index, chunk_rows, check,
                                                grad_wanted, reduction, overlap)
    return (loss, lse) if return_lse else loss


class ChunkLoss(torch.nn.Module):
    """Wraps an nn.Linear LM head so that head(hidden, labels) returns the loss
    (the plugin's replacement of the head's forward), never the logits."""

    def __init__(self, head: torch.nn.Linear, chunk_rows: int = 0, ignore_index: int = IGNORE_INDEX,
                 reduction: str = "mean"):
        super().__init__()
        if chunk_rows < 0:
            raise ValueError("chunk_rows must not be negative")
        _flags(reduction, False)
        self.head = head
        self.chunk_rows = chunk_rows
        self.ignore_index = ignore_index
        self.reduction = reduction

    def forward(self, hidden: torch.Tensor, labels: torch.Tensor) -> torch.Tensor:
        return linear_cross_entropy(hidden, self.head.weight, labels, self.head.bias, self.ignore_index,
                                    self.chunk_rows, reduction=self.reduction)
