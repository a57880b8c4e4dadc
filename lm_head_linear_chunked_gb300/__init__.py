"""Chunked linear cross-entropy on GB300: Python binding of liblce.so.

The functions named like the C ABI of include/lce.h (lce_forward,
lce_backward, lce_fused_fwd_bwd, ...) only marshal arguments: a tensor
argument may be a torch tensor (its data_ptr() is passed), an integer
address, or None (NULL); a stream may be a torch.cuda.Stream or a raw
handle.  A non-OK status from the library raises LCEError.  Every step of
the computation runs in the library's CUDA kernels; there is no fallback.
If liblce.so has not been built, the first call raises ImportError.

`workspace`, `forward`, `backward` and `fused` below are conveniences that
allocate the outputs and the workspace with torch and call the same entry
points.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

__all__ = [
    "LCEError", "IGNORE_INDEX", "WS_FORWARD", "WS_BACKWARD", "WS_FUSED", "WS_FUSED_MIN", "STATUS", "library_path", "lib",
    "lce_workspace_size", "lce_chunk_rows", "lce_forward", "lce_backward", "lce_fused_fwd_bwd",
    "lce_check_status", "lce_status_string", "lce_debug_gemm", "lce_debug_wait_timeout",
    "lce_debug_gradx_tail_plan",
    "lce_profile_begin", "lce_profile_end", "PROFILE_KINDS", "lce_forward_static_ws", "STATIC_SCRATCH_BYTES",
    "lce_static_ws_check_status",
    "lce_scale_grads",
    "workspace", "forward", "backward", "fused",
]

IGNORE_INDEX = -100
WS_FORWARD, WS_BACKWARD, WS_FUSED, WS_FUSED_MIN = 0, 1, 2, 3
STATUS = {0: "LCE_OK", 1: "LCE_ERR_INVALID_ARG", 2: "LCE_ERR_UNSUPPORTED", 3: "LCE_ERR_WORKSPACE",
          4: "LCE_ERR_LABEL_RANGE", 5: "LCE_ERR_TIMEOUT", 6: "LCE_ERR_CUDA", 7: "LCE_ERR_BOUNDS"}

_HERE = os.path.dirname(os.path.abspath(__file__))
# LCE_LIBRARY=debug in the environment loads the bounds-checking build
# (liblce_debug.so: the same entry points, every kernel checking its indices
# and reporting a failed check as LCE_ERR_BOUNDS) instead of liblce.so.
library_path = os.path.join(_HERE, "liblce_debug.so" if os.environ.get("LCE_LIBRARY") == "debug" else "liblce.so")

_lib = None
_lock = threading.Lock()

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_STATUS = ctypes.c_int

# name -> argument types, in the order of include/lce.h
_SIGS = {
    "lce_workspace_size": [_I64, _I64, _I64, _I64, ctypes.c_int, ctypes.c_int, ctypes.POINTER(ctypes.c_size_t)],
    "lce_chunk_rows": [_I64, _I64, _I64, _I64, ctypes.POINTER(_I64)],
    "lce_forward": [_I64, _I64, _I64, _P, _P, _P, _P, _I64, _I64, _P, _P, _P, _P, ctypes.c_size_t, _P],
    "lce_backward": [_I64, _I64, _I64, _P, _P, _P, _P, _I64, _I64, _P, ctypes.c_float, _P,
                     _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P],
    "lce_fused_fwd_bwd": [_I64, _I64, _I64, _P, _P, _P, _P, _I64, _I64, ctypes.c_float, _P,
                          _P, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P],
    "lce_forward_ex": [_I64, _I64, _I64, _P, _P, _P, _P, _I64, _I64, _P, _P, _P, _P, ctypes.c_size_t, _P,
                       ctypes.c_uint32],
    "lce_backward_ex": [_I64, _I64, _I64, _P, _P, _P, _P, _I64, _I64, _P, ctypes.c_float, _P,
                        _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P, ctypes.c_uint32],
    "lce_fused_fwd_bwd_ex": [_I64, _I64, _I64, _P, _P, _P, _P, _I64, _I64, ctypes.c_float, _P,
                             _P, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P, ctypes.c_uint32],
    "lce_check_status": [_P, _P],
    "lce_status_string": [_STATUS],
    "lce_debug_gemm": [ctypes.c_int, _I64, _I64, _I64, _P, _P, _P, _P, ctypes.c_size_t, _P],
    "lce_debug_wait_timeout": [ctypes.c_uint32, _P, ctypes.c_size_t, _P],
    "lce_debug_gradx_tail_plan": [_I64, _I64, _I64, _I64, ctypes.POINTER(_I64)],
    "lce_forward_static_ws": [_I64, _I64, _I64, _P, _P, _P, _P, _I64, _I64, _P, _P, _P, _P],
    "lce_static_ws_check_status": [_P],
    "lce_scale_grads": [_I64, _I64, _I64, _P, _P, _P, _P, _P, _P, _P],
    "lce_set_gemm_form": [ctypes.c_int],
    "lce_gemm_pair_slots": [],
    "lce_profile_begin": [],
    "lce_profile_end": [ctypes.POINTER(ctypes.c_double), ctypes.POINTER(_I64)],
}

PROFILE_KINDS = ("logits_lse", "recomputed_logits_softmax", "grad_x", "grad_w", "other")


class LCEError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)} ({lce_status_string(status)})")


def lib() -> ctypes.CDLL:
    """The loaded liblce.so (ImportError if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(library_path):
                raise ImportError(f"{library_path} is missing: build it with "
                                  "`python -c 'import __graft_entry__ as g; g.build()'`")
            L = ctypes.CDLL(library_path)
            for name, argtypes in _SIGS.items():
                f = getattr(L, name)
                f.argtypes = argtypes
                f.restype = (ctypes.c_char_p if name == "lce_status_string" else
                             ctypes.c_int if name in ("lce_set_gemm_form", "lce_gemm_pair_slots") else _STATUS)
            _lib = L
    return _lib


def _ptr(x) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x or None
    return x.data_ptr() or None


def _stream(s) -> Optional[int]:
    if s is None:
        return None
    if isinstance(s, int):
        return s or None
    return s.cuda_stream or None


def _check(status: int, where: str) -> None:
    if status != 0:
        raise LCEError(status, where)


# ---------------------------------------------------------------- the C ABI

def lce_status_string(status: int) -> str:
    return lib().lce_status_string(int(status)).decode()


def lce_workspace_size(N: int, H: int, V: int, chunk_rows: int, has_bias: bool, which: int) -> int:
    out = ctypes.c_size_t(0)
    _check(lib().lce_workspace_size(N, H, V, chunk_rows, int(bool(has_bias)), which, ctypes.byref(out)),
           "lce_workspace_size")
    return out.value


def lce_chunk_rows(N: int, H: int, V: int, chunk_rows: int) -> int:
    out = _I64(0)
    _check(lib().lce_chunk_rows(N, H, V, chunk_rows, ctypes.byref(out)), "lce_chunk_rows")
    return out.value


def lce_forward(N, H, V, X, W, b, y, ignore_index, chunk_rows, loss, lse, n_valid, ws, ws_bytes, stream) -> None:
    _check(lib().lce_forward(N, H, V, _ptr(X), _ptr(W), _ptr(b), _ptr(y), ignore_index, chunk_rows,
                             _ptr(loss), _ptr(lse), _ptr(n_valid), _ptr(ws), ws_bytes, _stream(stream)),
           "lce_forward")


def lce_backward(N, H, V, X, W, b, y, ignore_index, chunk_rows, lse, grad_scale, d_grad_output,
                 grad_X, grad_W, grad_b, grad_W_acc, grad_b_acc, ws, ws_bytes, stream) -> None:
    _check(lib().lce_backward(N, H, V, _ptr(X), _ptr(W), _ptr(b), _ptr(y), ignore_index, chunk_rows,
                              _ptr(lse), float(grad_scale), _ptr(d_grad_output), _ptr(grad_X), _ptr(grad_W),
                              _ptr(grad_b), _ptr(grad_W_acc), _ptr(grad_b_acc), _ptr(ws), ws_bytes,
                              _stream(stream)),
           "lce_backward")


def lce_fused_fwd_bwd(N, H, V, X, W, b, y, ignore_index, chunk_rows, grad_scale, d_grad_output, loss, lse,
                      n_valid, grad_X, grad_W, grad_b, grad_W_acc, grad_b_acc, ws, ws_bytes, stream) -> None:
    _check(lib().lce_fused_fwd_bwd(N, H, V, _ptr(X), _ptr(W), _ptr(b), _ptr(y), ignore_index, chunk_rows,
                                   float(grad_scale), _ptr(d_grad_output), _ptr(loss), _ptr(lse), _ptr(n_valid),
                                   _ptr(grad_X), _ptr(grad_W), _ptr(grad_b), _ptr(grad_W_acc), _ptr(grad_b_acc),
                                   _ptr(ws), ws_bytes, _stream(stream)),
           "lce_fused_fwd_bwd")


REDUCTION_SUM = 1   # LCE_REDUCTION_SUM
ACCUMULATE = 2      # LCE_ACCUMULATE


def lce_forward_ex(N, H, V, X, W, b, y, ignore_index, chunk_rows, loss, lse, n_valid, ws, ws_bytes, stream,
                   flags) -> None:
    _check(lib().lce_forward_ex(N, H, V, _ptr(X), _ptr(W), _ptr(b), _ptr(y), ignore_index, chunk_rows,
                                _ptr(loss), _ptr(lse), _ptr(n_valid), _ptr(ws), ws_bytes, _stream(stream),
                                int(flags)),
           "lce_forward_ex")


def lce_backward_ex(N, H, V, X, W, b, y, ignore_index, chunk_rows, lse, grad_scale, d_grad_output,
                    grad_X, grad_W, grad_b, grad_W_acc, grad_b_acc, ws, ws_bytes, stream, flags) -> None:
    _check(lib().lce_backward_ex(N, H, V, _ptr(X), _ptr(W), _ptr(b), _ptr(y), ignore_index, chunk_rows,
                                 _ptr(lse), float(grad_scale), _ptr(d_grad_output), _ptr(grad_X), _ptr(grad_W),
                                 _ptr(grad_b), _ptr(grad_W_acc), _ptr(grad_b_acc), _ptr(ws), ws_bytes,
                                 _stream(stream), int(flags)),
           "lce_backward_ex")


def lce_fused_fwd_bwd_ex(N, H, V, X, W, b, y, ignore_index, chunk_rows, grad_scale, d_grad_output, loss, lse,
                         n_valid, grad_X, grad_W, grad_b, grad_W_acc, grad_b_acc, ws, ws_bytes, stream,
                         flags) -> None:
    _check(lib().lce_fused_fwd_bwd_ex(N, H, V, _ptr(X), _ptr(W), _ptr(b), _ptr(y), ignore_index, chunk_rows,
                                      float(grad_scale), _ptr(d_grad_output), _ptr(loss), _ptr(lse),
                                      _ptr(n_valid), _ptr(grad_X), _ptr(grad_W), _ptr(grad_b), _ptr(grad_W_acc),
                                      _ptr(grad_b_acc), _ptr(ws), ws_bytes, _stream(stream), int(flags)),
           "lce_fused_fwd_bwd_ex")


def _flags(reduction: str, accumulate: bool) -> int:
    if reduction not in ("mean", "sum"):
        raise ValueError(f"reduction must be 'mean' or 'sum', got {reduction!r}")
    return (REDUCTION_SUM if reduction == "sum" else 0) | (ACCUMULATE if accumulate else 0)


STATIC_SCRATCH_BYTES = 32 << 20


def lce_forward_static_ws(N, H, V, X, W, b, y, ignore_index, chunk_rows, loss, lse, n_valid, stream) -> None:
    """lce_forward with the library's fixed device scratch array instead of a
    workspace argument, for callers that cannot allocate device memory."""
    _check(lib().lce_forward_static_ws(N, H, V, _ptr(X), _ptr(W), _ptr(b), _ptr(y), ignore_index, chunk_rows,
                                       _ptr(loss), _ptr(lse), _ptr(n_valid), _stream(stream)),
           "lce_forward_static_ws")


def lce_static_ws_check_status(stream) -> int:
    """Synchronises the stream; returns the device status code of the last
    lce_forward_static_ws call on the current device (no raise)."""
    return lib().lce_static_ws_check_status(_stream(stream))


def lce_scale_grads(N, H, V, d_grad_output, grad_X, grad_W_acc, grad_W, grad_b_acc, grad_b, stream) -> None:
    _check(lib().lce_scale_grads(N, H, V, _ptr(d_grad_output), _ptr(grad_X), _ptr(grad_W_acc), _ptr(grad_W),
                                 _ptr(grad_b_acc), _ptr(grad_b), _stream(stream)),
           "lce_scale_grads")


def lce_check_status(ws, stream) -> int:
    """Synchronises the stream; returns the device status code (no raise)."""
    return lib().lce_check_status(_ptr(ws), _stream(stream))


def lce_debug_gemm(layout, M, N, K, A, B, D, ws, ws_bytes, stream) -> None:
    _check(lib().lce_debug_gemm(layout, M, N, K, _ptr(A), _ptr(B), _ptr(D), _ptr(ws), ws_bytes, _stream(stream)),
           "lce_debug_gemm")


def lce_debug_wait_timeout(limit_us, ws, ws_bytes, stream) -> None:
    _check(lib().lce_debug_wait_timeout(limit_us, _ptr(ws), ws_bytes, _stream(stream)), "lce_debug_wait_timeout")


def lce_debug_gradx_tail_plan(tiles, slots, k_blocks, tile_cols=256) -> tuple:
    """(tiles computed whole, tiles split over K after them, slices per split
    tile, k-blocks per slice) of a pair-form grad_X launch whose tiles are
    256 rows x tile_cols (256 or 512) columns."""
    out = (_I64 * 4)()
    _check(lib().lce_debug_gradx_tail_plan(tiles, slots, k_blocks, tile_cols, out), "lce_debug_gradx_tail_plan")
    return tuple(int(v) for v in out)


GEMM_SINGLE, GEMM_PAIR = 0, 1
GEMM_FORMS = {"single": GEMM_SINGLE, "pair": GEMM_PAIR}


def lce_set_gemm_form(form) -> int:
    """Selects the GEMM form of later calls ("single"/0 or "pair"/1); returns the previous one."""
    f = GEMM_FORMS.get(form, form)
    prev = lib().lce_set_gemm_form(int(f))
    if prev < 0:
        raise ValueError(f"unknown GEMM form {form!r}")
    return prev


def lce_gemm_pair_slots() -> int:
    """CTA pairs of the pair form resident at once on the current device (0: not available)."""
    return int(lib().lce_gemm_pair_slots())


def lce_profile_begin() -> None:
    _check(lib().lce_profile_begin(), "lce_profile_begin")


def lce_profile_end() -> dict:
    """{kind: (milliseconds, launches)} of the kernels enqueued since lce_profile_begin()."""
    ms = (ctypes.c_double * len(PROFILE_KINDS))()
    n = (_I64 * len(PROFILE_KINDS))()
    _check(lib().lce_profile_end(ms, n), "lce_profile_end")
    return {k: (ms[i], n[i]) for i, k in enumerate(PROFILE_KINDS)}


# ---------------------------------------------------------------- torch conveniences

def _torch():
    import torch
    return torch


def _bits(t):
    """bf16 tensor -> its storage (the library takes bf16 bit patterns)."""
    torch = _torch()
    if t is None:
        return None
    if t.dtype not in (torch.bfloat16, torch.int16, torch.uint16):
        raise TypeError(f"expected a bf16 tensor, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return t


def workspace(N, H, V, chunk_rows=0, has_bias=False, which=WS_FUSED, device="cuda"):
    torch = _torch()
    n = lce_workspace_size(N, H, V, chunk_rows, has_bias, which)
    return torch.empty(n, dtype=torch.uint8, device=device)


def forward(X, W, b, y, ignore_index=IGNORE_INDEX, chunk_rows=0, ws=None, stream=None, reduction="mean"):
    """loss, lse, n_valid of the chunked linear cross-entropy (one lce_forward_ex call)."""
    torch = _torch()
    N, H = X.shape
    V = W.shape[0]
    dev = X.device
    if ws is None:
        ws = workspace(N, H, V, chunk_rows, b is not None, WS_FORWARD, dev)
    loss = torch.empty(1, dtype=torch.float32, device=dev)
    lse = torch.empty(N, dtype=torch.float32, device=dev)
    n_valid = torch.empty(1, dtype=torch.int64, device=dev)
    stream = stream or torch.cuda.current_stream(dev)
    lce_forward_ex(N, H, V, _bits(X), _bits(W), _bits(b), y, ignore_index, chunk_rows, loss, lse, n_valid,
                   ws, ws.numel(), stream, _flags(reduction, False))
    return {"loss": loss, "lse": lse, "n_valid": n_valid, "ws": ws}


def _accumulators(W, b, accumulate, grad_W_acc, grad_b_acc):
    """The FP32 accumulators: the caller's (required with accumulate), else new ones."""
    torch = _torch()
    V = W.shape[0]
    if accumulate:
        if grad_W_acc is None or (b is not None and grad_b_acc is None):
            raise ValueError("accumulate=True needs the running grad_W_acc (and grad_b_acc with a bias)")
        return grad_W_acc, grad_b_acc
    gw = grad_W_acc if grad_W_acc is not None else torch.empty(W.shape, dtype=torch.float32, device=W.device)
    gb = None
    if b is not None:
        gb = grad_b_acc if grad_b_acc is not None else torch.empty(V, dtype=torch.float32, device=W.device)
    return gw, gb


def backward(X, W, b, y, lse, ignore_index=IGNORE_INDEX, chunk_rows=0, grad_scale=1.0, grad_output=None,
             want_grad_X=True, ws=None, stream=None, reduction="mean", accumulate=False, grad_W_acc=None,
             grad_b_acc=None):
    """All gradients from a forward's lse (one lce_backward_ex call).  With
    accumulate=True the given FP32 accumulators are added to."""
    torch = _torch()
    N, H = X.shape
    V = W.shape[0]
    dev = X.device
    if ws is None:
        ws = workspace(N, H, V, chunk_rows, b is not None, WS_BACKWARD, dev)
    gw_acc, gb_acc = _accumulators(W, b, accumulate, grad_W_acc, grad_b_acc)
    out = {
        "grad_X": torch.empty_like(X) if want_grad_X else None,
        "grad_W": torch.empty_like(W),
        "grad_W_acc": gw_acc,
        "grad_b": torch.empty_like(b) if b is not None else None,
        "grad_b_acc": gb_acc,
        "ws": ws,
    }
    stream = stream or torch.cuda.current_stream(dev)
    lce_backward_ex(N, H, V, _bits(X), _bits(W), _bits(b), y, ignore_index, chunk_rows, lse, grad_scale,
                    grad_output, out["grad_X"], out["grad_W"], out["grad_b"], out["grad_W_acc"], out["grad_b_acc"],
                    ws, ws.numel(), stream, _flags(reduction, accumulate))
    return out


def fused(X, W, b, y, ignore_index=IGNORE_INDEX, chunk_rows=0, grad_scale=1.0, grad_output=None, ws=None,
          stream=None, reduction="mean", accumulate=False, grad_W_acc=None, grad_b_acc=None):
    """loss, lse, n_valid and all gradients (one lce_fused_fwd_bwd_ex call).
    With accumulate=True the given FP32 accumulators are added to."""
    torch = _torch()
    N, H = X.shape
    V = W.shape[0]
    dev = X.device
    if ws is None:
        ws = workspace(N, H, V, chunk_rows, b is not None, WS_FUSED, dev)
    gw_acc, gb_acc = _accumulators(W, b, accumulate, grad_W_acc, grad_b_acc)
    out = {
        "loss": torch.empty(1, dtype=torch.float32, device=dev),
        "lse": torch.empty(N, dtype=torch.float32, device=dev),
        "n_valid": torch.empty(1, dtype=torch.int64, device=dev),
        "grad_X": torch.empty_like(X),
        "grad_W": torch.empty_like(W),
        "grad_W_acc": gw_acc,
        "grad_b": torch.empty_like(b) if b is not None else None,
        "grad_b_acc": gb_acc,
        "ws": ws,
    }
    stream = stream or torch.cuda.current_stream(dev)
    lce_fused_fwd_bwd_ex(N, H, V, _bits(X), _bits(W), _bits(b), y, ignore_index, chunk_rows, grad_scale,
                         grad_output, out["loss"], out["lse"], out["n_valid"], out["grad_X"], out["grad_W"],
                         out["grad_b"], out["grad_W_acc"], out["grad_b_acc"], ws, ws.numel(), stream,
                         _flags(reduction, accumulate))
    return out
