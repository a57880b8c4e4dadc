"""Helpers shared by the GPU tests: moving seeded numpy inputs to the device
and comparing results with the oracle under the stated tolerances."""
from __future__ import annotations

import numpy as np

# (test, quantity, measured error, allowed error) of every check made in this
# process; conftest writes them out when LCE_PARITY_REPORT names a file.
RECORDS: list = []


def _record(what, err, allowed):
    import os
    RECORDS.append({"test": os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0], "quantity": what,
                    "error": float(err), "allowed": float(np.min(allowed)) if np.ndim(allowed) else float(allowed)})

# Tolerances: loss relative 1e-4; lse absolute 1e-3; bf16 gradients max-abs
# 1e-2 * max|ref|; fp32 accumulators max-abs 1e-4 * max|ref|.
LOSS_RTOL = 1e-4
LSE_ATOL = 1e-3
BF16_GRAD_TOL = 1e-2
F32_ACC_TOL = 1e-4


def dev_bf16(bits: np.ndarray, device="cuda"):
    import torch
    if bits is None:
        return None
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)


def dev_i64(a: np.ndarray, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int64)).to(device)


def host_f64(t) -> np.ndarray:
    import torch
    if t.dtype == torch.bfloat16:
        t = t.float()
    return t.double().cpu().numpy()


def max_rel_err(got: np.ndarray, ref: np.ndarray) -> float:
    scale = np.abs(ref).max()
    err = np.abs(got - ref).max()
    return float(err / scale) if scale > 0 else float(err)


def assert_grad(got, ref, tol, what, elem_bound=None):
    """max |got - ref| <= tol * max|ref|; with `elem_bound`, an element may
    instead lie within its own arithmetic bound (see fp16_acc_bound)."""
    got = host_f64(got) if not isinstance(got, np.ndarray) else got
    scale = np.abs(ref).max()
    diff = np.abs(got - ref)
    allowed = tol * max(scale, 1e-30)
    if elem_bound is not None:
        allowed = np.maximum(allowed, elem_bound)
    bad = diff > allowed
    _record(what, diff.max() if diff.size else 0.0, tol * max(scale, 1e-30))
    assert not bad.any() or (scale == 0 and diff.max() == 0), \
        f"{what}: max abs err {diff.max():.3e} > {tol:g} * max|ref| ({scale:.3e}) at {np.argwhere(bad)[0]}"


def fp16_acc_bound(X, W, b, y, lse, s, ignore_index=-100):
    """Per-element error bound of the fp32 grad_W accumulator that the
    arithmetic allows: the gradient GEMMs read the softmax P as fp16, rounded
    at most twice (the fused path stores 2^(t - tile max) in fp16 and rescales
    it to P in fp16; each rounding is <= 2^-11 relative), so
    |err[v,h]| <= s * 2^-10 * sum_i p[i,v] |x[i,h]|, plus 1e-5 * max|ref| for
    fp32 accumulation and the approximate exp.  The target entries p[i, y_i]
    are not 16-bit operands (their gradient is applied in fp32), so they are
    left out of the sum.
    Used for shapes outside the five workloads and the peaked-softmax cases
    (e.g. V = 8, one row), where a softmax with few classes puts O(1)
    probabilities in single non-target entries."""
    import oracle
    Xf, Wf, bf = oracle.as_f64(X), oracle.as_f64(W), oracle.as_f64(b)
    z = oracle.logits(Xf, Wf, bf)
    p = np.exp(z - np.asarray(lse)[:, None])
    y = np.asarray(y)
    p[y == ignore_index] = 0.0
    rows = np.nonzero(y != ignore_index)[0]
    p[rows, y[rows]] = 0.0
    return s * 2.0 ** -10 * (p.T @ np.abs(Xf))


def check_against_oracle(out: dict, ref: dict, has_bias: bool, fwd=True, bwd=True, grad_x=True, acc_bound=None):
    if fwd:
        loss = float(out["loss"].item())
        # relative 1e-4; the 1e-6 floor only matters for a loss near 0 (e.g.
        # V = 1), where fp32 rounding of lse = z leaves ~1e-10
        _record("loss (relative)", abs(loss - ref["loss"]) / max(abs(ref["loss"]), 1e-30), LOSS_RTOL)
        assert abs(loss - ref["loss"]) <= LOSS_RTOL * abs(ref["loss"]) + 1e-6, f"loss {loss} vs oracle {ref['loss']}"
        lse = host_f64(out["lse"])
        err = np.abs(lse - ref["lse"]).max()
        _record("lse (absolute)", err, LSE_ATOL)
        assert err <= LSE_ATOL, f"lse max abs err {err}"
        assert int(out["n_valid"].item()) == ref["n_valid"]
    if bwd:
        if grad_x:
            assert_grad(out["grad_X"], ref["grad_X"], BF16_GRAD_TOL, "grad_X")
        assert_grad(out["grad_W"], ref["grad_W"], BF16_GRAD_TOL, "grad_W")
        assert_grad(out["grad_W_acc"], ref["grad_W"], F32_ACC_TOL, "grad_W_acc (fp32)",
                    None if acc_bound is None else acc_bound + 1e-5 * np.abs(ref["grad_W"]).max())
        if has_bias:
            assert_grad(out["grad_b"], ref["grad_b"], BF16_GRAD_TOL, "grad_b")
            assert_grad(out["grad_b_acc"], ref["grad_b"], F32_ACC_TOL, "grad_b_acc (fp32)")
