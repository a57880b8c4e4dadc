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


def assert_grad(got, ref, tol, what):
    """max |got - ref| <= tol * max|ref|."""
    got = host_f64(got) if not isinstance(got, np.ndarray) else got
    scale = np.abs(ref).max()
    diff = np.abs(got - ref)
    allowed = tol * max(scale, 1e-30)
    bad = diff > allowed
    _record(what, diff.max() if diff.size else 0.0, allowed)
    assert not bad.any() or (scale == 0 and diff.max() == 0), \
        f"{what}: max abs err {diff.max():.3e} > {tol:g} * max|ref| ({scale:.3e}) at {np.argwhere(bad)[0]}"


def check_against_oracle(out: dict, ref: dict, has_bias: bool, fwd=True, bwd=True, grad_x=True):
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
        assert_grad(out["grad_W_acc"], ref["grad_W"], F32_ACC_TOL, "grad_W_acc (fp32)")
        if has_bias:
            assert_grad(out["grad_b"], ref["grad_b"], BF16_GRAD_TOL, "grad_b")
            assert_grad(out["grad_b_acc"], ref["grad_b"], F32_ACC_TOL, "grad_b_acc (fp32)")
