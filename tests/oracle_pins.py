"""Pins of the FP64 oracle against facts that do not come from the oracle.

Each check returns a list of failure strings (empty = pass), so the same
checks run against the real oracle (tests/test_oracle_pins.py) and against
oracles with a planted mistake (tests/test_oracle_mutants.py).

Sources: the chunk-loss autograd Function of the LlamaFactory PR #10762
analysis page (section 4: cross_entropy with reduction="none" and
ignore_index=-100 per row chunk; FP32-accumulated grad_weight/grad_bias)
and the chunking section of the TRL "1M 토큰 이상 학습" page (rows are
independent, so any row split gives the same result).
"""
from __future__ import annotations

import math

import numpy as np

IGN = -100


def _rng(seed):
    return np.random.default_rng(seed)


def tiny_problem(seed=0, N=6, H=8, V=16, bias=True, ignore=(1,), scale=1.0):
    r = _rng(seed)
    X = r.standard_normal((N, H)) * scale
    W = r.standard_normal((V, H)) * (scale / math.sqrt(H))
    b = r.standard_normal(V) * 0.3 if bias else None
    y = r.integers(0, V, N).astype(np.int64)
    for i in ignore:
        y[i] = IGN
    return X, W, b, y


def _close(a, b, rtol, atol=0.0):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    if a.shape != b.shape:
        return False
    return bool(np.all(np.abs(a - b) <= atol + rtol * np.maximum(1.0, np.abs(b).max(initial=0.0))))


def pin_zero_weight_closed_form(orc):
    """W = 0, b = 0: every logit is 0, so lse = ln V and loss = ln V; grad_X = 0;
    grad_W[v] = s * sum_valid (1/V - [y_i = v]) x_i; grad_b[v] = s (n_valid/V - count_v)."""
    fails = []
    for V in (1, 3, 16, 4096):
        N, H = 9, 5
        r = _rng(V)
        X = r.standard_normal((N, H))
        y = r.integers(0, V, N).astype(np.int64)
        y[[2, 7]] = IGN
        W = np.zeros((V, H))
        b = np.zeros(V)
        out = orc.fused(X, W, b, y)
        lnV = math.log(V)
        if abs(out["loss"] - lnV) > 1e-12 * max(1, lnV):
            fails.append(f"P1 loss {out['loss']} != ln {V}")
        if not np.allclose(out["lse"], lnV, rtol=0, atol=1e-12):
            fails.append("P1 lse != ln V")
        if np.abs(out["grad_X"]).max() > 1e-15:
            fails.append("P1 grad_X != 0")
        ok = y != IGN
        nv = int(ok.sum())
        s = 1.0 / nv
        gW = np.zeros((V, H))
        gb = np.zeros(V)
        for i in np.nonzero(ok)[0]:
            gW += s * (1.0 / V) * X[i][None, :]
            gW[y[i]] -= s * X[i]
            gb += s / V
            gb[y[i]] -= s
        if not _close(out["grad_W"], gW, 1e-12):
            fails.append("P1 grad_W closed form")
        if not _close(out["grad_b"], gb, 1e-12):
            fails.append("P1 grad_b closed form")
    return fails


def pin_rows_sum_to_zero(orc):
    """Each row of softmax - onehot sums to 0, so sum_v grad_W[v,:] = 0 and sum_v grad_b = 0."""
    X, W, b, y = tiny_problem(1, N=12, H=7, V=33)
    out = orc.fused(X, W, b, y)
    fails = []
    if np.abs(out["grad_W"].sum(axis=0)).max() > 1e-12 * np.abs(out["grad_W"]).max():
        fails.append("P2 sum_v grad_W != 0")
    if abs(out["grad_b"].sum()) > 1e-12 * np.abs(out["grad_b"]).max():
        fails.append("P2 sum grad_b != 0")
    return fails


def pin_ignored_rows(orc):
    """An ignored row contributes nothing: grad_X of that row is exactly 0 and
    changing its hidden state changes only its own lse."""
    X, W, b, y = tiny_problem(2, N=8, H=6, V=20, ignore=(3, 5))
    a = orc.fused(X, W, b, y)
    X2 = X.copy()
    X2[3] += 0.7
    c = orc.fused(X2, W, b, y)
    fails = []
    if np.any(a["grad_X"][[3, 5]] != 0.0):
        fails.append("P3 grad_X of ignored rows != 0")
    if abs(a["loss"] - c["loss"]) > 1e-14 or not _close(a["grad_W"], c["grad_W"], 1e-13) \
            or not _close(a["grad_b"], c["grad_b"], 1e-13):
        fails.append("P3 ignored row changed loss/grads")
    if abs(a["lse"][3] - c["lse"][3]) < 1e-6 or not np.array_equal(np.delete(a["lse"], 3), np.delete(c["lse"], 3)):
        fails.append("P3 lse changed for the wrong rows")
    if a["n_valid"] != 6:
        fails.append("P3 n_valid")
    return fails


def pin_finite_differences(orc):
    """Central differences of the loss (step 1e-6, float64) match the gradients."""
    X, W, b, y = tiny_problem(3, N=6, H=8, V=16, ignore=(4,))
    out = orc.fused(X, W, b, y)
    eps = 1e-6
    fails = []

    def loss_of(X_, W_, b_):
        return orc.forward(X_, W_, b_, y)["loss"]

    for name, arr, grad in (("X", X, out["grad_X"]), ("W", W, out["grad_W"]), ("b", b, out["grad_b"])):
        num = np.zeros_like(arr)
        it = np.nditer(arr, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            p = arr.copy(); p[idx] += eps
            m = arr.copy(); m[idx] -= eps
            args_p = {"X": (p, W, b), "W": (X, p, b), "b": (X, W, p)}[name]
            args_m = {"X": (m, W, b), "W": (X, m, b), "b": (X, W, m)}[name]
            num[idx] = (loss_of(*args_p) - loss_of(*args_m)) / (2 * eps)
        err = np.abs(num - grad).max() / max(np.abs(grad).max(), 1e-30)
        if not err <= 1e-6:
            fails.append(f"P5 finite differences for {name}: rel err {err:.2e}")
    return fails


def pin_shift_invariance(orc):
    """b += c shifts every lse by c and leaves loss and grads unchanged;
    W[v] += u for all v shifts row i's logits by x_i.u: loss, grad_X, grad_W unchanged."""
    X, W, b, y = tiny_problem(4, N=7, H=5, V=11, ignore=(0,))
    a = orc.fused(X, W, b, y)
    c = orc.fused(X, W, b + 3.25, y)
    fails = []
    if not np.allclose(c["lse"] - a["lse"], 3.25, atol=1e-12):
        fails.append("P6 lse does not shift with b")
    if abs(c["loss"] - a["loss"]) > 1e-12:
        fails.append("P6 loss changed under b shift")
    for k in ("grad_X", "grad_W", "grad_b"):
        if not _close(c[k], a[k], 1e-10):
            fails.append(f"P6 {k} changed under b shift")
    u = _rng(9).standard_normal(X.shape[1])
    d = orc.fused(X, W + u[None, :], b, y)
    if not np.allclose(d["lse"] - a["lse"], X @ u, atol=1e-12):
        fails.append("P6 lse does not shift with W rows")
    if abs(d["loss"] - a["loss"]) > 1e-12:
        fails.append("P6 loss changed under W shift")
    for k in ("grad_X", "grad_W", "grad_b"):
        if not _close(d[k], a[k], 1e-10):
            fails.append(f"P6 {k} changed under W shift")
    return fails


def pin_row_permutation(orc):
    """Permuting rows permutes lse and grad_X and leaves loss, grad_W, grad_b unchanged."""
    X, W, b, y = tiny_problem(5, N=9, H=6, V=14, ignore=(2, 6))
    perm = _rng(5).permutation(len(y))
    a = orc.fused(X, W, b, y)
    c = orc.fused(X[perm], W, b, y[perm])
    fails = []
    if not np.allclose(c["lse"], a["lse"][perm], atol=1e-13, rtol=0):
        fails.append("P7 lse not permuted")
    if not _close(c["grad_X"], a["grad_X"][perm], 1e-13):
        fails.append("P7 grad_X not permuted")
    if abs(c["loss"] - a["loss"]) > 1e-13:
        fails.append("P7 loss changed")
    for k in ("grad_W", "grad_b"):
        if not _close(c[k], a[k], 1e-12):
            fails.append(f"P7 {k} changed")
    return fails


def pin_torch_cross_entropy(orc):
    """Special case that is a library routine: torch CPU float64
    F.cross_entropy(X W^T + b, y, ignore_index=-100) (mean over valid rows)
    with autograd, scaled by grad_scale * grad_output; lse = torch.logsumexp."""
    import torch
    fails = []
    for seed, bias, scale, gs, go in ((6, True, 1.0, 1.0, 1.0), (7, False, 1.0, 0.5, 3.0),
                                      (8, True, 60.0, 1.0, 1.0)):
        X, W, b, y = tiny_problem(seed, N=10, H=12, V=23, bias=bias, ignore=(0, 9), scale=scale)
        out = orc.fused(X, W, b, y, grad_scale=gs, grad_output=go)
        tX = torch.tensor(X, requires_grad=True)
        tW = torch.tensor(W, requires_grad=True)
        tb = torch.tensor(b, requires_grad=True) if b is not None else None
        z = tX @ tW.T + (tb if tb is not None else 0.0)
        loss = torch.nn.functional.cross_entropy(z, torch.tensor(y), ignore_index=IGN)
        (loss * gs).backward(torch.tensor(go, dtype=torch.float64))
        if not math.isfinite(out["loss"]) or abs(out["loss"] - loss.item()) > 1e-12 * max(1.0, abs(loss.item())):
            fails.append(f"P8 loss {out['loss']} vs torch {loss.item()} (seed {seed})")
        if not np.allclose(out["lse"], torch.logsumexp(z.detach(), 1).numpy(), rtol=1e-13, atol=1e-12):
            fails.append(f"P8 lse (seed {seed})")
        for k, t in (("grad_X", tX), ("grad_W", tW)):
            if not _close(out[k], t.grad.numpy(), 1e-11):
                fails.append(f"P8 {k} (seed {seed})")
        if tb is not None and not _close(out["grad_b"], tb.grad.numpy(), 1e-11):
            fails.append(f"P8 grad_b (seed {seed})")
    return fails


def pin_torch_cross_entropy_sum(orc):
    """Reduction "sum" against torch CPU float64 F.cross_entropy(...,
    reduction="sum") with autograd: loss, and every gradient scaled by
    grad_scale * grad_output (no division by n_valid)."""
    import torch
    fails = []
    for seed, bias, gs, go in ((16, True, 1.0, 1.0), (17, False, 0.25, 2.0)):
        X, W, b, y = tiny_problem(seed, N=9, H=10, V=19, bias=bias, ignore=(2, 5))
        out = orc.fused(X, W, b, y, grad_scale=gs, grad_output=go, reduction="sum")
        tX = torch.tensor(X, requires_grad=True)
        tW = torch.tensor(W, requires_grad=True)
        tb = torch.tensor(b, requires_grad=True) if b is not None else None
        z = tX @ tW.T + (tb if tb is not None else 0.0)
        loss = torch.nn.functional.cross_entropy(z, torch.tensor(y), ignore_index=IGN, reduction="sum")
        (loss * gs).backward(torch.tensor(go, dtype=torch.float64))
        if abs(out["loss"] - loss.item()) > 1e-12 * max(1.0, abs(loss.item())):
            fails.append(f"P8s loss {out['loss']} vs torch {loss.item()} (seed {seed})")
        for k, t in (("grad_X", tX), ("grad_W", tW)):
            if not _close(out[k], t.grad.numpy(), 1e-11):
                fails.append(f"P8s {k} (seed {seed})")
        if tb is not None and not _close(out["grad_b"], tb.grad.numpy(), 1e-11):
            fails.append(f"P8s grad_b (seed {seed})")
    # no valid row: the empty sum is 0 and so is every gradient
    X, W, b, y = tiny_problem(18, N=3, H=4, V=5, ignore=(0, 1, 2))
    out = orc.fused(X, W, b, y, reduction="sum")
    if out["loss"] != 0.0 or np.abs(out["grad_W"]).max() != 0.0:
        fails.append("P8s all rows ignored")
    return fails


def pin_finite_differences_sum(orc):
    """Central differences of the summed loss match the reduction "sum" gradients."""
    X, W, b, y = tiny_problem(19, N=5, H=6, V=7, ignore=(3,))
    out = orc.fused(X, W, b, y, reduction="sum")
    eps = 1e-6
    fails = []
    for name, arr, grad in (("W", W, out["grad_W"]), ("b", b, out["grad_b"])):
        num = np.zeros_like(arr)
        it = np.nditer(arr, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            p = arr.copy(); p[idx] += eps
            m = arr.copy(); m[idx] -= eps
            args_p = {"W": (X, p, b), "b": (X, W, p)}[name]
            args_m = {"W": (X, m, b), "b": (X, W, m)}[name]
            num[idx] = (orc.forward(*args_p, y, reduction="sum")["loss"] -
                        orc.forward(*args_m, y, reduction="sum")["loss"]) / (2 * eps)
        err = np.abs(num - grad).max() / max(np.abs(grad).max(), 1e-30)
        if not err <= 1e-6:
            fails.append(f"P5s finite differences for {name}: rel err {err:.2e}")
    return fails


def pin_single_class(orc):
    """V = 1: the only class has probability 1, so loss = 0 and all grads = 0."""
    X, W, b, y = tiny_problem(10, N=5, H=4, V=1, ignore=(1,))
    y[y != IGN] = 0
    out = orc.fused(X, W, b, y)
    fails = []
    if abs(out["loss"]) > 1e-15:
        fails.append("P9 loss != 0 for V=1")
    for k in ("grad_X", "grad_W", "grad_b"):
        if np.abs(out[k]).max() > 1e-15:
            fails.append(f"P9 {k} != 0 for V=1")
    return fails


def pin_no_valid_rows(orc):
    """No valid row: loss 0 and zero grads (the trainer's division guard); lse still defined."""
    X, W, b, y = tiny_problem(11, N=4, H=3, V=6, ignore=(0, 1, 2, 3))
    out = orc.fused(X, W, b, y)
    fails = []
    if out["loss"] != 0.0 or out["n_valid"] != 0:
        fails.append("no-valid loss/n_valid")
    for k in ("grad_X", "grad_W", "grad_b"):
        if np.abs(out[k]).max() != 0.0:
            fails.append(f"no-valid {k}")
    import torch
    ref = torch.logsumexp(torch.tensor(X @ W.T + b), 1).numpy()
    if not np.allclose(out["lse"], ref, atol=1e-12):
        fails.append("no-valid lse")
    return fails


def pin_worked_example(orc):
    """Hand-derived case.  X = [[1,0],[0,1]], W = [[0,0],[1,0],[0,2]], no bias,
    y = [1, 0]: row 0 has logits (0, 1, 0), row 1 has (0, 0, 2).
    lse_0 = ln(2 + e), lse_1 = ln(2 + e^2);
    loss = ((ln(2+e) - 1) + ln(2+e^2)) / 2;
    with s = 1/2: G_0 = s((1, e, 1)/(2+e) - (0,1,0)), G_1 = s((1, 1, e^2)/(2+e^2) - (1,0,0));
    grad_X = G W, grad_W = G^T X (written out below)."""
    e = math.e
    X = np.array([[1.0, 0.0], [0.0, 1.0]])
    W = np.array([[0.0, 0.0], [1.0, 0.0], [0.0, 2.0]])
    y = np.array([1, 0], dtype=np.int64)
    out = orc.fused(X, W, None, y)
    d0, d1 = 2 + e, 2 + e * e
    G0 = np.array([1 / d0, e / d0 - 1, 1 / d0]) / 2
    G1 = np.array([1 / d1 - 1, 1 / d1, e * e / d1]) / 2
    gX = np.array([[G0[1], 2 * G0[2]], [G1[1], 2 * G1[2]]])
    gW = np.array([[G0[0], G1[0]], [G0[1], G1[1]], [G0[2], G1[2]]])
    fails = []
    if abs(out["loss"] - ((math.log(d0) - 1) + math.log(d1)) / 2) > 1e-15:
        fails.append("worked example loss")
    if not np.allclose(out["lse"], [math.log(d0), math.log(d1)], rtol=0, atol=1e-15):
        fails.append("worked example lse")
    if not _close(out["grad_X"], gX, 1e-15) or not _close(out["grad_W"], gW, 1e-15):
        fails.append("worked example grads")
    return fails


def pin_block_invariance(orc):
    """Rows are independent (TRL chunking section): the oracle's row blocking
    changes nothing beyond float64 rounding."""
    X, W, b, y = tiny_problem(12, N=23, H=9, V=31, ignore=(4, 5, 20))
    ref = orc.fused(X, W, b, y, block_rows=23)
    fails = []
    for br in (1, 7, 16):
        o = orc.fused(X, W, b, y, block_rows=br)
        if abs(o["loss"] - ref["loss"]) > 1e-13 or not np.allclose(o["lse"], ref["lse"], atol=1e-13):
            fails.append(f"block {br}: loss/lse")
        for k in ("grad_X", "grad_W", "grad_b"):
            if not _close(o[k], ref[k], 1e-13):
                fails.append(f"block {br}: {k}")
    return fails


def pin_row_sampled_pieces(orc):
    """The row-sampled functions match torch on their rows (per-row CE with
    reduction='none', autograd of the row losses with weight s)."""
    import torch
    X, W, b, y = tiny_problem(13, N=11, H=10, V=19, ignore=(2, 8))
    rows = np.array([0, 2, 5, 8, 10])
    nv = int((y != IGN).sum())
    s = 1.0 / nv
    rf = orc.rows_forward(X[rows], W, b, y[rows])
    tX = torch.tensor(X[rows], requires_grad=True)
    z = tX @ torch.tensor(W).T + torch.tensor(b)
    per = torch.nn.functional.cross_entropy(z, torch.tensor(y[rows]), ignore_index=IGN, reduction="none")
    (per.sum() * s).backward()
    fails = []
    if not np.allclose(rf["row_loss"], per.detach().numpy(), atol=1e-13):
        fails.append("rows_forward row_loss")
    if not np.allclose(rf["lse"], torch.logsumexp(z.detach(), 1).numpy(), atol=1e-13):
        fails.append("rows_forward lse")
    gx = orc.rows_grad_X(X[rows], W, b, y[rows], rf["lse"], s)
    if not _close(gx, tX.grad.numpy(), 1e-12):
        fails.append("rows_grad_X")
    zt = orc.target_logits(X, W, b, y, block_rows=4)
    ok = y != IGN
    ref = (X @ W.T + b)[np.nonzero(ok)[0], y[ok]]
    if not np.allclose(zt[ok], ref, atol=1e-13) or not np.all(np.isnan(zt[~ok])):
        fails.append("target_logits")
    return fails


def pin_column_slice(orc):
    """grad_W_columns against torch CPU float64 cross_entropy + autograd:
    the chosen columns of grad_W (all rows), grad_b, lse and the loss."""
    import torch
    fails = []
    for (h0, h1, block) in ((2, 5, 3), (0, 8, 100), (7, 8, 1)):
        X, W, b, y = tiny_problem(23, N=11, H=8, V=13, ignore=(0, 6))
        out = orc.grad_W_columns(X, W, b, y, h0, h1, grad_scale=0.7, grad_output=1.3, block_rows=block)
        Xt = torch.tensor(X, requires_grad=True)
        Wt = torch.tensor(W, requires_grad=True)
        bt = torch.tensor(b, requires_grad=True)
        z = Xt @ Wt.T + bt
        loss = torch.nn.functional.cross_entropy(z, torch.tensor(y), ignore_index=IGN)
        (loss * 0.7 * 1.3).backward()
        if not _close(out["grad_W_cols"], Wt.grad.numpy()[:, h0:h1], 1e-11):
            fails.append(f"column slice {h0}:{h1} grad_W")
        if not _close(out["grad_b"], bt.grad.numpy(), 1e-11):
            fails.append("column slice grad_b")
        if not _close(out["lse"], torch.logsumexp(z, 1).detach().numpy(), 1e-12):
            fails.append("column slice lse")
        if abs(out["loss"] - loss.item()) > 1e-12 * abs(loss.item()):
            fails.append("column slice loss")
    return fails


def pin_bf16_decode(orc):
    """bf16 bit patterns decode to the values their IEEE fields define:
    sign, 8 exponent bits (bias 127), 7 fraction bits; subnormals 0.f 2^-126.
    Written as hand-derived constants, independent of any decoder."""
    cases = {0x3F80: 1.0, 0xC020: -2.5, 0x0001: 2.0 ** -133, 0x7F7F: (2 - 2.0 ** -7) * 2.0 ** 127,
             0x4049: 3.140625, 0x0080: 2.0 ** -126, 0xBE00: -0.125, 0x4300: 128.0}
    bits = np.array(list(cases), dtype=np.uint16)
    got = orc.as_f64(bits)
    fails = [f"bf16 decode {hex(b)} -> {g} != {cases[b]}" for b, g in zip(cases, got) if g != cases[b]]
    z = orc.as_f64(np.array([0x8000], dtype=np.uint16))[0]
    if not (z == 0.0 and np.signbit(z)):
        fails.append("bf16 decode 0x8000 is not -0.0")
    return fails


ALL_PINS = [pin_bf16_decode, pin_column_slice, pin_zero_weight_closed_form, pin_rows_sum_to_zero, pin_ignored_rows,
            pin_finite_differences, pin_shift_invariance, pin_row_permutation,
            pin_torch_cross_entropy, pin_torch_cross_entropy_sum, pin_finite_differences_sum,
            pin_single_class, pin_no_valid_rows,
            pin_worked_example, pin_block_invariance, pin_row_sampled_pieces]


def run_all(orc):
    fails = []
    for p in ALL_PINS:
        try:
            fails += p(orc)
        except Exception as e:  # a crash is a failed pin too
            fails.append(f"{p.__name__} raised {type(e).__name__}: {e}")
    return fails
