"""GPU path (through the C ABI) against the CPU FP64 oracle on small seeded
problems: every output element by element, plus chunk-size invariance,
ragged shapes, the degenerate cases, the device error statuses, and guard
bytes around every output (out-of-bounds writes would show there)."""
import numpy as np
import pytest

import lce_inputs as L
import lm_head_linear_chunked_gb300 as lce
import oracle
from tests.gpu_util import (BF16_GRAD_TOL, F32_ACC_TOL, LSE_ATOL, assert_grad, check_against_oracle, dev_bf16,
                            dev_i64, host_f64)

pytestmark = pytest.mark.gpu

GUARD = 256  # elements of guard before and after each output
PATTERN = {"f32": 0x7FBADBAD, "bf16": 0x7FBA, "i64": 0x7FBADBAD7FBADBAD}


class Guarded:
    """An output tensor with guard elements on both sides."""

    def __init__(self, shape, kind):
        import torch
        dt = {"f32": torch.int32, "bf16": torch.int16, "i64": torch.int64}[kind]
        view_dt = {"f32": torch.float32, "bf16": torch.bfloat16, "i64": torch.int64}[kind]
        n = int(np.prod(shape))
        pat = PATTERN[kind]
        pat = pat - (1 << {"f32": 32, "bf16": 16, "i64": 64}[kind]) if pat >= (1 << ({"f32": 31, "bf16": 15, "i64": 63}[kind])) else pat
        self.buf = torch.full((n + 2 * GUARD,), pat, dtype=dt, device="cuda")
        self.pat = pat
        self.t = self.buf[GUARD:GUARD + n].view(view_dt).view(*shape)

    def intact(self):
        return bool((self.buf[:GUARD] == self.pat).all().item() and (self.buf[-GUARD:] == self.pat).all().item())


def random_problem(seed, N, H, V, bias, ignore_frac=0.1, w_sigma=None):
    w_sigma = w_sigma if w_sigma is not None else 2.0 / np.sqrt(H)
    X = L.normal_bf16(seed, L.TID_X, 0, N * H, 1.0).reshape(N, H)
    W = L.normal_bf16(seed, L.TID_W, 0, V * H, w_sigma).reshape(V, H)
    b = L.normal_bf16(seed, L.TID_B, 0, V, 0.1) if bias else None
    y = L.zipf_labels(seed, N, V)
    y[L.random_ignore_positions(seed, N, ignore_frac)] = L.IGNORE_INDEX
    return X, W, b, y


def run_fused(X, W, b, y, chunk_rows, grad_scale=1.0, grad_output=None, ignore_index=-100):
    import torch
    N, H = X.shape
    V = W.shape[0]
    has_b = b is not None
    out = {
        "loss": Guarded((1,), "f32"), "lse": Guarded((N,), "f32"), "n_valid": Guarded((1,), "i64"),
        "grad_X": Guarded((N, H), "bf16"), "grad_W": Guarded((V, H), "bf16"),
        "grad_W_acc": Guarded((V, H), "f32"),
    }
    if has_b:
        out["grad_b"] = Guarded((V,), "bf16")
        out["grad_b_acc"] = Guarded((V,), "f32")
    nws = lce.lce_workspace_size(N, H, V, chunk_rows, has_b, lce.WS_FUSED)
    ws = torch.empty(nws + 4096, dtype=torch.uint8, device="cuda")
    ws[nws:] = 0xA5
    go = torch.tensor([grad_output], dtype=torch.float32, device="cuda") if grad_output is not None else None
    s = torch.cuda.current_stream()
    Xd, Wd, bd, yd = dev_bf16(X), dev_bf16(W), dev_bf16(b), dev_i64(y)
    lce.lce_fused_fwd_bwd(N, H, V, Xd, Wd, bd, yd, ignore_index, chunk_rows, grad_scale, go,
                          out["loss"].t, out["lse"].t, out["n_valid"].t, out["grad_X"].t, out["grad_W"].t,
                          out["grad_b"].t if has_b else None, out["grad_W_acc"].t,
                          out["grad_b_acc"].t if has_b else None, ws, nws, s)
    status = lce.lce_check_status(ws, s)
    for k, g in out.items():
        assert g.intact(), f"guard bytes around {k} overwritten"
    assert bool((ws[nws:] == 0xA5).all().item()), "write past the end of the workspace"
    res = {k: g.t for k, g in out.items()}
    res["status"] = status
    return res


def oracle_of(X, W, b, y, grad_scale=1.0, grad_output=1.0):
    return oracle.fused(X, W, b, y, grad_scale=grad_scale, grad_output=grad_output)


# ---------------------------------------------------------------- the two small workloads

def test_tiny_workload_fused():
    w = L.WORKLOADS[0]
    P = L.problem(w)
    out = run_fused(P["X"], P["W"], None, P["y"], w.chunk_rows)
    assert out["status"] == 0
    check_against_oracle(out, oracle_of(P["X"], P["W"], None, P["y"]), has_bias=False)


def test_bias_workload_fused():
    w = L.WORKLOADS[1]
    P = L.problem(w)
    out = run_fused(P["X"], P["W"], P["b"], P["y"], w.chunk_rows)
    assert out["status"] == 0
    check_against_oracle(out, oracle_of(P["X"], P["W"], P["b"], P["y"]), has_bias=True)


def test_forward_and_backward_entry_points():
    import torch
    w = L.WORKLOADS[1]
    P = L.problem(w)
    X, W, b, y = dev_bf16(P["X"]), dev_bf16(P["W"]), dev_bf16(P["b"]), dev_i64(P["y"])
    f = lce.forward(X, W, b, y, chunk_rows=w.chunk_rows)
    s = torch.cuda.current_stream()
    assert lce.lce_check_status(f["ws"], s) == 0
    ref = oracle_of(P["X"], P["W"], P["b"], P["y"])
    check_against_oracle(f, ref, has_bias=True, bwd=False)
    # backward from the GPU's own lse, and from the oracle's lse
    for lse in (f["lse"], torch.from_numpy(ref["lse"].astype(np.float32)).cuda()):
        g = lce.backward(X, W, b, y, lse, chunk_rows=w.chunk_rows)
        assert lce.lce_check_status(g["ws"], s) == 0
        check_against_oracle(g, ref, has_bias=True, fwd=False)
    # grad_X may be skipped
    g = lce.backward(X, W, b, y, f["lse"], chunk_rows=w.chunk_rows, want_grad_X=False)
    assert lce.lce_check_status(g["ws"], s) == 0
    check_against_oracle(g, ref, has_bias=True, fwd=False, grad_x=False)


# ---------------------------------------------------------------- chunking

def test_chunk_size_invariance():
    """Rows are independent, so lse and loss are bitwise the same for every
    chunk size; gradients agree within the fp32-accumulation tolerance."""
    X, W, b, y = random_problem(21, 300, 128, 1000, bias=True)
    ref = oracle_of(X, W, b, y)
    base = None
    for chunk in (300, 0, 1, 7, 128, 256, 1000):
        out = run_fused(X, W, b, y, chunk)
        assert out["status"] == 0
        check_against_oracle(out, ref, has_bias=True)
        cur = (out["loss"].cpu().numpy().tobytes(), out["lse"].cpu().numpy().tobytes())
        if base is None:
            base = cur
        assert cur == base, f"lse/loss bits changed with chunk_rows={chunk}"


@pytest.mark.parametrize("N,H,V,bias", [
    (1, 64, 8, False), (129, 64, 257 * 8, True), (300, 192, 999, True), (513, 256, 4104, False),
    (77, 320, 2056, False), (256, 64, 16, True),
])
def test_ragged_shapes(N, H, V, bias):
    X, W, b, y = random_problem(N + H + V, N, H, V, bias=bias, ignore_frac=0.2)
    ref = oracle_of(X, W, b, y)
    for chunk in (0, 100):
        out = run_fused(X, W, b, y, chunk)
        assert out["status"] == 0
        check_against_oracle(out, ref, has_bias=bias)


# ---------------------------------------------------------------- scales and degenerate cases

def test_grad_scale_and_grad_output():
    X, W, b, y = random_problem(5, 256, 128, 512, bias=True)
    out = run_fused(X, W, b, y, 64, grad_scale=0.5, grad_output=3.0)
    assert out["status"] == 0
    ref = oracle_of(X, W, b, y, grad_scale=0.5, grad_output=3.0)
    check_against_oracle(out, ref, has_bias=True)


def test_all_rows_ignored():
    X, W, b, y = random_problem(6, 200, 64, 300 * 8 // 8 * 8, bias=True)
    y[:] = L.IGNORE_INDEX
    out = run_fused(X, W, b, y, 64)
    assert out["status"] == 0
    assert float(out["loss"].item()) == 0.0 and int(out["n_valid"].item()) == 0
    for k in ("grad_X", "grad_W", "grad_W_acc", "grad_b", "grad_b_acc"):
        assert float(out[k].float().abs().max().item()) == 0.0, k
    ref = oracle_of(X, W, b, y)
    assert np.abs(host_f64(out["lse"]) - ref["lse"]).max() <= LSE_ATOL


def test_single_class_vocabulary():
    """V = 1: the only class has probability 1, so the loss and every gradient
    are 0; fp32 leaves only rounding-level residues (p - 1 ~ 1e-7)."""
    for bias in (False, True):
        X, W, b, y = random_problem(7, 256, 64, 1, bias=bias)
        y[y != L.IGNORE_INDEX] = 0
        out = run_fused(X, W, b, y, 100)
        assert out["status"] == 0
        assert abs(float(out["loss"].item())) <= 1e-6
        ks = ("grad_X", "grad_W", "grad_W_acc") + (("grad_b", "grad_b_acc") if bias else ())
        for k in ks:
            assert float(out[k].float().abs().max().item()) <= 1e-6, k


def test_zero_weight_gives_log_V():
    """W = 0: every logit is 0, so loss = lse = ln V (a closed form)."""
    import math
    X, W, b, y = random_problem(8, 300, 128, 4096, bias=False)
    W[:] = 0
    out = run_fused(X, W, None, y, 128)
    assert out["status"] == 0
    assert abs(float(out["loss"].item()) - math.log(4096)) <= 1e-6 * math.log(4096)
    assert np.abs(host_f64(out["lse"]) - math.log(4096)).max() <= 1e-5
    assert float(out["grad_X"].float().abs().max().item()) == 0.0


def test_large_logits_do_not_overflow():
    X, W, b, y = random_problem(9, 256, 256, 2048, bias=False, w_sigma=1.0)  # logits ~ N(0, 256)
    out = run_fused(X, W, None, y, 0)
    assert out["status"] == 0
    ref = oracle_of(X, W, None, y)
    check_against_oracle(out, ref, has_bias=False)


def test_custom_ignore_index():
    X, W, b, y = random_problem(10, 256, 64, 512, bias=False)
    y[y == L.IGNORE_INDEX] = 511
    y[::5] = -1
    out = run_fused(X, W, None, y, 0, ignore_index=-1)
    assert out["status"] == 0
    ref = oracle.fused(X, W, None, y, ignore_index=-1)
    check_against_oracle(out, ref, has_bias=False)


def test_label_out_of_range_sets_status():
    X, W, b, y = random_problem(11, 128, 64, 256, bias=False)
    y[17] = 256
    out = run_fused(X, W, None, y, 0)
    assert out["status"] == 4  # LCE_ERR_LABEL_RANGE
    y[17] = -7
    out = run_fused(X, W, None, y, 0)
    assert out["status"] == 4


def test_repeatable_bits():
    X, W, b, y = random_problem(12, 384, 128, 2048, bias=True)
    a = run_fused(X, W, b, y, 128)
    c = run_fused(X, W, b, y, 128)
    for k in ("loss", "lse", "grad_X", "grad_W", "grad_W_acc", "grad_b", "grad_b_acc"):
        assert bool((a[k].view(-1) == c[k].view(-1)).all().item()) or k == "loss" and a[k].item() == c[k].item(), k


def test_chunk_spanning_several_label_blocks():
    """A chunk of more than 8192 rows is sorted and scattered in several
    label blocks; the labels repeat across blocks (Zipf), so the blocks'
    one-hot updates of the same grad_W rows must all land."""
    X, W, b, y = random_problem(13, 20000, 64, 512, bias=True)
    ref = oracle_of(X, W, b, y)
    for chunk in (20000, 9000):
        out = run_fused(X, W, b, y, chunk)
        assert out["status"] == 0
        check_against_oracle(out, ref, has_bias=True)


def test_overlapped_rescale_matches_oracle_and_recompute():
    """Chunks of >= 4096 rows without a bias: each chunk's forward also turns
    the previous chunk's kept exponentials into P (the epilogue warps' side
    job), and chunk c-1's backward runs after chunk c's forward.  Every
    output against the oracle, and grad_W_acc against the recomputing
    lce_forward + lce_backward path."""
    import torch
    X, W, b, y = random_problem(91, 9000, 128, 4096, bias=False, ignore_frac=0.2)
    ref = oracle_of(X, W, b, y)
    out = run_fused(X, W, b, y, 4096)
    assert out["status"] == 0
    check_against_oracle(out, ref, has_bias=False)
    Xd, Wd, yd = dev_bf16(X), dev_bf16(W), dev_i64(y)
    f = lce.forward(Xd, Wd, None, yd, chunk_rows=4096)
    g = lce.backward(Xd, Wd, None, yd, f["lse"], chunk_rows=4096)
    assert lce.lce_check_status(g["ws"], torch.cuda.current_stream()) == 0
    d = (out["grad_W_acc"].double() - g["grad_W_acc"].double()).abs().max().item()
    assert d <= 2e-4 * g["grad_W_acc"].abs().max().item(), d  # both within 1e-4 of the oracle
    # With only the minimum workspace the rescale runs as its own kernel,
    # after the chunk's forward: the same arithmetic, so the same bits.
    N, H = X.shape
    V = W.shape[0]
    nmin = lce.lce_workspace_size(N, H, V, 4096, False, lce.WS_FUSED_MIN)
    assert nmin < lce.lce_workspace_size(N, H, V, 4096, False, lce.WS_FUSED)
    seq = lce.fused(Xd, Wd, None, yd, chunk_rows=4096,
                    ws=torch.empty(nmin, dtype=torch.uint8, device="cuda"))
    assert lce.lce_check_status(seq["ws"], torch.cuda.current_stream()) == 0
    for k in ("loss", "lse", "grad_X", "grad_W", "grad_W_acc"):
        assert torch.equal(seq[k], out[k]), k
