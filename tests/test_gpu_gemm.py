"""The tensor-core GEMM core alone (lce_debug_gemm, through the C ABI)
against a float64 product of the same bf16 operands, for the three operand
layouts the loss uses: logits X W^T, grad_X = G W, grad_W = G^T X."""
import pytest

import lm_head_linear_chunked_gb300 as lce

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("layout", [0, 1, 2], ids=["A_Bt", "A_B", "At_B"])
@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (256, 512, 256), (200, 264, 72), (384, 1024, 1000),
                                   (1000, 304, 4096), (8, 8, 8), (4096, 4096, 512)])
def test_debug_gemm_matches_float64(layout, M, N, K):
    import torch
    torch.manual_seed(M * 7 + N * 3 + K + layout)
    dev = torch.device("cuda")
    a_shape = (M, K) if layout in (0, 1) else (K, M)
    b_shape = (N, K) if layout == 0 else (K, N)
    A = torch.randn(a_shape, device=dev).to(torch.bfloat16)
    B = torch.randn(b_shape, device=dev).to(torch.bfloat16)
    D = torch.full((M, N), float("nan"), dtype=torch.float32, device=dev)
    ws = torch.zeros(256, dtype=torch.uint8, device=dev)
    s = torch.cuda.current_stream()
    lce.lce_debug_gemm(layout, M, N, K, A, B, D, ws, ws.numel(), s)
    assert lce.lce_check_status(ws, s) == 0
    Ad, Bd = A.double(), B.double()
    ref = Ad @ Bd.T if layout == 0 else (Ad @ Bd if layout == 1 else Ad.T @ Bd)
    err = (D.double() - ref).abs().max().item()
    scale = ref.abs().max().item()
    assert err <= 1e-5 * scale * max(1.0, K / 512), f"max abs err {err} (max |ref| {scale})"


def test_wait_timeout_reports_status():
    import torch
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream()
    lce.lce_debug_wait_timeout(2000, ws, ws.numel(), s)
    assert lce.lce_check_status(ws, s) == 5  # LCE_ERR_TIMEOUT
    # the context is still usable afterwards
    x = torch.ones(4, device="cuda")
    assert float((x * 2).sum().item()) == 8.0
