"""Both forms of the tensor-core GEMM, whichever one the library uses by
default: one CTA per 128x256 tile (tcgen05 cta_group::1), and pairs of
CTAs on neighbouring SMs sharing 256x256 tiles (cta_group::2).  Each form is
checked against float64 products (the bare GEMM core) and against the FP64
oracle (the fused call), on shapes with ragged edges in every dimension,
odd numbers of 128-row tiles (a pair whose second half lies past the
rows), compacted chunks, split-K grad_X, and chunks large enough for the
forward to rescale the previous chunk's exponentials as a side job."""
import pytest

import lce_inputs as L
import lm_head_linear_chunked_gb300 as lce
from tests.gpu_util import check_against_oracle
from tests.test_gpu_parity import oracle_of, random_problem, run_fused

pytestmark = pytest.mark.gpu

FORMS = ["single", "pair"]


def test_pair_form_available():
    # the pair tests below run the pair form, not a fallback to single CTAs
    import torch
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    slots = lce.lce_gemm_pair_slots()
    assert sms // 4 <= slots <= sms // 2, (slots, sms)


@pytest.fixture(params=FORMS)
def form(request):
    prev = lce.lce_set_gemm_form(request.param)
    yield request.param
    lce.lce_set_gemm_form(prev)


@pytest.mark.parametrize("layout", [0, 1, 2], ids=["A_Bt", "A_B", "At_B"])
@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (256, 512, 256), (200, 264, 72), (384, 1024, 1000),
                                   (1000, 304, 4096), (8, 8, 8), (4096, 4096, 512), (640, 256, 128)])
def test_debug_gemm_forms(form, layout, M, N, K):
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
    assert err <= 1e-5 * scale * max(1.0, K / 512), f"{form}: max abs err {err} (max |ref| {scale})"


@pytest.mark.parametrize("N,H,V,bias,chunk", [
    (384, 128, 1000, False, 0),      # three 128-row tiles: one pair half past the rows
    (700, 192, 4100, True, 256),     # ragged rows and vocabulary, bias, 3 chunks
    (1300, 256, 2304, False, 640),   # ragged chunk of 20 rows
    (256, 512, 33000, False, 256),   # few output tiles: split-K grad_X
    (9000, 128, 4096, False, 4096),  # chunks of >= 4096 rows: each forward rescales the previous chunk's E
])
def test_fused_forms_match_oracle(form, N, H, V, bias, chunk):
    X, W, b, y = random_problem(31 + N, N, H, V, bias, ignore_frac=0.2)
    out = run_fused(X, W, b, y, chunk)
    assert out["status"] == 0
    ref = oracle_of(X, W, b, y)
    check_against_oracle(out, ref, has_bias=bias)


def test_forms_agree():
    """The two forms on the same problem: lse to a few FP32 ulps of the
    logits' scale, gradients to the fp16 operand rounding."""
    import torch
    X, W, b, y = random_problem(77, 1024, 256, 8192, False)
    outs = {}
    for f in FORMS:
        prev = lce.lce_set_gemm_form(f)
        try:
            outs[f] = run_fused(X, W, b, y, 512)
        finally:
            lce.lce_set_gemm_form(prev)
        assert outs[f]["status"] == 0
    a, p = outs["single"], outs["pair"]
    assert float((a["lse"] - p["lse"]).abs().max().item()) <= 1e-5
    acc = a["grad_W_acc"].double()
    assert float((acc - p["grad_W_acc"].double()).abs().max().item()) <= 1e-5 * float(acc.abs().max().item())
    gx = a["grad_X"].double()
    assert float((gx - p["grad_X"].double()).abs().max().item()) <= 1e-2 * float(gx.abs().max().item())
