"""Runtime contract of the C ABI on the GPU: the library allocates no device
memory of its own during a call, and it runs on the stream it is given."""
import numpy as np
import pytest

import lm_head_linear_chunked_gb300 as lce
from tests.gpu_util import dev_bf16, dev_i64
from tests.test_gpu_parity import random_problem

pytestmark = pytest.mark.gpu


def _buffers(N, H, V, chunk):
    import torch
    out = {"loss": torch.empty(1, device="cuda"), "lse": torch.empty(N, device="cuda"),
           "n_valid": torch.empty(1, dtype=torch.int64, device="cuda"),
           "gX": torch.empty((N, H), dtype=torch.bfloat16, device="cuda"),
           "gW": torch.empty((V, H), dtype=torch.bfloat16, device="cuda"),
           "acc": torch.empty((V, H), dtype=torch.float32, device="cuda")}
    nws = lce.lce_workspace_size(N, H, V, chunk, False, lce.WS_FUSED)
    out["ws"] = torch.empty(nws, dtype=torch.uint8, device="cuda")
    return out, nws


def _call(N, H, V, X, W, y, chunk, o, nws, stream):
    lce.lce_fused_fwd_bwd(N, H, V, X, W, None, y, -100, chunk, 1.0, None, o["loss"], o["lse"], o["n_valid"],
                          o["gX"], o["gW"], None, o["acc"], None, o["ws"], nws, stream)


def test_no_device_allocation_during_calls():
    import torch
    X, W, b, y = random_problem(41, 2048, 256, 8192, bias=False)
    N, H, V = 2048, 256, 8192
    Xd, Wd, yd = dev_bf16(X), dev_bf16(W), dev_i64(y)
    o, nws = _buffers(N, H, V, 512)
    s = torch.cuda.current_stream()
    _call(N, H, V, Xd, Wd, yd, 512, o, nws, s)          # warm-up: modules load here
    assert lce.lce_check_status(o["ws"], s) == 0
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        _call(N, H, V, Xd, Wd, yd, 512, o, nws, s)
    assert lce.lce_check_status(o["ws"], s) == 0
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, f"device free memory changed by {free0 - free1} bytes during the calls"


def test_side_stream_gives_the_same_bits():
    import torch
    X, W, b, y = random_problem(42, 1024, 128, 4096, bias=False)
    N, H, V = 1024, 128, 4096
    Xd, Wd, yd = dev_bf16(X), dev_bf16(W), dev_i64(y)
    a, nws = _buffers(N, H, V, 256)
    c, _ = _buffers(N, H, V, 256)
    _call(N, H, V, Xd, Wd, yd, 256, a, nws, torch.cuda.current_stream())
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        _call(N, H, V, Xd, Wd, yd, 256, c, nws, side)
    assert lce.lce_check_status(c["ws"], side) == 0
    torch.cuda.synchronize()
    for k in ("loss", "lse", "gX", "gW", "acc"):
        assert bool((a[k].view(-1) == c[k].view(-1)).all().item()), k


def test_cuda_graph_capture_and_replay():
    """After one warm-up call (which loads the kernels and sets their
    attributes), a fused call records into a CUDA graph; replays give the
    eager call's bits."""
    import torch
    X, W, b, y = random_problem(43, 1536, 128, 4096, bias=False)
    N, H, V = 1536, 128, 4096
    Xd, Wd, yd = dev_bf16(X), dev_bf16(W), dev_i64(y)
    eager, nws = _buffers(N, H, V, 512)
    s = torch.cuda.current_stream()
    _call(N, H, V, Xd, Wd, yd, 512, eager, nws, s)
    assert lce.lce_check_status(eager["ws"], s) == 0
    g_out, _ = _buffers(N, H, V, 512)
    side = torch.cuda.Stream()
    side.wait_stream(s)
    with torch.cuda.stream(side):
        _call(N, H, V, Xd, Wd, yd, 512, g_out, nws, side)   # warm-up on the capture stream
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        _call(N, H, V, Xd, Wd, yd, 512, g_out, nws, side)
    for _ in range(2):
        for k in ("loss", "lse", "gX", "gW", "acc"):
            g_out[k].zero_()
        graph.replay()
        torch.cuda.synchronize()
        for k in ("loss", "lse", "gX", "gW", "acc"):
            assert bool((eager[k].view(-1) == g_out[k].view(-1)).all().item()), k


def test_profile_counts_launches_per_role():
    """The per-kernel profiling hook sees one launch of each GEMM role per
    chunk in the fused call (no recomputed-logits GEMM there), and the
    recompute GEMM per chunk in lce_backward."""
    import torch
    X, W, b, y = random_problem(44, 1000, 128, 4096, bias=False)
    N, H, V, chunk = 1000, 128, 4096, 256
    chunks = -(-N // chunk)
    Xd, Wd, yd = dev_bf16(X), dev_bf16(W), dev_i64(y)
    o, nws = _buffers(N, H, V, chunk)
    s = torch.cuda.current_stream()
    lce.lce_profile_begin()
    _call(N, H, V, Xd, Wd, yd, chunk, o, nws, s)
    prof = lce.lce_profile_end()
    assert prof["logits_lse"][1] == chunks
    assert prof["recomputed_logits_softmax"][1] == 0
    assert prof["grad_w"][1] == chunks
    assert prof["grad_x"][1] in (chunks, 2 * chunks)  # a split product adds its reduction
    assert all(v[0] > 0 for k, v in prof.items() if v[1] > 0)
    nws_b = lce.lce_workspace_size(N, H, V, chunk, False, lce.WS_BACKWARD)
    ws_b = torch.empty(nws_b, dtype=torch.uint8, device="cuda")
    lce.lce_profile_begin()
    lce.lce_backward(N, H, V, Xd, Wd, None, yd, -100, chunk, o["lse"], 1.0, None, o["gX"], o["gW"], None,
                     o["acc"], None, ws_b, nws_b, s)
    prof = lce.lce_profile_end()
    assert prof["recomputed_logits_softmax"][1] == chunks and prof["logits_lse"][1] == 0
