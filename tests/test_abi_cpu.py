"""The C ABI without a GPU: the library loads, exports every entry point
include/lce.h declares, sizes workspaces, and rejects bad arguments on the
host before touching CUDA."""
import ctypes
import os
import re

import pytest

import __graft_entry__
import lm_head_linear_chunked_gb300 as lce

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "lce.h")


@pytest.fixture(scope="module", autouse=True)
def built():
    __graft_entry__.build()


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"LCE_API\s+[\w\s\*]*?\b(lce_\w+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_symbols()
    for n in ("lce_workspace_size", "lce_forward", "lce_backward", "lce_fused_fwd_bwd", "lce_check_status",
              "lce_status_string", "lce_chunk_rows", "lce_debug_gemm", "lce_debug_wait_timeout"):
        assert n in names


def test_library_exports_every_declared_symbol():
    L = ctypes.CDLL(lce.library_path)
    for n in declared_symbols():
        assert hasattr(L, n), n
    assert set(declared_symbols()) <= set(lce._SIGS)


def test_bounds_checking_library_has_the_same_entry_points():
    """liblce_debug.so (the sources compiled with LCE_DEBUG) is built beside
    liblce.so and exports the same declared entry points; its host-side
    argument checks answer the same way."""
    from lm_head_linear_chunked_gb300 import build
    lib_path, obj_dir, flags = build._variant(True)
    assert lib_path.endswith("liblce_debug.so") and "-DLCE_DEBUG" in flags and obj_dir != build.BUILD_DIR
    assert os.path.exists(lib_path)
    D = ctypes.CDLL(lib_path)
    for n in declared_symbols():
        assert hasattr(D, n), n
    out = ctypes.c_size_t(0)
    f = D.lce_workspace_size
    f.argtypes = [ctypes.c_int64] * 4 + [ctypes.c_int, ctypes.c_int, ctypes.POINTER(ctypes.c_size_t)]
    assert f(4096, 1024, 32768, 256, 1, lce.WS_FUSED, ctypes.byref(out)) == 0
    assert out.value == lce.lce_workspace_size(4096, 1024, 32768, 256, True, lce.WS_FUSED)
    assert f(0, 1024, 32768, 256, 1, lce.WS_FUSED, ctypes.byref(out)) == 1  # LCE_ERR_INVALID_ARG
    g = D.lce_status_string
    g.restype = ctypes.c_char_p
    g.argtypes = [ctypes.c_int]
    assert b"bounds" in g(7)


def test_status_strings():
    for code, name in lce.STATUS.items():
        assert lce.lce_status_string(code)
    assert lce.lce_status_string(99) == "unknown status"


@pytest.mark.parametrize("N,chunk,expect", [(512, 256, 256), (512, 0, 512), (100000, 0, 8192), (7, 1000, 7),
                                            (131072, 0, 8192), (4096, 1, 1)])
def test_chunk_rows(N, chunk, expect):
    assert lce.lce_chunk_rows(N, 1024, 32768, chunk) == expect


def test_workspace_sizes():
    N, H, V = 131072, 4096, 151936
    f = lce.lce_workspace_size(N, H, V, 0, False, lce.WS_FORWARD)
    b = lce.lce_workspace_size(N, H, V, 0, False, lce.WS_BACKWARD)
    fb = lce.lce_workspace_size(N, H, V, 0, False, lce.WS_FUSED)
    C, ldg, n_vt = 8192, V, -(-V // 256)
    second = C * ldg * 2 + 2 * n_vt * C * 4        # the overlapped chunk's E and half-tile maxes
    assert fb >= max(f, b) and fb <= f + b + second
    assert b >= C * V * 2                          # one chunk of fp16 P
    assert fb < N * V * 2 / 3                      # far below the logits it replaces
    with_bias = lce.lce_workspace_size(N, H, V, 0, True, lce.WS_FUSED)
    assert with_bias > b                           # no overlap with a bias: one E buffer
    assert with_bias < fb
    assert lce.lce_workspace_size(N, H, V, 256, False, lce.WS_FUSED) < fb
    # the fused call's minimum: one chunk of E, no overlap
    fmin = lce.lce_workspace_size(N, H, V, 0, False, lce.WS_FUSED_MIN)
    assert fmin == fb - second and max(f, b) <= fmin <= f + b
    assert lce.lce_workspace_size(N, H, V, 0, True, lce.WS_FUSED_MIN) == with_bias
    assert lce.lce_workspace_size(N, H, V, 128, False, lce.WS_FUSED_MIN) == \
        lce.lce_workspace_size(N, H, V, 128, False, lce.WS_FUSED)  # chunks too small to overlap


@pytest.mark.parametrize("args,code", [
    ((0, 64, 10, 0), 1), ((10, 64, 0, 0), 1), ((10, 0, 10, 0), 1), ((10, 64, 10, -1), 1),
    ((10, 100, 10, 0), 2), ((10, 32, 10, 0), 2), ((2**31, 64, 10, 0), 2),
])
def test_workspace_size_rejects(args, code):
    with pytest.raises(lce.LCEError) as e:
        lce.lce_workspace_size(*args, False, lce.WS_FUSED)
    assert e.value.status == code


def test_workspace_which_is_checked_4():
    with pytest.raises(lce.LCEError) as e:
        lce.lce_workspace_size(16, 64, 32, 0, False, 4)
    assert e.value.status == 1


def test_workspace_which_is_checked():
    with pytest.raises(lce.LCEError) as e:
        lce.lce_workspace_size(10, 64, 10, 0, False, 7)
    assert e.value.status == 1


# Fake, aligned, never-dereferenced addresses: these calls must return before
# any CUDA work, so they run without a GPU.
A = 1 << 20


def fwd(**kw):
    args = dict(N=16, H=64, V=32, X=A, W=A, b=None, y=A, ignore_index=-100, chunk_rows=0, loss=A, lse=A,
                n_valid=None, ws=A, ws_bytes=1 << 30, stream=None)
    args.update(kw)
    lce.lce_forward(*args.values())


def bwd(**kw):
    args = dict(N=16, H=64, V=32, X=A, W=A, b=None, y=A, ignore_index=-100, chunk_rows=0, lse=A, grad_scale=1.0,
                d_grad_output=None, grad_X=A, grad_W=A, grad_b=None, grad_W_acc=A, grad_b_acc=None, ws=A,
                ws_bytes=1 << 30, stream=None)
    args.update(kw)
    lce.lce_backward(*args.values())


@pytest.mark.parametrize("kw,code", [
    (dict(X=None), 1), (dict(W=None), 1), (dict(y=None), 1), (dict(lse=None), 1), (dict(loss=None), 1),
    (dict(ws=None), 1), (dict(X=A + 2), 1), (dict(ws=A + 16), 1), (dict(ws_bytes=100), 3),
    (dict(N=-3), 1), (dict(H=65), 2), (dict(chunk_rows=-5), 1),
])
def test_forward_host_errors(kw, code):
    with pytest.raises(lce.LCEError) as e:
        fwd(**kw)
    assert e.value.status == code


@pytest.mark.parametrize("kw,code", [
    (dict(grad_W_acc=None), 1), (dict(grad_b=A), 1), (dict(grad_b_acc=A), 1), (dict(b=A), 1),
    (dict(grad_W=A + 8), 1), (dict(ws_bytes=1000), 3),
])
def test_backward_host_errors(kw, code):
    with pytest.raises(lce.LCEError) as e:
        bwd(**kw)
    assert e.value.status == code


def test_debug_entry_points_host_errors():
    with pytest.raises(lce.LCEError) as e:
        lce.lce_debug_gemm(3, 128, 128, 64, A, A, A, A, 4096, None)
    assert e.value.status == 1
    with pytest.raises(lce.LCEError) as e:
        lce.lce_debug_gemm(0, 128, 100, 64, A, A, A, A, 4096, None)
    assert e.value.status == 2
    with pytest.raises(lce.LCEError) as e:
        lce.lce_debug_wait_timeout(10, A, 8, None)
    assert e.value.status == 3
    assert lce.lce_check_status(None, None) == 1


@pytest.mark.parametrize("kw,code", [
    (dict(d_grad_output=None), 1), (dict(grad_W=None), 1), (dict(grad_b=A), 1), (dict(grad_X=A + 4), 1),
    (dict(N=0), 1), (dict(H=12), 2),
])
def test_scale_grads_host_errors(kw, code):
    args = dict(N=16, H=64, V=32, d_grad_output=A, grad_X=A, grad_W_acc=A, grad_W=A, grad_b_acc=None,
                grad_b=None, stream=None)
    args.update(kw)
    with pytest.raises(lce.LCEError) as e:
        lce.lce_scale_grads(*args.values())
    assert e.value.status == code


def test_profile_end_without_begin_is_empty():
    lce.lce_profile_begin()
    out = lce.lce_profile_end()
    assert set(out) == set(lce.PROFILE_KINDS)
    assert all(v == (0.0, 0) for v in out.values())


@pytest.mark.parametrize("flags", [lce.ACCUMULATE, 4, 1 << 31])
def test_forward_ex_rejects_flags(flags):
    # accumulate has no meaning without gradients; unknown bits are errors
    args = dict(N=16, H=64, V=32, X=A, W=A, b=None, y=A, ignore_index=-100, chunk_rows=0, loss=A, lse=A,
                n_valid=None, ws=A, ws_bytes=1 << 30, stream=None, flags=flags)
    with pytest.raises(lce.LCEError) as e:
        lce.lce_forward_ex(*args.values())
    assert e.value.status == 1


@pytest.mark.parametrize("flags", [4, 8 | lce.REDUCTION_SUM])
def test_backward_ex_rejects_unknown_flags(flags):
    args = dict(N=16, H=64, V=32, X=A, W=A, b=None, y=A, ignore_index=-100, chunk_rows=0, lse=A, grad_scale=1.0,
                d_grad_output=None, grad_X=A, grad_W=A, grad_b=None, grad_W_acc=A, grad_b_acc=None, ws=A,
                ws_bytes=1 << 30, stream=None, flags=flags)
    with pytest.raises(lce.LCEError) as e:
        lce.lce_backward_ex(*args.values())
    assert e.value.status == 1


def test_reduction_names_are_checked():
    assert lce._flags("sum", True) == lce.REDUCTION_SUM | lce.ACCUMULATE
    assert lce._flags("mean", False) == 0
    with pytest.raises(ValueError):
        lce._flags("none", False)


@pytest.mark.parametrize("tiles,slots,kb,want", [
    (496, 76, 2374, (456, 40, 7, 340)),   # 8192-row chunk, 7782 valid rows, H = 4096, V = 151936
    (456, 76, 2374, (456, 0, 1, 2374)),   # whole rounds: nothing to split
    (151, 76, 2374, (151, 0, 1, 2374)),   # 75 tiles in the last round: no split saves an eighth of a tile
    (40, 76, 20, (40, 0, 1, 20)),         # K too short to split
    (0, 76, 100, (0, 0, 1, 100)),         # no valid rows
    (32, 76, 64, (0, 32, 2, 32)),         # fewer tiles than pairs: all of them split
    (5, 0, 64, (5, 0, 1, 64)),
])
def test_gradx_tail_plan(tiles, slots, kb, want):
    assert lce.lce_debug_gradx_tail_plan(tiles, slots, kb) == want


@pytest.mark.parametrize("tiles,slots,kb,want", [
    (248, 76, 2374, (228, 20, 7, 340)),   # 256 x 512 tiles of an 8192-row chunk (7782 valid rows), H = 4096
    (64, 76, 64, (64, 0, 1, 64)),         # 64 x 4 slices would pass the 160 partial tiles of 512 columns
    (20, 76, 128, (0, 20, 7, 19)),
])
def test_gradx_tail_plan_wide_tiles(tiles, slots, kb, want):
    assert lce.lce_debug_gradx_tail_plan(tiles, slots, kb, 512) == want


def test_gradx_tail_plan_properties():
    """On random launches: the slices cover K without an empty one, the
    partial tiles fit the workspace (320 of 256 columns, 160 of 512), and the split taken is the
    shortest tail among the allowed ones (none when none saves an eighth)."""
    rng = __import__("random").Random(5)

    def tail_time(r, s, slots):
        return -(-r * s // slots) / s

    for _ in range(3000):
        slots = rng.choice([1, 2, 37, 75, 76, 80, 148])
        tiles = rng.randrange(0, 6 * slots + 3)
        kb = rng.choice([1, 15, 32, 64, 127, 128, 2374, rng.randrange(1, 3000)])
        cols = rng.choice([256, 512])
        full, tail, s, kps = lce.lce_debug_gradx_tail_plan(tiles, slots, kb, cols)
        cap = 320 * 256 // cols
        r = tiles % slots
        allowed = [t for t in range(2, 9) if r * t <= cap and kb >= 16 * t]
        good = [t for t in allowed if 8 * -(-r * t // slots) <= 7 * t]
        if tail == 0:
            assert (full, s, kps) == (tiles, 1, kb)
            assert r == 0 or not good
            continue
        assert full + tail == tiles and full % slots == 0 and tail == r
        assert 2 <= s <= 8 and tail * s <= cap and (s - 1) * kps < kb <= s * kps and kps >= 16
        assert 8 * -(-tail * s // slots) <= 7 * s
        assert all(tail_time(r, s, slots) <= tail_time(r, t, slots) for t in allowed)


def test_gradx_tail_plan_rejects():
    for args in [(-1, 76, 10), (10, -1, 10), (10, 76, -1), (2**31, 76, 10), (10, 76, 10, 384)]:
        with pytest.raises(lce.LCEError) as e:
            lce.lce_debug_gradx_tail_plan(*args)
        assert e.value.status == 1
