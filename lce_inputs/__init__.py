"""Seeded synthetic inputs for chunked linear cross-entropy workloads.

This module is shared by the oracle and by the GPU library's tests and
benchmark, and holds none of the loss's arithmetic: it only produces the
hidden states X, the head weight W, the bias b and the labels y that both
sides consume, bit for bit the same.

Workload recipe (the five head shapes below).  The pages' own workload is
SFT of Qwen3 models on PG-19 ("1M 토큰 이상 학습" page, "실행" section);
neither the text nor trained weights are available, so these draws stand in
for them, with the head shapes of the models the pages name:

* X ~ N(0, 1), W ~ N(0, (2/sqrt(H))^2), b ~ N(0, 0.1^2) where a bias is
  used; every value rounded to bf16.  The logits then have standard
  deviation 2, so the softmax is peaked rather than uniform.
* Labels follow a Zipf law with exponent 1.1 over the vocabulary, truncated
  to ranks 1..V and drawn by inverse CDF; token id = rank - 1.
* Ignored rows (label -100, the ignore index of the LlamaFactory chunk-loss
  plugin): either exactly round(p*N) distinct positions drawn without
  replacement (the positions with the smallest keys of a seeded stream), or
  the first floor(0.3 * seq_len) positions of every sequence (a prompt
  mask, as in SFT).

Random stream: counter-based SplitMix64 (Steele, Lea and Flood, OOPSLA
2014) keyed by (seed, tensor id); normals by the Box-Muller transform.
`normal_bf16_reference` is the definition, in numpy; `normal_bf16` is the
fast multi-threaded C twin in seeded.c (tests check the two agree bit for
bit).  Tensor ids: X=0, W=1, b=2, labels=3, ignore mask=4.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading
from dataclasses import dataclass
from typing import Optional

import numpy as np

IGNORE_INDEX = -100

TID_X, TID_W, TID_B, TID_LABELS, TID_MASK = 0, 1, 2, 3, 4

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "seeded.c")
_LIB = os.path.join(_HERE, "_seeded.so")

_M64 = (1 << 64) - 1
_GAMMA = 0x9E3779B97F4A7C15


# ---------------------------------------------------------------------------
# the definition (numpy)
# ---------------------------------------------------------------------------

def _mix64(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
    z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
    return z ^ (z >> np.uint64(31))


def stream_key(seed: int, tensor_id: int) -> int:
    """Key of stream (seed, tensor_id); same formula as seeded.c."""
    with np.errstate(over="ignore"):
        a = _mix64(np.array([(seed + _GAMMA) & _M64], dtype=np.uint64))
        t = np.uint64((tensor_id * 0xD1B54A32D192ED03) & _M64)
        return int(_mix64(a ^ t)[0])


def draws_u64(seed: int, tensor_id: int, start: int, count: int) -> np.ndarray:
    """Draws start..start+count-1 of stream (seed, tensor_id), as uint64."""
    key = np.uint64(stream_key(seed, tensor_id))
    n = np.arange(start, start + count, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix64(key + (n + np.uint64(1)) * np.uint64(_GAMMA))


def uniform53(u: np.ndarray) -> np.ndarray:
    """Top 53 bits of a uint64 draw as a double in [0, 1)."""
    return (u >> np.uint64(11)).astype(np.float64) * 2.0 ** -53


def f32_to_bf16_bits(f: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit pattern (uint16), round to nearest even."""
    u = np.ascontiguousarray(f, dtype=np.float32).view(np.uint32).astype(np.uint64)
    nan_or_inf = (u & np.uint64(0x7F800000)) == np.uint64(0x7F800000)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = ((u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)).astype(np.uint16)
    quiet = np.where((u & np.uint64(0x007FFFFF)) != 0, np.uint64(0x40), np.uint64(0))
    keep = ((u >> np.uint64(16)) | quiet).astype(np.uint16)
    return np.where(nan_or_inf, keep, r)


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    """bf16 bit pattern (uint16) -> float64, exactly."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def normal_bf16_reference(seed: int, tensor_id: int, start: int, count: int,
                          sigma: float) -> np.ndarray:
    """Elements start..start+count-1 of the N(0, sigma^2) stream, as bf16 bits."""
    if count == 0:
        return np.zeros(0, dtype=np.uint16)
    k0, k1 = start // 2, (start + count - 1) // 2
    pairs = np.arange(k0, k1 + 1, dtype=np.uint64)
    a = draws_u64(seed, tensor_id, 2 * k0, 2 * (k1 - k0 + 1))
    u1 = 1.0 - uniform53(a[0::2])
    u2 = uniform53(a[1::2])
    r = np.sqrt(-2.0 * np.log(u1))
    t = 6.283185307179586476925286766559 * u2
    vals = np.empty(2 * len(pairs), dtype=np.float64)
    vals[0::2] = r * np.cos(t)
    vals[1::2] = r * np.sin(t)
    off = start - 2 * k0
    v = vals[off:off + count] * sigma
    return f32_to_bf16_bits(v.astype(np.float32))


# ---------------------------------------------------------------------------
# the fast twin (C, multi-threaded)
# ---------------------------------------------------------------------------

_lib = None
_lib_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile seeded.c into _seeded.so next to it (gcc, no CUDA)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-ffp-contract=off",
                               "-o", tmp, _SRC, "-lm", "-lpthread"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lib_lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.lce_inputs_normal_bf16.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64,
                                                   ctypes.c_uint64, ctypes.c_double, ctypes.c_void_p,
                                                   ctypes.c_int]
            lib.lce_inputs_normal_bf16.restype = ctypes.c_int
            lib.lce_inputs_stream_key.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
            lib.lce_inputs_stream_key.restype = ctypes.c_uint64
            _lib = lib
    return _lib


def default_threads() -> int:
    return max(1, min(64, os.cpu_count() or 1))


def normal_bf16_into(ptr: int, seed: int, tensor_id: int, start: int, count: int,
                     sigma: float, threads: Optional[int] = None) -> None:
    """Write `count` bf16 values (uint16 bits) to host address `ptr`."""
    if count <= 0:
        return
    rc = _load().lce_inputs_normal_bf16(seed, tensor_id, start, count, float(sigma),
                                        ctypes.c_void_p(ptr), threads or default_threads())
    if rc != 0:
        raise RuntimeError("lce_inputs: could not start generator threads")


def normal_bf16(seed: int, tensor_id: int, start: int, count: int, sigma: float,
                threads: Optional[int] = None) -> np.ndarray:
    out = np.empty(count, dtype=np.uint16)
    normal_bf16_into(out.ctypes.data, seed, tensor_id, start, count, sigma, threads)
    return out


# ---------------------------------------------------------------------------
# labels and ignore masks
# ---------------------------------------------------------------------------

def zipf_labels(seed: int, n: int, V: int, s: float = 1.1) -> np.ndarray:
    """n labels, P(token k-1) proportional to k^-s for ranks k = 1..V (inverse CDF)."""
    w = np.arange(1, V + 1, dtype=np.float64) ** (-s)
    cdf = np.cumsum(w)
    cdf /= cdf[-1]
    u = uniform53(draws_u64(seed, TID_LABELS, 0, n))
    lab = np.searchsorted(cdf, u, side="right")
    return np.minimum(lab, V - 1).astype(np.int64)


def random_ignore_positions(seed: int, n: int, p: float) -> np.ndarray:
    """Exactly round(p*n) distinct positions, without replacement."""
    m = int(round(p * n))
    if m == 0:
        return np.zeros(0, dtype=np.int64)
    keys = draws_u64(seed, TID_MASK, 0, n)
    return np.sort(np.argsort(keys, kind="stable")[:m]).astype(np.int64)


def prefix_ignore_positions(n: int, seq_len: int, frac: float) -> np.ndarray:
    """The first floor(frac*seq_len) positions of every seq_len-row sequence."""
    k = int(math.floor(frac * seq_len))
    starts = np.arange(0, n, seq_len, dtype=np.int64)
    pos = (starts[:, None] + np.arange(k, dtype=np.int64)[None, :]).reshape(-1)
    return pos[pos < n]


# ---------------------------------------------------------------------------
# the five workloads
# ---------------------------------------------------------------------------

@dataclass(frozen=True)
class Workload:
    name: str
    N: int
    seqs: int
    H: int
    V: int
    b_sigma: Optional[float]      # None: no bias
    mask: str                     # "random" or "prefix"
    mask_frac: float
    chunk_rows: int               # 0 = chosen by the library
    seed: int

    @property
    def seq_len(self) -> int:
        return self.N // self.seqs

    @property
    def x_sigma(self) -> float:
        return 1.0

    @property
    def w_sigma(self) -> float:
        return 2.0 / math.sqrt(self.H)

    @property
    def has_bias(self) -> bool:
        return self.b_sigma is not None

    def flops_fused(self) -> float:
        """8*N*H*V: forward logits, recomputed logits, grad_X and grad_W GEMMs."""
        return 8.0 * self.N * self.H * self.V


WORKLOADS = [
    Workload("tiny-N512-H256-V4096", 512, 2, 256, 4096, None, "random", 0.10, 256, 0),
    Workload("bias-N4096-H1024-V32768", 4096, 2, 1024, 32768, 0.1, "prefix", 0.30, 256, 1),
    Workload("qwen3-0.6b-head-N16384-H1024-V151936", 16384, 8, 1024, 151936, None, "prefix", 0.30, 256, 2),
    Workload("qwen3-8b-head-N131072-H4096-V151936", 131072, 1, 4096, 151936, None, "random", 0.05, 0, 3),
    Workload("qwen3-4b-head-N1048576-H2560-V151936", 1048576, 1, 2560, 151936, None, "random", 0.02, 0, 4),
]

BY_NAME = {w.name: w for w in WORKLOADS}


def labels(w: Workload) -> np.ndarray:
    y = zipf_labels(w.seed, w.N, w.V)
    if w.mask == "random":
        y[random_ignore_positions(w.seed, w.N, w.mask_frac)] = IGNORE_INDEX
    else:
        y[prefix_ignore_positions(w.N, w.seq_len, w.mask_frac)] = IGNORE_INDEX
    return y


def x_rows(w: Workload, rows: np.ndarray, threads: Optional[int] = None) -> np.ndarray:
    """bf16 bits of the given rows of X, shape [len(rows), H]."""
    out = np.empty((len(rows), w.H), dtype=np.uint16)
    for j, r in enumerate(np.asarray(rows, dtype=np.int64)):
        normal_bf16_into(out[j].ctypes.data, w.seed, TID_X, int(r) * w.H, w.H, w.x_sigma, 1)
    return out


def x_into(w: Workload, ptr: int, row0: int = 0, nrows: Optional[int] = None,
           threads: Optional[int] = None) -> None:
    nrows = w.N - row0 if nrows is None else nrows
    normal_bf16_into(ptr, w.seed, TID_X, row0 * w.H, nrows * w.H, w.x_sigma, threads)


def w_into(w: Workload, ptr: int, threads: Optional[int] = None) -> None:
    normal_bf16_into(ptr, w.seed, TID_W, 0, w.V * w.H, w.w_sigma, threads)


def b_into(w: Workload, ptr: int) -> None:
    if w.has_bias:
        normal_bf16_into(ptr, w.seed, TID_B, 0, w.V, w.b_sigma, 1)


def problem(w: Workload, threads: Optional[int] = None) -> dict:
    """The whole problem as numpy arrays (bf16 as uint16 bits)."""
    X = np.empty((w.N, w.H), dtype=np.uint16)
    W = np.empty((w.V, w.H), dtype=np.uint16)
    x_into(w, X.ctypes.data, threads=threads)
    w_into(w, W.ctypes.data, threads=threads)
    b = None
    if w.has_bias:
        b = np.empty(w.V, dtype=np.uint16)
        b_into(w, b.ctypes.data)
    return {"X": X, "W": W, "b": b, "y": labels(w)}
