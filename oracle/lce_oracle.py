"""CPU FP64 oracle for chunked linear cross-entropy.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
benchmark's CPU-baseline leg may import this module.  The GPU library
never calls it, shares no code with it, and must fail loudly rather than
fall back to it.

What it computes (plain definition, float64, every bf16 input converted
exactly to double):

  z[i, v]   = sum_h X[i, h] W[v, h] + b[v]           (b = 0 without a bias)
  lse[i]    = m_i + ln sum_v exp(z[i, v] - m_i),      m_i = max_v z[i, v]
  valid(i)  = y[i] != ignore_index
  n_valid   = #{i : valid(i)}
  loss      = (1 / n_valid) sum_{valid i} (lse[i] - z[i, y[i]])   (reduction "mean")
            =               sum_{valid i} (lse[i] - z[i, y[i]])   (reduction "sum")
  s         = grad_scale * grad_output / n_valid                  (mean)
            = grad_scale * grad_output                            (sum)
  G[i, v]   = s (exp(z[i, v] - lse[i]) - [v == y[i]])  for valid i, else 0
  grad_X    = G W,   grad_W = G^T X,   grad_b = sum_i G[i, :]

Sources, by page and section:
* LlamaFactory PR #10762 analysis page, section 4 (Chunk Loss implementation,
  `chunk_loss.py`): the loss of each row chunk is
  `F.cross_entropy(logits, labels, reduction="none", ignore_index=IGNORE_INDEX)`
  over the head's linear output; IGNORE_INDEX is -100; grad_weight and
  grad_bias are accumulated in FP32 and cast back to the weight dtype.
* Same page, section 3 (`BaseTrainer.fit`): the loss is normalised by the
  count of valid (non-ignored) tokens, with a guard against dividing by zero.
  That count is gathered over all ranks and micro-batches before the
  division, so a trainer may instead take the plain sum of a micro-batch's
  per-token losses and divide by its own count: reduction "sum".
* TRL "1M 토큰 이상 학습" page, section "매우 큰 logits 행렬: 청킹": the loss
  is a sum over rows and the softmax runs along one row's vocabulary, so
  any split of the rows gives the same result.  That is why this oracle may
  walk the rows in blocks of any size: each row is computed on its own.

Readings where the pages are silent:
* the per-token losses are reduced by a mean over valid rows;
* with no valid row, loss = 0 and every gradient is 0 (the trainer's
  division guard), lse is still defined for every row;
* lse is defined for ignored rows too (same formula);
* grad_scale * grad_output multiplies G before both gradient products
  (equivalent to scaling the saved gradients, as autograd's grad_output).

The full-problem functions materialise one block of rows' logits at a time.
The row-sampled functions let tests check the largest workloads row by row.
Matrix products use numpy's float64 matmul (a library primitive).
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from typing import Optional

import numpy as np

IGNORE_INDEX = -100


def as_f64(a) -> Optional[np.ndarray]:
    """bf16 bit patterns (uint16) -> float64 exactly; float arrays -> float64."""
    if a is None:
        return None
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def logits(X: np.ndarray, W: np.ndarray, b: Optional[np.ndarray]) -> np.ndarray:
    """z = X W^T + b for the given rows of X (float64)."""
    z = X @ W.T
    if b is not None:
        z += b[None, :]
    return z


def logsumexp_rows(z: np.ndarray) -> np.ndarray:
    """lse[i] = m_i + ln sum_v exp(z[i, v] - m_i), m_i = max_v z[i, v]."""
    m = z.max(axis=1)
    return m + np.log(np.exp(z - m[:, None]).sum(axis=1))


def valid_mask(y: np.ndarray, ignore_index: int = IGNORE_INDEX) -> np.ndarray:
    return np.asarray(y) != ignore_index


def count_valid(y: np.ndarray, ignore_index: int = IGNORE_INDEX) -> int:
    return int(valid_mask(y, ignore_index).sum())


def check_labels(y: np.ndarray, V: int, ignore_index: int = IGNORE_INDEX) -> None:
    """Labels must lie in [0, V) or equal ignore_index (cross_entropy's contract)."""
    y = np.asarray(y)
    bad = (y != ignore_index) & ((y < 0) | (y >= V))
    if bad.any():
        raise ValueError(f"label out of range at row {int(np.argmax(bad))}")


def grad_scale_per_row(grad_scale: float, grad_output: float, n_valid: int, reduction: str = "mean") -> float:
    """s = grad_scale * grad_output / n_valid (mean; 0 when there is no valid
    row), or grad_scale * grad_output (sum)."""
    if reduction == "sum":
        return float(grad_scale) * float(grad_output)
    if reduction != "mean":
        raise ValueError(f"reduction must be 'mean' or 'sum', got {reduction!r}")
    if n_valid == 0:
        return 0.0
    return float(grad_scale) * float(grad_output) / n_valid


def softmax_minus_onehot(z: np.ndarray, lse: np.ndarray, y: np.ndarray, s: float,
                         ignore_index: int = IGNORE_INDEX) -> np.ndarray:
    """G[i, v] = s (exp(z[i, v] - lse[i]) - [v == y[i]]) for valid rows, 0 otherwise."""
    G = np.exp(z - lse[:, None])
    ok = valid_mask(y, ignore_index)
    rows = np.nonzero(ok)[0]
    G[rows, np.asarray(y)[rows]] -= 1.0
    G[~ok, :] = 0.0
    return s * G


def _blocks(n: int, block_rows: int):
    return [(r, min(n, r + block_rows)) for r in range(0, n, block_rows)]


def _pool(threads: Optional[int]):
    return ThreadPoolExecutor(max_workers=threads or max(1, os.cpu_count() or 1))


def forward(X, W, b, y, ignore_index: int = IGNORE_INDEX, block_rows: int = 256,
            threads: Optional[int] = None, reduction: str = "mean") -> dict:
    """loss, lse [N] and n_valid of the whole problem."""
    X, W, b = as_f64(X), as_f64(W), as_f64(b)
    y = np.asarray(y, dtype=np.int64)
    N, V = X.shape[0], W.shape[0]
    check_labels(y, V, ignore_index)
    lse = np.empty(N)
    zt = np.zeros(N)

    def one(blk):
        r0, r1 = blk
        z = logits(X[r0:r1], W, b)
        lse[r0:r1] = logsumexp_rows(z)
        yy = y[r0:r1]
        ok = yy != ignore_index
        zt[r0:r1][ok] = z[np.nonzero(ok)[0], yy[ok]]

    with _pool(threads) as ex:
        list(ex.map(one, _blocks(N, block_rows)))
    ok = valid_mask(y, ignore_index)
    n_valid = int(ok.sum())
    total = float((lse[ok] - zt[ok]).sum())
    if reduction == "sum":
        loss = total
    elif reduction == "mean":
        loss = total / n_valid if n_valid else 0.0
    else:
        raise ValueError(f"reduction must be 'mean' or 'sum', got {reduction!r}")
    return {"loss": loss, "lse": lse, "n_valid": n_valid}


def backward(X, W, b, y, lse, ignore_index: int = IGNORE_INDEX, grad_scale: float = 1.0,
             grad_output: float = 1.0, block_rows: int = 256,
             threads: Optional[int] = None, reduction: str = "mean") -> dict:
    """grad_X [N,H], grad_W [V,H], grad_b [V] (None without a bias), given lse."""
    X, W, b = as_f64(X), as_f64(W), as_f64(b)
    y = np.asarray(y, dtype=np.int64)
    lse = np.asarray(lse, dtype=np.float64)
    N, H = X.shape
    V = W.shape[0]
    check_labels(y, V, ignore_index)
    s = grad_scale_per_row(grad_scale, grad_output, count_valid(y, ignore_index), reduction)
    grad_X = np.zeros((N, H))
    blocks = _blocks(N, block_rows)
    part_W = [None] * len(blocks)
    part_b = [None] * len(blocks)

    def one(j):
        r0, r1 = blocks[j]
        z = logits(X[r0:r1], W, b)
        G = softmax_minus_onehot(z, lse[r0:r1], y[r0:r1], s, ignore_index)
        grad_X[r0:r1] = G @ W
        part_W[j] = G.T @ X[r0:r1]
        part_b[j] = G.sum(axis=0)

    with _pool(threads) as ex:
        list(ex.map(one, range(len(blocks))))
    grad_W = np.zeros((V, H))
    grad_b = np.zeros(V)
    for j in range(len(blocks)):          # fixed order
        grad_W += part_W[j]
        grad_b += part_b[j]
    return {"grad_X": grad_X, "grad_W": grad_W, "grad_b": grad_b if b is not None else None}


def fused(X, W, b, y, ignore_index: int = IGNORE_INDEX, grad_scale: float = 1.0,
          grad_output: float = 1.0, block_rows: int = 256, threads: Optional[int] = None,
          reduction: str = "mean") -> dict:
    """forward() then backward() with the forward's lse."""
    f = forward(X, W, b, y, ignore_index, block_rows, threads, reduction)
    g = backward(X, W, b, y, f["lse"], ignore_index, grad_scale, grad_output, block_rows, threads, reduction)
    f.update(g)
    return f


# ---------------------------------------------------------------------------
# row-sampled pieces for the largest workloads
# ---------------------------------------------------------------------------

def rows_forward(X_rows, W, b, y_rows, ignore_index: int = IGNORE_INDEX) -> dict:
    """lse, target logit and per-row loss of the given rows (row-local work).

    For ignored rows the target logit and the row loss are NaN and 0."""
    Xr, W, b = as_f64(X_rows), as_f64(W), as_f64(b)
    y_rows = np.asarray(y_rows, dtype=np.int64)
    z = logits(Xr, W, b)
    lse = logsumexp_rows(z)
    ok = y_rows != ignore_index
    zt = np.full(len(y_rows), np.nan)
    zt[ok] = z[np.nonzero(ok)[0], y_rows[ok]]
    row_loss = np.where(ok, lse - np.where(ok, zt, 0.0), 0.0)
    return {"lse": lse, "z_target": zt, "row_loss": row_loss}


def rows_grad_X(X_rows, W, b, y_rows, lse_rows, s: float,
                ignore_index: int = IGNORE_INDEX) -> np.ndarray:
    """grad_X of the given rows: G[i, :] W with the scale s of the whole problem."""
    Xr, W, b = as_f64(X_rows), as_f64(W), as_f64(b)
    z = logits(Xr, W, b)
    G = softmax_minus_onehot(z, np.asarray(lse_rows, dtype=np.float64),
                             np.asarray(y_rows, dtype=np.int64), s, ignore_index)
    return G @ W


def grad_W_columns(X, W, b, y, h0: int, h1: int, ignore_index: int = IGNORE_INDEX,
                   grad_scale: float = 1.0, grad_output: float = 1.0, block_rows: int = 128,
                   threads: Optional[int] = None) -> dict:
    """Columns h0:h1 of grad_W = G^T X over ALL rows (reduction "mean"),
    with the whole problem's lse, loss and grad_b.

    Each block of rows gets its logits, its lse and its G (the definitions
    above, row by row), and contributes G^T X[:, h0:h1]; the blocks'
    contributions are added in row order.  This costs the full 2 N H V of
    logits but holds only one block's, so the FP32 accumulation over many
    chunks can be checked on all rows of a large problem."""
    X, W, b = as_f64(X), as_f64(W), as_f64(b)
    y = np.asarray(y, dtype=np.int64)
    N, V = X.shape[0], W.shape[0]
    check_labels(y, V, ignore_index)
    n_valid = count_valid(y, ignore_index)
    s = grad_scale_per_row(grad_scale, grad_output, n_valid)
    blocks = _blocks(N, block_rows)
    lse = np.empty(N)
    zt = np.zeros(N)
    slice_parts = [None] * len(blocks)
    bias_parts = [None] * len(blocks)

    def one(j):
        r0, r1 = blocks[j]
        z = logits(X[r0:r1], W, b)
        lse[r0:r1] = logsumexp_rows(z)
        yy = y[r0:r1]
        kept = np.nonzero(yy != ignore_index)[0]
        zt[r0 + kept] = z[kept, yy[kept]]
        G = softmax_minus_onehot(z, lse[r0:r1], yy, s, ignore_index)
        slice_parts[j] = G.T @ X[r0:r1, h0:h1]
        bias_parts[j] = G.sum(axis=0)

    with _pool(threads) as ex:
        list(ex.map(one, range(len(blocks))))
    cols = np.zeros((V, h1 - h0))
    grad_b = np.zeros(V)
    for j in range(len(blocks)):          # fixed order
        cols += slice_parts[j]
        grad_b += bias_parts[j]
    ok = valid_mask(y, ignore_index)
    loss = float((lse[ok] - zt[ok]).sum()) / n_valid if n_valid else 0.0
    return {"grad_W_cols": cols, "grad_b": grad_b if b is not None else None, "lse": lse, "loss": loss,
            "n_valid": n_valid}


def target_logits(X, W, b, y, ignore_index: int = IGNORE_INDEX,
                  block_rows: int = 65536) -> np.ndarray:
    """z[i, y[i]] for every row (NaN for ignored rows): N*H work, no full logits."""
    W, b = as_f64(W), as_f64(b)
    y = np.asarray(y, dtype=np.int64)
    out = np.full(len(y), np.nan)
    for r0, r1 in _blocks(len(y), block_rows):
        yy = y[r0:r1]
        ok = np.nonzero(yy != ignore_index)[0]
        Xb = as_f64(X[r0:r1][ok])
        zt = np.einsum("ij,ij->i", Xb, W[yy[ok]])
        if b is not None:
            zt += b[yy[ok]]
        out[r0 + ok] = zt
    return out
