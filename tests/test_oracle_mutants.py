"""Planted mistakes in the oracle (CPU only): each mutant of the oracle's
source must fail at least one pin, which shows the pins would catch that
kind of error in the oracle itself."""
import importlib.util
import os
import sys
import types

import pytest

from tests import oracle_pins

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "lce_oracle.py")

MUTANTS = {
    "drop_bias": ("        z += b[None, :]\n", "        pass\n"),
    "onehot_sign": ("    G[rows, np.asarray(y)[rows]] -= 1.0\n", "    G[rows, np.asarray(y)[rows]] += 1.0\n"),
    "onehot_off_by_one": ("    G[rows, np.asarray(y)[rows]] -= 1.0\n",
                          "    G[rows, (np.asarray(y)[rows] + 1) % G.shape[1]] -= 1.0\n"),
    "ignored_rows_kept": ("    G[~ok, :] = 0.0\n", "    pass\n"),
    "n_valid_counts_all": ("    return int(valid_mask(y, ignore_index).sum())\n", "    return int(len(y))\n"),
    "no_max_shift": ("    return m + np.log(np.exp(z - m[:, None]).sum(axis=1))\n",
                     "    return np.log(np.exp(z).sum(axis=1))\n"),
    "log2_not_ln": ("    return m + np.log(np.exp(z - m[:, None]).sum(axis=1))\n",
                    "    return m + np.log2(np.exp(z - m[:, None]).sum(axis=1))\n"),
    "grad_scale_dropped": ("    return float(grad_scale) * float(grad_output) / n_valid\n",
                           "    return 1.0 / n_valid\n"),
    "grad_W_wrong_rows": ("        part_W[j] = G.T @ X[r0:r1]\n", "        part_W[j] = G.T @ X[r0:r1][::-1]\n"),
    "grad_X_shifted_weight": ("        grad_X[r0:r1] = G @ W\n",
                                 "        grad_X[r0:r1] = G @ np.roll(W, 1, axis=1)\n"),
    "grad_b_wrong_axis": ("        part_b[j] = G.sum(axis=0)\n", "        part_b[j] = G.sum(axis=1).sum() + 0 * G.sum(axis=0)\n"),
    "mean_over_all_rows": ("        loss = total / n_valid if n_valid else 0.0\n",
                           "        loss = total / N if n_valid else 0.0\n"),
    "sum_loss_divided": ("        loss = total\n", "        loss = total / max(n_valid, 1)\n"),
    "sum_scale_divided": ("        return float(grad_scale) * float(grad_output)\n",
                          "        return float(grad_scale) * float(grad_output) / max(n_valid, 1)\n"),
    "lse_missing_max": ("    return m + np.log(np.exp(z - m[:, None]).sum(axis=1))\n",
                        "    return np.log(np.exp(z - m[:, None]).sum(axis=1))\n"),
    "softmax_not_normalised": ("    G = np.exp(z - lse[:, None])\n", "    G = np.exp(z - z.max(axis=1)[:, None])\n"),
    "ignored_rows_in_loss": ("    total = float((lse[ok] - zt[ok]).sum())\n", "    total = float((lse - zt).sum())\n"),
    "loss_sign": ("    total = float((lse[ok] - zt[ok]).sum())\n", "    total = float((zt[ok] - lse[ok]).sum())\n"),
    "bf16_decode_shift_15": ("        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)\n",
                             "        return (a.astype(np.uint32) << 15).view(np.float32).astype(np.float64)\n"),
    "bf16_decode_as_float16": ("        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)\n",
                               "        return a.view(np.float16).astype(np.float64)\n"),
    "bf16_decode_drops_sign": ("        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)\n",
                               "        return ((a.astype(np.uint32) & 0x7FFF) << 16).view(np.float32).astype(np.float64)\n"),
    "column_slice_offset": ("        slice_parts[j] = G.T @ X[r0:r1, h0:h1]\n",
                            "        slice_parts[j] = G.T @ X[r0:r1, h0 + 1:h1 + 1]\n"),
    "target_logit_wrong_column": ("        zt[r0:r1][ok] = z[np.nonzero(ok)[0], yy[ok]]\n",
                                  "        zt[r0:r1][ok] = z[np.nonzero(ok)[0], 0]\n"),
}


def _load_mutant(name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutant {name}: anchor not found exactly once"
    mod = types.ModuleType(f"lce_oracle_mutant_{name}")
    mod.__file__ = SRC
    exec(compile(src.replace(old, new), f"<mutant {name}>", "exec"), mod.__dict__)
    return mod


def test_unmutated_source_passes():
    mod = _load_mutant("none", "import numpy as np\n", "import numpy as np\n")
    assert oracle_pins.run_all(mod) == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name):
    old, new = MUTANTS[name]
    mod = _load_mutant(name, old, new)
    fails = oracle_pins.run_all(mod)
    assert fails, f"planted mistake {name} passed every pin"
