"""The oracle's bf16 decode (`as_f64`) against values the bit patterns define
by IEEE-754 binary16-brain layout (1 sign bit, 8 exponent bits with bias
127, 7 fraction bits), computed here from the fields in exact rational
arithmetic, and against torch's own bfloat16 -> float64 cast.  Every GPU
parity test feeds bf16 bit patterns through this decode, so a wrong shift,
a float16 reading or a lost sign here would be blamed on the kernels.
CPU only."""
from fractions import Fraction

import numpy as np

import oracle


def ieee_bf16_value(bits: int) -> float:
    """Value of a bf16 bit pattern from its fields (finite patterns only)."""
    sign = -1 if bits & 0x8000 else 1
    e = (bits >> 7) & 0xFF
    f = bits & 0x7F
    assert e != 0xFF
    if e == 0:   # subnormal: 0.f * 2^-126
        v = Fraction(f, 128) * Fraction(1, 2 ** 126)
    else:        # normal: 1.f * 2^(e - 127)
        v = (1 + Fraction(f, 128)) * (Fraction(2) ** (e - 127))
    return float(sign * v)


def test_hand_chosen_patterns():
    cases = {
        0x3F80: 1.0,
        0xC020: -2.5,
        0x0001: 2.0 ** -133,                    # smallest subnormal: 2^-7 * 2^-126
        0x7F7F: (2 - 2.0 ** -7) * 2.0 ** 127,   # largest finite
        0x4049: 3.140625,                       # 1.5703125 * 2
        0x3E00: 0.125,
        0x0080: 2.0 ** -126,                    # smallest normal
    }
    bits = np.array(list(cases), dtype=np.uint16)
    got = oracle.as_f64(bits)
    for b, g in zip(cases, got):
        assert g == cases[b], (hex(b), g, cases[b])
    z = oracle.as_f64(np.array([0x8000], dtype=np.uint16))[0]
    assert z == 0.0 and np.signbit(z)                                      # -0.0


def test_every_finite_pattern_against_the_fields():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    finite = ((bits >> 7) & 0xFF) != 0xFF
    got = oracle.as_f64(bits)
    want = np.array([ieee_bf16_value(int(b)) for b in bits[finite]])
    assert np.array_equal(got[finite], want)
    assert np.array_equal(np.signbit(got[finite]), (bits[finite] & 0x8000) != 0)
    # exponent all ones: infinities (fraction 0) and NaNs
    top = bits[~finite]
    g = got[~finite]
    frac0 = (top & 0x7F) == 0
    assert np.all(np.isinf(g[frac0])) and np.all(np.isnan(g[~frac0]))
    assert np.array_equal(np.signbit(g[frac0]), (top[frac0] & 0x8000) != 0)


def test_matches_torch_cast():
    import torch
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = oracle.as_f64(bits)
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    assert np.array_equal(np.isnan(got), np.isnan(ref))


def test_shape_and_float_passthrough():
    a = np.array([[0x3F80, 0x4000], [0xBF80, 0x0000]], dtype=np.uint16)
    assert np.array_equal(oracle.as_f64(a), np.array([[1.0, 2.0], [-1.0, 0.0]]))
    f = np.array([0.1, -3.0], dtype=np.float32)
    assert np.array_equal(oracle.as_f64(f), f.astype(np.float64))
    assert oracle.as_f64(None) is None
