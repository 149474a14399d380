"""Pins of the oracle's BF16 -> float64 widening (ZipFusion §II.A, KV Cache and BF16: a BF16 value
is 1 sign bit, 8 exponent bits and 7 fraction bits).  Every attention pin converts both of its
sides through this one function, so it is checked here against values fixed by the field
definition alone: a hand-listed table of patterns, and an independent decode of the three fields
(written with integer arithmetic and math.ldexp, no float32 reinterpretation) over all 65,536
patterns."""
import math

import numpy as np

from oracle import zf_oracle as O

# pattern -> exact value: sign, biased exponent e (bias 127), fraction f over 128
HAND = [
    (0x3F80, 1.0),                         # e = 127, f = 0
    (0xBF80, -1.0),                        # sign set
    (0x4000, 2.0),
    (0x3FC0, 1.5),                         # f = 64 / 128
    (0x4049, 3.140625),                    # e = 128, f = 73: 2 * (1 + 73/128)
    (0xC2F7, -123.5),                      # e = 133, f = 119: -64 * (1 + 119/128)
    (0x0000, 0.0),
    (0x8000, -0.0),
    (0x0001, 2.0 ** -133),                 # smallest subnormal: 2^-126 * 1/128
    (0x007F, 127 * 2.0 ** -133),           # largest subnormal
    (0x0080, 2.0 ** -126),                 # smallest normal
    (0x7F7F, (2 - 2.0 ** -7) * 2.0 ** 127),  # largest finite
    (0xFF7F, -(2 - 2.0 ** -7) * 2.0 ** 127),
    (0x7F80, math.inf),
    (0xFF80, -math.inf),
]


def test_hand_listed_patterns():
    bits = np.array([p for p, _ in HAND], dtype=np.uint16)
    got = O.bf16_to_f64(bits)
    assert got.dtype == np.float64
    for (p, want), g in zip(HAND, got):
        assert g == want, hex(p)
        assert math.copysign(1.0, g) == math.copysign(1.0, want), hex(p)     # -0.0 keeps its sign


def test_nan_patterns_give_nan():
    for p in (0x7FC0, 0x7F81, 0xFFC0, 0xFFFF):
        with np.errstate(invalid="ignore"):
            assert math.isnan(O.bf16_to_f64(np.array([p], dtype=np.uint16))[0]), hex(p)


def _field_decode(p: int) -> float:
    s, e, f = p >> 15, (p >> 7) & 0xFF, p & 0x7F
    sign = -1.0 if s else 1.0
    if e == 0xFF:
        return sign * math.inf if f == 0 else math.nan
    if e == 0:
        return sign * math.ldexp(f, -126 - 7)          # subnormal: 0.f * 2^-126
    return sign * math.ldexp(128 + f, e - 127 - 7)     # 1.f * 2^(e - 127)


def test_every_pattern_matches_an_independent_field_decode():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    with np.errstate(invalid="ignore"):          # NaN patterns widen to NaN
        got = O.bf16_to_f64(bits)
    want = np.array([_field_decode(p) for p in range(1 << 16)])
    nan = np.isnan(want)
    assert (np.isnan(got) == nan).all()
    assert (got[~nan] == want[~nan]).all()
    assert (np.signbit(got[~nan]) == np.signbit(want[~nan])).all()
