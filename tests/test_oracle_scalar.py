"""Oracle pins for the scalar rules of the finalizer.

* bf16 round trip ("The Finalizer's Sharp Edges": the NOPE path rounds y
  through bf16 and the RoPE values are stored as bf16): checked against
  torch's float32 -> bfloat16 cast, a library routine, on millions of values
  including ties and overflow edges.
* Quantisation exponent e = ceil(log2(a / 127)) ("How One Output Is
  Produced", NOPE quantisation): checked by its defining property in exact
  rational arithmetic -- 127 * 2^e >= a > 127 * 2^(e-1) -- and at hand-worked
  values.
"""
from fractions import Fraction

import numpy as np
import pytest

from kvc_testlib import torch_bf16_bits


def test_bf16_rne_matches_torch_random_bits(oracle_mod):
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 2**32, size=1 << 21, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x = x[np.isfinite(x)]
    got = oracle_mod.f32_to_bf16_bits_array(x)
    want = torch_bf16_bits(x)
    assert np.array_equal(got, want)


def test_bf16_rne_ties_and_edges(oracle_mod):
    rng = np.random.default_rng(2)
    hi = rng.integers(0, 0x7F7F, size=200000, dtype=np.uint32)
    sign = rng.integers(0, 2, size=hi.shape, dtype=np.uint32) << 31
    # exact ties (low half 0x8000), one below and one above the tie
    lows = np.array([0x8000, 0x7FFF, 0x8001, 0x0000, 0xFFFF], dtype=np.uint32)
    pats = ((hi[:, None] << 16) | lows[None, :]) | sign[:, None]
    x = pats.reshape(-1).view(np.float32)
    extra = np.array([0.0, -0.0, 3.3895314e38, -3.3895314e38, 3.4028235e38,
                      1e-45, -1e-45, 1.1754944e-38, 1.0, -1.0, 1.00390625,
                      1.01171875], dtype=np.float32)
    x = np.concatenate([x, extra])
    assert np.array_equal(oracle_mod.f32_to_bf16_bits_array(x), torch_bf16_bits(x))
    # hand-worked: 1 + 2^-8 is a tie between 1.0 (even) and 1 + 2^-7 -> 1.0
    assert oracle_mod.f32_to_bf16_bits(1.00390625) == 0x3F80
    # 1 + 3 * 2^-8 is a tie between 1 + 2^-7 (odd) and 1 + 2^-6 (even)
    assert oracle_mod.f32_to_bf16_bits(1.01171875) == 0x3F82


def _exact_ok(a: float, e: int) -> bool:
    fa = Fraction(a)
    return Fraction(127) * Fraction(2) ** e >= fa > Fraction(127) * Fraction(2) ** (e - 1)


def test_exponent_defining_property(oracle_mod):
    vals = []
    for k in range(-30, 30):
        edge = np.float32(np.ldexp(127.0, k))          # a / 127 exactly 2^k
        vals += [edge, np.nextafter(edge, np.float32(np.inf)),
                 np.nextafter(edge, np.float32(0))]
        vals += [np.float32(np.ldexp(1.0, k)), np.float32(np.ldexp(1.5, k))]
    rng = np.random.default_rng(3)
    vals += list(np.float32(10.0) ** rng.uniform(-4, 6, size=20000).astype(np.float32))
    # bf16-valued magnitudes, as the quantiser sees them
    b = rng.integers(0x3800, 0x4F00, size=20000).astype(np.uint32) << 16
    vals += list(b.view(np.float32))
    vals.append(np.float32(1e-4))
    for a in vals:
        a = float(np.float32(a))
        e = oracle_mod.scale_exponent(a)
        assert _exact_ok(a, e), (a, e)


@pytest.mark.parametrize("a,e", [
    (127.0, 0),        # log2(1) = 0
    (127.5, 1),        # just above 127 * 2^0
    (254.0, 1),        # 127 * 2
    (1.0, -6),         # log2(1/127) = -6.989
    (63.5, -1),        # 127 / 2 exactly
    (0.49609375, -8),  # 127 / 256 exactly, a bf16 value
    (float(np.float32(1e-4)), -20),  # the amax floor: log2(7.87e-7) = -20.28
])
def test_exponent_hand_worked(oracle_mod, a, e):
    assert oracle_mod.scale_exponent(a) == e
