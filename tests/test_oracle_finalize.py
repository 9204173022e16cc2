"""Oracle pins for RMSNorm, NOPE quantisation and RoPE.

"How One Output Is Produced" of the KernelGen Challenge 8 write-up:
  rho = (mean_d c_d^2 + eps)^(-1/2), y_d = c_d rho w_d;
  z = fp32(bf16(y)), per 64-dim group a = max(max|z|, 1e-4),
  e = ceil(log2(a/127)), q = int8(clip(z 2^-e, -127, 127)), scale = e + 127;
  GPT-J interleaved RoPE on dims 448..511 with cos/sin read from row
  pc = floor(p / C) * C of cos_sin_cache (cos in columns 0..31, sin 32..63).
"The Finalizer's Sharp Edges" fixes truncation toward zero and the bf16
rounding of the rotated values.

Pins: torch.nn.functional.rms_norm (library routine) and the exact scale
invariance of RMSNorm; complex multiplication for the rotation; the two
inequalities that characterise truncation toward zero; the code range that
follows from the exponent rule; norm preservation and inverse rotation.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

from kvc_testlib import bf16_bits_to_f32, torch_bf16_bits


def test_rmsnorm_matches_torch_rms_norm(oracle_mod):
    rng = np.random.default_rng(20)
    c = (rng.standard_normal((64, 512)) * rng.uniform(0.01, 10, (64, 1))).astype(np.float32)
    w = (1 + 0.1 * rng.standard_normal(512)).astype(np.float32)
    y = oracle_mod.rmsnorm(c, w, 1e-6)
    ref = F.rms_norm(torch.from_numpy(c).double(), (512,),
                     torch.from_numpy(w).double(), eps=float(np.float32(1e-6))).numpy()
    # two fp32 roundings after a correctly rounded rho: a few ulp
    assert np.allclose(y, ref, rtol=4 * 2 ** -24, atol=0)


def test_rmsnorm_unit_weight_gives_unit_rms(oracle_mod):
    rng = np.random.default_rng(21)
    c = rng.standard_normal((32, 512)).astype(np.float32)
    y = oracle_mod.rmsnorm(c, np.ones(512, np.float32), 1e-6)
    m = (c.astype(np.float64) ** 2).mean(1)
    rms = np.sqrt((y.astype(np.float64) ** 2).mean(1))
    assert np.allclose(rms, np.sqrt(m / (m + float(np.float32(1e-6)))), rtol=1e-6)


@pytest.mark.parametrize("k", [-20, -3, 1, 7, 30])
def test_rmsnorm_exact_power_of_two_scale_invariance(oracle_mod, k):
    # with eps = 0, rho(2^k c) = 2^-k rho(c) exactly, so y is bit-identical
    rng = np.random.default_rng(22)
    c = rng.standard_normal((8, 512)).astype(np.float32)
    w = (1 + 0.1 * rng.standard_normal(512)).astype(np.float32)
    y0 = oracle_mod.rmsnorm(c, w, 0.0)
    y1 = oracle_mod.rmsnorm(np.ldexp(c, k).astype(np.float32), w, 0.0)
    assert np.array_equal(y0, y1)


def _rope_row(theta):
    theta = np.asarray(theta, dtype=np.float64)
    return np.concatenate([np.cos(theta), np.sin(theta)]).astype(np.float32)


def _decode(payload, scale):
    q = payload[:448].view(np.int8).astype(np.int64)
    e = scale[:7].astype(np.int64) - 127
    rope = bf16_bits_to_f32(payload[448:].copy().view("<u2"))
    return q, e, rope


def test_rope_is_complex_multiplication(oracle_mod):
    rng = np.random.default_rng(23)
    mism = 0
    for _ in range(50):
        y = rng.standard_normal(512).astype(np.float32)
        theta = rng.uniform(-np.pi, np.pi, 32)
        cs = _rope_row(theta)
        payload, scale = oracle_mod.pack_slot(y, cs)
        _, _, rope = _decode(payload, scale)
        zc = (y[448::2].astype(np.float64) + 1j * y[449::2]) * \
             (cs[:32].astype(np.float64) + 1j * cs[32:].astype(np.float64))
        ref = np.empty(64)
        ref[0::2], ref[1::2] = zc.real, zc.imag
        ref_b = bf16_bits_to_f32(torch_bf16_bits(ref.astype(np.float32)))
        # fp32 intermediates may flip a bf16 rounding: at most one bf16 ulp
        ulp = np.ldexp(1.0, np.frexp(np.abs(ref_b) + 1e-30)[1] - 8)
        assert np.all(np.abs(rope - ref_b) <= ulp)
        mism += int(np.sum(rope != ref_b))
    assert mism <= 50 * 64 // 100


def test_rope_identity_at_zero_angle(oracle_mod):
    rng = np.random.default_rng(24)
    y = rng.standard_normal(512).astype(np.float32)
    payload, scale = oracle_mod.pack_slot(y, _rope_row(np.zeros(32)))
    assert np.array_equal(payload[448:].copy().view("<u2"), torch_bf16_bits(y[448:]))


def test_rope_pairs_are_interleaved_not_halves(oracle_mod):
    # 90 degree rotation: (u, w) -> (-w, u) on adjacent dims (448+2j, 449+2j)
    y = np.zeros(512, np.float32)
    y[448:] = np.arange(1, 65, dtype=np.float32)
    payload, scale = oracle_mod.pack_slot(y, _rope_row(np.full(32, np.pi / 2)))
    _, _, rope = _decode(payload, scale)
    want = np.empty(64, np.float32)
    want[0::2] = -y[449::2]
    want[1::2] = y[448::2]
    assert np.allclose(rope, want, atol=1e-6)


def test_rope_preserves_norm_and_inverts(oracle_mod):
    rng = np.random.default_rng(25)
    y = rng.standard_normal(512).astype(np.float32)
    theta = rng.uniform(-np.pi, np.pi, 32)
    _, _, r1 = _decode(*oracle_mod.pack_slot(y, _rope_row(theta)))
    n0 = np.hypot(y[448::2], y[449::2])
    n1 = np.hypot(r1[0::2], r1[1::2])
    assert np.allclose(n0, n1, rtol=2 ** -7)
    y2 = y.copy()
    y2[448:] = r1
    _, _, r2 = _decode(*oracle_mod.pack_slot(y2, _rope_row(-theta)))
    assert np.allclose(r2, y[448:], rtol=2 ** -6, atol=2 ** -7)


def test_quant_truncation_and_code_range(oracle_mod):
    rng = np.random.default_rng(26)
    total = 0
    for _ in range(200):
        y = (rng.standard_normal(512) * rng.uniform(1e-3, 1e3, 512)).astype(np.float32)
        payload, scale = oracle_mod.pack_slot(y, _rope_row(np.zeros(32)))
        q, e, rope = _decode(payload, scale)
        z = bf16_bits_to_f32(torch_bf16_bits(y[:448])).astype(np.float64)
        step = np.repeat(np.ldexp(1.0, e), 64)
        # truncation toward zero: |q| 2^e <= |z| < (|q| + 1) 2^e, same sign
        assert np.all(np.abs(q) * step <= np.abs(z))
        assert np.all(np.abs(z) < (np.abs(q) + 1) * step)
        assert np.all((q == 0) | (np.sign(q) == np.sign(z)))
        # ceil(log2(a/127)) => 63 <= max|q| <= 127 in every group (a > 1e-4)
        gmax = np.abs(q).reshape(7, 64).max(1)
        assert np.all((gmax >= 63) & (gmax <= 127))
        assert scale[7] == 0
        total += 1
    assert total == 200


def test_quant_floor_for_tiny_groups(oracle_mod):
    y = np.zeros(512, np.float32)
    y[:64] = 1e-6          # group 0 below the 1e-4 floor
    y[64:128] = -3e-5
    payload, scale = oracle_mod.pack_slot(y, _rope_row(np.zeros(32)))
    q, e, _ = _decode(payload, scale)
    # a = 1e-4 -> e = -20 (1e-4/127 = 2^-20.28); codes trunc(z * 2^20)
    assert list(e[:3]) == [-20, -20, -20]
    z0 = float(bf16_bits_to_f32(torch_bf16_bits(np.float32([1e-6])))[0])
    z1 = float(bf16_bits_to_f32(torch_bf16_bits(np.float32([-3e-5])))[0])
    assert np.all(q[:64] == int(z0 * 2 ** 20))   # 1.048 -> 1
    assert np.all(q[64:128] == int(z1 * 2 ** 20))  # -31.4 -> -31
    assert np.all(q[128:] == 0)


def test_quant_truncates_not_rounds(oracle_mod):
    # group 0: z = 1.0234375 * 2^k and the group max 1.984375 * 2^k (= 127 *
    # 2^(k-6)), so e = k - 6 and z * 2^-e = 65.5: truncation gives 65, any
    # rounding 66; the max element gives exactly 127.
    y = np.zeros(512, np.float32)
    y[0] = 1.984375 * 4
    y[1] = 1.0234375 * 4
    y[2] = -1.0234375 * 4
    payload, scale = oracle_mod.pack_slot(y, _rope_row(np.zeros(32)))
    q, e, _ = _decode(payload, scale)
    assert e[0] == 2 - 6
    assert (q[0], q[1], q[2]) == (127, 65, -65)
    assert payload[2] == 256 - 65                      # two's complement byte
