"""Oracle pins for the packed slot layout and the scatter.

* tests/golden/hand_worked_two_slots.json: every byte of two slots derived by
  hand from the formulas of "How One Output Is Produced" and the layout of
  "Gather and Scatter" (KernelGen Challenge 8 write-up).
* brute-force decoding: every written slot read back (codes * 2^e and the
  bf16 RoPE values) reproduces the oracle's own y within one quantisation
  step, and every byte outside the written slots keeps its prior value.
* the compressed position pc = floor(p / C) * C selects the cos/sin row.
"""
import json
import os

import numpy as np

from kv_cache_compression_c128_gb300 import inputs
from kvc_testlib import (bf16_bits_to_f32, decode_slot, dequant, slots_of_case,
                         torch_bf16_bits, written_mask)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _hand_worked_inputs():
    C, T = 8, 16
    d = np.arange(512)
    vA = np.where(d % 3 == 2, -1.0, 1.0)
    vB = np.where(d % 3 == 0, -2.0, 2.0)
    st = np.zeros((2, 8, 1024), np.float32)
    for i in range(8):
        st[1, i, :512] = vA
        st[1, i, 512:] = (i - 3.5) * ((d % 5) - 2) / 4.0
        st[0, i, :512] = vB
        st[0, i, 512:] = (i - 3.5) * ((d % 3) - 1) / 2.0
    w = np.ones(512, np.float64)
    for g in range(7):
        k = g - 3
        for j in range(64):
            m = {0: 1.984375, 1: 1.0234375, 2: 1.5}.get(j, 0.25)
            w[64 * g + j] = m * 2.0 ** k
    csc = np.zeros((16, 64), np.float32)
    csc[:, :32] = 1.0
    csc[8, :32], csc[8, 32:] = 0.0, 1.0
    csc[7, :32], csc[7, 32:] = 0.0, -1.0
    csc[15, :32], csc[15, 32:] = -1.0, 0.0
    sm = np.full(T, -1, np.int64)
    sm[7], sm[15] = 1, 0
    arrays = dict(
        state_bits=torch_bf16_bits(st).reshape(2, 8, 1024),
        token_to_req=np.zeros(T, np.int32), positions=np.arange(T, dtype=np.int64),
        boundary_token_indices=np.array([7, 15], np.int64),
        block_table=np.array([[1, 0]], np.int32),
        rms_norm_weight=w.astype(np.float32), cos_sin_cache=csc,
        kv_slot_mapping=sm, block_size=8, compress_ratio=C, rms_norm_eps=1e-6)
    return arrays, vA, vB


def _expected_hand_worked(spec, vA, vB):
    exp = spec["expected"]
    kv = np.full(37376, exp["untouched_byte"], np.uint8)
    one, mone = exp["rope_one_bf16_bits"], exp["rope_minus_one_bf16_bits"]
    for v, slot, rot in ((vA, 1, "identity"), (vB, 0, "quarter")):
        payload = np.zeros(576, np.uint8)
        for dd in range(448):
            code = exp["code_by_j"].get(str(dd % 64), exp["code_by_j"]["other"])
            payload[dd] = code if v[dd] > 0 else 256 - code
        rope = np.empty(64)
        if rot == "identity":
            rope[:] = np.sign(v[448:])
        else:  # (u, w) -> (-w, u)
            rope[0::2] = -np.sign(v[449::2])
            rope[1::2] = np.sign(v[448::2])
        bits = np.where(rope > 0, one, mone).astype("<u2")
        payload[448:] = bits.view(np.uint8)
        kv[slot * 576: slot * 576 + 576] = payload
        kv[36864 + slot * 8: 36864 + slot * 8 + 8] = np.array(exp["scale_bytes"], np.uint8)
    return kv


def test_hand_worked_golden_slots(oracle_mod):
    with open(os.path.join(GOLDEN, "hand_worked_two_slots.json")) as f:
        spec = json.load(f)
    arrays, vA, vB = _hand_worked_inputs()
    kv = np.full((1, 37376), spec["expected"]["untouched_byte"], np.uint8)
    res = oracle_mod.compress(kv_cache=kv, **arrays)
    assert res["status"] == 0
    assert np.array_equal(res["c"][0], vA.astype(np.float32))
    assert np.array_equal(res["c"][1], vB.astype(np.float32))
    want = _expected_hand_worked(spec, vA, vB)
    assert np.array_equal(kv.reshape(-1), want)


def test_decoded_slots_reproduce_y_and_leave_other_bytes(oracle_mod):
    case = inputs.make_case(2, 4096, 32, seed=30, kv_fill=31)   # 128 outputs, 2 pages
    before = case.kv_cache.copy()
    kv, res = oracle_mod.compress_case(case)
    assert res["status"] == 0
    y = res["y"].astype(np.float64)
    slots = slots_of_case(case)
    assert sorted(slots.tolist()) == list(range(case.num_outputs))
    for n, s in enumerate(slots):
        q, e, pad, rope = decode_slot(kv, s)
        assert pad == 0
        z = bf16_bits_to_f32(torch_bf16_bits(y[n, :448].astype(np.float32)))
        step = np.repeat(np.ldexp(1.0, e), 64)
        assert np.all(np.abs(dequant(q, e) - z) < step)
        # RoPE values: magnitude-preserving rotation of y's last 64 dims
        r0 = np.hypot(y[n, 448::2], y[n, 449::2])
        r1 = np.hypot(rope[0::2], rope[1::2])
        assert np.allclose(r0, r1, rtol=2 ** -7, atol=1e-6)
    m = written_mask(kv.shape, slots)
    assert np.array_equal(kv.reshape(-1)[~m], before.reshape(-1)[~m])
    assert not np.array_equal(kv.reshape(-1)[m], before.reshape(-1)[m])


def test_compressed_position_selects_cos_sin_row(oracle_mod):
    # C = 16; the output at p = 31 must read row pc = 16, not row 31 or 0
    case = inputs.make_case(1, 64, 16, seed=32)
    csc = np.zeros_like(case.cos_sin_cache)
    csc[:, :32] = 1.0                       # identity everywhere ...
    csc[16, :32], csc[16, 32:] = 0.0, 1.0   # ... except a quarter turn at 16
    case.cos_sin_cache = csc
    kv, res = oracle_mod.compress_case(case)
    y = res["y"]
    for n, b in enumerate(case.boundary_token_indices):
        p = int(case.positions[b])
        _, _, _, rope = decode_slot(kv, case.kv_slot_mapping[b])
        if p == 31:
            want = np.empty(64, np.float32)
            want[0::2], want[1::2] = -y[n, 449::2], y[n, 448::2]
        else:
            want = y[n, 448:]
        assert np.array_equal(rope, bf16_bits_to_f32(torch_bf16_bits(want)))


def test_negative_slot_is_skipped_and_slot_mapping_by_output(oracle_mod):
    case = inputs.make_case(1, 1024, 64, seed=33, kv_fill=34)
    kv_tok, _ = oracle_mod.compress_case(case)
    # the same slots given per output (length N) instead of per token
    per_out = case.kv_slot_mapping[case.boundary_token_indices].copy()
    kv_out = case.kv_cache.copy()
    res = oracle_mod.compress(case.state_bits, case.token_to_req, case.positions,
                              case.boundary_token_indices, case.block_table,
                              case.rms_norm_weight, case.cos_sin_cache, per_out,
                              kv_out, 8, 64)
    assert res["status"] == 0 and np.array_equal(kv_out, kv_tok)
    # slot -1 for output 3: its slot keeps the prior bytes
    skip = per_out.copy()
    old = int(skip[3])
    skip[3] = -1
    kv_skip = case.kv_cache.copy()
    oracle_mod.compress(case.state_bits, case.token_to_req, case.positions,
                        case.boundary_token_indices, case.block_table,
                        case.rms_norm_weight, case.cos_sin_cache, skip,
                        kv_skip, 8, 64)
    m = written_mask(kv_skip.shape, [old])
    assert np.array_equal(kv_skip.reshape(-1)[m], case.kv_cache.reshape(-1)[m])
    assert np.array_equal(kv_skip.reshape(-1)[~m], kv_tok.reshape(-1)[~m])


# ---- the reader direction: decode packed slots back to vectors -----------------

def test_dequantize_hand_worked_golden_slots(oracle_mod):
    # the two hand-worked slots decode to the hand-derived values:
    # group g has e = g - 9, so a code q reads back as q * 2^(g - 9); RoPE +-1
    with open(os.path.join(GOLDEN, "hand_worked_two_slots.json")) as f:
        spec = json.load(f)
    arrays, vA, vB = _hand_worked_inputs()
    kv = np.full((1, 37376), 0xAB, np.uint8)
    oracle_mod.compress(kv_cache=kv, **arrays)
    out, st = oracle_mod.dequantize(kv, np.array([1, 0, -1], np.int64))
    assert st == 0
    code = spec["expected"]["code_by_j"]
    for row, v in ((0, vA), (1, vB)):
        for d in range(448):
            q = code.get(str(d % 64), code["other"]) * (1 if v[d] > 0 else -1)
            assert out[row, d] == q * 2.0 ** (d // 64 - 9)
    assert np.all(np.abs(out[0, 448:]) == 1.0) and np.all(np.abs(out[1, 448:]) == 1.0)
    assert np.array_equal(np.sign(out[0, 448:]), np.sign(vA[448:]))
    assert np.all(out[2] == 0.0)                  # negative slot: zeros


def test_dequantize_edge_bytes(oracle_mod):
    kv = np.zeros((1, 37376), np.uint8)
    pay = kv[0, 0:576]
    sc = kv[0, 36864:36872]
    pay[0], sc[0] = 0x81, 127                     # -127 * 2^0
    pay[64], pay[65], sc[1] = 0x01, 0x00, 0       # 2^-127 (subnormal), 0
    pay[128], pay[129], sc[2] = 0x01, 0x00, 255   # 2^128 -> inf, 0 * 2^128 -> 0
    pay[448], pay[449] = 0x80, 0xBF               # bf16 0xBF80 = -1.0
    out, st = oracle_mod.dequantize(kv, np.array([0], np.int64))
    assert st == 0
    assert out[0, 0] == -127.0
    assert out[0, 64] == np.float32(2.0 ** -127) and out[0, 65] == 0.0
    assert np.isinf(out[0, 128]) and out[0, 128] > 0 and out[0, 129] == 0.0
    assert out[0, 448] == -1.0
    bits, _ = oracle_mod.dequantize(kv, np.array([0], np.int64), out_bf16=True)
    assert bits[0, 0] == 0xC2FE                   # -127 in bf16
    assert bits[0, 128] == 0x7F80 and bits[0, 448] == 0xBF80
    _, st = oracle_mod.dequantize(kv, np.array([64], np.int64))
    assert st == 4                                # slot beyond the last page


def test_dequantize_matches_bit_level_decoder(oracle_mod):
    # random bytes everywhere (codes and scale exponents over their full
    # range): the oracle's reader equals the tests' own byte decoder
    rng = np.random.default_rng(40)
    kv = rng.integers(0, 256, size=(2, 37376), dtype=np.uint8)
    slots = rng.permutation(128)[:50]
    out, st = oracle_mod.dequantize(kv, slots)
    assert st == 0
    for m, s in enumerate(slots):
        q, e, _, rope = decode_slot(kv, s)
        want = np.concatenate([dequant(q, e), rope.astype(np.float64)]).astype(np.float32)
        assert np.array_equal(out[m], want, equal_nan=True)
