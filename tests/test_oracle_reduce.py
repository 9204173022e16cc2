"""Oracle pins for the window gather and the per-dimension softmax sum.

"How One Output Is Produced" of the KernelGen Challenge 8 write-up: the
window of boundary token b is t_i = p - C + 1 + i, each t_i resolves through
block_table (block_size 8) to a physical row whose first 512 columns are
values v and next 512 are scores s, and c_d = sum_i softmax_i(s_{., d}) v_{i, d}
with the softmax taken along the window, separately for every dimension.

Pins (none re-types the oracle's loop):
* the page's own baseline ("The Baseline": gather [N, C, 1024], then
  softmax(dim=1) and a sum) evaluated by torch in float64;
* closed forms: equal scores give the window mean, a dominant score picks its
  row, a constant value row survives any scores;
* the window's position, through a value pattern equal to the token position;
* invariance under a relabelling of physical blocks and under a score shift.
"""
import numpy as np
import pytest
import torch

from kv_cache_compression_c128_gb300 import inputs
from kvc_testlib import bf16_bits_to_f32, gather_window_rows, torch_bf16_bits


def _reduce(oracle_mod, case):
    c, valid, status = oracle_mod.window_reduce(
        case.state_bits, case.token_to_req, case.positions,
        case.boundary_token_indices, case.block_table, case.compress_ratio,
        case.block_size)
    assert status == 0 and valid.all()
    return c


@pytest.mark.parametrize("R,T,C", [(1, 256, 8), (2, 512, 16), (2, 1024, 128),
                                   (1, 1024, 512), (3, 768, 64)])
def test_reduce_matches_torch_softmax(oracle_mod, R, T, C):
    case = inputs.make_case(R, T, C, seed=100 + C + R)
    c = _reduce(oracle_mod, case)
    rows = gather_window_rows(case)                         # [N, C]
    st = bf16_bits_to_f32(case.state_bits.reshape(-1, 1024)).astype(np.float64)
    all_rows = torch.from_numpy(st[rows.reshape(-1)]).reshape(rows.shape[0], C, 1024)
    v, s = all_rows[..., :512], all_rows[..., 512:]
    ref = (v * torch.softmax(s, dim=1)).sum(dim=1).numpy()
    # c is the float64 result rounded once to float32
    assert np.allclose(c, ref, rtol=2 ** -23, atol=1e-12)


@pytest.mark.parametrize("R,T,C,B", [(2, 1536, 37, 24), (1, 1024, 5, 16), (2, 2048, 300, 32),
                                     (3, 1536, 1, 8)])
def test_general_windows_match_torch_softmax(oracle_mod, R, T, C, B):
    # windows at random starts (not block aligned), block sizes other than 8
    case = inputs.make_case(R, T, C, seed=200 + C + B, block_size=B, boundaries_per_req=30)
    c = _reduce(oracle_mod, case)
    rows = gather_window_rows(case)
    st = bf16_bits_to_f32(case.state_bits.reshape(-1, 1024)).astype(np.float64)
    all_rows = torch.from_numpy(st[rows.reshape(-1)]).reshape(rows.shape[0], C, 1024)
    ref = (all_rows[..., :512] * torch.softmax(all_rows[..., 512:], dim=1)).sum(dim=1).numpy()
    assert np.allclose(c, ref, rtol=2 ** -23, atol=1e-12)
    starts = case.positions[case.boundary_token_indices] - C + 1
    assert C == 1 or np.any(starts % B != 0)     # the case does exercise unaligned starts


def _custom_case(C, T, v_fn, s_fn, R=1, seed=7):
    """A case whose state rows are set from token-level functions."""
    case = inputs.make_case(R, T, C, seed=seed)
    st = np.zeros((T // 8 * 8, 1024), dtype=np.float32)
    for tok in range(T):
        r = int(case.token_to_req[tok])
        t = int(case.positions[tok])
        row = int(case.block_table[r, t // 8]) * 8 + t % 8
        st[row, :512] = v_fn(r, t)
        st[row, 512:] = s_fn(r, t)
    case.state_bits = torch_bf16_bits(st).reshape(-1, 8, 1024)
    return case


def test_equal_scores_give_window_mean_of_positions(oracle_mod):
    # v_{t,d} = t (exact in bf16 for t <= 256), all scores equal:
    # c_d = mean of t over the window = p - (C - 1) / 2, exactly.
    C, T = 16, 256
    case = _custom_case(C, T, lambda r, t: np.full(512, t, np.float32),
                        lambda r, t: np.full(512, 0.75, np.float32))
    c = _reduce(oracle_mod, case)
    p = case.positions[case.boundary_token_indices]
    assert np.array_equal(c, np.repeat((p - (C - 1) / 2.0)[:, None], 512, 1).astype(np.float32))


def test_dominant_score_selects_its_row(oracle_mod):
    # score 60 at window offset i* = (d mod C) in dimension d, others N(0,1)
    # clipped to |s| <= 4: weight of the rest <= C * e^-56, so c_d = v_{i*, d}.
    C, T = 32, 256
    rng = np.random.default_rng(5)
    V = rng.standard_normal((T, 512)).astype(np.float32)
    S = np.clip(rng.standard_normal((T, 512)), -4, 4).astype(np.float32)
    d = np.arange(512)
    for t in range(T):
        S[t, (d % C) == (t % C)] = 60.0
    case = _custom_case(C, T, lambda r, t: V[t], lambda r, t: S[t])
    c = _reduce(oracle_mod, case)
    Vb = bf16_bits_to_f32(torch_bf16_bits(V))
    for n, b in enumerate(case.boundary_token_indices):
        p = int(case.positions[b])
        t_star = p - C + 1 + (d % C)          # row holding the 60 in dim d
        assert np.allclose(c[n], Vb[t_star, d], rtol=1e-6, atol=1e-7)


def test_constant_value_rows_survive_any_scores(oracle_mod):
    rng = np.random.default_rng(6)
    vals = rng.standard_normal(512).astype(np.float32)
    C, T = 128, 1024
    case = _custom_case(C, T, lambda r, t: vals,
                        lambda r, t: rng.standard_normal(512).astype(np.float32) * 3)
    c = _reduce(oracle_mod, case)
    vb = bf16_bits_to_f32(torch_bf16_bits(vals))
    assert np.array_equal(c, np.broadcast_to(vb, c.shape))


def test_block_relabelling_invariance(oracle_mod):
    case = inputs.make_case(2, 1024, 64, seed=9)
    c0 = _reduce(oracle_mod, case)
    nb = case.state_bits.shape[0]
    perm = np.random.default_rng(10).permutation(nb)   # new block id of old id
    new_state = np.empty_like(case.state_bits)
    new_state[perm] = case.state_bits
    case.state_bits = new_state
    case.block_table = perm[case.block_table].astype(np.int32)
    c1 = _reduce(oracle_mod, case)
    assert np.array_equal(c0, c1)


def test_score_shift_invariance(oracle_mod):
    # scores are multiples of 1/8 in [-4, 4]: adding 2.0 stays exact in bf16
    rng = np.random.default_rng(11)
    T, C = 512, 128
    V = rng.standard_normal((T, 512)).astype(np.float32)
    S = (rng.integers(-32, 33, size=(T, 512)) / 8.0).astype(np.float32)
    a = _reduce(oracle_mod, _custom_case(C, T, lambda r, t: V[t], lambda r, t: S[t]))
    b = _reduce(oracle_mod, _custom_case(C, T, lambda r, t: V[t], lambda r, t: S[t] + 2.0))
    assert np.allclose(a, b, rtol=2 ** -22, atol=1e-30)


def test_bad_indices_are_reported_and_skipped(oracle_mod):
    case = inputs.make_case(1, 256, 16, seed=12)
    case.block_table = case.block_table.copy()
    case.block_table[0, 5] = 10_000           # used by the window ending at p=47
    c, valid, status = oracle_mod.window_reduce(
        case.state_bits, case.token_to_req, case.positions,
        case.boundary_token_indices, case.block_table, 16, 8)
    assert status == 4
    bad = [n for n, b in enumerate(case.boundary_token_indices)
           if (case.positions[b] - 15) // 8 <= 5 <= case.positions[b] // 8]
    assert bad and all(valid[n] == 0 for n in bad)
    assert sum(valid) == len(valid) - len(bad)
