"""Oracle pins for the fp32 state and the strided state / block-table layouts.

"The Baseline" of the KernelGen Challenge 8 write-up counts the window's
source traffic with an fp32 state element, and "A Bit of Triton and GPU
Background" reads the state through explicit block / row / column strides.
The oracle's general entry points (window_reduce_ex, compress_strided) take
the state as bf16 or fp32 with element strides and the block table with
row / column strides.

Pins (none re-types the oracle's loop):
* closed form in fp32: values t + d/1024 (not representable in bf16) with
  equal scores give the window mean exactly, so a state read as the wrong
  dtype or at the wrong element fails;
* the page's baseline (gather, softmax along the window, sum) evaluated by
  torch in float64 on the fp32 state;
* an fp32 state holding bf16 values reproduces the bf16 path bit for bit
  (c, y and every kv byte);
* a state embedded at padded strides with NaN everywhere else, and a block
  table stored column-major or with padded rows (-1 elsewhere), reproduce
  the contiguous results bit for bit.
"""
import numpy as np
import pytest
import torch

from kv_cache_compression_c128_gb300 import inputs
from kvc_testlib import bf16_bits_to_f32, gather_window_rows

W = 1024


def _contiguous_args(case):
    G, B = case.num_state_blocks, case.block_size
    R, M = case.block_table.shape
    return dict(block_stride=B * W, row_stride=W, num_blocks=G, num_reqs=R,
                max_blocks_per_req=M, bt_row_stride=M, bt_col_stride=1)


def _run(oracle_mod, case, state, **over):
    a = _contiguous_args(case)
    table = over.pop("table", case.block_table)
    a.update(over)
    kv = case.kv_cache.copy()
    res = oracle_mod.compress_strided(
        state, a["block_stride"], a["row_stride"], a["num_blocks"], case.token_to_req,
        case.positions, case.boundary_token_indices, table, a["num_reqs"],
        a["max_blocks_per_req"], a["bt_row_stride"], a["bt_col_stride"],
        case.rms_norm_weight, case.cos_sin_cache, case.kv_slot_mapping, kv,
        case.block_size, case.compress_ratio, case.rms_norm_eps)
    assert res["status"] == 0 and res["valid"].all()
    return kv, res


def test_fp32_equal_scores_give_exact_window_mean(oracle_mod):
    # v_{t,d} = t + d/1024 (18 significant bits: exact in fp32, not in bf16),
    # equal scores: c_d = p - (C - 1)/2 + d/1024 exactly.
    C, T = 32, 256
    case = inputs.make_case(1, T, C, seed=60)
    st = np.zeros((T // 8, 8, W), np.float32)
    d = np.arange(512)
    for t in range(T):
        g = int(case.block_table[0, t // 8])
        st[g, t % 8, :512] = t + d / 1024.0
        st[g, t % 8, 512:] = -1.25
    _, res = _run(oracle_mod, case, st)
    p = case.positions[case.boundary_token_indices].astype(np.float64)
    want = (p[:, None] - (C - 1) / 2.0 + d[None, :] / 1024.0).astype(np.float32)
    assert np.array_equal(res["c"], want)


@pytest.mark.parametrize("R,T,C", [(1, 512, 16), (2, 1024, 128), (1, 1024, 512)])
def test_fp32_reduce_matches_torch_softmax(oracle_mod, R, T, C):
    case = inputs.make_case(R, T, C, seed=61 + C)
    st = inputs.fp32_state(case.num_state_blocks, 8, seed=62 + C)
    _, res = _run(oracle_mod, case, st)
    rows = gather_window_rows(case)
    all_rows = torch.from_numpy(st.reshape(-1, W).astype(np.float64)[rows.reshape(-1)])
    all_rows = all_rows.reshape(rows.shape[0], C, W)
    ref = (all_rows[..., :512] * torch.softmax(all_rows[..., 512:], dim=1)).sum(dim=1).numpy()
    assert np.allclose(res["c"], ref, rtol=2 ** -23, atol=1e-12)
    # the fp32 values are not bf16 values: the bf16 reading would differ
    assert not np.array_equal(st, bf16_bits_to_f32(inputs._bf16_bits_from_f32(st)))


def test_fp32_state_of_bf16_values_matches_bf16_path(oracle_mod):
    case = inputs.make_case(2, 1024, 64, seed=63, kv_fill=64)
    kv_b, res_b = oracle_mod.compress_case(case)
    st32 = bf16_bits_to_f32(case.state_bits).astype(np.float32)
    kv_f, res_f = _run(oracle_mod, case, st32)
    assert np.array_equal(res_f["c"], res_b["c"]) and np.array_equal(res_f["y"], res_b["y"])
    assert np.array_equal(kv_f, kv_b)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("pad_row,pad_block", [(0, 24), (64, 0), (136, 1000)])
def test_strided_state_with_poisoned_padding(oracle_mod, dtype, pad_row, pad_block):
    case = inputs.make_case(2, 1024, 48, seed=65, block_size=16, boundaries_per_req=20)
    st = case.state_bits if dtype == "bf16" else inputs.fp32_state(
        case.num_state_blocks, 16, seed=66)
    kv0, res0 = _run(oracle_mod, case, st)
    rs = W + pad_row
    bs = 16 * rs + pad_block
    flat = inputs.embed_strided(st, bs, rs)
    kv1, res1 = _run(oracle_mod, case, flat, block_stride=bs, row_stride=rs)
    assert np.array_equal(res1["c"], res0["c"]) and np.array_equal(kv1, kv0)
    assert np.isnan(res1["y"]).sum() == 0


def test_block_table_column_major_and_padded_rows(oracle_mod):
    case = inputs.make_case(3, 1536, 64, seed=67, kv_fill=68)
    kv0, res0 = _run(oracle_mod, case, case.state_bits)
    R, M = case.block_table.shape
    cm = inputs.strided_table(case.block_table, 1, R)
    kv1, res1 = _run(oracle_mod, case, case.state_bits, table=cm, bt_row_stride=1,
                     bt_col_stride=R)
    assert np.array_equal(kv1, kv0) and np.array_equal(res1["c"], res0["c"])
    padded = inputs.strided_table(case.block_table, M + 7, 1)
    kv2, res2 = _run(oracle_mod, case, case.state_bits, table=padded, bt_row_stride=M + 7)
    assert np.array_equal(kv2, kv0) and np.array_equal(res2["c"], res0["c"])
    # a stride that walks into the -1 padding is reported, not read as a block
    kv = case.kv_cache.copy()
    bad = oracle_mod.compress_strided(
        case.state_bits, 8 * W, W, case.num_state_blocks, case.token_to_req, case.positions,
        case.boundary_token_indices, padded, R, M, M, 1, case.rms_norm_weight,
        case.cos_sin_cache, case.kv_slot_mapping, kv, 8, 64)
    assert bad["status"] == 4 and not bad["valid"].all()
