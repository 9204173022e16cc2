"""GPU parity: the CUDA library (called through its C ABI) against the oracle.

Three checks per case, on the same seeded inputs (the bar of the write-up's
"Byte-Level Correctness" section, with the floating-point parts given a
tolerance because the kernel reduces in fp32 where the oracle uses double):

1. the pre-quantisation vector y (exported through y_out) is within 2e-3
   relative of the oracle's: |y_gpu - y_ref| <= 2e-3 |y_ref| + 1e-5 rms(y_ref);
2. the kv_cache bytes are bit-exact against the oracle's quantise / rotate /
   scatter step applied to the GPU's own y -- so quantisation codes, scale
   bytes, padding, RoPE bf16 bytes, slot placement and every byte outside the
   written slots are all checked exactly, the floating-point decisions being
   taken on the same fp32 input on both sides;
3. against the oracle's own bytes: every byte outside the written slots is
   identical; per element the dequantised NOPE values differ by at most one
   quantisation step, scale bytes by at most one; RoPE values by at most one
   bf16 ulp plus what the y tolerance allows after a norm-preserving
   rotation: 2e-3 |(u, w)| + 1.5e-5 rms(y) (where u cos ~ w sin cancel, a
   tiny difference in y is many ulps of the tiny result).
"""
import numpy as np
import pytest
import torch

from kv_cache_compression_c128_gb300 import inputs
from kvc_testlib import (assert_parity, run_gpu, slots_of_case, to_device,
                         written_mask)

pytestmark = pytest.mark.gpu

@pytest.fixture(scope="module")
def kvc():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import kv_cache_compression_c128_gb300 as kvc

    kvc.build()
    return kvc


def check_case(oracle_mod, case, flags=0, valid_outputs=None):
    """Run GPU and oracle on `case`, assert the three-way bar; return stats."""
    kv_g, y_g, err = run_gpu(case, flags)
    assert err == 0, f"device error {err}"
    return assert_parity(oracle_mod, case, kv_g, y_g)


SMALL = [(1, 256, 8), (2, 1024, 16), (2, 2048, 128), (1, 4096, 512), (3, 3072, 64),
         (4, 4096, 256)]


ROUTES = ([("auto", 0, 0)] + [("streamk", g, 0) for g in (1, 3, 7, 13, 64)]
          + [("cluster", n, S) for S in (1, 2, 4, 8, 16) for n in (0, 1, 3)])


@pytest.mark.parametrize("R,T,C", SMALL)
@pytest.mark.parametrize("route,count,S", ROUTES)
def test_small_cases_every_route(kvc, oracle_mod, R, T, C, route, count, S):
    if S > C // 8:
        pytest.skip("cluster larger than the window's block count")
    case = inputs.make_case(R, T, C, seed=inputs.BASE_SEED + 500 + C + R, kv_fill=11)
    check_case(oracle_mod, case, flags=kvc.make_flags(route, count, S))


@pytest.mark.parametrize("C", [128, 512])
@pytest.mark.parametrize("S", [1, 2, 4, 8, 16])
def test_full_size_every_cluster_size(kvc, oracle_mod, C, S):
    case = inputs.make_case(4, 32768, C, seed=inputs.BASE_SEED + 600 + C, kv_fill=12)
    check_case(oracle_mod, case, flags=kvc.make_flags("cluster", 0, S))


def test_full_size_stream_k_route(kvc, oracle_mod):
    check_case(oracle_mod, inputs.bench_case(3), flags=kvc.make_flags("streamk"))


@pytest.mark.parametrize("case_id", range(12))
def test_benchmark_shapes_full_size(kvc, oracle_mod, case_id):
    case = inputs.bench_case(case_id)
    check_case(oracle_mod, case)


@pytest.mark.parametrize("C", [128, 256, 512])
def test_ragged_variant(kvc, oracle_mod, C):
    case = inputs.ragged_case(C)
    check_case(oracle_mod, case)


def test_ragged_with_odd_grids(kvc, oracle_mod):
    L = inputs.ragged_lengths(5, 20480, 128, seed=77)
    case = inputs.make_case(5, 20480, 128, seed=78, lengths=L, kv_fill=79)
    for grid in (1, 5, 17, 151, 299):
        check_case(oracle_mod, case, flags=kvc.make_flags("streamk", grid))
    for n, S in ((1, 2), (5, 4), (17, 8), (7, 16), (151, 1)):
        check_case(oracle_mod, case, flags=kvc.make_flags("cluster", n, S))


def test_deterministic_repeat(kvc, oracle_mod):
    case = inputs.make_case(4, 8192, 256, seed=80)
    d = to_device(case)
    kv1, y1, e1 = run_gpu(case, dev_arrays=d)
    d["kv_cache"].copy_(torch.from_numpy(case.kv_cache))
    kv2, y2, e2 = run_gpu(case, dev_arrays=d)
    assert e1 == 0 and e2 == 0
    assert np.array_equal(kv1, kv2) and np.array_equal(y1.view(np.uint32), y2.view(np.uint32))


def test_zero_outputs(kvc):
    case = inputs.make_case(1, 256, 16, seed=81, kv_fill=82)
    d = to_device(case)
    d["boundary_token_indices"] = d["boundary_token_indices"][:0]
    kvc.c128_256_512_compress(block_size=8, compress_ratio=16, **d)
    assert kvc.kvc_get_device_error(torch.cuda.current_stream().cuda_stream) == 0
    assert np.array_equal(d["kv_cache"].cpu().numpy(), case.kv_cache)


def test_slot_mapping_by_output_and_negative_slot(kvc, oracle_mod):
    case = inputs.make_case(2, 4096, 64, seed=83, kv_fill=84)
    per_out = case.kv_slot_mapping[case.boundary_token_indices].copy()
    kv_tok, _, e0 = run_gpu(case)
    kv_out, _, e1 = run_gpu(case, slot_mapping=per_out)
    assert e0 == 0 and e1 == 0 and np.array_equal(kv_tok, kv_out)
    skip = per_out.copy()
    old = int(skip[5])
    skip[5] = -1
    kv_skip, y_skip, e2 = run_gpu(case, slot_mapping=skip)
    assert e2 == 0
    m = written_mask(kv_skip.shape, [old])
    assert np.array_equal(kv_skip.reshape(-1)[m], case.kv_cache.reshape(-1)[m])
    assert np.array_equal(kv_skip.reshape(-1)[~m], kv_tok.reshape(-1)[~m])
    assert np.all(np.isfinite(y_skip[5]))      # y is still produced


def _expect_device_error(kvc, case, code, bad_outputs, oracle_mod, grid=0):
    kv_g, y_g, err = run_gpu(case, flags=grid)
    assert err == code
    slots = slots_of_case(case)
    # skipped outputs leave their slots untouched
    m_bad = written_mask(kv_g.shape, [slots[n] for n in bad_outputs])
    assert np.array_equal(kv_g.reshape(-1)[m_bad], case.kv_cache.reshape(-1)[m_bad])
    # every other output is still written correctly (bytes follow from y)
    good = np.array([n not in set(bad_outputs) for n in range(case.num_outputs)])
    kv_y = case.kv_cache.copy()
    oracle_mod.quant_rope_scatter(y_g, case.positions, case.boundary_token_indices,
                                  case.compress_ratio, case.cos_sin_cache,
                                  case.kv_slot_mapping, kv_y, valid=good.astype(np.uint8))
    assert np.array_equal(kv_g, kv_y)
    return kv_g


@pytest.mark.parametrize("grid", [0, 3 | (1 << 24), 2 << 16, 8 << 16])
def test_bad_block_index_is_reported_and_skipped(kvc, oracle_mod, grid):
    case = inputs.make_case(2, 2048, 128, seed=85, kv_fill=86)
    case.block_table = case.block_table.copy()
    case.block_table[1, 20] = 10 ** 6            # output window 1 of request 1
    bad = [n for n, b in enumerate(case.boundary_token_indices)
           if case.token_to_req[b] == 1 and case.positions[b] // 128 == 1]
    _expect_device_error(kvc, case, 4, bad, oracle_mod, grid)


def test_window_before_sequence_start(kvc, oracle_mod):
    case = inputs.make_case(1, 1024, 64, seed=87, kv_fill=88)
    case.boundary_token_indices = case.boundary_token_indices.copy()
    case.boundary_token_indices[2] = 7          # p = 7 < C - 1
    _expect_device_error(kvc, case, 4, [2], oracle_mod)


def test_unaligned_window_stream_k_unsupported_cluster_exact(kvc, oracle_mod):
    case = inputs.make_case(1, 1024, 64, seed=89, kv_fill=90)
    case.boundary_token_indices = case.boundary_token_indices.copy()
    case.boundary_token_indices[3] += 1          # window starts at an odd row
    # the stream-K route handles only block-aligned windows: reported, skipped
    _expect_device_error(kvc, case, 2, [3], oracle_mod, grid=kvc.make_flags("streamk"))
    # the cluster route computes it like any other window
    check_case(oracle_mod, case)


def test_slot_and_position_out_of_range(kvc, oracle_mod):
    case = inputs.make_case(1, 2048, 64, seed=91, kv_fill=92)
    case.kv_slot_mapping = case.kv_slot_mapping.copy()
    b4 = case.boundary_token_indices[4]
    case.kv_slot_mapping[b4] = 64 * case.kv_cache.shape[0] + 3   # beyond the last page
    kv_g, _, err = run_gpu(case)
    assert err == 4
    # cos_sin_cache too short for the last window's compressed position
    case2 = inputs.make_case(1, 2048, 64, seed=93, kv_fill=94)
    case2.cos_sin_cache = case2.cos_sin_cache[:2000].copy()
    last = case2.num_outputs - 1                 # pc = 1984 < 2000 -> fine
    kv2, _, err2 = run_gpu(case2)
    assert err2 == 0
    case2.cos_sin_cache = case2.cos_sin_cache[:1984].copy()    # pc = 1984 now out of range
    _expect_device_error(kvc, case2, 4, [last], oracle_mod)


# ---- general windows: any start, any C >= 1, block_size >= 8 ------------------

GENERAL = [  # (num_reqs, total_tokens, C, block_size, boundaries per request)
    (2, 1024, 37, 8, 20),
    (2, 1024, 100, 16, 20),
    (1, 2048, 1, 8, 40),
    (3, 1440, 5, 24, 16),
    (2, 4096, 300, 64, 12),
    (1, 4096, 128, 8, 25),     # the benchmark's C at unaligned window starts
    (1, 4096, 512, 32, 10),
]


@pytest.mark.parametrize("R,T,C,B,nb", GENERAL)
@pytest.mark.parametrize("S", [0, 1, 2, 4, 8, 16])
def test_general_windows(kvc, oracle_mod, R, T, C, B, nb, S):
    if S > -(-C // 8):
        pytest.skip("cluster larger than the window's chunk count")
    case = inputs.make_case(R, T, C, seed=inputs.BASE_SEED + 700 + C + B, block_size=B,
                            boundaries_per_req=nb, kv_fill=13)
    check_case(oracle_mod, case, flags=kvc.make_flags("cluster", 0, S) if S else 0)


def test_general_windows_not_on_the_stream_k_route(kvc):
    case = inputs.make_case(1, 1024, 100, seed=5, block_size=16, boundaries_per_req=4)
    with pytest.raises(kvc.KvcError) as ei:
        run_gpu(case, flags=kvc.make_flags("streamk"))
    assert ei.value.status == kvc.KVC_ERR_UNSUPPORTED
