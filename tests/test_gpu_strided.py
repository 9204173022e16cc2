"""GPU parity for the fp32 state and the strided state / block-table layouts.

The fp32 element is the one "The Baseline" of the KernelGen Challenge 8
write-up counts the window's traffic with, and the block / row / column
strides are those of "A Bit of Triton and GPU Background".  The CUDA library
(kvc_compress_strided, reached through the torch wrapper, which passes the
tensors' own strides) is compared with the oracle's compress_strided on the
same seeded state, laid out in a buffer whose every other element is NaN, so
that a stride mistake on either side cannot pass.  The bar is the three-way
one of tests/test_gpu_parity.py.
"""
import numpy as np
import pytest
import torch

from kv_cache_compression_c128_gb300 import inputs
from kvc_testlib import assert_parity

pytestmark = pytest.mark.gpu

W = 1024


@pytest.fixture(scope="module")
def kvc():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import kv_cache_compression_c128_gb300 as kvc

    kvc.build()
    return kvc


class Layout:
    """A state (bf16 bits or fp32, [G, B, 1024]) embedded at element strides
    (block_stride, row_stride) and the case's block table stored row-major
    ("row"), column-major ("col") or with padded rows ("pad")."""

    def __init__(self, case, state, row_pad=0, block_pad=0, table="row"):
        G, B, _ = state.shape
        self.G, self.B = G, B
        self.rs = W + row_pad
        self.bs = B * self.rs + block_pad
        self.flat = inputs.embed_strided(state, self.bs, self.rs)
        self.f32 = state.dtype == np.float32
        R, M = case.block_table.shape
        self.R, self.M = R, M
        if table == "row":
            self.bt_rs, self.bt_cs = M, 1
        elif table == "col":
            self.bt_rs, self.bt_cs = 1, R
        else:
            self.bt_rs, self.bt_cs = M + 7, 1
        self.table = inputs.strided_table(case.block_table, self.bt_rs, self.bt_cs)

    def device(self, dev="cuda"):
        if self.f32:
            flat = torch.from_numpy(self.flat).to(dev)
        else:
            flat = torch.from_numpy(self.flat.view(np.int16)).view(torch.bfloat16).to(dev)
        st = flat.as_strided((self.G, self.B, W), (self.bs, self.rs, 1))
        tab = torch.from_numpy(self.table).to(dev).as_strided(
            (self.R, self.M), (self.bt_rs, self.bt_cs))
        return st, tab

    def oracle(self, oracle_mod, case, slot_mapping=None):
        kv = case.kv_cache.copy()
        sm = case.kv_slot_mapping if slot_mapping is None else slot_mapping
        res = oracle_mod.compress_strided(
            self.flat, self.bs, self.rs, self.G, case.token_to_req, case.positions,
            case.boundary_token_indices, self.table, self.R, self.M, self.bt_rs, self.bt_cs,
            case.rms_norm_weight, case.cos_sin_cache, sm, kv, case.block_size,
            case.compress_ratio, case.rms_norm_eps)
        return kv, res


def _index_arrays(case, dev="cuda"):
    t = lambda a: torch.from_numpy(a).to(dev)
    return dict(token_to_req=t(case.token_to_req), positions=t(case.positions),
                boundary_token_indices=t(case.boundary_token_indices),
                rms_norm_weight=t(case.rms_norm_weight), cos_sin_cache=t(case.cos_sin_cache),
                kv_slot_mapping=t(case.kv_slot_mapping), kv_cache=t(case.kv_cache.copy()))


def run_layout(kvc, case, lay, flags=0):
    st, tab = lay.device()
    d = _index_arrays(case)
    N = case.num_outputs
    y = torch.full((max(N, 1), 512), float("nan"), dtype=torch.float32, device="cuda")
    kvc.c128_256_512_compress(st, block_table=tab, block_size=case.block_size,
                              compress_ratio=case.compress_ratio,
                              rms_norm_eps=case.rms_norm_eps, y_out=y, flags=flags, **d)
    err = kvc.kvc_get_device_error(torch.cuda.current_stream().cuda_stream)
    return d["kv_cache"].cpu().numpy(), y[:N].cpu().numpy(), err


def check_layout(kvc, oracle_mod, case, lay, flags=0):
    kv_g, y_g, err = run_layout(kvc, case, lay, flags)
    assert err == 0, f"device error {err}"
    ref = lay.oracle(oracle_mod, case)
    assert ref[1]["status"] == 0
    return assert_parity(oracle_mod, case, kv_g, y_g, ref=ref)


def _fp32(case, seed):
    return inputs.fp32_state(case.num_state_blocks, case.block_size, seed)


# ---- fp32 state ----------------------------------------------------------------------

@pytest.mark.parametrize("S,count", [(0, 0), (1, 0), (2, 0), (4, 3), (8, 0), (16, 1)])
def test_fp32_every_cluster_size(kvc, oracle_mod, S, count):
    case = inputs.make_case(2, 4096, 256, seed=inputs.BASE_SEED + 800, kv_fill=81)
    lay = Layout(case, _fp32(case, 82))
    route = "auto" if S == 0 else "cluster"
    check_layout(kvc, oracle_mod, case, lay, kvc.make_flags(route, count, S))


@pytest.mark.parametrize("C,B", [(8, 8), (20, 8), (100, 16), (512, 40), (128, 8)])
def test_fp32_general_windows(kvc, oracle_mod, C, B):
    case = inputs.make_case(3, 6000 if B == 40 else 6144, C, seed=inputs.BASE_SEED + 810 + C,
                            block_size=B, boundaries_per_req=40, kv_fill=83)
    lay = Layout(case, _fp32(case, 84 + C))
    check_layout(kvc, oracle_mod, case, lay)
    if C >= 32:
        check_layout(kvc, oracle_mod, case, lay, kvc.make_flags("cluster", 5, 4))


def test_fp32_of_bf16_values_matches_the_bf16_call(kvc, oracle_mod):
    # the same values stored as fp32: both calls meet the bar against the
    # oracle's bf16 run, and their y differ only by fp32 summation order (the
    # bf16 kernel folds 16 rows per rescale, the fp32 kernel 8)
    case = inputs.make_case(2, 2048, 128, seed=inputs.BASE_SEED + 820, kv_fill=85)
    st32 = (case.state_bits.astype(np.uint32) << 16).view(np.float32)
    kv32, y32, e32 = run_layout(kvc, case, Layout(case, st32))
    kv16, y16, e16 = run_layout(kvc, case, Layout(case, case.state_bits))
    assert e32 == 0 and e16 == 0
    rms = np.sqrt((y16.astype(np.float64) ** 2).mean(1, keepdims=True))
    assert np.all(np.abs(y32 - y16) <= 1e-5 * (np.abs(y16) + rms))
    assert_parity(oracle_mod, case, kv32, y32)
    assert_parity(oracle_mod, case, kv16, y16)


def test_fp32_bad_block_is_reported_and_skipped(kvc, oracle_mod):
    case = inputs.make_case(1, 1024, 64, seed=inputs.BASE_SEED + 830, kv_fill=86)
    case.block_table = case.block_table.copy()
    case.block_table[0, 9] = 10_000
    lay = Layout(case, _fp32(case, 87))
    kv_g, y_g, err = run_layout(kvc, case, lay)
    assert err == 4
    kv_o, res = lay.oracle(oracle_mod, case)
    assert res["status"] == 4
    bad = res["valid"] == 0
    assert bad.any() and not bad.all()
    assert np.allclose(y_g[~bad], res["y"][~bad], rtol=2e-3, atol=1e-4)
    # the valid outputs' bytes follow from the GPU's y; the others stay untouched
    kv_y = case.kv_cache.copy()
    oracle_mod.quant_rope_scatter(y_g, case.positions, case.boundary_token_indices,
                                  case.compress_ratio, case.cos_sin_cache,
                                  case.kv_slot_mapping, kv_y, valid=(~bad).astype(np.uint8))
    assert np.array_equal(kv_g, kv_y)


# ---- strided state and block table -----------------------------------------------------

LAYOUTS = [(0, 256, "col"), (64, 0, "row"), (64, 512, "pad"), (8 * 16, 64, "col")]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("row_pad,block_pad,table", LAYOUTS)
def test_strided_general_windows(kvc, oracle_mod, dtype, row_pad, block_pad, table):
    case = inputs.make_case(2, 4096, 48, seed=inputs.BASE_SEED + 840, block_size=16,
                            boundaries_per_req=50, kv_fill=88)
    st = case.state_bits if dtype == "bf16" else _fp32(case, 89)
    lay = Layout(case, st, row_pad, block_pad, table)
    check_layout(kvc, oracle_mod, case, lay)
    check_layout(kvc, oracle_mod, case, lay, kvc.make_flags("cluster", 3, 2))


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("S", [1, 4, 16])
def test_strided_rows_aligned_windows(kvc, oracle_mod, dtype, S):
    case = inputs.make_case(4, 8192, 128, seed=inputs.BASE_SEED + 850, kv_fill=90)
    st = case.state_bits if dtype == "bf16" else _fp32(case, 91)
    lay = Layout(case, st, row_pad=64, block_pad=128, table="pad")
    check_layout(kvc, oracle_mod, case, lay, kvc.make_flags("cluster", 0, S))


@pytest.mark.parametrize("grid", [0, 1, 7, 64])
def test_stream_k_with_padded_blocks_and_column_major_table(kvc, oracle_mod, grid):
    case = inputs.make_case(3, 6144, 128, seed=inputs.BASE_SEED + 860, kv_fill=92)
    lay = Layout(case, case.state_bits, row_pad=0, block_pad=512, table="col")
    check_layout(kvc, oracle_mod, case, lay, kvc.make_flags("streamk", grid))


def test_stream_k_rejects_fp32_and_split_rows(kvc):
    case = inputs.make_case(1, 1024, 64, seed=inputs.BASE_SEED + 870)
    for lay in (Layout(case, _fp32(case, 93)), Layout(case, case.state_bits, row_pad=64)):
        with pytest.raises(kvc.KvcError) as ei:
            run_layout(kvc, case, lay, kvc.make_flags("streamk"))
        assert ei.value.status == 2


def test_query_launch_ex_matches_bf16_footprint(kvc):
    a = kvc.kvc_query_launch_ex(1024, 128, kvc.KVC_DTYPE_F32)
    b = kvc.kvc_query_launch(1024, 128)
    assert a[2] == b[2] and a[3] == b[3] and a[0] >= 1 and a[1] >= 1


# ---- full sizes ----------------------------------------------------------------------

@pytest.mark.parametrize("C", [128, 512])
def test_fp32_headline_shape_full_size(kvc, oracle_mod, C):
    # 8 requests x 16384 tokens, fp32 state (512 MiB), every output checked
    case = inputs.make_case(8, 131072, C, seed=inputs.BASE_SEED + 880 + C)
    lay = Layout(case, _fp32(case, 94 + C))
    check_layout(kvc, oracle_mod, case, lay)


def test_bf16_split_rows_headline_shape_full_size(kvc, oracle_mod):
    # rows 64 elements apart (one bulk copy per row), padded table rows
    case = inputs.headline_case()
    lay = Layout(case, case.state_bits, row_pad=64, block_pad=0, table="pad")
    check_layout(kvc, oracle_mod, case, lay)


# ---- rows apart: tensor-map copies against row-by-row copies ---------------------------

@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("C,B,nb,route", [
    (128, 8, None, "auto"),     # aligned windows: every chunk is one tensor copy
    (256, 8, None, "s4"),       # the same through a cluster of 4
    (48, 16, 50, "auto"),       # general windows: chunks split between blocks go row by row
    (100, 24, 40, "s2"),
    (512, 64, 12, "auto"),
])
def test_rows_apart_tensor_and_row_copies_agree(kvc, oracle_mod, dtype, C, B, nb, route):
    # Rows apart are copied 8 at a time through a TMA tensor map per layer;
    # with KVC_FLAG_ROW_COPIES one bulk copy per row.  Both fill the ring with
    # the same bytes, so results are identical, and both meet the bar.  The
    # gaps between rows hold NaN, so a box that strayed would show.
    T = 3 * (2064 if B == 24 else 2048)  # requests of whole blocks
    case = inputs.make_case(3, T, C, seed=inputs.BASE_SEED + 880 + C, block_size=B,
                            boundaries_per_req=nb, kv_fill=94)
    f32 = dtype == "f32"
    st = _fp32(case, 95) if f32 else case.state_bits
    lay = Layout(case, st, row_pad=32 if f32 else 64, block_pad=256, table="pad")
    S = 0 if route == "auto" else int(route[1:])
    flags = kvc.make_flags("auto" if S == 0 else "cluster", 0, S)
    kv_t, y_t, e_t = run_layout(kvc, case, lay, flags)
    kv_r, y_r, e_r = run_layout(kvc, case, lay, flags | kvc.KVC_FLAG_ROW_COPIES)
    assert e_t == 0 and e_r == 0 and case.num_outputs > 0
    assert np.array_equal(kv_t, kv_r)
    assert np.array_equal(y_t.view(np.uint32), y_r.view(np.uint32))
    ref = lay.oracle(oracle_mod, case)
    assert ref[1]["status"] == 0
    assert_parity(oracle_mod, case, kv_t, y_t, ref=ref)
