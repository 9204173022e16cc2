"""C-ABI checks that need no GPU.

The library is compiled for sm_103a on the CPU machine (nvcc cross-compiles),
loaded with ctypes, and checked to export every function include/kvc.h
declares.  Every argument check kvc_compress performs on the host happens
before any CUDA call, so the error paths run here too.
"""
import ctypes
import os
import re
import shutil

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

pytestmark = pytest.mark.skipif(shutil.which("nvcc") is None and
                                not os.path.exists("/usr/local/cuda/bin/nvcc"),
                                reason="nvcc not available")


@pytest.fixture(scope="module")
def kvc():
    import kv_cache_compression_c128_gb300 as kvc

    kvc.build()
    return kvc


def _declared_functions():
    with open(os.path.join(ROOT, "include", "kvc.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kvc_[a-z_]+)\s*\(", text)))


def test_header_declares_the_abi():
    names = _declared_functions()
    assert {"kvc_compress", "kvc_workspace_bytes", "kvc_get_device_error",
            "kvc_error_string", "kvc_version", "kvc_query_launch"} <= set(names)


def test_library_exports_every_declared_symbol(kvc):
    lib = ctypes.CDLL(kvc.LIB_PATH)
    for name in _declared_functions():
        assert hasattr(lib, name), f"{name} declared in kvc.h but not exported"


def test_library_is_built_for_sm_103a(kvc):
    # the fatbin carries an sm_103a cubin: the ELF note lists the arch name
    with open(kvc.LIB_PATH, "rb") as f:
        blob = f.read()
    assert b"sm_103a" in blob or b"sm_103" in blob


def test_strings(kvc):
    assert kvc.kvc_error_string(0) == "ok"
    assert "index" in kvc.kvc_error_string(4)
    assert kvc.kvc_error_string(99) == "unknown status"
    assert "sm_103a" in kvc.kvc_version()


# a valid-looking argument set; pointers are fake (never dereferenced on the
# host, and every case below is rejected before any CUDA call)
_GOOD = dict(state_cache=0x10000, num_state_blocks=1024, token_to_req=0x20000,
             positions=0x30000, num_tokens=8192, boundary_token_indices=0x40000,
             num_outputs=64, block_table=0x50000, num_reqs=1, max_blocks_per_req=1024,
             rms_norm_weight=0x60000, cos_sin_cache=0x70000, num_positions=8192,
             kv_slot_mapping=0x80000, slot_mapping_len=8192, kv_cache=0x90000,
             num_kv_pages=1, block_size=8, compress_ratio=128, rms_norm_eps=1e-6,
             y_out=0, workspace=0xA0000, workspace_bytes=1 << 24, flags=0, stream=0)


@pytest.mark.parametrize("change,status", [
    (dict(block_size=4), 2),
    (dict(block_size=0), 2),
    (dict(compress_ratio=0), 1),
    (dict(compress_ratio=-8), 1),
    (dict(num_outputs=-1), 1),
    (dict(flags=1 << 28), 1),
    (dict(rms_norm_eps=float("nan")), 1),
    (dict(rms_norm_eps=-1.0), 1),
    (dict(state_cache=0), 1),
    (dict(kv_cache=0), 1),
    (dict(workspace=0), 1),
    (dict(num_kv_pages=0), 1),
    (dict(slot_mapping_len=77), 1),
    (dict(state_cache=0x10008), 1),      # not 16-byte aligned
    (dict(kv_cache=0x90004), 1),
    (dict(positions=0x30004), 1),
    (dict(y_out=0xB0004), 1),
])
def test_host_argument_validation(kvc, change, status):
    args = dict(_GOOD, **change)
    assert kvc.kvc_compress(**args) == status


def test_zero_outputs_is_a_no_op(kvc):
    assert kvc.kvc_compress(**dict(_GOOD, num_outputs=0)) == 0


def test_query_launch_rejects_bad_arguments(kvc):
    with pytest.raises(kvc.KvcError):
        kvc.kvc_query_launch(64, 0)
    with pytest.raises(kvc.KvcError):
        kvc.kvc_query_launch(-1, 128)
    with pytest.raises(kvc.KvcError):
        kvc.kvc_query_launch(64, 128, 1 << 28)


def test_make_flags(kvc):
    assert kvc.make_flags() == 0
    assert kvc.make_flags("cluster", 3, 8) == 3 | (8 << 16)
    assert kvc.make_flags("streamk", 13) == 13 | (1 << 24)
    assert kvc.make_flags(row_copies=True) == 1 << 25


def test_flag_constants_match_the_header(kvc):
    # the Python constants and the header's #defines name the same bits
    import os

    hdr = open(os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "kvc.h")).read()
    for name, value in (("KVC_FLAG_STREAM_K", kvc.KVC_FLAG_STREAM_K),
                        ("KVC_FLAG_ROW_COPIES", kvc.KVC_FLAG_ROW_COPIES)):
        m = re.search(r"#define %s \(1u << (\d+)\)" % name, hdr)
        assert m and (1 << int(m.group(1))) == value


def test_row_copies_flag_is_accepted(kvc):
    # bit 25 is a known flag: the call gets past the flag check (an unknown
    # bit returns INVALID_ARG) to the block-size check (UNSUPPORTED)
    small = dict(_GOOD, block_size=4)
    assert kvc.kvc_compress(**dict(small, flags=kvc.KVC_FLAG_ROW_COPIES)) == 2
    assert kvc.kvc_compress(**dict(small, flags=1 << 26)) == 1


def test_torch_wrapper_rejects_cpu_tensors(kvc):
    import torch

    from kv_cache_compression_c128_gb300 import inputs

    case = inputs.make_case(1, 256, 16, seed=1)
    st = torch.from_numpy(case.state_bits.view("int16")).view(torch.bfloat16)
    t = torch.from_numpy
    with pytest.raises(ValueError, match="no CPU path"):
        kvc.c128_256_512_compress(st, t(case.token_to_req), t(case.positions),
                                  t(case.boundary_token_indices), t(case.block_table),
                                  t(case.rms_norm_weight), t(case.cos_sin_cache),
                                  t(case.kv_slot_mapping), t(case.kv_cache), 8, 16)


@pytest.mark.parametrize("change,status", [
    (dict(out_dtype=7), 1),
    (dict(num_slots=-1), 1),
    (dict(kv_cache=0), 1),
    (dict(out=0x30004), 1),            # fp32 output must be 16-byte aligned
    (dict(slots=0x20004), 1),
    (dict(num_kv_pages=0), 1),
])
def test_dequantize_host_validation(kvc, change, status):
    args = dict(kv_cache=0x10000, num_kv_pages=1, slots=0x20000, num_slots=8, out=0x30000,
                out_dtype=0, stream=0)
    args.update(change)
    assert kvc.kvc_dequantize(**args) == status


def test_dequantize_zero_slots_is_a_no_op(kvc):
    assert kvc.kvc_dequantize(0x10000, 1, 0x20000, 0, 0x30000, 0, 0) == 0


def test_layers_host_validation(kvc):
    args = dict(_GOOD)
    for k in ("state_cache", "rms_norm_weight", "kv_cache"):
        args.pop(k)
    base = dict(num_layers=2, state_caches=[0x10000, 0x11000], rms_norm_weights=[0x60000, 0x61000],
                kv_caches=[0x90000, 0x91000], **args)
    assert kvc.kvc_compress_layers(**dict(base, num_layers=0)) == 1
    assert kvc.kvc_compress_layers(**dict(base, num_layers=65, state_caches=[0x10000] * 65,
                                          rms_norm_weights=[0x60000] * 65,
                                          kv_caches=[0x90000] * 65)) == 1
    assert kvc.kvc_compress_layers(**dict(base, state_caches=[0x10000, 0])) == 1
    assert kvc.kvc_compress_layers(**dict(base, kv_caches=[0x90000, 0x91004])) == 1
    assert kvc.kvc_compress_layers(**dict(base, num_outputs=0)) == 0


def _strided_args(**change):
    args = dict(_GOOD)
    args.update(state_dtype=1, state_block_stride=8 * 1024, state_row_stride=1024,
                block_table_row_stride=1024, block_table_col_stride=1)
    args.update(change)
    return args


@pytest.mark.parametrize("change,status", [
    (dict(state_dtype=2), 1),                       # unknown element type
    (dict(state_dtype=-1), 1),
    (dict(state_block_stride=-8), 1),
    (dict(state_row_stride=-1024), 1),
    (dict(block_table_row_stride=-1), 1),
    (dict(block_table_col_stride=-1), 1),
    (dict(state_row_stride=1028), 2),               # bf16: 2056 B, not a multiple of 16
    (dict(state_block_stride=8 * 1024 + 4), 2),
    (dict(state_dtype=0, state_row_stride=1026), 2),  # fp32: 4104 B
    (dict(state_block_stride=1 << 62), 1),          # byte offsets overflow int64
    (dict(block_table_row_stride=1 << 62, num_reqs=8), 1),
    (dict(block_size=4), 2),
    (dict(state_cache=0x10008), 1),
])
def test_strided_host_validation(kvc, change, status):
    assert kvc.kvc_compress_strided(**_strided_args(**change)) == status


def test_strided_zero_outputs_is_a_no_op(kvc):
    assert kvc.kvc_compress_strided(**_strided_args(num_outputs=0)) == 0
    assert kvc.kvc_compress_strided(**_strided_args(num_outputs=0, state_dtype=0)) == 0


def test_query_launch_ex_rejects_bad_dtype(kvc):
    with pytest.raises(kvc.KvcError):
        kvc.kvc_query_launch_ex(64, 128, 5)


def test_torch_wrapper_rejects_strided_columns(kvc):
    import torch

    from kv_cache_compression_c128_gb300 import inputs

    case = inputs.make_case(1, 256, 16, seed=1)
    st = torch.zeros((32, 1024, 8), dtype=torch.float32).transpose(1, 2)
    t = torch.from_numpy
    with pytest.raises(ValueError):
        kvc.c128_256_512_compress(st, t(case.token_to_req), t(case.positions),
                                  t(case.boundary_token_indices), t(case.block_table),
                                  t(case.rms_norm_weight), t(case.cos_sin_cache),
                                  t(case.kv_slot_mapping), t(case.kv_cache), 8, 16)


def test_selftest_wait_rejects_bad_limits(kvc):
    assert kvc.kvc_selftest_wait_timeout(0) == 1
    assert kvc.kvc_selftest_wait_timeout(4_000_000_001) == 1


def test_selftest_wait_limit_range(kvc):
    # host-side range check only (no launch): 0 restores the default
    assert kvc.kvc_selftest_set_wait_limit(4_000_000_001) == 1
    assert kvc.kvc_selftest_set_wait_limit(500) == 0
    assert kvc.kvc_selftest_set_wait_limit(0) == 0


def test_selftest_poison_guesses_range(kvc):
    # host-side range check only (no launch): 0 restores normal guesses
    assert kvc.lib().kvc_selftest_poison_guesses(2) == 1
    assert kvc.lib().kvc_selftest_poison_guesses(-1) == 1
    assert kvc.kvc_selftest_poison_guesses(True) == 0
    assert kvc.kvc_selftest_poison_guesses(False) == 0


def test_selftest_first_pass_rejections_needs_an_output(kvc):
    lib = kvc.lib()
    assert lib.kvc_selftest_first_pass_rejections(None, None) == 1
