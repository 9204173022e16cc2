"""GPU parity of the reader direction (kvc_dequantize) against the oracle.

Decoding is exact arithmetic (int8 code times a power of two, bf16 widened),
so the bar is bit-exact: the GPU's fp32 and bf16 outputs equal the oracle's
reader on the same kv_cache bytes -- caches written by the GPU compressor,
and random bytes covering every code and scale exponent.  Negative slots read
as zeros; slots beyond the last page read as zeros and raise the device error
word.  A round trip (compress, then read) returns the NOPE values within one
quantisation step of bf16(y).
"""
import numpy as np
import pytest
import torch

from kv_cache_compression_c128_gb300 import inputs
from kvc_testlib import bf16_bits_to_f32, run_gpu, slots_of_case, torch_bf16_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvc():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import kv_cache_compression_c128_gb300 as kvc

    kvc.build()
    return kvc


def _read(kvc, kv_np, slots, dtype):
    kv = torch.from_numpy(kv_np).cuda()
    sl = torch.from_numpy(np.ascontiguousarray(slots, dtype=np.int64)).cuda()
    out = kvc.dequantize(kv, sl, dtype=dtype)
    err = kvc.kvc_get_device_error(torch.cuda.current_stream().cuda_stream)
    if dtype == torch.bfloat16:
        return out.view(torch.int16).cpu().numpy().view(np.uint16), err
    return out.cpu().numpy(), err


@pytest.mark.parametrize("case_id", [0, 3, 8])
def test_reader_exact_on_compressed_cache(kvc, oracle_mod, case_id):
    case = inputs.bench_case(case_id)
    kv_g, y_g, err = run_gpu(case)
    assert err == 0
    slots = slots_of_case(case)
    for dtype, bf in ((torch.float32, False), (torch.bfloat16, True)):
        got, e = _read(kvc, kv_g, slots, dtype)
        want, st = oracle_mod.dequantize(kv_g, slots, out_bf16=bf)
        assert e == 0 and st == 0
        assert np.array_equal(got.view(np.uint32 if not bf else np.uint16),
                              want.view(np.uint32 if not bf else np.uint16))
    # round trip: NOPE values within one quantisation step of bf16(y)
    got, _ = _read(kvc, kv_g, slots, torch.float32)
    z = bf16_bits_to_f32(torch_bf16_bits(y_g[:, :448]))
    for n, s in enumerate(slots):
        pg, off = divmod(int(s), 64)
        e = kv_g[pg, 36864 + off * 8: 36864 + off * 8 + 7].astype(np.int64) - 127
        step = np.repeat(np.ldexp(1.0, e), 64)
        assert np.all(np.abs(got[n, :448].astype(np.float64) - z[n]) < step)


def test_reader_exact_on_random_bytes(kvc, oracle_mod):
    rng = np.random.default_rng(41)
    kv = rng.integers(0, 256, size=(5, 37376), dtype=np.uint8)
    slots = np.concatenate([rng.permutation(5 * 64), [-1, -7, 3]]).astype(np.int64)
    for dtype, bf in ((torch.float32, False), (torch.bfloat16, True)):
        got, e = _read(kvc, kv, slots, dtype)
        want, st = oracle_mod.dequantize(kv, slots, out_bf16=bf)
        assert e == 0 and st == 0
        view = np.uint16 if bf else np.uint32
        assert np.array_equal(got.view(view), want.view(view))
    assert np.all(got[-3:-1] == 0)


def test_reader_slot_beyond_last_page(kvc, oracle_mod):
    kv = np.random.default_rng(42).integers(0, 256, size=(1, 37376), dtype=np.uint8)
    slots = np.array([5, 64, 70, 2], np.int64)        # 64 and 70 are past page 0
    got, e = _read(kvc, kv, slots, torch.float32)
    want, st = oracle_mod.dequantize(kv, slots)
    assert e == 4 and st == 4
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
    assert np.all(got[1:3] == 0)


@pytest.mark.parametrize("M", [2433, 20011, 120000])
def test_reader_large_calls_exact_on_random_bytes(kvc, oracle_mod, M):
    # beyond a device-full of slot pairs the reader switches to its
    # warp-per-slot persistent kernel; every byte pattern, slot order,
    # negative slot, ragged tail and out-of-range slot must read back as the
    # oracle's reader reads it
    rng = np.random.default_rng(43 + M)
    pages = 64
    kv = rng.integers(0, 256, size=(pages, 37376), dtype=np.uint8)
    slots = rng.integers(0, pages * 64, size=M).astype(np.int64)
    slots[rng.choice(M, size=M // 50, replace=False)] = -1
    for dtype, bf in ((torch.float32, False), (torch.bfloat16, True)):
        got, e = _read(kvc, kv, slots, dtype)
        want, st = oracle_mod.dequantize(kv, slots, out_bf16=bf)
        assert e == 0 and st == 0
        view = np.uint16 if bf else np.uint32
        assert np.array_equal(got.view(view), want.view(view))
    bad = slots.copy()
    bad[M // 2] = pages * 64 + 5           # past the last page
    got, e = _read(kvc, kv, bad, torch.float32)
    want, st = oracle_mod.dequantize(kv, bad)
    assert e == 4 and st == 4
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


@pytest.mark.parametrize("M", [20011, 120000])
def test_reader_large_bf16_into_8_byte_aligned_output(kvc, oracle_mod, M):
    # bf16 output needs only 8-byte alignment: a 16-byte-aligned output takes
    # the 8-dims-per-lane kernel (the test above), an output 8 bytes off a
    # 16-byte boundary the 4-dims-per-lane one; both must read back the
    # oracle's bits
    rng = np.random.default_rng(47 + M)
    pages = 64
    kv = rng.integers(0, 256, size=(pages, 37376), dtype=np.uint8)
    slots = rng.integers(0, pages * 64, size=M).astype(np.int64)
    slots[rng.choice(M, size=M // 50, replace=False)] = -1
    buf = torch.full((M * 512 + 4,), float("nan"), dtype=torch.bfloat16, device="cuda")
    out = buf[4:].view(M, 512)
    assert out.data_ptr() % 16 == 8
    kvc.dequantize(torch.from_numpy(kv).cuda(), torch.from_numpy(slots).cuda(),
                   dtype=torch.bfloat16, out=out)
    assert kvc.kvc_get_device_error(torch.cuda.current_stream().cuda_stream) == 0
    want, st = oracle_mod.dequantize(kv, slots, out_bf16=True)
    assert st == 0
    got = out.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(got, want.view(np.uint16))
    assert torch.isnan(buf[:4]).all()
