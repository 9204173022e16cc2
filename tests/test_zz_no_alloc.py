"""kvc_compress_static: the entry point for callers that cannot allocate.

Plugins handed only input/output pointers, engines that own the whole device
memory pool, and latency-critical paths that cannot pay cudaMalloc's implicit
synchronisation cannot supply the workspace kvc_compress asks for.  The
static entry point uses the library's own 8 MiB scratch buffer instead.  These
tests call it through the C ABI and check it against kvc_compress (with a
caller workspace) on the same inputs, on two calls in a row, within the
tolerances the parity tests use; and check that oversized problems are
refused and that repeated calls take no device memory.

This file sorts last so that, in a run that stops at the first failure,
every other test has already run.
"""
import numpy as np
import pytest
import torch

from kv_cache_compression_c128_gb300 import inputs
from kvc_testlib import to_device

pytestmark = pytest.mark.gpu

Y_RTOL = 2e-3
Y_ATOL_RMS = 1e-5


@pytest.fixture(scope="module")
def kvc():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import kv_cache_compression_c128_gb300 as kvc

    kvc.build()
    return kvc


def _raw_args(d, case, y, stream):
    """Positional arguments shared by the two entry points (raw pointers)."""
    return [d["state_cache"].data_ptr(), d["state_cache"].shape[0],
            d["token_to_req"].data_ptr(), d["positions"].data_ptr(), d["positions"].numel(),
            d["boundary_token_indices"].data_ptr(), case.num_outputs,
            d["block_table"].data_ptr(), d["block_table"].shape[0], d["block_table"].shape[1],
            d["rms_norm_weight"].data_ptr(), d["cos_sin_cache"].data_ptr(),
            d["cos_sin_cache"].shape[0], d["kv_slot_mapping"].data_ptr(),
            d["kv_slot_mapping"].numel(), d["kv_cache"].data_ptr(), d["kv_cache"].shape[0],
            case.block_size, case.compress_ratio, case.rms_norm_eps, y.data_ptr()]


@pytest.mark.parametrize("R,T,C,route", [(2, 4096, 128, "streamk"), (1, 8192, 512, "streamk"),
                                         (8, 131072, 128, "streamk"), (2, 4096, 128, "auto")])
def test_static_entry_matches_workspace_entry_on_two_calls(kvc, R, T, C, route):
    # the stream-K route splits outputs between CTAs, so the scratch (partial
    # states + arrival counters) is used
    case = inputs.make_case(R, T, C, seed=inputs.BASE_SEED + 4242 + C, kv_fill=5)
    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream
    d = to_device(case)
    N = case.num_outputs

    ws = torch.zeros(kvc.kvc_workspace_bytes(N), dtype=torch.uint8, device="cuda")
    y_ref = torch.empty((N, 512), dtype=torch.float32, device="cuda")
    flags = kvc.make_flags(route)
    st = kvc.kvc_compress(*_raw_args(d, case, y_ref, sp), ws.data_ptr(), ws.numel(), flags, sp)
    assert st == kvc.KVC_OK
    assert kvc.kvc_get_device_error(sp) == 0
    kv_ref = d["kv_cache"].cpu().numpy()
    y_ref = y_ref.cpu().numpy()
    rms = np.sqrt((y_ref.astype(np.float64) ** 2).mean(1, keepdims=True))

    for call in range(2):
        d["kv_cache"].copy_(torch.from_numpy(case.kv_cache))
        y = torch.full((N, 512), float("nan"), dtype=torch.float32, device="cuda")
        st = kvc.kvc_compress_static(*_raw_args(d, case, y, sp), flags, sp)
        assert st == kvc.KVC_OK, f"call {call}: {kvc.kvc_error_string(st)}"
        assert kvc.kvc_get_device_error(sp) == 0
        y_np = y.cpu().numpy()
        err = np.abs(y_np.astype(np.float64) - y_ref)
        assert np.all(err <= Y_RTOL * np.abs(y_ref) + Y_ATOL_RMS * rms), f"call {call}: y"
        assert np.array_equal(d["kv_cache"].cpu().numpy(), kv_ref), f"call {call}: kv bytes"


def _other_compute_processes():
    """PIDs of other processes holding a context on this GPU (None: unknown)."""
    import os
    import subprocess

    try:
        uuid = str(torch.cuda.get_device_properties(0).uuid)
        out = subprocess.run(["nvidia-smi", "--query-compute-apps=gpu_uuid,pid",
                              "--format=csv,noheader"], capture_output=True, text=True,
                             timeout=30).stdout
    except (OSError, subprocess.SubprocessError, AttributeError):
        return None
    pids = set()
    for line in out.splitlines():
        parts = [x.strip() for x in line.split(",")]
        if len(parts) == 2 and uuid.replace("GPU-", "") in parts[0] and parts[1].isdigit():
            pids.add(int(parts[1]))
    return pids - {os.getpid()}


def _free_bytes(reads=3):
    """Device free memory, the largest of a few readings after a sync."""
    torch.cuda.synchronize()
    return max(torch.cuda.mem_get_info()[0] for _ in range(reads))


def test_static_entry_takes_no_device_memory_per_call(kvc):
    # Free device memory is a device-wide figure: the comparison assumes that
    # this process is alone on the GPU, and is skipped when nvidia-smi shows
    # another process holding a context there.
    others = _other_compute_processes()
    if others:
        pytest.skip(f"other processes on this GPU ({sorted(others)}): free memory is not ours alone")
    case = inputs.make_case(4, 32768, 256, seed=inputs.BASE_SEED + 4343)
    sp = torch.cuda.current_stream().cuda_stream
    d = to_device(case)
    y = torch.empty((case.num_outputs, 512), dtype=torch.float32, device="cuda")
    args = _raw_args(d, case, y, sp)
    flags = kvc.make_flags("streamk")
    assert kvc.kvc_compress_static(*args, flags, sp) == kvc.KVC_OK   # first call: set-up
    free0 = _free_bytes()
    for _ in range(5):
        assert kvc.kvc_compress_static(*args, flags, sp) == kvc.KVC_OK
    free1 = _free_bytes()
    assert free1 >= free0
    assert kvc.kvc_get_device_error(sp) == 0


def test_static_entry_refuses_problems_beyond_its_buffer(kvc):
    # ten million outputs need more counters than the 8 MiB buffer holds; the
    # call returns before touching any pointer (these are placeholders)
    fake = 1 << 20
    args = [fake, 1, fake, fake, 1, fake, 10_000_000, fake, 1, 1, fake, fake, 1, fake, 1,
            fake, 1, 8, 128, 1e-6, 0, 0, 0]
    st = kvc.kvc_compress_static(*args)
    assert st == kvc.KVC_ERR_SCRATCH_LIMIT
    assert "8 MiB" in kvc.kvc_error_string(st)
