"""GPU failure path: a pipeline wait that runs out reports, it does not hang.

Every wait of the kernels on a shared-memory barrier is bounded; when the
bound passes the kernel records KVC_ERR_TIMEOUT in the device error word and
returns.  kvc_selftest_wait_timeout makes one such wait run out on purpose (a
barrier nothing completes, a ~1 ms limit), with no fault and no trap.  The
test reads the status back and checks that the context is still usable: the
compressor runs and meets the parity bar right after.
"""
import pytest
import torch

from kv_cache_compression_c128_gb300 import inputs
from kvc_testlib import assert_parity, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvc():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import kv_cache_compression_c128_gb300 as kvc

    kvc.build()
    return kvc


def test_wait_timeout_is_reported_and_context_survives(kvc, oracle_mod):
    stream = torch.cuda.current_stream().cuda_stream
    assert kvc.kvc_get_device_error(stream) == 0
    for _ in range(2):
        assert kvc.kvc_selftest_wait_timeout(2_000_000, stream) == 0
        assert kvc.kvc_get_device_error(stream) == 5        # KVC_ERR_TIMEOUT
        assert kvc.kvc_get_device_error(stream) == 0        # read clears it
    case = inputs.make_case(2, 2048, 128, seed=inputs.BASE_SEED + 900, kv_fill=95)
    kv_g, y_g, err = run_gpu(case)
    assert err == 0
    assert_parity(oracle_mod, case, kv_g, y_g)
