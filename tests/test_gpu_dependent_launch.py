"""GPU: a call that reads what the call before it on the stream writes.

The cluster kernel is launched with programmatic stream serialisation: it
may start while the previous kernel on the stream is still running, and it
warms L2 with its first stages, from the index arrays as they stand, before
its grid dependency wait.  Only loads after the wait may reach a result.

Here call A writes its y output, and call B, queued right behind it on the
same stream, reads that same memory as its fp32 state.  B must produce
exactly what it produces when the host synchronises between the two calls,
and not what it produced on the buffer's earlier contents.
"""
import numpy as np
import pytest
import torch

from kv_cache_compression_c128_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvc():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import kv_cache_compression_c128_gb300 as kvc

    kvc.build()
    return kvc


def _dev(case):
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    st = t(case.state_bits.view(np.int16)).view(torch.bfloat16)
    return st, dict(token_to_req=t(case.token_to_req), positions=t(case.positions),
                    boundary_token_indices=t(case.boundary_token_indices),
                    block_table=t(case.block_table), rms_norm_weight=t(case.rms_norm_weight),
                    cos_sin_cache=t(case.cos_sin_cache), kv_slot_mapping=t(case.kv_slot_mapping),
                    kv_cache=t(case.kv_cache))


@pytest.mark.parametrize("route", ["auto", "s2"])
def test_call_reads_the_previous_calls_output(kvc, route):
    # A: 4096 outputs of 16 rows each; its y (8 MiB of fp32) is rewritten by every run
    a = inputs.make_case(2, 65536, 16, seed=inputs.BASE_SEED + 7000, kv_fill=3)
    a_state, a_args = _dev(a)
    y = torch.empty((a.num_outputs, 512), dtype=torch.float32, device="cuda")
    # B: reads the first 4 MiB of y as its fp32 state [128 blocks, 8 rows, 1024]
    b = inputs.make_case(1, 1024, 64, seed=inputs.BASE_SEED + 7001, kv_fill=4)
    G = b.num_state_blocks
    assert y.numel() >= G * 8 * 1024
    b_state = y.view(-1)[:G * 8 * 1024].view(G, 8, 1024)
    _, b_args = _dev(b)
    flags = 0 if route == "auto" else kvc.make_flags("cluster", 0, 2)

    def run_a():
        kvc.c128_256_512_compress(a_state, block_size=8, compress_ratio=16, y_out=y, **a_args)

    def run_b():
        kv = b_args["kv_cache"].clone()
        yb = torch.zeros((b.num_outputs, 512), dtype=torch.float32, device="cuda")
        kvc.c128_256_512_compress(b_state, block_size=8, compress_ratio=64, y_out=yb, flags=flags,
                                  **dict(b_args, kv_cache=kv))
        return kv, yb

    # stale contents first, read once by B so that its lines sit in the caches
    y.copy_(torch.randn_like(y))
    torch.cuda.synchronize()
    kv_stale, y_stale = run_b()
    torch.cuda.synchronize()
    # A then B back to back on one stream: B may start before A ends
    for _ in range(3):
        run_a()
        kv_chain, y_chain = run_b()
        torch.cuda.synchronize()
        assert kvc.kvc_get_device_error(torch.cuda.current_stream().cuda_stream) == 0
        # the same with the host waiting for A before B is queued
        kv_sync, y_sync = run_b()
        torch.cuda.synchronize()
        assert torch.equal(kv_chain, kv_sync)
        assert torch.equal(y_chain.view(torch.int32), y_sync.view(torch.int32))
        assert not torch.equal(y_chain, y_stale)
        y.copy_(torch.randn_like(y))  # stale again for the next round
        torch.cuda.synchronize()
        run_b()
        torch.cuda.synchronize()
