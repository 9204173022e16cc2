"""GPU: the compressor inside CUDA graphs and on concurrent streams.

A serving loop captures its decode step once and replays it.  These tests
capture kvc_compress (every route), kvc_compress_strided and
kvc_compress_layers in torch CUDA graphs, replay them on new inputs written
into the captured buffers, and hold each replay to the three-way parity bar
against the oracle.  Two calls on two streams with separate workspaces run
concurrently and both meet the bar.
"""
import numpy as np
import pytest
import torch

from kv_cache_compression_c128_gb300 import inputs
from kvc_testlib import assert_parity, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvc():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import kv_cache_compression_c128_gb300 as kvc

    kvc.build()
    return kvc


def _bits(case):
    return torch.from_numpy(case.state_bits.view(np.int16)).view(torch.bfloat16)


@pytest.mark.parametrize("route,count,S", [("auto", 0, 0), ("cluster", 0, 4), ("streamk", 0, 0)])
def test_captured_call_replays_on_new_inputs(kvc, oracle_mod, route, count, S):
    # two cases of the same shape: capture on the first, replay on the second
    a = inputs.make_case(2, 4096, 128, seed=inputs.BASE_SEED + 950, kv_fill=96)
    b = inputs.make_case(2, 4096, 128, seed=inputs.BASE_SEED + 951, kv_fill=97)
    for name in ("token_to_req", "positions", "boundary_token_indices", "cos_sin_cache"):
        assert np.array_equal(getattr(a, name), getattr(b, name))   # same shape of call
    d = to_device(a)
    N = a.num_outputs
    y = torch.full((N, 512), float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.zeros(kvc.kvc_workspace_bytes(N), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.Stream()
    flags = kvc.make_flags(route, count, S)
    with torch.cuda.stream(stream):
        kvc.c128_256_512_compress(block_size=8, compress_ratio=128, y_out=y, flags=flags,
                                  stream=stream, workspace=ws, **d)   # set-up outside capture
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            kvc.c128_256_512_compress(block_size=8, compress_ratio=128, y_out=y, flags=flags,
                                      stream=stream, workspace=ws, **d)
    for case in (b, a, b):
        d["state_cache"].copy_(_bits(case))
        d["block_table"].copy_(torch.from_numpy(case.block_table))
        d["rms_norm_weight"].copy_(torch.from_numpy(case.rms_norm_weight))
        d["kv_slot_mapping"].copy_(torch.from_numpy(case.kv_slot_mapping))
        d["kv_cache"].copy_(torch.from_numpy(case.kv_cache))
        with torch.cuda.stream(stream):
            g.replay()
        stream.synchronize()
        assert kvc.kvc_get_device_error(stream.cuda_stream) == 0
        assert_parity(oracle_mod, case, d["kv_cache"].cpu().numpy(), y.cpu().numpy())


def test_captured_strided_and_layers_calls(kvc, oracle_mod):
    case = inputs.make_case(2, 2048, 64, seed=inputs.BASE_SEED + 952, kv_fill=98)
    d = to_device(case)
    N = case.num_outputs
    # fp32 state, column-major block table
    st32 = d["state_cache"].float()
    R, M = case.block_table.shape
    bt_cm = torch.from_numpy(np.ascontiguousarray(case.block_table.T)).cuda().t()
    y = torch.zeros((N, 512), dtype=torch.float32, device="cuda")
    # two layers: the same state twice, separate kv caches
    kv2 = [d["kv_cache"].clone(), d["kv_cache"].clone()]
    y2 = torch.zeros((2 * N, 512), dtype=torch.float32, device="cuda")
    ws = torch.zeros(kvc.kvc_workspace_bytes(N), dtype=torch.uint8, device="cuda")
    ws2 = torch.zeros(kvc.kvc_workspace_bytes(N), dtype=torch.uint8, device="cuda")
    base = {k: v for k, v in d.items() if k not in ("state_cache", "block_table")}
    stream = torch.cuda.Stream()

    def step():
        kvc.c128_256_512_compress(st32, block_table=bt_cm, block_size=8, compress_ratio=64,
                                  y_out=y, stream=stream, workspace=ws, **base)
        kvc.compress_layers([d["state_cache"], d["state_cache"]], d["token_to_req"],
                            d["positions"], d["boundary_token_indices"], d["block_table"],
                            [d["rms_norm_weight"]] * 2, d["cos_sin_cache"],
                            d["kv_slot_mapping"], kv2, 8, 64, y_out=y2, stream=stream,
                            workspace=ws2)

    with torch.cuda.stream(stream):
        step()
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            step()
        for t in [base["kv_cache"]] + kv2:
            t.copy_(torch.from_numpy(case.kv_cache))
        g.replay()
    stream.synchronize()
    assert kvc.kvc_get_device_error(stream.cuda_stream) == 0
    for kv_t, y_t in ((base["kv_cache"], y), (kv2[0], y2[:N]), (kv2[1], y2[N:])):
        assert_parity(oracle_mod, case, kv_t.cpu().numpy(), y_t.cpu().numpy())


def test_two_streams_run_concurrently(kvc, oracle_mod):
    cases = [inputs.make_case(4, 16384, 128, seed=inputs.BASE_SEED + 953 + i, kv_fill=99 + i)
             for i in range(2)]
    ds = [to_device(c) for c in cases]
    ys = [torch.zeros((c.num_outputs, 512), dtype=torch.float32, device="cuda") for c in cases]
    wss = [torch.zeros(kvc.kvc_workspace_bytes(c.num_outputs), dtype=torch.uint8, device="cuda")
           for c in cases]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    torch.cuda.synchronize()
    for _ in range(3):
        for c, d, y, ws, s in zip(cases, ds, ys, wss, streams):
            d["kv_cache"].copy_(torch.from_numpy(c.kv_cache))
        torch.cuda.synchronize()
        for c, d, y, ws, s in zip(cases, ds, ys, wss, streams):
            kvc.c128_256_512_compress(block_size=8, compress_ratio=128, y_out=y, stream=s,
                                      workspace=ws, **d)
        torch.cuda.synchronize()
        assert kvc.kvc_get_device_error(0) == 0
        for c, d, y in zip(cases, ds, ys):
            assert_parity(oracle_mod, c, d["kv_cache"].cpu().numpy(), y.cpu().numpy())
