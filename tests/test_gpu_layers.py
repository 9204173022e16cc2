"""GPU parity of the multi-layer entry point (kvc_compress_layers).

L layers share every index array (boundary tokens, windows, block table,
slots, cos/sin) and each has its own state cache, RMSNorm weight and
kv_cache.  Each layer's result must meet the same three-way bar against the
oracle run on that layer's inputs, on every route; one layer reproduces
kvc_compress bit for bit.
"""
import copy

import numpy as np
import pytest
import torch

from kv_cache_compression_c128_gb300 import inputs
from kvc_testlib import assert_parity, run_gpu, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvc():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import kv_cache_compression_c128_gb300 as kvc

    kvc.build()
    return kvc


def _layer_cases(base, L, seed):
    """L copies of `base` with their own state, weights and kv prefill."""
    rng = np.random.default_rng(seed)
    out = []
    for l in range(L):
        c = copy.copy(base)
        st = rng.standard_normal(base.state_bits.shape, dtype=np.float32)
        c.state_bits = inputs._bf16_bits_from_f32(st).reshape(base.state_bits.shape)
        c.rms_norm_weight = (1.0 + 0.1 * rng.standard_normal(512)).astype(np.float32)
        c.kv_cache = rng.integers(0, 256, size=base.kv_cache.shape, dtype=np.uint8)
        out.append(c)
    return out


def _run_layers(kvc, cases, flags=0):
    d = to_device(cases[0])
    states = [torch.from_numpy(c.state_bits.view(np.int16)).view(torch.bfloat16).cuda()
              for c in cases]
    weights = [torch.from_numpy(c.rms_norm_weight).cuda() for c in cases]
    kvs = [torch.from_numpy(c.kv_cache.copy()).cuda() for c in cases]
    L, N = len(cases), cases[0].num_outputs
    y = torch.full((L * N, 512), float("nan"), dtype=torch.float32, device="cuda")
    kvc.compress_layers(states, d["token_to_req"], d["positions"], d["boundary_token_indices"],
                        d["block_table"], weights, d["cos_sin_cache"], d["kv_slot_mapping"], kvs,
                        cases[0].block_size, cases[0].compress_ratio, cases[0].rms_norm_eps,
                        y_out=y, flags=flags)
    err = kvc.kvc_get_device_error(torch.cuda.current_stream().cuda_stream)
    return [k.cpu().numpy() for k in kvs], y.cpu().numpy().reshape(L, N, 512), err


ROUTES = [("auto", 0, 0), ("cluster", 0, 1), ("cluster", 0, 2), ("cluster", 0, 8),
          ("cluster", 3, 4), ("streamk", 0, 0)]


@pytest.mark.parametrize("route,count,S", ROUTES)
def test_layers_each_layer_meets_the_bar(kvc, oracle_mod, route, count, S):
    base = inputs.make_case(2, 4096, 128, seed=inputs.BASE_SEED + 800, kv_fill=3)
    cases = _layer_cases(base, 4, seed=801)
    kvs, ys, err = _run_layers(kvc, cases, flags=kvc.make_flags(route, count, S))
    assert err == 0
    for l, c in enumerate(cases):
        assert_parity(oracle_mod, c, kvs[l], ys[l])


def test_layers_general_windows(kvc, oracle_mod):
    base = inputs.make_case(2, 2048, 100, seed=inputs.BASE_SEED + 802, block_size=16,
                            boundaries_per_req=24, kv_fill=4)
    cases = _layer_cases(base, 3, seed=803)
    kvs, ys, err = _run_layers(kvc, cases)
    assert err == 0
    for l, c in enumerate(cases):
        assert_parity(oracle_mod, c, kvs[l], ys[l])


def test_one_layer_is_kvc_compress(kvc):
    case = inputs.make_case(4, 32768, 256, seed=inputs.BASE_SEED + 804, kv_fill=5)
    kv1, y1, e1 = run_gpu(case)
    kvs, ys, e2 = _run_layers(kvc, [case])
    assert e1 == 0 and e2 == 0
    assert np.array_equal(kvs[0], kv1)
    assert np.array_equal(ys[0].view(np.uint32), y1.view(np.uint32))


def test_sixty_four_layers(kvc, oracle_mod):
    base = inputs.make_case(1, 512, 64, seed=inputs.BASE_SEED + 805, kv_fill=6)
    cases = _layer_cases(base, 64, seed=806)
    kvs, ys, err = _run_layers(kvc, cases)
    assert err == 0
    for l in (0, 17, 63):
        assert_parity(oracle_mod, cases[l], kvs[l], ys[l])


@pytest.mark.parametrize("f32,row_pad,block_pad,table,L", [
    (True, 0, 0, "col", 3), (False, 64, 256, "pad", 3), (True, 32, 8, "row", 3),
    (False, 64, 0, "row", 8),    # rows apart: the most layers that get tensor maps
    (False, 64, 0, "row", 9),    # one more: every layer goes row by row
])
def test_strided_layers_match_the_oracle(kvc, oracle_mod, f32, row_pad, block_pad, table, L):
    # kvc_compress_layers_strided: every layer's state in the same strided
    # layout (NaN between the rows), one strided block table
    from test_gpu_strided import Layout

    case = inputs.make_case(2, 4096, 48, seed=inputs.BASE_SEED + 1200 + row_pad, block_size=16,
                            boundaries_per_req=40, kv_fill=71)
    lays = []
    for l in range(L):
        st = inputs.fp32_state(case.num_state_blocks, 16, 72 + l) if f32 else \
            inputs.make_case(2, 4096, 48, seed=inputs.BASE_SEED + 1300 + l, block_size=16,
                             boundaries_per_req=40).state_bits
        lays.append(Layout(case, st, row_pad, block_pad, table))
    devs = [lay.device() for lay in lays]
    states = [dv[0] for dv in devs]
    tab = devs[0][1]
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    weights = [t(case.rms_norm_weight * (1.0 + 0.1 * l)).float() for l in range(L)]
    kvs = [t(case.kv_cache) for _ in range(L)]
    N = case.num_outputs
    y = torch.zeros((L * N, 512), dtype=torch.float32, device="cuda")
    kvc.compress_layers(states, t(case.token_to_req), t(case.positions),
                        t(case.boundary_token_indices), tab, weights, t(case.cos_sin_cache),
                        t(case.kv_slot_mapping), kvs, 16, 48, y_out=y)
    assert kvc.kvc_get_device_error(torch.cuda.current_stream().cuda_stream) == 0
    for l in range(L):
        lc = inputs.make_case(2, 4096, 48, seed=inputs.BASE_SEED + 1200 + row_pad, block_size=16,
                              boundaries_per_req=40, kv_fill=71)
        lc.rms_norm_weight = weights[l].cpu().numpy()
        ref = lays[l].oracle(oracle_mod, lc)
        assert ref[1]["status"] == 0
        assert_parity(oracle_mod, lc, kvs[l].cpu().numpy(), y[l * N:(l + 1) * N].cpu().numpy(),
                      ref=ref)
