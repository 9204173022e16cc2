"""GPU: the compressor's own abort path, driven on real launches.

Every pipeline wait of the kernels (a copy stage landing, a stage being
freed, a hand-off between the resolver and issuer warps) is bounded.  When
one runs past its limit the kernel records KVC_ERR_TIMEOUT, stops issuing
copies, waits for the copies already in flight, still completes its side of
every exchange between the CTAs of a cluster, and returns.  The test hook
kvc_selftest_set_wait_limit shortens that limit to a few hundred or thousand
SM cycles, far less than a copy takes to land, so real calls give up part
way.  Nothing faults or hangs: the final drain of in-flight copies and the
cluster exchanges keep the default limit, so every wait in the test ends
when the data it waits for arrives.

Checked per call: the launch succeeds; the device error word reads
KVC_ERR_TIMEOUT; at least one output was abandoned; every slot is either
untouched or holds exactly the bytes an undisturbed call writes (and its y
row likewise); every byte outside the slots is untouched; and, with the
default limit restored, the next call on the same workspace meets the
parity bar against the oracle.  Cluster size 1 comes first, then the
cluster sizes whose ranks exchange partial states, then the stream-K route.
"""
import numpy as np
import pytest
import torch

from kv_cache_compression_c128_gb300 import inputs
from kvc_testlib import assert_parity, slot_byte_ranges, slots_of_case, to_device, written_mask

pytestmark = pytest.mark.gpu

KVC_ERR_TIMEOUT = 5


@pytest.fixture(scope="module")
def kvc():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import kv_cache_compression_c128_gb300 as kvc

    kvc.build()
    yield kvc
    kvc.kvc_selftest_set_wait_limit(0)


def _call(kvc, case, d, ws, flags, layers=1):
    """One compression of `case` on the device arrays `d`; returns y (NaN
    where nothing was written) after checking the launch status."""
    N = case.num_outputs
    y = torch.full((layers * N, 512), float("nan"), dtype=torch.float32, device="cuda")
    if layers == 1:
        kvc.c128_256_512_compress(block_size=case.block_size, compress_ratio=case.compress_ratio,
                                  rms_norm_eps=case.rms_norm_eps, y_out=y, flags=flags,
                                  workspace=ws, **d)
    else:
        kvc.compress_layers([d["state_cache"]] * layers, d["token_to_req"], d["positions"],
                            d["boundary_token_indices"], d["block_table"],
                            [d["rms_norm_weight"]] * layers, d["cos_sin_cache"],
                            d["kv_slot_mapping"], d["kv_layers"], case.block_size,
                            case.compress_ratio, case.rms_norm_eps, y_out=y, flags=flags,
                            workspace=ws)
    return y


def _check_abandoned_call(case, kv_prefill, kv_got, y_got, kv_ref, y_ref):
    """Every slot untouched or whole; bytes outside slots untouched; y rows
    NaN or equal to the undisturbed call's.  Returns (abandoned, written)."""
    slots = slots_of_case(case)
    m = written_mask(kv_got.shape, slots)
    flat_got, flat_pre, flat_ref = kv_got.reshape(-1), kv_prefill.reshape(-1), kv_ref.reshape(-1)
    assert np.array_equal(flat_got[~m], flat_pre[~m]), "bytes outside the slots changed"
    abandoned = written = 0
    for n, s in enumerate(slots):
        if s < 0:
            continue
        p0, s0 = slot_byte_ranges(s)
        got = np.concatenate([flat_got[p0:p0 + 576], flat_got[s0:s0 + 8]])
        pre = np.concatenate([flat_pre[p0:p0 + 576], flat_pre[s0:s0 + 8]])
        ref = np.concatenate([flat_ref[p0:p0 + 576], flat_ref[s0:s0 + 8]])
        if np.array_equal(got, ref) and not np.array_equal(ref, pre):
            written += 1
            assert np.array_equal(y_got[n], y_ref[n]), f"output {n}: slot written, y differs"
        else:
            assert np.array_equal(got, pre), f"output {n}: slot neither untouched nor whole"
            assert np.all(np.isnan(y_got[n])), f"output {n}: slot untouched, y written"
            abandoned += 1
    return abandoned, written


CASES = [
    # (name, num_reqs, total_tokens, C, route, cluster size, wait limit in SM cycles)
    ("s1", 4, 32768, 128, "cluster", 1, 200),
    ("s1_limit_2000", 4, 32768, 128, "cluster", 1, 2000),
    # a call small enough that the resolver issues the ring's first pass itself
    ("s1_small_call", 1, 8192, 128, "cluster", 1, 200),
    ("s1_small_call_limit_3000", 1, 8192, 512, "cluster", 1, 3000),
    ("s2", 4, 32768, 256, "cluster", 2, 200),
    ("s4", 4, 32768, 512, "cluster", 4, 500),
    ("s8", 1, 8192, 256, "cluster", 8, 500),
    ("s16", 1, 8192, 512, "cluster", 16, 500),
    ("streamk", 4, 32768, 128, "streamk", 0, 500),
    ("auto_headline", 8, 131072, 128, "auto", 0, 1000),
]


@pytest.mark.parametrize("name,R,T,C,route,S,limit", CASES, ids=[c[0] for c in CASES])
def test_pipeline_timeout_abandons_cleanly(kvc, oracle_mod, name, R, T, C, route, S, limit):
    case = inputs.make_case(R, T, C, seed=inputs.BASE_SEED + 5100 + C + S, kv_fill=77)
    sp = torch.cuda.current_stream().cuda_stream
    flags = kvc.make_flags(route, cluster_size=S)
    d = to_device(case)
    ws = torch.zeros(kvc.kvc_workspace_bytes(case.num_outputs), dtype=torch.uint8, device="cuda")
    assert kvc.kvc_get_device_error(sp) == 0

    # the undisturbed call: the bytes a finished output must have
    y_ref = _call(kvc, case, d, ws, flags).cpu().numpy()
    assert kvc.kvc_get_device_error(sp) == 0
    kv_ref = d["kv_cache"].cpu().numpy()

    d["kv_cache"].copy_(torch.from_numpy(case.kv_cache))
    assert kvc.kvc_selftest_set_wait_limit(limit) == 0
    try:
        y = _call(kvc, case, d, ws, flags)
        err = kvc.kvc_get_device_error(sp)      # synchronises: the kernel returned
    finally:
        assert kvc.kvc_selftest_set_wait_limit(0) == 0
    assert err == KVC_ERR_TIMEOUT
    abandoned, _ = _check_abandoned_call(case, case.kv_cache, d["kv_cache"].cpu().numpy(),
                                         y.cpu().numpy(), kv_ref, y_ref)
    assert abandoned >= 1

    # the default limit again: the next call on the same workspace is whole
    d["kv_cache"].copy_(torch.from_numpy(case.kv_cache))
    y2 = _call(kvc, case, d, ws, flags).cpu().numpy()
    assert kvc.kvc_get_device_error(sp) == 0
    kv2 = d["kv_cache"].cpu().numpy()
    assert np.array_equal(kv2, kv_ref) and np.array_equal(y2, y_ref)
    assert_parity(oracle_mod, case, kv2, y2)


def test_pipeline_timeout_in_a_multi_layer_call(kvc, oracle_mod):
    L = 3
    case = inputs.make_case(2, 8192, 256, seed=inputs.BASE_SEED + 5200, kv_fill=61)
    sp = torch.cuda.current_stream().cuda_stream
    d = to_device(case)
    d["kv_layers"] = [d["kv_cache"].clone() for _ in range(L)]
    ws = torch.zeros(kvc.kvc_workspace_bytes(case.num_outputs), dtype=torch.uint8, device="cuda")

    y_ref = _call(kvc, case, d, ws, 0, layers=L).cpu().numpy()
    assert kvc.kvc_get_device_error(sp) == 0
    kv_ref = [k.cpu().numpy() for k in d["kv_layers"]]
    for k in d["kv_layers"]:
        k.copy_(torch.from_numpy(case.kv_cache))
    assert kvc.kvc_selftest_set_wait_limit(300) == 0
    try:
        y = _call(kvc, case, d, ws, 0, layers=L)
        err = kvc.kvc_get_device_error(sp)
    finally:
        assert kvc.kvc_selftest_set_wait_limit(0) == 0
    assert err == KVC_ERR_TIMEOUT
    N = case.num_outputs
    y = y.cpu().numpy()
    total = 0
    for l in range(L):
        ab, _ = _check_abandoned_call(case, case.kv_cache, d["kv_layers"][l].cpu().numpy(),
                                      y[l * N:(l + 1) * N], kv_ref[l], y_ref[l * N:(l + 1) * N])
        total += ab
    assert total >= 1
    for k in d["kv_layers"]:
        k.copy_(torch.from_numpy(case.kv_cache))
    y2 = _call(kvc, case, d, ws, 0, layers=L).cpu().numpy()
    assert kvc.kvc_get_device_error(sp) == 0
    for l in range(L):
        kv2 = d["kv_layers"][l].cpu().numpy()
        assert np.array_equal(kv2, kv_ref[l])
        if l == 0:
            assert_parity(oracle_mod, case, kv2, y2[:N])
