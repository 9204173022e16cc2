"""GPU: byte offsets beyond 2^31, and extreme window lengths and output counts.

A small case is laid out inside large tensors: its physical blocks are placed
at block ids above 131072 of a 4.6 GiB bf16 state (and of a 9.2 GiB fp32
one), so every state byte offset exceeds 2^31, and its slots are moved to
slot ids around 4 million of a 2.4 GB kv_cache.  Renumbering blocks and
slots changes no arithmetic, so the results must equal, bit for bit, those
of the same call on the compact case, which itself meets the parity bar.

The extremes: windows of 8192 and 16384 rows (1024 and 2048 chunks, up to
clusters of 16), and 32768 one-row windows (128 outputs per CTA, the
per-output record ring wrapping many times).
"""
import numpy as np
import pytest
import torch

from kv_cache_compression_c128_gb300 import inputs
from kvc_testlib import assert_parity, run_gpu, to_device

pytestmark = pytest.mark.gpu

W = 1024
BIG_BLOCKS = 300_000            # bf16: 300000 * 16 KiB = 4.6 GiB
SLOT_BASE = 4_000_000           # page 62500: byte offset 2.34e9


@pytest.fixture(scope="module")
def kvc():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import kv_cache_compression_c128_gb300 as kvc

    kvc.build()
    return kvc


@pytest.mark.parametrize("f32", [False, True])
def test_offsets_beyond_2_pow_31(kvc, oracle_mod, f32):
    case = inputs.make_case(2, 2048, 128, seed=inputs.BASE_SEED + 5000, kv_fill=61)
    G = case.num_state_blocks
    d = to_device(case)
    state_small = d["state_cache"].float() if f32 else d["state_cache"]
    # compact reference run
    N = case.num_outputs
    y_ref = torch.zeros((N, 512), dtype=torch.float32, device="cuda")
    kv_ref = d["kv_cache"].clone()
    kvc.c128_256_512_compress(state_small, d["token_to_req"], d["positions"],
                              d["boundary_token_indices"], d["block_table"],
                              d["rms_norm_weight"], d["cos_sin_cache"], d["kv_slot_mapping"],
                              kv_ref, 8, 128, y_out=y_ref)
    assert kvc.kvc_get_device_error(torch.cuda.current_stream().cuda_stream) == 0
    assert_parity(oracle_mod, case, kv_ref.cpu().numpy(), y_ref.cpu().numpy())

    # the same blocks at ids >= 150000 of a large state
    new_id = 150_000 + np.arange(G, dtype=np.int64) * 499
    assert new_id.max() < BIG_BLOCKS
    big = torch.empty((BIG_BLOCKS, 8, W), dtype=state_small.dtype, device="cuda")
    big[torch.from_numpy(new_id).cuda()] = state_small
    table = torch.from_numpy(new_id[case.block_table].astype(np.int32)).cuda()
    # the same slots moved to ids around 4 million of a large kv_cache
    slots = case.kv_slot_mapping.copy()
    sel = slots >= 0
    slots[sel] += SLOT_BASE
    pages = (int(slots.max()) // 64) + 1
    kv_big = torch.zeros((pages, 64 * (576 + 8)), dtype=torch.uint8, device="cuda")
    base_page = SLOT_BASE // 64
    kv_big[base_page:base_page + kv_ref.shape[0]] = torch.from_numpy(case.kv_cache).cuda()
    y = torch.zeros((N, 512), dtype=torch.float32, device="cuda")
    kvc.c128_256_512_compress(big, d["token_to_req"], d["positions"], d["boundary_token_indices"],
                              table, d["rms_norm_weight"], d["cos_sin_cache"],
                              torch.from_numpy(slots).cuda(), kv_big, 8, 128, y_out=y)
    assert kvc.kvc_get_device_error(torch.cuda.current_stream().cuda_stream) == 0
    assert torch.equal(y, y_ref)
    assert torch.equal(kv_big[base_page:base_page + kv_ref.shape[0]], kv_ref)
    assert int(kv_big[:base_page].count_nonzero()) == 0
    del big, kv_big
    torch.cuda.empty_cache()


@pytest.mark.parametrize("R,T,C,route", [
    (2, 16384, 8192, "auto"),          # 1024 chunks per window
    (1, 16384, 16384, "auto"),         # the whole request is one window
    (2, 16384, 8192, "s16"),
    (4, 32768, 1, "auto"),             # 32768 outputs of one row each
    (4, 32768, 1, "streamk"),
])
def test_extreme_window_lengths_and_output_counts(kvc, oracle_mod, R, T, C, route):
    case = inputs.make_case(R, T, C, seed=inputs.BASE_SEED + 5100 + C, kv_fill=62)
    if route == "streamk":
        if C % 8:
            # one-row windows are not block-aligned: the stream-K route refuses them
            with pytest.raises(kvc.KvcError):
                run_gpu(case, kvc.make_flags("streamk"))
            return
        flags = kvc.make_flags("streamk")
    elif route.startswith("s"):
        flags = kvc.make_flags("cluster", 0, int(route[1:]))
    else:
        flags = 0
    kv_g, y_g, err = run_gpu(case, flags)
    assert err == 0
    assert_parity(oracle_mod, case, kv_g, y_g)
