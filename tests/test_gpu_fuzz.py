"""GPU parity on seeded random configurations.

Each seed draws one call at random:

- 1–4 requests, block_size in {8, 16, 24, 32, 64}, compress_ratio from 1 to
  600, windows at random starts;
- slots given per token or per output, a few of them -1 (skipped);
- a bf16 or fp32 state, adjacent or padded rows and blocks, a row-major or
  column-major block table; rows apart copied through tensor maps or row by
  row;
- an automatic or forced cluster size, or the stream-K route where it
  applies.

Every call is held to the three-way bar against the oracle's strided
compress on the same arrays.  The seeds are fixed, so a failure is
reproducible.
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


def _draw(seed, block_sizes=(8, 16, 24, 32, 64)):
    rng = np.random.Generator(np.random.PCG64(seed))
    R = int(rng.integers(1, 5))
    B = int(rng.choice(list(block_sizes)))
    C = int(rng.choice([1, 2, 7, 8, 13, 16, 31, 64, 100, 128, 256, 300, 512, 600]))
    per_req = max(C, B)
    lengths = [B * int(np.ceil((per_req + int(rng.integers(0, 4 * B + 200))) / B)) for _ in range(R)]
    T = int(sum(lengths))
    nb = int(rng.integers(1, 40))
    case = inputs.make_case(R, T, C, seed=seed, block_size=B, lengths=lengths,
                            boundaries_per_req=nb, kv_fill=int(rng.integers(0, 1000)))
    case.rms_norm_eps = float(rng.choice([1e-6, 1e-5, 0.0]))
    per_output = bool(rng.integers(0, 2))
    slots = case.kv_slot_mapping[case.boundary_token_indices].copy() if per_output else \
        case.kv_slot_mapping.copy()
    if case.num_outputs > 2:
        drop = rng.choice(case.num_outputs, size=max(1, case.num_outputs // 10), replace=False)
        if per_output:
            slots[drop] = -1
        else:
            slots[case.boundary_token_indices[drop]] = -1
    f32 = bool(rng.integers(0, 2))
    row_pad = int(rng.choice([0, 0, 64, 128])) // (2 if f32 else 1)  # elements; rows stay 16 B aligned
    block_pad = int(rng.choice([0, 0, 8, 256]))
    table = str(rng.choice(["row", "col", "pad"]))
    K = -(-C // 8)
    routes = ["auto"] + [f"s{S}" for S in (1, 2, 4, 8, 16) if S <= K]
    aligned_sk = (B == 8 and C % 8 == 0 and not f32 and row_pad == 0
                  and np.all((case.positions[case.boundary_token_indices] - C + 1) % 8 == 0))
    if aligned_sk:
        routes.append("streamk")
    route = str(rng.choice(routes))
    count = int(rng.choice([0, 0, 1, 3, 17]))
    row_copies = bool(rng.integers(0, 2)) if row_pad else False
    return case, slots, f32, row_pad, block_pad, table, route, count, row_copies


@pytest.mark.parametrize("seed", range(4000, 4200))
def test_random_configuration(kvc, oracle_mod, seed):
    _check_draw(kvc, oracle_mod, seed, _draw(seed))


@pytest.mark.parametrize("seed", range(5000, 5060))
def test_random_configuration_blocks_not_multiple_of_8(kvc, oracle_mod, seed):
    # block sizes that are not a multiple of 8: most chunks straddle two
    # blocks, with rows apart copied row by row around the tensor copies
    _check_draw(kvc, oracle_mod, seed, _draw(seed, (9, 12, 20, 40, 100)))


def _check_draw(kvc, oracle_mod, seed, draw):
    case, slots, f32, row_pad, block_pad, table, route, count, row_copies = draw
    state = inputs.fp32_state(case.num_state_blocks, case.block_size, seed + 1) if f32 \
        else case.state_bits
    G, B, _ = state.shape
    rs = W + row_pad
    bs = B * rs + block_pad
    flat = inputs.embed_strided(state, bs, rs)
    R, M = case.block_table.shape
    bt_rs, bt_cs = {"row": (M, 1), "col": (1, R), "pad": (M + 3, 1)}[table]
    tab = inputs.strided_table(case.block_table, bt_rs, bt_cs)

    # oracle on the same layout
    kv_o = case.kv_cache.copy()
    res = oracle_mod.compress_strided(flat, bs, rs, G, case.token_to_req, case.positions,
                                      case.boundary_token_indices, tab, R, M, bt_rs, bt_cs,
                                      case.rms_norm_weight, case.cos_sin_cache, slots, kv_o,
                                      B, case.compress_ratio, case.rms_norm_eps)
    assert res["status"] == 0

    dev = torch.device("cuda")
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    st = (t(flat) if f32 else t(flat.view(np.int16)).view(torch.bfloat16)).as_strided(
        (G, B, W), (bs, rs, 1))
    bt = t(tab).as_strided((R, M), (bt_rs, bt_cs))
    kv = t(case.kv_cache)
    N = case.num_outputs
    y = torch.full((max(N, 1), 512), float("nan"), dtype=torch.float32, device=dev)
    if route == "auto":
        flags = kvc.make_flags("auto", count)
    elif route == "streamk":
        flags = kvc.make_flags("streamk", count)
    else:
        flags = kvc.make_flags("cluster", count, int(route[1:]))
    if row_copies:
        flags |= kvc.KVC_FLAG_ROW_COPIES
    kvc.c128_256_512_compress(st, t(case.token_to_req), t(case.positions),
                              t(case.boundary_token_indices), bt, t(case.rms_norm_weight),
                              t(case.cos_sin_cache), t(slots), kv, B, case.compress_ratio,
                              case.rms_norm_eps, y_out=y, flags=flags)
    assert kvc.kvc_get_device_error(torch.cuda.current_stream().cuda_stream) == 0
    kv_g, y_g = kv.cpu().numpy(), y[:N].cpu().numpy()
    # the bar, with this call's slots (as a per-token mapping) in place of the case's
    if len(slots) == len(case.kv_slot_mapping):
        case.kv_slot_mapping = slots
    else:
        per_token = np.full_like(case.kv_slot_mapping, -1)
        per_token[case.boundary_token_indices] = slots
        case.kv_slot_mapping = per_token
    assert_parity(oracle_mod, case, kv_g, y_g, ref=(kv_o, res))
