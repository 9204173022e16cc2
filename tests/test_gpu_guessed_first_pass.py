"""GPU: the guessed first pass of a call queued behind another, and its recovery.

A CTA of the cluster kernel that is resident while the previous kernel on
its stream still runs reads the index arrays before its grid dependency
wait, issues the ring's first copies from those guesses as soon as the wait
releases, and then checks every guess against the indices read after the
release.  A failed check marks the copied stages to be skipped, and the
issuer copies the right rows one ring pass later.  This only happens to a
call queued right behind another kernel, so every call here is queued back
to back with others on one stream, into buffers made before the first is
queued (a copy or fill between two calls would end the overlap), behind a
spin kernel that holds the stream until the host has queued them all.

kvc_selftest_poison_guesses makes every guess name the next physical block,
so every guessed first pass fails its check.  Checked per layout: with the
poison, the device counts rejected first passes, and every call of the
chain writes exactly the bytes (and y) of the same call made alone, which
meets the parity bar against the oracle; without it, no first pass is
rejected, since nothing changes the indices.
"""
import numpy as np
import pytest
import torch

from kv_cache_compression_c128_gb300 import inputs
from kvc_testlib import assert_parity, slot_byte_ranges, slots_of_case, to_device, written_mask

pytestmark = pytest.mark.gpu

CHAIN = 6  # calls queued back to back


@pytest.fixture(scope="module")
def kvc():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import kv_cache_compression_c128_gb300 as kvc

    kvc.build()
    yield kvc
    kvc.kvc_selftest_poison_guesses(False)


def _stream():
    return torch.cuda.current_stream().cuda_stream


HOLD_CYCLES = 20_000_000  # about 10 ms of spinning: far longer than queueing the calls takes


def _calls(kvc, case, d, n, layers=1, flags=0):
    """n calls of `case` queued back to back, each into its own copies of
    the prefilled kv_cache (one per layer) and its own y; returns
    [(kv arrays per layer, y)] after checking the device error word.  With
    n > 1 the calls wait behind a spin kernel while the host queues them, so
    that each starts inside the one before it."""
    N = case.num_outputs
    kvs = [[d["kv_cache"].clone() for _ in range(layers)] for _ in range(n)]
    ys = [torch.full((layers * N, 512), float("nan"), dtype=torch.float32, device="cuda")
          for _ in range(n)]
    torch.cuda.synchronize()
    if n > 1:
        torch.cuda._sleep(HOLD_CYCLES)
    for kv, y in zip(kvs, ys):
        if layers == 1:
            kvc.c128_256_512_compress(block_size=case.block_size,
                                      compress_ratio=case.compress_ratio,
                                      rms_norm_eps=case.rms_norm_eps, y_out=y, flags=flags,
                                      **dict(d, kv_cache=kv[0]))
        else:
            kvc.compress_layers([d["state_cache"]] * layers, d["token_to_req"], d["positions"],
                                d["boundary_token_indices"], d["block_table"],
                                [d["rms_norm_weight"]] * layers, d["cos_sin_cache"],
                                d["kv_slot_mapping"], kv, case.block_size, case.compress_ratio,
                                case.rms_norm_eps, y_out=y, flags=flags)
    assert kvc.kvc_get_device_error(_stream()) == 0
    return [([k.cpu().numpy() for k in kv], y.cpu().numpy()) for kv, y in zip(kvs, ys)]


def _check_chain(kvc, oracle_mod, case, d, layers=1, flags=0, oracle=True):
    # the call alone: nothing before it on the stream but the buffer fills
    kvc.kvc_selftest_first_pass_rejections(_stream())  # clears the count
    (kv_ref, y_ref), = _calls(kvc, case, d, 1, layers, flags)
    if oracle:
        assert_parity(oracle_mod, case, kv_ref[0], y_ref[:case.num_outputs])
    kvc.kvc_selftest_first_pass_rejections(_stream())

    # without the poison every guess holds
    for kv, y in _calls(kvc, case, d, CHAIN, layers, flags):
        assert all(np.array_equal(a, b) for a, b in zip(kv, kv_ref))
        assert np.array_equal(y.view(np.int32), y_ref.view(np.int32))
    assert kvc.kvc_selftest_first_pass_rejections(_stream()) == 0

    # with it every guessed first pass is rejected, and the results stand
    assert kvc.kvc_selftest_poison_guesses(True) == 0
    try:
        chain = _calls(kvc, case, d, CHAIN, layers, flags)
        rejected = kvc.kvc_selftest_first_pass_rejections(_stream())
    finally:
        assert kvc.kvc_selftest_poison_guesses(False) == 0
    assert rejected > 0
    for kv, y in chain:
        assert all(np.array_equal(a, b) for a, b in zip(kv, kv_ref))
        assert np.array_equal(y.view(np.int32), y_ref.view(np.int32))
    return rejected


CASES = [
    # (name, num_reqs, total_tokens, C, block_size, boundaries per request, cluster size)
    # 16 outputs on 8-CTA clusters: 128 CTAs, the next call wholly resident early
    ("r1_c512", 1, 8192, 512, 8, None, 0),
    # 64 outputs on 4-CTA clusters: the first pass is each CTA's whole window
    ("r1_c128", 1, 8192, 128, 8, None, 0),
    # 256 CTAs of one output each: 48 of the next call's CTAs resident early
    ("r4_c128", 4, 32768, 128, 8, None, 0),
    ("r4_c256_s2", 4, 32768, 256, 8, None, 2),
    # windows at any start in blocks of 16 rows: chunks split between blocks
    ("general_b16", 2, 4096, 100, 16, 24, 0),
    ("general_b24_s4", 3, 1440, 37, 24, 16, 4),
]


@pytest.mark.parametrize("name,R,T,C,B,nb,S", CASES, ids=[c[0] for c in CASES])
def test_rejected_guesses_leave_results_alone(kvc, oracle_mod, name, R, T, C, B, nb, S):
    case = inputs.make_case(R, T, C, seed=inputs.BASE_SEED + 5300 + C + B, block_size=B,
                            boundaries_per_req=nb, kv_fill=91)
    flags = kvc.make_flags("cluster", 0, S) if S else 0
    _check_chain(kvc, oracle_mod, case, to_device(case), flags=flags)


def test_rejected_guesses_on_an_fp32_state(kvc, oracle_mod):
    case = inputs.make_case(2, 8192, 128, seed=inputs.BASE_SEED + 5400, kv_fill=92)
    d = to_device(case)
    st32 = inputs.fp32_state(case.num_state_blocks, case.block_size, inputs.BASE_SEED + 5401)
    d["state_cache"] = torch.from_numpy(st32).cuda()
    # parity of the fp32 state itself is covered elsewhere; here the chain
    # must reproduce the call made alone
    _check_chain(kvc, oracle_mod, case, d, oracle=False)


def test_rejected_guesses_in_a_multi_layer_call(kvc, oracle_mod):
    case = inputs.make_case(1, 8192, 256, seed=inputs.BASE_SEED + 5500, kv_fill=93)
    _check_chain(kvc, oracle_mod, case, to_device(case), layers=4)


KVC_ERR_TIMEOUT = 5


@pytest.mark.parametrize("R,T,C,limit", [(1, 8192, 512, 500), (4, 32768, 128, 500)],
                         ids=["r1_c512", "r4_c128"])
def test_abort_after_rejected_guesses(kvc, oracle_mod, R, T, C, limit):
    # both test hooks at once: every guessed first pass fails its check and
    # the pipeline waits give up early.  The stages copied from the guesses
    # are counted as issued, so each CTA still waits for them to land before
    # it exits; every slot must end up whole or untouched.
    case = inputs.make_case(R, T, C, seed=inputs.BASE_SEED + 5600 + C, kv_fill=94)
    d = to_device(case)
    (kv_ref, y_ref), = _calls(kvc, case, d, 1)
    kv_ref, y_ref = kv_ref[0], y_ref[:case.num_outputs]
    kvc.kvc_selftest_first_pass_rejections(_stream())
    assert kvc.kvc_selftest_poison_guesses(True) == 0
    assert kvc.kvc_selftest_set_wait_limit(limit) == 0
    try:
        N = case.num_outputs
        kvs = [d["kv_cache"].clone() for _ in range(CHAIN)]
        ys = [torch.full((N, 512), float("nan"), dtype=torch.float32, device="cuda")
              for _ in range(CHAIN)]
        torch.cuda.synchronize()
        torch.cuda._sleep(HOLD_CYCLES)
        for kv, y in zip(kvs, ys):
            kvc.c128_256_512_compress(block_size=case.block_size,
                                      compress_ratio=case.compress_ratio,
                                      rms_norm_eps=case.rms_norm_eps, y_out=y,
                                      **dict(d, kv_cache=kv))
        err = kvc.kvc_get_device_error(_stream())  # synchronises: every call returned
        rejected = kvc.kvc_selftest_first_pass_rejections(_stream())
    finally:
        assert kvc.kvc_selftest_set_wait_limit(0) == 0
        assert kvc.kvc_selftest_poison_guesses(False) == 0
    assert err == KVC_ERR_TIMEOUT
    assert rejected > 0
    slots = slots_of_case(case)
    inside = written_mask(case.kv_cache.shape, slots).reshape(-1)
    pre = case.kv_cache.reshape(-1)
    ref = kv_ref.reshape(-1)
    abandoned = 0
    for kv, y in zip(kvs, ys):
        got, yg = kv.cpu().numpy().reshape(-1), y.cpu().numpy()
        assert np.array_equal(got[~inside], pre[~inside]), "bytes outside the slots changed"
        for n, s in enumerate(slots):
            if s < 0:
                continue
            p0, s0 = slot_byte_ranges(s)
            rng = np.r_[p0:p0 + 576, s0:s0 + 8]
            if np.array_equal(got[rng], ref[rng]) and not np.array_equal(ref[rng], pre[rng]):
                assert np.array_equal(yg[n].view(np.int32), y_ref[n].view(np.int32))
            else:
                assert np.array_equal(got[rng], pre[rng]), f"output {n}: slot neither whole nor untouched"
                assert np.all(np.isnan(yg[n]))
                abandoned += 1
    assert abandoned >= 1
    # hooks off: the next chain is whole again
    for kv, y in _calls(kvc, case, d, 2):
        assert np.array_equal(kv[0], kv_ref)
        assert np.array_equal(y.view(np.int32), y_ref.view(np.int32))


def _rows_apart(case, state, row_pad):
    """`state` ([G, B, 1024], bf16 bits or fp32) on the device with each row
    `row_pad` elements after the previous one's end (NaN in the gaps)."""
    G, B, W = state.shape
    rs, bs = W + row_pad, B * (W + row_pad)
    flat = inputs.embed_strided(state, bs, rs)
    if flat.dtype == np.float32:
        dev = torch.from_numpy(flat).cuda()
    else:
        dev = torch.from_numpy(flat.view(np.int16)).view(torch.bfloat16).cuda()
    return dev.as_strided((G, B, W), (bs, rs, 1))


@pytest.mark.parametrize("dtype,R,T,C,B,nb", [
    ("bf16", 2, 8192, 128, 8, None),
    ("bf16", 1, 8192, 512, 8, None),
    ("fp32", 2, 8192, 256, 8, None),
    # windows at any start in blocks of 16 rows: chunks split between two
    # blocks go row by row, the others by one tensor copy
    ("bf16", 2, 4096, 100, 16, 24),
], ids=["bf16_c128", "bf16_c512", "fp32_c256", "bf16_general_b16"])
def test_rejected_guesses_with_rows_apart(kvc, oracle_mod, dtype, R, T, C, B, nb):
    # rows 64 elements apart are copied through per-layer TMA tensor maps,
    # and the guessed first pass there issues tensor copies too
    case = inputs.make_case(R, T, C, seed=inputs.BASE_SEED + 5700 + C + B, block_size=B,
                            boundaries_per_req=nb, kv_fill=95)
    d = to_device(case)
    st = case.state_bits if dtype == "bf16" else \
        inputs.fp32_state(case.num_state_blocks, case.block_size, inputs.BASE_SEED + 5701)
    d["state_cache"] = _rows_apart(case, st, 64)
    rejected = _check_chain(kvc, oracle_mod, case, d, oracle=dtype == "bf16")
    assert rejected > 0


def test_rejected_guesses_in_a_multi_layer_call_with_rows_apart(kvc, oracle_mod):
    # 3 layers whose states share one strided view (rows 64 elements
    # apart): the per-layer tensor maps and the guessed tensor copies
    case = inputs.make_case(1, 8192, 256, seed=inputs.BASE_SEED + 5800, kv_fill=96)
    d = to_device(case)
    d["state_cache"] = _rows_apart(case, case.state_bits, 64)
    rejected = _check_chain(kvc, oracle_mod, case, d, layers=3)
    assert rejected > 0


@pytest.mark.parametrize("poison", [False, True], ids=["guesses", "poisoned"])
def test_headline_graph_replay_equals_the_call_alone(kvc, oracle_mod, poison):
    # The bench times the headline shape (8 requests x 16384 tokens, C = 128)
    # as back-to-back calls replayed from a CUDA graph, where the next
    # launch's CTAs start inside the previous one and take the guessed first
    # pass.  Every replayed call must write exactly the bytes of the call
    # made alone, which meets the parity bar.
    case = inputs.headline_case()
    d = to_device(case)
    N, n = case.num_outputs, 8
    stream = torch.cuda.Stream()
    ws = torch.zeros(kvc.kvc_workspace_bytes(N), dtype=torch.uint8, device="cuda")
    kvs = [d["kv_cache"].clone() for _ in range(n + 1)]
    ys = [torch.full((N, 512), float("nan"), dtype=torch.float32, device="cuda") for _ in range(n + 1)]

    def call(i):
        kvc.c128_256_512_compress(block_size=case.block_size, compress_ratio=case.compress_ratio,
                                  rms_norm_eps=case.rms_norm_eps, y_out=ys[i], stream=stream,
                                  workspace=ws, **dict(d, kv_cache=kvs[i]))

    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        call(n)                            # the call alone (also warms the library up)
        stream.synchronize()
        assert kvc.kvc_get_device_error(stream.cuda_stream) == 0
        kv_ref, y_ref = kvs[n].cpu().numpy(), ys[n].cpu().numpy()
        # the launch parameters, the poison setting among them, are fixed
        # when the graph is captured
        assert kvc.kvc_selftest_poison_guesses(poison) == 0
        try:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for i in range(n):
                    call(i)
        finally:
            assert kvc.kvc_selftest_poison_guesses(False) == 0
        for k, y in zip(kvs[:n], ys[:n]):  # capturing runs nothing; start from the prefill anyway
            k.copy_(d["kv_cache"])
            y.fill_(float("nan"))
        stream.synchronize()
        kvc.kvc_selftest_first_pass_rejections(stream.cuda_stream)
        g.replay()
        assert kvc.kvc_get_device_error(stream.cuda_stream) == 0
        rejected = kvc.kvc_selftest_first_pass_rejections(stream.cuda_stream)
    assert (rejected > 0) if poison else (rejected == 0)
    for k, y in zip(kvs[:n], ys[:n]):
        assert np.array_equal(k.cpu().numpy(), kv_ref)
        assert np.array_equal(y.cpu().numpy().view(np.int32), y_ref.view(np.int32))
    assert_parity(oracle_mod, case, kv_ref, y_ref)
