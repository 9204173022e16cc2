"""GPU: a call that reads what the call before it on the stream writes.

The cluster kernel is launched with programmatic stream serialisation: it
may start while the previous kernel on the stream is still running, and it
warms L2 with its first stages, from the index arrays as they stand, before
its grid dependency wait.  Only loads after the wait may reach a result.

In the first test call A writes its y output, and call B, queued right
behind it on the same stream, reads that same memory as its fp32 state; in
the second, B reads A's packed slots as its positions array.  B must
produce exactly what it produces when the host synchronises between the two
calls, and not what it produced on the buffer's earlier contents.  B's
outputs are allocated before A is queued, so that no other kernel or copy
sits between the two on the stream.
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

    def out_b():
        # B's outputs are made before A is queued: any kernel or copy between
        # A and B on the stream would keep B from starting inside A
        return (b_args["kv_cache"].clone(),
                torch.zeros((b.num_outputs, 512), dtype=torch.float32, device="cuda"))

    def run_b(kv, yb):
        kvc.c128_256_512_compress(b_state, block_size=8, compress_ratio=64, y_out=yb, flags=flags,
                                  **dict(b_args, kv_cache=kv))
        return kv, yb

    # stale contents first, read once by B so that its lines sit in the caches
    y.copy_(torch.randn_like(y))
    torch.cuda.synchronize()
    kv_stale, y_stale = run_b(*out_b())
    torch.cuda.synchronize()
    # A then B back to back on one stream: B may start before A ends
    for _ in range(3):
        outs = out_b()
        run_a()
        kv_chain, y_chain = run_b(*outs)
        torch.cuda.synchronize()
        assert kvc.kvc_get_device_error(torch.cuda.current_stream().cuda_stream) == 0
        # the same with the host waiting for A before B is queued
        kv_sync, y_sync = run_b(*out_b())
        torch.cuda.synchronize()
        assert torch.equal(kv_chain, kv_sync)
        assert torch.equal(y_chain.view(torch.int32), y_sync.view(torch.int32))
        assert not torch.equal(y_chain, y_stale)
        y.copy_(torch.randn_like(y))  # stale again for the next round
        torch.cuda.synchronize()
        run_b(*out_b())
        torch.cuda.synchronize()


@pytest.mark.parametrize("route", ["auto", "s2"])
def test_call_reads_its_positions_from_the_previous_calls_slots(kvc, route):
    # Before its grid dependency wait the kernel resolves its first chunks
    # from the index arrays as they stand, to warm L2; only what it loads
    # after the wait may reach a result.  Here call B's positions array IS
    # call A's kv_cache, so B's early pass can see positions A has not
    # written yet, and B must still produce what it produces after A is done.
    #
    # A: 512 windows whose values are exactly 1 in dims d = 0 mod 8 (d < 448)
    # and 0 elsewhere, unit weights.  Then c is exactly that 0/1 pattern
    # (every sum of a softmax weight times 1 equals the matching denominator
    # term), and each of A's 64-dim groups codes to q at dims 0 mod 8 and 0
    # elsewhere: every 8-byte word of a code region reads as the int64 q.
    a = inputs.make_case(8, 65536, 128, seed=inputs.BASE_SEED + 7100)
    cols = np.arange(512)
    vals = np.where((cols % 8 == 0) & (cols < 448), 0x3F80, 0).astype(np.uint16)
    a.state_bits[:, :, :512] = vals
    a.rms_norm_weight[:] = 1.0
    a_state, a_args = _dev(a)
    a_kv = a_args["kv_cache"]
    words = a_kv.view(-1).view(torch.int64)                # B's positions [pages * 4672]
    # B: windows of 16 rows in one request of 16 blocks, at the positions held
    # by 256 code words of A's slots (word m of slot s: page*4672 + off*72 + m)
    rng = np.random.Generator(np.random.PCG64(inputs.BASE_SEED + 7101))
    slots = rng.choice(a.num_outputs, size=256, replace=True)
    m = rng.integers(0, 56, size=256)
    bti = np.unique((slots // 64) * 4672 + (slots % 64) * 72 + m)
    n_b = bti.size
    t_b = words.numel()
    b_state = torch.from_numpy(
        inputs.make_case(1, 128, 16, seed=inputs.BASE_SEED + 7102).state_bits.view(np.int16)
    ).view(torch.bfloat16).cuda()
    t = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()
    b_args = dict(token_to_req=torch.zeros(t_b, dtype=torch.int32, device="cuda"),
                  positions=words, boundary_token_indices=t(bti.astype(np.int64)),
                  block_table=t(rng.permutation(16).astype(np.int32)[None, :]),
                  rms_norm_weight=t(a.rms_norm_weight), cos_sin_cache=t(inputs._cos_sin_table(128)),
                  kv_slot_mapping=t(rng.permutation(n_b).astype(np.int64)))
    flags = 0 if route == "auto" else kvc.make_flags("cluster", 0, 2)
    stream = torch.cuda.current_stream().cuda_stream

    def run_a():
        kvc.c128_256_512_compress(a_state, block_size=8, compress_ratio=128, **a_args)

    def out_b():  # made before A is queued, so that B directly follows A
        return (torch.zeros((4, inputs.KV_PAGE_BYTES), dtype=torch.uint8, device="cuda"),
                torch.zeros((n_b, 512), dtype=torch.float32, device="cuda"))

    def run_b(kv, yb):
        kvc.c128_256_512_compress(b_state, block_size=8, compress_ratio=16, y_out=yb,
                                  flags=flags, kv_cache=kv, **b_args)
        return kv, yb

    run_a()
    torch.cuda.synchronize()
    q = words[torch.from_numpy(bti).cuda()]
    assert int(q.min()) >= 63 and int(q.max()) <= 127, "A's code words"
    kv_sync, y_sync = run_b(*out_b())
    torch.cuda.synchronize()
    assert kvc.kvc_get_device_error(stream) == 0
    for _ in range(3):
        words.fill_(40)                                    # another valid position
        kv_stale, _ = run_b(*out_b())                      # B on the stale positions
        torch.cuda.synchronize()
        assert not torch.equal(kv_stale, kv_sync)
        outs = out_b()
        run_a()
        kv_chain, y_chain = run_b(*outs)                   # queued right behind A
        torch.cuda.synchronize()
        assert kvc.kvc_get_device_error(stream) == 0
        assert torch.equal(kv_chain, kv_sync)
        assert torch.equal(y_chain.view(torch.int32), y_sync.view(torch.int32))


def _coded_case_a(kvc):
    """Call A of the index tests: 512 windows whose c is a 0/1 pattern (ones at
    dims 0 mod 8 below 448), so every 8-byte word of a slot's code region, and
    every other 4-byte word, reads back as the same code q (checked)."""
    a = inputs.make_case(8, 65536, 128, seed=inputs.BASE_SEED + 7100)
    cols = np.arange(512)
    a.state_bits[:, :, :512] = np.where((cols % 8 == 0) & (cols < 448), 0x3F80, 0).astype(np.uint16)
    a.rms_norm_weight[:] = 1.0
    a_state, a_args = _dev(a)

    def run_a():
        kvc.c128_256_512_compress(a_state, block_size=8, compress_ratio=128, **a_args)

    return a, a_args["kv_cache"], run_a


def _chain_b_against_sync(kvc, run_a, run_b, out_b, index_buf, stale_value):
    """A then B back to back must equal B after a host sync, and differ from
    B on stale index contents (index_buf filled with stale_value)."""
    stream = torch.cuda.current_stream().cuda_stream
    run_a()
    torch.cuda.synchronize()
    kv_sync, y_sync = run_b(*out_b())
    torch.cuda.synchronize()
    assert kvc.kvc_get_device_error(stream) == 0
    for _ in range(3):
        index_buf.fill_(stale_value)
        kv_stale, _ = run_b(*out_b())
        torch.cuda.synchronize()
        assert kvc.kvc_get_device_error(stream) == 0
        assert not torch.equal(kv_stale, kv_sync)
        outs = out_b()
        run_a()
        kv_chain, y_chain = run_b(*outs)                   # queued right behind A
        torch.cuda.synchronize()
        assert kvc.kvc_get_device_error(stream) == 0
        assert torch.equal(kv_chain, kv_sync)
        assert torch.equal(y_chain.view(torch.int32), y_sync.view(torch.int32))


@pytest.mark.parametrize("route", ["auto", "s2"])
def test_call_reads_its_requests_from_the_previous_calls_slots(kvc, route):
    # B's token_to_req IS A's kv_cache read as int32: the request of each of
    # B's boundary tokens is a code A writes.  A guess of B's index chain made
    # before the grid dependency wait may hold a stale request; B must still
    # produce what it produces after A is done.
    a, a_kv, run_a = _coded_case_a(kvc)
    words = a_kv.view(-1).view(torch.int32)
    rng = np.random.Generator(np.random.PCG64(inputs.BASE_SEED + 7201))
    slots = rng.choice(a.num_outputs, size=256, replace=True)
    j = rng.integers(0, 56, size=256)
    bti = np.unique((slots // 64) * 9344 + (slots % 64) * 144 + 2 * j)   # code words of A's slots
    n_b, t_b, R = bti.size, words.numel(), 128
    blocks = 256
    b_state = torch.from_numpy(
        inputs.make_case(1, 8 * blocks, 16, seed=inputs.BASE_SEED + 7202).state_bits.view(np.int16)
    ).view(torch.bfloat16).cuda()
    t = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()
    b_args = dict(token_to_req=words, positions=torch.full((t_b,), 15, dtype=torch.int64, device="cuda"),
                  boundary_token_indices=t(bti.astype(np.int64)),
                  block_table=t(rng.integers(0, blocks, size=(R, 2)).astype(np.int32)),
                  rms_norm_weight=t(a.rms_norm_weight), cos_sin_cache=t(inputs._cos_sin_table(16)),
                  kv_slot_mapping=t(rng.permutation(n_b).astype(np.int64)))
    flags = 0 if route == "auto" else kvc.make_flags("cluster", 0, 2)

    def out_b():
        return (torch.zeros(((n_b + 63) // 64, inputs.KV_PAGE_BYTES), dtype=torch.uint8, device="cuda"),
                torch.zeros((n_b, 512), dtype=torch.float32, device="cuda"))

    def run_b(kv, yb):
        kvc.c128_256_512_compress(b_state, block_size=8, compress_ratio=16, y_out=yb,
                                  flags=flags, kv_cache=kv, **b_args)
        return kv, yb

    run_a()
    torch.cuda.synchronize()
    r = words[torch.from_numpy(bti).cuda()]
    assert int(r.min()) >= 63 and int(r.max()) < R, "A's code words"
    _chain_b_against_sync(kvc, run_a, run_b, out_b, words, 40)


@pytest.mark.parametrize("route", ["auto", "s2"])
def test_call_reads_its_boundary_tokens_from_the_previous_calls_slots(kvc, route):
    # B's boundary_token_indices IS the start of A's kv_cache read as int64:
    # the 56 code words of A's first slot.  A guess made before the wait may
    # hold a stale boundary token; B must still match the synchronised run.
    a, a_kv, run_a = _coded_case_a(kvc)
    words = a_kv.view(-1).view(torch.int64)
    n_b = 56
    bti = words[:n_b]
    rng = np.random.Generator(np.random.PCG64(inputs.BASE_SEED + 7301))
    b_state = torch.from_numpy(
        inputs.make_case(1, 128, 16, seed=inputs.BASE_SEED + 7302).state_bits.view(np.int16)
    ).view(torch.bfloat16).cuda()
    t = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()
    b_args = dict(token_to_req=torch.zeros(128, dtype=torch.int32, device="cuda"),
                  positions=torch.arange(128, dtype=torch.int64, device="cuda"),
                  boundary_token_indices=bti,
                  block_table=t(rng.permutation(16).astype(np.int32)[None, :]),
                  rms_norm_weight=t(a.rms_norm_weight), cos_sin_cache=t(inputs._cos_sin_table(128)),
                  kv_slot_mapping=t(rng.permutation(n_b).astype(np.int64)))
    flags = 0 if route == "auto" else kvc.make_flags("cluster", 0, 2)

    def out_b():
        return (torch.zeros((1, inputs.KV_PAGE_BYTES), dtype=torch.uint8, device="cuda"),
                torch.zeros((n_b, 512), dtype=torch.float32, device="cuda"))

    def run_b(kv, yb):
        kvc.c128_256_512_compress(b_state, block_size=8, compress_ratio=16, y_out=yb,
                                  flags=flags, kv_cache=kv, **b_args)
        return kv, yb

    run_a()
    torch.cuda.synchronize()
    assert int(bti.min()) >= 63 and int(bti.max()) < 128, "A's code words"
    _chain_b_against_sync(kvc, run_a, run_b, out_b, bti, 40)
