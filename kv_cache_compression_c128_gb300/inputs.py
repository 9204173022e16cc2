"""Seeded synthetic workloads for the KV-cache window compressor.

This module only *builds input arrays*.  It holds none of the compressor's
arithmetic (no softmax, normalisation, quantisation or RoPE rotation), so both
the CUDA path and the CPU oracle can be fed from it without sharing any of
the method.

Shapes follow the benchmark table of "From Attention to KV Cache Compression:
Notes from a KernelGen Optimization" (section "Competition Background and
Problem Statement"): ``num_reqs/total_tokens`` in {1/8192, 4/32768, 8/65536,
8/131072} times ``compress_ratio`` in {128, 256, 512}, ``block_size`` = 8.
The argument list and the packed slot layout are the ones of the sections
"The Compression Operator" and "Gather and Scatter" of the same page.

Recipe (every array is a pure function of the shape and the seed):

* ``state_cache``: bf16 ``[T/8, 8, 1024]``; N(0,1) drawn in fp32 (numpy PCG64)
  then rounded to bf16 (round-to-nearest-even, done by torch's dtype cast).
  Columns 0..511 are the values and 512..1023 the scores; both use the same
  distribution.
* ``block_table``: int32 ``[R, max_len/8]``.  One seeded permutation of the
  ``T/8`` physical blocks is cut into per-request runs, so requests own
  disjoint, randomly placed blocks.  Unused tail entries of shorter (ragged)
  requests hold -1.
* ``token_to_req``: int32 ``[T]``, requests are concatenated in token order.
* ``positions``: int64 ``[T]``, restarting at 0 for each request.
* ``boundary_token_indices``: int64 ``[N]``, the tokens whose position ``p``
  has ``(p + 1) % C == 0``, in token order.
* ``rms_norm_weight``: fp32 ``[512]``, ``1 + 0.1 * N(0,1)``; eps = 1e-6.
* ``cos_sin_cache``: fp32 ``[max_len, 64]``: columns 0..31 hold
  ``cos(pos * theta**(-j/32))`` and 32..63 the matching ``sin``, theta=10000
  (the standard RoPE table, evaluated in float64 then rounded to fp32).
* ``kv_slot_mapping``: int64 ``[T]``: -1 at ordinary tokens, a seeded
  permutation of ``0..N-1`` at the boundary tokens.
* ``kv_cache``: uint8 ``[ceil(N/64), 64*576 + 64*8]`` filled with zeros (or a
  seeded byte pattern, for the untouched-bytes tests).

Layout variants (the fp32 state the page's traffic count of "The Baseline"
assumes, and the explicit block / row / column strides of "A Bit of Triton
and GPU Background"):

* ``fp32_state``: fp32 ``[T/8, 8, 1024]``, N(0,1) drawn from its own seed and
  kept in fp32 (most values are not representable in bf16).
* ``embed_strided``: places a state in a larger flat buffer at element
  ``g * block_stride + o * row_stride + col``; every other element holds a
  poison value (NaN by default), so a stride mistake cannot go unnoticed.
* ``strided_table``: the same for the block table, entry ``(r, l)`` at
  ``r * row_stride + l * col_stride``, the rest -1.
"""
from __future__ import annotations

import dataclasses
from typing import Optional, Sequence

import numpy as np

HEAD_DIM = 512
STATE_WIDTH = 2 * HEAD_DIM
BLOCK_SIZE = 8
KV_BLOCK_SIZE = 64
TOKEN_STRIDE = 576
SCALE_DIM = 8
KV_PAGE_BYTES = KV_BLOCK_SIZE * (TOKEN_STRIDE + SCALE_DIM)
ROPE_THETA = 10000.0
RMS_EPS = 1.0e-6
BASE_SEED = 20260614

# The twelve benchmark shapes: (num_reqs, total_tokens, compress_ratio).
BENCH_SHAPES = [
    (r, t, c)
    for c in (128, 256, 512)
    for (r, t) in ((1, 8192), (4, 32768), (8, 65536), (8, 131072))
]


@dataclasses.dataclass
class Case:
    """One synthetic call of the compressor (host numpy arrays)."""

    name: str
    num_reqs: int
    total_tokens: int
    compress_ratio: int
    block_size: int
    lengths: np.ndarray              # int64 [R]
    state_bits: np.ndarray           # uint16 [T/8, 8, 1024] raw bf16 bits
    token_to_req: np.ndarray         # int32 [T]
    positions: np.ndarray            # int64 [T]
    boundary_token_indices: np.ndarray  # int64 [N]
    block_table: np.ndarray          # int32 [R, max_blocks]
    rms_norm_weight: np.ndarray      # float32 [512]
    cos_sin_cache: np.ndarray        # float32 [P, 64]
    kv_slot_mapping: np.ndarray      # int64 [T]
    kv_cache: np.ndarray             # uint8 [pages, 37376]
    rms_norm_eps: float = RMS_EPS

    @property
    def num_outputs(self) -> int:
        return int(self.boundary_token_indices.shape[0])

    @property
    def num_state_blocks(self) -> int:
        return int(self.state_bits.shape[0])

    def algorithmic_bytes(self) -> int:
        """Bytes the method must move for one call (reads + writes).

        state rows N*C*2048, block-table entries N*(C/8)*4, per-output
        metadata N*(8+4+8+8) (boundary index, request, position, slot),
        one cos/sin row N*256, the weight vector 2048, and the written
        slot bytes N*(576+8).
        """
        n, c = self.num_outputs, self.compress_ratio
        return (n * c * STATE_WIDTH * 2 + n * (c // self.block_size) * 4
                + n * 28 + n * 256 + HEAD_DIM * 4
                + n * (TOKEN_STRIDE + SCALE_DIM))


def _bf16_bits_from_f32(x: np.ndarray) -> np.ndarray:
    """Round fp32 -> bf16 (RNE) through torch's cast; returns uint16 bits."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _cos_sin_table(num_positions: int) -> np.ndarray:
    j = np.arange(32, dtype=np.float64)
    inv_freq = ROPE_THETA ** (-(2.0 * j) / 64.0)
    ang = np.arange(num_positions, dtype=np.float64)[:, None] * inv_freq[None, :]
    return np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32)


def make_case(num_reqs: int, total_tokens: int, compress_ratio: int, *,
              seed: int, block_size: int = BLOCK_SIZE,
              lengths: Optional[Sequence[int]] = None,
              kv_fill: Optional[int] = None, name: str = "",
              boundaries_per_req: Optional[int] = None) -> Case:
    """Build one seeded synthetic call.

    ``lengths`` (per-request token counts, each a multiple of ``block_size``;
    of ``compress_ratio`` too unless ``boundaries_per_req`` is given) defaults
    to equal requests.  Boundary tokens are those with ``(p + 1) % C == 0``,
    as in the benchmark; with ``boundaries_per_req`` set they are instead
    that many distinct positions per request drawn uniformly from
    ``[C - 1, L - 1]`` (windows at arbitrary offsets, for the general-window
    tests).  ``kv_fill``: None -> zero-filled kv_cache; an int -> a seeded
    byte pattern drawn from that seed (to check that unwritten bytes stay
    untouched).
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    R, T, C, B = num_reqs, total_tokens, compress_ratio, block_size
    if lengths is None:
        assert T % R == 0
        lengths = [T // R] * R
    lengths = np.asarray(lengths, dtype=np.int64)
    assert lengths.shape == (R,) and int(lengths.sum()) == T
    assert all(int(L) % B == 0 for L in lengths)
    if boundaries_per_req is None:
        assert all(int(L) % C == 0 for L in lengths)

    num_blocks = T // B
    state = rng.standard_normal((num_blocks, B, STATE_WIDTH), dtype=np.float32)
    state_bits = _bf16_bits_from_f32(state).reshape(num_blocks, B, STATE_WIDTH)
    del state

    perm = rng.permutation(num_blocks).astype(np.int32)
    max_blocks = int(lengths.max()) // B
    block_table = np.full((R, max_blocks), -1, dtype=np.int32)
    assert num_blocks == T // B
    token_to_req = np.empty(T, dtype=np.int32)
    positions = np.empty(T, dtype=np.int64)
    start_tok = 0
    start_blk = 0
    for r, L in enumerate(lengths.tolist()):
        nb = L // B
        block_table[r, :nb] = perm[start_blk:start_blk + nb]
        token_to_req[start_tok:start_tok + L] = r
        positions[start_tok:start_tok + L] = np.arange(L, dtype=np.int64)
        start_tok += L
        start_blk += nb

    if boundaries_per_req is None:
        bti = np.nonzero((positions + 1) % C == 0)[0].astype(np.int64)
    else:
        picks = []
        start = 0
        for L in lengths.tolist():
            k = min(boundaries_per_req, L - C + 1)
            pos = rng.choice(np.arange(C - 1, L), size=k, replace=False)
            picks.append(start + np.sort(pos))
            start += L
        bti = np.concatenate(picks).astype(np.int64)
    N = int(bti.shape[0])
    weight = (1.0 + 0.1 * rng.standard_normal(HEAD_DIM)).astype(np.float32)
    csc = _cos_sin_table(int(lengths.max()))
    slot_map = np.full(T, -1, dtype=np.int64)
    slot_map[bti] = rng.permutation(N).astype(np.int64)
    pages = (N + KV_BLOCK_SIZE - 1) // KV_BLOCK_SIZE
    if kv_fill is None:
        kv = np.zeros((pages, KV_PAGE_BYTES), dtype=np.uint8)
    else:
        kv = np.random.Generator(np.random.PCG64(kv_fill)).integers(
            0, 256, size=(pages, KV_PAGE_BYTES), dtype=np.uint8)
    return Case(name=name or f"r{R}_t{T}_c{C}", num_reqs=R, total_tokens=T,
                compress_ratio=C, block_size=B, lengths=lengths,
                state_bits=state_bits, token_to_req=token_to_req,
                positions=positions, boundary_token_indices=bti,
                block_table=block_table, rms_norm_weight=weight,
                cos_sin_cache=csc, kv_slot_mapping=slot_map, kv_cache=kv)


def fp32_state(num_blocks: int, block_size: int, seed: int) -> np.ndarray:
    """fp32 state [num_blocks, block_size, 1024] drawn N(0,1), seed `seed`."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return rng.standard_normal((num_blocks, block_size, STATE_WIDTH), dtype=np.float32)


def embed_strided(state: np.ndarray, block_stride: int, row_stride: int,
                  fill=None) -> np.ndarray:
    """Flat copy of `state` ([G, B, 1024], uint16 bf16 bits or float32) with
    element (g, o, col) at g * block_stride + o * row_stride + col; every
    other element holds `fill` (default: a quiet NaN of the dtype)."""
    G, B, W = state.shape
    assert W == STATE_WIDTH and row_stride >= W and block_stride >= (B - 1) * row_stride + W
    size = (G - 1) * block_stride + (B - 1) * row_stride + W
    if fill is None:
        fill = np.uint16(0x7FC1) if state.dtype == np.uint16 else np.float32(np.nan)
    out = np.full(size, fill, dtype=state.dtype)
    e = out.itemsize
    view = np.lib.stride_tricks.as_strided(out, shape=(G, B, W),
                                           strides=(block_stride * e, row_stride * e, e))
    view[...] = state
    return out


def strided_table(block_table: np.ndarray, row_stride: int, col_stride: int) -> np.ndarray:
    """Flat int32 copy of `block_table` ([R, M]) with entry (r, l) at
    r * row_stride + l * col_stride; other entries hold -1."""
    R, M = block_table.shape
    size = (R - 1) * row_stride + (M - 1) * col_stride + 1
    out = np.full(size, -1, dtype=np.int32)
    idx = np.arange(R)[:, None] * row_stride + np.arange(M)[None, :] * col_stride
    assert np.unique(idx).size == idx.size
    out[idx] = block_table
    return out


def ragged_lengths(num_reqs: int, total_tokens: int, compress_ratio: int,
                   seed: int) -> list:
    """Unequal request lengths L_i = C * (1 + m_i), m ~ Multinomial(T/C - R)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    extra = rng.multinomial(total_tokens // compress_ratio - num_reqs,
                            [1.0 / num_reqs] * num_reqs)
    return [compress_ratio * (1 + int(m)) for m in extra]


def bench_case(case_id: int) -> Case:
    """Case ``case_id`` (0..11) of the benchmark table, seed BASE_SEED+id."""
    R, T, C = BENCH_SHAPES[case_id]
    return make_case(R, T, C, seed=BASE_SEED + case_id,
                     name=f"r{R}_t{T}_c{C}")


def ragged_case(compress_ratio: int = 128, total_tokens: int = 131072,
                num_reqs: int = 8) -> Case:
    """The ragged variant: 8 unequal requests summing to 131072 tokens."""
    seed = BASE_SEED + 100 + compress_ratio
    L = ragged_lengths(num_reqs, total_tokens, compress_ratio, seed)
    return make_case(num_reqs, total_tokens, compress_ratio, seed=seed + 1,
                     lengths=L, name=f"ragged_r{num_reqs}_t{total_tokens}_c{compress_ratio}")


def general_window_case(compress_ratio: int = 128, block_size: int = 16) -> Case:
    """Headline-sized call with general windows: 8 requests x 16384 tokens,
    block_size 16, 128 windows per request at random starts (1024 outputs)."""
    seed = BASE_SEED + 300 + compress_ratio + block_size
    return make_case(8, 131072, compress_ratio, seed=seed, block_size=block_size,
                     boundaries_per_req=128,
                     name=f"general_r8_t131072_c{compress_ratio}_b{block_size}")


def block16_case() -> Case:
    """The headline shape (8 x 16384 tokens, C = 128, block-aligned windows)
    with block_size 16: the same bytes in 32 KiB physical blocks."""
    return make_case(8, 131072, 128, seed=BASE_SEED + 400, block_size=16,
                     name="r8_t131072_c128_b16")


def headline_case() -> Case:
    """8 requests x 16384 tokens, compress_ratio 128: the largest case."""
    return bench_case(BENCH_SHAPES.index((8, 131072, 128)))
