"""CPU oracle for the KV-cache window compressor -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline /
reference leg of ``bench.py`` may import this package.  The product library
(``kv_cache_compression_c128_gb300``) never imports, links or runs it, and
the two share no code: the arithmetic lives in ``kvc_oracle.c`` (plain,
single-threaded C, pinned by ``tests/test_oracle_*.py``), this module only
compiles it with gcc and marshals numpy arrays through ctypes.

Every function follows "From Attention to KV Cache Compression: Notes from
a KernelGen Optimization", sections "How One Output Is Produced" (window,
paged rows, per-dimension softmax sum, RMSNorm, quantisation, RoPE,
scatter), "Gather and Scatter" (slot layout) and "The Finalizer's Sharp
Edges" (fp32 finalizer, bf16 round trip, truncation, byte encoding).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvc_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libkvc_oracle.so")
_lock = threading.Lock()
_lib = None

HEAD_DIM = 512


def build(force: bool = False) -> str:
    """Compile kvc_oracle.c into _build/libkvc_oracle.so (gcc, no contraction)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
               "-fno-fast-math", "-Wall", "-Wextra", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I64, I32, F32 = ctypes.c_int64, ctypes.c_int32, ctypes.c_float
            lib.kvc_oracle_f32_to_bf16.argtypes = [F32]
            lib.kvc_oracle_f32_to_bf16.restype = ctypes.c_uint16
            lib.kvc_oracle_f32_to_bf16_n.argtypes = [P, P, I64]
            lib.kvc_oracle_f32_to_bf16_n.restype = None
            lib.kvc_oracle_bf16_round.argtypes = [F32]
            lib.kvc_oracle_bf16_round.restype = F32
            lib.kvc_oracle_scale_exponent.argtypes = [F32]
            lib.kvc_oracle_scale_exponent.restype = ctypes.c_int
            lib.kvc_oracle_window_reduce.argtypes = [
                P, I64, I32, P, P, I64, P, I64, P, I64, I64, I32, P, P]
            lib.kvc_oracle_window_reduce.restype = ctypes.c_int
            lib.kvc_oracle_window_reduce_ex.argtypes = [
                P, I32, I64, I64, I64, I32, P, P, I64, P, I64, P, I64, I64, I64, I64, I32, P, P]
            lib.kvc_oracle_window_reduce_ex.restype = ctypes.c_int
            lib.kvc_oracle_rmsnorm.argtypes = [P, P, F32, I64, P]
            lib.kvc_oracle_rmsnorm.restype = None
            lib.kvc_oracle_pack_slot.argtypes = [P, P, P, P]
            lib.kvc_oracle_pack_slot.restype = None
            lib.kvc_oracle_quant_rope_scatter.argtypes = [
                P, P, I64, P, P, I64, I32, P, I64, P, I64, P, I64]
            lib.kvc_oracle_quant_rope_scatter.restype = ctypes.c_int
            lib.kvc_oracle_compress.argtypes = [
                P, I64, P, P, I64, P, I64, P, I64, I64, P, P, I64, P, I64, P,
                I64, I32, I32, F32, P, P, P]
            lib.kvc_oracle_compress.restype = ctypes.c_int
            lib.kvc_oracle_compress_ex.argtypes = [
                P, I32, I64, I64, I64, P, P, I64, P, I64, P, I64, I64, I64, I64, P, P, I64, P,
                I64, P, I64, I32, I32, F32, P, P, P]
            lib.kvc_oracle_compress_ex.restype = ctypes.c_int
            lib.kvc_oracle_dequantize.argtypes = [P, I64, P, I64, P, I32]
            lib.kvc_oracle_dequantize.restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


# ---- scalar helpers -------------------------------------------------------

def f32_to_bf16_bits(x: float) -> int:
    """bf16 round-to-nearest-even of one float, as raw 16-bit pattern."""
    return int(_load().kvc_oracle_f32_to_bf16(float(x)))


def f32_to_bf16_bits_array(x) -> np.ndarray:
    """Vectorised f32_to_bf16_bits (uint16 array of the same shape)."""
    x = _c(x, np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    _load().kvc_oracle_f32_to_bf16_n(_ptr(x), _ptr(out), x.size)
    return out


def bf16_round(x: float) -> float:
    return float(_load().kvc_oracle_bf16_round(float(x)))


def scale_exponent(a: float) -> int:
    """ceil(log2(a / 127)) for a > 0 (exact)."""
    return int(_load().kvc_oracle_scale_exponent(float(a)))


# ---- pipeline steps -------------------------------------------------------

def window_reduce(state_bits, token_to_req, positions, boundary_token_indices,
                  block_table, compress_ratio, block_size=8
                  ) -> Tuple[np.ndarray, np.ndarray, int]:
    """Per-dimension softmax-weighted window sum c[N, 512] (float32).

    Returns (c, valid[N] uint8, status)."""
    st = _c(state_bits, np.uint16)
    t2r = _c(token_to_req, np.int32)
    pos = _c(positions, np.int64)
    bti = _c(boundary_token_indices, np.int64)
    bt = _c(block_table, np.int32)
    N = bti.shape[0]
    c = np.zeros((N, HEAD_DIM), dtype=np.float32)
    valid = np.zeros(N, dtype=np.uint8)
    status = _load().kvc_oracle_window_reduce(
        _ptr(st), st.shape[0], block_size, _ptr(t2r), _ptr(pos), pos.shape[0],
        _ptr(bti), N, _ptr(bt), bt.shape[0], bt.shape[1], compress_ratio,
        _ptr(c), _ptr(valid))
    return c, valid, int(status)


def window_reduce_ex(state, block_stride, row_stride, num_blocks, block_size, token_to_req,
                     positions, boundary_token_indices, block_table, max_blocks_per_req,
                     bt_row_stride, bt_col_stride, compress_ratio):
    """window_reduce over a strided state: `state` is a flat numpy array of
    uint16 (bf16 bits) or float32 elements, addressed as block g, row o,
    column col at g * block_stride + o * row_stride + col; block_table is a
    flat int32 array addressed as r * bt_row_stride + l * bt_col_stride."""
    st = np.ascontiguousarray(state).reshape(-1)
    dtype = 2 if st.dtype == np.float32 else 1
    assert st.dtype in (np.float32, np.uint16)
    t2r = _c(token_to_req, np.int32)
    pos = _c(positions, np.int64)
    bti = _c(boundary_token_indices, np.int64)
    bt = _c(block_table, np.int32).reshape(-1)
    N = bti.shape[0]
    num_reqs = int(t2r.max()) + 1 if t2r.size else 1
    c = np.zeros((N, HEAD_DIM), dtype=np.float32)
    valid = np.zeros(N, dtype=np.uint8)
    status = _load().kvc_oracle_window_reduce_ex(
        _ptr(st), dtype, block_stride, row_stride, num_blocks, block_size, _ptr(t2r), _ptr(pos),
        pos.shape[0], _ptr(bti), N, _ptr(bt), num_reqs, max_blocks_per_req, bt_row_stride,
        bt_col_stride, compress_ratio, _ptr(c), _ptr(valid))
    return c, valid, int(status)


def rmsnorm(c, weight, eps=1e-6) -> np.ndarray:
    c = _c(c, np.float32)
    w = _c(weight, np.float32)
    y = np.empty_like(c)
    _load().kvc_oracle_rmsnorm(_ptr(c), _ptr(w), float(eps), c.shape[0], _ptr(y))
    return y


def pack_slot(y_row, cos_sin_row) -> Tuple[np.ndarray, np.ndarray]:
    """576 payload bytes and 8 scale bytes of one normalised vector y[512]."""
    y = _c(y_row, np.float32)
    cs = _c(cos_sin_row, np.float32)
    assert y.shape == (HEAD_DIM,) and cs.shape == (64,)
    payload = np.zeros(576, dtype=np.uint8)
    scale = np.zeros(8, dtype=np.uint8)
    _load().kvc_oracle_pack_slot(_ptr(y), _ptr(cs), _ptr(payload), _ptr(scale))
    return payload, scale


def quant_rope_scatter(y, positions, boundary_token_indices, compress_ratio,
                       cos_sin_cache, kv_slot_mapping, kv_cache,
                       valid=None) -> int:
    """Quantise/rotate every y row and scatter it into kv_cache (in place)."""
    y = _c(y, np.float32)
    pos = _c(positions, np.int64)
    bti = _c(boundary_token_indices, np.int64)
    csc = _c(cos_sin_cache, np.float32)
    sm = _c(kv_slot_mapping, np.int64)
    assert kv_cache.flags.c_contiguous and kv_cache.dtype == np.uint8
    v = None if valid is None else _c(valid, np.uint8)
    return int(_load().kvc_oracle_quant_rope_scatter(
        _ptr(y), _ptr(v), y.shape[0], _ptr(bti), _ptr(pos), pos.shape[0],
        compress_ratio, _ptr(csc), csc.shape[0], _ptr(sm), sm.shape[0],
        _ptr(kv_cache), kv_cache.shape[0]))


def compress(state_bits, token_to_req, positions, boundary_token_indices,
             block_table, rms_norm_weight, cos_sin_cache, kv_slot_mapping,
             kv_cache, block_size, compress_ratio, rms_norm_eps=1e-6):
    """The whole operator on host arrays; kv_cache (uint8) is written in place.

    Returns a dict with c, y (float32 [N, 512]), valid (uint8 [N]) and status.
    """
    st = _c(state_bits, np.uint16)
    t2r = _c(token_to_req, np.int32)
    pos = _c(positions, np.int64)
    bti = _c(boundary_token_indices, np.int64)
    bt = _c(block_table, np.int32)
    w = _c(rms_norm_weight, np.float32)
    csc = _c(cos_sin_cache, np.float32)
    sm = _c(kv_slot_mapping, np.int64)
    assert kv_cache.flags.c_contiguous and kv_cache.dtype == np.uint8
    N = bti.shape[0]
    c = np.zeros((N, HEAD_DIM), dtype=np.float32)
    y = np.zeros((N, HEAD_DIM), dtype=np.float32)
    valid = np.zeros(N, dtype=np.uint8)
    status = _load().kvc_oracle_compress(
        _ptr(st), st.shape[0], _ptr(t2r), _ptr(pos), pos.shape[0], _ptr(bti), N,
        _ptr(bt), bt.shape[0], bt.shape[1], _ptr(w), _ptr(csc), csc.shape[0],
        _ptr(sm), sm.shape[0], _ptr(kv_cache), kv_cache.shape[0], block_size,
        compress_ratio, float(rms_norm_eps), _ptr(c), _ptr(y), _ptr(valid))
    return {"c": c, "y": y, "valid": valid, "status": int(status)}


def compress_strided(state, block_stride, row_stride, num_blocks, token_to_req, positions,
                     boundary_token_indices, block_table, num_reqs, max_blocks_per_req,
                     bt_row_stride, bt_col_stride, rms_norm_weight, cos_sin_cache,
                     kv_slot_mapping, kv_cache, block_size, compress_ratio, rms_norm_eps=1e-6):
    """compress over a strided state of bf16 bits (uint16) or float32: `state`
    is a flat array addressed as g * block_stride + o * row_stride + col, and
    `block_table` a flat int32 array addressed as r * bt_row_stride +
    l * bt_col_stride.  kv_cache (uint8) is written in place; returns the same
    dict as compress."""
    st = np.ascontiguousarray(state).reshape(-1)
    assert st.dtype in (np.float32, np.uint16)
    dtype = 2 if st.dtype == np.float32 else 1
    t2r = _c(token_to_req, np.int32)
    pos = _c(positions, np.int64)
    bti = _c(boundary_token_indices, np.int64)
    bt = _c(block_table, np.int32).reshape(-1)
    w = _c(rms_norm_weight, np.float32)
    csc = _c(cos_sin_cache, np.float32)
    sm = _c(kv_slot_mapping, np.int64)
    assert kv_cache.flags.c_contiguous and kv_cache.dtype == np.uint8
    N = bti.shape[0]
    c = np.zeros((N, HEAD_DIM), dtype=np.float32)
    y = np.zeros((N, HEAD_DIM), dtype=np.float32)
    valid = np.zeros(N, dtype=np.uint8)
    status = _load().kvc_oracle_compress_ex(
        _ptr(st), dtype, block_stride, row_stride, num_blocks, _ptr(t2r), _ptr(pos),
        pos.shape[0], _ptr(bti), N, _ptr(bt), num_reqs, max_blocks_per_req, bt_row_stride,
        bt_col_stride, _ptr(w), _ptr(csc), csc.shape[0], _ptr(sm), sm.shape[0],
        _ptr(kv_cache), kv_cache.shape[0], block_size, compress_ratio, float(rms_norm_eps),
        _ptr(c), _ptr(y), _ptr(valid))
    return {"c": c, "y": y, "valid": valid, "status": int(status)}


def dequantize(kv_cache, slots, out_bf16: bool = False):
    """Decode slots back to vectors: float32 [M, 512], or raw bf16 bits
    (uint16 [M, 512]) when out_bf16.  Returns (out, status)."""
    assert kv_cache.flags.c_contiguous and kv_cache.dtype == np.uint8
    sl = _c(slots, np.int64)
    out = np.zeros((sl.shape[0], HEAD_DIM), dtype=np.uint16 if out_bf16 else np.float32)
    st = _load().kvc_oracle_dequantize(_ptr(kv_cache), kv_cache.shape[0], _ptr(sl),
                                       sl.shape[0], _ptr(out), 1 if out_bf16 else 0)
    return out, int(st)


def compress_case(case, kv_cache=None):
    """Run the oracle on an inputs.Case; returns (kv_cache, result dict)."""
    kv = case.kv_cache.copy() if kv_cache is None else kv_cache
    res = compress(case.state_bits, case.token_to_req, case.positions,
                   case.boundary_token_indices, case.block_table,
                   case.rms_norm_weight, case.cos_sin_cache,
                   case.kv_slot_mapping, kv, case.block_size,
                   case.compress_ratio, case.rms_norm_eps)
    return kv, res
