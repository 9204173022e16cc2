"""GB300-native KV-cache window compressor (``c128_256_512_compress``).

The computation runs in the CUDA library ``_lib/libkvc.so`` (sources in
``csrc/``, C ABI in ``include/kvc.h``); this module only marshals arguments
through ctypes.  There is no CPU fallback: if the library is missing or no
CUDA device is present, the calls raise.

The operator is the one of "From Attention to KV Cache Compression: Notes
from a KernelGen Optimization" (KernelGen Challenge 8 write-up), section
"The Compression Operator", with the layout of "Gather and Scatter".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor
from typing import Optional

_HERE = os.path.dirname(os.path.abspath(__file__))
_ROOT = os.path.dirname(_HERE)
_CSRC = os.path.join(_HERE, "csrc")
_INCLUDE = os.path.join(_ROOT, "include")
_LIB_DIR = os.path.join(_HERE, "_lib")
LIB_PATH = os.path.join(_LIB_DIR, "libkvc.so")
_SOURCES = ["kvc_cluster.cu", "kvc_streamk.cu", "kvc_reader.cu", "kvc_api.cu", "kvc_static.cu",
            "kvc_selftest.cu"]
ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]

KVC_OK = 0
KVC_ERR_INVALID_ARG = 1
KVC_ERR_UNSUPPORTED = 2
KVC_ERR_CUDA = 3
KVC_ERR_BAD_INDEX = 4
KVC_ERR_TIMEOUT = 5
KVC_ERR_SCRATCH_LIMIT = 6
KVC_FLAG_GRID_MASK = 0xFFFF
KVC_DTYPE_F32 = 0
KVC_DTYPE_BF16 = 1
KVC_FLAG_CLUSTER_SHIFT = 16
KVC_FLAG_STREAM_K = 1 << 24
KVC_FLAG_ROW_COPIES = 1 << 25


def make_flags(route: str = "auto", count: int = 0, cluster_size: int = 0,
               row_copies: bool = False) -> int:
    """kvc_compress flags: route 'auto' | 'cluster' | 'streamk', a forced
    launch size (clusters or CTAs; 0 = automatic), cluster size, and, for
    rows apart, row-by-row copies instead of TMA tensor maps."""
    f = int(count) & KVC_FLAG_GRID_MASK
    if route == "streamk":
        f |= KVC_FLAG_STREAM_K
    else:
        f |= (int(cluster_size) & 0x1F) << KVC_FLAG_CLUSTER_SHIFT
    if row_copies:
        f |= KVC_FLAG_ROW_COPIES
    return f

HEAD_DIM = 512
KV_PAGE_BYTES = 64 * (576 + 8)

_lock = threading.Lock()
_lib = None


class KvcError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {kvc_error_string(status)} (status {status})")


# ---- build -------------------------------------------------------------------

def _nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _stale() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    deps = [os.path.join(_CSRC, f) for f in os.listdir(_CSRC)]
    deps.append(os.path.join(_INCLUDE, "kvc.h"))
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile csrc/*.cu for sm_103a into _lib/libkvc.so (in-tree)."""
    if not force and not _stale():
        return LIB_PATH
    os.makedirs(_LIB_DIR, exist_ok=True)
    nvcc = _nvcc()
    common = ARCH_FLAGS + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
                           "-I", _INCLUDE]
    objs = [os.path.join(_LIB_DIR, s.replace(".cu", ".o")) for s in _SOURCES]

    def compile_one(src_obj):
        src, obj = src_obj
        cmd = [nvcc] + common + ["-c", os.path.join(_CSRC, src), "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        return r.stderr

    with ThreadPoolExecutor(len(_SOURCES)) as ex:
        logs = list(ex.map(compile_one, zip(_SOURCES, objs)))
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    r = subprocess.run([nvcc, "-shared"] + ARCH_FLAGS + objs + ["-o", tmp],
                       capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB_PATH)
    if verbose:
        print("".join(logs))
    return LIB_PATH


# ---- loading -----------------------------------------------------------------

def lib():
    """The loaded libkvc.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it with "
                    "kv_cache_compression_c128_gb300.build() (there is no CPU fallback)")
            L = ctypes.CDLL(LIB_PATH)
            P, I64, I32, U32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_uint32
            L.kvc_workspace_bytes.argtypes = [I64]
            L.kvc_workspace_bytes.restype = ctypes.c_size_t
            L.kvc_compress.argtypes = [
                P, I64, P, P, I64, P, I64, P, I64, I64, P, P, I64, P, I64, P, I64,
                I32, I32, ctypes.c_float, P, P, ctypes.c_size_t, U32, P]
            L.kvc_compress.restype = ctypes.c_int
            L.kvc_compress_static.argtypes = [
                P, I64, P, P, I64, P, I64, P, I64, I64, P, P, I64, P, I64, P, I64,
                I32, I32, ctypes.c_float, P, U32, P]
            L.kvc_compress_static.restype = ctypes.c_int
            L.kvc_compress_layers.argtypes = [
                I32, P, I64, P, P, I64, P, I64, P, I64, I64, P, P, I64, P, I64, P, I64,
                I32, I32, ctypes.c_float, P, P, ctypes.c_size_t, U32, P]
            L.kvc_compress_layers.restype = ctypes.c_int
            L.kvc_compress_layers_strided.argtypes = [
                I32, P, I32, I64, I64, I64, P, P, I64, P, I64, P, I64, I64, I64, I64, P, P, I64,
                P, I64, P, I64, I32, I32, ctypes.c_float, P, P, ctypes.c_size_t, U32, P]
            L.kvc_compress_layers_strided.restype = ctypes.c_int
            L.kvc_dequantize.argtypes = [P, I64, P, I64, P, I32, P]
            L.kvc_dequantize.restype = ctypes.c_int
            L.kvc_compress_strided.argtypes = [
                P, I32, I64, I64, I64, P, P, I64, P, I64, P, I64, I64, I64, I64, P, P, I64, P,
                I64, P, I64, I32, I32, ctypes.c_float, P, P, ctypes.c_size_t, U32, P]
            L.kvc_compress_strided.restype = ctypes.c_int
            L.kvc_query_launch.argtypes = [I64, I32, U32, P, P, P, P]
            L.kvc_query_launch.restype = ctypes.c_int
            L.kvc_query_launch_ex.argtypes = [I64, I32, I32, U32, P, P, P, P]
            L.kvc_query_launch_ex.restype = ctypes.c_int
            L.kvc_selftest_wait_timeout.argtypes = [ctypes.c_uint64, P]
            L.kvc_selftest_wait_timeout.restype = ctypes.c_int
            L.kvc_selftest_set_wait_limit.argtypes = [ctypes.c_uint64]
            L.kvc_selftest_set_wait_limit.restype = ctypes.c_int
            L.kvc_selftest_poison_guesses.argtypes = [I32]
            L.kvc_selftest_poison_guesses.restype = ctypes.c_int
            L.kvc_selftest_first_pass_rejections.argtypes = [P, P]
            L.kvc_selftest_first_pass_rejections.restype = ctypes.c_int
            L.kvc_get_device_error.argtypes = [P, P]
            L.kvc_get_device_error.restype = ctypes.c_int
            L.kvc_error_string.argtypes = [ctypes.c_int]
            L.kvc_error_string.restype = ctypes.c_char_p
            L.kvc_version.argtypes = []
            L.kvc_version.restype = ctypes.c_char_p
            _lib = L
    return _lib


# ---- the C ABI, one Python function per entry point ---------------------------

def kvc_error_string(status: int) -> str:
    return lib().kvc_error_string(int(status)).decode()


def kvc_version() -> str:
    return lib().kvc_version().decode()


def kvc_workspace_bytes(num_outputs: int) -> int:
    return int(lib().kvc_workspace_bytes(int(num_outputs)))


def kvc_query_launch(num_outputs: int, compress_ratio: int, flags: int = 0):
    """(ctas, cluster size, threads, dynamic smem bytes) of the launch."""
    c, k, t, s = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
    st = lib().kvc_query_launch(int(num_outputs), int(compress_ratio), int(flags),
                                ctypes.byref(c), ctypes.byref(k), ctypes.byref(t),
                                ctypes.byref(s))
    if st != KVC_OK:
        raise KvcError(st, "kvc_query_launch")
    return c.value, k.value, t.value, s.value


def kvc_query_launch_ex(num_outputs: int, compress_ratio: int, state_dtype: int,
                        flags: int = 0):
    """kvc_query_launch for a state of element type state_dtype (KVC_DTYPE_*)."""
    c, k, t, s = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
    st = lib().kvc_query_launch_ex(int(num_outputs), int(compress_ratio), int(state_dtype),
                                   int(flags), ctypes.byref(c), ctypes.byref(k),
                                   ctypes.byref(t), ctypes.byref(s))
    if st != KVC_OK:
        raise KvcError(st, "kvc_query_launch_ex")
    return c.value, k.value, t.value, s.value


def kvc_selftest_wait_timeout(limit_cycles: int, stream: Optional[int] = None) -> int:
    """Launch the bounded-wait self-test (a wait that runs out after
    limit_cycles and records KVC_ERR_TIMEOUT); returns the launch status."""
    return int(lib().kvc_selftest_wait_timeout(int(limit_cycles), ctypes.c_void_p(stream or 0)))


def kvc_selftest_set_wait_limit(limit_cycles: int) -> int:
    """Test hook: the limit (SM cycles) on each pipeline wait of later
    compressions in this process; 0 restores the default.  Returns the
    status."""
    return int(lib().kvc_selftest_set_wait_limit(int(limit_cycles)))


def kvc_selftest_poison_guesses(on: bool) -> int:
    """Test hook: make every guessed first pass of later calls in this
    process fail its check (True) or guess normally (False).  Returns the
    status."""
    return int(lib().kvc_selftest_poison_guesses(1 if on else 0))


def kvc_selftest_first_pass_rejections(stream: Optional[int] = None) -> int:
    """Synchronise `stream`, read and clear the count of guessed first passes
    that failed their check on the current device."""
    n = ctypes.c_uint64()
    st = lib().kvc_selftest_first_pass_rejections(ctypes.c_void_p(stream or 0), ctypes.byref(n))
    if st != KVC_OK:
        raise KvcError(st, "kvc_selftest_first_pass_rejections")
    return int(n.value)


def kvc_get_device_error(stream: Optional[int] = None) -> int:
    """Synchronise `stream` (a cudaStream_t as int), read and clear the
    device error code."""
    code = ctypes.c_uint32()
    st = lib().kvc_get_device_error(ctypes.c_void_p(stream or 0), ctypes.byref(code))
    if st != KVC_OK:
        raise KvcError(st, "kvc_get_device_error")
    return int(code.value)


def kvc_compress(state_cache, num_state_blocks, token_to_req, positions, num_tokens,
                 boundary_token_indices, num_outputs, block_table, num_reqs,
                 max_blocks_per_req, rms_norm_weight, cos_sin_cache, num_positions,
                 kv_slot_mapping, slot_mapping_len, kv_cache, num_kv_pages, block_size,
                 compress_ratio, rms_norm_eps, y_out, workspace, workspace_bytes,
                 flags, stream) -> int:
    """The C entry point with raw integer pointers; returns the status."""
    v = ctypes.c_void_p
    return int(lib().kvc_compress(
        v(state_cache), num_state_blocks, v(token_to_req), v(positions), num_tokens,
        v(boundary_token_indices), num_outputs, v(block_table), num_reqs,
        max_blocks_per_req, v(rms_norm_weight), v(cos_sin_cache), num_positions,
        v(kv_slot_mapping), slot_mapping_len, v(kv_cache), num_kv_pages, block_size,
        compress_ratio, ctypes.c_float(rms_norm_eps), v(y_out), v(workspace),
        workspace_bytes, flags, v(stream)))


def kvc_compress_strided(state_cache, state_dtype, num_state_blocks, state_block_stride,
                         state_row_stride, token_to_req, positions, num_tokens,
                         boundary_token_indices, num_outputs, block_table, num_reqs,
                         max_blocks_per_req, block_table_row_stride, block_table_col_stride,
                         rms_norm_weight, cos_sin_cache, num_positions, kv_slot_mapping,
                         slot_mapping_len, kv_cache, num_kv_pages, block_size, compress_ratio,
                         rms_norm_eps, y_out, workspace, workspace_bytes, flags, stream) -> int:
    """The strided / fp32-state C entry point with raw integer pointers."""
    v = ctypes.c_void_p
    return int(lib().kvc_compress_strided(
        v(state_cache), int(state_dtype), num_state_blocks, state_block_stride,
        state_row_stride, v(token_to_req), v(positions), num_tokens,
        v(boundary_token_indices), num_outputs, v(block_table), num_reqs, max_blocks_per_req,
        block_table_row_stride, block_table_col_stride, v(rms_norm_weight), v(cos_sin_cache),
        num_positions, v(kv_slot_mapping), slot_mapping_len, v(kv_cache), num_kv_pages,
        int(block_size), int(compress_ratio), float(rms_norm_eps), v(y_out), v(workspace),
        int(workspace_bytes), int(flags), v(stream)))


def kvc_compress_static(state_cache, num_state_blocks, token_to_req, positions, num_tokens,
                        boundary_token_indices, num_outputs, block_table, num_reqs,
                        max_blocks_per_req, rms_norm_weight, cos_sin_cache, num_positions,
                        kv_slot_mapping, slot_mapping_len, kv_cache, num_kv_pages, block_size,
                        compress_ratio, rms_norm_eps, y_out, flags, stream) -> int:
    """kvc_compress without a workspace, for callers that cannot allocate
    device memory: the library's built-in 8 MiB scratch buffer is used
    instead (shared by all calls on a device; order overlapping calls).
    Raw integer pointers; returns the status."""
    v = ctypes.c_void_p
    return int(lib().kvc_compress_static(
        v(state_cache), num_state_blocks, v(token_to_req), v(positions), num_tokens,
        v(boundary_token_indices), num_outputs, v(block_table), num_reqs,
        max_blocks_per_req, v(rms_norm_weight), v(cos_sin_cache), num_positions,
        v(kv_slot_mapping), slot_mapping_len, v(kv_cache), num_kv_pages, block_size,
        compress_ratio, ctypes.c_float(rms_norm_eps), v(y_out), flags, v(stream)))


def kvc_compress_layers(num_layers, state_caches, num_state_blocks, token_to_req, positions,
                        num_tokens, boundary_token_indices, num_outputs, block_table, num_reqs,
                        max_blocks_per_req, rms_norm_weights, cos_sin_cache, num_positions,
                        kv_slot_mapping, slot_mapping_len, kv_caches, num_kv_pages, block_size,
                        compress_ratio, rms_norm_eps, y_out, workspace, workspace_bytes, flags,
                        stream) -> int:
    """The multi-layer entry point; the three per-layer arguments are
    sequences of integer device pointers.  Returns the status."""
    v = ctypes.c_void_p
    arr = lambda xs: (ctypes.c_void_p * len(xs))(*[int(x) for x in xs])
    return int(lib().kvc_compress_layers(
        int(num_layers), arr(state_caches), num_state_blocks, v(token_to_req), v(positions),
        num_tokens, v(boundary_token_indices), num_outputs, v(block_table), num_reqs,
        max_blocks_per_req, arr(rms_norm_weights), v(cos_sin_cache), num_positions,
        v(kv_slot_mapping), slot_mapping_len, arr(kv_caches), num_kv_pages, block_size,
        compress_ratio, ctypes.c_float(rms_norm_eps), v(y_out), v(workspace), workspace_bytes,
        flags, v(stream)))


def kvc_compress_layers_strided(num_layers, state_caches, state_dtype, num_state_blocks,
                                state_block_stride, state_row_stride, token_to_req, positions,
                                num_tokens, boundary_token_indices, num_outputs, block_table,
                                num_reqs, max_blocks_per_req, block_table_row_stride,
                                block_table_col_stride, rms_norm_weights, cos_sin_cache,
                                num_positions, kv_slot_mapping, slot_mapping_len, kv_caches,
                                num_kv_pages, block_size, compress_ratio, rms_norm_eps, y_out,
                                workspace, workspace_bytes, flags, stream) -> int:
    """The strided multi-layer entry point (raw integer pointers, per-layer
    sequences for the three per-layer arguments).  Returns the status."""
    v = ctypes.c_void_p
    arr = lambda xs: (ctypes.c_void_p * len(xs))(*[int(x) for x in xs])
    return int(lib().kvc_compress_layers_strided(
        int(num_layers), arr(state_caches), int(state_dtype), num_state_blocks,
        state_block_stride, state_row_stride, v(token_to_req), v(positions), num_tokens,
        v(boundary_token_indices), num_outputs, v(block_table), num_reqs, max_blocks_per_req,
        block_table_row_stride, block_table_col_stride, arr(rms_norm_weights), v(cos_sin_cache),
        num_positions, v(kv_slot_mapping), slot_mapping_len, arr(kv_caches), num_kv_pages,
        int(block_size), int(compress_ratio), ctypes.c_float(rms_norm_eps), v(y_out),
        v(workspace), int(workspace_bytes), int(flags), v(stream)))


def kvc_dequantize(kv_cache, num_kv_pages, slots, num_slots, out, out_dtype, stream) -> int:
    """Decode slots back to vectors (raw integer pointers); returns the status."""
    v = ctypes.c_void_p
    return int(lib().kvc_dequantize(v(kv_cache), num_kv_pages, v(slots), num_slots, v(out),
                                    int(out_dtype), v(stream)))


# ---- torch-facing wrappers ----------------------------------------------------

def dequantize(kv_cache, slots, dtype=None, out=None, stream=None):
    """Read slots of a packed kv_cache back as [len(slots), 512] vectors
    (torch.float32 or torch.bfloat16) on the cache's device."""
    import torch

    dtype = torch.float32 if dtype is None else dtype
    if dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("dtype must be torch.float32 or torch.bfloat16")
    dev = kv_cache.device
    if dev.type != "cuda":
        raise ValueError("kv_cache must be a CUDA tensor (there is no CPU path)")
    _check(kv_cache, "kv_cache", torch.uint8, dev)
    _check(slots, "slots", torch.int64, dev)
    M = slots.numel()
    if out is None:
        out = torch.empty((M, HEAD_DIM), dtype=dtype, device=dev)
    _check(out, "out", dtype, dev)
    with torch.cuda.device(dev):
        s = stream if stream is not None else torch.cuda.current_stream(dev)
        st = kvc_dequantize(kv_cache.data_ptr(), kv_cache.shape[0], slots.data_ptr(), M,
                            out.data_ptr(),
                            KVC_DTYPE_BF16 if dtype == torch.bfloat16 else KVC_DTYPE_F32,
                            int(s.cuda_stream))
    if st != KVC_OK:
        raise KvcError(st, "kvc_dequantize")
    return out


# ---- torch-facing wrapper with the statement's signature ----------------------

_workspaces = {}


def workspace_for(device, stream_ptr: int, num_outputs: int):
    """A zero-initialised workspace cached per (device, stream)."""
    import torch

    need = kvc_workspace_bytes(num_outputs)
    key = (device.index, stream_ptr)
    ws = _workspaces.get(key)
    if ws is None or ws.numel() < need:
        ws = torch.zeros(max(need, 1 << 20), dtype=torch.uint8, device=device)
        _workspaces[key] = ws
    return ws


def _check(t, name, dtype, device, contiguous=True):
    import torch

    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    dtypes = dtype if isinstance(dtype, tuple) else (dtype,)
    if t.dtype not in dtypes:
        raise TypeError(f"{name} must have dtype {' or '.join(map(str, dtypes))}, got {t.dtype}")
    if t.device != device:
        raise ValueError(f"{name} must be on {device}, got {t.device}")
    if contiguous and not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def c128_256_512_compress(state_cache, token_to_req, positions, boundary_token_indices,
                          block_table, rms_norm_weight, cos_sin_cache, kv_slot_mapping,
                          kv_cache, block_size, compress_ratio, rms_norm_eps=1.0e-6, *,
                          y_out=None, flags: int = 0, stream=None, workspace=None):
    """Compress every boundary token's window into its kv_cache slot, in place.

    state_cache bf16 or fp32 [blocks, block_size, 1024] (any block and row
    strides, columns contiguous); token_to_req int32 [T]; positions int64
    [T]; boundary_token_indices int64 [N]; block_table int32 [R, Lb] (any
    strides); rms_norm_weight fp32 [512]; cos_sin_cache fp32 [P, 64];
    kv_slot_mapping int64 [T] (or [N]); kv_cache uint8 [pages, 37376].  All
    on one CUDA device.  Optional y_out fp32 [N, 512] receives the
    normalised vectors.  A contiguous bf16 state with a contiguous table goes
    through kvc_compress, anything else through kvc_compress_strided.
    Returns kv_cache.
    """
    import torch

    dev = state_cache.device
    if dev.type != "cuda":
        raise ValueError("state_cache must be a CUDA tensor (there is no CPU path)")
    _check(state_cache, "state_cache", (torch.bfloat16, torch.float32), dev, contiguous=False)
    _check(token_to_req, "token_to_req", torch.int32, dev)
    _check(positions, "positions", torch.int64, dev)
    _check(boundary_token_indices, "boundary_token_indices", torch.int64, dev)
    _check(block_table, "block_table", torch.int32, dev, contiguous=False)
    _check(rms_norm_weight, "rms_norm_weight", torch.float32, dev)
    _check(cos_sin_cache, "cos_sin_cache", torch.float32, dev)
    _check(kv_slot_mapping, "kv_slot_mapping", torch.int64, dev)
    _check(kv_cache, "kv_cache", torch.uint8, dev)
    if state_cache.dim() != 3 or state_cache.shape[2] != 2 * HEAD_DIM:
        raise ValueError("state_cache must be [num_blocks, block_size, 1024]")
    if state_cache.stride(2) != 1:
        raise ValueError("state_cache columns must be contiguous (stride(2) == 1)")
    if state_cache.shape[1] != block_size:
        raise ValueError("state_cache.shape[1] must equal block_size")
    if block_table.dim() != 2 or cos_sin_cache.dim() != 2 or cos_sin_cache.shape[1] != 64:
        raise ValueError("block_table must be 2-D and cos_sin_cache [P, 64]")
    if rms_norm_weight.numel() != HEAD_DIM:
        raise ValueError("rms_norm_weight must have 512 elements")
    if kv_cache.dim() != 2 or kv_cache.shape[1] != KV_PAGE_BYTES:
        raise ValueError(f"kv_cache must be [num_pages, {KV_PAGE_BYTES}] uint8")
    if token_to_req.numel() != positions.numel():
        raise ValueError("token_to_req and positions must have one entry per token")
    N = boundary_token_indices.numel()
    if y_out is not None:
        _check(y_out, "y_out", torch.float32, dev)
        if y_out.numel() < N * HEAD_DIM:
            raise ValueError("y_out must hold num_outputs * 512 floats")
    with torch.cuda.device(dev):
        s = stream if stream is not None else torch.cuda.current_stream(dev)
        sp = int(s.cuda_stream)
        ws = workspace if workspace is not None else workspace_for(dev, sp, N)
        y_ptr = 0 if y_out is None else y_out.data_ptr()
        if (state_cache.dtype == torch.bfloat16 and state_cache.is_contiguous()
                and block_table.is_contiguous()):
            name = "kvc_compress"
            st = kvc_compress(
                state_cache.data_ptr(), state_cache.shape[0], token_to_req.data_ptr(),
                positions.data_ptr(), positions.numel(), boundary_token_indices.data_ptr(), N,
                block_table.data_ptr(), block_table.shape[0], block_table.shape[1],
                rms_norm_weight.data_ptr(), cos_sin_cache.data_ptr(), cos_sin_cache.shape[0],
                kv_slot_mapping.data_ptr(), kv_slot_mapping.numel(), kv_cache.data_ptr(),
                kv_cache.shape[0], int(block_size), int(compress_ratio), float(rms_norm_eps),
                y_ptr, ws.data_ptr(), ws.numel(), int(flags), sp)
        else:
            name = "kvc_compress_strided"
            st = kvc_compress_strided(
                state_cache.data_ptr(),
                KVC_DTYPE_F32 if state_cache.dtype == torch.float32 else KVC_DTYPE_BF16,
                state_cache.shape[0], state_cache.stride(0), state_cache.stride(1),
                token_to_req.data_ptr(), positions.data_ptr(), positions.numel(),
                boundary_token_indices.data_ptr(), N, block_table.data_ptr(),
                block_table.shape[0], block_table.shape[1], block_table.stride(0),
                block_table.stride(1), rms_norm_weight.data_ptr(), cos_sin_cache.data_ptr(),
                cos_sin_cache.shape[0], kv_slot_mapping.data_ptr(), kv_slot_mapping.numel(),
                kv_cache.data_ptr(), kv_cache.shape[0], int(block_size), int(compress_ratio),
                float(rms_norm_eps), y_ptr, ws.data_ptr(), ws.numel(), int(flags), sp)
    if st != KVC_OK:
        raise KvcError(st, name)
    return kv_cache


def compress_layers(state_caches, token_to_req, positions, boundary_token_indices, block_table,
                    rms_norm_weights, cos_sin_cache, kv_slot_mapping, kv_caches, block_size,
                    compress_ratio, rms_norm_eps=1.0e-6, *, y_out=None, flags: int = 0,
                    stream=None, workspace=None):
    """c128_256_512_compress for several layers in one launch: lists of
    per-layer state caches, RMSNorm weights and kv caches (same shapes and
    dtypes as the single-layer call) sharing every index array.  The state
    caches are bf16 or fp32, all of one dtype and one set of strides (any
    block and row strides, columns contiguous); the block table may have any
    strides.  y_out, if given, is fp32 [L * N, 512] (layer-major).  Returns
    kv_caches."""
    import torch

    L = len(state_caches)
    if not (len(rms_norm_weights) == L == len(kv_caches)) or L < 1:
        raise ValueError("state_caches, rms_norm_weights and kv_caches need one entry per layer")
    dev = state_caches[0].device
    if dev.type != "cuda":
        raise ValueError("state caches must be CUDA tensors (there is no CPU path)")
    s0 = state_caches[0]
    for l in range(L):
        _check(state_caches[l], f"state_caches[{l}]", (torch.bfloat16, torch.float32), dev,
               contiguous=False)
        _check(rms_norm_weights[l], f"rms_norm_weights[{l}]", torch.float32, dev)
        _check(kv_caches[l], f"kv_caches[{l}]", torch.uint8, dev)
        if state_caches[l].shape != s0.shape or kv_caches[l].shape != kv_caches[0].shape:
            raise ValueError("all layers need the same state and kv_cache shapes")
        if state_caches[l].dtype != s0.dtype or state_caches[l].stride() != s0.stride():
            raise ValueError("all layers need the same state dtype and strides")
    if s0.dim() != 3 or s0.shape[2] != 2 * HEAD_DIM or s0.stride(2) != 1:
        raise ValueError("state caches must be [num_blocks, block_size, 1024] with contiguous columns")
    for name, t, dt in (("token_to_req", token_to_req, torch.int32), ("positions", positions, torch.int64),
                        ("boundary_token_indices", boundary_token_indices, torch.int64),
                        ("cos_sin_cache", cos_sin_cache, torch.float32),
                        ("kv_slot_mapping", kv_slot_mapping, torch.int64)):
        _check(t, name, dt, dev)
    _check(block_table, "block_table", torch.int32, dev, contiguous=False)
    N = boundary_token_indices.numel()
    if y_out is not None:
        _check(y_out, "y_out", torch.float32, dev)
        if y_out.numel() < L * N * HEAD_DIM:
            raise ValueError("y_out must hold num_layers * num_outputs * 512 floats")
    with torch.cuda.device(dev):
        s = stream if stream is not None else torch.cuda.current_stream(dev)
        sp = int(s.cuda_stream)
        ws = workspace if workspace is not None else workspace_for(dev, sp, N)
        y_ptr = 0 if y_out is None else y_out.data_ptr()
        if s0.dtype == torch.bfloat16 and s0.is_contiguous() and block_table.is_contiguous():
            name = "kvc_compress_layers"
            st = kvc_compress_layers(
                L, [t.data_ptr() for t in state_caches], s0.shape[0],
                token_to_req.data_ptr(), positions.data_ptr(), positions.numel(),
                boundary_token_indices.data_ptr(), N, block_table.data_ptr(), block_table.shape[0],
                block_table.shape[1], [t.data_ptr() for t in rms_norm_weights],
                cos_sin_cache.data_ptr(), cos_sin_cache.shape[0], kv_slot_mapping.data_ptr(),
                kv_slot_mapping.numel(), [t.data_ptr() for t in kv_caches], kv_caches[0].shape[0],
                int(block_size), int(compress_ratio), float(rms_norm_eps), y_ptr, ws.data_ptr(),
                ws.numel(), int(flags), sp)
        else:
            name = "kvc_compress_layers_strided"
            st = kvc_compress_layers_strided(
                L, [t.data_ptr() for t in state_caches],
                KVC_DTYPE_F32 if s0.dtype == torch.float32 else KVC_DTYPE_BF16, s0.shape[0],
                s0.stride(0), s0.stride(1), token_to_req.data_ptr(), positions.data_ptr(),
                positions.numel(), boundary_token_indices.data_ptr(), N, block_table.data_ptr(),
                block_table.shape[0], block_table.shape[1], block_table.stride(0),
                block_table.stride(1), [t.data_ptr() for t in rms_norm_weights],
                cos_sin_cache.data_ptr(), cos_sin_cache.shape[0], kv_slot_mapping.data_ptr(),
                kv_slot_mapping.numel(), [t.data_ptr() for t in kv_caches], kv_caches[0].shape[0],
                int(block_size), int(compress_ratio), float(rms_norm_eps), y_ptr, ws.data_ptr(),
                ws.numel(), int(flags), sp)
    if st != KVC_OK:
        raise KvcError(st, name)
    return kv_caches
