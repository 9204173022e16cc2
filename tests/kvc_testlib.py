"""Helpers shared by the tests: a brute-force decoder of the packed kv_cache
slot layout and bf16 conversions through torch (a library routine).

Layout ("Gather and Scatter" and "How One Output Is Produced" of the
KernelGen Challenge 8 write-up): a page holds 64 slots; slot ``off`` of page
``pg`` keeps 576 payload bytes at ``[pg, off*576]`` -- 448 int8 NOPE codes then
64 little-endian bf16 RoPE values -- and 8 scale bytes at
``[pg, 64*576 + off*8]``: 7 exponent bytes ``e + 127`` and one padding byte.
"""
from __future__ import annotations

import numpy as np
import torch

PAGE_SLOTS = 64
TOKEN_STRIDE = 576
SCALE_DIM = 8
PAGE_BYTES = PAGE_SLOTS * (TOKEN_STRIDE + SCALE_DIM)
SCALE_BASE = PAGE_SLOTS * TOKEN_STRIDE


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def torch_bf16_bits(x: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def slot_byte_ranges(slot: int):
    """(payload_start, scale_start) flat byte offsets of ``slot`` in kv_cache."""
    pg, off = divmod(int(slot), PAGE_SLOTS)
    return pg * PAGE_BYTES + off * TOKEN_STRIDE, pg * PAGE_BYTES + SCALE_BASE + off * SCALE_DIM


def decode_slot(kv: np.ndarray, slot: int):
    """Read one slot back: (q int8[448], e int[7], pad byte, rope f32[64])."""
    flat = kv.reshape(-1)
    p0, s0 = slot_byte_ranges(slot)
    payload = flat[p0:p0 + TOKEN_STRIDE]
    scale = flat[s0:s0 + SCALE_DIM]
    q = payload[:448].view(np.int8).astype(np.int64)
    e = scale[:7].astype(np.int64) - 127
    rope_bits = payload[448:].copy().view("<u2")
    return q, e, int(scale[7]), bf16_bits_to_f32(rope_bits)


def dequant(q: np.ndarray, e: np.ndarray) -> np.ndarray:
    """NOPE values back from codes: q * 2^e, per 64-dim group (float64)."""
    return q.astype(np.float64) * np.repeat(np.ldexp(1.0, e), 64)


def written_mask(kv_shape, slots) -> np.ndarray:
    """Boolean mask (flat) of the bytes owned by the given slots."""
    m = np.zeros(int(np.prod(kv_shape)), dtype=bool)
    for s in slots:
        if s < 0:
            continue
        p0, s0 = slot_byte_ranges(s)
        m[p0:p0 + TOKEN_STRIDE] = True
        m[s0:s0 + SCALE_DIM] = True
    return m


def slots_of_case(case) -> np.ndarray:
    """Slot written by each output n (kv_slot_mapping indexed by token)."""
    return case.kv_slot_mapping[case.boundary_token_indices]


def gather_window_rows(case) -> np.ndarray:
    """The page's baseline gather: flat row ids [N, C] through block_table.

    Restates "The Baseline" (flat_idx = block_numbers * block_size +
    block_offsets) in numpy, for the torch cross-check of the reduction.
    """
    B, C = case.block_size, case.compress_ratio
    b = case.boundary_token_indices
    r = case.token_to_req[b].astype(np.int64)
    p = case.positions[b]
    t = p[:, None] - C + 1 + np.arange(C)[None, :]
    blk = case.block_table[r[:, None], t // B].astype(np.int64)
    return blk * B + t % B


# ---- running a case through the CUDA library (GPU tests) --------------------

def to_device(case, device="cuda"):
    """The case's arrays as torch tensors on `device` (kv_cache copied)."""
    st = torch.from_numpy(case.state_bits.view(np.int16)).view(torch.bfloat16)
    return dict(
        state_cache=st.to(device),
        token_to_req=torch.from_numpy(case.token_to_req).to(device),
        positions=torch.from_numpy(case.positions).to(device),
        boundary_token_indices=torch.from_numpy(case.boundary_token_indices).to(device),
        block_table=torch.from_numpy(case.block_table).to(device),
        rms_norm_weight=torch.from_numpy(case.rms_norm_weight).to(device),
        cos_sin_cache=torch.from_numpy(case.cos_sin_cache).to(device),
        kv_slot_mapping=torch.from_numpy(case.kv_slot_mapping).to(device),
        kv_cache=torch.from_numpy(case.kv_cache.copy()).to(device),
    )


def run_gpu(case, flags=0, dev_arrays=None, slot_mapping=None):
    """Run the CUDA library on a case; returns (kv np, y np, device error)."""
    import kv_cache_compression_c128_gb300 as kvc

    d = dev_arrays if dev_arrays is not None else to_device(case)
    if slot_mapping is not None:
        d = dict(d, kv_slot_mapping=torch.from_numpy(slot_mapping).to(d["kv_cache"].device))
    N = case.num_outputs
    y = torch.full((max(N, 1), 512), float("nan"), dtype=torch.float32, device=d["kv_cache"].device)
    kvc.c128_256_512_compress(block_size=case.block_size, compress_ratio=case.compress_ratio,
                              rms_norm_eps=case.rms_norm_eps, y_out=y, flags=flags, **d)
    err = kvc.kvc_get_device_error(torch.cuda.current_stream().cuda_stream)
    return d["kv_cache"].cpu().numpy(), y[:N].cpu().numpy(), err


# ---- the parity bar (see tests/test_gpu_parity.py for its statement) -----------

Y_RTOL = 2e-3
Y_ATOL_RMS = 1e-5


def _y_ok(y_gpu, y_ref):
    rms = np.sqrt((y_ref.astype(np.float64) ** 2).mean(1, keepdims=True))
    err = np.abs(y_gpu.astype(np.float64) - y_ref)
    return np.all(err <= Y_RTOL * np.abs(y_ref) + Y_ATOL_RMS * rms), float(
        (err / (np.abs(y_ref) + rms)).max())


def assert_parity(oracle_mod, case, kv_g, y_g, ref=None):
    """The three-way parity bar between GPU results (kv bytes, y) and the
    oracle on `case`: y within 2e-3 relative; kv bytes bit-exact against the
    oracle's finalizer applied to the GPU's y; against the oracle's own bytes
    within one quantisation step / one scale step / a bf16 ulp plus the y
    tolerance, every other byte untouched.  `ref` = (kv, result dict) of an
    oracle run already made (e.g. on an fp32 or strided state); default: the
    oracle on the case's own bf16 state.  Returns stats."""
    kv_o, res = oracle_mod.compress_case(case) if ref is None else ref
    assert res["status"] == 0
    ok, worst = _y_ok(y_g, res["y"])
    assert ok, f"y outside 2e-3 relative (worst scaled error {worst:.3g})"

    # (2) bytes exactly determined by the GPU's y
    kv_y = case.kv_cache.copy()
    oracle_mod.quant_rope_scatter(y_g, case.positions, case.boundary_token_indices,
                                  case.compress_ratio, case.cos_sin_cache,
                                  case.kv_slot_mapping, kv_y)
    if not np.array_equal(kv_g, kv_y):
        bad = np.nonzero(kv_g.reshape(-1) != kv_y.reshape(-1))[0]
        raise AssertionError(f"{bad.size} bytes differ from oracle(y_gpu); first at {bad[:8]}")

    # (3) against the oracle's own bytes
    slots = slots_of_case(case)
    m = written_mask(kv_g.shape, slots)
    assert np.array_equal(kv_g.reshape(-1)[~m], kv_o.reshape(-1)[~m])
    assert np.array_equal(kv_g.reshape(-1)[~m], case.kv_cache.reshape(-1)[~m])
    n_code_diff = 0
    y_rms = np.sqrt((res["y"].astype(np.float64) ** 2).mean(1))
    for n, s in enumerate(slots):
        if s < 0:
            continue
        qg, eg, pg, rg = decode_slot(kv_g, s)
        qo, eo, po, ro = decode_slot(kv_o, s)
        assert pg == 0 and po == 0
        assert np.all(np.abs(eg - eo) <= 1)
        step = np.maximum(np.repeat(np.ldexp(1.0, eg), 64), np.repeat(np.ldexp(1.0, eo), 64))
        assert np.all(np.abs(dequant(qg, eg) - dequant(qo, eo)) <= step)
        mag = np.maximum(np.abs(ro), np.abs(rg))
        ulp = np.ldexp(1.0, np.frexp(np.maximum(mag, 1e-30))[1] - 8)
        pair = np.repeat(np.hypot(res["y"][n, 448::2], res["y"][n, 449::2]), 2)
        tol = ulp + Y_RTOL * pair + 1.5 * Y_ATOL_RMS * y_rms[n]
        assert np.all(np.abs(rg.astype(np.float64) - ro) <= tol)
        n_code_diff += int(np.sum(qg != qo))
    # differing codes come only from y values within rounding of a code edge
    assert n_code_diff <= max(8, 2e-3 * 448 * max(1, case.num_outputs))
    return {"worst_y": worst, "code_diff": n_code_diff}


