"""Benchmark of the fused KV-cache window compressor on one GB300 (or N).

One step = one call of the whole operator (gather, window reduce, RMSNorm,
quantisation, RoPE, scatter) over the largest benchmark shape of the
KernelGen Challenge 8 write-up: 8 requests x 16384 tokens, compress_ratio
128, block_size 8 (1024 outputs, 256 MiB of bf16 state).  The line printed
is the operator's effective HBM bandwidth (algorithmic bytes / time).

Timing: inputs resident in HBM; the state is rotated over >= 3 copies whose
total size is several times the L2, so no call reads what the previous one
left in L2; the K timed launches are replayed from CUDA graphs and timed
with CUDA events on the launching stream, between device synchronisations
(and a barrier plus max over ranks under torchrun).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
                  [--no-sweep] [--no-e2e] [--no-cpu] [--state-layout L]
                  [--sweep-only [--shape NAME]] [--reader-only]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import platform
import re
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = ("µs/call and effective HBM GB/s (% of GB300 peak) over the 12 "
          "compress shapes")
HEADLINE = (8, 131072, 128)
L2_BYTES = 126 * 2 ** 20
ROTATE_MIN_BYTES = 3 * L2_BYTES


# ---- helpers shared with the multi-rank path (tested on CPU with gloo) -------

def dist_env():
    """(rank, world_size, local_rank) from the torchrun environment."""
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def rank_seed(base_seed: int, rank: int) -> int:
    """Each rank compresses its own, independent batch of requests."""
    return base_seed + 7919 * rank


def max_over_ranks(value: float, device=None) -> float:
    """Max of a float over all ranks (identity without a process group)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()):
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier():
    import torch.distributed as dist

    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# ---- measured peaks, profiles, clocks ------------------------------------------

def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


KERNEL_SOURCES = ("kvc_cluster.cu", "kvc_streamk.cu", "kvc_device.cuh", "kvc_internal.h")


def _code_only(text: str) -> str:
    """C++ source without comments and with whitespace collapsed, so that a
    comment edit does not orphan the ncu counters taken on the same code."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_hash() -> str:
    """Hash of the fused kernel's code (ties ncu counters to a kernel)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "kv_cache_compression_c128_gb300", "csrc")
    for f in KERNEL_SOURCES:
        with open(os.path.join(csrc, f), encoding="utf-8") as fh:
            h.update(f.encode() + b"\0" + _code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(layout: str = "bf16"):
    """DRAM bytes per launch from the committed ncu summary of the headline
    workload in `layout`, if it was taken on the current kernel sources
    (else None)."""
    tag = "" if layout == "bf16" else f"_{layout}"
    p = os.path.join(ROOT, "profiles", f"kvc_compress_headline{tag}_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    if d.get("kernel_source_hash") != kernel_source_hash():
        return None
    return d.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock / throttle samples (100 ms) around the timed region."""

    FIELDS = ("index,uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None):
        self.uuid = uuid
        self.samples = []
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [x.strip() for x in line.split(",")]))

    def mark(self, begin: bool):
        if begin:
            self.t0 = time.time()
        else:
            self.t1 = time.time()

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = [(t, r) for t, r in self.samples if len(r) >= 10]
        if self.uuid:
            mine = [(t, r) for t, r in rows if self.uuid in r[1]]
            rows = mine or rows
        inside = [r for t, r in rows if self.t0 - 0.1 <= t <= self.t1 + 0.1]
        if not inside and rows:  # timed region shorter than one sample period
            mid = 0.5 * (self.t0 + self.t1)
            inside = [min(rows, key=lambda tr: abs(tr[0] - mid))[1]]
        if not inside:
            return None

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(r[2]) for r in inside if num(r[2]) is not None]
        reasons = set()
        for r in inside:
            for name, col in (("hw_slowdown", 6), ("hw_thermal_slowdown", 7),
                              ("sw_thermal_slowdown", 8), ("sw_power_cap", 9)):
                if r[col].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": num(inside[0][3]), "samples": len(inside),
                "reasons": sorted(reasons),
                "power_w_max": max((num(r[4]) or 0.0) for r in inside)}


# ---- workload ------------------------------------------------------------------

def _tensors(case, device, copies):
    import torch

    states = []
    if copies > 0:
        st_host = torch.from_numpy(case.state_bits.view(np.int16)).view(torch.bfloat16)
        states = [st_host.to(device)]
        for _ in range(copies - 1):
            states.append(states[0].clone())
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(device)
    d = dict(token_to_req=t(case.token_to_req), positions=t(case.positions),
             boundary_token_indices=t(case.boundary_token_indices),
             block_table=t(case.block_table), rms_norm_weight=t(case.rms_norm_weight),
             cos_sin_cache=t(case.cos_sin_cache), kv_slot_mapping=t(case.kv_slot_mapping),
             kv_cache=t(case.kv_cache))
    return states, d


def _copies_for(case) -> int:
    b = case.state_bits.nbytes
    return max(3, -(-ROTATE_MIN_BYTES // b))


def time_device(kvc, case, device, steps: int, warmup: int, sampler=None,
                graph_chunk: int = 250, states=None, block_table=None, sync_ranks: bool = False):
    """Average seconds per call over `steps` graph-replayed launches.
    `states` (rotating state tensors, any layout) and `block_table` replace
    the case's own contiguous bf16 state and table when given.  With
    `sync_ranks` every rank must call it: the timed region starts and ends
    with a barrier (the headline); rank-0-only measurements leave it off."""
    import torch

    if states is None:
        copies = _copies_for(case)
        states, d = _tensors(case, device, copies)
    else:
        copies = len(states)
        _, d = _tensors(case, device, 0)
    if block_table is not None:
        d = dict(d, block_table=block_table)
    stream = torch.cuda.Stream(device)
    N = case.num_outputs
    ws = torch.zeros(kvc.kvc_workspace_bytes(N), dtype=torch.uint8, device=device)

    def call(i, s):
        kvc.c128_256_512_compress(states[i % copies], block_size=case.block_size,
                                  compress_ratio=case.compress_ratio,
                                  rms_norm_eps=case.rms_norm_eps, stream=s, workspace=ws, **d)

    with torch.cuda.stream(stream):
        for i in range(max(3, warmup)):
            call(i, stream)
    stream.synchronize()
    assert kvc.kvc_get_device_error(stream.cuda_stream) == 0
    # graphs of up to graph_chunk launches, rotating the state copies
    chunk = max(1, min(graph_chunk, steps))
    graphs = []
    remaining = steps
    pos = 0
    while remaining > 0:
        m = min(chunk, remaining)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(m):
                call(pos + i, stream)
        graphs.append(g)
        pos += m
        remaining -= m
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    # replay() launches on the current stream: make it the timed stream
    with torch.cuda.stream(stream):
        graphs[0].replay()                    # warm the graph path itself
        torch.cuda.synchronize(device)
        if sync_ranks:
            barrier()
        if sampler:
            sampler.mark(True)
        ev0.record(stream)
        for g in graphs:
            g.replay()
        ev1.record(stream)
        torch.cuda.synchronize(device)
    if sampler:
        sampler.mark(False)
    if sync_ranks:
        barrier()
    elapsed = ev0.elapsed_time(ev1) / 1e3
    assert kvc.kvc_get_device_error(stream.cuda_stream) == 0
    del graphs
    return elapsed / steps, elapsed


def time_distribution(kvc, case, device, iters: int = 200, warm: bool = False):
    """Per-call device times (CUDA events around every call, no graph): the
    median, p10 and p90 in microseconds.  Cold: the state rotates over
    copies larger than L2 together; warm: one copy, read again and again.
    A sleep kernel holds the stream while the host enqueues every call, so
    the GPU never waits for the host between them and each event pair
    brackets one kernel (the events also keep consecutive calls from
    overlapping, unlike the graph-replayed headline)."""
    import torch

    copies = 1 if warm else _copies_for(case)
    states, d = _tensors(case, device, copies)
    ws = torch.zeros(kvc.kvc_workspace_bytes(case.num_outputs), dtype=torch.uint8, device=device)
    stream = torch.cuda.Stream(device)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(iters)]
    with torch.cuda.stream(stream):
        for i in range(5):
            kvc.c128_256_512_compress(states[i % copies], block_size=case.block_size,
                                      compress_ratio=case.compress_ratio,
                                      rms_norm_eps=case.rms_norm_eps, stream=stream,
                                      workspace=ws, **d)
        stream.synchronize()
        torch.cuda._sleep(150000 * iters)  # ~75 us of SM clock per queued call
        for i in range(iters):
            ev[i][0].record(stream)
            kvc.c128_256_512_compress(states[i % copies], block_size=case.block_size,
                                      compress_ratio=case.compress_ratio,
                                      rms_norm_eps=case.rms_norm_eps, stream=stream,
                                      workspace=ws, **d)
            ev[i][1].record(stream)
        stream.synchronize()
    assert kvc.kvc_get_device_error(stream.cuda_stream) == 0
    t = np.array([a.elapsed_time(b) * 1e3 for a, b in ev])
    return {"shape": case.name, "l2": "warm" if warm else "cold", "calls": iters,
            "median_us": round(float(np.median(t)), 2), "p10_us": round(float(np.percentile(t, 10)), 2),
            "p90_us": round(float(np.percentile(t, 90)), 2)}


def time_reader(kvc, case, device, steps: int = 2000):
    """Per-call time of kvc_dequantize reading back every slot of `case`
    (fp32 and bf16 outputs), after one compression fills the cache."""
    import torch

    states, d = _tensors(case, device, 1)
    kvc.c128_256_512_compress(states[0], block_size=case.block_size,
                              compress_ratio=case.compress_ratio, **d)
    slots = torch.from_numpy(case.kv_slot_mapping[case.boundary_token_indices]).to(device)
    M = slots.numel()
    res = {}
    for name, dtype, width in (("f32", torch.float32, 4), ("bf16", torch.bfloat16, 2)):
        out = torch.empty((M, 512), dtype=dtype, device=device)
        stream = torch.cuda.Stream(device)
        with torch.cuda.stream(stream):
            for _ in range(5):
                kvc.dequantize(d["kv_cache"], slots, dtype=dtype, out=out, stream=stream)
            stream.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for _ in range(200):
                    kvc.dequantize(d["kv_cache"], slots, dtype=dtype, out=out, stream=stream)
            g.replay()
            torch.cuda.synchronize(device)
            ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            ev0.record(stream)
            for _ in range(max(1, steps // 200)):
                g.replay()
            ev1.record(stream)
            torch.cuda.synchronize(device)
        t = ev0.elapsed_time(ev1) / 1e3 / (max(1, steps // 200) * 200)
        b = M * (576 + 8 + 8) + M * 512 * width
        res[name] = {"us_per_call": round(t * 1e6, 3), "bytes": b, "gb_s": round(b / t / 1e9, 1)}
    assert kvc.kvc_get_device_error(torch.cuda.current_stream(device).cuda_stream) == 0
    res["large"] = time_reader_large(kvc, device)
    return {"slots": M, **res}


def time_reader_large(kvc, device, pages: int = 4096, reps: int = 20):
    """kvc_dequantize over a 262144-slot cache (4096 pages of seeded random
    bytes, 153 MB) read in a random slot order into fp32 and bf16 outputs:
    the reader at a size where bandwidth, not launch latency, decides."""
    import torch

    gen = torch.Generator(device=device).manual_seed(20260614)
    kv = torch.randint(0, 256, (pages, 64 * (576 + 8)), dtype=torch.uint8, device=device,
                       generator=gen)
    M = pages * 64
    slots = torch.randperm(M, device=device, generator=gen)
    res = {"slots": M}
    stream = torch.cuda.Stream(device)
    for name, dtype, width in (("f32", torch.float32, 4), ("bf16", torch.bfloat16, 2)):
        out = torch.empty((M, 512), dtype=dtype, device=device)
        with torch.cuda.stream(stream):
            for _ in range(3):
                kvc.dequantize(kv, slots, dtype=dtype, out=out, stream=stream)
            stream.synchronize()
            ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            ev0.record(stream)
            for _ in range(reps):
                kvc.dequantize(kv, slots, dtype=dtype, out=out, stream=stream)
            ev1.record(stream)
            stream.synchronize()
        t = ev0.elapsed_time(ev1) / 1e3 / reps
        b = M * (576 + 8 + 8) + M * 512 * width
        res[name] = {"us_per_call": round(t * 1e6, 2), "bytes": b, "gb_s": round(b / t / 1e9, 1)}
        del out
    assert kvc.kvc_get_device_error(stream.cuda_stream) == 0
    return res


def time_layers(kvc, case, device, L: int = 8, steps: int = 1000):
    """Per-call time of kvc_compress_layers over L layers of `case` (each
    layer its own state copy, weight and kv_cache; >= 3 rotating sets so the
    L * state bytes are not served from L2), against the per-call time of the
    single-layer call on the same shape."""
    import torch

    sets = max(3, -(-ROTATE_MIN_BYTES // (L * case.state_bits.nbytes)))
    states0, d = _tensors(case, device, 1)
    states = [[states0[0].clone() for _ in range(L)] for _ in range(sets)]
    weights = [d["rms_norm_weight"].clone() for _ in range(L)]
    kvs = [d["kv_cache"].clone() for _ in range(L)]
    ws = torch.zeros(kvc.kvc_workspace_bytes(case.num_outputs), dtype=torch.uint8, device=device)
    stream = torch.cuda.Stream(device)

    def call(i):
        kvc.compress_layers(states[i % sets], d["token_to_req"], d["positions"],
                            d["boundary_token_indices"], d["block_table"], weights,
                            d["cos_sin_cache"], d["kv_slot_mapping"], kvs, case.block_size,
                            case.compress_ratio, case.rms_norm_eps, stream=stream, workspace=ws)

    with torch.cuda.stream(stream):
        for i in range(5):
            call(i)
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        chunk = 100
        with torch.cuda.graph(g, stream=stream):
            for i in range(chunk):
                call(i)
        g.replay()
        torch.cuda.synchronize(device)
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = max(1, steps // chunk)
        ev0.record(stream)
        for _ in range(reps):
            g.replay()
        ev1.record(stream)
        torch.cuda.synchronize(device)
    assert kvc.kvc_get_device_error(stream.cuda_stream) == 0
    t = ev0.elapsed_time(ev1) / 1e3 / (reps * chunk)
    b = L * bytes_for(case)
    single, _ = time_device(kvc, case, device, 1000, 20)
    return {"shape": case.name, "layers": L, "us_per_call": round(t * 1e6, 3),
            "gb_s": round(b / t / 1e9, 1), "us_per_layer": round(t * 1e6 / L, 3),
            "single_layer_us_per_call": round(single * 1e6, 3),
            "speedup_vs_single_calls": round(L * single / t, 2)}


def time_e2e(kvc, case, device, steps: int, warmup: int):
    """Seconds per call through the public API from pinned host buffers:
    every step copies all of its inputs host->device, makes the call, and
    reads kv_cache back device->host, all inside the timed region.  Two
    device input sets alternate, so one step's copy-in runs on a copy
    stream while the previous step computes and copies out on the compute
    stream (each step waits for its own inputs; a buffer is refilled only
    after the step that used it has copied its result out)."""
    import torch

    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
    host = dict(state_cache=pin(case.state_bits.view(np.int16)).view(torch.bfloat16),
                token_to_req=pin(case.token_to_req), positions=pin(case.positions),
                boundary_token_indices=pin(case.boundary_token_indices),
                block_table=pin(case.block_table), rms_norm_weight=pin(case.rms_norm_weight),
                cos_sin_cache=pin(case.cos_sin_cache), kv_slot_mapping=pin(case.kv_slot_mapping),
                kv_cache=pin(case.kv_cache))
    devs = [{k: torch.empty_like(v, device=device) for k, v in host.items()} for _ in range(2)]
    outs = [torch.empty_like(host["kv_cache"]).pin_memory() for _ in range(2)]
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = outs[0].numel() * outs[0].element_size()
    copy_s = torch.cuda.Stream(device)
    comp_s = torch.cuda.Stream(device)
    ws = torch.zeros(kvc.kvc_workspace_bytes(case.num_outputs), dtype=torch.uint8, device=device)
    copied = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]

    def step(i):
        b = i % 2
        dev = devs[b]
        with torch.cuda.stream(copy_s):
            if i >= 2:
                copy_s.wait_event(done[b])
            for k in host:
                dev[k].copy_(host[k], non_blocking=True)
            copied[b].record(copy_s)
        with torch.cuda.stream(comp_s):
            comp_s.wait_event(copied[b])
            kvc.c128_256_512_compress(block_size=case.block_size,
                                      compress_ratio=case.compress_ratio,
                                      rms_norm_eps=case.rms_norm_eps, stream=comp_s,
                                      workspace=ws, **dev)
            outs[b].copy_(dev["kv_cache"], non_blocking=True)
            done[b].record(comp_s)

    for i in range(max(3, warmup)):
        step(i)
    torch.cuda.synchronize(device)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    barrier()
    ev0.record(copy_s)
    comp_s.wait_event(ev0)
    for i in range(steps):
        step(i)
    copy_s.wait_stream(comp_s)
    ev1.record(copy_s)
    torch.cuda.synchronize(device)
    elapsed = ev0.elapsed_time(ev1) / 1e3
    assert outs[0].shape == host["kv_cache"].shape
    return elapsed / steps, h2d, d2h


def time_oracle(case, max_outputs: int, min_seconds: float = 0.0, max_passes: int = 1):
    """Single-threaded oracle on the first `max_outputs` outputs of `case`,
    repeated (up to max_passes) until min_seconds have passed.  Returns
    (seconds, outputs computed in all passes)."""
    import oracle

    oracle.build()
    n = min(max_outputs, case.num_outputs)
    done = 0
    t0 = time.perf_counter()
    for _ in range(max(1, max_passes)):
        kv = case.kv_cache.copy()
        res = oracle.compress(case.state_bits, case.token_to_req, case.positions,
                              case.boundary_token_indices[:n], case.block_table,
                              case.rms_norm_weight, case.cos_sin_cache, case.kv_slot_mapping, kv,
                              case.block_size, case.compress_ratio, case.rms_norm_eps)
        assert res["status"] == 0
        done += n
        if time.perf_counter() - t0 >= min_seconds:
            break
    return time.perf_counter() - t0, done


def time_oracle_threads(case, threads: int, min_seconds: float = 10.0, max_passes: int = 60,
                        kv_out=None, max_outputs: int | None = None):
    """The same unchanged single-threaded oracle on `threads` host threads at
    once: thread i runs it on the i-th contiguous slice of the outputs (the
    ctypes call releases the GIL; slices write disjoint slots), all threads
    repeated until min_seconds have passed.  Returns (seconds, outputs
    computed in all passes); the last pass's kv_cache is appended to kv_out
    when given.  max_outputs: only the first that many outputs."""
    from concurrent.futures import ThreadPoolExecutor

    import oracle

    oracle.build()
    N = case.num_outputs if max_outputs is None else min(max_outputs, case.num_outputs)
    cuts = [N * i // threads for i in range(threads + 1)]

    def part(i, kv):
        res = oracle.compress(case.state_bits, case.token_to_req, case.positions,
                              case.boundary_token_indices[cuts[i]:cuts[i + 1]], case.block_table,
                              case.rms_norm_weight, case.cos_sin_cache, case.kv_slot_mapping, kv,
                              case.block_size, case.compress_ratio, case.rms_norm_eps)
        return res["status"]

    done = 0
    t0 = time.perf_counter()
    with ThreadPoolExecutor(max_workers=threads) as ex:
        for _ in range(max(1, max_passes)):
            kv = case.kv_cache.copy()
            assert all(st == 0 for st in ex.map(lambda i: part(i, kv), range(threads)))
            done += N
            if time.perf_counter() - t0 >= min_seconds:
                break
    dt = time.perf_counter() - t0
    if kv_out is not None:
        kv_out.append(kv)
    return dt, done


def bytes_for(case, n_outputs=None, elem_bytes: int = 2) -> int:
    """Algorithmic bytes of a call: state rows (1024 elements of elem_bytes),
    block-table entries (one per 8-row chunk of the window, two where a
    chunk straddles blocks; counted as one), per-output metadata, one
    cos/sin row, the weights, the slot."""
    n = case.num_outputs if n_outputs is None else n_outputs
    c = case.compress_ratio
    return (n * c * 1024 * elem_bytes + n * (-(-c // 8)) * 4 + n * 28 + n * 256 + 2048
            + n * 584)


# Other layouts of the headline state: name -> (bytes per element, kind).
LAYOUTS = {
    "bf16": (2, "contiguous bf16"),
    "fp32_contiguous": (4, "fp32 elements (the seeded bf16 values widened), contiguous"),
    "bf16_rows_64_apart": (2, "bf16 rows 1088 elements apart: one TMA tensor copy per 8-row chunk"),
    "bf16_blocks_512_apart_colmajor_table": (
        2, "bf16 blocks 8*1024+512 elements apart, column-major block table"),
}


def layout_states(case, name, device, copies):
    """`copies` device state tensors holding the case's values in layout
    `name` (every element outside the rows is NaN), and the block table to
    pass with them (None: the case's own row-major table)."""
    import torch

    from kv_cache_compression_c128_gb300 import inputs

    G, B = case.num_state_blocks, case.block_size
    R, M = case.block_table.shape
    bits = torch.from_numpy(case.state_bits.view(np.int16)).view(torch.bfloat16).to(device)

    def embedded(src, rs, bs):
        size = (G - 1) * bs + (B - 1) * rs + 1024
        flat = torch.full((size,), float("nan"), dtype=src.dtype, device=device)
        view = flat.as_strided((G, B, 1024), (bs, rs, 1))
        view.copy_(src)
        return view

    table = None
    if name == "bf16":
        make = lambda: bits.clone()
    elif name == "fp32_contiguous":
        make = lambda: bits.float()
    elif name == "bf16_rows_64_apart":
        make = lambda: embedded(bits, 1088, 8 * 1088)
    elif name == "bf16_blocks_512_apart_colmajor_table":
        make = lambda: embedded(bits, 1024, 8 * 1024 + 512)
        table = torch.from_numpy(inputs.strided_table(case.block_table, 1, R)).to(device)
        table = table.as_strided((R, M), (1, R))
    else:
        raise ValueError(f"unknown state layout {name}")
    states = [make() for _ in range(copies)]
    del bits
    return states, table


def time_layouts(kvc, device, peak: float, steps: int = 600):
    """The headline shape with the state in the other layouts of LAYOUTS
    (fp32 elements; bf16 rows apart; padded bf16 blocks with a column-major
    table), each built on the device from the case's seeded values, three
    rotating copies (> L2)."""
    from kv_cache_compression_c128_gb300 import inputs

    case = inputs.headline_case()
    out = []
    for name, (eb, _) in LAYOUTS.items():
        if name == "bf16":
            continue
        states, table = layout_states(case, name, device, 3)
        t, _ = time_device(kvc, case, device, steps, 20, states=states, block_table=table)
        b = bytes_for(case, elem_bytes=eb)
        dt = kvc.KVC_DTYPE_F32 if eb == 4 else kvc.KVC_DTYPE_BF16
        ctas, clu, _, _ = kvc.kvc_query_launch_ex(case.num_outputs, case.compress_ratio, dt)
        out.append({"layout": name, "shape": case.name, "bytes": b, "ctas": ctas,
                    "cluster_size": clu, "us_per_call": round(t * 1e6, 3),
                    "gb_s": round(b / t / 1e9, 1), "pct_of_peak": round(100 * b / t / 1e9 / peak, 1)})
        del states
    return out


def windows_overlap(case) -> bool:
    """Whether two windows of `case` share a row of the same request."""
    b = case.boundary_token_indices
    r = case.token_to_req[b].astype(np.int64)
    p = case.positions[b]
    order = np.lexsort((p, r))
    r, p = r[order], p[order]
    same = r[1:] == r[:-1]
    return bool(np.any(same & (p[1:] - p[:-1] < case.compress_ratio)))


def run_sweep(kvc, inputs, device, peak: float, steps=None, warmup: int = 20,
              detail: bool = False, only: str | None = None):
    """The 12 benchmark shapes, the 3 ragged variants, the general-window
    headline and the headline with block_size 16, each timed like the
    headline (steps: 2000 for the small states, 600 for the large ones,
    unless given).  With `detail`, each shape also gets its per-call
    distribution (100 calls, L2 cold and warm) and one single-threaded
    oracle pass on the host.  `only`: time just the shape of that name."""
    out = []
    makers = ([lambda i=i: inputs.bench_case(i) for i in range(12)]
              + [lambda c=c: inputs.ragged_case(c) for c in (128, 256, 512)]
              + [lambda: inputs.general_window_case(128, 16), inputs.block16_case])
    for make in makers:
        cs = make()
        if only is not None and cs.name != only:
            continue
        n_steps = steps or (2000 if cs.state_bits.nbytes < 100 * 2 ** 20 else 600)
        tc, _ = time_device(kvc, cs, device, n_steps, warmup)
        b = bytes_for(cs)
        sctas, sclu, _, _ = kvc.kvc_query_launch(cs.num_outputs, cs.compress_ratio)
        row = {"shape": cs.name, "outputs": cs.num_outputs, "bytes": b,
               "ctas": sctas, "cluster_size": sclu,
               "us_per_call": round(tc * 1e6, 3)}
        if windows_overlap(cs):
            # L2 serves the rows that several windows share, so bytes / time
            # is not a DRAM rate and has no place against the HBM peak
            row.update({"window_rows_gb_s": round(b / tc / 1e9, 1), "pct_of_peak": None,
                        "note": "windows overlap: the rate counts window rows, not DRAM "
                                "bytes (L2 serves the shared rows), so it is not compared "
                                "with the HBM peak"})
        else:
            row.update({"gb_s": round(b / tc / 1e9, 1),
                        "pct_of_peak": round(100 * b / tc / 1e9 / peak, 1)})
        if detail:
            cold = time_distribution(kvc, cs, device, 100)
            warm = time_distribution(kvc, cs, device, 100, warm=True)
            row["cold_us"] = {k: cold[k] for k in ("median_us", "p10_us", "p90_us")}
            row["warm_us"] = {k: warm[k] for k in ("median_us", "p10_us", "p90_us")}
            dt, _ = time_oracle(cs, cs.num_outputs)
            row["oracle_ms_1_core"] = round(dt * 1e3, 1)
        out.append(row)
        del cs
    return out


def workload_config(case, state_layout: str = "bf16", n_copies: int | None = None) -> dict:
    """The `config` object of the JSON line: the workload alone, the same in
    both arms (how each arm runs it goes under `run`)."""
    R, T, C = case.num_reqs, case.total_tokens, case.compress_ratio
    eb = LAYOUTS[state_layout][0]
    copies = n_copies if n_copies is not None else _copies_for(case)
    return {"workload": f"{R} reqs x {T // R} tokens, compress_ratio {C}, block_size "
                        f"{case.block_size} ({case.num_outputs} outputs)",
            "num_reqs": R, "total_tokens": T, "compress_ratio": C,
            "block_size": case.block_size, "outputs": case.num_outputs,
            "state_layout": f"{state_layout}: {LAYOUTS[state_layout][1]}",
            "algorithmic_bytes_per_call": bytes_for(case, elem_bytes=eb),
            "l2": f"GPU arm: the state rotates over {copies} copies "
                  f"({copies * case.state_bits.nbytes * eb // 2 >> 20} MiB > L2) between "
                  f"calls; CPU arm: host memory"}


# ---- main ------------------------------------------------------------------------

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["kvc", "reference"], default="kvc")
    ap.add_argument("--no-sweep", action="store_true",
                    help="time the headline only: no shape sweep, reader, layers or layouts")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--sweep-only", action="store_true",
                    help="time only the shape sweep, --steps launches per shape (for ncu)")
    ap.add_argument("--shape", default=None,
                    help="with --sweep-only: time only the sweep shape of this name")
    ap.add_argument("--reader-only", action="store_true",
                    help="time only the reader (kvc_dequantize) calls (for ncu)")
    ap.add_argument("--state-layout", choices=sorted(LAYOUTS), default="bf16",
                    help="layout of the timed headline state (default: contiguous bf16)")
    args = ap.parse_args()
    rank, world, local_rank = dist_env()
    from kv_cache_compression_c128_gb300 import inputs

    R, T, C = HEADLINE
    workload = f"{R} reqs x {T // R} tokens, compress_ratio {C}, block_size 8 ({T // C} outputs)"

    if args.impl == "reference":
        if rank != 0:
            return
        run_reference(args, inputs, workload)
        return

    import torch

    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    device = torch.device("cuda", local_rank if world > 1 else 0)
    torch.cuda.set_device(device)
    import kv_cache_compression_c128_gb300 as kvc

    # one rank compiles (if the library is out of date); the others then load it
    if rank == 0:
        kvc.build()
    barrier()
    kvc.build()
    if args.sweep_only:
        peak, _ = measured_peaks()
        print(json.dumps({"sweep": run_sweep(kvc, inputs, device, peak, args.steps,
                                             args.warmup, only=args.shape)}))
        return
    if args.reader_only:
        print(json.dumps({"reader": time_reader(kvc, inputs.headline_case(), device)}))
        return
    case = inputs.make_case(R, T, C, seed=rank_seed(inputs.BASE_SEED + inputs.BENCH_SHAPES.index(HEADLINE), rank),
                            name="headline")
    elem_bytes = LAYOUTS[args.state_layout][0]
    per_call_bytes = bytes_for(case, elem_bytes=elem_bytes)
    states = table = None
    if args.state_layout != "bf16":
        states, table = layout_states(case, args.state_layout, device,
                                      max(3, -(-ROTATE_MIN_BYTES // (case.state_bits.nbytes
                                                                   * elem_bytes // 2))))
    props = torch.cuda.get_device_properties(device)
    uuid = str(getattr(props, "uuid", "") or "")
    sampler = ClockSampler(uuid.replace("GPU-", "") if uuid else None)
    sampler.start()
    time.sleep(0.3)
    t_call, t_total = time_device(kvc, case, device, args.steps, args.warmup, sampler,
                                  states=states, block_table=table, sync_ranks=True)
    n_copies = len(states) if states is not None else _copies_for(case)
    del states, table
    clocks = sampler.stop()
    t_max = max_over_ranks(t_total, device if world > 1 else None)
    ms_per_step = t_max / args.steps * 1e3
    value = world * per_call_bytes * args.steps / t_max / 1e9
    peak, peak_kind = measured_peaks()
    achieved = per_call_bytes / t_call / 1e9
    f32 = elem_bytes == 4
    ctas, cluster, threads, smem = kvc.kvc_query_launch_ex(
        case.num_outputs, C, kvc.KVC_DTYPE_F32 if f32 else kvc.KVC_DTYPE_BF16)

    e2e = None
    if not args.no_e2e and args.state_layout == "bf16":
        e_steps = max(3, min(50, args.steps))
        t_e2e, h2d, d2h = time_e2e(kvc, case, device, e_steps, 3)
        t_e2e = max_over_ranks(t_e2e, device if world > 1 else None)
        e2e = {"value": round(world * per_call_bytes / t_e2e / 1e9, 3), "unit": "GB/s",
               "us_per_call": round(t_e2e * 1e6, 2), "steps": e_steps,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}

    extras = rank == 0 and not args.no_sweep
    # NVTX ranges name each part, so that ncu can capture one of them alone
    # (--nvtx --nvtx-include "reader/")
    nvtx = torch.cuda.nvtx
    reader = layers = layouts = None
    if extras:
        nvtx.range_push("reader")
        reader = time_reader(kvc, case, device)
        nvtx.range_pop()
        nvtx.range_push("layers")
        layers = time_layers(kvc, inputs.bench_case(0), device, 8)
        nvtx.range_pop()
        nvtx.range_push("layouts")
        layouts = time_layouts(kvc, device, peak)
        nvtx.range_pop()
    distribution = None
    isolated = None
    if rank == 0 and args.state_layout == "bf16":
        isolated = time_distribution(kvc, case, device)
    if extras:
        small = inputs.bench_case(0)
        distribution = [isolated, time_distribution(kvc, small, device),
                        time_distribution(kvc, small, device, warm=True)]

    sweep = (run_sweep(kvc, inputs, device, peak, detail=not args.no_cpu)
             if not args.no_sweep and rank == 0 else None)

    cpu = cpu_all = None
    if not args.no_cpu and rank == 0 and world >= 1:
        dt, n = time_oracle(case, case.num_outputs, min_seconds=10.0, max_passes=60)
        cpu = {"value": round(bytes_for(case, n) / dt / 1e9, 4), "unit": "GB/s", "cores": 1,
               "kind": "oracle",
               "sample": f"all {case.num_outputs} outputs of the headline workload, "
                         f"{n // case.num_outputs} passes ({dt:.1f} s), single-threaded C "
                         f"(float64 reduce) on one of {os.cpu_count()} "
                         f"{platform.machine()} host cores"}
        nthr = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
        dt_a, n_a = time_oracle_threads(case, nthr)
        cpu_all = {"value": round(bytes_for(case, n_a) / dt_a / 1e9, 4), "unit": "GB/s",
                   "cores": nthr, "kind": "oracle",
                   "sample": f"all {case.num_outputs} outputs of the headline workload, "
                             f"{n_a // case.num_outputs} passes ({dt_a:.1f} s), the same "
                             f"single-threaded C oracle on {nthr} threads at once, each on "
                             f"its own slice of the outputs"}

    if rank != 0:
        return
    traffic = profiled_traffic(args.state_layout)
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 6),
        "us_per_call": round(ms_per_step * 1e3, 3),
        "pct_of_peak": round(100 * value / world / peak, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32" if f32 else "bf16",
        "data": "synthetic: seeded N(0,1) bf16 state, random block permutation, "
                "1+0.1N(0,1) weights, RoPE theta 10000, permuted slots",
        "config": workload_config(case, args.state_layout, n_copies),
        "run": {"timing": "CUDA graphs of <=250 launches, CUDA events on the launching "
                          "stream; consecutive launches overlap (programmatic dependent "
                          "launch: each launch's first reads start in the previous one's "
                          "tail), so ms_per_step is back-to-back throughput; "
                          "roofline.frac_isolated is the per-call figure",
                "launch": {"ctas": ctas, "cluster_size": cluster, "threads": threads,
                           "smem_bytes": smem, "route": "cluster" if cluster else "stream-k"},
                "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "frac_basis": "back to back: bytes / graph-replayed time per launch "
                                   "(consecutive launches overlap)",
                     "frac_isolated": (round(per_call_bytes / (isolated["median_us"] * 1e-6)
                                             / 1e9 / peak, 4) if isolated else None),
                     "isolated_median_us": isolated["median_us"] if isolated else None,
                     "frac_isolated_basis": "per call: bytes / median of 200 calls each timed "
                                            "alone (L2 cold, nothing overlaps)",
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_kind == "measured" else "fallback 6.8 TB/s",
                     "traffic": traffic,
                     "kernel": (f"kvc_cluster_kernel<{cluster}, {'true' if f32 else 'false'}, "
                                f"{'true' if args.state_layout == 'bf16_rows_64_apart' else 'false'}>"
                                if cluster else "kvc_streamk_kernel"),
                     "algorithmic_bytes_per_launch": per_call_bytes},
        "gpu_launches": args.steps,
        "clocks": clocks,
        "e2e": e2e,
        "reader": reader,
        "layers": layers,
        "layouts": layouts,
        "distribution": distribution,
        "cpu_baseline": cpu,
        "cpu_baseline_all_cores": cpu_all,
        "sweep": sweep,
        "kernel_source_hash": kernel_source_hash(),
    }
    print(json.dumps(line))


def run_reference(args, inputs, workload):
    """The reference arm: the CPU oracle, as it stands, on the host cores."""
    R, T, C = HEADLINE
    case = inputs.make_case(R, T, C, seed=inputs.BASE_SEED + inputs.BENCH_SHAPES.index(HEADLINE),
                            name="headline")
    # every host thread runs the unchanged single-threaded oracle on its own
    # slice of a step's outputs; each step's sample is sized so that the
    # whole run takes about a minute
    nthr = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    dt1, n1 = time_oracle_threads(case, nthr, min_seconds=0.0, max_passes=1,
                                  max_outputs=8 * nthr)
    per_output = dt1 / n1
    n_sample = int(max(nthr, min(case.num_outputs, 60.0 / max(1, args.steps) / per_output)))
    for _ in range(max(0, min(args.warmup, 1))):
        time_oracle_threads(case, nthr, min_seconds=0.0, max_passes=1, max_outputs=n_sample)
    tot = 0.0
    n = 0
    for _ in range(args.steps):
        dt, n = time_oracle_threads(case, nthr, min_seconds=0.0, max_passes=1,
                                    max_outputs=n_sample)
        tot += dt
    per = tot / max(1, args.steps)
    value = bytes_for(case, n) / per / 1e9
    sample = (f"each step: first {n} of the {case.num_outputs} outputs of the headline "
              f"workload, the unchanged single-threaded C oracle (float64 reduce) on {nthr} "
              f"host threads at once, each on its own slice of the outputs")
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(per * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(case),
            "run": {"timing": "host wall clock (time.perf_counter) around each step",
                    "parallelism": f"{nthr} host threads"},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": nthr,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


if __name__ == "__main__":
    main()
