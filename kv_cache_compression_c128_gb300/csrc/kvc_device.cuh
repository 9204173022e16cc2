// Device-side building blocks shared by the two kernels of the KV-cache
// window compressor (kvc_streamk.cu, kvc_cluster.cu): PTX wrappers for
// mbarriers, bulk copies and cluster shared memory, the per-dimension online
// softmax fold, block-table resolution, and the finaliser (RMSNorm, NOPE
// quantisation, RoPE, slot store) of "How One Output Is Produced" in the
// KernelGen Challenge 8 write-up, with the byte rules of its section "The
// Finalizer's Sharp Edges".
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "kvc_internal.h"

namespace kvc {
namespace dev {

constexpr uint32_t kErrUnsupported = 2;
constexpr uint32_t kErrBadIndex = 4;
constexpr uint32_t kErrTimeout = 5;
constexpr long long kWaitLimitCycles = kDefaultWaitLimitCycles;
constexpr float kLog2e = 1.4426950408889634f;

// Slot record of one output piece, handed from the copy-issuing warp to the
// consumer warps through shared memory.
struct alignas(16) MetaRec {
  long long slot;  // destination slot (< 0: do not write)
  long long pc;    // compressed position (< 0: invalid output)
};

// ---- PTX wrappers -------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(unsigned long long* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(unsigned long long* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(unsigned long long* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

// Raise the barrier's expected transaction bytes without arriving (a stage
// filled by several copies announces each one; the last arrives).
__device__ __forceinline__ void mbar_expect_tx(unsigned long long* bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(unsigned long long* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Non-blocking probe of the phase of `bar` with the given parity.
__device__ __forceinline__ bool mbar_test_wait(unsigned long long* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Limits below this many cycles are polled with test_wait and the clock read
// after every probe: a try_wait may suspend the thread for a hardware-chosen
// time that can exceed such a limit.  (Only the test hook that shortens the
// pipeline waits asks for limits this short.)
constexpr long long kPollBelowCycles = 100000;

// Wait for the phase of `bar` with the given parity; false once more than
// `limit` SM clock cycles have passed.
static __device__ __noinline__ bool mbar_wait_bounded_for(unsigned long long* bar, uint32_t parity,
                                                          long long limit) {
  if (limit < kPollBelowCycles) {
    const long long t0 = clock64();
    while (!mbar_test_wait(bar, parity))
      if (clock64() - t0 > limit) return false;
    return true;
  }
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (clock64() - t0 > limit) return false;
  }
}

// A pipeline wait (a stage, a FIFO half): bounded by the call's limit
// (Params::wait_limit; kWaitLimitCycles unless a test shortened it).
__device__ __forceinline__ bool mbar_wait_bounded(unsigned long long* bar, uint32_t parity,
                                                  long long limit) {
  return mbar_wait_bounded_for(bar, parity, limit);
}

// The final drain of a CTA's own bulk copies always takes the long limit: a
// CTA must not exit while a copy may still write into its shared memory, and
// a copy of valid addresses always lands.
__device__ __forceinline__ bool mbar_wait_drain(unsigned long long* bar, uint32_t parity) {
  return mbar_wait_bounded_for(bar, parity, kWaitLimitCycles);
}

// As mbar_wait_bounded, with cluster-scope acquire: for barriers completed by
// other CTAs of the cluster (remote stores with complete_tx).
__device__ __forceinline__ bool mbar_try_wait_cluster(unsigned long long* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

static __device__ __noinline__ bool mbar_wait_cluster_bounded(unsigned long long* bar,
                                                              uint32_t parity) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait_cluster(bar, parity)) return true;
    if (clock64() - t0 > kWaitLimitCycles) return false;
  }
}

__device__ __forceinline__ uint64_t evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// One tensor copy global -> shared through the 4-D map `map` (a generic
// address of a CUtensorMap in parameter space): the box at element
// coordinates (0, 0, row, block), completing on `bar` as tx bytes.  `dst`
// 128-byte aligned.
__device__ __forceinline__ void tensor_copy_g2s(void* dst, const void* map, int row, int block,
                                                unsigned long long* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(smem_addr(dst)),
      "l"(map), "r"(0), "r"(0), "r"(row), "r"(block), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// The same box prefetched into L2.
__device__ __forceinline__ void tensor_prefetch_l2(const void* map, int row, int block) {
  asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];" ::"l"(map),
               "r"(0), "r"(0), "r"(row), "r"(block)
               : "memory");
}

// Bulk prefetch of `bytes` (a multiple of 16) into L2 from a 16-byte aligned
// global address.  It moves no data into the SM and completes on nothing.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// One bulk (1-D) copy global -> shared, completing on `bar` as tx bytes.
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes,
                                              unsigned long long* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// Named barrier 1 over the 256 consumer threads (the other warps never join).
__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumerThreads) : "memory");
}

// OR of `v` over the consumer threads (also a consumer barrier).
__device__ __forceinline__ bool consumer_any(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, 1, %2, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v)), "n"(kConsumerThreads)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void record_error(uint32_t* err, uint32_t code) { atomicCAS(err, 0u, code); }

// ---- cluster shared memory ----------------------------------------------------

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Shared-memory address of `local` (this CTA) in the CTA of cluster rank r.
__device__ __forceinline__ uint32_t peer_addr(uint32_t local, uint32_t r) {
  uint32_t a;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(local), "r"(r));
  return a;
}

// Remote stores into another CTA's shared memory that complete `bytes` of
// transaction count on that CTA's mbarrier once the data is visible there.
__device__ __forceinline__ void st_async_f2(uint32_t remote, float x, float y, uint32_t remote_bar) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];" ::"r"(remote),
      "f"(x), "f"(y), "r"(remote_bar)
      : "memory");
}

__device__ __forceinline__ void st_async_f32(uint32_t remote, float x, uint32_t remote_bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.f32 [%0], %1, [%2];" ::"r"(remote),
               "f"(x), "r"(remote_bar)
               : "memory");
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

// The two halves of a cluster barrier, for a thread that has work to do in
// between.  Every thread of the cluster arrives once, then waits once,
// before it arrives again.  The relaxed arrive publishes mbarrier
// initialisation when fence_mbar_init() came before it.
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire;" ::: "memory");
}

// ---- bf16 and float helpers -----------------------------------------------------

__device__ __forceinline__ uint32_t bf16x2_max(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ float fast_ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ unsigned long long pack2(float a, float b) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}

__device__ __forceinline__ void unpack2(unsigned long long r, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}

__device__ __forceinline__ unsigned long long fma2(unsigned long long a, unsigned long long b,
                                                   unsigned long long c) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

__device__ __forceinline__ unsigned long long add2(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// ceil(log2(a / 127)) for a finite, normal a > 0, exactly: with a = m 2^E,
// m in [1, 2), 127 * 2^e >= a  <=>  e >= E + log2(m / 127), and
// log2(m / 127) lies in (-7, -5]; it exceeds -6 exactly when m > 127/64,
// i.e. when the 23-bit mantissa field exceeds 0x7E0000.
__device__ __forceinline__ int scale_exponent(float a) {
  const uint32_t bits = __float_as_uint(a);
  const int e_a = static_cast<int>(bits >> 23) - 127;
  return e_a - 6 + ((bits & 0x7FFFFFu) > 0x7E0000u ? 1 : 0);
}

__device__ __forceinline__ uint32_t bf16_bits_rn(float x) {
  return static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(x)));
}

// ---- online softmax over the window -----------------------------------------------

struct SoftmaxState {
  float m0, m1, d0, d1, a0, a1;  // running max, denominator, numerator (2 dims)
};

__device__ __forceinline__ void state_reset(SoftmaxState& s) {
  s.m0 = s.m1 = -INFINITY;
  s.d0 = s.d1 = s.a0 = s.a1 = 0.f;
}

// Fold kRows consecutive staged rows (each [512 values | 512 scores] bf16,
// 2 KiB apart) into thread t's dimensions 2t, 2t+1: the rows' score maximum
// (bf16x2, exact) rescales the running state once, then every row adds
// exp(s - m) to the denominator and exp(s - m) * v to the numerator (packed
// f32x2 arithmetic; exp as ex2 of a log2e-scaled argument).  kRows = 8 is
// one chunk; 16 is a stage of two full chunks, which share one rescale.
template <int kRows>
__device__ __forceinline__ void fold_rows_n(const uint8_t* blk, int t, SoftmaxState& s) {
  const uint32_t* w = reinterpret_cast<const uint32_t*>(blk);
  uint32_t sw[kRows];
#pragma unroll
  for (int r = 0; r < kRows; ++r) sw[r] = w[r * (kRowElems / 2) + (kHeadDim / 2) + t];
  uint32_t mx = sw[0];
#pragma unroll
  for (int r = 1; r < kRows; ++r) mx = bf16x2_max(mx, sw[r]);
  const float nm0 = fmaxf(s.m0, bf16_lo(mx));
  const float nm1 = fmaxf(s.m1, bf16_hi(mx));
  const float r0 = fast_ex2((s.m0 - nm0) * kLog2e);  // 0 on the first rows
  const float r1 = fast_ex2((s.m1 - nm1) * kLog2e);
  const unsigned long long l2 = pack2(kLog2e, kLog2e);
  const unsigned long long negmb = pack2(-nm0 * kLog2e, -nm1 * kLog2e);
  unsigned long long dd = 0ull, aa = 0ull;
#pragma unroll
  for (int r = 0; r < kRows; ++r) {
    const uint32_t vw = w[r * (kRowElems / 2) + t];
    float x0, x1;
    unpack2(fma2(pack2(bf16_lo(sw[r]), bf16_hi(sw[r])), l2, negmb), x0, x1);
    const unsigned long long e = pack2(fast_ex2(x0), fast_ex2(x1));
    dd = add2(dd, e);
    aa = fma2(e, pack2(bf16_lo(vw), bf16_hi(vw)), aa);
  }
  float d0, d1, a0, a1;
  unpack2(dd, d0, d1);
  unpack2(aa, a0, a1);
  s.d0 = fmaf(s.d0, r0, d0);
  s.d1 = fmaf(s.d1, r1, d1);
  s.a0 = fmaf(s.a0, r0, a0);
  s.a1 = fmaf(s.a1, r1, a1);
  s.m0 = nm0;
  s.m1 = nm1;
}

// One staged 8-row block.
__device__ __forceinline__ void fold_block(const uint8_t* blk, int t, SoftmaxState& s) {
  fold_rows_n<kBlockRows>(blk, t, s);
}

// ---- block table resolution -------------------------------------------------------

// Physical block of unit (n, k) of the window (blk = -1, error recorded, if
// any index is bad) and, when want_meta, the output's slot and compressed
// position pc = floor(p / C) * C.  The slot is loaded together with the
// request and position, so the chain before the first bulk copy is three
// dependent loads deep.
__device__ __forceinline__ void resolve_unit(const Params& p, int64_t n, int k, bool want_meta,
                                             long long& blk, MetaRec& rec) {
  blk = -1;
  rec = MetaRec{-1, -1};
  const int64_t b = __ldg(p.bti + n);
  if (b < 0 || b >= p.num_tokens) { record_error(p.error, kErrBadIndex); return; }
  const int64_t r = __ldg(p.token_to_req + b);
  const int64_t pos = __ldg(p.positions + b);
  const int64_t slot = want_meta ? __ldg(p.slot_map + (p.slot_by_token ? b : n)) : -1;
  const int64_t t0 = pos - p.compress_ratio + 1;
  if (r < 0 || r >= p.num_reqs || t0 < 0) { record_error(p.error, kErrBadIndex); return; }
  if (t0 & (kBlockRows - 1)) { record_error(p.error, kErrUnsupported); return; }
  const int64_t l = t0 / kBlockRows + k;
  if (l >= p.max_blocks) { record_error(p.error, kErrBadIndex); return; }
  const int64_t g = __ldg(p.block_table + r * p.bt_row_stride + l * p.bt_col_stride);
  if (g < 0 || g >= p.num_blocks) { record_error(p.error, kErrBadIndex); return; }
  blk = g;
  if (want_meta) {
    const int64_t pc = (pos / p.compress_ratio) * p.compress_ratio;
    if (pc >= p.num_positions) { record_error(p.error, kErrBadIndex); blk = -1; return; }
    if (slot >= 0 && (slot / kSlotsPerPage) >= p.num_pages) {
      record_error(p.error, kErrBadIndex);
      blk = -1;
      return;
    }
    rec.slot = slot;
    rec.pc = pc;
  }
}

// Rows of window chunk k (rows t0 + 8k .. t0 + 8k + nr - 1 of the request, nr
// = min(8, C - 8k)) as at most two runs of rows that each lie in one
// physical block: the part in logical block l1 = (t0 + 8k) / B from offset
// o1, and the rest at the start of block l1 + 1 (block_size B >= 8, so a
// chunk never touches three blocks).  Runs are given as byte offsets from
// the state's base: block g, row o starts at g * block_bytes + o * row_bytes.
struct ChunkRuns {
  long long off1, off2;  // byte offset of each run's first row (off1 < 0: bad chunk)
  int n1, n2;            // rows in each run (n2 = 0: one run)
  int g1, o1;            // block and first row of run 1 (g1 valid below 2^31 only)
};

// Index loads of resolve_chunk_t.  The speculative pass (kSpec) loads
// through L2 only (ld.global.cg), so it leaves no line in L1 that a load
// after the grid dependency wait could hit.
template <bool kSpec>
__device__ __forceinline__ int64_t ld_index(const int32_t* a) {
  if constexpr (kSpec) {
    int32_t v;
    asm volatile("ld.global.cg.s32 %0, [%1];" : "=r"(v) : "l"(a));
    return v;
  } else {
    return __ldg(a);
  }
}
template <bool kSpec>
__device__ __forceinline__ int64_t ld_index(const int64_t* a) {
  if constexpr (kSpec) {
    int64_t v;
    asm volatile("ld.global.cg.s64 %0, [%1];" : "=l"(v) : "l"(a));
    return v;
  } else {
    return __ldg(a);
  }
}

// Resolve chunk k of output n for the cluster route (any window start, any
// C >= 1, any B >= 8, any state and block-table strides), and, when
// want_meta, the output's slot and compressed position.  All loads of one
// level are issued together: the chain before the first copy is boundary
// index -> (request, position, slot) -> one or two block-table entries.
// kSpec: the speculative pass, which runs before the grid dependency wait on
// indices that may still be changing; every index is bounds-checked all the
// same (a bad one yields off1 < 0), but nothing is recorded.
template <bool kSpec>
__device__ __forceinline__ void resolve_chunk_t(const Params& p, int64_t n, int k, bool want_meta,
                                                ChunkRuns& cr, MetaRec& rec) {
  cr = ChunkRuns{-1, -1, 0, 0, 0, 0};
  rec = MetaRec{-1, -1};
  const auto bad = [&]() {
    if constexpr (!kSpec) record_error(p.error, kErrBadIndex);
  };
  const int64_t b = ld_index<kSpec>(p.bti + n);
  if (b < 0 || b >= p.num_tokens) { bad(); return; }
  const int64_t r = ld_index<kSpec>(p.token_to_req + b);
  const int64_t pos = ld_index<kSpec>(p.positions + b);
  const int64_t slot = want_meta ? ld_index<kSpec>(p.slot_map + (p.slot_by_token ? b : n)) : -1;
  const int64_t C = p.compress_ratio, B = p.block_size;
  const int64_t t0 = pos - C + 1;
  if (r < 0 || r >= p.num_reqs || t0 < 0) { bad(); return; }
  const int64_t first = t0 + static_cast<int64_t>(kBlockRows) * k;
  const int64_t left = C - static_cast<int64_t>(kBlockRows) * k;
  const int nr = static_cast<int>(left < kBlockRows ? left : kBlockRows);
  const int64_t l1 = first / B, o1 = first - l1 * B;
  const int n1 = static_cast<int>(B - o1 < nr ? B - o1 : nr);
  const int n2 = nr - n1;
  if (l1 + (n2 > 0 ? 1 : 0) >= p.max_blocks) { bad(); return; }
  const int32_t* row = p.block_table + r * p.bt_row_stride;
  const int64_t g1 = ld_index<kSpec>(row + l1 * p.bt_col_stride);
  const int64_t g2 = n2 > 0 ? ld_index<kSpec>(row + (l1 + 1) * p.bt_col_stride) : 0;
  if (g1 < 0 || g1 >= p.num_blocks || g2 < 0 || g2 >= p.num_blocks) {
    bad();
    return;
  }
  if (want_meta) {
    const int64_t pc = (pos / C) * C;
    if (pc >= p.num_positions || (slot >= 0 && (slot / kSlotsPerPage) >= p.num_pages)) {
      bad();
      return;
    }
    rec.slot = slot;
    rec.pc = pc;
  }
  cr.off1 = g1 * p.state_block_bytes + o1 * p.state_row_bytes;
  cr.n1 = n1;
  cr.off2 = n2 > 0 ? g2 * p.state_block_bytes : -1;
  cr.n2 = n2;
  cr.g1 = static_cast<int>(g1);
  cr.o1 = static_cast<int>(o1);
}

__device__ __forceinline__ void resolve_chunk(const Params& p, int64_t n, int k, bool want_meta,
                                              ChunkRuns& cr, MetaRec& rec) {
  resolve_chunk_t<false>(p, n, k, want_meta, cr, rec);
}

// fold_block for a chunk holding only its first `nrows` (1..7) rows: the
// missing rows act as score -inf, value 0 (they add nothing and do not move
// the maximum).
__device__ __forceinline__ void fold_rows(const uint8_t* blk, int t, SoftmaxState& s, int nrows) {
  const uint32_t* w = reinterpret_cast<const uint32_t*>(blk);
  uint32_t sw[kBlockRows], vw[kBlockRows];
#pragma unroll
  for (int r = 0; r < kBlockRows; ++r) {
    const bool in = r < nrows;
    sw[r] = in ? w[r * (kRowElems / 2) + (kHeadDim / 2) + t] : 0xFF80FF80u;  // bf16 -inf pair
    vw[r] = in ? w[r * (kRowElems / 2) + t] : 0u;
  }
  const uint32_t mx = bf16x2_max(bf16x2_max(bf16x2_max(sw[0], sw[1]), bf16x2_max(sw[2], sw[3])),
                                 bf16x2_max(bf16x2_max(sw[4], sw[5]), bf16x2_max(sw[6], sw[7])));
  const float nm0 = fmaxf(s.m0, bf16_lo(mx));
  const float nm1 = fmaxf(s.m1, bf16_hi(mx));
  const float r0 = fast_ex2((s.m0 - nm0) * kLog2e);
  const float r1 = fast_ex2((s.m1 - nm1) * kLog2e);
  float d0 = 0.f, d1 = 0.f, a0 = 0.f, a1 = 0.f;
#pragma unroll
  for (int r = 0; r < kBlockRows; ++r) {
    if (r < nrows) {
      const float e0 = fast_ex2(fmaf(bf16_lo(sw[r]), kLog2e, -nm0 * kLog2e));
      const float e1 = fast_ex2(fmaf(bf16_hi(sw[r]), kLog2e, -nm1 * kLog2e));
      d0 += e0;
      d1 += e1;
      a0 = fmaf(e0, bf16_lo(vw[r]), a0);
      a1 = fmaf(e1, bf16_hi(vw[r]), a1);
    }
  }
  s.d0 = fmaf(s.d0, r0, d0);
  s.d1 = fmaf(s.d1, r1, d1);
  s.a0 = fmaf(s.a0, r0, a0);
  s.a1 = fmaf(s.a1, r1, a1);
  s.m0 = nm0;
  s.m1 = nm1;
}

// fold_block / fold_rows for a staged fp32 chunk (8 rows x [512 values | 512
// scores] fp32, 4 KiB per row): thread t reads float2 pairs of its dims.
// With kFull the chunk holds all 8 rows; otherwise only its first `nrows`,
// and the missing rows act as score -inf, value 0 (exp gives exactly 0).
template <bool kFull>
__device__ __forceinline__ void fold_f32(const uint8_t* blk, int t, SoftmaxState& s, int nrows) {
  const float2* w = reinterpret_cast<const float2*>(blk);
  float2 sw[kBlockRows], vw[kBlockRows];
#pragma unroll
  for (int r = 0; r < kBlockRows; ++r) {
    const bool in = kFull || r < nrows;
    sw[r] = in ? w[r * (kRowElems / 2) + (kHeadDim / 2) + t] : make_float2(-INFINITY, -INFINITY);
    vw[r] = in ? w[r * (kRowElems / 2) + t] : make_float2(0.f, 0.f);
  }
  float mx0 = fmaxf(fmaxf(fmaxf(sw[0].x, sw[1].x), fmaxf(sw[2].x, sw[3].x)),
                    fmaxf(fmaxf(sw[4].x, sw[5].x), fmaxf(sw[6].x, sw[7].x)));
  float mx1 = fmaxf(fmaxf(fmaxf(sw[0].y, sw[1].y), fmaxf(sw[2].y, sw[3].y)),
                    fmaxf(fmaxf(sw[4].y, sw[5].y), fmaxf(sw[6].y, sw[7].y)));
  const float nm0 = fmaxf(s.m0, mx0);
  const float nm1 = fmaxf(s.m1, mx1);
  const float r0 = fast_ex2((s.m0 - nm0) * kLog2e);  // 0 on the first chunk
  const float r1 = fast_ex2((s.m1 - nm1) * kLog2e);
  const unsigned long long l2 = pack2(kLog2e, kLog2e);
  const unsigned long long negmb = pack2(-nm0 * kLog2e, -nm1 * kLog2e);
  unsigned long long dd = 0ull, aa = 0ull;
#pragma unroll
  for (int r = 0; r < kBlockRows; ++r) {
    float x0, x1;
    unpack2(fma2(pack2(sw[r].x, sw[r].y), l2, negmb), x0, x1);
    const unsigned long long e = pack2(fast_ex2(x0), fast_ex2(x1));
    dd = add2(dd, e);
    aa = fma2(e, pack2(vw[r].x, vw[r].y), aa);
  }
  float d0, d1, a0, a1;
  unpack2(dd, d0, d1);
  unpack2(aa, a0, a1);
  s.d0 = fmaf(s.d0, r0, d0);
  s.d1 = fmaf(s.d1, r1, d1);
  s.a0 = fmaf(s.a0, r0, a0);
  s.a1 = fmaf(s.a1, r1, a1);
  s.m0 = nm0;
  s.m1 = nm1;
}

// ---- finaliser ------------------------------------------------------------------------

// Shared-memory scratch of the finaliser (one per CTA).
struct FinalScratch {
  alignas(16) uint8_t pack[kTokenStride + kScaleDim];  // the slot's 584 bytes
  float red[kConsumerWarps];
};

// Sum of c0^2 + c1^2 over the 256 consumer threads (each owning 2 dims).
__device__ __forceinline__ float consumer_sum_squares(FinalScratch& fs, float c0, float c1) {
  const int t = threadIdx.x;
  const float ss = warp_sum(c0 * c0 + c1 * c1);
  if ((t & 31) == 0) fs.red[t >> 5] = ss;
  consumer_sync();
  float tot = 0.f;
#pragma unroll
  for (int i = 0; i < kConsumerWarps; ++i) tot += fs.red[i];
  return tot;
}

// RMSNorm, NOPE quantisation, RoPE and the store of dims [dbase, dbase + wd)
// of output row `row` (= layer * num_outputs + n: the y_out row) of layer
// `layer`.  Thread t < wd/2 is `active` and owns dims d0 = dbase + 2t and
// d0 + 1 with window sums c0, c1 and RMSNorm weights w (loaded by the caller
// ahead of time, so the load's latency is not spent here); `total` is the
// sum of c^2 over all 512 dims.  wd is a multiple of 64, so every 64-dim quantisation group lies in
// one warp and the RoPE dims 448..511 in the last.  The slice's bytes are
// [dbase, dbase + wd) of the payload (up to 576 for the slice holding the
// RoPE dims) and scale bytes [dbase/64, (dbase + wd)/64) (the last one is
// the zero padding byte).  All 256 consumer threads call this (it holds
// consumer barriers).
__device__ __forceinline__ void finalize_slice(const Params& p, FinalScratch& fs, int layer,
                                               int64_t row, bool active, int d0, float c0, float c1,
                                               float2 w, bool bad, const MetaRec& meta, float cs,
                                               float sn, float total, int dbase, int wd) {
  const int t = threadIdx.x, lane = t & 31;
  const bool invalid = consumer_any(bad) || meta.pc < 0;
  const float rho = __frsqrt_rn(total * (1.0f / kHeadDim) + p.eps);
  if (active) {
    const float y0 = __fmul_rn(__fmul_rn(c0, rho), w.x);
    const float y1 = __fmul_rn(__fmul_rn(c1, rho), w.y);
    if (p.y_out != nullptr && !invalid)
      *reinterpret_cast<float2*>(p.y_out + row * kHeadDim + d0) = make_float2(y0, y1);
    if (d0 < kNopeDim) {
      // bf16 round trip, group amax (one warp = one 64-dim group), exponent,
      // truncating codes, two's-complement bytes
      const float z0 = __bfloat162float(__float2bfloat16_rn(y0));
      const float z1 = __bfloat162float(__float2bfloat16_rn(y1));
      const float a = fmaxf(warp_max(fmaxf(fabsf(z0), fabsf(z1))), 1.0e-4f);
      const int e = scale_exponent(a);
      const float inv = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);  // 2^-e, exact
      int q0 = __float2int_rz(__fmul_rn(z0, inv));
      int q1 = __float2int_rz(__fmul_rn(z1, inv));
      q0 = max(-127, min(127, q0));
      q1 = max(-127, min(127, q1));
      *reinterpret_cast<uint16_t*>(fs.pack + d0) =
          static_cast<uint16_t>((q0 & 0xFF) | ((q1 & 0xFF) << 8));
      if (lane == 0) fs.pack[kTokenStride + d0 / kGroup] = static_cast<uint8_t>(e + 127);
    } else {
      // GPT-J pair j on dims (448 + 2j, 449 + 2j), one rounding per operation
      const int j = (d0 - kNopeDim) >> 1;
      const float ru = __fsub_rn(__fmul_rn(y0, cs), __fmul_rn(y1, sn));
      const float rw = __fadd_rn(__fmul_rn(y1, cs), __fmul_rn(y0, sn));
      *reinterpret_cast<uint32_t*>(fs.pack + kNopeDim + 4 * j) =
          bf16_bits_rn(ru) | (bf16_bits_rn(rw) << 16);
      if (j == 0) fs.pack[kTokenStride + kScaleDim - 1] = 0;
    }
  }
  consumer_sync();
  if (!invalid && meta.slot >= 0) {
    uint8_t* page = p.kvs[layer] + (meta.slot / kSlotsPerPage) * kPageBytes;
    const int64_t off = meta.slot % kSlotsPerPage;
    const int pb0 = dbase;
    const int pb1 = (dbase + wd == kHeadDim) ? kTokenStride : dbase + wd;
    const int chunks = (pb1 - pb0) / 16;
    const int sb0 = dbase / kGroup, sb1 = (dbase + wd) / kGroup;
    if (t < chunks) {
      reinterpret_cast<uint4*>(page + off * kTokenStride + pb0)[t] =
          reinterpret_cast<const uint4*>(fs.pack + pb0)[t];
    } else if (t < chunks + (sb1 - sb0)) {
      if (sb1 - sb0 == kScaleDim) {  // whole scale record: one 8-byte store
        if (t == chunks)
          *reinterpret_cast<uint2*>(page + kScaleBase + off * kScaleDim) =
              *reinterpret_cast<const uint2*>(fs.pack + kTokenStride);
      } else {
        const int i = sb0 + (t - chunks);
        page[kScaleBase + off * kScaleDim + i] = fs.pack[kTokenStride + i];
      }
    }
  }
  consumer_sync();  // fs is reused by the next output
}

}  // namespace dev
}  // namespace kvc
