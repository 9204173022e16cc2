// Fused KV-cache window compressor for sm_103a (GB300).
//
// Computes c128_256_512_compress of "From Attention to KV Cache Compression:
// Notes from a KernelGen Optimization" (KernelGen Challenge 8 write-up) in
// one launch: paged window gather, per-dimension softmax-weighted window sum
// ("How One Output Is Produced"; streamed as in "Online Softmax: Streaming
// Away the Window"), RMSNorm, NOPE int8 quantisation, GPT-J RoPE and the
// packed slot scatter ("Gather and Scatter"; byte rules of "The Finalizer's
// Sharp Edges").
//
// Work decomposition.  One unit = one 8-row physical block of one output's
// window (16 KiB of bf16: 8 rows x [512 values | 512 scores]); the units of
// all outputs form one sequence u = n * K + k (K = C / 8).  A persistent grid
// of G CTAs takes contiguous, equal slices of that sequence (stream-K), so
// every CTA streams the same number of bytes whatever N and C are.  An output
// whose units fall in one CTA is finalised there; an output split between
// CTAs leaves partial softmax states (m, den, num per dimension) in the
// workspace and the last CTA to arrive on the output's counter merges them
// and finalises -- nobody waits for anybody.
//
// Inside a CTA, warp 8 (the producer) resolves block_table entries and issues
// one cp.async.bulk copy of 16 KiB per unit into a kStages-deep shared-memory
// ring, each stage guarded by a full/empty mbarrier pair.  Warps 0..7 (the
// consumers) run the online softmax: thread t owns dimensions 2t and 2t+1,
// keeps (m, den, num) for both in registers and folds one 8-row block per
// stage (tile max in bf16x2, one rescale per block, one ex2 per element).
// At the end of an output the consumers reduce the sum of squares across the
// CTA, quantise (warp w < 7 owns NOPE group w, so the group amax is a warp
// reduction), rotate (warp 7, lane j owns RoPE pair j), stage the 584 bytes
// in shared memory and store them with 16-byte stores.
//
// Every wait is bounded: on timeout the kernel records KVC_ERR_TIMEOUT,
// stops issuing copies, waits (bounded) for the copies already issued and
// returns.  Invalid indices are recorded as errors and the affected outputs
// are skipped; nothing traps.

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "kvc_internal.h"

namespace kvc {
namespace {

// Device error word: the first error code recorded since the last clear.
__device__ uint32_t g_error_word;

constexpr uint32_t kErrUnsupported = 2;
constexpr uint32_t kErrBadIndex = 4;
constexpr uint32_t kErrTimeout = 5;
constexpr long long kWaitLimitCycles = 4000000000LL;  // ~2 s at 2 GHz
constexpr float kLog2e = 1.4426950408889634f;

struct alignas(16) MetaRec {
  long long slot;  // destination slot (< 0: do not write)
  long long pc;    // compressed position (< 0: invalid output)
};

struct SmemTail {
  unsigned long long full_bar[kStages];
  unsigned long long empty_bar[kStages];
  MetaRec meta[kMetaRing];
  alignas(16) uint8_t pack[kTokenStride + kScaleDim];
  float red[kConsumerWarps];
  uint32_t stage_ok[kStages];
  int abort_flag;
  int ticket;
};

// ---- small PTX helpers ---------------------------------------------------

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

// Wait for the phase of `bar` with the given parity; false after the limit.
__device__ __noinline__ bool mbar_wait_bounded(unsigned long long* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (clock64() - t0 > kWaitLimitCycles) return false;
  }
}

__device__ __forceinline__ uint64_t evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
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

__device__ __forceinline__ void record_error(uint32_t code) { atomicCAS(&g_error_word, 0u, code); }

// ---- the finaliser's scalar rules -----------------------------------------

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

// cta_of(u): the CTA whose slice [floor(g U / G), floor((g+1) U / G)) holds u.
__device__ __forceinline__ int64_t cta_of(int64_t u, int64_t U, int64_t G) {
  return ((u + 1) * G - 1) / U;
}

// Per-output metadata: slot and compressed position (pc < 0 when invalid).
__device__ MetaRec load_meta(const Params& p, int64_t n) {
  MetaRec rec{-1, -1};
  const int64_t b = __ldg(p.bti + n);
  if (b < 0 || b >= p.num_tokens) return rec;
  const int64_t pos = __ldg(p.positions + b);
  const int64_t slot = __ldg(p.slot_map + (p.slot_by_token ? b : n));
  if (pos < 0) return rec;
  const int64_t pc = (pos / p.compress_ratio) * p.compress_ratio;
  if (pc >= p.num_positions) { record_error(kErrBadIndex); return rec; }
  if (slot >= 0 && (slot / kSlotsPerPage) >= p.num_pages) { record_error(kErrBadIndex); return rec; }
  rec.slot = slot;
  rec.pc = pc;
  return rec;
}

// Physical block of unit (n, k), or -1 (error recorded) if any index is bad.
__device__ long long resolve_block(const Params& p, int64_t n, int k) {
  const int64_t b = __ldg(p.bti + n);
  if (b < 0 || b >= p.num_tokens) { record_error(kErrBadIndex); return -1; }
  const int64_t r = __ldg(p.token_to_req + b);
  const int64_t pos = __ldg(p.positions + b);
  const int64_t t0 = pos - p.compress_ratio + 1;
  if (r < 0 || r >= p.num_reqs || t0 < 0) { record_error(kErrBadIndex); return -1; }
  if (t0 & (kBlockRows - 1)) { record_error(kErrUnsupported); return -1; }
  const int64_t l = t0 / kBlockRows + k;
  if (l >= p.max_blocks) { record_error(kErrBadIndex); return -1; }
  const int64_t g = __ldg(p.block_table + r * p.max_blocks + l);
  if (g < 0 || g >= p.num_blocks) { record_error(kErrBadIndex); return -1; }
  return g;
}

// ---- producer warp ----------------------------------------------------------

__device__ void producer(const Params& p, SmemTail& sh, uint8_t* ring, int64_t u0, int64_t u1) {
  const int lane = threadIdx.x & 31;
  const int K = p.blocks_per_output;
  const uint64_t policy = evict_first_policy();
  int stage = 0;
  uint32_t phase = 0;
  uint32_t issued = 0, last_parity = 0;  // per-stage bit masks (lane 0)
  bool aborted = false;
  for (int64_t base = u0; base < u1 && !aborted; base += 32) {
    const int64_t u = base + lane;
    long long blk = -1;
    MetaRec rec{-1, -1};
    int first = 0;
    int64_t n = 0;
    if (u < u1) {
      n = u / K;
      const int k = static_cast<int>(u - n * K);
      first = (k == 0 || u == u0);
      blk = resolve_block(p, n, k);
      if (first) rec = load_meta(p, n);
    }
    const int cnt = static_cast<int>(u1 - base < 32 ? u1 - base : 32);
    for (int j = 0; j < cnt; ++j) {
      const long long gb = __shfl_sync(0xffffffffu, blk, j);
      const int fj = __shfl_sync(0xffffffffu, first, j);
      const long long nj = __shfl_sync(0xffffffffu, static_cast<long long>(n), j);
      const long long slot_j = __shfl_sync(0xffffffffu, rec.slot, j);
      const long long pc_j = __shfl_sync(0xffffffffu, rec.pc, j);
      if (lane == 0) {
        if (*reinterpret_cast<volatile int*>(&sh.abort_flag)) {
          aborted = true;
        } else if (!mbar_wait_bounded(&sh.empty_bar[stage], phase ^ 1u)) {
          record_error(kErrTimeout);
          *reinterpret_cast<volatile int*>(&sh.abort_flag) = 1;
          aborted = true;
        } else {
          if (fj) {
            MetaRec& m = sh.meta[nj % kMetaRing];
            m.slot = slot_j;
            m.pc = pc_j;
          }
          if (gb >= 0) {
            sh.stage_ok[stage] = 1;
            mbar_arrive_expect_tx(&sh.full_bar[stage], kBlockBytes);
            bulk_copy_g2s(ring + static_cast<size_t>(stage) * kBlockBytes,
                          p.state + gb * (kBlockRows * kRowElems), kBlockBytes,
                          &sh.full_bar[stage], policy);
          } else {
            sh.stage_ok[stage] = 0;
            mbar_arrive(&sh.full_bar[stage]);
          }
          issued |= 1u << stage;
          last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
        }
      }
      aborted = __shfl_sync(0xffffffffu, aborted, 0);
      if (aborted) break;
      if (++stage == kStages) { stage = 0; phase ^= 1u; }
    }
  }
  // No bulk copy may still target this CTA's shared memory when it exits.
  if (lane == 0) {
    for (int s = 0; s < kStages; ++s)
      if ((issued >> s) & 1u)
        if (!mbar_wait_bounded(&sh.full_bar[s], (last_parity >> s) & 1u)) record_error(kErrTimeout);
  }
}

// ---- consumer warps --------------------------------------------------------

struct SoftmaxState {
  float m0, m1, d0, d1, a0, a1;  // running max, denominator, numerator
};

__device__ __forceinline__ void state_reset(SoftmaxState& s) {
  s.m0 = s.m1 = -INFINITY;
  s.d0 = s.d1 = s.a0 = s.a1 = 0.f;
}

// Fold one staged 8-row block into thread t's two dimensions.
__device__ __forceinline__ void fold_block(const uint8_t* blk, int t, SoftmaxState& s) {
  const uint32_t* w = reinterpret_cast<const uint32_t*>(blk);
  uint32_t sw[kBlockRows], vw[kBlockRows];
#pragma unroll
  for (int r = 0; r < kBlockRows; ++r) {
    sw[r] = w[r * (kRowElems / 2) + (kHeadDim / 2) + t];
    vw[r] = w[r * (kRowElems / 2) + t];
  }
  const uint32_t mx = bf16x2_max(bf16x2_max(bf16x2_max(sw[0], sw[1]), bf16x2_max(sw[2], sw[3])),
                                 bf16x2_max(bf16x2_max(sw[4], sw[5]), bf16x2_max(sw[6], sw[7])));
  const float nm0 = fmaxf(s.m0, bf16_lo(mx));
  const float nm1 = fmaxf(s.m1, bf16_hi(mx));
  const float r0 = fast_ex2((s.m0 - nm0) * kLog2e);  // 0 on the first block
  const float r1 = fast_ex2((s.m1 - nm1) * kLog2e);
  const float mb0 = nm0 * kLog2e, mb1 = nm1 * kLog2e;
  float d0 = 0.f, d1 = 0.f, a0 = 0.f, a1 = 0.f;
#pragma unroll
  for (int r = 0; r < kBlockRows; ++r) {
    const float e0 = fast_ex2(fmaf(bf16_lo(sw[r]), kLog2e, -mb0));
    const float e1 = fast_ex2(fmaf(bf16_hi(sw[r]), kLog2e, -mb1));
    d0 += e0;
    d1 += e1;
    a0 = fmaf(e0, bf16_lo(vw[r]), a0);
    a1 = fmaf(e1, bf16_hi(vw[r]), a1);
  }
  s.d0 = fmaf(s.d0, r0, d0);
  s.d1 = fmaf(s.d1, r1, d1);
  s.a0 = fmaf(s.a0, r0, a0);
  s.a1 = fmaf(s.a1, r1, a1);
  s.m0 = nm0;
  s.m1 = nm1;
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

// RMSNorm, quantisation, RoPE and the slot store of output n.  All 256
// consumer threads call this together (it contains consumer barriers).
__device__ void finalize(const Params& p, SmemTail& sh, int64_t n, float c0, float c1, bool bad,
                         const MetaRec& meta, float cs, float sn) {
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const bool invalid = consumer_any(bad) || meta.pc < 0;

  // rho = (mean(c^2) + eps)^-1/2 over the 512 dimensions
  const float ss = warp_sum(c0 * c0 + c1 * c1);
  if (lane == 0) sh.red[warp] = ss;
  consumer_sync();
  float tot = 0.f;
#pragma unroll
  for (int i = 0; i < kConsumerWarps; ++i) tot += sh.red[i];
  const float rho = __frsqrt_rn(tot * (1.0f / kHeadDim) + p.eps);
  const float2 w = __ldg(reinterpret_cast<const float2*>(p.weight) + t);
  const float y0 = __fmul_rn(__fmul_rn(c0, rho), w.x);
  const float y1 = __fmul_rn(__fmul_rn(c1, rho), w.y);
  if (p.y_out != nullptr && !invalid)
    reinterpret_cast<float2*>(p.y_out + n * kHeadDim)[t] = make_float2(y0, y1);

  if (warp < kNopeDim / kGroup) {
    // NOPE group `warp`: bf16 round trip, amax, exponent, truncating codes
    const float z0 = __bfloat162float(__float2bfloat16_rn(y0));
    const float z1 = __bfloat162float(__float2bfloat16_rn(y1));
    const float a = fmaxf(warp_max(fmaxf(fabsf(z0), fabsf(z1))), 1.0e-4f);
    const int e = scale_exponent(a);
    const float inv = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);  // 2^-e
    int q0 = __float2int_rz(__fmul_rn(z0, inv));
    int q1 = __float2int_rz(__fmul_rn(z1, inv));
    q0 = max(-127, min(127, q0));
    q1 = max(-127, min(127, q1));
    reinterpret_cast<uint16_t*>(sh.pack)[t] =
        static_cast<uint16_t>((q0 & 0xFF) | ((q1 & 0xFF) << 8));
    if (lane == 0) sh.pack[kTokenStride + warp] = static_cast<uint8_t>(e + 127);
  } else {
    // RoPE pair j = lane on dims (448 + 2j, 449 + 2j)
    const float ru = __fsub_rn(__fmul_rn(y0, cs), __fmul_rn(y1, sn));
    const float rw = __fadd_rn(__fmul_rn(y1, cs), __fmul_rn(y0, sn));
    reinterpret_cast<uint32_t*>(sh.pack + kNopeDim)[lane] = bf16_bits_rn(ru) | (bf16_bits_rn(rw) << 16);
    if (lane == 0) sh.pack[kTokenStride + kScaleDim - 1] = 0;
  }
  consumer_sync();
  if (!invalid && meta.slot >= 0) {
    uint8_t* page = p.kv + (meta.slot / kSlotsPerPage) * kPageBytes;
    const int64_t off = meta.slot % kSlotsPerPage;
    if (t < kTokenStride / 16) {
      reinterpret_cast<uint4*>(page + off * kTokenStride)[t] = reinterpret_cast<const uint4*>(sh.pack)[t];
    } else if (t == kTokenStride / 16) {
      *reinterpret_cast<uint2*>(page + kScaleBase + off * kScaleDim) =
          *reinterpret_cast<const uint2*>(sh.pack + kTokenStride);
    }
  }
  consumer_sync();  // sh.pack / sh.red are reused by the next output
}

// Store this CTA's partial state of output n; the last CTA to arrive merges
// all partials of n and finalises it.
__device__ void flush_partial(const Params& p, SmemTail& sh, int64_t n, int64_t g, int64_t G,
                              int64_t n_first, const SoftmaxState& s, bool bad) {
  const int t = threadIdx.x;
  const int64_t U = p.num_units, K = p.blocks_per_output;
  const int which = (n == n_first) ? 0 : 1;
  float* rec = p.partials + (g * 2 + which) * kPartialFloats;
  __stcg(reinterpret_cast<float2*>(rec) + t, make_float2(s.m0, s.m1));
  __stcg(reinterpret_cast<float2*>(rec + kHeadDim) + t, make_float2(s.d0, s.d1));
  __stcg(reinterpret_cast<float2*>(rec + 2 * kHeadDim) + t, make_float2(s.a0, s.a1));
  const bool any_bad = consumer_any(bad);
  if (t == 0) __stcg(p.part_status + g * 2 + which, any_bad ? 1 : 0);
  __threadfence();
  consumer_sync();
  if (t == 0) sh.ticket = atomicAdd(p.counters + n, 1);
  consumer_sync();
  const int64_t gf = cta_of(n * K, U, G), gl = cta_of(n * K + K - 1, U, G);
  if (sh.ticket != static_cast<int>(gl - gf)) return;  // uniform across consumers

  // Last arrival: every other piece of n is published.
  __threadfence();
  if (t == 0) p.counters[n] = 0;  // ready for the next call
  float M0 = -INFINITY, M1 = -INFINITY;
  for (int64_t gg = gf; gg <= gl; ++gg) {
    const int wh = (n == (gg * U / G) / K) ? 0 : 1;
    const float2 m = __ldcg(reinterpret_cast<const float2*>(p.partials + (gg * 2 + wh) * kPartialFloats) + t);
    M0 = fmaxf(M0, m.x);
    M1 = fmaxf(M1, m.y);
  }
  float D0 = 0.f, D1 = 0.f, A0 = 0.f, A1 = 0.f;
  bool mbad = false;
  for (int64_t gg = gf; gg <= gl; ++gg) {
    const int wh = (n == (gg * U / G) / K) ? 0 : 1;
    const float* r = p.partials + (gg * 2 + wh) * kPartialFloats;
    const float2 m = __ldcg(reinterpret_cast<const float2*>(r) + t);
    const float2 d = __ldcg(reinterpret_cast<const float2*>(r + kHeadDim) + t);
    const float2 a = __ldcg(reinterpret_cast<const float2*>(r + 2 * kHeadDim) + t);
    const float f0 = fast_ex2((m.x - M0) * kLog2e), f1 = fast_ex2((m.y - M1) * kLog2e);
    D0 = fmaf(d.x, f0, D0);
    D1 = fmaf(d.y, f1, D1);
    A0 = fmaf(a.x, f0, A0);
    A1 = fmaf(a.y, f1, A1);
    mbad |= __ldcg(p.part_status + gg * 2 + wh) != 0;
  }
  const MetaRec meta = load_meta(p, n);
  float cs = 1.f, sn = 0.f;
  const int warp = t >> 5, lane = t & 31;
  if (warp == kConsumerWarps - 1 && meta.pc >= 0) {
    cs = __ldg(p.cos_sin + meta.pc * kRopeDim + lane);
    sn = __ldg(p.cos_sin + meta.pc * kRopeDim + kRopeDim / 2 + lane);
  }
  finalize(p, sh, n, A0 / D0, A1 / D1, mbad, meta, cs, sn);
}

__device__ void consumer(const Params& p, SmemTail& sh, const uint8_t* ring, int64_t u0,
                         int64_t u1, int64_t g, int64_t G) {
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int K = p.blocks_per_output;
  const int64_t n_first = u0 / K;
  int64_t n = n_first;
  int k = static_cast<int>(u0 - n * K);
  bool from_start = (k == 0);
  int stage = 0;
  uint32_t phase = 0;
  SoftmaxState s;
  state_reset(s);
  bool bad = false;
  MetaRec meta{-1, -1};
  float cs = 1.f, sn = 0.f;
  for (int64_t u = u0; u < u1; ++u) {
    bool ready = false;
    if (!*reinterpret_cast<volatile int*>(&sh.abort_flag)) {
      ready = mbar_wait_bounded(&sh.full_bar[stage], phase);
      if (!ready) {
        record_error(kErrTimeout);
        *reinterpret_cast<volatile int*>(&sh.abort_flag) = 1;
      }
    }
    if (u == u0 || k == 0) {  // first unit of a piece: take the output's record
      if (ready) {
        meta = sh.meta[n % kMetaRing];
        if (warp == kConsumerWarps - 1 && meta.pc >= 0) {
          cs = __ldg(p.cos_sin + meta.pc * kRopeDim + lane);
          sn = __ldg(p.cos_sin + meta.pc * kRopeDim + kRopeDim / 2 + lane);
        }
      } else {
        meta = MetaRec{-1, -1};
      }
    }
    if (ready && sh.stage_ok[stage]) {
      fold_block(ring + static_cast<size_t>(stage) * kBlockBytes, t, s);
    } else {
      bad = true;
    }
    __syncwarp();
    if (ready && lane == 0) mbar_arrive(&sh.empty_bar[stage]);
    if (++stage == kStages) { stage = 0; phase ^= 1u; }

    const bool end_of_output = (k == K - 1);
    if (end_of_output || u == u1 - 1) {
      if (from_start && end_of_output) {
        finalize(p, sh, n, s.a0 / s.d0, s.a1 / s.d1, bad, meta, cs, sn);
      } else {
        flush_partial(p, sh, n, g, G, n_first, s, bad);
      }
      state_reset(s);
      bad = false;
      from_start = true;
      if (end_of_output) { ++n; k = 0; }
    } else {
      ++k;
    }
  }
}

__global__ void __launch_bounds__(kThreads, 2) kvc_compress_kernel(const Params p) {
  extern __shared__ __align__(128) uint8_t smem[];
  SmemTail& sh = *reinterpret_cast<SmemTail*>(smem + static_cast<size_t>(kStages) * kBlockBytes);
  const int64_t U = p.num_units, G = gridDim.x, g = blockIdx.x;
  const int64_t u0 = g * U / G, u1 = (g + 1) * U / G;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sh.full_bar[s], 1);
      mbar_init(&sh.empty_bar[s], kConsumerWarps);
    }
    sh.abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (u0 >= u1) return;
  if (threadIdx.x >= kConsumerThreads) {
    producer(p, sh, smem, u0, u1);
  } else {
    consumer(p, sh, smem, u0, u1, g, G);
  }
}

}  // namespace

size_t dynamic_smem_bytes() {
  return static_cast<size_t>(kStages) * kBlockBytes + sizeof(SmemTail);
}

const void* kernel_symbol() { return reinterpret_cast<const void*>(&kvc_compress_kernel); }

uint32_t* device_error_word() {
  void* ptr = nullptr;
  if (cudaGetSymbolAddress(&ptr, g_error_word) != cudaSuccess) return nullptr;
  return static_cast<uint32_t*>(ptr);
}

cudaError_t launch(const Params& p, int ctas, cudaStream_t stream) {
  kvc_compress_kernel<<<ctas, kThreads, dynamic_smem_bytes(), stream>>>(p);
  return cudaGetLastError();
}

WorkspaceLayout workspace_layout(int max_ctas, int64_t num_outputs) {
  auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  WorkspaceLayout L;
  L.partials = 0;
  L.status = up(static_cast<size_t>(2) * max_ctas * kPartialFloats * sizeof(float));
  L.counters = L.status + up(static_cast<size_t>(2) * max_ctas * sizeof(int32_t));
  L.total = L.counters + up(static_cast<size_t>(num_outputs > 0 ? num_outputs : 0) * sizeof(int32_t));
  return L;
}

}  // namespace kvc
