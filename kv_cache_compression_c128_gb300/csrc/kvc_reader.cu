// Reader direction of the KV-cache window compressor: decode packed slots
// back into 512-vectors for the attention side.
//
// The slot layout is the one of "Gather and Scatter" in "From Attention to
// KV Cache Compression: Notes from a KernelGen Optimization" (KernelGen
// Challenge 8 write-up); the values are the ones its quantisation equation
// ("How One Output Is Produced") encodes: NOPE dim d < 448 reads back as
// q_d * 2^(scale[d / 64] - 127), RoPE dims 448..511 as the stored bf16.
//
// Small calls: one slot per 128 threads, 4 dims per thread: a thread reads 4
// int8 codes (or 4 bf16 RoPE values) and the group's scale byte, scales
// exactly (see "exact decode") and writes one 16-byte (fp32) or 8-byte
// (bf16) vector.
// Large calls (more slot pairs than fit on the device at once): one warp per
// slot on a persistent grid, 4 (fp32 output) or 2 (bf16) slots per warp in
// flight, every load and store coalesced.  584 bytes read and 1 or 2 KiB written per slot.

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "kvc_internal.h"

namespace kvc {
namespace {

constexpr int kReaderThreads = 256;
constexpr int kThreadsPerSlot = kHeadDim / 4;   // 128
constexpr int kSlotsPerCta = kReaderThreads / kThreadsPerSlot;
constexpr uint32_t kErrBadIndexReader = 4;

// ---- exact decode -----------------------------------------------------------
//
// A stored value is q * 2^e for an int8 code q (any of its 256 byte values)
// and e = b - 127 for a scale byte b (any of its 256 values).  The product
// has at most 8 significant bits, so it is exact in fp32 -- and in bf16 --
// unless |q| 2^e reaches 2^128, where correct rounding gives +-inf; zero
// codes give +0.  It is formed from exact pieces with no conversion
// instruction and no library scaling call:
//   q       = float(2^23 + (q + 128)) - (2^23 + 128): the byte (q + 128) is
//             placed in the mantissa of 2^23 (integer bit operations), and
//             the subtraction of two integers below 2^24 is exact;
//   2^(e-1) = the fp32 with those bits: exponent field b - 1 for b >= 2,
//             the subnormals 2^-127 (b = 1) and 2^-128 (b = 0);
//   q 2^e   = (q * 2^(e-1)) * 2: both products are exact or overflow, and
//             b = 255 (e = 128, whose 2^e is not an fp32 value) needs no
//             special case: a zero code stays +0, any other overflows.
// The fp32 result's low 16 bits are zero (at most 8 significant bits, and
// subnormal results keep their bits at or above 2^-128), so its bf16 form
// is exactly its high half.

// 2^(e - 1) for the scale byte b = e + 127.
__device__ __forceinline__ float half_scale(uint32_t b) {
  return __uint_as_float(b >= 2u ? (b - 1u) << 23 : 0x00200000u << b);
}

// The four codes of `word` (little-endian int8) times 2^e, hs = half_scale.
__device__ __forceinline__ void decode4(uint32_t word, float hs, float v[4]) {
  const uint32_t x = word ^ 0x80808080u;  // q + 128 in every byte
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    // bytes (q + 128, 0, 0, 0x4B): 2^23 + q + 128
    const float q = __uint_as_float(__byte_perm(x, 0x4B00u, 0x5440u | i)) - 8388736.0f;
    v[i] = (q * hs) * 2.0f;
  }
}

// Two decoded values (each exactly a bf16) as one word of bf16 bits.
__device__ __forceinline__ uint32_t bf16_pair(float lo, float hi) {
  return __byte_perm(__float_as_uint(lo), __float_as_uint(hi), 0x7632u);
}

// What one thread reads for its 4 dims of one slot.
struct Piece {
  uint32_t codes;  // 4 int8 codes (NOPE dims)
  uint2 raw;       // 4 bf16 words (RoPE dims)
  uint32_t b;      // the group's scale byte
  bool ok;         // the slot is read (non-negative and on a page)
};

__device__ __forceinline__ Piece load_piece(const uint8_t* __restrict__ kv, int64_t num_pages,
                                            int64_t slot, int d0, int t, uint32_t* err) {
  Piece pc{0u, make_uint2(0u, 0u), 0u, false};
  if (slot < 0) return pc;
  const int64_t page = slot / kSlotsPerPage, off = slot % kSlotsPerPage;
  if (page >= num_pages) {
    if (t == 0) atomicCAS(err, 0u, kErrBadIndexReader);
    return pc;
  }
  const uint8_t* pg = kv + page * kPageBytes;
  const uint8_t* payload = pg + off * kTokenStride;
  if (d0 < kNopeDim) {
    pc.codes = __ldg(reinterpret_cast<const uint32_t*>(payload + d0));
    pc.b = __ldg(pg + kScaleBase + off * kScaleDim + d0 / kGroup);
  } else {
    pc.raw = __ldg(reinterpret_cast<const uint2*>(payload + kNopeDim + 2 * (d0 - kNopeDim)));
  }
  pc.ok = true;
  return pc;
}

__device__ __forceinline__ void store_piece(const Piece& pc, int d0, int t, int64_t m, void* out,
                                            int out_bf16) {
  float v[4] = {0.f, 0.f, 0.f, 0.f};
  const bool rope = pc.ok && d0 >= kNopeDim;  // RoPE dims: the stored bf16 words, copied as they are
  if (pc.ok && !rope) {
    decode4(pc.codes, half_scale(pc.b), v);
  } else if (rope) {
    v[0] = __uint_as_float(pc.raw.x << 16);
    v[1] = __uint_as_float(pc.raw.x & 0xFFFF0000u);
    v[2] = __uint_as_float(pc.raw.y << 16);
    v[3] = __uint_as_float(pc.raw.y & 0xFFFF0000u);
  }
  if (out_bf16 && rope) {
    reinterpret_cast<uint2*>(static_cast<uint16_t*>(out) + m * kHeadDim)[t] = pc.raw;
  } else if (out_bf16) {
    reinterpret_cast<uint2*>(static_cast<uint16_t*>(out) + m * kHeadDim)[t] =
        make_uint2(bf16_pair(v[0], v[1]), bf16_pair(v[2], v[3]));
  } else {
    reinterpret_cast<float4*>(static_cast<float*>(out) + m * kHeadDim)[t] =
        make_float4(v[0], v[1], v[2], v[3]);
  }
}

// Grid-stride over the slots, kUnroll per 128-thread slot lane and pass: the
// slot indices, then the codes and exponents of all kUnroll slots are loaded
// before any is decoded and stored, so each thread keeps kUnroll chains in
// flight, and at most a device-full of CTAs is launched.
// kUnroll = 1 (the launcher's choice for calls of up to a device-full of
// slot pairs): one slot per 128-thread lane.
template <int kUnroll>
__global__ void __launch_bounds__(kReaderThreads) kvc_dequant_kernel(
    const uint8_t* __restrict__ kv, int64_t num_pages, const int64_t* __restrict__ slots,
    int64_t num_slots, void* __restrict__ out, int out_bf16, uint32_t* err) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int lane_slot = threadIdx.x / kThreadsPerSlot;
  const int t = threadIdx.x % kThreadsPerSlot;
  const int d0 = 4 * t;
  // the kUnroll slots of one pass lie one grid-width apart, so a grid with
  // a CTA per two slots (small calls) gives every lane one slot, and the
  // persistent grid of large calls gives every lane kUnroll per pass
  const int64_t width = static_cast<int64_t>(gridDim.x) * kSlotsPerCta;
  for (int64_t base = static_cast<int64_t>(blockIdx.x) * kSlotsPerCta + lane_slot;
       base < num_slots; base += width * kUnroll) {
    int64_t sl[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t m = base + u * width;
      sl[u] = m < num_slots ? __ldg(slots + m) : -1;
    }
    Piece pc[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) pc[u] = load_piece(kv, num_pages, sl[u], d0, t, err);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t m = base + u * width;
      if (m < num_slots) store_piece(pc[u], d0, t, m, out, out_bf16);
    }
  }
}

// One warp per slot: lane L handles dims 4L + 128k for k = 0..3, so every
// load and store instruction of a warp covers one contiguous run of the slot
// (128 code bytes, 512 fp32 or 256 bf16 output bytes).  Dims 0..447 are
// NOPE; in pass k = 3, lanes 16..31 hold the RoPE dims 448..511.  The
// slot's 8-byte scale record is read once per lane.  kUnroll slots per warp
// and pass, one grid-width of warps apart, are loaded before any is written,
// on a persistent grid: the large calls, where the bytes in flight per SM
// decide the rate.  kStream: streaming (evict-first) stores, for outputs
// that are not read back soon.
template <int kUnroll, bool kStream>
__global__ void __launch_bounds__(kReaderThreads) kvc_dequant_warp_kernel(
    const uint8_t* __restrict__ kv, int64_t num_pages, const int64_t* __restrict__ slots,
    int64_t num_slots, void* __restrict__ out, int out_bf16, uint32_t* err) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  constexpr int kWarps = kReaderThreads / 32;
  const int lane = threadIdx.x & 31;
  const bool rope_lane = lane >= 16;  // in pass 3
  const int64_t width = static_cast<int64_t>(gridDim.x) * kWarps;
  for (int64_t base = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
       base < num_slots; base += width * kUnroll) {
    int64_t sl[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t m = base + u * width;
      sl[u] = m < num_slots ? __ldg(slots + m) : -1;
    }
    uint32_t codes[kUnroll][4];
    uint2 scale[kUnroll], rope[kUnroll];
    bool ok[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
#pragma unroll
      for (int k = 0; k < 4; ++k) codes[u][k] = 0u;
      scale[u] = rope[u] = make_uint2(0u, 0u);
      ok[u] = false;
      if (sl[u] < 0) continue;
      const int64_t page = sl[u] / kSlotsPerPage, off = sl[u] % kSlotsPerPage;
      if (page >= num_pages) {
        if (lane == 0) atomicCAS(err, 0u, kErrBadIndexReader);
        continue;
      }
      const uint8_t* pg = kv + page * kPageBytes;
      const uint8_t* payload = pg + off * kTokenStride;
      scale[u] = __ldg(reinterpret_cast<const uint2*>(pg + kScaleBase + off * kScaleDim));
#pragma unroll
      for (int k = 0; k < 3; ++k)
        codes[u][k] = __ldg(reinterpret_cast<const uint32_t*>(payload + 4 * lane + 128 * k));
      if (!rope_lane)
        codes[u][3] = __ldg(reinterpret_cast<const uint32_t*>(payload + 4 * lane + 384));
      else
        rope[u] = __ldg(reinterpret_cast<const uint2*>(payload + kNopeDim + 8 * (lane - 16)));
      ok[u] = true;
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t m = base + u * width;
      if (m >= num_slots) continue;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int d = 4 * lane + 128 * k;
        const bool is_rope = k == 3 && rope_lane;
        float v[4] = {0.f, 0.f, 0.f, 0.f};
        if (ok[u] && !is_rope) {
          const int g = d / kGroup;  // 2k + lane / 16
          const uint32_t sw = g < 4 ? scale[u].x : scale[u].y;
          decode4(codes[u][k], half_scale((sw >> (8 * (g & 3))) & 0xFFu), v);
        } else if (is_rope) {
          v[0] = __uint_as_float(rope[u].x << 16);
          v[1] = __uint_as_float(rope[u].x & 0xFFFF0000u);
          v[2] = __uint_as_float(rope[u].y << 16);
          v[3] = __uint_as_float(rope[u].y & 0xFFFF0000u);
        }
        if (out_bf16) {
          uint2 o;
          if (is_rope) {  // the stored bf16 words, copied as they are
            o = rope[u];
          } else {
            o = make_uint2(bf16_pair(v[0], v[1]), bf16_pair(v[2], v[3]));
          }
          uint2* dst = reinterpret_cast<uint2*>(static_cast<uint16_t*>(out) + m * kHeadDim + d);
          if constexpr (kStream) {
            __stcs(dst, o);
          } else {
            *dst = o;
          }
        } else {
          float4* dst = reinterpret_cast<float4*>(static_cast<float*>(out) + m * kHeadDim + d);
          if constexpr (kStream) {
            __stcs(dst, make_float4(v[0], v[1], v[2], v[3]));
          } else {
            *dst = make_float4(v[0], v[1], v[2], v[3]);
          }
        }
      }
    }
  }
}

// bf16 output of a large call into 16-byte-aligned memory: lane L covers
// dims 256k + 8L .. 256k + 8L + 7 of the slot (k = 0, 1), so a slot is one
// 8-byte code load per lane and half (lanes 24..31 of half 1 load the 16
// bytes of RoPE words instead), the 8-byte scale record, and one 16-byte
// store per lane and half: 512-byte store instructions, half as many as the
// 4-dims-per-lane layout.  Same values, bit for bit.
template <int kUnroll>
__global__ void __launch_bounds__(kReaderThreads) kvc_dequant_wide16_kernel(
    const uint8_t* __restrict__ kv, int64_t num_pages, const int64_t* __restrict__ slots,
    int64_t num_slots, uint16_t* __restrict__ out, uint32_t* err) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  constexpr int kWarps = kReaderThreads / 32;
  const int lane = threadIdx.x & 31;
  const bool rope_lane = lane >= 24;  // in half 1: dims 448..511
  const int64_t width = static_cast<int64_t>(gridDim.x) * kWarps;
  for (int64_t base = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
       base < num_slots; base += width * kUnroll) {
    int64_t sl[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t m = base + u * width;
      sl[u] = m < num_slots ? __ldg(slots + m) : -1;
    }
    uint2 codes[kUnroll][2], scale[kUnroll];
    uint4 rope[kUnroll];
    bool ok[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      codes[u][0] = codes[u][1] = scale[u] = make_uint2(0u, 0u);
      rope[u] = make_uint4(0u, 0u, 0u, 0u);
      ok[u] = false;
      if (sl[u] < 0) continue;
      const int64_t page = sl[u] / kSlotsPerPage, off = sl[u] % kSlotsPerPage;
      if (page >= num_pages) {
        if (lane == 0) atomicCAS(err, 0u, kErrBadIndexReader);
        continue;
      }
      const uint8_t* pg = kv + page * kPageBytes;
      const uint8_t* payload = pg + off * kTokenStride;
      scale[u] = __ldg(reinterpret_cast<const uint2*>(pg + kScaleBase + off * kScaleDim));
      codes[u][0] = __ldg(reinterpret_cast<const uint2*>(payload + 8 * lane));
      if (!rope_lane)
        codes[u][1] = __ldg(reinterpret_cast<const uint2*>(payload + 256 + 8 * lane));
      else
        rope[u] = __ldg(reinterpret_cast<const uint4*>(payload + kNopeDim + 16 * (lane - 24)));
      ok[u] = true;
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t m = base + u * width;
      if (m >= num_slots) continue;
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int d = 256 * k + 8 * lane;
        uint4 o;
        if (k == 1 && rope_lane) {  // the stored bf16 words, copied as they are
          o = rope[u];
        } else {
          o = make_uint4(0u, 0u, 0u, 0u);
          if (ok[u]) {
            const int g = d / kGroup;
            const uint32_t sw = g < 4 ? scale[u].x : scale[u].y;
            const float hs = half_scale((sw >> (8 * (g & 3))) & 0xFFu);
            float v[8];
            decode4(codes[u][k].x, hs, v);
            decode4(codes[u][k].y, hs, v + 4);
            o = make_uint4(bf16_pair(v[0], v[1]), bf16_pair(v[2], v[3]), bf16_pair(v[4], v[5]),
                           bf16_pair(v[6], v[7]));
          }
        }
        *reinterpret_cast<uint4*>(out + m * kHeadDim + d) = o;
      }
    }
  }
}

}  // namespace

namespace {

// Large-call kernels, measured on 262,144 slots in random order, with the
// exact decode (no conversion instruction, no library scaling call):
// fp32 output: 4 slots per warp and pass, streaming stores: 111.9 us
//   (2 / 6 / 8 slots: 118.4 / 119.5 / 137.4 us; plain stores at 4: 113.5;
//   the earlier ldexpf decode at 8 slots: 112.2);
// bf16 output (16-byte aligned, wide16): 2 slots per warp and pass, plain
//   stores: 68.2 us (72.2 with the ldexpf decode and a cvt per value).
constexpr auto kWarpF32 = &kvc_dequant_warp_kernel<4, true>;
constexpr auto kWarpBf16 = &kvc_dequant_warp_kernel<2, false>;
constexpr auto kWide16Bf16 = &kvc_dequant_wide16_kernel<2>;

// CTAs of a kernel that fit on the current device at once (cached per device).
int resident_ctas(int dev, const void* kernel, std::atomic<int>* cache) {
  int n = cache[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    int sms = 0, per_sm = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kReaderThreads, 0) !=
            cudaSuccess)
      return 0;
    n = sms * (per_sm > 0 ? per_sm : 1);
    cache[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

}  // namespace

cudaError_t launch_dequantize(const uint8_t* kv, int64_t num_pages, const int64_t* slots,
                              int64_t num_slots, void* out, int out_bf16, uint32_t* err,
                              cudaStream_t stream) {
  static std::atomic<int> small_cap[64], f32_cap[64], bf16_cap[64], wide_cap[64];  // 0: unknown
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  const void* small_fn = reinterpret_cast<const void*>(&kvc_dequant_kernel<1>);
  const bool wide16 = out_bf16 && (reinterpret_cast<uintptr_t>(out) & 15u) == 0;
  const void* large_fn = wide16     ? reinterpret_cast<const void*>(kWide16Bf16)
                         : out_bf16 ? reinterpret_cast<const void*>(kWarpBf16)
                                    : reinterpret_cast<const void*>(kWarpF32);
  const int cap_s = resident_ctas(dev, small_fn, small_cap);
  const int cap_l = resident_ctas(dev, large_fn, wide16 ? wide_cap : out_bf16 ? bf16_cap : f32_cap);
  if (cap_s == 0 || cap_l == 0) return cudaErrorInvalidDevice;
  // up to a device-full of slot pairs: one CTA per pair, 128 threads per slot
  // (the shortest chain); beyond that a persistent grid of warp-per-slot CTAs
  const int64_t pairs = (num_slots + kSlotsPerCta - 1) / kSlotsPerCta;
  const bool large = pairs > cap_s;
  const int64_t warps8 = (num_slots + 7) / 8;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(large ? (warps8 < cap_l ? warps8 : cap_l) : pairs));
  cfg.blockDim = dim3(kReaderThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e;
  if (!large) {
    e = cudaLaunchKernelEx(&cfg, &kvc_dequant_kernel<1>, kv, num_pages, slots, num_slots, out,
                           out_bf16, err);
  } else if (wide16) {
    e = cudaLaunchKernelEx(&cfg, kWide16Bf16, kv, num_pages, slots, num_slots,
                           static_cast<uint16_t*>(out), err);
  } else if (out_bf16) {
    e = cudaLaunchKernelEx(&cfg, kWarpBf16, kv, num_pages, slots, num_slots, out, out_bf16, err);
  } else {
    e = cudaLaunchKernelEx(&cfg, kWarpF32, kv, num_pages, slots, num_slots, out, out_bf16, err);
  }
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace kvc
