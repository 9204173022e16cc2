// Reader direction of the KV-cache window compressor: decode packed slots
// back into 512-vectors for the attention side.
//
// The slot layout is the one of "Gather and Scatter" in "From Attention to
// KV Cache Compression: Notes from a KernelGen Optimization" (KernelGen
// Challenge 8 write-up); the values are the ones its quantisation equation
// ("How One Output Is Produced") encodes: NOPE dim d < 448 reads back as
// q_d * 2^(scale[d / 64] - 127), RoPE dims 448..511 as the stored bf16.
//
// One slot per 128 threads, 4 dims per thread: a thread reads 4 int8 codes
// (or 4 bf16 RoPE values) and the group's scale byte, scales exactly with
// ldexpf and writes one 16-byte (fp32) or 8-byte (bf16) vector.  Memory-bound:
// 584 bytes read and 1 or 2 KiB written per slot.

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "kvc_internal.h"

namespace kvc {
namespace {

constexpr int kReaderThreads = 256;
constexpr int kThreadsPerSlot = kHeadDim / 4;   // 128
constexpr int kSlotsPerCta = kReaderThreads / kThreadsPerSlot;
constexpr uint32_t kErrBadIndexReader = 4;

__global__ void __launch_bounds__(kReaderThreads) kvc_dequant_kernel(
    const uint8_t* __restrict__ kv, int64_t num_pages, const int64_t* __restrict__ slots,
    int64_t num_slots, void* __restrict__ out, int out_bf16, uint32_t* err) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int64_t m = static_cast<int64_t>(blockIdx.x) * kSlotsPerCta + threadIdx.x / kThreadsPerSlot;
  if (m >= num_slots) return;
  const int t = threadIdx.x % kThreadsPerSlot;
  const int d0 = 4 * t;
  float v[4] = {0.f, 0.f, 0.f, 0.f};
  bool rope_bits = false;  // RoPE dims: the stored bf16 words, copied as they are
  uint2 raw = make_uint2(0u, 0u);
  const int64_t slot = __ldg(slots + m);
  if (slot >= 0) {
    const int64_t page = slot / kSlotsPerPage, off = slot % kSlotsPerPage;
    if (page >= num_pages) {
      if (t == 0) atomicCAS(err, 0u, kErrBadIndexReader);
    } else {
      const uint8_t* pg = kv + page * kPageBytes;
      const uint8_t* payload = pg + off * kTokenStride;
      if (d0 < kNopeDim) {
        const uint32_t w = __ldg(reinterpret_cast<const uint32_t*>(payload + d0));
        const int e = static_cast<int>(__ldg(pg + kScaleBase + off * kScaleDim + d0 / kGroup)) - 127;
#pragma unroll
        for (int i = 0; i < 4; ++i)
          v[i] = ldexpf(static_cast<float>(static_cast<int8_t>((w >> (8 * i)) & 0xFFu)), e);
      } else {
        raw = __ldg(reinterpret_cast<const uint2*>(payload + kNopeDim + 2 * (d0 - kNopeDim)));
        rope_bits = true;
        v[0] = __uint_as_float(raw.x << 16);
        v[1] = __uint_as_float(raw.x & 0xFFFF0000u);
        v[2] = __uint_as_float(raw.y << 16);
        v[3] = __uint_as_float(raw.y & 0xFFFF0000u);
      }
    }
  }
  if (out_bf16 && rope_bits) {
    reinterpret_cast<uint2*>(static_cast<uint16_t*>(out) + m * kHeadDim)[t] = raw;
  } else if (out_bf16) {
    uint2 o;
    o.x = static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(v[0]))) |
          (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(v[1]))) << 16);
    o.y = static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(v[2]))) |
          (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(v[3]))) << 16);
    reinterpret_cast<uint2*>(static_cast<uint16_t*>(out) + m * kHeadDim)[t] = o;
  } else {
    reinterpret_cast<float4*>(static_cast<float*>(out) + m * kHeadDim)[t] =
        make_float4(v[0], v[1], v[2], v[3]);
  }
}

}  // namespace

cudaError_t launch_dequantize(const uint8_t* kv, int64_t num_pages, const int64_t* slots,
                              int64_t num_slots, void* out, int out_bf16, uint32_t* err,
                              cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((num_slots + kSlotsPerCta - 1) / kSlotsPerCta));
  cfg.blockDim = dim3(kReaderThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, &kvc_dequant_kernel, kv, num_pages, slots, num_slots,
                                           out, out_bf16, err);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace kvc
