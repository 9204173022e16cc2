// Stream-K route of the KV-cache window compressor (sm_103a).
//
// The same computation as the cluster route (kvc_cluster.cu) -- the
// window compressor of "How One Output Is Produced" in the KernelGen
// Challenge 8 write-up -- with a different work split: one unit is one 8-row
// physical block of one output's window, the units of all outputs form one
// sequence u = n K + k, and a persistent grid of G CTAs takes contiguous,
// equal slices of it.  An output whose units fall in one CTA is finalised
// there; an output split between CTAs leaves partial softmax states
// (m, den, num per dimension) in the caller's workspace and the last CTA to
// arrive on the output's counter merges them and finalises (no waiting).
// It needs no thread-block clusters; it is the route for devices or
// configurations where the cluster route is unavailable, and it is the route
// that uses scratch memory (the workspace, or the library's static buffer).
// It takes a bf16 state whose 8-row blocks are 16 KiB contiguous (any block
// stride, any block-table strides) and block-aligned windows.
// One launch compresses one layer (the layer-0 pointers of its Params); the
// host launches it once per layer of a multi-layer call.
//
// Warp 8 resolves block_table entries 32 units at a time and issues one
// cp.async.bulk of 16 KiB per unit into a kStages ring; warps 0-7 fold the
// staged blocks (thread t owns dims 2t, 2t+1).  Every wait is bounded.

#include <cuda_runtime.h>

#include "kvc_device.cuh"

namespace kvc {
namespace {

using namespace dev;

struct StreamKShared {
  unsigned long long full_bar[kStages];
  unsigned long long empty_bar[kStages];
  MetaRec meta[kMetaRing];
  FinalScratch fs;
  uint32_t stage_ok[kStages];
  int abort_flag;
  int ticket;
};

// cta_of(u): the CTA whose slice [floor(g U / G), floor((g+1) U / G)) holds u.
__device__ __forceinline__ int64_t cta_of(int64_t u, int64_t U, int64_t G) {
  return ((u + 1) * G - 1) / U;
}

__device__ void producer(const Params& p, StreamKShared& sh, uint8_t* ring, int64_t u0, int64_t u1) {
  const int lane = threadIdx.x & 31;
  const int K = p.blocks_per_output;
  const uint64_t policy = evict_first_policy();
  int stage = 0;
  uint32_t phase = 0;
  uint32_t issued = 0, last_parity = 0;  // per-stage bit masks (lane 0)
  long long piece_base = 0;              // pieces started before this chunk
  bool stop = false;
  for (int64_t base = u0; base < u1 && !stop; base += 32) {
    const int64_t u = base + lane;
    long long blk = -1;
    MetaRec rec{-1, -1};
    int first = 0;
    if (u < u1) {
      const int64_t n = u / K;
      const int k = static_cast<int>(u - n * K);
      first = (k == 0 || u == u0);
      resolve_unit(p, n, k, first != 0, blk, rec);
    }
    const uint32_t fm = __ballot_sync(0xffffffffu, first);
    const long long piece = piece_base + __popc(fm & ((1u << lane) - 1u));
    piece_base += __popc(fm);
    const int cnt = static_cast<int>(u1 - base < 32 ? u1 - base : 32);
    for (int j = 0; j < cnt; ++j) {
      const long long gb = __shfl_sync(0xffffffffu, blk, j);
      const long long pj = __shfl_sync(0xffffffffu, piece, j);
      const long long slot_j = __shfl_sync(0xffffffffu, rec.slot, j);
      const long long pc_j = __shfl_sync(0xffffffffu, rec.pc, j);
      if (lane == 0) {
        if (*reinterpret_cast<volatile int*>(&sh.abort_flag)) {
          stop = true;
        } else if (!mbar_wait_bounded(&sh.empty_bar[stage], phase ^ 1u, p.wait_limit)) {
          record_error(p.error, kErrTimeout);
          *reinterpret_cast<volatile int*>(&sh.abort_flag) = 1;
          stop = true;
        } else {
          if ((fm >> j) & 1u) {
            MetaRec& m = sh.meta[pj % kMetaRing];
            m.slot = slot_j;
            m.pc = pc_j;
          }
          if (gb >= 0) {
            sh.stage_ok[stage] = 1;
            mbar_arrive_expect_tx(&sh.full_bar[stage], kBlockBytes);
            bulk_copy_g2s(ring + static_cast<size_t>(stage) * kBlockBytes,
                          p.states[0] + gb * p.state_block_bytes, kBlockBytes,
                          &sh.full_bar[stage], policy);
          } else {
            sh.stage_ok[stage] = 0;
            mbar_arrive(&sh.full_bar[stage]);
          }
          issued |= 1u << stage;
          last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
        }
      }
      stop = __shfl_sync(0xffffffffu, stop, 0);
      if (stop) break;
      if (++stage == kStages) { stage = 0; phase ^= 1u; }
    }
  }
  // No bulk copy may still target this CTA's shared memory when it exits.
  if (lane == 0) {
    for (int s = 0; s < kStages; ++s)
      if ((issued >> s) & 1u)
        if (!mbar_wait_drain(&sh.full_bar[s], (last_parity >> s) & 1u))
          record_error(p.error, kErrTimeout);
  }
}

__device__ __forceinline__ void finalize_whole(const Params& p, StreamKShared& sh, int64_t n, float c0,
                                               float c1, bool bad, const MetaRec& meta, float cs,
                                               float sn) {
  const float2 w = __ldg(reinterpret_cast<const float2*>(p.weights[0] + 2 * threadIdx.x));
  const float total = consumer_sum_squares(sh.fs, c0, c1);
  finalize_slice(p, sh.fs, 0, n, true, 2 * threadIdx.x, c0, c1, w, bad, meta, cs, sn, total, 0,
                 kHeadDim);
}

// Store this CTA's partial state of output n; the last CTA to arrive merges
// every partial of n (loads issued four pieces at a time) and finalises it.
__device__ void flush_partial(const Params& p, StreamKShared& sh, int64_t n, int64_t g, int64_t G,
                              int64_t n_first, const SoftmaxState& s, bool bad, const MetaRec& meta,
                              float cs, float sn) {
  const int t = threadIdx.x;
  const int64_t U = p.num_units, K = p.blocks_per_output;
  const int which = (n == n_first) ? 0 : 1;  // this CTA's first or last piece
  float* rec = p.partials + (g * 2 + which) * kPartialFloats;
  __stcg(reinterpret_cast<float2*>(rec) + t, make_float2(s.m0, s.m1));
  __stcg(reinterpret_cast<float2*>(rec + kHeadDim) + t, make_float2(s.d0, s.d1));
  __stcg(reinterpret_cast<float2*>(rec + 2 * kHeadDim) + t, make_float2(s.a0, s.a1));
  const bool any_bad = consumer_any(bad);  // also orders every thread's stores before t0's
  if (t == 0) {
    __stcg(p.part_status + g * 2 + which, any_bad ? 1 : 0);
    int ticket;
    // release: this CTA's partial is visible before the count moves;
    // acquire: if last, every other CTA's partial is visible to this CTA
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;"
                 : "=r"(ticket)
                 : "l"(p.counters + n)
                 : "memory");
    sh.ticket = ticket;
  }
  consumer_sync();
  const int64_t gf = cta_of(n * K, U, G), gl = cta_of(n * K + K - 1, U, G);
  if (sh.ticket != static_cast<int>(gl - gf)) return;  // uniform across consumers

  if (t == 0) p.counters[n] = 0;  // ready for the next call
  float M0 = -INFINITY, M1 = -INFINITY, D0 = 0.f, D1 = 0.f, A0 = 0.f, A1 = 0.f;
  bool mbad = false;
  for (int64_t g0 = gf; g0 <= gl; g0 += 4) {
    float2 m[4], d[4], a[4];
    int st[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int64_t gg = g0 + q;
      if (gg <= gl) {
        const int wh = (n == (gg * U / G) / K) ? 0 : 1;
        const float* r = p.partials + (gg * 2 + wh) * kPartialFloats;
        m[q] = __ldcg(reinterpret_cast<const float2*>(r) + t);
        d[q] = __ldcg(reinterpret_cast<const float2*>(r + kHeadDim) + t);
        a[q] = __ldcg(reinterpret_cast<const float2*>(r + 2 * kHeadDim) + t);
        st[q] = __ldcg(p.part_status + gg * 2 + wh);
      } else {
        m[q] = make_float2(-INFINITY, -INFINITY);
        d[q] = a[q] = make_float2(0.f, 0.f);
        st[q] = 0;
      }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float n0 = fmaxf(M0, m[q].x), n1 = fmaxf(M1, m[q].y);
      const float r0 = fast_ex2((M0 - n0) * kLog2e), r1 = fast_ex2((M1 - n1) * kLog2e);
      const float f0 = fast_ex2((m[q].x - n0) * kLog2e), f1 = fast_ex2((m[q].y - n1) * kLog2e);
      D0 = fmaf(d[q].x, f0, D0 * r0);
      D1 = fmaf(d[q].y, f1, D1 * r1);
      A0 = fmaf(a[q].x, f0, A0 * r0);
      A1 = fmaf(a[q].y, f1, A1 * r1);
      M0 = n0;
      M1 = n1;
      mbad |= st[q] != 0;
    }
  }
  finalize_whole(p, sh, n, A0 / D0, A1 / D1, mbad, meta, cs, sn);
}

__device__ void consumer(const Params& p, StreamKShared& sh, const uint8_t* ring, int64_t u0,
                         int64_t u1, int64_t g, int64_t G) {
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int K = p.blocks_per_output;
  const int64_t n_first = u0 / K;
  int64_t n = n_first;
  int k = static_cast<int>(u0 - n * K);
  int stage = 0;
  uint32_t phase = 0;
  long long piece = -1;
  SoftmaxState s;
  state_reset(s);
  bool bad = false, from_start = false;
  MetaRec meta{-1, -1};
  float cs = 1.f, sn = 0.f;
  for (int64_t u = u0; u < u1; ++u) {
    bool ready = false;
    if (!*reinterpret_cast<volatile int*>(&sh.abort_flag)) {
      ready = mbar_wait_bounded(&sh.full_bar[stage], phase, p.wait_limit);
      if (!ready) {
        record_error(p.error, kErrTimeout);
        *reinterpret_cast<volatile int*>(&sh.abort_flag) = 1;
      }
    }
    if (k == 0 || u == u0) {  // first unit of a piece: take its record
      ++piece;
      from_start = (k == 0);
      if (ready) {
        meta = sh.meta[piece % kMetaRing];
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
        finalize_whole(p, sh, n, s.a0 / s.d0, s.a1 / s.d1, bad, meta, cs, sn);
      } else {
        flush_partial(p, sh, n, g, G, n_first, s, bad, meta, cs, sn);
      }
      state_reset(s);
      bad = false;
    }
    if (++k == K) { k = 0; ++n; }
  }
}

__global__ void __launch_bounds__(kThreads, 2) kvc_streamk_kernel(const Params p) {
  extern __shared__ __align__(128) uint8_t smem[];
  StreamKShared& sh = *reinterpret_cast<StreamKShared*>(smem + static_cast<size_t>(kStages) * kBlockBytes);
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
  // Wait for the previous grid on the stream (programmatic dependent launch)
  // before touching any global memory, and let the next one start launching.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  __syncthreads();
  if (u0 >= u1) return;
  if (threadIdx.x >= kConsumerThreads) {
    producer(p, sh, smem, u0, u1);
  } else {
    consumer(p, sh, smem, u0, u1, g, G);
  }
}

}  // namespace

size_t streamk_smem_bytes() {
  return static_cast<size_t>(kStages) * kBlockBytes + sizeof(StreamKShared);
}

const void* streamk_kernel_symbol() { return reinterpret_cast<const void*>(&kvc_streamk_kernel); }

cudaError_t launch_streamk(const Params& p, int ctas, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(ctas));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = streamk_smem_bytes();
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, &kvc_streamk_kernel, p);
  return e != cudaSuccess ? e : cudaGetLastError();
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
