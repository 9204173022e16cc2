// kvc_compress_static: the same compression as kvc_compress, for callers
// that cannot allocate device memory.
//
// Some callers have no way to call cudaMalloc: plugins that are handed only
// their input and output pointers by a host engine, engines that reserve the
// whole device memory pool up front and forbid allocation at run time, and
// latency-critical paths where cudaMalloc's implicit device synchronisation
// is not acceptable.  They cannot provide the workspace kvc_compress needs
// for outputs whose window is split between CTAs.  This entry point instead
// uses a scratch buffer that lives inside the library: a file-scope
// __device__ array that every device loading the library holds until the
// process exits.
//
// The buffer is shared by every call on a device and keeps what the last call
// left in it.  Its arrival counters are cleared (cudaMemsetAsync on the
// caller's stream) once every argument check has passed, right before the
// launch, so a refused call writes nothing; calls that overlap on the GPU
// would use the same buffer at once and race, so callers must order them
// (one stream, or events).

#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/kvc.h"
#include "kvc_internal.h"

namespace {

// Size of the library-owned scratch buffer: 8 MiB.  On a 152-SM GPU the
// partial softmax states take about 3.6 MiB of it and the rest holds the
// arrival counters, one int per output (about a million outputs).
constexpr size_t kStaticScratchBytes = size_t{8} << 20;

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_static_mutex;
struct StaticAddress {
  unsigned long long ctx = 0;  // context the address belongs to (kvc::context_id)
  void* ptr = nullptr;
};
StaticAddress g_static[kMaxDevices];

// Device address of g_static_scratch on the current device.  Host code only
// sees a host-side stand-in under the array's name; a kernel must be given
// the address cudaGetSymbolAddress returns.  Looked up once per device and
// context: after cudaDeviceReset the library's module is loaded again in a
// new context, and the address is looked up again.
kvc_status static_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KVC_ERR_CUDA;
  const unsigned long long ctx = kvc::context_id();
  std::lock_guard<std::mutex> lock(g_static_mutex);
  StaticAddress& a = g_static[dev];
  if (a.ptr == nullptr || ctx == 0 || a.ctx != ctx) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_static_scratch) != cudaSuccess || ptr == nullptr)
      return KVC_ERR_CUDA;
    a.ptr = ptr;
    a.ctx = kvc::context_id();  // the lookup made a context current
  }
  *out = a.ptr;
  return KVC_OK;
}

// The bytes to clear before a launch: the arrival counters.
struct ClearRange {
  unsigned char* at;
  size_t bytes;
};

cudaError_t clear_counters(void* ctx, cudaStream_t stream) {
  const ClearRange* r = static_cast<const ClearRange*>(ctx);
  return cudaMemsetAsync(r->at, 0, r->bytes, stream);
}

}  // namespace

extern "C" kvc_status kvc_compress_static(
    const void* state_cache, int64_t num_state_blocks, const int32_t* token_to_req,
    const int64_t* positions, int64_t num_tokens, const int64_t* boundary_token_indices,
    int64_t num_outputs, const int32_t* block_table, int64_t num_reqs,
    int64_t max_blocks_per_req, const float* rms_norm_weight, const float* cos_sin_cache,
    int64_t num_positions, const int64_t* kv_slot_mapping, int64_t slot_mapping_len,
    uint8_t* kv_cache, int64_t num_kv_pages, int32_t block_size, int32_t compress_ratio,
    float rms_norm_eps, float* y_out, uint32_t flags, void* stream) {
  void* scratch = nullptr;
  ClearRange clear{nullptr, 0};
  if (num_outputs > 0) {
    // Workspace layout: partial states first, the arrival counters from
    // offset kvc_workspace_bytes(0) to kvc_workspace_bytes(num_outputs).
    const size_t counters_at = kvc_workspace_bytes(0);
    const size_t need = kvc_workspace_bytes(num_outputs);
    if (counters_at == 0 || need == 0) return KVC_ERR_CUDA;
    if (need > kStaticScratchBytes) return KVC_ERR_SCRATCH_LIMIT;
    const kvc_status st = static_scratch(&scratch);
    if (st != KVC_OK) return st;
    clear = ClearRange{static_cast<unsigned char*>(scratch) + counters_at, need - counters_at};
  }
  const kvc::PreLaunch hook{&clear_counters, &clear};
  return kvc::compress_hooked(state_cache, num_state_blocks, token_to_req, positions, num_tokens,
                              boundary_token_indices, num_outputs, block_table, num_reqs,
                              max_blocks_per_req, rms_norm_weight, cos_sin_cache, num_positions,
                              kv_slot_mapping, slot_mapping_len, kv_cache, num_kv_pages,
                              block_size, compress_ratio, rms_norm_eps, y_out, scratch,
                              scratch ? kStaticScratchBytes : 0, flags, stream,
                              scratch ? &hook : nullptr);
}
