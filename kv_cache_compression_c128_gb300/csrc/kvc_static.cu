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
// caller's stream) before each launch; calls that overlap on the GPU would
// use the same buffer at once and race, so callers must order them (one
// stream, or events).

#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/kvc.h"

namespace {

// Size of the library-owned scratch buffer: 8 MiB.  On a 152-SM GPU the
// partial softmax states take about 3.6 MiB of it and the rest holds the
// arrival counters, one int per output (about a million outputs).
constexpr size_t kStaticScratchBytes = size_t{8} << 20;

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_static_mutex;
void* g_static_ptr[kMaxDevices] = {};

// Device address of g_static_scratch on the current device.  Host code only
// sees a host-side stand-in under the array's name; a kernel must be given
// the address cudaGetSymbolAddress returns.  Looked up once per device.
kvc_status static_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KVC_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_static_mutex);
  if (g_static_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_static_scratch) != cudaSuccess || ptr == nullptr)
      return KVC_ERR_CUDA;
    g_static_ptr[dev] = ptr;
  }
  *out = g_static_ptr[dev];
  return KVC_OK;
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
  if (num_outputs > 0) {
    const kvc_status st = static_scratch(&scratch);
    if (st != KVC_OK) return st;
    // Workspace layout: partial states first, the arrival counters from
    // offset kvc_workspace_bytes(0) to kvc_workspace_bytes(num_outputs).
    const size_t counters_at = kvc_workspace_bytes(0);
    const size_t need = kvc_workspace_bytes(num_outputs);
    if (counters_at == 0 || need == 0) return KVC_ERR_CUDA;
    if (need > kStaticScratchBytes) return KVC_ERR_SCRATCH_LIMIT;
    if (cudaMemsetAsync(static_cast<unsigned char*>(scratch) + counters_at, 0, need - counters_at,
                        static_cast<cudaStream_t>(stream)) != cudaSuccess)
      return KVC_ERR_CUDA;
  }
  return kvc_compress(state_cache, num_state_blocks, token_to_req, positions, num_tokens,
                      boundary_token_indices, num_outputs, block_table, num_reqs,
                      max_blocks_per_req, rms_norm_weight, cos_sin_cache, num_positions,
                      kv_slot_mapping, slot_mapping_len, kv_cache, num_kv_pages, block_size,
                      compress_ratio, rms_norm_eps, y_out, scratch,
                      scratch ? kStaticScratchBytes : 0, flags, stream);
}
