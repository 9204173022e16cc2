// C ABI of the KV-cache window compressor (declared in include/kvc.h):
// host-side argument validation, per-device launch capacity, workspace
// sizing, device error reporting.  The computation itself is the fused
// kernel of kvc_compress.cu.

#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "../../include/kvc.h"
#include "kvc_internal.h"

namespace {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  bool ready = false;
  int sms = 0;
  int ctas_per_sm = 0;
  uint32_t* error_word = nullptr;
};

std::mutex g_mutex;
DeviceInfo g_devices[kMaxDevices];

// Per-device set-up on first use: shared-memory opt-in, occupancy, error word.
kvc_status device_info(DeviceInfo* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KVC_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceInfo& d = g_devices[dev];
  if (!d.ready) {
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return KVC_ERR_CUDA;
    const size_t smem = kvc::dynamic_smem_bytes();
    if (cudaFuncSetAttribute(kvc::kernel_symbol(), cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return KVC_ERR_CUDA;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kvc::kernel_symbol(), kvc::kThreads,
                                                      smem) != cudaSuccess ||
        per_sm < 1)
      return KVC_ERR_CUDA;
    uint32_t* err = kvc::device_error_word();
    if (err == nullptr) return KVC_ERR_CUDA;
    d.sms = sms;
    d.ctas_per_sm = per_sm;
    d.error_word = err;
    d.ready = true;
  }
  *out = d;
  return KVC_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int pick_ctas(const DeviceInfo& d, int64_t units, uint32_t flags) {
  const int64_t cap = static_cast<int64_t>(d.sms) * d.ctas_per_sm;
  int64_t g = (flags & KVC_FLAG_GRID_MASK) ? static_cast<int64_t>(flags & KVC_FLAG_GRID_MASK) : cap;
  if (g > cap) g = cap;
  if (g > units) g = units;
  return static_cast<int>(g < 1 ? 1 : g);
}

}  // namespace

extern "C" {

size_t kvc_workspace_bytes(int64_t num_outputs) {
  DeviceInfo d;
  if (device_info(&d) != KVC_OK) return 0;
  return kvc::workspace_layout(d.sms * d.ctas_per_sm, num_outputs).total;
}

kvc_status kvc_query_launch(int64_t num_outputs, int32_t compress_ratio, uint32_t flags,
                            int32_t* ctas, int32_t* threads, int32_t* smem_bytes) {
  if (num_outputs < 0 || compress_ratio <= 0 || compress_ratio % kvc::kBlockRows != 0 ||
      (flags & ~KVC_FLAG_GRID_MASK) != 0)
    return KVC_ERR_INVALID_ARG;
  DeviceInfo d;
  const kvc_status st = device_info(&d);
  if (st != KVC_OK) return st;
  const int64_t units = num_outputs * (compress_ratio / kvc::kBlockRows);
  if (ctas) *ctas = units > 0 ? pick_ctas(d, units, flags) : 0;
  if (threads) *threads = kvc::kThreads;
  if (smem_bytes) *smem_bytes = static_cast<int32_t>(kvc::dynamic_smem_bytes());
  return KVC_OK;
}

kvc_status kvc_compress(const void* state_cache, int64_t num_state_blocks,
                        const int32_t* token_to_req, const int64_t* positions, int64_t num_tokens,
                        const int64_t* boundary_token_indices, int64_t num_outputs,
                        const int32_t* block_table, int64_t num_reqs, int64_t max_blocks_per_req,
                        const float* rms_norm_weight, const float* cos_sin_cache,
                        int64_t num_positions, const int64_t* kv_slot_mapping,
                        int64_t slot_mapping_len, uint8_t* kv_cache, int64_t num_kv_pages,
                        int32_t block_size, int32_t compress_ratio, float rms_norm_eps,
                        float* y_out, void* workspace, size_t workspace_bytes, uint32_t flags,
                        void* stream) {
  if (num_outputs < 0 || (flags & ~KVC_FLAG_GRID_MASK) != 0) return KVC_ERR_INVALID_ARG;
  if (block_size != kvc::kBlockRows) return KVC_ERR_UNSUPPORTED;
  if (compress_ratio <= 0 || compress_ratio % kvc::kBlockRows != 0) return KVC_ERR_UNSUPPORTED;
  if (!std::isfinite(rms_norm_eps) || rms_norm_eps < 0.f) return KVC_ERR_INVALID_ARG;
  if (num_outputs == 0) return KVC_OK;
  if (!state_cache || !token_to_req || !positions || !boundary_token_indices || !block_table ||
      !rms_norm_weight || !cos_sin_cache || !kv_slot_mapping || !kv_cache || !workspace)
    return KVC_ERR_INVALID_ARG;
  if (num_state_blocks <= 0 || num_tokens <= 0 || num_reqs <= 0 || max_blocks_per_req <= 0 ||
      num_positions <= 0 || num_kv_pages <= 0)
    return KVC_ERR_INVALID_ARG;
  if (slot_mapping_len != num_tokens && slot_mapping_len != num_outputs) return KVC_ERR_INVALID_ARG;
  if (!aligned(state_cache, 16) || !aligned(kv_cache, 16) || !aligned(workspace, 16) ||
      !aligned(rms_norm_weight, 8) || (y_out && !aligned(y_out, 8)) ||
      !aligned(token_to_req, 4) || !aligned(block_table, 4) || !aligned(cos_sin_cache, 4) ||
      !aligned(positions, 8) || !aligned(boundary_token_indices, 8) || !aligned(kv_slot_mapping, 8))
    return KVC_ERR_INVALID_ARG;

  DeviceInfo d;
  const kvc_status st = device_info(&d);
  if (st != KVC_OK) return st;
  const int max_ctas = d.sms * d.ctas_per_sm;
  const kvc::WorkspaceLayout L = kvc::workspace_layout(max_ctas, num_outputs);
  if (workspace_bytes < L.total) return KVC_ERR_INVALID_ARG;

  kvc::Params p;
  p.state = static_cast<const uint16_t*>(state_cache);
  p.num_blocks = num_state_blocks;
  p.token_to_req = token_to_req;
  p.positions = positions;
  p.num_tokens = num_tokens;
  p.bti = boundary_token_indices;
  p.num_outputs = num_outputs;
  p.block_table = block_table;
  p.num_reqs = num_reqs;
  p.max_blocks = max_blocks_per_req;
  p.weight = rms_norm_weight;
  p.cos_sin = cos_sin_cache;
  p.num_positions = num_positions;
  p.slot_map = kv_slot_mapping;
  p.slot_by_token = (slot_mapping_len == num_tokens) ? 1 : 0;
  p.kv = kv_cache;
  p.num_pages = num_kv_pages;
  p.y_out = y_out;
  p.compress_ratio = compress_ratio;
  p.blocks_per_output = compress_ratio / kvc::kBlockRows;
  p.num_units = num_outputs * p.blocks_per_output;
  p.eps = rms_norm_eps;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  p.partials = reinterpret_cast<float*>(ws + L.partials);
  p.part_status = reinterpret_cast<int32_t*>(ws + L.status);
  p.counters = reinterpret_cast<int32_t*>(ws + L.counters);

  const int ctas = pick_ctas(d, p.num_units, flags);
  if (kvc::launch(p, ctas, static_cast<cudaStream_t>(stream)) != cudaSuccess) return KVC_ERR_CUDA;
  return KVC_OK;
}

kvc_status kvc_get_device_error(void* stream, uint32_t* out_code) {
  if (out_code == nullptr) return KVC_ERR_INVALID_ARG;
  DeviceInfo d;
  const kvc_status st = device_info(&d);
  if (st != KVC_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return KVC_ERR_CUDA;
  uint32_t code = 0;
  if (cudaMemcpy(&code, d.error_word, sizeof code, cudaMemcpyDeviceToHost) != cudaSuccess)
    return KVC_ERR_CUDA;
  if (code != 0 && cudaMemset(d.error_word, 0, sizeof code) != cudaSuccess) return KVC_ERR_CUDA;
  *out_code = code;
  return KVC_OK;
}

const char* kvc_error_string(kvc_status status) {
  switch (status) {
    case KVC_OK: return "ok";
    case KVC_ERR_INVALID_ARG: return "invalid argument";
    case KVC_ERR_UNSUPPORTED: return "unsupported configuration";
    case KVC_ERR_CUDA: return "CUDA runtime error";
    case KVC_ERR_BAD_INDEX: return "index outside its array";
    case KVC_ERR_TIMEOUT: return "pipeline wait timed out";
    case KVC_ERR_SCRATCH_LIMIT:
      return "problem needs more scratch than the library's built-in 8 MiB buffer holds";
  }
  return "unknown status";
}

const char* kvc_version(void) {
  return "kvc 0.1.0 sm_103a fused stream-K window compressor (bulk-copy ring, 6x16KiB stages)";
}

}  // extern "C"
