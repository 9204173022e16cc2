// C ABI of the KV-cache window compressor (declared in include/kvc.h):
// host-side argument validation, per-device set-up, the choice between the
// cluster route (kvc_cluster.cu) and the stream-K route (kvc_streamk.cu),
// workspace sizing and device error reporting.

#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "../../include/kvc.h"
#include "kvc_internal.h"

namespace {

// Limit on one pipeline wait of the kernels, in SM clock cycles: the default
// unless kvc_selftest_set_wait_limit shortened it.
std::atomic<long long> g_wait_limit{kvc::kDefaultWaitLimitCycles};

// Whether calls launched from now on poison their guessed first passes
// (kvc_selftest_poison_guesses).
std::atomic<int> g_poison_guesses{0};

// A driver entry point looked up through the runtime (no link against the
// driver library); null when the driver does not offer it.
template <typename Fn>
Fn driver_entry(const char* name) {
  void* f = nullptr;
  cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
  if (cudaGetDriverEntryPointByVersion(name, &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess) {
    (void)cudaGetLastError();
    return nullptr;
  }
  return reinterpret_cast<Fn>(f);
}

}  // namespace

namespace kvc {

unsigned long long context_id() {
  using GetCurrent = CUresult (*)(CUcontext*);
  using GetId = CUresult (*)(CUcontext, unsigned long long*);
  static const GetCurrent get_current = driver_entry<GetCurrent>("cuCtxGetCurrent");
  static const GetId get_id = driver_entry<GetId>("cuCtxGetId");
  CUcontext ctx = nullptr;
  if (get_current == nullptr || get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  unsigned long long id = 0;
  if (get_id != nullptr && get_id(ctx, &id) == CUDA_SUCCESS) return id + 1;  // never 0
  return static_cast<unsigned long long>(reinterpret_cast<uintptr_t>(ctx));
}

}  // namespace kvc

namespace {

// Device error word: the first error code a kernel recorded since the last
// kvc_get_device_error.  Kernels get its device address in Params::error.
__device__ uint32_t g_error_word;

// Guessed first passes that failed their check since the last
// kvc_selftest_first_pass_rejections.  Kernels get it in Params::rejections.
__device__ unsigned long long g_rejections;

constexpr int kMaxDevices = 64;

constexpr int kClusterSizes[] = {1, 2, 4, 8, 16};
constexpr int kNumClusterSizes = 5;

struct DeviceInfo {
  bool ready = false;
  unsigned long long ctx = 0;  // context the set-up was made in (kvc::context_id)
  int sms = 0;
  int streamk_ctas_per_sm = 0;
  int cluster_cap[kNumClusterSizes] = {};  // co-resident clusters per size
  uint32_t* error_word = nullptr;
  unsigned long long* rejections = nullptr;
};

std::mutex g_mutex;
DeviceInfo g_devices[kMaxDevices];

// Per-device set-up on first use (with that device current): shared-memory
// opt-in and occupancy of both routes, address of the error word.  All of it
// belongs to the CUDA context it was made in; when another context is
// current (after cudaDeviceReset, or a context the caller created), the
// set-up is made again.
kvc_status device_info(DeviceInfo* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KVC_ERR_CUDA;
  const unsigned long long ctx = kvc::context_id();
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceInfo& d = g_devices[dev];
  if (!d.ready || ctx == 0 || d.ctx != ctx) {
    d.ready = false;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return KVC_ERR_CUDA;
    const size_t smem = kvc::streamk_smem_bytes();
    if (cudaFuncSetAttribute(kvc::streamk_kernel_symbol(),
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return KVC_ERR_CUDA;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kvc::streamk_kernel_symbol(),
                                                      kvc::kThreads, smem) != cudaSuccess ||
        per_sm < 1)
      return KVC_ERR_CUDA;
    for (int i = 0; i < kNumClusterSizes; ++i) d.cluster_cap[i] = kvc::cluster_capacity(kClusterSizes[i]);
    void* err = nullptr;
    if (cudaGetSymbolAddress(&err, g_error_word) != cudaSuccess || err == nullptr) return KVC_ERR_CUDA;
    void* rej = nullptr;
    if (cudaGetSymbolAddress(&rej, g_rejections) != cudaSuccess || rej == nullptr) return KVC_ERR_CUDA;
    d.sms = sms;
    d.streamk_ctas_per_sm = per_sm;
    d.error_word = static_cast<uint32_t*>(err);
    d.rejections = static_cast<unsigned long long*>(rej);
    d.ctx = kvc::context_id();  // the set-up's runtime calls made a context current
    d.ready = true;
  }
  *out = d;
  return KVC_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Bytes of one 8-row chunk of a state row type.
double chunk_bytes_of(int32_t dtype) {
  return static_cast<double>(kvc::kBlockRows) * kvc::kRowElems * (dtype == KVC_DTYPE_F32 ? 4 : 2);
}

struct Route {
  bool stream_k;
  int count;     // stream-K: CTAs; cluster route: clusters
  int cluster;   // cluster route: CTAs per output
};

int cluster_index(int S) {
  for (int i = 0; i < kNumClusterSizes; ++i)
    if (kClusterSizes[i] == S) return i;
  return -1;
}

// Clusters for N outputs at a capacity of `cap` co-resident clusters: the
// fewest that keep the largest per-cluster output count at its minimum, so
// that every CTA streams (nearly) the same number of blocks.
int64_t balanced_clusters(int64_t N, int cap) {
  const int64_t most = N < cap ? N : cap;
  const int64_t rounds = (N + most - 1) / most;
  return (N + rounds - 1) / rounds;
}

// Cluster size for N outputs of K chunks of chunk_bytes each: the estimated
// time of the slowest CTA -- its chunks times the time one chunk takes when
// A CTAs share the HBM (about 6.4 TB/s in all; one CTA's copy pipeline alone
// delivers about 34 GB/s) -- plus about 1 us per cross-CTA merge.  Ties go
// to the smaller cluster.  0 if no cluster size fits.
int auto_cluster_size(const DeviceInfo& d, int64_t N, int64_t K, double chunk_bytes) {
  constexpr double kTotalBytesPerUs = 6.4e6, kCtaBytesPerUs = 3.4e4, kMergeUs = 1.0;
  int best = 0;
  double best_t = 1e300;
  for (int i = 0; i < kNumClusterSizes; ++i) {
    const int S = kClusterSizes[i];
    if (S > K || d.cluster_cap[i] < 1) continue;
    const int64_t ncl = balanced_clusters(N, d.cluster_cap[i]);
    const double rounds = static_cast<double>((N + ncl - 1) / ncl);
    const double kmax = static_cast<double>((K + S - 1) / S);
    const double A = static_cast<double>(ncl) * S;
    const double rate = kCtaBytesPerUs < kTotalBytesPerUs / A ? kCtaBytesPerUs : kTotalBytesPerUs / A;
    const double t = rounds * kmax * chunk_bytes / rate + (S > 1 ? rounds * kMergeUs : 0.0);
    if (t < best_t * (1.0 - 1e-9)) {
      best_t = t;
      best = S;
    }
  }
  return best;
}

// Route for N outputs of K chunks of chunk_bytes.  `streamk_ok` = a bf16
// state with adjacent rows, block_size 8 and C a multiple of 8 (the stream-K
// route handles only those; the window start is checked on the device).
bool pick_route(const DeviceInfo& d, int64_t N, int64_t K, bool streamk_ok, double chunk_bytes,
                uint32_t flags, Route* r) {
  const int forced_count = static_cast<int>(flags & KVC_FLAG_GRID_MASK);
  const int forced_s = static_cast<int>((flags & KVC_FLAG_CLUSTER_MASK) >> KVC_FLAG_CLUSTER_SHIFT);
  const int S = (flags & KVC_FLAG_STREAM_K)
                    ? 0
                    : (forced_s ? forced_s : auto_cluster_size(d, N, K, chunk_bytes));
  if (S == 0) {  // stream-K: asked for, or no cluster size fits this device
    if (!streamk_ok) return false;
    const int64_t units = N * K;
    const int64_t cap = static_cast<int64_t>(d.sms) * d.streamk_ctas_per_sm;
    int64_t g = forced_count ? forced_count : cap;
    if (g > cap) g = cap;
    if (g > units) g = units;
    *r = Route{true, static_cast<int>(g < 1 ? 1 : g), 0};
    return true;
  }
  const int ci = cluster_index(S);
  if (ci < 0 || S > K || d.cluster_cap[ci] < 1) return false;
  int64_t ncl = forced_count ? forced_count : balanced_clusters(N, d.cluster_cap[ci]);
  if (ncl > d.cluster_cap[ci]) ncl = d.cluster_cap[ci];
  if (ncl > N) ncl = N;
  *r = Route{false, static_cast<int>(ncl < 1 ? 1 : ncl), S};
  return true;
}

}  // namespace

extern "C" {

size_t kvc_workspace_bytes(int64_t num_outputs) {
  DeviceInfo d;
  if (device_info(&d) != KVC_OK) return 0;
  return kvc::workspace_layout(d.sms * d.streamk_ctas_per_sm, num_outputs).total;
}

kvc_status kvc_query_launch_ex(int64_t num_outputs, int32_t compress_ratio,
                               int32_t state_dtype, uint32_t flags, int32_t* ctas,
                               int32_t* cluster_size, int32_t* threads, int32_t* smem_bytes) {
  if (num_outputs < 0 || compress_ratio <= 0 || (flags & ~KVC_FLAG_ALL) != 0 ||
      (state_dtype != KVC_DTYPE_BF16 && state_dtype != KVC_DTYPE_F32))
    return KVC_ERR_INVALID_ARG;
  DeviceInfo d;
  const kvc_status st = device_info(&d);
  if (st != KVC_OK) return st;
  Route r{false, 0, 1};
  const int64_t K = (compress_ratio + kvc::kBlockRows - 1) / kvc::kBlockRows;
  const bool bf16 = state_dtype == KVC_DTYPE_BF16;
  if (num_outputs > 0 &&
      !pick_route(d, num_outputs, K, bf16 && compress_ratio % kvc::kBlockRows == 0,
                  chunk_bytes_of(state_dtype), flags, &r))
    return KVC_ERR_UNSUPPORTED;
  if (ctas) *ctas = num_outputs > 0 ? (r.stream_k ? r.count : r.count * r.cluster) : 0;
  if (cluster_size) *cluster_size = r.stream_k ? 0 : r.cluster;
  if (threads) *threads = r.stream_k ? kvc::kThreads : kvc::cluster_threads();
  if (smem_bytes)
    *smem_bytes = static_cast<int32_t>(r.stream_k ? kvc::streamk_smem_bytes()
                                                  : kvc::cluster_smem_bytes(r.cluster));
  return KVC_OK;
}

kvc_status kvc_query_launch(int64_t num_outputs, int32_t compress_ratio, uint32_t flags,
                            int32_t* ctas, int32_t* cluster_size, int32_t* threads,
                            int32_t* smem_bytes) {
  return kvc_query_launch_ex(num_outputs, compress_ratio, KVC_DTYPE_BF16, flags, ctas,
                             cluster_size, threads, smem_bytes);
}

}  // extern "C"

namespace {

// State element type and strides (elements), block-table strides.
struct StateLayout {
  int32_t dtype;
  int64_t block_stride, row_stride;
  int64_t bt_row_stride, bt_col_stride;
};

StateLayout contiguous_layout(int32_t block_size, int64_t max_blocks_per_req) {
  return StateLayout{KVC_DTYPE_BF16, static_cast<int64_t>(block_size) * kvc::kRowElems,
                     kvc::kRowElems, max_blocks_per_req, 1};
}

// kvc_compress for L layers that share every index array: host arrays of L
// device pointers for the state caches, weights and kv caches.
kvc_status compress_layers(int32_t L, const void* const* state_caches, const StateLayout& lay,
                           int64_t num_state_blocks,
                           const int32_t* token_to_req, const int64_t* positions,
                           int64_t num_tokens, const int64_t* boundary_token_indices,
                           int64_t num_outputs, const int32_t* block_table, int64_t num_reqs,
                           int64_t max_blocks_per_req, const float* const* rms_norm_weights,
                           const float* cos_sin_cache, int64_t num_positions,
                           const int64_t* kv_slot_mapping, int64_t slot_mapping_len,
                           uint8_t* const* kv_caches, int64_t num_kv_pages, int32_t block_size,
                           int32_t compress_ratio, float rms_norm_eps, float* y_out,
                           void* workspace, size_t workspace_bytes, uint32_t flags, void* stream,
                           const kvc::PreLaunch* pre_launch = nullptr) {
  if (num_outputs < 0 || (flags & ~KVC_FLAG_ALL) != 0) return KVC_ERR_INVALID_ARG;
  if (L < 1 || L > kvc::kMaxLayers) return KVC_ERR_INVALID_ARG;
  if (lay.dtype != KVC_DTYPE_BF16 && lay.dtype != KVC_DTYPE_F32) return KVC_ERR_INVALID_ARG;
  if (lay.block_stride < 0 || lay.row_stride < 0 || lay.bt_row_stride < 0 || lay.bt_col_stride < 0)
    return KVC_ERR_INVALID_ARG;
  const int64_t esize = lay.dtype == KVC_DTYPE_F32 ? 4 : 2;
  if ((lay.block_stride * esize) % 16 != 0 || (lay.row_stride * esize) % 16 != 0)
    return KVC_ERR_UNSUPPORTED;
  if (block_size < kvc::kBlockRows) return KVC_ERR_UNSUPPORTED;
  if (compress_ratio <= 0) return KVC_ERR_INVALID_ARG;
  if (!std::isfinite(rms_norm_eps) || rms_norm_eps < 0.f) return KVC_ERR_INVALID_ARG;
  if (num_outputs == 0) return KVC_OK;
  if (!state_caches || !rms_norm_weights || !kv_caches) return KVC_ERR_INVALID_ARG;
  for (int l = 0; l < L; ++l) {
    if (!state_caches[l] || !rms_norm_weights[l] || !kv_caches[l]) return KVC_ERR_INVALID_ARG;
    if (!aligned(state_caches[l], 16) || !aligned(kv_caches[l], 16) ||
        !aligned(rms_norm_weights[l], 8))
      return KVC_ERR_INVALID_ARG;
  }
  if (!token_to_req || !positions || !boundary_token_indices || !block_table || !cos_sin_cache ||
      !kv_slot_mapping || !workspace)
    return KVC_ERR_INVALID_ARG;
  if (num_state_blocks <= 0 || num_tokens <= 0 || num_reqs <= 0 || max_blocks_per_req <= 0 ||
      num_positions <= 0 || num_kv_pages <= 0)
    return KVC_ERR_INVALID_ARG;
  if (slot_mapping_len != num_tokens && slot_mapping_len != num_outputs) return KVC_ERR_INVALID_ARG;
  // every byte offset the kernels form must fit in int64
  const __int128 state_end = static_cast<__int128>(lay.block_stride) * (num_state_blocks - 1) +
                             static_cast<__int128>(lay.row_stride) * (block_size - 1) + kvc::kRowElems;
  const __int128 table_end = static_cast<__int128>(lay.bt_row_stride) * (num_reqs - 1) +
                             static_cast<__int128>(lay.bt_col_stride) * (max_blocks_per_req - 1);
  if (state_end * esize > INT64_MAX || table_end > INT64_MAX / 4) return KVC_ERR_INVALID_ARG;
  if (!aligned(workspace, 16) || (y_out && !aligned(y_out, 8)) || !aligned(token_to_req, 4) ||
      !aligned(block_table, 4) || !aligned(cos_sin_cache, 4) || !aligned(positions, 8) ||
      !aligned(boundary_token_indices, 8) || !aligned(kv_slot_mapping, 8))
    return KVC_ERR_INVALID_ARG;

  DeviceInfo d;
  const kvc_status st = device_info(&d);
  if (st != KVC_OK) return st;
  const int max_ctas = d.sms * d.streamk_ctas_per_sm;
  const kvc::WorkspaceLayout WL = kvc::workspace_layout(max_ctas, num_outputs);
  if (workspace_bytes < WL.total) return KVC_ERR_INVALID_ARG;

  kvc::Params p = {};
  for (int l = 0; l < L; ++l) {
    p.states[l] = static_cast<const uint8_t*>(state_caches[l]);
    p.weights[l] = rms_norm_weights[l];
    p.kvs[l] = kv_caches[l];
  }
  p.num_layers = L;
  p.num_blocks = num_state_blocks;
  p.state_block_bytes = lay.block_stride * esize;
  p.state_row_bytes = lay.row_stride * esize;
  p.state_f32 = lay.dtype == KVC_DTYPE_F32 ? 1 : 0;
  p.rows_contiguous = lay.row_stride == kvc::kRowElems ? 1 : 0;
  p.token_to_req = token_to_req;
  p.positions = positions;
  p.num_tokens = num_tokens;
  p.bti = boundary_token_indices;
  p.num_outputs = num_outputs;
  p.block_table = block_table;
  p.num_reqs = num_reqs;
  p.max_blocks = max_blocks_per_req;
  p.bt_row_stride = lay.bt_row_stride;
  p.bt_col_stride = lay.bt_col_stride;
  p.cos_sin = cos_sin_cache;
  p.num_positions = num_positions;
  p.slot_map = kv_slot_mapping;
  p.slot_by_token = (slot_mapping_len == num_tokens) ? 1 : 0;
  p.num_pages = num_kv_pages;
  p.y_out = y_out;
  p.compress_ratio = compress_ratio;
  p.block_size = block_size;
  p.blocks_per_output = (compress_ratio + kvc::kBlockRows - 1) / kvc::kBlockRows;
  p.num_units = num_outputs * p.blocks_per_output;
  p.eps = rms_norm_eps;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  p.partials = reinterpret_cast<float*>(ws + WL.partials);
  p.part_status = reinterpret_cast<int32_t*>(ws + WL.status);
  p.counters = reinterpret_cast<int32_t*>(ws + WL.counters);
  p.error = d.error_word;
  p.wait_limit = g_wait_limit.load(std::memory_order_relaxed);
  p.rejections = d.rejections;
  p.poison_guesses = g_poison_guesses.load(std::memory_order_relaxed);

  const bool streamk_ok = lay.dtype == KVC_DTYPE_BF16 && p.rows_contiguous &&
                          block_size == kvc::kBlockRows && compress_ratio % kvc::kBlockRows == 0;
  const double chunk = chunk_bytes_of(lay.dtype);
  Route r;
  if (!pick_route(d, num_outputs * L, p.blocks_per_output, streamk_ok, chunk, flags, &r))
    return KVC_ERR_UNSUPPORTED;
  p.cluster_size = r.cluster;
  if (!r.stream_k && !p.rows_contiguous && L <= kvc::kMaxMapLayers &&
      (flags & KVC_FLAG_ROW_COPIES) == 0) {
    bool ok = true;
    for (int l = 0; l < L && ok; ++l)
      ok = kvc::encode_rows_map(&p.maps[l], state_caches[l], p.state_f32 != 0, block_size,
                           num_state_blocks, p.state_row_bytes, p.state_block_bytes);
    p.use_maps = ok ? 1 : 0;
  }
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (pre_launch != nullptr && pre_launch->fn(pre_launch->ctx, s) != cudaSuccess) return KVC_ERR_CUDA;
  if (!r.stream_k) return kvc::launch_cluster(p, r.count, s) == cudaSuccess ? KVC_OK : KVC_ERR_CUDA;
  // stream-K: one launch per layer (each reuses the workspace, in stream order)
  const int ctas =
      pick_route(d, num_outputs, p.blocks_per_output, streamk_ok, chunk, flags, &r) ? r.count : 1;
  for (int l = 0; l < L; ++l) {
    kvc::Params pl = p;
    pl.states[0] = p.states[l];
    pl.weights[0] = p.weights[l];
    pl.kvs[0] = p.kvs[l];
    pl.num_layers = 1;
    pl.y_out = y_out ? y_out + static_cast<int64_t>(l) * num_outputs * kvc::kHeadDim : nullptr;
    if (kvc::launch_streamk(pl, ctas, s) != cudaSuccess) return KVC_ERR_CUDA;
  }
  return KVC_OK;
}

}  // namespace

namespace kvc {

kvc_status compress_hooked(const void* state_cache, int64_t num_state_blocks,
                           const int32_t* token_to_req, const int64_t* positions,
                           int64_t num_tokens, const int64_t* boundary_token_indices,
                           int64_t num_outputs, const int32_t* block_table, int64_t num_reqs,
                           int64_t max_blocks_per_req, const float* rms_norm_weight,
                           const float* cos_sin_cache, int64_t num_positions,
                           const int64_t* kv_slot_mapping, int64_t slot_mapping_len,
                           uint8_t* kv_cache, int64_t num_kv_pages, int32_t block_size,
                           int32_t compress_ratio, float rms_norm_eps, float* y_out,
                           void* workspace, size_t workspace_bytes, uint32_t flags, void* stream,
                           const PreLaunch* pre_launch) {
  return compress_layers(1, &state_cache, contiguous_layout(block_size, max_blocks_per_req),
                         num_state_blocks, token_to_req, positions, num_tokens,
                         boundary_token_indices, num_outputs, block_table, num_reqs,
                         max_blocks_per_req, &rms_norm_weight, cos_sin_cache, num_positions,
                         kv_slot_mapping, slot_mapping_len, &kv_cache, num_kv_pages, block_size,
                         compress_ratio, rms_norm_eps, y_out, workspace, workspace_bytes, flags,
                         stream, pre_launch);
}

}  // namespace kvc

extern "C" {

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
  return compress_layers(1, &state_cache, contiguous_layout(block_size, max_blocks_per_req),
                         num_state_blocks, token_to_req, positions, num_tokens,
                         boundary_token_indices, num_outputs, block_table, num_reqs,
                         max_blocks_per_req, &rms_norm_weight, cos_sin_cache, num_positions,
                         kv_slot_mapping, slot_mapping_len, &kv_cache, num_kv_pages, block_size,
                         compress_ratio, rms_norm_eps, y_out, workspace, workspace_bytes, flags,
                         stream);
}

kvc_status kvc_compress_layers(int32_t num_layers, const void* const* state_caches,
                               int64_t num_state_blocks, const int32_t* token_to_req,
                               const int64_t* positions, int64_t num_tokens,
                               const int64_t* boundary_token_indices, int64_t num_outputs,
                               const int32_t* block_table, int64_t num_reqs,
                               int64_t max_blocks_per_req, const float* const* rms_norm_weights,
                               const float* cos_sin_cache, int64_t num_positions,
                               const int64_t* kv_slot_mapping, int64_t slot_mapping_len,
                               uint8_t* const* kv_caches, int64_t num_kv_pages, int32_t block_size,
                               int32_t compress_ratio, float rms_norm_eps, float* y_out,
                               void* workspace, size_t workspace_bytes, uint32_t flags,
                               void* stream) {
  return compress_layers(num_layers, state_caches,
                         contiguous_layout(block_size, max_blocks_per_req), num_state_blocks,
                         token_to_req, positions,
                         num_tokens, boundary_token_indices, num_outputs, block_table, num_reqs,
                         max_blocks_per_req, rms_norm_weights, cos_sin_cache, num_positions,
                         kv_slot_mapping, slot_mapping_len, kv_caches, num_kv_pages, block_size,
                         compress_ratio, rms_norm_eps, y_out, workspace, workspace_bytes, flags,
                         stream);
}

kvc_status kvc_compress_strided(
    const void* state_cache, int32_t state_dtype, int64_t num_state_blocks,
    int64_t state_block_stride, int64_t state_row_stride, const int32_t* token_to_req,
    const int64_t* positions, int64_t num_tokens, const int64_t* boundary_token_indices,
    int64_t num_outputs, const int32_t* block_table, int64_t num_reqs, int64_t max_blocks_per_req,
    int64_t block_table_row_stride, int64_t block_table_col_stride, const float* rms_norm_weight,
    const float* cos_sin_cache, int64_t num_positions, const int64_t* kv_slot_mapping,
    int64_t slot_mapping_len, uint8_t* kv_cache, int64_t num_kv_pages, int32_t block_size,
    int32_t compress_ratio, float rms_norm_eps, float* y_out, void* workspace,
    size_t workspace_bytes, uint32_t flags, void* stream) {
  const StateLayout lay{state_dtype, state_block_stride, state_row_stride, block_table_row_stride,
                        block_table_col_stride};
  return compress_layers(1, &state_cache, lay, num_state_blocks, token_to_req, positions,
                         num_tokens, boundary_token_indices, num_outputs, block_table, num_reqs,
                         max_blocks_per_req, &rms_norm_weight, cos_sin_cache, num_positions,
                         kv_slot_mapping, slot_mapping_len, &kv_cache, num_kv_pages, block_size,
                         compress_ratio, rms_norm_eps, y_out, workspace, workspace_bytes, flags,
                         stream);
}

kvc_status kvc_compress_layers_strided(
    int32_t num_layers, const void* const* state_caches, int32_t state_dtype,
    int64_t num_state_blocks, int64_t state_block_stride, int64_t state_row_stride,
    const int32_t* token_to_req, const int64_t* positions, int64_t num_tokens,
    const int64_t* boundary_token_indices, int64_t num_outputs, const int32_t* block_table,
    int64_t num_reqs, int64_t max_blocks_per_req, int64_t block_table_row_stride,
    int64_t block_table_col_stride, const float* const* rms_norm_weights,
    const float* cos_sin_cache, int64_t num_positions, const int64_t* kv_slot_mapping,
    int64_t slot_mapping_len, uint8_t* const* kv_caches, int64_t num_kv_pages, int32_t block_size,
    int32_t compress_ratio, float rms_norm_eps, float* y_out, void* workspace,
    size_t workspace_bytes, uint32_t flags, void* stream) {
  const StateLayout lay{state_dtype, state_block_stride, state_row_stride, block_table_row_stride,
                        block_table_col_stride};
  return compress_layers(num_layers, state_caches, lay, num_state_blocks, token_to_req, positions,
                         num_tokens, boundary_token_indices, num_outputs, block_table, num_reqs,
                         max_blocks_per_req, rms_norm_weights, cos_sin_cache, num_positions,
                         kv_slot_mapping, slot_mapping_len, kv_caches, num_kv_pages, block_size,
                         compress_ratio, rms_norm_eps, y_out, workspace, workspace_bytes, flags,
                         stream);
}

kvc_status kvc_dequantize(const uint8_t* kv_cache, int64_t num_kv_pages, const int64_t* slots,
                          int64_t num_slots, void* out, int32_t out_dtype, void* stream) {
  if (num_slots < 0 || (out_dtype != KVC_DTYPE_F32 && out_dtype != KVC_DTYPE_BF16))
    return KVC_ERR_INVALID_ARG;
  if (num_slots == 0) return KVC_OK;
  if (!kv_cache || !slots || !out || num_kv_pages <= 0) return KVC_ERR_INVALID_ARG;
  if (!aligned(kv_cache, 16) || !aligned(slots, 8) ||
      !aligned(out, out_dtype == KVC_DTYPE_F32 ? 16 : 8))
    return KVC_ERR_INVALID_ARG;
  DeviceInfo d;
  const kvc_status st = device_info(&d);
  if (st != KVC_OK) return st;
  const cudaError_t e = kvc::launch_dequantize(kv_cache, num_kv_pages, slots, num_slots, out,
                                               out_dtype == KVC_DTYPE_BF16, d.error_word,
                                               static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KVC_OK : KVC_ERR_CUDA;
}

kvc_status kvc_selftest_wait_timeout(uint64_t limit_cycles, void* stream) {
  if (limit_cycles < 1 || limit_cycles > 4000000000ull) return KVC_ERR_INVALID_ARG;
  DeviceInfo d;
  const kvc_status st = device_info(&d);
  if (st != KVC_OK) return st;
  const cudaError_t e = kvc::launch_selftest_wait(static_cast<long long>(limit_cycles),
                                                  d.error_word, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KVC_OK : KVC_ERR_CUDA;
}

kvc_status kvc_selftest_set_wait_limit(uint64_t limit_cycles) {
  if (limit_cycles > static_cast<uint64_t>(kvc::kDefaultWaitLimitCycles)) return KVC_ERR_INVALID_ARG;
  g_wait_limit.store(limit_cycles == 0 ? kvc::kDefaultWaitLimitCycles
                                       : static_cast<long long>(limit_cycles),
                     std::memory_order_relaxed);
  return KVC_OK;
}

kvc_status kvc_selftest_poison_guesses(int32_t on) {
  if (on != 0 && on != 1) return KVC_ERR_INVALID_ARG;
  g_poison_guesses.store(on, std::memory_order_relaxed);
  return KVC_OK;
}

kvc_status kvc_selftest_first_pass_rejections(void* stream, uint64_t* out_count) {
  if (out_count == nullptr) return KVC_ERR_INVALID_ARG;
  DeviceInfo d;
  const kvc_status st = device_info(&d);
  if (st != KVC_OK) return st;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return KVC_ERR_CUDA;
  unsigned long long n = 0;
  if (cudaMemcpy(&n, d.rejections, sizeof n, cudaMemcpyDeviceToHost) != cudaSuccess)
    return KVC_ERR_CUDA;
  if (n != 0 && cudaMemset(d.rejections, 0, sizeof n) != cudaSuccess) return KVC_ERR_CUDA;
  *out_count = n;
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
  return "kvc 0.3.0 sm_103a: cluster route (S=1..16, bf16/fp32 strided state, bulk-copy ring "
         "96KiB, st.async merges) + stream-K route";
}

}  // extern "C"
