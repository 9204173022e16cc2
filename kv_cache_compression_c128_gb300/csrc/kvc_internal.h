// Internal interface between the C ABI layer (kvc_api.cu) and the two
// kernel routes (kvc_cluster.cu, kvc_streamk.cu).  Not part of the ABI.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda.h>  // CUtensorMap (a plain struct; no driver call is linked)
#include <cuda_runtime.h>

#include "../../include/kvc.h"  // kvc_status

namespace kvc {

// Constants of the section "Gather and Scatter" of the KernelGen Challenge 8
// write-up, plus the paged state geometry (block_size 8, 512 values + 512
// scores per row).
constexpr int kHeadDim = 512;
constexpr int kNopeDim = 448;
constexpr int kRopeDim = 64;
constexpr int kGroup = 64;
constexpr int kRowElems = 2 * kHeadDim;                    // elements per state row
constexpr int kBlockRows = 8;                              // rows per chunk (block_size 8)
constexpr int kBlockBytes = kBlockRows * kRowElems * 2;    // 16 KiB per bf16 chunk
constexpr int kSlotsPerPage = 64;
constexpr int kTokenStride = 576;
constexpr int kScaleDim = 8;
constexpr int64_t kPageBytes = kSlotsPerPage * (kTokenStride + kScaleDim);
constexpr int kScaleBase = kSlotsPerPage * kTokenStride;   // 36864

// CTA shape: 8 consumer warps (thread t owns dims 2t, 2t+1) + 1 producer
// warp (stream-K route; the cluster route adds a resolver warp).
constexpr int kConsumerWarps = 8;
constexpr int kConsumerThreads = kConsumerWarps * 32;
constexpr int kThreads = kConsumerThreads + 32;
constexpr int kMaxClusterSize = 16;
constexpr int kMaxFinalizers = 8;
constexpr int kStages = 6;                                 // 16 KiB ring stages (bf16)
constexpr int kRingBytes = kStages * kBlockBytes;          // 96 KiB: 6 bf16 or 3 fp32 chunks
constexpr int kMetaRing = kStages + 2;                     // per-output records

// A split output's partial softmax state: m[512], den[512], num[512].
constexpr int kPartialFloats = 3 * kHeadDim;

// Layers one multi-layer call may compress (per-layer pointers travel in the
// kernel parameters).
constexpr int kMaxLayers = 64;

// Layers that get a TMA tensor map when the rows of a block are apart (one
// tensor copy per full 8-row run instead of one bulk copy per row).  The maps
// travel in the kernel parameters, 128 bytes each.
constexpr int kMaxMapLayers = 8;

// The 4-D view of a state that the maps describe, innermost first: 256
// elements, 4 segments of a row (kRowElems = 4 x 256), rows of a block,
// blocks; the box is 256 x 4 x 8 x 1, i.e. 8 whole rows.
constexpr int kMapInner = 256;
constexpr int kMapSegments = kRowElems / kMapInner;

struct Params {
  const uint8_t* states[kMaxLayers];   // per layer: state base (bf16 or fp32 elements)
  const float* weights[kMaxLayers];    // per layer: rms_norm_weight [512]
  uint8_t* kvs[kMaxLayers];            // per layer: kv_cache [num_pages, 37376]
  int num_layers;                      // L; outputs of the call = L * num_outputs
  int64_t num_blocks;
  int64_t state_block_bytes;           // bytes between physical blocks
  int64_t state_row_bytes;             // bytes between rows of a block
  int state_f32;                       // 1: fp32 elements, 0: bf16
  int rows_contiguous;                 // state_row_bytes == one row's bytes
  const int32_t* token_to_req;
  const int64_t* positions;
  int64_t num_tokens;
  const int64_t* bti;             // boundary_token_indices
  int64_t num_outputs;
  const int32_t* block_table;
  int64_t num_reqs;
  int64_t max_blocks;
  int64_t bt_row_stride;          // block_table[r, l] at r * bt_row_stride + l * bt_col_stride
  int64_t bt_col_stride;
  const float* cos_sin;
  int64_t num_positions;
  const int64_t* slot_map;
  int slot_by_token;              // 1: slot_map[b], 0: slot_map[n]
  int64_t num_pages;
  float* y_out;                   // optional: [L * num_outputs, 512], layer-major
  int compress_ratio;             // C
  int block_size;                 // B: rows per physical state block
  int blocks_per_output;          // K = ceil(C / 8): 8-row chunks per window
  int64_t num_units;              // U = N * K: one unit = one 8-row chunk
  float eps;
  int cluster_size;               // cluster route: CTAs per output (S)
  float* partials;                // [2 * max_ctas][kPartialFloats]
  int32_t* part_status;           // [2 * max_ctas]
  int32_t* counters;              // [num_outputs]
  uint32_t* error;                // device error word (first error code wins)
  long long wait_limit;           // SM cycles a pipeline wait may take before the kernel
                                  // records KVC_ERR_TIMEOUT and abandons the call
  unsigned long long* rejections; // device counter of guessed first passes that failed their check
  int poison_guesses;             // test hook: guesses name the next physical block
  int use_maps;                   // rows apart and every layer has a map (cluster route)
  CUtensorMap maps[kMaxMapLayers];  // per layer, when use_maps
};

// Workspace layout (byte offsets), given the device's CTA capacity.
struct WorkspaceLayout {
  size_t partials, status, counters, total;
};
WorkspaceLayout workspace_layout(int max_ctas, int64_t num_outputs);

// stream-K route (kvc_streamk.cu)
size_t streamk_smem_bytes();
const void* streamk_kernel_symbol();
cudaError_t launch_streamk(const Params& p, int ctas, cudaStream_t stream);

// cluster route (kvc_cluster.cu); cluster sizes 1, 2, 4, 8, 16; both state
// dtypes use the same shared-memory footprint, so one capacity serves both
int cluster_threads();
size_t cluster_smem_bytes(int cluster_size);
int cluster_capacity(int cluster_size);  // sets the kernel up; co-resident clusters (0: refused)
cudaError_t launch_cluster(const Params& p, int clusters, cudaStream_t stream);
// The TMA tensor map of one layer's state with rows apart (host; false when
// it cannot be encoded, and the call then copies row by row).
bool encode_rows_map(CUtensorMap* map, const void* base, bool f32, int64_t block_size,
                     int64_t num_blocks, int64_t row_bytes, int64_t block_bytes);

// reader direction (kvc_reader.cu)
cudaError_t launch_dequantize(const uint8_t* kv, int64_t num_pages, const int64_t* slots,
                              int64_t num_slots, void* out, int out_bf16, uint32_t* err,
                              cudaStream_t stream);

// failure-path self-test (kvc_selftest.cu): one bounded wait that runs out
cudaError_t launch_selftest_wait(long long limit_cycles, uint32_t* err, cudaStream_t stream);

// The kernels' default limit on one wait, in SM clock cycles (~2 s at 2 GHz).
constexpr long long kDefaultWaitLimitCycles = 4000000000LL;

// Identity of the CUDA context current on the calling thread (0: none).
// Per-device set-up (function attributes, symbol addresses) belongs to one
// context and is made again when another one is current.
unsigned long long context_id();

// A host step the ABI layer runs on the call's stream after every argument
// check has passed, right before the launch (kvc_static.cu clears its
// counters this way, so a refused call writes nothing).
struct PreLaunch {
  cudaError_t (*fn)(void* ctx, cudaStream_t stream);
  void* ctx;
};

// kvc_compress (include/kvc.h) with a PreLaunch step (null: none).
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
                           const PreLaunch* pre_launch);

}  // namespace kvc
