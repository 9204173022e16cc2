/*
 * kvc.h -- C ABI of the GB300 KV-cache window compressor.
 *
 * The operator is c128_256_512_compress from "From Attention to KV Cache
 * Compression: Notes from a KernelGen Optimization" (KernelGen Challenge 8
 * write-up): section "The Compression Operator" gives the argument list,
 * "Gather and Scatter" the constants and the packed slot layout, and "How
 * One Output Is Produced" the computation:
 *
 *   for every boundary token b = boundary_token_indices[n]:
 *     r = token_to_req[b], p = positions[b], window t = p-C+1 .. p;
 *     row(t) = block_table[r, t/B] * B + t%B of state_cache (block_size B);
 *     c_d = sum_t softmax_t(score[row(t), d]) * value[row(t), d], d < 512
 *           (softmax along the window, separately per dimension);
 *     y = c * (mean(c^2) + eps)^-1/2 * rms_norm_weight;
 *     dims 0..447: z = bf16(y); per 64-dim group a = max(max|z|, 1e-4),
 *       e = ceil(log2(a/127)), q = trunc(z * 2^-e) clipped to +-127 (int8),
 *       scale byte = e + 127;
 *     dims 448..511: GPT-J interleaved RoPE with the cos/sin row
 *       pc = floor(p/C)*C, stored as bf16;
 *     slot = kv_slot_mapping[b]: 576 payload bytes at
 *       kv_cache[slot/64, (slot%64)*576] and 8 scale bytes (7 exponents + a
 *       zero padding byte) at kv_cache[slot/64, 64*576 + (slot%64)*8].
 *
 * All pointers name device memory of the current CUDA device unless stated
 * otherwise; the caller owns every buffer.  Calls are asynchronous on the
 * given stream and never synchronise it (kvc_get_device_error excepted).
 * A call may start while the kernel before it on the stream still runs
 * (programmatic dependent launch).  It may then read its index arrays,
 * warm L2 with its first rows and even copy rows those indices name, but
 * every value that reaches a result is read, or checked against a read,
 * after that kernel has finished: a call may read what the kernel before
 * it writes.
 * The library's own per-device set-up (kernel attributes, the addresses of
 * its device-side words) is made at the first call in a CUDA context and made
 * again when another context is current on that device, e.g. after
 * cudaDeviceReset.
 *
 * Two choices of this interface that a reader of the statement's signature
 * might not expect:
 *   - Index checking is always on: every index is range-checked on its way
 *     to an address, and a bad one is reported through kvc_get_device_error.
 *     There is no "checked mode" flag.  The low 16 bits of `flags` force the
 *     launch size instead (see below): flags = 1 runs the whole call on ONE
 *     cluster, which computes the same bytes but many times slower.  Pass 0.
 *   - kvc_compress does not allocate.  Scratch for outputs whose window is
 *     split between CTAs is a caller-owned, zero-filled workspace
 *     (kvc_workspace_bytes); the Python binding keeps one per device and
 *     stream.  kvc_compress_static uses a buffer inside the library instead.
 */
#ifndef KVC_H_
#define KVC_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  KVC_OK = 0,
  KVC_ERR_INVALID_ARG = 1,  /* null pointer, bad size, misalignment, small workspace */
  KVC_ERR_UNSUPPORTED = 2,  /* block_size < 8; a cluster size the problem or device
                               cannot take; a state stride that is not a multiple of
                               16 bytes; the stream-K route asked for with block_size
                               != 8, C not a multiple of 8, an fp32 state or rows of
                               a block that are not adjacent, or (device, stream-K
                               route) a window not starting on an 8-row block */
  KVC_ERR_CUDA = 3,         /* a CUDA runtime call failed */
  KVC_ERR_BAD_INDEX = 4,    /* (device) an index outside its array */
  KVC_ERR_TIMEOUT = 5,      /* (device) a pipeline wait ran past its limit */
  KVC_ERR_SCRATCH_LIMIT = 6 /* kvc_compress_static: the problem needs more scratch
                               than the library's built-in buffer holds */
} kvc_status;

/*
 * flags (0 = automatic choice of everything; use 0 outside tuning and tests):
 *   bits 0..15   force the launch size: clusters for the cluster route, CTAs
 *                for the stream-K route (capped at what fits on the device);
 *                NOT a "checked mode" switch -- checking is always on, and
 *                flags = 1 forces a single cluster;
 *   bits 16..20  force the cluster size S (1, 2, 4, 8 or 16, at most C/8);
 *   bit 24       use the stream-K route instead of the cluster route;
 *   bit 25       rows apart (kvc_compress_strided): copy one row at a time
 *                even where a TMA tensor map could move 8 rows at once.
 * The routes and copy modes compute the same bytes (see kvc_query_launch);
 * the flags exist for tuning and testing.  Other bits must be zero.
 */
#define KVC_FLAG_GRID_MASK 0xFFFFu
#define KVC_FLAG_CLUSTER_SHIFT 16
#define KVC_FLAG_CLUSTER_MASK (0x1Fu << KVC_FLAG_CLUSTER_SHIFT)
#define KVC_FLAG_STREAM_K (1u << 24)
#define KVC_FLAG_ROW_COPIES (1u << 25)
#define KVC_FLAG_ALL \
  (KVC_FLAG_GRID_MASK | KVC_FLAG_CLUSTER_MASK | KVC_FLAG_STREAM_K | KVC_FLAG_ROW_COPIES)

/* Element types: of the state (kvc_compress_strided, kvc_query_launch_ex)
 * and of the output of kvc_dequantize. */
#define KVC_DTYPE_F32 0
#define KVC_DTYPE_BF16 1

/*
 * Bytes of device workspace kvc_compress needs for num_outputs outputs on
 * the current device.  The workspace holds the partial softmax states of
 * outputs whose window is split between two or more CTAs and one arrival
 * counter per output.  Returns 0 on error (no CUDA device).
 */
size_t kvc_workspace_bytes(int64_t num_outputs);

/*
 * Compress every boundary token's window into its kv_cache slot.
 *
 * state_cache      bf16 [num_state_blocks, block_size, 1024], contiguous,
 *                  16-byte aligned; row columns 0..511 are values, 512..1023
 *                  scores.
 * token_to_req     int32 [num_tokens]: request of each token.
 * positions        int64 [num_tokens]: position of each token in its request.
 * boundary_token_indices  int64 [num_outputs]: token index b of each output.
 * block_table      int32 [num_reqs, max_blocks_per_req] (row stride
 *                  max_blocks_per_req): physical block of each logical block.
 * rms_norm_weight  fp32 [512].
 * cos_sin_cache    fp32 [num_positions, 64]: cos in columns 0..31, sin 32..63.
 * kv_slot_mapping  int64: indexed by token (slot_mapping_len == num_tokens)
 *                  or by output (slot_mapping_len == num_outputs).  A
 *                  negative slot skips that output.
 * kv_cache         uint8 [num_kv_pages, 37376], 16-byte aligned; written in
 *                  place, only at the 576 + 8 bytes of each written slot.
 * block_size       B >= 8 rows per physical block (the write-up's is 8).
 * compress_ratio   C >= 1 (the write-up's are 128, 256, 512).  Windows may
 *                  start at any position p - C + 1 >= 0 (the benchmark's start
 *                  on a block boundary).
 * rms_norm_eps     finite, >= 0 (the write-up's default is 1e-6).
 * y_out            optional fp32 [num_outputs, 512], 8-byte aligned, or NULL:
 *                  receives the RMS-normalised vector y of each output (before
 *                  the bf16 rounding, quantisation and RoPE).
 * workspace        device buffer of at least kvc_workspace_bytes(num_outputs)
 *                  bytes, 16-byte aligned, ZERO-FILLED before its first use.
 *                  Every completed call leaves its counters at zero again, so
 *                  one workspace serves any number of calls in stream order.
 *                  Calls that may run concurrently need separate workspaces.
 * stream           cudaStream_t (NULL = legacy default stream).
 *
 * Host-detected errors return before anything is launched.  Device-detected
 * errors (an index outside its array, a window that starts before position
 * 0 or off an 8-row block boundary) never trap: the offending output's slot
 * is left untouched, the other outputs are written, and a sticky device
 * error code is recorded for kvc_get_device_error.  Every wait of the
 * kernels is bounded: a wait that runs past its limit records
 * KVC_ERR_TIMEOUT, the kernel stops issuing copies, waits for the ones in
 * flight and returns.  When a pipeline wait (a copy stage, a hand-off
 * between warps) ran out, every slot is either written whole, with the bytes
 * an undisturbed call writes, or left untouched; when an exchange between
 * the CTAs of a cluster ran out (a peer that stopped answering), the slots
 * of the outputs that exchange served are unspecified.
 */
kvc_status kvc_compress(
    const void* state_cache, int64_t num_state_blocks,
    const int32_t* token_to_req, const int64_t* positions, int64_t num_tokens,
    const int64_t* boundary_token_indices, int64_t num_outputs,
    const int32_t* block_table, int64_t num_reqs, int64_t max_blocks_per_req,
    const float* rms_norm_weight,
    const float* cos_sin_cache, int64_t num_positions,
    const int64_t* kv_slot_mapping, int64_t slot_mapping_len,
    uint8_t* kv_cache, int64_t num_kv_pages,
    int32_t block_size, int32_t compress_ratio, float rms_norm_eps,
    float* y_out, void* workspace, size_t workspace_bytes,
    uint32_t flags, void* stream);

/*
 * kvc_compress for num_layers layers (1..64) that share every index array:
 * the same boundary tokens, windows, block table, slots, cos/sin table and
 * eps, each layer with its own state cache, RMSNorm weight and kv_cache
 * (per-layer caches of a model: the write-up's motivation is long-context
 * decoding, where every layer compresses the same windows).  One launch
 * serves all layers: the index chain is resolved per window and the work of
 * all layers is split evenly over the GPU.
 *
 * state_caches, rms_norm_weights, kv_caches: HOST arrays of num_layers
 * DEVICE pointers, each with the shape, alignment and meaning of the single
 * buffer of kvc_compress.  y_out (optional): fp32 [num_layers * num_outputs,
 * 512], layer-major.  workspace: kvc_workspace_bytes(num_outputs) bytes
 * (the stream-K route processes one layer at a time).  Everything else as for
 * kvc_compress, whose results each layer reproduces.
 */
kvc_status kvc_compress_layers(
    int32_t num_layers, const void* const* state_caches, int64_t num_state_blocks,
    const int32_t* token_to_req, const int64_t* positions, int64_t num_tokens,
    const int64_t* boundary_token_indices, int64_t num_outputs,
    const int32_t* block_table, int64_t num_reqs, int64_t max_blocks_per_req,
    const float* const* rms_norm_weights,
    const float* cos_sin_cache, int64_t num_positions,
    const int64_t* kv_slot_mapping, int64_t slot_mapping_len,
    uint8_t* const* kv_caches, int64_t num_kv_pages,
    int32_t block_size, int32_t compress_ratio, float rms_norm_eps,
    float* y_out, void* workspace, size_t workspace_bytes,
    uint32_t flags, void* stream);

/*
 * kvc_compress over a state of either element type, laid out with explicit
 * strides, and a strided block table.  "The Baseline" of the write-up counts
 * the window's source traffic with an fp32 state element, and "A Bit of
 * Triton and GPU Background" reads the state through block / row / column
 * strides; this entry point takes both.  (kvc_compress is this call with a
 * contiguous bf16 state and a row-major block table.)
 *
 * state_cache         bf16 (state_dtype KVC_DTYPE_BF16) or fp32
 *                     (KVC_DTYPE_F32) elements, 16-byte aligned.  Element
 *                     (g, o, col) of physical block g < num_state_blocks,
 *                     row o < block_size, column col < 1024 is at element
 *                     offset g * state_block_stride + o * state_row_stride +
 *                     col (columns are contiguous); the caller guarantees
 *                     that every such element lies in the buffer.
 * state_block_stride, state_row_stride
 *                     >= 0, in elements; each a multiple of 16 bytes
 *                     (KVC_ERR_UNSUPPORTED otherwise: the rows are moved by
 *                     bulk copies).  Rows that are adjacent (row stride 1024)
 *                     are copied a run at a time.  Rows apart are copied 8 at
 *                     a time through a TMA tensor map per layer (calls of up
 *                     to 8 layers; the library encodes the maps on the host at
 *                     each call), one at a time where a chunk's 8 rows span
 *                     two blocks, with more layers, or with
 *                     KVC_FLAG_ROW_COPIES.
 * block_table         int32; entry (r, l) of request r < num_reqs, logical
 *                     block l < max_blocks_per_req at element offset
 *                     r * block_table_row_stride + l * block_table_col_stride
 *                     (both >= 0; e.g. 1 and num_reqs for a column-major
 *                     table), 4-byte aligned.
 * Everything else (arguments, results, errors, flags) as for kvc_compress.
 * The results meet kvc_compress's bar on the same values: the window sum
 * runs in fp32 over the elements as stored (bf16 widened exactly); only the
 * order of the fp32 sums differs between element types.  The stream-K route
 * takes only a bf16 state with adjacent rows.
 */
kvc_status kvc_compress_strided(
    const void* state_cache, int32_t state_dtype, int64_t num_state_blocks,
    int64_t state_block_stride, int64_t state_row_stride,
    const int32_t* token_to_req, const int64_t* positions, int64_t num_tokens,
    const int64_t* boundary_token_indices, int64_t num_outputs,
    const int32_t* block_table, int64_t num_reqs, int64_t max_blocks_per_req,
    int64_t block_table_row_stride, int64_t block_table_col_stride,
    const float* rms_norm_weight,
    const float* cos_sin_cache, int64_t num_positions,
    const int64_t* kv_slot_mapping, int64_t slot_mapping_len,
    uint8_t* kv_cache, int64_t num_kv_pages,
    int32_t block_size, int32_t compress_ratio, float rms_norm_eps,
    float* y_out, void* workspace, size_t workspace_bytes,
    uint32_t flags, void* stream);

/*
 * kvc_compress_layers over states of either element type at explicit
 * strides, with a strided block table: the layout arguments of
 * kvc_compress_strided (one layout shared by every layer), the per-layer
 * pointer arrays of kvc_compress_layers.  Everything else, results and
 * errors as for those two calls.
 */
kvc_status kvc_compress_layers_strided(
    int32_t num_layers, const void* const* state_caches, int32_t state_dtype,
    int64_t num_state_blocks, int64_t state_block_stride, int64_t state_row_stride,
    const int32_t* token_to_req, const int64_t* positions, int64_t num_tokens,
    const int64_t* boundary_token_indices, int64_t num_outputs,
    const int32_t* block_table, int64_t num_reqs, int64_t max_blocks_per_req,
    int64_t block_table_row_stride, int64_t block_table_col_stride,
    const float* const* rms_norm_weights,
    const float* cos_sin_cache, int64_t num_positions,
    const int64_t* kv_slot_mapping, int64_t slot_mapping_len,
    uint8_t* const* kv_caches, int64_t num_kv_pages,
    int32_t block_size, int32_t compress_ratio, float rms_norm_eps,
    float* y_out, void* workspace, size_t workspace_bytes,
    uint32_t flags, void* stream);

/*
 * Read packed slots back as 512-vectors (the reader side of the cache: the
 * attention that consumes the compressed keys).  Layout of "Gather and
 * Scatter" in the write-up; values of its quantisation equation ("How One
 * Output Is Produced"):
 *   out[m, d] = q_d * 2^(scale[d / 64] - 127)   d < 448, q_d the int8 code,
 *   out[m, d] = the stored bf16 RoPE value       d >= 448,
 * computed exactly (a power-of-two scaling) and written as fp32
 * (out_dtype KVC_DTYPE_F32, out 16-byte aligned, float [num_slots, 512]) or
 * bf16 (KVC_DTYPE_BF16, out 8-byte aligned, [num_slots, 512]; every such
 * value is exactly representable in bf16 unless it overflows).
 *
 * kv_cache  uint8 [num_kv_pages, 37376], 16-byte aligned, read only.
 * slots     int64 [num_slots]: slot m to read; a negative slot yields zeros;
 *           a slot beyond the last page yields zeros and records
 *           KVC_ERR_BAD_INDEX in the device error word.
 * Asynchronous on `stream`; allocates nothing.
 */
kvc_status kvc_dequantize(const uint8_t* kv_cache, int64_t num_kv_pages,
                          const int64_t* slots, int64_t num_slots, void* out,
                          int32_t out_dtype, void* stream);

/*
 * kvc_compress without a workspace argument, for callers that cannot
 * allocate device memory: plugins that are handed only their input and
 * output pointers, engines that reserve the whole device memory pool up front
 * and forbid allocation at run time, and latency-critical paths that cannot
 * afford cudaMalloc's implicit device synchronisation.  (The write-up has no
 * counterpart; this is a property of this library's interface.)
 *
 * Scratch comes from an 8 MiB buffer inside the library (a file-scope
 * __device__ array, held by every device that loads the library until the
 * process exits).  Nothing is allocated: no cudaMalloc, no cudaFree, no
 * allocating library routine.  The first call on a device (and the first
 * after the device's context changed, e.g. after cudaDeviceReset) looks up
 * the buffer's device address (cudaGetSymbolAddress) and sets up the kernel
 * for that device; make that first call before any stream capture on the
 * device.  Once every argument check has passed, each call clears the
 * buffer's arrival counters with cudaMemsetAsync on `stream`, then computes
 * exactly what kvc_compress computes; a call refused by a check writes
 * nothing.
 *
 * Every call on a device shares the one buffer, which keeps the last call's
 * contents: calls that overlap on the GPU (different streams, not ordered by
 * events) race on it.  Order them.
 *
 * Limit: on a 152-SM GPU the buffer serves up to about one million outputs
 * per call (kvc_workspace_bytes(num_outputs) must not exceed 8 MiB); larger
 * problems return KVC_ERR_SCRATCH_LIMIT before anything is launched.
 * Arguments, errors and flags are otherwise those of kvc_compress.
 */
kvc_status kvc_compress_static(
    const void* state_cache, int64_t num_state_blocks,
    const int32_t* token_to_req, const int64_t* positions, int64_t num_tokens,
    const int64_t* boundary_token_indices, int64_t num_outputs,
    const int32_t* block_table, int64_t num_reqs, int64_t max_blocks_per_req,
    const float* rms_norm_weight,
    const float* cos_sin_cache, int64_t num_positions,
    const int64_t* kv_slot_mapping, int64_t slot_mapping_len,
    uint8_t* kv_cache, int64_t num_kv_pages,
    int32_t block_size, int32_t compress_ratio, float rms_norm_eps,
    float* y_out, uint32_t flags, void* stream);

/*
 * Launch shape kvc_compress would use for this problem on the current
 * device: total CTAs, cluster size (0 for the stream-K route), threads per
 * CTA and dynamic shared memory bytes per CTA.  Any out pointer may be NULL.
 * flags as for kvc_compress; KVC_ERR_UNSUPPORTED if they ask for a cluster
 * size the problem or the device cannot take.
 */
kvc_status kvc_query_launch(int64_t num_outputs, int32_t compress_ratio,
                            uint32_t flags, int32_t* ctas, int32_t* cluster_size,
                            int32_t* threads, int32_t* smem_bytes);

/*
 * kvc_query_launch for a state of element type state_dtype (KVC_DTYPE_BF16
 * or KVC_DTYPE_F32): the launch kvc_compress_strided would use.
 * kvc_query_launch is this call with KVC_DTYPE_BF16.
 */
kvc_status kvc_query_launch_ex(int64_t num_outputs, int32_t compress_ratio,
                               int32_t state_dtype, uint32_t flags, int32_t* ctas,
                               int32_t* cluster_size, int32_t* threads,
                               int32_t* smem_bytes);

/*
 * Self-test of the failure path that every pipeline wait of the kernels
 * takes.  Launches one thread on `stream` that waits, through the same
 * bounded mbarrier wait the kernels use, on a barrier nothing will ever
 * complete, with a limit of limit_cycles SM clock cycles (1 .. 4e9; the
 * kernels' own limit is 4e9, about 2 s).  The wait runs out, the thread
 * records KVC_ERR_TIMEOUT in the device error word (read it with
 * kvc_get_device_error) and returns: nothing traps or hangs, and the
 * context stays usable.  KVC_ERR_INVALID_ARG for a limit outside the range.
 */
kvc_status kvc_selftest_wait_timeout(uint64_t limit_cycles, void* stream);

/*
 * Test hook for the kernels' abort path: sets the limit, in SM clock cycles,
 * on each pipeline wait (a copy stage, a hand-off between warps) of every
 * compression launched afterwards by this process, on any device.
 * limit_cycles 0 restores the default (4e9 cycles, about 2 s); 1 .. 4e9 sets
 * it; larger values return KVC_ERR_INVALID_ARG.  Limits below 100000 cycles
 * are polled without suspending the waiting thread, so they run out on time.
 * A short limit makes real calls give up part way: each records
 * KVC_ERR_TIMEOUT, stops issuing copies, drains the copies already in flight
 * (that drain, and the exchanges between the CTAs of a cluster, keep the
 * default limit, so no CTA exits while a copy or a peer may still write into
 * it) and returns, with every slot either written whole or untouched.  It
 * exists so that this path can be tested on real launches; production
 * callers never need it.  Not synchronised with calls in flight on other
 * host threads.
 */
kvc_status kvc_selftest_set_wait_limit(uint64_t limit_cycles);

/*
 * Test hook for the guessed first pass of a call on a state whose rows are
 * adjacent.  A CTA that is resident while the previous kernel on its stream
 * still runs reads the index arrays as they stand (they may still change),
 * issues its first copies from those guesses the moment the grid
 * dependency wait releases, and then checks every guess against the
 * indices read after the release.  A failed check throws the copied rows
 * away and copies the right ones; results never depend on which happened.
 * on = 1: every guess made by calls launched afterwards in this process, on
 * any device, names the next physical block instead of the right one, so
 * every guessed first pass fails its check (given at least 2 physical
 * blocks) and takes that recovery.  on = 0 restores normal guesses; other
 * values return KVC_ERR_INVALID_ARG.  Not synchronised with calls in flight
 * on other host threads.
 */
kvc_status kvc_selftest_poison_guesses(int32_t on);

/*
 * Synchronises `stream`, then reads and clears the number of guessed first
 * passes whose check failed, counted by the kernels of this library on the
 * current device since the last read.  Indices that no earlier kernel on
 * the stream changes always pass, so outside kvc_selftest_poison_guesses
 * the count stays 0 unless a call reads indices the kernel before it writes.
 */
kvc_status kvc_selftest_first_pass_rejections(void* stream, uint64_t* out_count);

/*
 * Synchronises `stream`, then reads and clears the device error code
 * recorded by kernels of this library on the current device (KVC_OK if
 * none).  The code is the first one recorded since the last clear.
 */
kvc_status kvc_get_device_error(void* stream, uint32_t* out_code);

/* Static description of a status code. */
const char* kvc_error_string(kvc_status status);

/* Library identification: version, target architecture and kernel route. */
const char* kvc_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KVC_H_ */
