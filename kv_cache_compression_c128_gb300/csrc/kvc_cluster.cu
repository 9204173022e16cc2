// Cluster route of the KV-cache window compressor (sm_103a).
//
// Computes c128_256_512_compress of "From Attention to KV Cache Compression:
// Notes from a KernelGen Optimization" (KernelGen Challenge 8 write-up): the
// per-dimension softmax-weighted window sum of "How One Output Is Produced",
// streamed as in "Online Softmax: Streaming Away the Window", then RMSNorm,
// NOPE quantisation, RoPE and the packed slot store.
//
// Work decomposition.  A window of C rows is cut into K = ceil(C/8) chunks of
// 8 rows (the last may be shorter); with the benchmark's block-aligned
// windows and block_size 8 a chunk is exactly one 16 KiB physical block, in
// general it is at most two runs of rows, each inside one physical block
// (block_size >= 8).  The state is bf16 or fp32 ("The Baseline" sizes its
// traffic with an fp32 element) and is addressed through block and row
// strides ("A Bit of Triton and GPU Background"); the kernel is templated on
// the element type, with a 16 KiB (bf16) or 32 KiB (fp32) chunk and the same
// 96 KiB ring of 32 KiB stages either way.  Output n is handled by one
// thread-block cluster of S CTAs (S = 1, 2, 4, 8, 16); rank j streams chunks
// [j K/S, (j+1) K/S).  Persistent clusters take contiguous, equal ranges of
// outputs, so every CTA streams the same number of chunks.  A multi-layer
// call simply has L * N outputs: output o is window o mod N of layer o / N
// (same chunks, that layer's state cache, weight and kv_cache), so all
// layers share one launch and one balanced split.
//
// Inside a CTA (320 threads):
//   warp 9  resolver: turns units into physical blocks (boundary index ->
//           request/position/slot -> block_table) 32 at a time, two chunks
//           ahead, into a shared-memory FIFO;
//   warp 8  issuer: one cp.async.bulk per run of rows into a ring of three
//           32 KiB stages (two bf16 chunks or one fp32 chunk each), each
//           stage guarded by a full/empty mbarrier pair.  When the rows of a
//           block are not adjacent: one TMA tensor copy per chunk through a
//           per-layer tensor map, or one bulk copy per row without one.
//           With adjacent rows the ring's first pass goes out from the
//           resolver, or, when the CTA is resident before the grid
//           dependency wait releases, from the whole issuer warp, on indices
//           read early and checked after the release;
//   warps 0-7 consumers: thread t owns dims 2t, 2t+1 and folds every staged
//           chunk into its (max, denominator, numerator), a stage of two
//           full bf16 chunks as 16 rows with one rescale.  Before the grid
//           dependency wait, warp 0 warms L2 with the CTA's first stages.
// With S = 1 the consumers then finalise the output directly.  With S > 1
// every rank pushes its partial state to the finaliser rank owning each dim
// (F = min(S, 8) finalisers, 512/F dims each) with st.async, which completes
// transaction bytes on that rank's mbarrier -- no fences, no remote polling.
// Each finaliser merges the S partials from its own shared memory, pushes its
// partial sum of squares to every rank the same way, and stores its slice of
// the slot.  The sum-of-squares exchange also tells senders that their
// previous partials were consumed, so a receive buffer is never overwritten
// early.  Every wait is bounded; invalid indices are recorded, not trapped.

#include <cuda_runtime.h>

#include "kvc_device.cuh"

namespace kvc {
namespace {

using namespace dev;

constexpr int kClusterWarps = kConsumerWarps + 2;  // + issuer + resolver
constexpr int kClusterThreads = kClusterWarps * 32;
constexpr int kIssuerWarp = kConsumerWarps;
constexpr int kResolverWarp = kConsumerWarps + 1;
constexpr int kFifoChunk = 32;

// Ring geometry of a state element type: a stage holds kChunksPerStage
// consecutive 8-row chunks of one output (two 16 KiB bf16 chunks or one
// 32 KiB fp32 chunk), so every stage is 32 KiB and the ring has 3 of them.
template <bool F32>
struct StateTraits {
  static constexpr int kRowBytes = kRowElems * (F32 ? 4 : 2);
  static constexpr int kChunkBytes = kBlockRows * kRowBytes;
  static constexpr int kChunksPerStage = F32 ? 1 : 2;
  static constexpr int kStageBytes = kChunksPerStage * kChunkBytes;
  static constexpr int kNumStages = kRingBytes / kStageBytes;
  static_assert(kNumStages >= 2 && kNumStages <= kStages, "ring geometry");
  static_assert(kChunksPerStage * 8 <= 32, "rows of a stage's chunks are packed 8 bits each");
};

// Stages of the ring's first pass over a CTA's `units` chunks (kj per
// output): their copies go out from the resolver right after it resolves
// them, or from the issuer warp on guessed indices (guessed_first_pass),
// instead of through the FIFO (adjacent rows only).  A stage holds up to
// kChunksPerStage consecutive chunks of one output.
template <bool F32>
__device__ __forceinline__ int first_pass_stages(int64_t units, int kj) {
  using T = StateTraits<F32>;
  const int64_t per_output = (kj + T::kChunksPerStage - 1) / T::kChunksPerStage;
  const int64_t total = units / kj * per_output;
  return static_cast<int>(total < T::kNumStages ? total : T::kNumStages);
}

// Chunks in the first n_pre stages (a stage never holds chunks of two
// outputs, so an output of kj chunks fills ceil(kj / kChunksPerStage)).
template <bool F32>
__device__ __forceinline__ int first_pass_units(int n_pre, int kj) {
  using T = StateTraits<F32>;
  const int per_output = (kj + T::kChunksPerStage - 1) / T::kChunksPerStage;
  const int rest = (n_pre % per_output) * T::kChunksPerStage;
  return (n_pre / per_output) * kj + (rest < kj ? rest : kj);
}

struct alignas(16) FifoEntry {
  long long off1, off2;  // byte offsets of the chunk's row runs (off1 < 0: unresolved)
  long long slot;        // output slot (first unit of an output only)
  long long pc;          // compressed position (first unit of an output only)
  int n1, n2;            // rows in each run
  int kk;                // chunk index within this CTA's range of its output
  int piece;             // output index relative to the cluster's first output
  int layer;             // layer whose state cache the chunk is read from
  int g1, o1;            // block and first row of run 1 (for a tensor copy)
};

template <int S>
struct ClusterShared {
  static constexpr int F = S < 8 ? S : 8;          // finaliser ranks
  static constexpr int WD = kHeadDim / F;          // dims per finaliser
  unsigned long long full_bar[kStages];
  unsigned long long empty_bar[kStages];
  unsigned long long fifo_full[2];
  unsigned long long fifo_empty[2];
  unsigned long long part_bar;                     // partials received
  unsigned long long ss_bar;                       // partial sums received
  FifoEntry fifo[2][kFifoChunk];
  MetaRec meta[kMetaRing];
  float recv[S > 1 ? S * 3 * WD : 1];              // [sender][m|den|num][WD]
  float recv_bad[S > 1 ? S : 1];
  float ss_recv[kMaxFinalizers];
  FinalScratch fs;
  uint32_t stage_rows[kStages];  // valid rows of each chunk of a stage, 8 bits each (0: unresolved)
  int abort_flag;
  int first_pass_owner;       // who issues the ring's first pass: 0 not yet, 1 issuer, 2 resolver
  long long resolver_start;   // clock64() when the resolver started (0: not yet)
};

__device__ __forceinline__ bool aborted(const int* flag) {
  return *reinterpret_cast<const volatile int*>(flag) != 0;
}

__device__ __forceinline__ void set_abort(int* flag) { *reinterpret_cast<volatile int*>(flag) = 1; }

// The resolver's issue of the ring's first pass (see resolver): called by
// the whole warp with each lane's FIFO entry of the first block.  Out of
// line, so that the resolver's loop stays as compact as it was: a larger
// kernel measured slower even where this code does not run.
// (The entry's fields travel as separate arguments, in registers: a
// reference would put the entry in local memory on the CTA's critical path.)
template <int S, bool F32>
__device__ __noinline__ void pre_issue_first_pass(const Params& p, ClusterShared<S>& sh, uint8_t* ring,
                                                  long long off1, long long off2, int n1, int n2,
                                                  int kk, int piece, int layer, long long slot,
                                                  long long pc, bool in_range, int kj, int n_pre) {
  using T = StateTraits<F32>;
  constexpr int CPS = T::kChunksPerStage;
  const int per_output = (kj + CPS - 1) / CPS;
  const int g = in_range ? piece * per_output + kk / CPS : n_pre;  // stage of the pass
  const bool mine = g < n_pre;
  const int half = kk % CPS;
  const bool valid = mine && off1 >= 0;
  const int nr = valid ? n1 + n2 : 0;
  if (valid) mbar_expect_tx(&sh.full_bar[g], static_cast<uint32_t>(nr * T::kRowBytes));
  if (mine && kk == 0) {
    MetaRec& m = sh.meta[piece % kMetaRing];
    m.slot = slot;
    m.pc = pc;
  }
  // rows of each chunk of the stage, 8 bits per chunk (the closing lane's
  // word takes its predecessor's chunk when the stage holds two)
  const uint32_t rows = static_cast<uint32_t>(nr) << (8 * half);
  const uint32_t prev = __shfl_up_sync(0xffffffffu, rows, 1);
  const bool closes = mine && (half == CPS - 1 || kk == kj - 1);
  __syncwarp();  // every byte count is announced before any stage's arrival
  if (valid) {
    const uint64_t policy = evict_first_policy();
    uint8_t* dst = ring + static_cast<size_t>(g) * T::kStageBytes +
                   static_cast<size_t>(half) * T::kChunkBytes;
    const uint8_t* state = p.states[layer];
    bulk_copy_g2s(dst, state + off1, n1 * T::kRowBytes, &sh.full_bar[g], policy);
    if (n2 > 0)
      bulk_copy_g2s(dst + n1 * T::kRowBytes, state + off2, n2 * T::kRowBytes, &sh.full_bar[g],
                    policy);
  }
  if (closes) {
    sh.stage_rows[g] = rows | (half == 1 ? prev : 0u);
    mbar_arrive(&sh.full_bar[g]);
  }
}

// The stage word of a first-pass stage whose guessed rows were wrong: the
// consumers skip the stage unread (a real word holds at most 8 rows a chunk).
constexpr uint32_t kJunkStage = 0xFFFFFFFFu;

// The issuer warp claims the ring's first pass only while the resolver has
// been running for fewer SM clocks than this (about 0.5 us); after that the
// resolver's own issue, which needs no check, comes first.  Measured in
// graph replay over the 12 benchmark shapes: 1000 and 1500 did best; 2000
// left one 64 MiB shape 0.5 % slower than without guesses, 3000 2 %.
constexpr long long kClaimWindow = 1000;

// The ring's first pass issued from guesses, by the whole issuer warp, with
// bulk copies of runs of adjacent rows, or (kTensorCopies, rows apart) a
// tensor copy per chunk lying in one block and row copies for a chunk split
// between two.  A CTA that is resident while the previous grid on
// the stream still runs would otherwise idle until the grid dependency wait
// releases, then walk the index chain (boundary index, then request and
// position, then block-table entry: three dependent loads, 1-1.5 us from L2
// under load) before its first copy.  Here lane i resolves unit i of the
// first pass from the index arrays as they stand, before the wait (L2-only
// loads, every index bounds-checked, nothing recorded), and the copies go
// out as soon as the wait releases.  One level of loads then checks every
// guess: the boundary index, request, position, slot and block-table
// entries, all at addresses the guesses give.  They are issued before the
// copies, since a load issued behind this SM's bulk copies waits for their
// data (measured: the check finished 1.8-2.6 us after the release that way,
// about 1.0 us this way).
//   Every guess held: the lanes write the outputs' slot records and the
//     stage words, and each stage gets its one arrival, as in the resolver's
//     own issue (pre_issue_first_pass).
//   Any guess failed: each stage still gets its arrival (the copies in
//     flight complete it) with the word kJunkStage; the consumers skip those
//     stages and the issuer copies the first pass again from the resolver's
//     FIFO, one ring pass later.  The results are the same either way.
// This warp claims the first pass with a compare-and-swap in shared memory,
// and only within kClaimWindow of the resolver's start: a CTA that became
// resident after the release would finish its guesses too late to gain.
// With adjacent rows the resolver makes the same claim after its own chain
// and issues the first pass when it wins; with rows apart it never does, so
// when this warp does not claim it the issuer starts from the first stage.
// Returns false only when this warp issued the first pass and a guess
// failed (the same on every lane).
// Measured in graph replay against the resolver's issue alone: the
// headline and every 128 and 256 MiB shape 1.6-1.9 % faster, 1 / 8192 at
// C = 512 8.5 %; the other 16 and 64 MiB shapes -2.3 .. +0.6 %; calls timed
// alone unchanged (no earlier grid, so no early CTA).  Rows apart: the
// headline shape 2.8 % faster, level with adjacent rows.
template <int S, bool F32, bool kTensorCopies>
__device__ __noinline__ bool guessed_first_pass(const Params& p, ClusterShared<S>& sh, uint8_t* ring,
                                                int64_t n0, int64_t units, int k_lo, int kj) {
  using T = StateTraits<F32>;
  constexpr int CPS = T::kChunksPerStage;
  const int lane = threadIdx.x & 31;
  // this warp's part in letting the next grid start launching (the CTA's
  // other threads give theirs after the wait)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int n_pre = first_pass_stages<F32>(units, kj);
  const int pre_units = first_pass_units<F32>(n_pre, kj);
  const bool mine = lane < pre_units;
  const int piece = lane / kj, kk = lane - piece * kj;
  const int64_t o = n0 + piece;  // output of the L * N space
  const int layer = static_cast<int>(o / p.num_outputs);
  const int64_t n = o - static_cast<int64_t>(layer) * p.num_outputs;
  const int64_t C = p.compress_ratio, B = p.block_size;
  const int64_t first_rel = static_cast<int64_t>(kBlockRows) * (k_lo + kk) - C + 1;  // + pos
  // the guess: the chain of resolve_chunk on the indices as they stand
  int64_t b = -1, r = -1, pos = -1, l1 = 0, g1 = -1, g2 = 0;
  int n1 = 0, n2 = 0;
  bool valid = false;
  if (mine) {
    b = ld_index<true>(p.bti + n);
    if (b >= 0 && b < p.num_tokens) {
      r = ld_index<true>(p.token_to_req + b);
      pos = ld_index<true>(p.positions + b);
      const int64_t left = C - static_cast<int64_t>(kBlockRows) * (k_lo + kk);
      if (r >= 0 && r < p.num_reqs && pos - C + 1 >= 0) {
        const int64_t first = pos + first_rel;
        const int nr = static_cast<int>(left < kBlockRows ? left : kBlockRows);
        l1 = first / B;
        const int64_t o1 = first - l1 * B;
        n1 = static_cast<int>(B - o1 < nr ? B - o1 : nr);
        n2 = nr - n1;
        if (l1 + (n2 > 0 ? 1 : 0) < p.max_blocks) {
          const int32_t* row = p.block_table + r * p.bt_row_stride;
          g1 = ld_index<true>(row + l1 * p.bt_col_stride);
          g2 = n2 > 0 ? ld_index<true>(row + (l1 + 1) * p.bt_col_stride) : 0;
          valid = g1 >= 0 && g1 < p.num_blocks && g2 >= 0 && g2 < p.num_blocks;
          if (valid && p.poison_guesses) g1 = g1 + 1 < p.num_blocks ? g1 + 1 : 0;
        }
      }
    }
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
  int won = 0;
  if (lane == 0) {
    const long long started = *reinterpret_cast<volatile long long*>(&sh.resolver_start);
    if (started == 0 || clock64() - started < kClaimWindow)
      won = atomicCAS(&sh.first_pass_owner, 0, 1) == 0;
  }
  if (!__shfl_sync(0xffffffffu, won, 0)) return true;  // the resolver issues it
  // the check's loads, ahead of the copies
  int64_t b2 = -1, r2 = -1, pos2 = -1, h1 = -1, h2 = 0, slot = -1;
  if (valid) {
    const int32_t* row = p.block_table + r * p.bt_row_stride;
    b2 = ld_index<true>(p.bti + n);
    r2 = ld_index<true>(p.token_to_req + b);
    pos2 = ld_index<true>(p.positions + b);
    h1 = ld_index<true>(row + l1 * p.bt_col_stride);
    if (n2 > 0) h2 = ld_index<true>(row + (l1 + 1) * p.bt_col_stride);
    if (kk == 0) slot = ld_index<true>(p.slot_map + (p.slot_by_token ? b : n));
  }
  // the copies of the guessed rows (the protocol of pre_issue_first_pass)
  const int g = piece * ((kj + CPS - 1) / CPS) + kk / CPS;  // stage of the pass
  const int half = kk % CPS;
  const int nr = n1 + n2;
  if (valid) mbar_expect_tx(&sh.full_bar[g], static_cast<uint32_t>(nr * T::kRowBytes));
  __syncwarp();  // every byte count is announced before any copy is issued
  if (valid) {
    const uint64_t policy = evict_first_policy();
    uint8_t* dst = ring + static_cast<size_t>(g) * T::kStageBytes +
                   static_cast<size_t>(half) * T::kChunkBytes;
    const uint8_t* state = p.states[layer];
    const int64_t o1 = pos + first_rel - l1 * B;
    if constexpr (!kTensorCopies) {
      bulk_copy_g2s(dst, state + g1 * p.state_block_bytes + o1 * p.state_row_bytes,
                    n1 * T::kRowBytes, &sh.full_bar[g], policy);
      if (n2 > 0)
        bulk_copy_g2s(dst + n1 * T::kRowBytes, state + g2 * p.state_block_bytes, n2 * T::kRowBytes,
                      &sh.full_bar[g], policy);
    } else if (n1 == kBlockRows) {  // the chunk's 8 rows in one block: one tensor copy
      tensor_copy_g2s(dst, &p.maps[layer], static_cast<int>(o1), static_cast<int>(g1),
                      &sh.full_bar[g], policy);
    } else {  // split between two blocks: row by row
      for (int r = 0; r < nr; ++r) {
        const long long off = r < n1 ? g1 * p.state_block_bytes + (o1 + r) * p.state_row_bytes
                                     : g2 * p.state_block_bytes + (r - n1) * p.state_row_bytes;
        bulk_copy_g2s(dst + r * T::kRowBytes, state + off, T::kRowBytes, &sh.full_bar[g], policy);
      }
    }
  }
  // the check: with the same boundary index, request and position the chunk
  // has the same runs, so equal block-table entries mean equal rows; the
  // output's slot record passes resolve_chunk's bounds checks
  bool match = !mine;
  int64_t pc = -1;
  if (valid) {
    match = b2 == b && r2 == r && pos2 == pos && h1 == g1 && h2 == g2;
    if (kk == 0) {
      pc = (pos / C) * C;
      match = match && pc < p.num_positions && (slot < 0 || slot / kSlotsPerPage < p.num_pages);
    }
  }
  const bool ok = __all_sync(0xffffffffu, match);
  if (ok && mine && kk == 0) {
    MetaRec& m = sh.meta[piece % kMetaRing];
    m.slot = slot;
    m.pc = pc;
  }
  // rows of each chunk of the stage, 8 bits per chunk (the closing lane's
  // word takes its predecessor's chunk when the stage holds two)
  const uint32_t rows = static_cast<uint32_t>(nr) << (8 * half);
  const uint32_t prev = __shfl_up_sync(0xffffffffu, rows, 1);
  const bool closes = mine && (half == CPS - 1 || kk == kj - 1);
  __syncwarp();  // the slot records are written before any stage's arrival
  if (closes) {
    sh.stage_rows[g] = ok ? (rows | (half == 1 ? prev : 0u)) : kJunkStage;
    mbar_arrive(&sh.full_bar[g]);
  }
  if (!ok && lane == 0) atomicAdd(p.rejections, 1ull);
  return ok;
}

// kBlocks: also pass each chunk's block and first row (tensor copies need
// them; adjacent rows leave the two fields alone).
//
// With adjacent rows (!kBlocks) the resolver also issues the copies of the
// ring's first pass (first_pass_stages) as soon as it has resolved them: the
// first chunks then start moving without waiting for the FIFO hand-off and
// the issuer's wake-up (about 0.75 us of every CTA's start, measured).  In
// graph replay every benchmark shape got faster, by 0.4-0.6 % on the
// 256 MiB ones, 1.1-2.9 % on the 64 and 128 MiB ones and 1.0 / 3.0 / 10.1 %
// on the 16 MiB ones at C = 128 / 256 / 512.  The
// protocol matches the issuer's: every lane announces its chunk's bytes on
// the stage barrier first (expect_tx, no arrival), then, after the warp has
// synchronised, issues its copies, and the lane holding a stage's last chunk
// writes the stage's row counts and makes the stage's one arrival.  The
// entries still go through the FIFO, where the issuer only keeps count.
// A CTA resident before the release may have issued the first pass from
// guesses already (guessed_first_pass): the resolver issues it only if it
// wins the claim, which it makes whatever happens (even after an abort),
// because the issuer counts those stages as issued and its final drain
// waits for them.
template <int S, bool F32, bool kBlocks>
__device__ void resolver(const Params& p, ClusterShared<S>& sh, uint8_t* ring, int64_t n0,
                         int64_t units, int k_lo, int kj) {
  using T = StateTraits<F32>;
  const int lane = threadIdx.x & 31;
  const int n_pre = kBlocks ? 0 : first_pass_stages<F32>(units, kj);
  if (lane == 0) *reinterpret_cast<volatile long long*>(&sh.resolver_start) = clock64();
  for (int64_t c = 0; c * kFifoChunk < units; ++c) {
    const int64_t i = c * kFifoChunk + lane;
    FifoEntry e{-1, -1, -1, -1, 0, 0, 0, 0, 0, 0, 0};
    if (i < units) {
      const int64_t q = i / kj;
      const int kk = static_cast<int>(i - q * kj);
      const int64_t o = n0 + q;                       // output of the L * N space
      const int layer = static_cast<int>(o / p.num_outputs);
      MetaRec rec;
      ChunkRuns cr;
      resolve_chunk(p, o - static_cast<int64_t>(layer) * p.num_outputs, k_lo + kk, kk == 0, cr, rec);
      e.layer = layer;
      e.off1 = cr.off1;
      e.off2 = cr.off2;
      e.n1 = cr.n1;
      e.n2 = cr.n2;
      if (kBlocks) {
        e.g1 = cr.g1;
        e.o1 = cr.o1;
      }
      e.slot = rec.slot;
      e.pc = rec.pc;
      e.kk = kk;
      e.piece = static_cast<int>(q);
    }
    if (c == 0 && n_pre > 0) {
      int won = 0;
      if (lane == 0) won = atomicCAS(&sh.first_pass_owner, 0, 2) == 0;
      if (__shfl_sync(0xffffffffu, won, 0))
        pre_issue_first_pass<S, F32>(p, sh, ring, e.off1, e.off2, e.n1, e.n2, e.kk, e.piece,
                                     e.layer, e.slot, e.pc, i < units, kj, n_pre);
    }
    const int h = static_cast<int>(c & 1);
    const uint32_t ph = static_cast<uint32_t>((c >> 1) & 1);
    bool ok = true;
    if (lane == 0) {
      ok = !aborted(&sh.abort_flag) && mbar_wait_bounded(&sh.fifo_empty[h], ph ^ 1u, p.wait_limit);
      if (!ok && !aborted(&sh.abort_flag)) {
        record_error(p.error, kErrTimeout);
        set_abort(&sh.abort_flag);
      }
    }
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (!ok) return;
    if (i < units) sh.fifo[h][lane] = e;
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh.fifo_full[h]);
  }
}

// How the issuer moves a chunk's rows into the ring.
//   kRuns:   rows of a block are adjacent; one bulk copy per run of rows.
//   kTensor: rows are apart and the layer has a TMA tensor map; one tensor
//            copy moves a chunk whose 8 rows lie in one block (a 256 x 4 x 8
//            box), and a chunk split between two blocks goes row by row.
//   kRows:   rows are apart, no map; one bulk copy per row, issued by the
//            lanes of the warp in parallel.
// Each copy has a fixed cost in the TMA unit, so eight 2 KiB copies take far
// longer than one of 16 KiB: with rows 64 elements apart the headline took
// 67.2 us with one lane issuing row copies, 52.0 us with eight lanes (kRows)
// and 42 us with tensor copies; per-row copies on adjacent rows were as slow
// (52.9 us), so the layout itself costs nothing.
enum class Copy { kRuns, kTensor, kRows };

// kRuns, kTensor: lane 0 alone walks the FIFO (the other lanes leave at
// once).  kRows: the whole warp walks it (lane 0 waits, announces bytes and
// arrives; the walk costs about 2.5 % against lane 0 alone).
template <int S, bool F32, Copy kCopy>
__device__ void issuer(const Params& p, ClusterShared<S>& sh, uint8_t* ring, int64_t units, int kj,
                       bool first_pass_held) {
  using T = StateTraits<F32>;
  constexpr bool kSplitRows = kCopy == Copy::kRows;
  const int lane = threadIdx.x & 31;
  if (!kSplitRows && lane != 0) return;
  const auto lane0_says = [](bool v) { return kSplitRows ? __shfl_sync(0xffffffffu, v, 0) : v; };
  const uint64_t policy = evict_first_policy();
  // the first pass's stages are issued by the resolver or from guesses
  // (adjacent rows), or from guesses alone (rows apart through tensor maps);
  // they count as issued at phase 0 from the start, so the drain waits for
  // them.  The issuer starts at the stage that follows them, with the units
  // after them, or with the first unit again when the guessed first pass
  // failed its check (first_pass_held false).
  // (rows apart through tensor maps: only when this warp claimed the first
  // pass, since the resolver never issues it there)
  const int n_pre = kCopy == Copy::kRuns ||
                            (kCopy == Copy::kTensor && sh.first_pass_owner == 1)
                        ? first_pass_stages<F32>(units, kj)
                        : 0;
  const int pre_units = n_pre > 0 ? first_pass_units<F32>(n_pre, kj) : 0;
  int stage = n_pre == T::kNumStages ? 0 : n_pre;
  uint32_t phase = n_pre == T::kNumStages ? 1u : 0u;
  uint32_t issued = (1u << n_pre) - 1u, last_parity = 0;
  uint32_t rows_word = 0;  // rows of each chunk of the open stage, 8 bits per chunk
  bool open = false;       // the current stage has copies announced but no arrival yet
  bool stop = false;
  for (int64_t c = 0; c * kFifoChunk < units && !stop; ++c) {
    const int h = static_cast<int>(c & 1);
    const uint32_t ph = static_cast<uint32_t>((c >> 1) & 1);
    bool ok = true;
    if (lane == 0) {
      ok = !aborted(&sh.abort_flag) && mbar_wait_bounded(&sh.fifo_full[h], ph, p.wait_limit);
      if (!ok && !aborted(&sh.abort_flag)) {
        record_error(p.error, kErrTimeout);
        set_abort(&sh.abort_flag);
      }
    }
    if (!lane0_says(ok)) break;
    const int64_t cnt = units - c * kFifoChunk < kFifoChunk ? units - c * kFifoChunk : kFifoChunk;
    for (int j = c == 0 && first_pass_held ? pre_units : 0; j < cnt; ++j) {
      const FifoEntry e = sh.fifo[h][j];
      const int half = e.kk % T::kChunksPerStage;  // which chunk of its stage
      const bool closes = half == T::kChunksPerStage - 1 || e.kk == kj - 1;
      if (half == 0) {
        bool free = true;
        if (lane == 0) {
          free = !aborted(&sh.abort_flag) && mbar_wait_bounded(&sh.empty_bar[stage], phase ^ 1u, p.wait_limit);
          if (!free && !aborted(&sh.abort_flag)) {
            record_error(p.error, kErrTimeout);
            set_abort(&sh.abort_flag);
          }
        }
        if (!lane0_says(free)) {
          stop = true;
          break;
        }
        rows_word = 0;
        open = true;
      }
      if (lane == 0 && e.kk == 0) {
        MetaRec& m = sh.meta[e.piece % kMetaRing];
        m.slot = e.slot;
        m.pc = e.pc;
      }
      if (e.off1 >= 0) {
        constexpr uint32_t kRowBytes = T::kRowBytes;
        uint8_t* dst = ring + static_cast<size_t>(stage) * T::kStageBytes +
                       static_cast<size_t>(half) * T::kChunkBytes;
        const int nr = e.n1 + e.n2;
        rows_word |= static_cast<uint32_t>(nr) << (8 * half);
        if (lane == 0) {
          if (closes) {
            sh.stage_rows[stage] = rows_word;
            mbar_arrive_expect_tx(&sh.full_bar[stage], nr * kRowBytes);
          } else {
            mbar_expect_tx(&sh.full_bar[stage], nr * kRowBytes);
          }
        }
        const uint8_t* state = p.states[e.layer];
        if constexpr (kCopy == Copy::kRuns) {
          bulk_copy_g2s(dst, state + e.off1, e.n1 * kRowBytes, &sh.full_bar[stage], policy);
          if (e.n2 > 0)
            bulk_copy_g2s(dst + e.n1 * kRowBytes, state + e.off2, e.n2 * kRowBytes,
                          &sh.full_bar[stage], policy);
        } else if constexpr (kCopy == Copy::kTensor) {
          if (e.n1 == kBlockRows) {
            tensor_copy_g2s(dst, &p.maps[e.layer], e.o1, e.g1, &sh.full_bar[stage], policy);
          } else {
            for (int r = 0; r < nr; ++r) {
              const long long off = r < e.n1 ? e.off1 + r * p.state_row_bytes
                                             : e.off2 + (r - e.n1) * p.state_row_bytes;
              bulk_copy_g2s(dst + r * kRowBytes, state + off, kRowBytes, &sh.full_bar[stage], policy);
            }
          }
        } else {
          __syncwarp();  // the bytes are announced before any row copy is issued
          if (lane < nr) {
            const long long off = lane < e.n1 ? e.off1 + lane * p.state_row_bytes
                                              : e.off2 + (lane - e.n1) * p.state_row_bytes;
            bulk_copy_g2s(dst + lane * kRowBytes, state + off, kRowBytes, &sh.full_bar[stage],
                          policy);
          }
        }
      } else if (closes && lane == 0) {  // an unresolved chunk keeps 0 rows
        sh.stage_rows[stage] = rows_word;
        mbar_arrive(&sh.full_bar[stage]);
      }
      if (closes) {
        open = false;
        issued |= 1u << stage;
        last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
        if (++stage == T::kNumStages) { stage = 0; phase ^= 1u; }
      }
    }
    if (kSplitRows) __syncwarp();  // every lane has read this FIFO half before it is handed back
    if (!stop && lane == 0) mbar_arrive(&sh.fifo_empty[h]);
  }
  if (lane != 0) return;
  if (open) {  // abandoned between the chunks of a stage: close it so the drain can wait on it
    sh.stage_rows[stage] = 0;
    mbar_arrive(&sh.full_bar[stage]);
    issued |= 1u << stage;
    last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
  }
  // No bulk copy may still target this CTA's shared memory when it exits.
  for (int s = 0; s < T::kNumStages; ++s)
    if ((issued >> s) & 1u)
      if (!mbar_wait_drain(&sh.full_bar[s], (last_parity >> s) & 1u)) record_error(p.error, kErrTimeout);
}

// cluster_waited: whether this thread has completed the start-up cluster
// barrier; if not, the consumers complete it before their first chunk
// (S > 1).
template <int S, bool F32>
__device__ void consumers(const Params& p, ClusterShared<S>& sh, const uint8_t* ring, int64_t n0,
                          int64_t n1, int kj, uint32_t rank, bool& cluster_waited) {
  using Sh = ClusterShared<S>;
  using T = StateTraits<F32>;
  constexpr int F = Sh::F, WD = Sh::WD;
  const int t = threadIdx.x, lane = t & 31;
  const bool finalizer = static_cast<int>(rank) < F;
  const int dbase = finalizer ? static_cast<int>(rank) * WD : 0;
  const bool active = finalizer && t < WD / 2;
  const int d0 = dbase + 2 * t;
  const bool rope = active && d0 >= kNopeDim;
  const int jp = (d0 - kNopeDim) >> 1;
  // where this thread's partial goes (S > 1): finaliser f, dim offset x
  const int f = (2 * t) / WD, x = 2 * t - f * WD;
  const uint32_t recv_l = smem_addr(sh.recv), bad_l = smem_addr(sh.recv_bad);
  const uint32_t ss_l = smem_addr(sh.ss_recv);
  const uint32_t part_bar_l = smem_addr(&sh.part_bar), ss_bar_l = smem_addr(&sh.ss_bar);
  if (S > 1 && !cluster_waited) {  // every rank's barriers exist before the first remote store
    cluster_wait();                 // (here the chunks are still on their way: off the critical path)
    cluster_waited = true;
  }
  int stage = 0;
  uint32_t phase = 0, mph = 0;
  for (int64_t q = 0; q < n1 - n0; ++q) {
    const int64_t o = n0 + q;  // output row of the L * N space
    const int layer = static_cast<int>(o / p.num_outputs);
    SoftmaxState s;
    state_reset(s);
    bool bad = false;
    MetaRec meta{-1, -1};
    float cs = 1.f, sn = 0.f;
    float2 w = make_float2(0.f, 0.f);  // RMSNorm weights of this thread's dims
    for (int kk = 0; kk < kj; kk += T::kChunksPerStage) {
      bool ready = false;
      if (!aborted(&sh.abort_flag)) {
        ready = mbar_wait_bounded(&sh.full_bar[stage], phase, p.wait_limit);
        if (!ready) {
          record_error(p.error, kErrTimeout);
          set_abort(&sh.abort_flag);
        }
      }
      const uint32_t word = ready ? sh.stage_rows[stage] : 0u;
      if (word == kJunkStage) {  // a guessed first-pass stage that failed its check
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.empty_bar[stage]);
        if (++stage == T::kNumStages) { stage = 0; phase ^= 1u; }
        kk -= T::kChunksPerStage;
        continue;
      }
      if (kk == 0 && ready) {
        // load what the finalise needs now, so its latency hides behind the window
        if (active) w = __ldg(reinterpret_cast<const float2*>(p.weights[layer] + d0));
        meta = sh.meta[q % kMetaRing];
        if (rope && meta.pc >= 0) {
          cs = __ldg(p.cos_sin + meta.pc * kRopeDim + jp);
          sn = __ldg(p.cos_sin + meta.pc * kRopeDim + kRopeDim / 2 + jp);
        }
      }
      constexpr uint32_t kTwoFull = kBlockRows | (kBlockRows << 8);
      if (!F32 && T::kChunksPerStage == 2 && kk + 1 < kj && word == kTwoFull) {
        // two full chunks: 16 rows, 2 KiB apart, one shared rescale
        fold_rows_n<2 * kBlockRows>(ring + static_cast<size_t>(stage) * T::kStageBytes, t, s);
      } else {
#pragma unroll
        for (int c = 0; c < T::kChunksPerStage; ++c) {
          if (kk + c >= kj) break;
          const uint32_t rows = (word >> (8 * c)) & 0xFFu;
          const uint8_t* chunk = ring + static_cast<size_t>(stage) * T::kStageBytes +
                                 static_cast<size_t>(c) * T::kChunkBytes;
          if (rows == kBlockRows) {
            if constexpr (F32) fold_f32<true>(chunk, t, s, kBlockRows);
            else fold_block(chunk, t, s);
          } else if (rows > 0) {
            if constexpr (F32) fold_f32<false>(chunk, t, s, static_cast<int>(rows));
            else fold_rows(chunk, t, s, static_cast<int>(rows));
          } else {
            bad = true;
          }
        }
      }
      __syncwarp();
      if (ready && lane == 0) mbar_arrive(&sh.empty_bar[stage]);
      if (++stage == T::kNumStages) { stage = 0; phase ^= 1u; }
    }

    if constexpr (S == 1) {
      const float c0 = s.a0 / s.d0, c1 = s.a1 / s.d1;
      const float total = consumer_sum_squares(sh.fs, c0, c1);
      finalize_slice(p, sh.fs, layer, o, true, 2 * t, c0, c1, w, bad, meta, cs, sn, total, 0, kHeadDim);
    } else {
      // push this rank's partial state to the finaliser of each dim
      const uint32_t fbar = peer_addr(part_bar_l, f);
      st_async_f2(peer_addr(recv_l + 4u * ((rank * 3 + 0) * WD + x), f), s.m0, s.m1, fbar);
      st_async_f2(peer_addr(recv_l + 4u * ((rank * 3 + 1) * WD + x), f), s.d0, s.d1, fbar);
      st_async_f2(peer_addr(recv_l + 4u * ((rank * 3 + 2) * WD + x), f), s.a0, s.a1, fbar);
      const bool any_bad = consumer_any(bad);
      if (t < F)
        st_async_f32(peer_addr(bad_l + 4u * rank, t), any_bad ? 1.f : 0.f, peer_addr(part_bar_l, t));
      float c0 = 0.f, c1 = 0.f;
      bool mbad = any_bad;
      if (finalizer) {
        if (t == 0) mbar_arrive_expect_tx(&sh.part_bar, S * (WD * 12 + 4));
        if (!mbar_wait_cluster_bounded(&sh.part_bar, mph)) {
          record_error(p.error, kErrTimeout);
          set_abort(&sh.abort_flag);
          mbad = true;
        }
        if (active) {
          float M0 = -INFINITY, M1 = -INFINITY, D0 = 0.f, D1 = 0.f, A0 = 0.f, A1 = 0.f;
#pragma unroll
          for (int j = 0; j < S; ++j) {
            const float2 m = *reinterpret_cast<const float2*>(sh.recv + (j * 3 + 0) * WD + 2 * t);
            const float2 d = *reinterpret_cast<const float2*>(sh.recv + (j * 3 + 1) * WD + 2 * t);
            const float2 a = *reinterpret_cast<const float2*>(sh.recv + (j * 3 + 2) * WD + 2 * t);
            const float nm0 = fmaxf(M0, m.x), nm1 = fmaxf(M1, m.y);
            const float r0 = fast_ex2((M0 - nm0) * kLog2e), r1 = fast_ex2((M1 - nm1) * kLog2e);
            const float f0 = fast_ex2((m.x - nm0) * kLog2e), f1 = fast_ex2((m.y - nm1) * kLog2e);
            D0 = fmaf(d.x, f0, D0 * r0);
            D1 = fmaf(d.y, f1, D1 * r1);
            A0 = fmaf(a.x, f0, A0 * r0);
            A1 = fmaf(a.y, f1, A1 * r1);
            M0 = nm0;
            M1 = nm1;
            mbad |= sh.recv_bad[j] != 0.f;
          }
          c0 = A0 / D0;
          c1 = A1 / D1;
        }
        // this slice's sum of squares, pushed to every rank
        const float ssw = warp_sum(active ? c0 * c0 + c1 * c1 : 0.f);
        if (lane == 0) sh.fs.red[t >> 5] = ssw;
        consumer_sync();
        if (t == 0) {
          float mine = 0.f;
#pragma unroll
          for (int i = 0; i < kConsumerWarps; ++i) mine += sh.fs.red[i];
#pragma unroll
          for (int r = 0; r < S; ++r) st_async_f32(peer_addr(ss_l + 4u * rank, r), mine, peer_addr(ss_bar_l, r));
        }
      }
      if (t == 0) mbar_arrive_expect_tx(&sh.ss_bar, F * 4);
      if (!mbar_wait_cluster_bounded(&sh.ss_bar, mph)) {
        record_error(p.error, kErrTimeout);
        set_abort(&sh.abort_flag);
        mbad = true;
      }
      mph ^= 1u;
      if (finalizer) {
        float total = 0.f;
#pragma unroll
        for (int i = 0; i < F; ++i) total += sh.ss_recv[i];
        finalize_slice(p, sh.fs, layer, o, active, d0, c0, c1, w, mbad, meta, cs, sn, total, dbase,
                       WD);
      } else {
        consumer_sync();  // sh.fs.red is rewritten by the next output
      }
    }
  }
}

// Before the grid dependency wait, the previous grid on the stream may still
// be writing this call's inputs, so nothing read then may reach a result;
// it may still warm L2.  Lane i resolves unit i of the CTA from the index
// arrays as they stand (L2-only loads, every index bounds-checked, nothing
// recorded), which brings the index lines of the resolver's first FIFO
// block into L2, and the lanes of the first stages prefetch their chunk's
// rows into L2.  A prefetch changes only what the cache holds and L2 stays
// coherent with the previous grid's writes, so no result can go stale.  When
// that grid is still running, this grid's first reads start in its tail
// instead of after the wait; when none is, they still start before the
// resolver-to-issuer hand-off.
template <bool F32>
__device__ void prefetch_first_stages(const Params& p, int64_t n0, int64_t units, int k_lo, int kj,
                                      bool maps) {
  using T = StateTraits<F32>;
  const int lane = threadIdx.x & 31;
  if (lane >= units) return;
  const int64_t q = lane / kj;
  const int kk = lane - static_cast<int>(q) * kj;
  const int64_t o = n0 + q;
  const int layer = static_cast<int>(o / p.num_outputs);
  ChunkRuns cr;
  MetaRec rec;
  resolve_chunk_t<true>(p, o - static_cast<int64_t>(layer) * p.num_outputs, k_lo + kk, false, cr, rec);
  // How much to prefetch, as measured on the bf16 shapes: the ring's first
  // pass, i.e. the chunks the issuer copies before it first waits for a
  // free stage.  Against two stages this took 0.5 % off the headline in
  // graph replay and cost some mid-size calls with no earlier grid to
  // overlap about 1 us (their prefetches queue ahead of the real copies);
  // ten chunks, past the ring, were slower both ways (up to 4.5 % in replay
  // and 10 % cold on the 64 MiB shapes).  Rows apart without a map take
  // one prefetch per row: the first stage alone.
  const int first = (p.rows_contiguous || maps ? T::kNumStages : 1) * T::kChunksPerStage;
  if (cr.off1 < 0 || lane >= first) return;
  const uint8_t* state = p.states[layer];
  if (p.rows_contiguous) {
    bulk_prefetch_l2(state + cr.off1, cr.n1 * T::kRowBytes);
    if (cr.n2 > 0) bulk_prefetch_l2(state + cr.off2, cr.n2 * T::kRowBytes);
  } else if (maps && cr.n1 == kBlockRows) {
    tensor_prefetch_l2(&p.maps[layer], cr.o1, cr.g1);
  } else {
    for (int r = 0; r < cr.n1 + cr.n2; ++r) {
      const long long off = r < cr.n1 ? cr.off1 + r * p.state_row_bytes
                                      : cr.off2 + (r - cr.n1) * p.state_row_bytes;
      bulk_prefetch_l2(state + off, T::kRowBytes);
    }
  }
}

// kApart: the rows of a block are apart (tensor or row copies); otherwise
// adjacent (run copies).  The tensor-copy path lives in the kApart kernels
// only: in the same kernel as the run copies it cost the adjacent-row
// headline 0.4-0.6 %.  The parameters are __grid_constant__ so that the
// tensor maps in them can be addressed in place by the TMA unit.
template <int S, bool F32, bool kApart>
__global__ void __launch_bounds__(kClusterThreads, 2)
    kvc_cluster_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(128) uint8_t smem[];
  ClusterShared<S>& sh = *reinterpret_cast<ClusterShared<S>*>(smem + kRingBytes);
  const uint32_t rank = S > 1 ? cluster_ctarank() : 0u;
  const int64_t c = blockIdx.x / S, ncl = gridDim.x / S;
  const int64_t N = p.num_outputs * p.num_layers;  // outputs of all layers
  const int64_t n0 = c * N / ncl, n1 = (c + 1) * N / ncl;
  const int K = p.blocks_per_output;
  const int k_lo = static_cast<int>(rank) * K / S;
  const int kj = (static_cast<int>(rank) + 1) * K / S - k_lo;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sh.full_bar[s], 1);
      mbar_init(&sh.empty_bar[s], kConsumerWarps);
    }
    for (int h = 0; h < 2; ++h) {
      mbar_init(&sh.fifo_full[h], 1);
      mbar_init(&sh.fifo_empty[h], 1);
    }
    mbar_init(&sh.part_bar, 1);
    mbar_init(&sh.ss_bar, 1);
    sh.abort_flag = 0;
    sh.first_pass_owner = 0;
    sh.resolver_start = 0;
    fence_mbar_init();
  }
  // With S > 1 the peers' barriers must exist before the first remote store.
  // For clusters of 2 and 4 the cluster barrier that ensures it is split:
  // every thread arrives now, the consumers wait before their first chunk
  // and the rest at the end, so the resolver and the issuer start without
  // waiting for the slowest rank to come up.  Measured in graph replay: the
  // 64 MiB shapes at C = 256 and 512 (S = 2 and 4) 3-4 % faster; clusters of
  // 8 were 1-2 % slower split, so they keep one barrier here.
  constexpr bool kSplitStart = S == 2 || S == 4;
  bool cluster_waited = !kSplitStart;
  if constexpr (kSplitStart) {
    __syncthreads();  // this CTA's barriers exist before its own threads use them
    cluster_arrive_relaxed();
  } else if constexpr (S > 1) {
    cluster_sync_all();  // every rank's barriers exist before any remote store
  } else {
    __syncthreads();
  }
  // Tensor copies need the ring 128-byte aligned and the maps 64-byte aligned;
  // failing either, rows apart go row by row.
  const bool maps = kApart && p.use_maps && (smem_addr(smem) & 127u) == 0 &&
                    (reinterpret_cast<uintptr_t>(&p.maps[0]) & 63u) == 0;
  // Warp 0 (a consumer warp, idle until the first chunk lands) warms L2; the
  // other warps go straight on.
  if (threadIdx.x < 32 && n0 < n1 && kj > 0)
    prefetch_first_stages<F32>(p, n0, (n1 - n0) * kj, k_lo, kj, maps);
  // Wait for the previous grid on the stream (programmatic dependent launch)
  // before reading any input for a result, and let the next one start
  // launching.  With adjacent rows, or rows apart copied through tensor
  // maps, the issuer warp waits inside guessed_first_pass.
  const int warp = threadIdx.x >> 5;
  bool first_pass_held = true;
  if (!kApart && warp == kIssuerWarp && p.rows_contiguous && n0 < n1 && kj > 0) {
    first_pass_held = guessed_first_pass<S, F32, false>(p, sh, smem, n0, (n1 - n0) * kj, k_lo, kj);
  } else if (kApart && maps && warp == kIssuerWarp && n0 < n1 && kj > 0) {
    first_pass_held = guessed_first_pass<S, F32, true>(p, sh, smem, n0, (n1 - n0) * kj, k_lo, kj);
  } else {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  }
  if (n0 < n1 && kj > 0) {
    const int64_t units = (n1 - n0) * kj;
    if (warp == kResolverWarp) {
      resolver<S, F32, kApart>(p, sh, smem, n0, units, k_lo, kj);
    } else if (warp == kIssuerWarp) {
      if constexpr (!kApart) {
        // Rows are adjacent whenever this kernel runs.  The row-copy branch
        // stays in its code all the same: without it the kernel's code layout
        // changed and the 64 MiB C = 128 shape measured 1.5 % slower.
        if (p.rows_contiguous) issuer<S, F32, Copy::kRuns>(p, sh, smem, units, kj, first_pass_held);
        else issuer<S, F32, Copy::kRows>(p, sh, smem, units, kj, true);
      } else if (maps) {
        issuer<S, F32, Copy::kTensor>(p, sh, smem, units, kj, first_pass_held);
      } else {
        issuer<S, F32, Copy::kRows>(p, sh, smem, units, kj, true);
      }
    } else {
      consumers<S, F32>(p, sh, smem, n0, n1, kj, rank, cluster_waited);
    }
  }
  if (S > 1) {
    if (!cluster_waited) cluster_wait();
    cluster_sync_all();  // no CTA leaves while a peer may still write to it
  }
}

template <int S>
size_t smem_bytes_of() {
  return static_cast<size_t>(kRingBytes) + sizeof(ClusterShared<S>);
}

template <int S>
cudaLaunchConfig_t config_of(int clusters, cudaStream_t stream, cudaLaunchAttribute* attrs) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(clusters * S));
  cfg.blockDim = dim3(kClusterThreads);
  cfg.dynamicSmemBytes = smem_bytes_of<S>();
  cfg.stream = stream;
  attrs[0].id = cudaLaunchAttributeClusterDimension;
  attrs[0].val.clusterDim.x = static_cast<unsigned>(S);
  attrs[0].val.clusterDim.y = 1;
  attrs[0].val.clusterDim.z = 1;
  attrs[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = 2;
  return cfg;
}

template <int S, bool F32, bool kApart>
int prepare_and_capacity() {
  const void* fn = reinterpret_cast<const void*>(&kvc_cluster_kernel<S, F32, kApart>);
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem_bytes_of<S>())) != cudaSuccess)
    return 0;
  if (S > 8 && cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
    return 0;
  cudaLaunchAttribute attrs[2];
  cudaLaunchConfig_t cfg = config_of<S>(1, nullptr, attrs);
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, &kvc_cluster_kernel<S, F32, kApart>, &cfg) != cudaSuccess)
    return 0;
  return n;
}

// Every kernel of a cluster size shares the footprint; the capacity is the
// smallest one.
template <int S>
int prepare_and_capacity_both() {
  const int c[4] = {prepare_and_capacity<S, false, false>(), prepare_and_capacity<S, true, false>(),
                    prepare_and_capacity<S, false, true>(), prepare_and_capacity<S, true, true>()};
  int n = c[0];
  for (int i = 1; i < 4; ++i) n = c[i] < n ? c[i] : n;
  return n;
}

template <int S>
cudaError_t launch_of(const Params& p, int clusters, cudaStream_t stream) {
  cudaLaunchAttribute attrs[2];
  cudaLaunchConfig_t cfg = config_of<S>(clusters, stream, attrs);
  cudaError_t e;
  if (p.rows_contiguous) {
    e = p.state_f32 ? cudaLaunchKernelEx(&cfg, &kvc_cluster_kernel<S, true, false>, p)
                    : cudaLaunchKernelEx(&cfg, &kvc_cluster_kernel<S, false, false>, p);
  } else {
    e = p.state_f32 ? cudaLaunchKernelEx(&cfg, &kvc_cluster_kernel<S, true, true>, p)
                    : cudaLaunchKernelEx(&cfg, &kvc_cluster_kernel<S, false, true>, p);
  }
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

int cluster_threads() { return kClusterThreads; }

// cuTensorMapEncodeTiled, looked up once through the runtime (no link against
// the driver library).  Null when the driver does not offer it.
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

namespace {

EncodeTiledFn encode_tiled() {
  static const EncodeTiledFn fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess) {
      (void)cudaGetLastError();
      return static_cast<EncodeTiledFn>(nullptr);
    }
    return reinterpret_cast<EncodeTiledFn>(f);
  }();
  return fn;
}

}  // namespace

// The TMA tensor map of one layer's state when its rows are apart: the 4-D
// view (256 elements, 4 row segments, block_size rows, num_blocks blocks)
// with strides (256 elements, row stride, block stride) in bytes, and a box
// of 8 whole rows.  L2 fills in 128-byte granules: rows start on 128-byte
// boundaries, and 256-byte fills read 3 % more than the rows (part of the
// gap after every other row).  False when the driver refuses the map or a
// coordinate would not fit the 32-bit tensor coordinates; the call then
// copies row by row.
bool encode_rows_map(CUtensorMap* m, const void* base, bool f32, int64_t block_size,
                     int64_t num_blocks, int64_t row_bytes, int64_t block_bytes) {
  const EncodeTiledFn fn = encode_tiled();
  if (!fn || num_blocks > INT32_MAX || block_size > INT32_MAX || row_bytes <= 0 ||
      block_bytes <= 0 || row_bytes >= (int64_t{1} << 40) || block_bytes >= (int64_t{1} << 40))
    return false;
  const cuuint64_t esize = f32 ? 4 : 2;
  const cuuint64_t dims[4] = {kMapInner, kMapSegments, static_cast<cuuint64_t>(block_size),
                              static_cast<cuuint64_t>(num_blocks)};
  const cuuint64_t strides[3] = {kMapInner * esize, static_cast<cuuint64_t>(row_bytes),
                                 static_cast<cuuint64_t>(block_bytes)};
  const cuuint32_t box[4] = {kMapInner, kMapSegments, kBlockRows, 1};
  const cuuint32_t unit[4] = {1, 1, 1, 1};
  return fn(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
            const_cast<void*>(base), dims, strides, box, unit, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t cluster_smem_bytes(int S) {
  switch (S) {
    case 1: return smem_bytes_of<1>();
    case 2: return smem_bytes_of<2>();
    case 4: return smem_bytes_of<4>();
    case 8: return smem_bytes_of<8>();
    case 16: return smem_bytes_of<16>();
  }
  return 0;
}

int cluster_capacity(int S) {
  int n = 0;
  switch (S) {
    case 1: n = prepare_and_capacity_both<1>(); break;
    case 2: n = prepare_and_capacity_both<2>(); break;
    case 4: n = prepare_and_capacity_both<4>(); break;
    case 8: n = prepare_and_capacity_both<8>(); break;
    case 16: n = prepare_and_capacity_both<16>(); break;
  }
  (void)cudaGetLastError();  // a refused size leaves no sticky error behind
  return n;
}

cudaError_t launch_cluster(const Params& p, int clusters, cudaStream_t stream) {
  switch (p.cluster_size) {
    case 1: return launch_of<1>(p, clusters, stream);
    case 2: return launch_of<2>(p, clusters, stream);
    case 4: return launch_of<4>(p, clusters, stream);
    case 8: return launch_of<8>(p, clusters, stream);
    case 16: return launch_of<16>(p, clusters, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace kvc
