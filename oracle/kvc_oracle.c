/*
 * CPU oracle for the KV-cache window compressor -- TEST INFRASTRUCTURE ONLY.
 *
 * This file is the plain, slow definition the CUDA library is checked
 * against.  Only the tests, the smoke check and the benchmark's CPU-baseline
 * leg may load it; the product path never does.  It shares no code, header,
 * table or constant generator with the CUDA library.
 *
 * Source of every step: "From Attention to KV Cache Compression: Notes from a
 * KernelGen Optimization" (KernelGen Challenge 8 write-up), sections
 *   "Gather and Scatter"           - constants and the packed slot layout,
 *   "How One Output Is Produced"   - window, paged addressing, per-dimension
 *                                    softmax sum, RMSNorm, NOPE quantisation,
 *                                    GPT-J RoPE and the scatter address,
 *   "The Baseline"                 - gather-then-softmax semantics, and its
 *                                    traffic count with an fp32 state element,
 *   "A Bit of Triton and GPU Background" - the state read through explicit
 *                                    block / row / column strides,
 *   "The Finalizer's Sharp Edges"  - fp32 finalizer, bf16 round trip,
 *                                    truncation toward zero, byte encoding.
 *
 * Precision: the window reduction and rho are evaluated in double (the pages
 * fix fp32 only for the compressed vector they hand on, so the oracle takes
 * the tighter route and rounds c to float at the end).  The finalizer (y,
 * quantisation, RoPE) is evaluated in fp32 exactly as the page's finalizer
 * does, one rounded operation at a time; build with -ffp-contract=off.
 *
 * The state may be bf16 or fp32 and strided (kvc_oracle_*_ex): every element
 * is widened exactly to double, so both dtypes follow one definition.
 *
 * The reader direction (kvc_oracle_dequantize) decodes a packed slot back to
 * a 512-vector: NOPE values q * 2^(scale - 127), RoPE values as stored.
 *
 * Parity pins: every function here is pinned by tests/test_oracle_*.py
 * against closed forms, library routines (torch softmax / rms_norm / bf16
 * cast, complex multiplication), exact rational arithmetic and hand-worked
 * fixtures in tests/golden/.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

/* constants of the section "Gather and Scatter" */
enum {
  OR_HEAD_DIM = 512,       /* width of the compressed vector            */
  OR_ROPE_DIM = 64,        /* last 64 dims: RoPE, stored as bf16        */
  OR_NOPE_DIM = 448,       /* first 448 dims: int8 with per-64 scales   */
  OR_GROUP = 64,           /* dims per quantisation group               */
  OR_SLOTS_PER_PAGE = 64,  /* KV_BLOCK_SIZE                             */
  OR_TOKEN_STRIDE = 576,   /* payload bytes per slot                    */
  OR_SCALE_DIM = 8,        /* scale bytes per slot (7 used + 1 padding) */
};
#define OR_PAGE_BYTES (OR_SLOTS_PER_PAGE * (OR_TOKEN_STRIDE + OR_SCALE_DIM))

/* error codes returned by the oracle (0 = ok) */
enum { OR_OK = 0, OR_BAD_INDEX = 4 };

/* ---- bf16 helpers --------------------------------------------------- */

/* A bf16 value is the upper half of an IEEE binary32; widening is exact. */
static float or_bf16_bits_to_float(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/*
 * Round a finite binary32 to bf16, round-to-nearest, ties-to-even, written
 * from the definition: the two bf16 neighbours of x are x with the low 16
 * bits cleared (toward zero) and the next bf16 away from zero; the low 16
 * bits measure the distance to the lower one in units of 2^-16 ulp.
 */
uint16_t kvc_oracle_f32_to_bf16(float x) {
  uint32_t u;
  memcpy(&u, &x, sizeof u);
  uint32_t toward_zero = u >> 16;        /* sign|exp|7 mantissa bits       */
  uint32_t rest = u & 0xFFFFu;           /* discarded low mantissa bits    */
  uint32_t away = toward_zero + 1u;      /* next magnitude (carries into e)*/
  if (rest > 0x8000u) return (uint16_t)away;
  if (rest < 0x8000u) return (uint16_t)toward_zero;
  return (uint16_t)((toward_zero & 1u) ? away : toward_zero); /* tie: even */
}

float kvc_oracle_bf16_round(float x) {
  return or_bf16_bits_to_float(kvc_oracle_f32_to_bf16(x));
}

/* The same rounding over an array (lets the tests sweep many inputs). */
void kvc_oracle_f32_to_bf16_n(const float* x, uint16_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = kvc_oracle_f32_to_bf16(x[i]);
}

/* ---- quantisation exponent ------------------------------------------ */

/*
 * e = ceil(log2(a / 127)) for a > 0, evaluated exactly: it is the smallest
 * integer e with 127 * 2^e >= a.  127 * 2^e and a (a float) are both exact
 * doubles, so the comparisons are exact.  frexp gives a first guess.
 */
int kvc_oracle_scale_exponent(float a) {
  int ea;
  (void)frexp((double)a / 127.0, &ea);  /* a/127 in [2^(ea-1), 2^ea) approx */
  int e = ea + 1;
  while (ldexp(127.0, e - 1) >= (double)a) --e;
  while (ldexp(127.0, e) < (double)a) ++e;
  return e;
}

/* ---- step 1+2: window gather and per-dimension softmax sum ----------- */

/* Element `col` of physical row (g, o) of the state, widened exactly to
 * double.  state_dtype 1 = bf16, 2 = fp32; strides in elements. */
static double or_state_elem(const void* state, int state_dtype, int64_t block_stride,
                            int64_t row_stride, int64_t g, int64_t o, int64_t col) {
  int64_t idx = g * block_stride + o * row_stride + col;
  if (state_dtype == 2) return (double)((const float*)state)[idx];
  return (double)or_bf16_bits_to_float(((const uint16_t*)state)[idx]);
}

/*
 * For each output n (boundary token b = boundary_token_indices[n]):
 *   r = token_to_req[b], p = positions[b], t_i = p - C + 1 + i (0 <= i < C),
 *   l_i = floor(t_i / B), o_i = t_i mod B, g_i = block_table[r, l_i],
 *   row_i = (g_i, o_i); v = state[row_i, 0:512], s = state[row_i, 512:1024]
 *   c_d = sum_i softmax_i(s_{., d}) * v_{i, d}   (softmax along the window).
 * Two-pass softmax in double: max, then sum of exp and weighted sum.
 * The state is bf16 (state_dtype 1) or fp32 (2) with the given element
 * strides between physical blocks and between rows of a block (columns are
 * contiguous); block_table[r, l] is at r * bt_row_stride + l * bt_col_stride.
 * c is written as float [N, 512].  Returns OR_BAD_INDEX on any index that
 * falls outside its array; nothing is written for that output then and
 * valid_out[n] (if valid_out is not NULL) is set to 0, else to 1.
 */
int kvc_oracle_window_reduce_ex(
    const void* state, int32_t state_dtype, int64_t state_block_stride,
    int64_t state_row_stride, int64_t num_state_blocks, int32_t block_size,
    const int32_t* token_to_req, const int64_t* positions, int64_t num_tokens,
    const int64_t* boundary_token_indices, int64_t num_outputs,
    const int32_t* block_table, int64_t num_reqs, int64_t max_blocks_per_req,
    int64_t bt_row_stride, int64_t bt_col_stride,
    int32_t compress_ratio, float* c_out, uint8_t* valid_out) {
  const int64_t C = compress_ratio, B = block_size;
  int status = OR_OK;
  double m[OR_HEAD_DIM], den[OR_HEAD_DIM], num[OR_HEAD_DIM];
  for (int64_t n = 0; n < num_outputs; ++n) {
    if (valid_out) valid_out[n] = 0;
    int64_t b = boundary_token_indices[n];
    if (b < 0 || b >= num_tokens) { status = OR_BAD_INDEX; continue; }
    int64_t r = token_to_req[b];
    int64_t p = positions[b];
    if (r < 0 || r >= num_reqs || p - C + 1 < 0) { status = OR_BAD_INDEX; continue; }
    /* resolve every row of the window first */
    int ok = 1;
    for (int64_t i = 0; i < C && ok; ++i) {
      int64_t t = p - C + 1 + i;
      int64_t l = t / B;
      if (l >= max_blocks_per_req) { ok = 0; break; }
      int64_t g = block_table[r * bt_row_stride + l * bt_col_stride];
      if (g < 0 || g >= num_state_blocks) ok = 0;
    }
    if (!ok) { status = OR_BAD_INDEX; continue; }
    for (int d = 0; d < OR_HEAD_DIM; ++d) { m[d] = -INFINITY; den[d] = 0.0; num[d] = 0.0; }
    /* pass 1: per-dimension maximum of the scores */
    for (int64_t i = 0; i < C; ++i) {
      int64_t t = p - C + 1 + i;
      int64_t g = block_table[r * bt_row_stride + (t / B) * bt_col_stride];
      for (int d = 0; d < OR_HEAD_DIM; ++d) {
        double sd = or_state_elem(state, state_dtype, state_block_stride, state_row_stride, g,
                                  t % B, OR_HEAD_DIM + d);
        if (sd > m[d]) m[d] = sd;
      }
    }
    /* pass 2: denominators and weighted numerators */
    for (int64_t i = 0; i < C; ++i) {
      int64_t t = p - C + 1 + i;
      int64_t g = block_table[r * bt_row_stride + (t / B) * bt_col_stride];
      for (int d = 0; d < OR_HEAD_DIM; ++d) {
        double sd = or_state_elem(state, state_dtype, state_block_stride, state_row_stride, g,
                                  t % B, OR_HEAD_DIM + d);
        double vd = or_state_elem(state, state_dtype, state_block_stride, state_row_stride, g,
                                  t % B, d);
        double e = exp(sd - m[d]);
        den[d] += e;
        num[d] += e * vd;
      }
    }
    for (int d = 0; d < OR_HEAD_DIM; ++d)
      c_out[n * OR_HEAD_DIM + d] = (float)(num[d] / den[d]);
    if (valid_out) valid_out[n] = 1;
  }
  return status;
}

/* The same for a contiguous bf16 state [num_blocks, B, 1024] and a
 * row-major block_table [num_reqs, max_blocks_per_req]. */
int kvc_oracle_window_reduce(
    const uint16_t* state, int64_t num_state_blocks, int32_t block_size,
    const int32_t* token_to_req, const int64_t* positions, int64_t num_tokens,
    const int64_t* boundary_token_indices, int64_t num_outputs,
    const int32_t* block_table, int64_t num_reqs, int64_t max_blocks_per_req,
    int32_t compress_ratio, float* c_out, uint8_t* valid_out) {
  const int64_t W = 2 * OR_HEAD_DIM;
  return kvc_oracle_window_reduce_ex(
      state, 1, (int64_t)block_size * W, W, num_state_blocks, block_size, token_to_req,
      positions, num_tokens, boundary_token_indices, num_outputs, block_table, num_reqs,
      max_blocks_per_req, max_blocks_per_req, 1, compress_ratio, c_out, valid_out);
}

/* ---- step 3: RMSNorm ------------------------------------------------ */

/*
 * rho = (mean_d c_d^2 + eps)^(-1/2), y_d = c_d * rho * w_d.
 * The mean and rho are taken in double and rho is rounded to float; the two
 * products are fp32 operations in the page's order ((c * rho) * w).
 */
void kvc_oracle_rmsnorm(const float* c, const float* weight, float eps,
                        int64_t num_outputs, float* y_out) {
  for (int64_t n = 0; n < num_outputs; ++n) {
    const float* cn = c + n * OR_HEAD_DIM;
    double ss = 0.0;
    for (int d = 0; d < OR_HEAD_DIM; ++d) ss += (double)cn[d] * (double)cn[d];
    double mean = ss / OR_HEAD_DIM;
    float rho = (float)(1.0 / sqrt(mean + (double)eps));
    for (int d = 0; d < OR_HEAD_DIM; ++d) {
      float t = cn[d] * rho;
      y_out[n * OR_HEAD_DIM + d] = t * weight[d];
    }
  }
}

/* ---- steps 4-6: NOPE quantisation, RoPE, scatter --------------------- */

/*
 * Builds the 576 payload bytes and 8 scale bytes of one output from its
 * normalised vector y[512]:
 *   z_d = fp32(bf16(y_d)) for d < 448; per 64-group g:
 *     a_g = max(max |z_d|, 1e-4), e_g = ceil(log2(a_g / 127)),
 *     q_d = int8(clip(z_d * 2^-e_g, -127, 127)) truncated toward zero,
 *     scale byte g = e_g + 127;  byte 7 of the scale record is 0 (padding).
 *   RoPE on dims 448..511, GPT-J interleaved pairs (448+2j, 449+2j):
 *     u' = u cos_j - w sin_j, w' = w cos_j + u sin_j, in fp32, then bf16;
 *     cos_j = cos_sin[pc, j], sin_j = cos_sin[pc, 32 + j].
 * Payload = [448 int8 bytes][64 bf16 little-endian = 128 bytes].
 */
void kvc_oracle_pack_slot(const float* y, const float* cos_row,
                          uint8_t payload[576], uint8_t scale[8]) {
  for (int g = 0; g < OR_NOPE_DIM / OR_GROUP; ++g) {
    float z[OR_GROUP];
    float a = 0.0f;
    for (int k = 0; k < OR_GROUP; ++k) {
      z[k] = kvc_oracle_bf16_round(y[g * OR_GROUP + k]);
      float mag = fabsf(z[k]);
      if (mag > a) a = mag;
    }
    if (a < 1.0e-4f) a = 1.0e-4f;
    int e = kvc_oracle_scale_exponent(a);
    for (int k = 0; k < OR_GROUP; ++k) {
      double scaled = ldexp((double)z[k], -e);  /* exact: power-of-two scale */
      if (scaled > 127.0) scaled = 127.0;
      if (scaled < -127.0) scaled = -127.0;
      int q = (int)trunc(scaled);
      payload[g * OR_GROUP + k] = (uint8_t)(q & 0xFF);  /* two's complement */
    }
    scale[g] = (uint8_t)(e + 127);
  }
  scale[7] = 0;
  for (int j = 0; j < OR_ROPE_DIM / 2; ++j) {
    float u = y[OR_NOPE_DIM + 2 * j];
    float w = y[OR_NOPE_DIM + 2 * j + 1];
    float cs = cos_row[j], sn = cos_row[OR_ROPE_DIM / 2 + j];
    float uc = u * cs, ws = w * sn, wc = w * cs, us = u * sn;
    float ru = uc - ws;
    float rw = wc + us;
    uint16_t hu = kvc_oracle_f32_to_bf16(ru), hw = kvc_oracle_f32_to_bf16(rw);
    uint8_t* o = payload + OR_NOPE_DIM + 4 * j;
    o[0] = (uint8_t)(hu & 0xFF); o[1] = (uint8_t)(hu >> 8);
    o[2] = (uint8_t)(hw & 0xFF); o[3] = (uint8_t)(hw >> 8);
  }
}

/*
 * Quantise, rotate and scatter every output.  slot = kv_slot_mapping[b]
 * when slot_mapping_len == num_tokens (indexed by token), else
 * kv_slot_mapping[n]; a negative slot means "do not write".
 *   page = slot / 64, off = slot % 64,
 *   payload at kv[page, off * 576], scale at kv[page, 64 * 576 + off * 8].
 * The compressed position is pc = floor(p / C) * C.  Outputs with
 * valid[n] == 0 are skipped (valid may be NULL: all outputs valid).
 */
int kvc_oracle_quant_rope_scatter(
    const float* y, const uint8_t* valid, int64_t num_outputs,
    const int64_t* boundary_token_indices, const int64_t* positions,
    int64_t num_tokens, int32_t compress_ratio,
    const float* cos_sin_cache, int64_t num_positions,
    const int64_t* kv_slot_mapping, int64_t slot_mapping_len,
    uint8_t* kv_cache, int64_t num_kv_pages) {
  int status = OR_OK;
  const int by_token = (slot_mapping_len == num_tokens);
  for (int64_t n = 0; n < num_outputs; ++n) {
    if (valid && !valid[n]) continue;
    int64_t b = boundary_token_indices[n];
    if (b < 0 || b >= num_tokens) { status = OR_BAD_INDEX; continue; }
    int64_t p = positions[b];
    int64_t slot = by_token ? kv_slot_mapping[b] : kv_slot_mapping[n];
    if (slot < 0) continue;
    if (p < 0) { status = OR_BAD_INDEX; continue; }
    int64_t pc = (p / compress_ratio) * compress_ratio;
    int64_t page = slot / OR_SLOTS_PER_PAGE, off = slot % OR_SLOTS_PER_PAGE;
    if (pc >= num_positions || page >= num_kv_pages) { status = OR_BAD_INDEX; continue; }
    uint8_t payload[OR_TOKEN_STRIDE], scale[OR_SCALE_DIM];
    kvc_oracle_pack_slot(y + n * OR_HEAD_DIM, cos_sin_cache + pc * OR_ROPE_DIM,
                         payload, scale);
    uint8_t* pg = kv_cache + page * (int64_t)OR_PAGE_BYTES;
    memcpy(pg + off * OR_TOKEN_STRIDE, payload, OR_TOKEN_STRIDE);
    memcpy(pg + OR_SLOTS_PER_PAGE * OR_TOKEN_STRIDE + off * OR_SCALE_DIM, scale,
           OR_SCALE_DIM);
  }
  return status;
}

/*
 * The whole operator, in the argument order of c128_256_512_compress, on
 * host arrays.  The caller provides the intermediate buffers, which keeps
 * this file free of allocation: c and y are float [N, 512] (they receive the
 * compressed and the normalised vectors), valid is uint8 [N].  An output
 * whose window has an index outside its array is skipped; the other
 * outputs are still written and OR_BAD_INDEX is returned.
 */
int kvc_oracle_compress_ex(
    const void* state, int32_t state_dtype, int64_t state_block_stride,
    int64_t state_row_stride, int64_t num_state_blocks,
    const int32_t* token_to_req, const int64_t* positions, int64_t num_tokens,
    const int64_t* boundary_token_indices, int64_t num_outputs,
    const int32_t* block_table, int64_t num_reqs, int64_t max_blocks_per_req,
    int64_t bt_row_stride, int64_t bt_col_stride,
    const float* rms_norm_weight, const float* cos_sin_cache,
    int64_t num_positions, const int64_t* kv_slot_mapping,
    int64_t slot_mapping_len, uint8_t* kv_cache, int64_t num_kv_pages,
    int32_t block_size, int32_t compress_ratio, float rms_norm_eps,
    float* c, float* y, uint8_t* valid) {
  memset(c, 0, sizeof(float) * (size_t)(num_outputs * OR_HEAD_DIM));
  int st1 = kvc_oracle_window_reduce_ex(
      state, state_dtype, state_block_stride, state_row_stride, num_state_blocks, block_size,
      token_to_req, positions, num_tokens, boundary_token_indices, num_outputs, block_table,
      num_reqs, max_blocks_per_req, bt_row_stride, bt_col_stride, compress_ratio, c, valid);
  kvc_oracle_rmsnorm(c, rms_norm_weight, rms_norm_eps, num_outputs, y);
  int st2 = kvc_oracle_quant_rope_scatter(
      y, valid, num_outputs, boundary_token_indices, positions, num_tokens,
      compress_ratio, cos_sin_cache, num_positions, kv_slot_mapping,
      slot_mapping_len, kv_cache, num_kv_pages);
  return st1 != OR_OK ? st1 : st2;
}

/* kvc_oracle_compress_ex for a contiguous bf16 state [num_blocks, B, 1024]
 * and a row-major block_table [num_reqs, max_blocks_per_req]. */
int kvc_oracle_compress(
    const uint16_t* state, int64_t num_state_blocks,
    const int32_t* token_to_req, const int64_t* positions, int64_t num_tokens,
    const int64_t* boundary_token_indices, int64_t num_outputs,
    const int32_t* block_table, int64_t num_reqs, int64_t max_blocks_per_req,
    const float* rms_norm_weight, const float* cos_sin_cache,
    int64_t num_positions, const int64_t* kv_slot_mapping,
    int64_t slot_mapping_len, uint8_t* kv_cache, int64_t num_kv_pages,
    int32_t block_size, int32_t compress_ratio, float rms_norm_eps,
    float* c, float* y, uint8_t* valid) {
  const int64_t W = 2 * OR_HEAD_DIM;
  return kvc_oracle_compress_ex(
      state, 1, (int64_t)block_size * W, W, num_state_blocks, token_to_req, positions,
      num_tokens, boundary_token_indices, num_outputs, block_table, num_reqs,
      max_blocks_per_req, max_blocks_per_req, 1, rms_norm_weight, cos_sin_cache,
      num_positions, kv_slot_mapping, slot_mapping_len, kv_cache, num_kv_pages, block_size,
      compress_ratio, rms_norm_eps, c, y, valid);
}

/*
 * Read slots back ("Gather and Scatter" layout; the values the quantisation
 * equation of "How One Output Is Produced" encodes): for each slot m,
 *   out[m, d] = q_d * 2^(scale[d / 64] - 127)   for d < 448 (q_d the int8 code),
 *   out[m, d] = the stored bf16 RoPE value       for d >= 448,
 * written as float (out_bf16 == 0, `out` is float [M, 512]) or as bf16 bits
 * (out_bf16 != 0, `out` is uint16 [M, 512], float value rounded to nearest
 * even).  q * 2^e is evaluated exactly in double before the single rounding.
 * A negative slot yields zeros; a slot beyond the last page yields zeros and
 * OR_BAD_INDEX.
 */
int kvc_oracle_dequantize(const uint8_t* kv_cache, int64_t num_kv_pages,
                          const int64_t* slots, int64_t num_slots, void* out,
                          int32_t out_bf16) {
  int status = OR_OK;
  for (int64_t m = 0; m < num_slots; ++m) {
    float vals[OR_HEAD_DIM];
    for (int d = 0; d < OR_HEAD_DIM; ++d) vals[d] = 0.0f;
    int64_t slot = slots[m];
    int64_t page = slot / OR_SLOTS_PER_PAGE, off = slot % OR_SLOTS_PER_PAGE;
    if (slot >= 0 && page >= num_kv_pages) status = OR_BAD_INDEX;
    if (slot >= 0 && page < num_kv_pages) {
      const uint8_t* pg = kv_cache + page * (int64_t)OR_PAGE_BYTES;
      const uint8_t* payload = pg + off * OR_TOKEN_STRIDE;
      const uint8_t* scale = pg + OR_SLOTS_PER_PAGE * OR_TOKEN_STRIDE + off * OR_SCALE_DIM;
      for (int d = 0; d < OR_NOPE_DIM; ++d) {
        int q = (int)(int8_t)payload[d];
        int e = (int)scale[d / OR_GROUP] - 127;
        vals[d] = (float)ldexp((double)q, e);
      }
      for (int j = 0; j < OR_ROPE_DIM; ++j) {
        const uint8_t* b = payload + OR_NOPE_DIM + 2 * j;
        vals[OR_NOPE_DIM + j] = or_bf16_bits_to_float((uint16_t)(b[0] | (b[1] << 8)));
      }
    }
    for (int d = 0; d < OR_HEAD_DIM; ++d) {
      if (out_bf16)
        ((uint16_t*)out)[m * OR_HEAD_DIM + d] = kvc_oracle_f32_to_bf16(vals[d]);
      else
        ((float*)out)[m * OR_HEAD_DIM + d] = vals[d];
    }
  }
  return status;
}
