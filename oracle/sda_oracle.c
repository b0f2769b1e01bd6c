/*
 * sda_oracle.c -- plain, slow, fp64 CPU oracle for sparse sink decode attention
 * over a unified KV pool, for the ragged index builder in front of it, and for
 * the fused q/kv RMSNorm + RoPE + SWA ring store that fills the pool (end of
 * this file, with its own sources).
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this code.  It shares nothing with the
 * CUDA library: no header, helper, constant or table.  Status-bit values that
 * both sides report are fixed by the documented contract, not by shared code.
 *
 * Sources (all from the sglang pull-request summary page "为 AMD V4 内核添加
 * ATOM 来源注释" (sglang PR 28392), section "关键源码片段", the docstring of
 * paged_decode.py):
 *   - caller convention, unified_kv: one [total_pages, D] bf16 table, page
 *     size 1; slots [0, swa_pages) are SWA entries state_slot*win + ring,
 *     slots [swa_pages, ...) are compressed entries block_id*K_PER_BLOCK +
 *     slot_in_block (offset by swa_pages);
 *   - caller convention, kv_indices / kv_indptr: token t attends over
 *     kv_indices[kv_indptr[t] : kv_indptr[t+1]]; every entry is a valid slot;
 *     padded tokens get an empty slice;
 *   - caller convention, attn_sink: per-head learnable softmax denominator bias;
 *   - returns: out [N, H, D] in q's dtype (here returned in fp64);
 *   - numerics: online softmax in the log2 domain with the sink merged as a
 *     virtual key.  The log2 form is the same function as the natural-log form
 *     written below (2^(x*log2 e) = e^x), so the oracle uses the plain
 *     definition with libm exp() in double precision.
 *
 * Readings where the page is silent:
 *   - the sink is a natural-log logit that is NOT multiplied by softmax_scale;
 *     its value vector is zero (a "virtual key" that only adds e^sink to the
 *     denominator);
 *   - empty slice with a finite sink -> 0 (follows from the definition);
 *     empty slice with sink = -inf (0/0) -> 0;
 *   - sink = +inf -> 0 for every token;
 *   - duplicated slots each count once per occurrence.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* bf16 bit pattern -> double, exactly (bf16 is the top half of an fp32). */
static double bf16_bits_to_double(uint16_t b) {
  uint32_t u = ((uint32_t)b) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/*
 * FP8 E4M3 code -> double, exactly, from the format's definition (sign bit,
 * 4 exponent bits with bias 7, 3 mantissa bits; exponent field 0 encodes
 * subnormals m/8 * 2^-6; no infinities; S.1111.111 is NaN; largest finite
 * magnitude 1.75 * 2^8 = 448).  The pool format that stores one code per
 * element and one fp32 dequantisation scale per row is not on the pages (see
 * the header of oracle_sda_decode_fp8).
 */
double oracle_e4m3_to_double(uint8_t c) {
  const int sign = c >> 7, e = (c >> 3) & 15, m = c & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0) v = ldexp((double)m / 8.0, -6);
  else v = ldexp(1.0 + (double)m / 8.0, e - 7);
  return sign ? -v : v;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Return codes of the oracle entry points. */
#define ORACLE_OK 0
#define ORACLE_BAD_SHAPE 1
#define ORACLE_BAD_INDPTR 2
#define ORACLE_BAD_SLOT 3
#define ORACLE_NO_MEMORY 4

/*
 * Sparse decode attention with an attention sink, fp64.
 *
 * q           [N, H, D] bf16 bits
 * unified_kv  [total_pages, D] bf16 bits; row s is both key and value
 * kv_indices  [total_indices] int32
 * kv_indptr   [N + 1] int32, non-decreasing, within [0, total_indices]
 * attn_sink   [H] fp32 (may be +-inf)
 * softmax_scale  fp32, applied to the q.k dot product only
 * tokens      optional list of n_tokens token ids to evaluate (NULL = all N,
 *             in which case n_tokens must equal N)
 * out         [n_tokens, H, D] fp64, row i belongs to token tokens[i]
 *
 * For token t, head h, with S = kv_indices[kv_indptr[t] : kv_indptr[t+1]]:
 *   x_j = softmax_scale * sum_d q[t,h,d] * kv[S_j, d]
 *   M   = max(sink_h, max_j x_j)
 *   Z   = e^(sink_h - M) + sum_j e^(x_j - M)
 *   out = sum_j e^(x_j - M) * kv[S_j, :] / Z
 * The whole input is validated first; nothing out of range is ever read.
 */
/* Row value of the pool: bf16 bits, or an E4M3 code times the row's scale. */
typedef struct {
  const uint16_t* bf16;  /* [total_pages, D] bf16 bits, or NULL */
  const uint8_t* fp8;    /* [total_pages, D] E4M3 codes, or NULL */
  const float* scale;    /* [total_pages] fp32 dequantisation scale (fp8 only) */
} Pool;

static double pool_value(const Pool* p, int64_t s, int d, int D) {
  if (p->bf16) return bf16_bits_to_double(p->bf16[(size_t)s * D + d]);
  return oracle_e4m3_to_double(p->fp8[(size_t)s * D + d]) * (double)p->scale[s];
}

static int decode_core(const uint16_t* q, const Pool* pool, int64_t total_pages,
                       const int32_t* kv_indices, int64_t total_indices,
                       const int32_t* kv_indptr, const float* attn_sink, float softmax_scale,
                       int N, int H, int D, const int32_t* tokens, int n_tokens, double* out) {
  if (N < 0 || H <= 0 || D <= 0 || total_pages <= 0 || total_indices < 0 || n_tokens < 0)
    return ORACLE_BAD_SHAPE;
  if (tokens == NULL && n_tokens != N) return ORACLE_BAD_SHAPE;
  for (int t = 0; t < N; ++t) {
    if (kv_indptr[t] < 0 || kv_indptr[t + 1] < kv_indptr[t] || kv_indptr[t + 1] > total_indices)
      return ORACLE_BAD_INDPTR;
  }
  for (int i = 0; i < n_tokens; ++i) {
    int t = tokens ? tokens[i] : i;
    if (t < 0 || t >= N) return ORACLE_BAD_SHAPE;
    for (int32_t e = kv_indptr[t]; e < kv_indptr[t + 1]; ++e)
      if (kv_indices[e] < 0 || (int64_t)kv_indices[e] >= total_pages) return ORACLE_BAD_SLOT;
  }
  const double scale = (double)softmax_scale;
  int failed = 0;

#pragma omp parallel for collapse(2) schedule(dynamic, 1)
  for (int i = 0; i < n_tokens; ++i) {
    for (int h = 0; h < H; ++h) {
      const int t = tokens ? tokens[i] : i;
      const int32_t begin = kv_indptr[t];
      const int32_t len = kv_indptr[t + 1] - begin;
      const double sink = (double)attn_sink[h];
      double* o = out + ((size_t)i * H + h) * D;
      for (int d = 0; d < D; ++d) o[d] = 0.0;
      if (sink == INFINITY) continue;        /* reading: an infinite sink absorbs all mass */
      double* x = (double*)malloc(sizeof(double) * (len > 0 ? len : 1));
      if (!x) {
#pragma omp atomic write
        failed = 1;
        continue;
      }
      const uint16_t* qh = q + ((size_t)t * H + h) * D;
      /* logits */
      double M = sink;
      for (int32_t j = 0; j < len; ++j) {
        const int64_t s = kv_indices[begin + j];
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += bf16_bits_to_double(qh[d]) * pool_value(pool, s, d, D);
        x[j] = scale * dot;
        if (x[j] > M) M = x[j];
      }
      if (M == -INFINITY) {                  /* empty slice and sink = -inf: 0/0, reading -> 0 */
        free(x);
        continue;
      }
      /* denominator: the sink's term plus one term per listed slot */
      double Z = exp(sink - M);
      for (int32_t j = 0; j < len; ++j) Z += exp(x[j] - M);
      /* numerator: probability-weighted sum of the value rows (the same rows) */
      for (int32_t j = 0; j < len; ++j) {
        const double w = exp(x[j] - M) / Z;
        const int64_t s = kv_indices[begin + j];
        for (int d = 0; d < D; ++d) o[d] += w * pool_value(pool, s, d, D);
      }
      free(x);
    }
  }
  return failed ? ORACLE_NO_MEMORY : ORACLE_OK;
}

int oracle_sda_decode(const uint16_t* q, const uint16_t* unified_kv, int64_t total_pages,
                      const int32_t* kv_indices, int64_t total_indices,
                      const int32_t* kv_indptr, const float* attn_sink, float softmax_scale,
                      int N, int H, int D, const int32_t* tokens, int n_tokens, double* out) {
  const Pool pool = {unified_kv, NULL, NULL};
  return decode_core(q, &pool, total_pages, kv_indices, total_indices, kv_indptr, attn_sink,
                     softmax_scale, N, H, D, tokens, n_tokens, out);
}

/*
 * The same attention over a pool stored in FP8: row s, element d has the value
 * e4m3(kv_fp8[s, d]) * kv_scale[s] (exact in double).  Everything else --
 * logits, sink, softmax, weighted sum -- is oracle_sda_decode's definition.
 * The pages keep unified_kv in bf16; this format (one E4M3 code per element,
 * one fp32 scale per row) is a reading, for the FP8-pool variant of the path.
 */
int oracle_sda_decode_fp8(const uint16_t* q, const uint8_t* kv_fp8, const float* kv_scale,
                          int64_t total_pages, const int32_t* kv_indices, int64_t total_indices,
                          const int32_t* kv_indptr, const float* attn_sink, float softmax_scale,
                          int N, int H, int D, const int32_t* tokens, int n_tokens, double* out) {
  const Pool pool = {NULL, kv_fp8, kv_scale};
  return decode_core(q, &pool, total_pages, kv_indices, total_indices, kv_indptr, attn_sink,
                     softmax_scale, N, H, D, tokens, n_tokens, out);
}

/*
 * Index builder: packs, per token, its SWA ring slots and its compressed-cache
 * slots into one ragged list (the "index scatter" the same page names
 * write_v4_paged_decode_indices; its inputs are not on the page -- reading:
 * the plainest inputs that produce the two slot formulas of the docstring).
 *
 * state_slot [N]        < 0 marks a padded token (empty slice, not an error)
 * swa_len    [N]        number of valid ring entries, 0..win
 * swa_head   [N]        ring position of the newest entry, 0..win-1
 * comp_indptr [N + 1]   token t's compressed entries are
 * comp_block / comp_slot  [comp_indptr[t], comp_indptr[t+1])
 * Emission order (reading): SWA entries oldest -> newest, ring position
 * (swa_head - swa_len + 1 + j) mod win, as slot state_slot*win + ring; then
 * compressed entries in input order as swa_pages + block*k_per_block + slot.
 * Tokens with any bad field get an empty slice and raise a status bit:
 *   1  swa_len outside [0, win]
 *   2  swa_head outside [0, win) while swa_len > 0
 *   4  comp_indptr decreasing, or outside [0, comp_total]
 *   8  a compressed entry with block < 0 or slot outside [0, k_per_block)
 *   16 an emitted slot outside its region (SWA slot >= swa_pages, or
 *      compressed slot >= total_pages)
 *   32 the packed list would exceed `capacity`; then every slice is empty
 * kv_indptr[0] = 0 and kv_indptr is the prefix sum of the emitted lengths.
 */
int oracle_build_indices(const int32_t* state_slot, const int32_t* swa_len, const int32_t* swa_head,
                         const int32_t* comp_indptr, const int32_t* comp_block,
                         const int32_t* comp_slot, int64_t comp_total, int N, int win,
                         int k_per_block, int64_t swa_pages, int64_t total_pages,
                         int32_t* kv_indices, int64_t capacity, int32_t* kv_indptr,
                         int32_t* status) {
  if (N < 0 || win <= 0 || k_per_block <= 0 || swa_pages < 0 || total_pages <= 0 ||
      swa_pages > total_pages || capacity < 0 || comp_total < 0)
    return ORACLE_BAD_SHAPE;
  int32_t flags = 0;
  int64_t* len = (int64_t*)calloc((size_t)(N > 0 ? N : 1), sizeof(int64_t));
  if (!len) return ORACLE_NO_MEMORY;
  for (int t = 0; t < N; ++t) {
    if (state_slot[t] < 0) continue;          /* padded token */
    int32_t bad = 0;
    const int32_t n_swa = swa_len[t];
    if (n_swa < 0 || n_swa > win) bad |= 1;
    else if (n_swa > 0 && (swa_head[t] < 0 || swa_head[t] >= win)) bad |= 2;
    else if (n_swa > 0 && (int64_t)state_slot[t] * win + win > swa_pages) bad |= 16;
    const int32_t c0 = comp_indptr[t], c1 = comp_indptr[t + 1];
    if (c0 < 0 || c1 < c0 || (int64_t)c1 > comp_total) bad |= 4;
    else {
      for (int32_t e = c0; e < c1; ++e) {
        if (comp_block[e] < 0 || comp_slot[e] < 0 || comp_slot[e] >= k_per_block) { bad |= 8; continue; }
        const int64_t s = swa_pages + (int64_t)comp_block[e] * k_per_block + comp_slot[e];
        if (s >= total_pages) bad |= 16;
      }
    }
    flags |= bad;
    if (!bad) len[t] = (int64_t)n_swa + (c1 - c0);
  }
  int64_t total = 0;
  for (int t = 0; t < N; ++t) total += len[t];
  if (total > capacity) {
    flags |= 32;
    for (int t = 0; t < N; ++t) len[t] = 0;
  }
  kv_indptr[0] = 0;
  int64_t pos = 0;
  for (int t = 0; t < N; ++t) {
    if (len[t] > 0) {
      const int32_t n_swa = swa_len[t];
      for (int32_t j = 0; j < n_swa; ++j) {
        const int32_t ring = (int32_t)((((int64_t)swa_head[t] - n_swa + 1 + j) % win + win) % win);
        kv_indices[pos++] = (int32_t)((int64_t)state_slot[t] * win + ring);
      }
      for (int32_t e = comp_indptr[t]; e < comp_indptr[t + 1]; ++e)
        kv_indices[pos++] = (int32_t)(swa_pages + (int64_t)comp_block[e] * k_per_block + comp_slot[e]);
    }
    kv_indptr[t + 1] = (int32_t)pos;
  }
  free(len);
  *status = flags;
  return ORACLE_OK;
}

/*
 * Index validation (the docstring's requirement that every entry is a valid
 * slot and that kv_indptr is a true prefix sum).  status[0] bits:
 *   1 kv_indptr decreasing somewhere;  2 kv_indptr outside [0, total_indices];
 *   4 some entry of kv_indices outside [0, total_pages).
 * status[1] = number of entries of kv_indices[0 : total_indices] out of range.
 */
int oracle_validate_indices(const int32_t* kv_indices, int64_t total_indices,
                            const int32_t* kv_indptr, int N, int64_t total_pages,
                            int32_t* status) {
  if (N < 0 || total_indices < 0 || total_pages <= 0) return ORACLE_BAD_SHAPE;
  int32_t flags = 0;
  for (int t = 0; t <= N; ++t) {
    if (kv_indptr[t] < 0 || (int64_t)kv_indptr[t] > total_indices) flags |= 2;
    if (t < N && kv_indptr[t + 1] < kv_indptr[t]) flags |= 1;
  }
  int64_t n_bad = 0;
  for (int64_t e = 0; e < total_indices; ++e)
    if (kv_indices[e] < 0 || (int64_t)kv_indices[e] >= total_pages) ++n_bad;
  if (n_bad) flags |= 4;
  status[0] = flags;
  status[1] = (int32_t)(n_bad > INT32_MAX ? INT32_MAX : n_bad);
  return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/*
 * Fused q / kv RMSNorm + RoPE + SWA ring store, fp64.
 *
 * Source: the sglang PR 25898 summary page ("修复 DSV4 在 AMD GPU 上的运行时
 * 崩溃与 JIT 不兼容"), section "关键文件": fused_qk_norm_rope_store.py is one
 * kernel that does the per-head RMSNorm of Q, the RMSNorm of the new KV, RoPE,
 * FP8 quantisation and the paged SWA store; section "关键符号" names its parts
 * (_batched_rmsnorm, _gptj_rotate, _batched_rope, fused_qk_norm_rope_swa_store);
 * section "实现拆解" item 2 names the cos_cache / sin_cache it reads.  The SWA
 * slot of an entry is state_slot * win + ring (the paged_decode.py docstring
 * on the PR 28392 page).
 *
 * Readings where the pages are silent:
 *   - RMSNorm of a row x of length D with weight w:
 *       y_d = x_d / sqrt(mean_d x_d^2 + eps) * w_d      (one weight [D] per
 *     tensor, shared by all heads of q);
 *   - RoPE acts on the last R dims of each row; "GPT-J" rotation pairs
 *     adjacent elements: for i < R/2, d = D - R + 2i,
 *       (y_d, y_{d+1}) <- (y_d c - y_{d+1} s,  y_{d+1} c + y_d s),
 *     c = cos_cache[pos, i], s = sin_cache[pos, i] (caches [max_pos, R/2]);
 *   - norm and rotation happen in full precision and the result is rounded
 *     once: to bf16 (nearest even) for q and for a bf16 pool, or quantised for
 *     an FP8 pool;
 *   - the new KV row goes to ring position pos mod win of its state:
 *     slot = state_slot * win + pos mod win, which must be < swa_pages;
 *   - state_slot < 0 marks a padded token: its q row is 0 and nothing is
 *     stored; a real token whose position is outside [0, max_pos) is treated
 *     the same way and raises status bit 1; a slot outside [0, swa_pages)
 *     raises bit 2 and is not stored (q is still produced).
 *
 * q [N,H,D], kv [N,D], q_norm_w [D], kv_norm_w [D]: bf16 bits.
 * Outputs: q_val [N,H,D] and kv_val [N,D] the exact (unrounded) results,
 * slot [N] the pool row written (-1 if none), *status the bits above.
 */
int oracle_qk_norm_rope_store(const uint16_t* q, const uint16_t* kv, const uint16_t* q_norm_w,
                              const uint16_t* kv_norm_w, const float* cos_cache,
                              const float* sin_cache, int max_pos, const int32_t* positions,
                              const int32_t* state_slot, int N, int H, int D, int R, float eps,
                              int win, int64_t swa_pages, double* q_val, double* kv_val,
                              int64_t* slot, int32_t* status) {
  if (N < 0 || H <= 0 || D <= 0 || R < 0 || R > D || (R & 1) || win <= 0 || swa_pages < 0 ||
      max_pos < 0)
    return ORACLE_BAD_SHAPE;
  int32_t flags = 0;
  for (int t = 0; t < N; ++t) {
    const int pos = positions[t];
    int live = state_slot[t] >= 0;
    if (live && (pos < 0 || pos >= max_pos)) {
      flags |= 1;
      live = 0;
    }
    slot[t] = -1;
    for (int r = 0; r <= H; ++r) {            /* rows 0..H-1: q heads; row H: the KV row */
      const uint16_t* x = r < H ? q + ((size_t)t * H + r) * D : kv + (size_t)t * D;
      const uint16_t* w = r < H ? q_norm_w : kv_norm_w;
      double* y = r < H ? q_val + ((size_t)t * H + r) * D : kv_val + (size_t)t * D;
      if (!live) {
        for (int d = 0; d < D; ++d) y[d] = 0.0;
        continue;
      }
      double ss = 0.0;
      for (int d = 0; d < D; ++d) ss += bf16_bits_to_double(x[d]) * bf16_bits_to_double(x[d]);
      const double inv_rms = 1.0 / sqrt(ss / D + (double)eps);
      for (int d = 0; d < D; ++d)
        y[d] = bf16_bits_to_double(x[d]) * inv_rms * bf16_bits_to_double(w[d]);
      for (int i = 0; i < R / 2; ++i) {
        const int d = D - R + 2 * i;
        const double c = cos_cache[(size_t)pos * (R / 2) + i];
        const double s = sin_cache[(size_t)pos * (R / 2) + i];
        const double a = y[d], b = y[d + 1];
        y[d] = a * c - b * s;
        y[d + 1] = b * c + a * s;
      }
    }
    if (live) {
      const int64_t sl = (int64_t)state_slot[t] * win + pos % win;
      if (sl >= swa_pages) flags |= 2;
      else slot[t] = sl;
    }
  }
  *status = flags;
  return ORACLE_OK;
}

/* Round to the nearest bf16, ties to even, from the format's definition
 * (8 significant bits, exponent range of fp32): returns the bit pattern. */
uint16_t oracle_bf16_rne(double v) {
  if (isnan(v)) return 0x7FC0;
  const uint16_t sign = signbit(v) ? 0x8000 : 0;
  const double a = fabs(v);
  if (a == 0.0) return sign;
  int e2;
  frexp(a, &e2);                      /* a = m * 2^e2, m in [0.5, 1) */
  int E = e2 - 1;                     /* floor(log2 a) */
  if (E < -126) E = -126;             /* subnormal range: fixed quantum 2^-133 */
  const double quantum = ldexp(1.0, E - 7);
  const double r = rint(a / quantum) * quantum;   /* rint: nearest, ties to even */
  if (r >= ldexp(1.0, 128)) return sign | 0x7F80;  /* rounds past the largest finite */
  const float f = (float)r;           /* exact: r has at most 8 significant bits */
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  return (uint16_t)(sign | (u >> 16));
}

/* Round to the nearest FP8 E4M3 value, ties to even, saturating at +-448
 * (format: bias 7, 3 mantissa bits, subnormal quantum 2^-9): returns the code. */
uint8_t oracle_e4m3_rne(double v) {
  if (isnan(v)) return 0x7F;
  const uint8_t sign = signbit(v) ? 0x80 : 0;
  const double a = fabs(v);
  if (a == 0.0) return sign;
  int e2;
  frexp(a, &e2);
  int E = e2 - 1;
  if (E < -6) E = -6;                 /* subnormals share the quantum of binade -6 */
  const double quantum = ldexp(1.0, E - 3);
  double r = rint(a / quantum) * quantum;
  if (r > 448.0) r = 448.0;
  if (r < ldexp(1.0, -6)) return (uint8_t)(sign | (uint8_t)(r / ldexp(1.0, -9)));  /* 0..7 */
  frexp(r, &e2);
  const int Er = e2 - 1;              /* 2^Er <= r < 2^(Er+1) */
  const int mant = (int)(r / ldexp(1.0, Er) * 8.0) - 8;
  return (uint8_t)(sign | ((Er + 7) << 3) | mant);
}

/* Power-of-two row scale of the FP8 store: 2^e with e the smallest integer
 * such that 448 * 2^e >= amax (so every element divided by it fits in E4M3),
 * e >= -126; amax = 0 gives 1.  Returns e. */
int oracle_fp8_scale_exponent(double amax) {
  if (!(amax > 0.0)) return 0;
  int e = (int)ceil(log2(amax / 448.0));
  while (ldexp(448.0, e) < amax) ++e;
  while (ldexp(448.0, e - 1) >= amax) --e;
  return e < -126 ? -126 : e;
}

/* bf16 bits of n values, each rounded to nearest even. */
void oracle_bf16_rne_array(const double* v, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_bf16_rne(v[i]);
}

/* FP8 quantisation of `rows` rows of D values (the FP8 pool's format: one
 * E4M3 code per element and one fp32 scale per row, element = code * scale):
 * scale = 2^oracle_fp8_scale_exponent(max_d |y_d|), code = E4M3 of y / scale
 * rounded to nearest even.  Dividing by a power of two is exact. */
void oracle_fp8_quantise_rows(const double* y, int64_t rows, int D, uint8_t* codes, float* scale) {
  for (int64_t r = 0; r < rows; ++r) {
    const double* yr = y + (size_t)r * D;
    double amax = 0.0;
    for (int d = 0; d < D; ++d)
      if (fabs(yr[d]) > amax) amax = fabs(yr[d]);
    const int e = oracle_fp8_scale_exponent(amax);
    scale[r] = (float)ldexp(1.0, e);
    for (int d = 0; d < D; ++d) codes[(size_t)r * D + d] = oracle_e4m3_rne(ldexp(yr[d], -e));
  }
}

/* E4M3 codes of n values, each rounded to nearest even (saturating). */
void oracle_e4m3_rne_array(const double* v, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_rne(v[i]);
}

/* ------------------------------------------------------------------------ */
/*
 * Top-k selection of compressed-cache entries -> slot lists (the input of the
 * index builder), fp32 scores.
 *
 * Source: the sglang attention tag page, entry "DSV4.1 新增索引器内核，重做
 * Top-K v2 分派": the selection pads with NaN rather than a very small value so
 * that a legitimate -inf score stays selectable, and a separate page-table
 * transform ("PageTransform") turns selected positions into cache locations.
 * The positions map to pool entries by the compressed-slot formula of the
 * paged_decode.py docstring (PR 28392 page): block_id * K_PER_BLOCK +
 * slot_in_block, the block being the token's block_table entry.
 *
 * Readings where the page is silent:
 *   - token t's candidates are positions p in [0, n_t), n_t = lengths[t], with
 *     scores[t * score_stride + p]; positions at or past n_t are padding and
 *     are never read or selected; lengths outside [0, score_stride] count as
 *     0 and raise status bit 1;
 *   - ranking: larger score first; -0 equals +0; a NaN inside [0, n_t) ranks
 *     below -inf (as padding does) but is still a candidate (status bit 8);
 *     equal scores are taken in increasing position;
 *   - the token keeps min(k, n_t) positions, emitted in increasing position;
 *   - position p -> (block_table[t * bt_stride + p / k_per_block],
 *     p % k_per_block); a negative block id raises bit 4 and is emitted as is
 *     (the index builder rejects it);
 *   - comp_indptr[0] = 0, comp_indptr[t + 1] = comp_indptr[t] + min(k, n_t).
 */
typedef struct {
  uint32_t key;  /* order-preserving image of the score: larger score, larger key */
  int32_t pos;
} KeyPos;

static uint32_t score_key(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  if (isnan(f)) return 0;                         /* below every number, -inf included */
  if (u == 0x80000000u) u = 0;                    /* -0 ranks as +0 */
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

static int keypos_order(const void* a, const void* b) {
  const KeyPos* x = (const KeyPos*)a;
  const KeyPos* y = (const KeyPos*)b;
  if (x->key != y->key) return x->key > y->key ? -1 : 1;  /* larger score first */
  return (x->pos > y->pos) - (x->pos < y->pos);            /* then smaller position */
}

static int int_order(const void* a, const void* b) {
  const int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;
  return (x > y) - (x < y);
}

int oracle_topk_slots(const float* scores, int64_t score_stride, const int32_t* lengths,
                      const int32_t* block_table, int64_t bt_stride, int N, int k,
                      int k_per_block, int32_t* comp_indptr, int32_t* comp_block,
                      int32_t* comp_slot, int32_t* status) {
  if (N < 0 || k < 0 || k_per_block <= 0 || score_stride < 0 || bt_stride < 0 ||
      bt_stride * (int64_t)k_per_block < score_stride)
    return ORACLE_BAD_SHAPE;
  int32_t flags = 0;
  comp_indptr[0] = 0;
  for (int t = 0; t < N; ++t) {
    int64_t n = lengths[t];
    if (n < 0 || n > score_stride) {
      flags |= 1;
      n = 0;
    }
    const int64_t kk = n < k ? n : k;
    comp_indptr[t + 1] = (int32_t)(comp_indptr[t] + kk);
    if (kk == 0) continue;
    KeyPos* c = (KeyPos*)malloc(sizeof(KeyPos) * (size_t)n);
    int32_t* sel = (int32_t*)malloc(sizeof(int32_t) * (size_t)kk);
    if (!c || !sel) {
      free(c);
      free(sel);
      return ORACLE_NO_MEMORY;
    }
    for (int64_t p = 0; p < n; ++p) {
      const float f = scores[(size_t)t * score_stride + p];
      if (isnan(f)) flags |= 8;
      c[p].key = score_key(f);
      c[p].pos = (int32_t)p;
    }
    qsort(c, (size_t)n, sizeof(KeyPos), keypos_order);
    for (int64_t i = 0; i < kk; ++i) sel[i] = c[i].pos;
    qsort(sel, (size_t)kk, sizeof(int32_t), int_order);
    for (int64_t i = 0; i < kk; ++i) {
      const int32_t p = sel[i];
      const int32_t blk = block_table[(size_t)t * bt_stride + p / k_per_block];
      if (blk < 0) flags |= 4;
      comp_block[comp_indptr[t] + i] = blk;
      comp_slot[comp_indptr[t] + i] = p % k_per_block;
    }
    free(c);
    free(sel);
  }
  *status = flags;
  return ORACLE_OK;
}
