/*
 * paged_attn_oracle.c -- plain fp64 CPU oracle for paged grouped-query attention.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the correctness reference for the CUDA library
 * in paged_gqa_attention_hd512_gb300/.  It shares no code with it: it is only compiled
 * and called by tests/, by __graft_entry__.smoke() and by bench.py's cpu_baseline leg.
 * It is deliberately slow and written for reading: no tiling, no split, no fusion.
 *
 * What it computes (the pages never print the formula; this is the standard softmax
 * attention they name):
 *   For sequence b, query row i (0 <= i < qo_len) and query head h, with kv head
 *   kvh = h / (Hq / Hkv) and query position pos = kv_len - qo_len + i:
 *     key j (0 <= j < kv_len) is allowed when (causal ? j <= pos : 1) and
 *       (window_left >= 0 ? j >= pos - window_left : 1);
 *     s_j = sm_scale * sum_d q[d] * K^[j][d]          (fp64, q read exactly from bf16)
 *     m = max_j s_j,  l = sum_j exp(s_j - m),
 *     o = sum_j exp(s_j - m) * V^[j] / l,   lse = m + ln(l)   (natural log)
 *   With no allowed key: o = 0, lse = -inf.
 *   K^ and V^ are the dequantised cache values: bf16 exactly; FP8 e4m3 code * per-tensor
 *   scale; NVFP4 e2m1 nibble * e4m3 block scale * fp32 global scale.
 *
 * Sources (page title, section):
 *  - "[None][feat] Run Gemma4 head_dim 512 attention on Triton" (TensorRT-LLM PR #17772),
 *    Approach: the combined HND cache [num_pages, 2, num_kv_heads, page_size, head_dim],
 *    read through kv_indptr / kv_indices / kv_last_page_len; prefill is causal when no
 *    custom mask is given; FP8 KV is cast on load.  Test Coverage: partial and
 *    exact-multiple last pages, GQA ratios with non-power-of-two groups, sliding windows,
 *    split-K.
 *  - "feat(attention): asymmetric VO-split NVFP4 paged prefill (qk=512/vo=256) for
 *    Gemma-4 on SM120/121" (FlashInfer PR #3684), Summary: head_dim_qk = 512 with
 *    head_dim_vo = 256, independent K and V strides, a contiguous [all-data | all-SF]
 *    scale layout; NVFP4 split-KV correctness: packed e2m1 with one FP8 scale per 16
 *    consecutive head-dim elements of one token; commit "support-or-reject-explicitly":
 *    the reference consumes the exact same quantised bytes as the kernel.
 *
 * Readings taken where the pages are silent:
 *  - lse uses the natural log of the scaled scores.
 *  - window: a query at pos sees keys [pos - window_left, pos]; -1 means no window.
 *  - causal alignment is bottom-right: pos = kv_len - qo_len + i.
 *  - q head h reads kv head h / (Hq / Hkv).
 *  - with d_qk != d_vo, page p holds the K block [Hkv][page_size][d_qk] followed by the
 *    V block [Hkv][page_size][d_vo]; with d_qk == d_vo this is the pages' layout.
 *  - NVFP4: element 2i is the low nibble of byte i; the scale pool holds, per page,
 *    [Hkv][page_size][d_qk/16] K scales then [Hkv][page_size][d_vo/16] V scales.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { KV_BF16 = 0, KV_FP8_E4M3 = 1, KV_NVFP4 = 2 };

/* ---------------------------------------------------------------- number formats */

/* bf16 is the upper half of an IEEE binary32. */
double oracle_bf16_value(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* e4m3 "fn": 1 sign, 4 exponent (bias 7), 3 mantissa bits; exponent 15 with mantissa 7
 * is NaN, there is no infinity; exponent 0 is subnormal (m/8 * 2^-6). */
double oracle_e4m3_value(uint8_t code) {
  int s = code >> 7, e = (code >> 3) & 15, m = code & 7;
  double mag;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    mag = ldexp((double)m / 8.0, -6);
  else
    mag = ldexp(1.0 + (double)m / 8.0, e - 7);
  return s ? -mag : mag;
}

/* e2m1: 1 sign, 2 exponent (bias 1), 1 mantissa bit; exponent 0 is subnormal (m * 0.5). */
double oracle_e2m1_value(uint8_t nibble) {
  int s = (nibble >> 3) & 1, e = (nibble >> 1) & 3, m = nibble & 1;
  double mag;
  if (e == 0)
    mag = 0.5 * (double)m;
  else
    mag = ldexp(1.0 + 0.5 * (double)m, e - 1);
  return s ? -mag : mag;
}

/* ---------------------------------------------------------------- cache addressing */

typedef struct {
  const uint8_t* kv_cache;
  const int32_t* kv_indptr;
  const int32_t* kv_indices;
  const int32_t* kv_last_page_len;
  const uint8_t* sf;
  int Hkv, d_qk, d_vo, page_size, kv_dtype;
  double k_scale, v_scale;
} kv_view;

static int64_t seq_kv_len(const kv_view* kv, int b) {
  int64_t npages = kv->kv_indptr[b + 1] - kv->kv_indptr[b];
  if (npages <= 0) return 0;
  return (npages - 1) * (int64_t)kv->page_size + kv->kv_last_page_len[b];
}

/* Elements per page: K block then V block. */
static int64_t page_elems(const kv_view* kv) {
  return (int64_t)kv->Hkv * kv->page_size * (kv->d_qk + kv->d_vo);
}

/* One dequantised element of token t (logical, within sequence b) of kv head kvh.
 * is_v selects the V block.  Token t lives in page kv_indices[kv_indptr[b] + t/ps],
 * slot t % ps. */
static double kv_element(const kv_view* kv, int b, int kvh, int64_t t, int is_v, int d) {
  int ps = kv->page_size;
  int64_t page = kv->kv_indices[kv->kv_indptr[b] + t / ps];
  int64_t slot = t % ps;
  int dim = is_v ? kv->d_vo : kv->d_qk;
  int64_t block_base = is_v ? (int64_t)kv->Hkv * ps * kv->d_qk : 0;
  int64_t elem = page * page_elems(kv) + block_base + ((int64_t)kvh * ps + slot) * dim + d;
  if (kv->kv_dtype == KV_BF16) {
    uint16_t bits;
    memcpy(&bits, kv->kv_cache + elem * 2, 2);
    return oracle_bf16_value(bits);
  }
  if (kv->kv_dtype == KV_FP8_E4M3) {
    double scale = is_v ? kv->v_scale : kv->k_scale;
    return oracle_e4m3_value(kv->kv_cache[elem]) * scale;
  }
  /* NVFP4 */
  {
    uint8_t byte = kv->kv_cache[elem / 2];
    uint8_t nib = (elem % 2 == 0) ? (byte & 15) : (byte >> 4);
    int64_t sf_index = elem / 16; /* 16 consecutive head-dim elements of one token */
    double block = oracle_e4m3_value(kv->sf[sf_index]);
    double global = is_v ? kv->v_scale : kv->k_scale;
    return oracle_e2m1_value(nib) * block * global;
  }
}

/* ---------------------------------------------------------------- attention rows */

static int find_seq(const int32_t* qo_indptr, int batch, int64_t tok) {
  int lo = 0, hi = batch - 1;
  while (lo < hi) { /* last b with qo_indptr[b] <= tok */
    int mid = (lo + hi + 1) / 2;
    if (qo_indptr[mid] <= tok) lo = mid; else hi = mid - 1;
  }
  return lo;
}

/*
 * oracle_rows: attention output for a list of (query token, query head) rows.
 *
 *  q            bf16 bits [total_q][Hq][d_qk]
 *  qo_indptr    [batch+1] query rows of each sequence (decode: 0,1,...,batch)
 *  kv_cache     cache bytes (layout above); kv_indptr [batch+1]; kv_indices [nnz];
 *  kv_last_page_len [batch]; sf NVFP4 scale pool or NULL
 *  k_scale/v_scale  FP8 per-tensor scales or NVFP4 global scales (ignored for bf16)
 *  row_tok[n], row_head[n]   which rows to compute
 *  key_lo/key_hi  optional per-row restriction of keys to [key_lo, key_hi) (NULL = all);
 *                 used to form split-K partials
 *  mask, mask_indptr  optional custom mask (NULL = none): for sequence b, query row i
 *                 (0 <= i < qo_len) may attend key j only when bit mask_indptr[b] * 8 +
 *                 i * kv_len + j of the byte array `mask` is 1 (bit k of a byte is its
 *                 2^k bit); it narrows the causal / window rules, it does not replace them.
 *                 ("[None][feat] Run Gemma4 head_dim 512 attention on Triton", Approach:
 *                 prefill is causal when no custom mask is given.)
 *  out [n][d_vo], lse [n]    fp64 results
 * Returns 0, or -1 on a malformed argument.
 */
int oracle_rows(const uint16_t* q, const int32_t* qo_indptr, const uint8_t* kv_cache,
                const int32_t* kv_indptr, const int32_t* kv_indices,
                const int32_t* kv_last_page_len, const uint8_t* sf, int batch, int Hq, int Hkv,
                int d_qk, int d_vo, int page_size, int kv_dtype, double k_scale, double v_scale,
                double sm_scale, int window_left, int causal, int64_t n_rows,
                const int64_t* row_tok, const int32_t* row_head, const int64_t* key_lo,
                const int64_t* key_hi, const uint8_t* mask, const int64_t* mask_indptr,
                double* out, double* lse, int n_threads) {
  if (batch <= 0 || Hkv <= 0 || Hq % Hkv != 0 || page_size <= 0 || d_qk <= 0 || d_vo <= 0)
    return -1;
  if (kv_dtype == KV_NVFP4 && (sf == NULL || d_qk % 16 || d_vo % 16)) return -1;
  kv_view kv = {kv_cache, kv_indptr, kv_indices, kv_last_page_len, sf,
                Hkv, d_qk, d_vo, page_size, kv_dtype, k_scale, v_scale};
  int group = Hq / Hkv;
  int64_t n_units = (int64_t)batch * Hkv;

  /* group the requested rows by (sequence, kv head) so each unit gathers its keys once */
  int64_t* unit_of = (int64_t*)malloc(sizeof(int64_t) * (n_rows ? n_rows : 1));
  int64_t* unit_start = (int64_t*)calloc(n_units + 1, sizeof(int64_t));
  int64_t* order = (int64_t*)malloc(sizeof(int64_t) * (n_rows ? n_rows : 1));
  int64_t* fill = (int64_t*)calloc(n_units + 1, sizeof(int64_t));
  for (int64_t r = 0; r < n_rows; ++r) {
    int b = find_seq(qo_indptr, batch, row_tok[r]);
    unit_of[r] = (int64_t)b * Hkv + row_head[r] / group;
    unit_start[unit_of[r] + 1]++;
  }
  for (int64_t u = 0; u < n_units; ++u) unit_start[u + 1] += unit_start[u];
  for (int64_t r = 0; r < n_rows; ++r) order[unit_start[unit_of[r]] + fill[unit_of[r]]++] = r;

#ifdef _OPENMP
  if (n_threads > 0) omp_set_num_threads(n_threads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
  for (int64_t u = 0; u < n_units; ++u) {
    if (unit_start[u] == unit_start[u + 1]) continue;
    int b = (int)(u / Hkv), kvh = (int)(u % Hkv);
    int64_t kv_len = seq_kv_len(&kv, b);
    int64_t qo_len = qo_indptr[b + 1] - qo_indptr[b];
    /* gather the dequantised keys and values of this (sequence, kv head) */
    double* K = (double*)malloc(sizeof(double) * (kv_len ? kv_len : 1) * d_qk);
    double* V = (double*)malloc(sizeof(double) * (kv_len ? kv_len : 1) * d_vo);
    double* s = (double*)malloc(sizeof(double) * (kv_len ? kv_len : 1));
    for (int64_t j = 0; j < kv_len; ++j) {
      for (int d = 0; d < d_qk; ++d) K[j * d_qk + d] = kv_element(&kv, b, kvh, j, 0, d);
      for (int d = 0; d < d_vo; ++d) V[j * d_vo + d] = kv_element(&kv, b, kvh, j, 1, d);
    }
    for (int64_t k = unit_start[u]; k < unit_start[u + 1]; ++k) {
      int64_t r = order[k];
      int64_t i = row_tok[r] - qo_indptr[b];
      int h = row_head[r];
      int64_t pos = kv_len - qo_len + i;
      int64_t lo = key_lo ? key_lo[r] : 0, hi = key_hi ? key_hi[r] : kv_len;
      const uint16_t* qrow = q + (row_tok[r] * Hq + h) * (int64_t)d_qk;
      double m = -INFINITY;
      for (int64_t j = 0; j < kv_len; ++j) {
        int allowed = (j >= lo && j < hi);
        if (causal && j > pos) allowed = 0;
        if (window_left >= 0 && j < pos - window_left) allowed = 0;
        if (mask) {
          int64_t bit = mask_indptr[b] * 8 + i * kv_len + j;
          if (!((mask[bit >> 3] >> (bit & 7)) & 1)) allowed = 0;
        }
        if (!allowed) { s[j] = -INFINITY; continue; }
        double dot = 0.0;
        for (int d = 0; d < d_qk; ++d) dot += oracle_bf16_value(qrow[d]) * K[j * d_qk + d];
        s[j] = sm_scale * dot;
        if (s[j] > m) m = s[j];
      }
      double* o = out + r * (int64_t)d_vo;
      for (int d = 0; d < d_vo; ++d) o[d] = 0.0;
      if (m == -INFINITY) { lse[r] = -INFINITY; continue; }
      double l = 0.0;
      for (int64_t j = 0; j < kv_len; ++j) {
        if (s[j] == -INFINITY) continue;
        double p = exp(s[j] - m);
        l += p;
        for (int d = 0; d < d_vo; ++d) o[d] += p * V[j * d_vo + d];
      }
      for (int d = 0; d < d_vo; ++d) o[d] /= l;
      lse[r] = m + log(l);
    }
    free(K); free(V); free(s);
  }
  free(unit_of); free(unit_start); free(order); free(fill);
  return 0;
}

/*
 * oracle_merge: combine split-K partials of one row.  Partial s holds the normalised
 * output o_s over its key subset and lse_s = m_s + ln l_s.  The whole-row result is
 *   lse = ln sum_s exp(lse_s),   o = sum_s exp(lse_s - lse) * o_s.
 * Empty partials carry lse_s = -inf and contribute nothing.  ("split-K", Not covered and
 * Test Coverage of "Run Gemma4 head_dim 512 attention on Triton".)
 */
void oracle_merge(int n_parts, const double* lse_parts, const double* o_parts, int d,
                  double* o, double* lse) {
  double M = -INFINITY;
  for (int s = 0; s < n_parts; ++s)
    if (lse_parts[s] > M) M = lse_parts[s];
  for (int k = 0; k < d; ++k) o[k] = 0.0;
  if (M == -INFINITY) { *lse = -INFINITY; return; }
  double L = 0.0;
  for (int s = 0; s < n_parts; ++s) L += exp(lse_parts[s] - M);
  *lse = M + log(L);
  for (int s = 0; s < n_parts; ++s) {
    if (lse_parts[s] == -INFINITY) continue;
    double w = exp(lse_parts[s] - *lse);
    for (int k = 0; k < d; ++k) o[k] += w * o_parts[(int64_t)s * d + k];
  }
}

/* Dequantise one whole (sequence, kv head, K or V) block into fp64 [kv_len][dim]; for
 * tests that compare against contiguous-layout attention. */
int oracle_gather(const uint8_t* kv_cache, const int32_t* kv_indptr, const int32_t* kv_indices,
                  const int32_t* kv_last_page_len, const uint8_t* sf, int Hkv, int d_qk,
                  int d_vo, int page_size, int kv_dtype, double k_scale, double v_scale, int b,
                  int kvh, int is_v, double* dst) {
  kv_view kv = {kv_cache, kv_indptr, kv_indices, kv_last_page_len, sf,
                Hkv, d_qk, d_vo, page_size, kv_dtype, k_scale, v_scale};
  int64_t kv_len = seq_kv_len(&kv, b);
  int dim = is_v ? d_vo : d_qk;
  for (int64_t j = 0; j < kv_len; ++j)
    for (int d = 0; d < dim; ++d) dst[j * dim + d] = kv_element(&kv, b, kvh, j, is_v, d);
  return (int)kv_len;
}

/* ================================================================ append (quantise-on-write)
 *
 * Writes the K and V rows of new tokens (bf16) into the cache as the last tokens of each
 * sequence, converted to the cache's element type.  The step that produces the FP8 /
 * NVFP4 caches read above ("feat(attention): asymmetric VO-split NVFP4 paged prefill
 * (qk=512/vo=256) for Gemma-4 on SM120/121": caches quantised from bf16 sources by an
 * in-tree NVFP4 KV quantisation kernel; "[None][feat] Run Gemma4 head_dim 512 attention on
 * Triton", Approach: FP8 KV with per-tensor scales).  The pages name the step but not its
 * rounding; the reading used here (stated with the C ABI):
 *   FP8    code = e4m3(x / s), nearest, ties to even, saturating at +-448;
 *   NVFP4  per 16 consecutive head-dim elements of one token and head, global scale G:
 *          amax = max |x|, sf = e4m3((amax / 6) / G), d = value(sf) * G,
 *          code = e2m1(x / d) (nearest, ties to even, saturating at +-6), 0 when d = 0.
 * Every arithmetic step is one fp32 operation in this order (the precision the codes are
 * decided in); the rounding to a code is decided exactly, in double, by comparing the
 * fp32 operand with every representable magnitude.  A code carries the operand's sign,
 * also when it rounds to zero.
 * ==================================================================================== */

/* Nearest of the n increasing non-negative magnitudes vals[0..n-1] to a >= 0, ties to the
 * even index (the code whose mantissa ends in 0); at or above vals[n-1]: n - 1. */
static int nearest_code(double a, const double* vals, int n) {
  if (a >= vals[n - 1]) return n - 1;
  int best = 0;
  double bd = fabs(a - vals[0]);
  for (int c = 1; c < n; ++c) {
    double dd = fabs(a - vals[c]);
    if (dd < bd || (dd == bd && (c & 1) == 0)) {
      best = c;
      bd = dd;
    }
  }
  return best;
}

static double g_e4m3_mag[127];
static double g_e2m1_mag[8];
static int g_tables_ready = 0;

static void build_tables(void) {
  if (g_tables_ready) return;
  for (int c = 0; c < 127; ++c) g_e4m3_mag[c] = oracle_e4m3_value((uint8_t)c);  /* 0x7F is NaN */
  for (int c = 0; c < 8; ++c) g_e2m1_mag[c] = oracle_e2m1_value((uint8_t)c);
  g_tables_ready = 1;
}

uint8_t oracle_e4m3_encode(float v) {
  build_tables();
  int code = nearest_code(fabs((double)v), g_e4m3_mag, 127);
  return (uint8_t)(code | (signbit(v) ? 0x80 : 0));
}

uint8_t oracle_e2m1_encode(float v) {
  build_tables();
  int code = nearest_code(fabs((double)v), g_e2m1_mag, 8);
  return (uint8_t)(code | (signbit(v) ? 0x8 : 0));
}

static float bf16_float(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* Returns the number of new rows skipped because their position falls outside the
 * sequence or their page id outside [0, num_pages). */
int oracle_append_kv(const uint16_t* k_new, const uint16_t* v_new, const int32_t* append_indptr,
                     uint8_t* kv_cache, const int32_t* kv_indptr, const int32_t* kv_indices,
                     const int32_t* kv_last_page_len, int batch, int num_pages, int Hkv, int d_qk,
                     int d_vo, int page_size, int kv_dtype, float k_scale, float v_scale,
                     uint8_t* sf) {
  build_tables();
  const int64_t x2 = kv_dtype == KV_BF16 ? 4 : (kv_dtype == KV_FP8_E4M3 ? 2 : 1);
  const int64_t rows = (int64_t)Hkv * page_size;
  const int64_t k_row = (int64_t)d_qk * x2 / 2, v_row = (int64_t)d_vo * x2 / 2;
  const int64_t page_bytes = rows * (k_row + v_row);
  const int64_t sf_page = rows * (d_qk / 16 + d_vo / 16);
  int skipped = 0;
  for (int b = 0; b < batch; ++b) {
    int n = append_indptr[b + 1] - append_indptr[b];
    int np = kv_indptr[b + 1] - kv_indptr[b];
    int64_t kv_len = np > 0 ? (int64_t)(np - 1) * page_size + kv_last_page_len[b] : 0;
    for (int j = 0; j < n; ++j) {
      int64_t i = append_indptr[b] + j;      /* new row */
      int64_t t = kv_len - n + j;            /* its position in the sequence */
      if (t < 0 || t >= kv_len) { ++skipped; continue; }
      int page = kv_indices[kv_indptr[b] + t / page_size];
      if (page < 0 || page >= num_pages) { ++skipped; continue; }
      int64_t slot = t % page_size;
      for (int h = 0; h < Hkv; ++h)
        for (int is_v = 0; is_v < 2; ++is_v) {
          int dim = is_v ? d_vo : d_qk;
          const uint16_t* src = (is_v ? v_new : k_new) + (i * Hkv + h) * dim;
          int64_t row = (int64_t)h * page_size + slot;
          uint8_t* dst = kv_cache + page * page_bytes + (is_v ? rows * k_row + row * v_row : row * k_row);
          float s = is_v ? v_scale : k_scale;
          if (kv_dtype == KV_BF16) {
            memcpy(dst, src, (size_t)dim * 2);
          } else if (kv_dtype == KV_FP8_E4M3) {
            for (int d = 0; d < dim; ++d) dst[d] = oracle_e4m3_encode(bf16_float(src[d]) / s);
          } else {
            uint8_t* sfd = sf + page * sf_page + (is_v ? rows * (d_qk / 16) + row * (d_vo / 16) : row * (d_qk / 16));
            for (int blk = 0; blk < dim / 16; ++blk) {
              float x[16], amax = 0.0f;
              for (int e = 0; e < 16; ++e) {
                x[e] = bf16_float(src[blk * 16 + e]);
                float a = fabsf(x[e]);
                if (a > amax) amax = a;
              }
              uint8_t sfc = oracle_e4m3_encode((amax / 6.0f) / s);
              float dd = (float)oracle_e4m3_value(sfc) * s;
              sfd[blk] = sfc;
              for (int e = 0; e < 16; e += 2) {
                uint8_t lo = dd != 0.0f ? oracle_e2m1_encode(x[e] / dd) : 0;
                uint8_t hi = dd != 0.0f ? oracle_e2m1_encode(x[e + 1] / dd) : 0;
                dst[blk * 8 + e / 2] = (uint8_t)(lo | (hi << 4));
              }
            }
          }
        }
    }
  }
  return skipped;
}
