/*
 * Paged-attention decode oracle: a plain, slow CPU implementation in double
 * precision. TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the
 * CPU-baseline leg of the benchmark are its only users; the product path never
 * links or calls it. It shares no code with the CUDA library.
 *
 * What it computes (the plain definition the split-KV kernels reach up to
 * rounding):
 *
 *   For sequence b, query index i in [0, QL), query head h, KV head
 *   g = h / (Hq / Hkv)  (GQA grouping, PR "Add paged-attention Tile kernel",
 *   host wrapper: query_group_size = num_q_heads // num_kv_heads):
 *     L = ctx_lens[b], query position p = L - QL + i (the context includes the
 *     new tokens: PR "Merge gfx1250 PA decode partitions ...", the non-causal
 *     commit note says one row's causal bound is the whole context);
 *     visible tokens T = { t in [0, L) : (!causal || t <= p)
 *                                        && (W == 0 || t > p - W) }
 *       (a window of W tokens includes the query's own token, so W = 1 leaves
 *        only t = p; PR "Extend packed D256 PA decode pipe ...", Validation,
 *        windows 0/1/17/257/8193);
 *     sparse decode instead uses T = { idx[b][j] : 0 <= idx < L }.
 *     K/V row of token t: page = block_table[b][t / S], slot = t % S,
 *       dequantised exactly (FP8 e4m3fn code times its per-tensor or per-token
 *       scale; BF16 widened), PR "Add paged-attention Tile kernel" (scales are
 *       a scalar or [num_blocks, num_kv_heads, block_size]); MXFP4 (PR "Merge
 *       gfx1250 PA decode partitions ...", the merge-resolution notes name
 *       MXFP4 K/V without a layout): the OCP Microscaling (MX) v1.0 format,
 *       blocks of 32 consecutive head dims of one token row, each an E8M0
 *       scale times 32 FP4 E2M1 elements (see kv_element for the layout).
 *     Transposed V (PR "Extend packed D256 PA decode pipe to page16,
 *       transposed V and sliding windows", and the D64 note of PR "Merge
 *       gfx1250 PA decode partitions ..."): a page's BF16 V rows stored as
 *       chunks of 8 consecutive tokens per head dim, [S/8][D][8], so one
 *       chunk's dims sit 16 bytes apart and consecutive chunks 16 * D bytes
 *       apart.
 *     x_t = sm_scale * sum_d q[d] * k[d]  (q widened exactly from BF16 or FP16:
 *       PR "Extend packed D256 PA decode pipe ...", Validation, and PR "Merge
 *       gfx1250 PA decode partitions ...", Validation, run BF16 and FP16
 *       queries)
 *     with sink s_h: m = max(max_t x_t, s_h), den = sum_t e^(x_t-m) + e^(s_h-m)
 *     without:        m = max_t x_t,          den = sum_t e^(x_t-m)
 *     out = sum_t e^(x_t-m) v_t / den; out = 0 when T is empty.
 *
 * Reading of the pages where they are silent (also listed in the design
 * notes): the sink is an extra logit in natural-log units, not multiplied by
 * sm_scale, with no value row; an empty visible set gives zeros, sink or not.
 *
 * Partials and their merge (PR "Merge gfx1250 PA decode partitions ...",
 * Partition merges): a partial over a token subset is (m, l, O) with
 * m = max x_t, l = sum e^(x_t - m), O = sum e^(x_t - m) v_t; merging a list of
 * partials in order gives M = max(m_j [, s]), L = sum l_j e^(m_j - M)
 * [+ e^(s - M)], out = sum O_j e^(m_j - M) / L.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define PA_ORACLE_OK 0
#define PA_ORACLE_BAD_ARG 1
#define PA_ORACLE_BAD_PAGE 2
#define PA_ORACLE_NO_MEM 3

enum { ORACLE_KV_FP8 = 0, ORACLE_KV_BF16 = 1, ORACLE_KV_MXFP4 = 2 };
enum { ORACLE_Q_BF16 = 0, ORACLE_Q_FP16 = 1 };
enum { ORACLE_SCALE_NONE = 0, ORACLE_SCALE_PER_TENSOR = 1, ORACLE_SCALE_PER_TOKEN = 2, ORACLE_SCALE_MX_BLOCK = 3 };
#define ORACLE_MX_BLOCK 32
enum { ORACLE_V_PLAIN = 0, ORACLE_V_TRANSPOSED = 1 };
#define ORACLE_V_CHUNK 8 /* tokens per transposed-V chunk */

typedef struct {
  int batch;
  int num_q_heads;
  int num_kv_heads;
  int head_dim;
  int query_len;
  int page_size;
  int max_pages_per_seq;
  int num_pages;
  int kv_dtype;   /* ORACLE_KV_FP8, ORACLE_KV_BF16 or ORACLE_KV_MXFP4 */
  int scale_mode; /* ORACLE_SCALE_* (FP8: NONE/PER_TENSOR/PER_TOKEN; MXFP4: MX_BLOCK) */
  int causal;
  int window; /* 0 = off */
  int has_sinks;
  int topk; /* 0 = dense decode; > 0 = sparse index-list decode (QL must be 1) */
  double sm_scale;
  int q_dtype;  /* ORACLE_Q_BF16 or ORACLE_Q_FP16 (the query's element type) */
  int v_layout; /* ORACLE_V_PLAIN or ORACLE_V_TRANSPOSED (BF16 caches) */
} pa_oracle_shape;

/* OCP 8-bit floating point, E4M3 ("fn": no infinities, S.1111.111 is NaN):
 * exponent bias 7, normal value (1 + m/8) * 2^(e-7), subnormal (m/8) * 2^-6. */
double pa_oracle_e4m3_to_double(uint8_t code) {
  int sign = (code >> 7) & 1;
  int e = (code >> 3) & 0xF;
  int m = code & 0x7;
  double mag;
  if (e == 0xF && m == 0x7) return NAN;
  if (e == 0)
    mag = ldexp((double)m / 8.0, -6);
  else
    mag = ldexp(1.0 + (double)m / 8.0, e - 7);
  return sign ? -mag : mag;
}

/* OCP MX v1.0 FP4 element, E2M1: sign bit 3, exponent bits 2..1 (bias 1),
 * mantissa bit 0; normal value (1 + m/2) * 2^(e-1), subnormal (e = 0) m/2.
 * No infinities or NaNs. */
double pa_oracle_e2m1_to_double(uint8_t code) {
  int sign = (code >> 3) & 1;
  int e = (code >> 1) & 0x3;
  int m = code & 0x1;
  double mag = e == 0 ? 0.5 * (double)m : ldexp(1.0 + 0.5 * (double)m, e - 1);
  return sign ? -mag : mag;
}

/* OCP MX v1.0 shared scale, E8M0: an unsigned biased exponent, value
 * 2^(code - 127); 0xFF is NaN. */
double pa_oracle_e8m0_to_double(uint8_t code) {
  if (code == 0xFF) return NAN;
  return ldexp(1.0, (int)code - 127);
}

/* BF16 is the upper half of an IEEE binary32: widening is exact. */
double pa_oracle_bf16_to_double(uint16_t bits) {
  uint32_t w = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &w, sizeof f);
  return (double)f;
}

/* IEEE 754 binary16: sign, 5 exponent bits (bias 15), 10 fraction bits;
 * exponent field 0 holds the subnormals f * 2^-24, 31 the infinities and
 * NaNs. Widening is exact. */
double pa_oracle_f16_to_double(uint16_t bits) {
  int sign = (bits >> 15) & 1;
  int e = (bits >> 10) & 0x1F;
  int f = bits & 0x3FF;
  double mag;
  if (e == 0x1F)
    mag = f ? NAN : INFINITY;
  else if (e == 0)
    mag = ldexp((double)f, -24);
  else
    mag = ldexp(1024.0 + (double)f, e - 25);
  return sign ? -mag : mag;
}

static double q_element(const pa_oracle_shape* sh, const uint16_t* qrow, int d) {
  return sh->q_dtype == ORACLE_Q_FP16 ? pa_oracle_f16_to_double(qrow[d]) : pa_oracle_bf16_to_double(qrow[d]);
}

/* Round a double to BF16 (8 significant bits, exponent range of binary32),
 * round-to-nearest, ties to even; returns the BF16 bit pattern. */
uint16_t pa_oracle_round_bf16(double x) {
  double r;
  float f;
  uint32_t w;
  if (isnan(x)) return 0x7FC0;
  if (x == 0.0) return signbit(x) ? 0x8000 : 0x0000;
  if (isinf(x)) return x > 0 ? 0x7F80 : 0xFF80;
  {
    int e;
    double a = fabs(x);
    (void)frexp(a, &e); /* a = f * 2^e with f in [0.5, 1) */
    /* quantum: 2^(e-8) for normals, 2^-133 below the binary32 normal range */
    int qexp = e - 8;
    if (qexp < -133) qexp = -133;
    r = nearbyint(ldexp(a, -qexp)); /* default rounding mode: ties to even */
    r = ldexp(r, qexp);
    if (r > 3.3895313892515355e38) r = INFINITY; /* above the largest finite BF16 */
    if (signbit(x)) r = -r;
  }
  f = (float)r; /* exact: r is representable in BF16, hence in binary32 */
  memcpy(&w, &f, sizeof w);
  return (uint16_t)(w >> 16);
}

/* Element d of the K or V row (page, g, slot). `scale` holds binary32 scales
 * (FP8: one, or one per token row) or, for MXFP4, the E8M0 bytes.
 * MXFP4 layout (this library's reading; the pages give none): the row's D
 * elements are D/2 bytes, element d in the low nibble of byte d/2 when d is
 * even and in the high nibble when odd; its D/32 scale bytes sit at
 * scale[row * D/32 + d/32], row = (page * Hkv + g) * page_size + slot. */
static double kv_element(const pa_oracle_shape* sh, const void* cache, const void* scale,
                         int page, int g, int slot, int d) {
  size_t row = ((size_t)page * sh->num_kv_heads + g) * sh->page_size + slot;
  size_t idx = row * sh->head_dim + d;
  if (sh->kv_dtype == ORACLE_KV_BF16) return pa_oracle_bf16_to_double(((const uint16_t*)cache)[idx]);
  if (sh->kv_dtype == ORACLE_KV_MXFP4) {
    uint8_t byte = ((const uint8_t*)cache)[row * (size_t)(sh->head_dim / 2) + (size_t)(d / 2)];
    uint8_t code = (d & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 0xF);
    uint8_t x = ((const uint8_t*)scale)[row * (size_t)(sh->head_dim / ORACLE_MX_BLOCK) + (size_t)(d / ORACLE_MX_BLOCK)];
    return pa_oracle_e2m1_to_double(code) * pa_oracle_e8m0_to_double(x);
  }
  {
    double v = pa_oracle_e4m3_to_double(((const uint8_t*)cache)[idx]);
    if (sh->scale_mode == ORACLE_SCALE_PER_TENSOR)
      v *= (double)((const float*)scale)[0];
    else if (sh->scale_mode == ORACLE_SCALE_PER_TOKEN)
      v *= (double)((const float*)scale)[row];
    return v;
  }
}

/* Element d of the V row (page, g, slot): the plain layout, or the transposed
 * one (BF16 only), where the page block of head g is [S/8 chunks][D][8 tokens]. */
static double v_element(const pa_oracle_shape* sh, const void* cache, const void* scale,
                        int page, int g, int slot, int d) {
  if (sh->v_layout == ORACLE_V_TRANSPOSED) {
    size_t block = ((size_t)page * sh->num_kv_heads + g) * (size_t)(sh->page_size / ORACLE_V_CHUNK);
    size_t idx = ((block + (size_t)(slot / ORACLE_V_CHUNK)) * sh->head_dim + d) * ORACLE_V_CHUNK + slot % ORACLE_V_CHUNK;
    return pa_oracle_bf16_to_double(((const uint16_t*)cache)[idx]);
  }
  return kv_element(sh, cache, scale, page, g, slot, d);
}

/* Physical page holding logical token t of sequence b, or -1 if the table
 * entry is out of the pool. */
static int token_page(const pa_oracle_shape* sh, const int32_t* block_table, int b, int t) {
  int page = block_table[(size_t)b * sh->max_pages_per_seq + t / sh->page_size];
  if (page < 0 || page >= sh->num_pages) return -1;
  return page;
}

/* Visible token list of query row (b, i): dense mask or sparse index list. */
static int visible_tokens(const pa_oracle_shape* sh, const int32_t* ctx_lens, const int32_t* topk_idx,
                          int b, int i, int32_t* tokens) {
  int L = ctx_lens[b];
  int n = 0;
  if (sh->topk > 0) {
    for (int j = 0; j < sh->topk; ++j) {
      int t = topk_idx[(size_t)b * sh->topk + j];
      if (t >= 0 && t < L) tokens[n++] = t;
    }
    return n;
  }
  {
    int p = L - sh->query_len + i;
    for (int t = 0; t < L; ++t) {
      if (sh->causal && t > p) continue;
      if (sh->window > 0 && t <= p - sh->window) continue;
      tokens[n++] = t;
    }
  }
  return n;
}

/* Partial (m, l, O[D]) of query row (b, i, h) over an explicit token list,
 * natural-log units. Empty list: m = -inf, l = 0, O = 0. */
int pa_oracle_row_partial(const pa_oracle_shape* sh, const uint16_t* q, const void* k_cache,
                          const void* v_cache, const int32_t* block_table, const void* k_scale,
                          const void* v_scale, int b, int i, int h, const int32_t* tokens,
                          int ntok, double* m_out, double* l_out, double* o_out) {
  int D = sh->head_dim;
  int G = sh->num_q_heads / sh->num_kv_heads;
  int g = h / G;
  const uint16_t* qrow = q + (((size_t)b * sh->query_len + i) * sh->num_q_heads + h) * D;
  double* x = (double*)malloc(sizeof(double) * (ntok > 0 ? ntok : 1));
  double m = -INFINITY, l = 0.0;
  if (!x) return PA_ORACLE_NO_MEM;
  for (int d = 0; d < D; ++d) o_out[d] = 0.0;
  for (int j = 0; j < ntok; ++j) {
    int t = tokens[j];
    int page = token_page(sh, block_table, b, t);
    double s = 0.0;
    if (page < 0) {
      free(x);
      return PA_ORACLE_BAD_PAGE;
    }
    for (int d = 0; d < D; ++d)
      s += q_element(sh, qrow, d) * kv_element(sh, k_cache, k_scale, page, g, t % sh->page_size, d);
    x[j] = sh->sm_scale * s;
    if (x[j] > m) m = x[j];
  }
  for (int j = 0; j < ntok; ++j) {
    int t = tokens[j];
    int page = token_page(sh, block_table, b, t);
    double w = exp(x[j] - m);
    l += w;
    for (int d = 0; d < D; ++d)
      o_out[d] += w * v_element(sh, v_cache, v_scale, page, g, t % sh->page_size, d);
  }
  free(x);
  *m_out = m;
  *l_out = l;
  return PA_ORACLE_OK;
}

/* Merge partials j = 0..n-1 in order, with an optional sink logit. */
void pa_oracle_merge(int n, int D, const double* m, const double* l, const double* o, int has_sink,
                     double sink, double* out) {
  double M = -INFINITY, L = 0.0;
  for (int j = 0; j < n; ++j)
    if (m[j] > M) M = m[j];
  if (has_sink && sink > M) M = sink;
  for (int d = 0; d < D; ++d) out[d] = 0.0;
  if (M == -INFINITY) return; /* no token, no sink */
  for (int j = 0; j < n; ++j) {
    double a;
    if (m[j] == -INFINITY) continue; /* empty partial contributes nothing */
    a = exp(m[j] - M);
    L += l[j] * a;
    for (int d = 0; d < D; ++d) out[d] += o[(size_t)j * D + d] * a;
  }
  if (has_sink) L += exp(sink - M);
  if (L == 0.0) {
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    return;
  }
  for (int d = 0; d < D; ++d) out[d] /= L;
}

static int check_shape(const pa_oracle_shape* sh) {
  if (sh->batch < 0 || sh->num_q_heads <= 0 || sh->num_kv_heads <= 0 || sh->head_dim <= 0 ||
      sh->query_len <= 0 || sh->page_size <= 0 || sh->max_pages_per_seq <= 0 || sh->num_pages <= 0)
    return PA_ORACLE_BAD_ARG;
  if (sh->num_q_heads % sh->num_kv_heads != 0) return PA_ORACLE_BAD_ARG;
  if (sh->topk > 0 && sh->query_len != 1) return PA_ORACLE_BAD_ARG;
  if (sh->window < 0) return PA_ORACLE_BAD_ARG;
  if (sh->q_dtype != ORACLE_Q_BF16 && sh->q_dtype != ORACLE_Q_FP16) return PA_ORACLE_BAD_ARG;
  if (sh->kv_dtype != ORACLE_KV_FP8 && sh->kv_dtype != ORACLE_KV_BF16 && sh->kv_dtype != ORACLE_KV_MXFP4)
    return PA_ORACLE_BAD_ARG;
  if ((sh->kv_dtype == ORACLE_KV_MXFP4) != (sh->scale_mode == ORACLE_SCALE_MX_BLOCK)) return PA_ORACLE_BAD_ARG;
  if (sh->kv_dtype == ORACLE_KV_MXFP4 && sh->head_dim % ORACLE_MX_BLOCK != 0) return PA_ORACLE_BAD_ARG;
  if (sh->v_layout != ORACLE_V_PLAIN && sh->v_layout != ORACLE_V_TRANSPOSED) return PA_ORACLE_BAD_ARG;
  if (sh->v_layout == ORACLE_V_TRANSPOSED && (sh->kv_dtype != ORACLE_KV_BF16 || sh->page_size % ORACLE_V_CHUNK != 0))
    return PA_ORACLE_BAD_ARG;
  return PA_ORACLE_OK;
}

/* Full decode. out: double [B*QL, Hq, D]. unit_mask (optional, [B*Hkv]):
 * rows of units whose mask byte is 0 are skipped (left untouched). */
int pa_oracle_decode(const pa_oracle_shape* sh, const uint16_t* q, const void* k_cache,
                     const void* v_cache, const int32_t* block_table, const int32_t* ctx_lens,
                     const void* k_scale, const void* v_scale, const float* sinks,
                     const int32_t* topk_idx, const uint8_t* unit_mask, double* out) {
  int rc = check_shape(sh);
  int D, G, maxL = 0;
  int32_t* tokens;
  double* o;
  if (rc) return rc;
  D = sh->head_dim;
  G = sh->num_q_heads / sh->num_kv_heads;
  for (int b = 0; b < sh->batch; ++b)
    if (ctx_lens[b] > maxL) maxL = ctx_lens[b];
  if (sh->topk > maxL) maxL = sh->topk;
  for (int b = 0; b < sh->batch; ++b)
    if ((long long)ctx_lens[b] > (long long)sh->max_pages_per_seq * sh->page_size || ctx_lens[b] < 0)
      return PA_ORACLE_BAD_ARG;
  tokens = (int32_t*)malloc(sizeof(int32_t) * (maxL > 0 ? maxL : 1));
  o = (double*)malloc(sizeof(double) * D);
  if (!tokens || !o) {
    free(tokens);
    free(o);
    return PA_ORACLE_NO_MEM;
  }
  for (int b = 0; b < sh->batch && rc == PA_ORACLE_OK; ++b) {
    for (int i = 0; i < sh->query_len && rc == PA_ORACLE_OK; ++i) {
      int ntok = visible_tokens(sh, ctx_lens, topk_idx, b, i, tokens);
      for (int h = 0; h < sh->num_q_heads; ++h) {
        double m, l;
        double* dst = out + (((size_t)b * sh->query_len + i) * sh->num_q_heads + h) * D;
        if (unit_mask && !unit_mask[(size_t)b * sh->num_kv_heads + h / G]) continue;
        rc = pa_oracle_row_partial(sh, q, k_cache, v_cache, block_table, k_scale, v_scale, b, i, h,
                                   tokens, ntok, &m, &l, o);
        if (rc) break;
        if (ntok == 0) {
          for (int d = 0; d < D; ++d) dst[d] = 0.0;
          continue;
        }
        {
          double den = l;
          double M = m;
          double a = 1.0;
          if (sh->has_sinks) {
            double s = (double)sinks[h];
            if (s > M) M = s;
            a = exp(m - M);
            den = l * a + exp(s - M);
          }
          for (int d = 0; d < D; ++d) dst[d] = o[d] * a / den;
        }
      }
    }
  }
  free(tokens);
  free(o);
  return rc;
}

/* Round a double array to BF16 bit patterns. */
void pa_oracle_round_bf16_array(const double* x, uint16_t* bits, size_t n) {
  for (size_t k = 0; k < n; ++k) bits[k] = pa_oracle_round_bf16(x[k]);
}

/*
 * Indexer logits (PR "[FlyDSL] fp8_mqa_logits gfx942: add LDS-staged variant,
 * use it by default", Summary and Changes: FP8 queries and KV, a ReLU x
 * weight epilogue reduced over the heads, per-row KV windows, -inf written
 * outside them when clean_logits is set). For query row r and KV token j:
 *
 *   inside the window (ks[r] <= j < ke[r], 0 <= j < num_kv):
 *     logit = sum_h w[r][h] * max(0, kv_scale[j] * sum_d q[r][h][d] * kv[j][d])
 *   outside: -inf
 *
 * with q and kv e4m3 codes decoded exactly. The reading where the page is
 * silent: the per-token KV scale multiplies the dot product before the ReLU.
 * Computed for the n listed (r, j) pairs; bound[i] receives
 * sum_h |w| * |kv_scale| * sum_d |q * kv| (the magnitude an FP32 evaluation's
 * rounding is proportional to), 0 outside the window.
 */
int pa_oracle_mqa_logits(int rows, int heads, int dim, int num_kv, const uint8_t* q, const uint8_t* kv,
                         const float* kv_scale, const float* weights, const int32_t* ks, const int32_t* ke,
                         int n, const int32_t* pr, const int32_t* pj, double* out, double* bound) {
  if (rows < 0 || heads <= 0 || dim <= 0 || num_kv < 0 || n < 0) return PA_ORACLE_BAD_ARG;
  for (int i = 0; i < n; ++i) {
    int r = pr[i], j = pj[i];
    if (r < 0 || r >= rows || j < 0 || j >= num_kv) return PA_ORACLE_BAD_ARG;
    if (!(j >= ks[r] && j < ke[r])) {
      out[i] = -INFINITY;
      bound[i] = 0.0;
      continue;
    }
    {
      double sc = (double)kv_scale[j], acc = 0.0, mag = 0.0;
      for (int h = 0; h < heads; ++h) {
        double s = 0.0, a = 0.0, w = (double)weights[(size_t)r * heads + h];
        for (int d = 0; d < dim; ++d) {
          double x = pa_oracle_e4m3_to_double(q[((size_t)r * heads + h) * dim + d]) *
                     pa_oracle_e4m3_to_double(kv[(size_t)j * dim + d]);
          s += x;
          a += fabs(x);
        }
        s *= sc;
        acc += w * (s > 0.0 ? s : 0.0);
        mag += fabs(w) * fabs(sc) * a;
      }
      out[i] = acc;
      bound[i] = mag;
    }
  }
  return PA_ORACLE_OK;
}
