/*
 * kivi_oracle.c -- plain, slow CPU oracle for the KIVI asymmetric 2-bit KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or call
 * this file: only the test suite, the smoke check and the benchmark's CPU-baseline
 * leg use it.  It shares no code, header, table or constant with the CUDA library;
 * it is written from the method's description, step by step, so that a reader can
 * check it against the text by eye.
 *
 * Source of the method: "KIVI: A Tuning-Free Asymmetric 2bit Quantization for KV
 * Cache" as summarised on the page "Makale Bulteni -- KIVI" (cmlonder.com, radar /
 * paper-to-prod, 2026-11-01):
 *   - headline paragraph: keys are quantized per channel, values per token, in an
 *     asymmetric 2-bit format;
 *   - section "Iddia ve Gerceklik", 2nd paragraph: key outlier channels are fixed
 *     along the sequence, so keys are grouped along the channel axis; values have no
 *     outlier channels and the attention output is a weighted sum of values, so their
 *     error is kept per token;
 *   - same section, 3rd paragraph: because a new token's channel min/max is not known
 *     in advance, keys are split into groups of G = 32 or 64 tokens and the trailing
 *     tokens of an unfilled group stay in a full-precision residual buffer.
 *
 * Readings where the page is silent (each is listed in the design notes):
 *   R1  asymmetric 2-bit = min/max zero-point and scale: z = min, s = (max-min)/3.
 *   R2  fp32 arithmetic with round-to-nearest-even for every operation of the
 *       quantizer; s is rounded to fp16 and the codes are computed with that stored
 *       fp16 scale; the division is a true division, not a reciprocal multiply.
 *   R3  code = clamp(rint_half_even((x - min) / s), 0, 3); a group with s16 == 0
 *       gets all-zero codes.
 *   R4  scale and zero are stored as fp16 {s, z}; a zero-point of -0 is stored as +0.
 *   R5  values: one (s, z) per token and KV head over all D channels.
 *   R6  only keys have a residual; a full group is flushed as soon as it fills, so
 *       r = n mod G tokens are residual.
 *   R7  packing: a token row is D/16 words; word w holds channels 16w..16w+15 and
 *       channel 16w+i sits in bits [2i, 2i+1].
 *   R8  attention over the dequantized cache in fp64:
 *       score_t = sigma * q . K'_t,  p = softmax(score),  out = sum_t p_t V'_t,
 *       with query head h reading KV head h / (Hq / Hkv).
 *   R10 (variant, bits = 4) the same rule with 2^4 - 1 = 15 levels:
 *       s = (max - min) / 15, code = clamp(round_half_even((x - min) / s), 0, 15),
 *       packed 8 per word: word w holds channels 8w..8w+7, channel 8w+i in bits
 *       [4i, 4i+3].  bits = 2 is R1-R7 unchanged.
 *   R9  (variant, when a value residual buffer is given) values keep the same
 *       residual as keys: the last n mod G values stay fp16, and when the key group
 *       flushes its G values are quantized per token (R5) at once.  Without the
 *       buffer, R6 holds: every value is quantized when it arrives.
 *   R11 (variant, value group vg < D) a value token is quantized in D / vg groups of
 *       vg consecutive channels, group g = channels g*vg .. g*vg + vg - 1, each with
 *       its own {s, z} by R1-R4 (R10 for bits = 4); the token's meta entries are
 *       its groups in order.  vg = D is R5.  The codes are packed as in R7 / R10.
 *   R12 (prefill attention, "Kod ve Entegrasyon Haritasi": FlashAttention runs the
 *       prefill) the prompt attends to itself in full precision, causally: for
 *       position i, out_i = sum_{j <= i} softmax_j(sigma * q_i . k_j) v_j over the
 *       raw fp16 keys and values, fp64, query head h reading KV head h / (Hq / Hkv);
 *       the cache is then quantized from the same fp16 K and V (R1-R11).
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fopenmp -shared -fPIC.  No fast-math and
 * no FMA contraction, so every fp32 operation is a single IEEE-754 RNE operation.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef _Float16 f16; /* IEEE-754 binary16; float -> f16 conversion rounds to nearest even */

static float h2f(uint16_t bits) {
  f16 h;
  memcpy(&h, &bits, sizeof h);
  return (float)h;
}

static uint16_t f2h(float x) {
  f16 h = (f16)x;
  uint16_t bits;
  memcpy(&bits, &h, sizeof bits);
  return bits;
}

/* fp16 <-> fp32 conversions, exported so the tests can pin them to numpy. */
float oracle_h2f(uint16_t bits) { return h2f(bits); }
uint16_t oracle_f2h(float x) { return f2h(x); }

int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Threads of the batch entry points' OpenMP loops (timing only; results do not
 * depend on it: each (batch, head) is computed by one thread). */
void oracle_set_threads(int n) {
#ifdef _OPENMP
  omp_set_num_threads(n > 0 ? n : 1);
#else
  (void)n;
#endif
}

/*
 * Quantize one group of `count` fp16 values x[i * stride] (R1-R4).
 * A key group is one channel of G consecutive tokens; a value group is one token
 * row of D channels.  Writes the fp16 scale and zero bit patterns and one code
 * (0..3) per element.
 */
void oracle_quantize_group(const uint16_t *x, int64_t count, int64_t stride, int bits,
                           uint16_t *s_out, uint16_t *z_out, uint8_t *codes) {
  const float levels = (float)((1 << bits) - 1); /* 3 (R1) or 15 (R10) */
  /* step 1: min and max (exact: both are fp16 values) */
  float mn = h2f(x[0]);
  float mx = mn;
  for (int64_t i = 1; i < count; ++i) {
    float v = h2f(x[i * stride]);
    if (v < mn) mn = v;
    if (v > mx) mx = v;
  }
  /* step 2: scale = (max - min) / (2^bits - 1) in fp32, then stored as fp16 */
  float range = mx - mn;
  float s32 = range / levels;
  uint16_t s16 = f2h(s32);
  float s = h2f(s16);
  /* step 3: zero-point = min, stored as fp16 (exact); -0 is stored as +0 */
  uint16_t z16 = f2h(mn);
  if (z16 == 0x8000u) z16 = 0x0000u;
  *s_out = s16;
  *z_out = z16;
  /* step 4: code = clamp(round_half_even((x - min) / s), 0, 2^bits - 1) */
  for (int64_t i = 0; i < count; ++i) {
    if (s == 0.0f) {
      codes[i] = 0;
      continue;
    }
    float d = h2f(x[i * stride]) - mn;
    float u = d / s;
    float r = rintf(u); /* default rounding mode: nearest, ties to even */
    if (r < 0.0f) r = 0.0f;
    if (r > levels) r = levels;
    codes[i] = (uint8_t)r;
  }
}

/* R7 / R10: pack the D codes of one token row into D * bits / 32 words: word w
 * holds the 32 / bits channels starting at w * 32 / bits, channel i of the word in
 * bits [bits * i, bits * i + bits - 1]. */
void oracle_pack_row(const uint8_t *codes, int D, int bits, uint32_t *words) {
  const int per_word = 32 / bits;
  const uint32_t mask = (1u << bits) - 1u;
  for (int w = 0; w < D / per_word; ++w) {
    uint32_t word = 0;
    for (int i = 0; i < per_word; ++i) word |= (uint32_t)(codes[per_word * w + i] & mask) << (bits * i);
    words[w] = word;
  }
}

/* words of one packed token row */
#define WPR(D, bits) ((D) * (bits) / 32)

/* inverse of oracle_pack_row */
static uint8_t unpack_code(const uint32_t *row, int bits, int c) {
  const int per_word = 32 / bits;
  return (uint8_t)((row[c / per_word] >> (bits * (c % per_word))) & ((1u << bits) - 1u));
}

static uint32_t meta_word(uint16_t s, uint16_t z) { return (uint32_t)s | ((uint32_t)z << 16); }
static uint16_t meta_s(uint32_t m) { return (uint16_t)(m & 0xffffu); }
static uint16_t meta_z(uint32_t m) { return (uint16_t)(m >> 16); }

/*
 * Key group quantization (R1-R4, R7): `rows` holds G token rows of D fp16 channels.
 * Each channel is quantized over the G tokens; the codes are packed per token row
 * into codes_out (G rows of D*bits/32 words) and the per-channel {s, z} go to meta_out[D].
 */
static void quantize_key_group(const uint16_t *rows, int D, int G, int bits, uint32_t *codes_out,
                               uint32_t *meta_out) {
  uint8_t *col = (uint8_t *)malloc((size_t)G);
  uint8_t *mat = (uint8_t *)malloc((size_t)G * D); /* [G][D] codes */
  for (int c = 0; c < D; ++c) {
    uint16_t s, z;
    oracle_quantize_group(rows + c, G, D, bits, &s, &z, col);
    meta_out[c] = meta_word(s, z);
    for (int t = 0; t < G; ++t) mat[(size_t)t * D + c] = col[t];
  }
  for (int t = 0; t < G; ++t) oracle_pack_row(mat + (size_t)t * D, D, bits, codes_out + (size_t)t * WPR(D, bits));
  free(mat);
  free(col);
}

/* Meta entries per value token: one per channel group (R5, R11). */
#define VMW(D, vg) ((D) / (vg))

/* Value token quantization (R5, R7, R10, R11): one row of D channels -> D*bits/32
 * words + D/vg {s, z}, group g over channels g*vg .. g*vg + vg - 1. */
static void quantize_value_token(const uint16_t *row, int D, int bits, int vg, uint32_t *codes_out,
                                 uint32_t *meta_out) {
  uint8_t *codes = (uint8_t *)malloc((size_t)D);
  for (int g = 0; g < VMW(D, vg); ++g) {
    uint16_t s, z;
    oracle_quantize_group(row + (size_t)g * vg, vg, 1, bits, &s, &z, codes + (size_t)g * vg);
    meta_out[g] = meta_word(s, z);
  }
  oracle_pack_row(codes, D, bits, codes_out);
  free(codes);
}

/*
 * One (batch, KV head): quantize a prompt of n tokens (R6, R9).
 *   k, v     : [n][D] fp16
 *   k_codes  : [max_tokens][D*bits/32]   rows < floor(n/G)*G written
 *   k_meta   : [max_tokens/G][D]    groups < floor(n/G) written
 *   k_res    : [G][D]               slots < n mod G written (token nq + j in slot j)
 *   v_codes  : [max_tokens][D*bits/32]   rows < n written (rows < nq with a value residual)
 *   v_meta   : [max_tokens][D/vg]   rows < n written (< nq with a value residual)
 *   v_res    : [G][D] or NULL       with a value residual: slots < n mod G written
 */
void oracle_prefill_head(int D, int G, int bits, int vg, int64_t n, const uint16_t *k, const uint16_t *v,
                         uint32_t *k_codes, uint32_t *k_meta, uint16_t *k_res,
                         uint32_t *v_codes, uint32_t *v_meta, uint16_t *v_res) {
  int64_t n_groups = n / G;
  int64_t nq = n_groups * G;
  for (int64_t g = 0; g < n_groups; ++g)
    quantize_key_group(k + (size_t)g * G * D, D, G, bits, k_codes + (size_t)g * G * WPR(D, bits),
                       k_meta + (size_t)g * D);
  for (int64_t j = 0; j < n - nq; ++j)
    memcpy(k_res + (size_t)j * D, k + (size_t)(nq + j) * D, (size_t)D * sizeof(uint16_t));
  int64_t n_quantized_values = v_res ? nq : n;
  for (int64_t t = 0; t < n_quantized_values; ++t)
    quantize_value_token(v + (size_t)t * D, D, bits, vg, v_codes + (size_t)t * WPR(D, bits),
                         v_meta + (size_t)t * VMW(D, vg));
  if (v_res)
    for (int64_t j = 0; j < n - nq; ++j)
      memcpy(v_res + (size_t)j * D, v + (size_t)(nq + j) * D, (size_t)D * sizeof(uint16_t));
}

/*
 * One (batch, KV head): append token n (the cache holds n tokens before the call).
 * The key goes to residual slot n mod G; the value is quantized at once (R6), or
 * with a value residual (R9) goes to the same slot of v_res.  When the residual
 * fills, its G keys are quantized as group n / G (and, with a value residual, its
 * G values token by token) and the residual empties.  Returns the new length n + 1.
 */
int64_t oracle_append_head(int D, int G, int bits, int vg, int64_t n, const uint16_t *k_new, const uint16_t *v_new,
                           uint32_t *k_codes, uint32_t *k_meta, uint16_t *k_res,
                           uint32_t *v_codes, uint32_t *v_meta, uint16_t *v_res) {
  int64_t r = n % G;
  memcpy(k_res + (size_t)r * D, k_new, (size_t)D * sizeof(uint16_t));
  if (v_res)
    memcpy(v_res + (size_t)r * D, v_new, (size_t)D * sizeof(uint16_t));
  else
    quantize_value_token(v_new, D, bits, vg, v_codes + (size_t)n * WPR(D, bits), v_meta + (size_t)n * VMW(D, vg));
  if (r + 1 == G) {
    int64_t g = n / G;
    quantize_key_group(k_res, D, G, bits, k_codes + (size_t)g * G * WPR(D, bits), k_meta + (size_t)g * D);
    if (v_res)
      for (int64_t j = 0; j < G; ++j)
        quantize_value_token(v_res + (size_t)j * D, D, bits, vg, v_codes + (size_t)(g * G + j) * WPR(D, bits),
                             v_meta + (size_t)(g * G + j) * VMW(D, vg));
  }
  return n + 1;
}

/* Dequantized key t of one head, fp64: z + code * s for quantized tokens, the fp16
 * residual value itself for the last n mod G tokens. */
static void dequant_key_f64(int D, int G, int bits, int64_t n, int64_t t, const uint32_t *k_codes,
                            const uint32_t *k_meta, const uint16_t *k_res, double *out) {
  int64_t nq = (n / G) * G;
  if (t < nq) {
    const uint32_t *row = k_codes + (size_t)t * WPR(D, bits);
    const uint32_t *meta = k_meta + (size_t)(t / G) * D;
    for (int c = 0; c < D; ++c)
      out[c] = (double)h2f(meta_z(meta[c])) + (double)unpack_code(row, bits, c) * (double)h2f(meta_s(meta[c]));
  } else {
    const uint16_t *res = k_res + (size_t)(t - nq) * D;
    for (int c = 0; c < D; ++c) out[c] = (double)h2f(res[c]);
  }
}

/* Dequantized value t of one head, fp64: z + code * s of the channel's group (R11),
 * or with a value residual (R9) the fp16 value itself for the last n mod G tokens. */
static void dequant_value_f64(int D, int G, int bits, int vg, int64_t n, int64_t t, const uint32_t *v_codes,
                              const uint32_t *v_meta, const uint16_t *v_res, double *out) {
  int64_t nq = (n / G) * G;
  if (v_res && t >= nq) {
    const uint16_t *res = v_res + (size_t)(t - nq) * D;
    for (int c = 0; c < D; ++c) out[c] = (double)h2f(res[c]);
    return;
  }
  const uint32_t *row = v_codes + (size_t)t * WPR(D, bits);
  const uint32_t *meta = v_meta + (size_t)t * VMW(D, vg);
  for (int c = 0; c < D; ++c) {
    double s = (double)h2f(meta_s(meta[c / vg]));
    double z = (double)h2f(meta_z(meta[c / vg]));
    out[c] = z + (double)unpack_code(row, bits, c) * s;
  }
}

/* Dequantize one head's n tokens to fp64 [n][D] (keys and values). */
void oracle_dequantize_head_f64(int D, int G, int bits, int vg, int64_t n, const uint32_t *k_codes,
                                const uint32_t *k_meta, const uint16_t *k_res,
                                const uint32_t *v_codes, const uint32_t *v_meta, const uint16_t *v_res,
                                double *k_out, double *v_out) {
  for (int64_t t = 0; t < n; ++t) {
    dequant_key_f64(D, G, bits, n, t, k_codes, k_meta, k_res, k_out + (size_t)t * D);
    dequant_value_f64(D, G, bits, vg, n, t, v_codes, v_meta, v_res, v_out + (size_t)t * D);
  }
}

/* Dequantize one head's n tokens to fp32 [n][D]: fp32(z) + fp32(code) * fp32(s),
 * a product that is exact in fp32 followed by one RNE addition. */
void oracle_dequantize_head_f32(int D, int G, int bits, int vg, int64_t n, const uint32_t *k_codes,
                                const uint32_t *k_meta, const uint16_t *k_res,
                                const uint32_t *v_codes, const uint32_t *v_meta, const uint16_t *v_res,
                                float *k_out, float *v_out) {
  int64_t nq = (n / G) * G;
  for (int64_t t = 0; t < n; ++t) {
    float *ko = k_out + (size_t)t * D;
    if (t < nq) {
      const uint32_t *row = k_codes + (size_t)t * WPR(D, bits);
      const uint32_t *meta = k_meta + (size_t)(t / G) * D;
      for (int c = 0; c < D; ++c) {
        float prod = (float)unpack_code(row, bits, c) * h2f(meta_s(meta[c]));
        ko[c] = h2f(meta_z(meta[c])) + prod;
      }
    } else {
      const uint16_t *res = k_res + (size_t)(t - nq) * D;
      for (int c = 0; c < D; ++c) ko[c] = h2f(res[c]);
    }
    float *vo = v_out + (size_t)t * D;
    if (v_res && t >= nq) {
      const uint16_t *res = v_res + (size_t)(t - nq) * D;
      for (int c = 0; c < D; ++c) vo[c] = h2f(res[c]);
      continue;
    }
    const uint32_t *vrow = v_codes + (size_t)t * WPR(D, bits);
    const uint32_t *vmeta = v_meta + (size_t)t * VMW(D, vg);
    for (int c = 0; c < D; ++c) {
      float prod = (float)unpack_code(vrow, bits, c) * h2f(meta_s(vmeta[c / vg]));
      vo[c] = h2f(meta_z(vmeta[c / vg])) + prod;
    }
  }
}

/*
 * R8: attention of one query vector q (D fp16) over one head's n-token cache, fp64.
 *   score_t = sigma * sum_c q_c K'_{t,c};  p = softmax(score) (max subtracted);
 *   out_c = sum_t p_t V'_{t,c}.
 * Returns 0, or -1 when n <= 0 (softmax over an empty set is undefined).
 */
int oracle_attention_head(int D, int G, int bits, int vg, int64_t n, const uint32_t *k_codes,
                          const uint32_t *k_meta,
                          const uint16_t *k_res, const uint32_t *v_codes, const uint32_t *v_meta,
                          const uint16_t *v_res, const uint16_t *q, double sigma, double *out) {
  if (n <= 0) return -1;
  double *score = (double *)malloc((size_t)n * sizeof(double));
  double *row = (double *)malloc((size_t)D * sizeof(double));
  double *qd = (double *)malloc((size_t)D * sizeof(double));
  for (int c = 0; c < D; ++c) qd[c] = (double)h2f(q[c]);
  double m = -INFINITY;
  for (int64_t t = 0; t < n; ++t) {
    dequant_key_f64(D, G, bits, n, t, k_codes, k_meta, k_res, row);
    double acc = 0.0;
    for (int c = 0; c < D; ++c) acc += qd[c] * row[c];
    score[t] = sigma * acc;
    if (score[t] > m) m = score[t];
  }
  double l = 0.0;
  for (int64_t t = 0; t < n; ++t) {
    score[t] = exp(score[t] - m);
    l += score[t];
  }
  for (int c = 0; c < D; ++c) out[c] = 0.0;
  for (int64_t t = 0; t < n; ++t) {
    dequant_value_f64(D, G, bits, vg, n, t, v_codes, v_meta, v_res, row);
    double p = score[t] / l;
    for (int c = 0; c < D; ++c) out[c] += p * row[c];
  }
  free(qd);
  free(row);
  free(score);
  return 0;
}

/*
 * Attention of one query vector over an unquantized fp16 cache (k, v: [n][D] fp16),
 * fp64: the same definition as oracle_attention_head with K' = K and V' = V.  It is
 * the reference for the fp16-cache decode kernel that serves as a comparison point.
 */
int oracle_attention_raw_head(int D, int64_t n, const uint16_t *k, const uint16_t *v, const uint16_t *q,
                              double sigma, double *out) {
  if (n <= 0) return -1;
  double *score = (double *)malloc((size_t)n * sizeof(double));
  double m = -INFINITY;
  for (int64_t t = 0; t < n; ++t) {
    double acc = 0.0;
    for (int c = 0; c < D; ++c) acc += (double)h2f(q[c]) * (double)h2f(k[(size_t)t * D + c]);
    score[t] = sigma * acc;
    if (score[t] > m) m = score[t];
  }
  double l = 0.0;
  for (int64_t t = 0; t < n; ++t) {
    score[t] = exp(score[t] - m);
    l += score[t];
  }
  for (int c = 0; c < D; ++c) out[c] = 0.0;
  for (int64_t t = 0; t < n; ++t) {
    double p = score[t] / l;
    for (int c = 0; c < D; ++c) out[c] += p * (double)h2f(v[(size_t)t * D + c]);
  }
  free(score);
  return 0;
}

/*
 * R12: causal prefill attention of one query head over one KV head's prompt, fp64.
 *   q [n][D], k [n][D], v [n][D] fp16;  out [n][D] fp64 with, for every position i,
 *   out_i = sum_{j <= i} p_ij v_j,  p_i = softmax_j (sigma * q_i . k_j) over j <= i.
 * Returns 0, or -1 when n <= 0.
 */
/* One row of R12: position i's query q_i [D] over keys and values 0 .. i; score is
 * scratch space of i + 1 doubles. */
static void prefill_attention_row(int D, int64_t i, const uint16_t *q_i, const uint16_t *k, const uint16_t *v,
                                  double sigma, double *score, double *o) {
  double m = -INFINITY;
  for (int64_t j = 0; j <= i; ++j) {
    double acc = 0.0;
    for (int c = 0; c < D; ++c) acc += (double)h2f(q_i[c]) * (double)h2f(k[(size_t)j * D + c]);
    score[j] = sigma * acc;
    if (score[j] > m) m = score[j];
  }
  double l = 0.0;
  for (int64_t j = 0; j <= i; ++j) {
    score[j] = exp(score[j] - m);
    l += score[j];
  }
  for (int c = 0; c < D; ++c) o[c] = 0.0;
  for (int64_t j = 0; j <= i; ++j) {
    double p = score[j] / l;
    for (int c = 0; c < D; ++c) o[c] += p * (double)h2f(v[(size_t)j * D + c]);
  }
}

int oracle_prefill_attention_head(int D, int64_t n, const uint16_t *q, const uint16_t *k, const uint16_t *v,
                                  double sigma, double *out) {
  if (n <= 0) return -1;
  double *score = (double *)malloc((size_t)n * sizeof(double));
  for (int64_t i = 0; i < n; ++i) prefill_attention_row(D, i, q + (size_t)i * D, k, v, sigma, score, out + (size_t)i * D);
  free(score);
  return 0;
}

/* R12 at selected positions of one head: rows[r] in [0, n), q [n][D] the head's queries,
 * out [nr][D] fp64.  Returns 0, or -1 on an empty prompt or a position outside it. */
int oracle_prefill_attention_rows(int D, int64_t n, int64_t nr, const int64_t *rows, const uint16_t *q,
                                  const uint16_t *k, const uint16_t *v, double sigma, double *out) {
  if (n <= 0) return -1;
  for (int64_t r = 0; r < nr; ++r)
    if (rows[r] < 0 || rows[r] >= n) return -1;
  double *score = (double *)malloc((size_t)n * sizeof(double));
  for (int64_t r = 0; r < nr; ++r)
    prefill_attention_row(D, rows[r], q + (size_t)rows[r] * D, k, v, sigma, score, out + (size_t)r * D);
  free(score);
  return 0;
}

/* ---------------------------------------------------------------------------------
 * Whole-batch wrappers over the per-head functions.  Buffer shapes:
 *   k, v      [B][Hkv][n][D] fp16         k_new, v_new [B][Hkv][D] fp16
 *   k_codes   [B][Hkv][max_tokens][D*bits/32]  k_meta [B][Hkv][max_tokens/G][D]
 *   k_res     [B][Hkv][G][D] fp16         v_codes [B][Hkv][max_tokens][D*bits/32]
 *   v_meta    [B][Hkv][max_tokens][D/vg]  q [B][Hq][D] fp16, out [B][Hq][D] fp64
 * Heads are independent, so the loops run in parallel over (b, head).
 * ------------------------------------------------------------------------------- */
#define KC(bh) (k_codes + (size_t)(bh) * max_tokens * WPR(D, bits))
#define KM(bh) (k_meta + (size_t)(bh) * (max_tokens / G) * D)
#define KR(bh) (k_res + (size_t)(bh) * G * D)
#define VC(bh) (v_codes + (size_t)(bh) * max_tokens * WPR(D, bits))
#define VM(bh) (v_meta + (size_t)(bh) * max_tokens * VMW(D, vg))
#define VR(bh) (v_res ? v_res + (size_t)(bh) * G * D : NULL)

void oracle_prefill(int B, int Hkv, int D, int G, int bits, int vg, int64_t max_tokens, int64_t n, const uint16_t *k,
                    const uint16_t *v, uint32_t *k_codes, uint32_t *k_meta, uint16_t *k_res,
                    uint32_t *v_codes, uint32_t *v_meta, uint16_t *v_res) {
  int64_t heads = (int64_t)B * Hkv;
#pragma omp parallel for schedule(dynamic)
  for (int64_t bh = 0; bh < heads; ++bh)
    oracle_prefill_head(D, G, bits, vg, n, k + (size_t)bh * n * D, v + (size_t)bh * n * D, KC(bh), KM(bh),
                        KR(bh), VC(bh), VM(bh), VR(bh));
}

int64_t oracle_append(int B, int Hkv, int D, int G, int bits, int vg, int64_t max_tokens, int64_t n,
                      const uint16_t *k_new, const uint16_t *v_new, uint32_t *k_codes,
                      uint32_t *k_meta, uint16_t *k_res, uint32_t *v_codes, uint32_t *v_meta,
                      uint16_t *v_res) {
  int64_t heads = (int64_t)B * Hkv;
#pragma omp parallel for schedule(static)
  for (int64_t bh = 0; bh < heads; ++bh)
    oracle_append_head(D, G, bits, vg, n, k_new + (size_t)bh * D, v_new + (size_t)bh * D, KC(bh), KM(bh),
                       KR(bh), VC(bh), VM(bh), VR(bh));
  return n + 1;
}

int oracle_attention(int B, int Hq, int Hkv, int D, int G, int bits, int vg, int64_t max_tokens, int64_t n,
                     const uint32_t *k_codes, const uint32_t *k_meta, const uint16_t *k_res,
                     const uint32_t *v_codes, const uint32_t *v_meta, const uint16_t *v_res,
                     const uint16_t *q, double sigma, double *out) {
  if (n <= 0 || Hkv <= 0 || Hq % Hkv != 0) return -1;
  int group = Hq / Hkv;
  int64_t rows = (int64_t)B * Hq;
#pragma omp parallel for schedule(dynamic)
  for (int64_t bq = 0; bq < rows; ++bq) {
    int64_t b = bq / Hq;
    int h = (int)(bq % Hq);
    int64_t bh = b * Hkv + h / group;
    oracle_attention_head(D, G, bits, vg, n, KC(bh), KM(bh), KR(bh), VC(bh), VM(bh), VR(bh), q + (size_t)bq * D,
                          sigma, out + (size_t)bq * D);
  }
  return 0;
}

/* R12 for the batch: q [B][Hq][n][D], k, v [B][Hkv][n][D] fp16 -> out [B][Hq][n][D] fp64. */
int oracle_prefill_attention(int B, int Hq, int Hkv, int D, int64_t n, const uint16_t *q, const uint16_t *k,
                             const uint16_t *v, double sigma, double *out) {
  if (n <= 0 || Hkv <= 0 || Hq % Hkv != 0) return -1;
  int group = Hq / Hkv;
  int64_t rows = (int64_t)B * Hq;
#pragma omp parallel for schedule(dynamic)
  for (int64_t bq = 0; bq < rows; ++bq) {
    int64_t b = bq / Hq;
    int h = (int)(bq % Hq);
    int64_t bh = b * Hkv + h / group;
    oracle_prefill_attention_head(D, n, q + (size_t)bq * n * D, k + (size_t)bh * n * D, v + (size_t)bh * n * D,
                                  sigma, out + (size_t)bq * n * D);
  }
  return 0;
}

int oracle_attention_raw(int B, int Hq, int Hkv, int D, int64_t n, const uint16_t *k, const uint16_t *v,
                         const uint16_t *q, double sigma, double *out) {
  if (n <= 0 || Hkv <= 0 || Hq % Hkv != 0) return -1;
  int group = Hq / Hkv;
  int64_t rows = (int64_t)B * Hq;
#pragma omp parallel for schedule(dynamic)
  for (int64_t bq = 0; bq < rows; ++bq) {
    int64_t b = bq / Hq;
    int h = (int)(bq % Hq);
    int64_t bh = b * Hkv + h / group;
    oracle_attention_raw_head(D, n, k + (size_t)bh * n * D, v + (size_t)bh * n * D, q + (size_t)bq * D, sigma,
                              out + (size_t)bq * D);
  }
  return 0;
}
