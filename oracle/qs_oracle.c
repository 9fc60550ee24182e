/*
 * qs_oracle.c -- plain CPU oracle for the QuantSpec hierarchical quantized KV
 * cache hot path.  TEST INFRASTRUCTURE ONLY: the product path never links,
 * loads or calls this file; only the tests, the smoke check and the timed CPU
 * baseline of the benchmark do.
 *
 * Sources (page titles as extracted):
 *  [P3] "QuantSpec: Self-Speculative Decoding with Hierarchical Quantized KV
 *       Cache" (Pith review), section "What carries the argument":
 *       C_INT8 = 2^4 * C_U + C_L, scale and zero-point shared by both levels,
 *       a double full-precision buffer of two halves of G, rejected tokens
 *       dropped before quantization, quantization once every G steps.
 *       Figure 7 caption / Appendix D: keys quantized per channel (group =
 *       G tokens), values per token (group = G channels), asymmetric.
 *       Appendix E: compatible with Flash Decoding.
 *  [P1] "QuantSpec Guide: Self-Speculative Decoding & Quantized KV", section
 *       "1. Hierarchical Quantizer with Bit-Packing": min/max asymmetric
 *       quantization to 255 levels, round, clamp to [0,255], upper = q >> 4,
 *       lower = q & 0xF, draft dequantization at the nibble midpoint (| 0x08).
 *
 * Everything here is written for a reader to check by eye: no blocking, no
 * streaming softmax, no reordering.  Floating point:
 *  - quantization follows the convention QS-RN-v1 (below) in IEEE fp32 with
 *    round-to-nearest-even, exactly as written (compile with
 *    -ffp-contract=off, no fast-math);
 *  - attention is evaluated in fp64 from the stored codes.
 *
 * Convention QS-RN-v1 for one group x_0..x_{n-1} of fp16 values (our reading
 * of the pages, which print no rounding rule for the stored scale):
 *   mn = min x_i, mx = max x_i                         (exact)
 *   r  = fp32(mx) - fp32(mn)                           (fp32, RNE)
 *   s  = r == 0 ? 0 : fp16_round_up(r / 255.0f)        (fp32 RNE divide, then
 *                                                       fp16 toward +inf)
 *   z  = mn  (stored fp16; a zero minimum is stored as +0)
 *   q_i = s == 0 ? 0 : clamp(rne((fp32(x_i) - fp32(z)) / fp32(s)), 0, 255)
 *   C_U = q >> 4, C_L = q & 15
 *   deq8 = s * (16*C_U + C_L) + z,   deqU = s * (16*C_U + 8) + z
 * A draft that reads the top k bits instead of four ([P3], "Editorial
 * extensions", "Reading between the lines" raises other values of k as an
 * open question; only k = 4 is evaluated on the pages) reconstructs, as our
 * reading, at the middle of the 2^(8-k) codes
 * sharing those bits, as the k = 4 midpoint does: with sh = 8 - k,
 *   deqK = s * (2^sh * (q >> sh) + 2^(sh-1)) + z     (k = 2: 64*C_U2 + 32).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define QSO_STATE_WORDS 8
#define QSO_N_GROUPS 0
#define QSO_FILL 1
#define QSO_PENDING 2
#define QSO_HALF_BASE 3
#define QSO_ERR 4

/* device-side error bits (same meaning as the library's) */
#define QSO_DEV_OVERFLOW 1
#define QSO_DEV_OVER_ROLLBACK 2
#define QSO_DEV_FLUSH_UNCOMMITTED 4
#define QSO_DEV_CAPACITY 8
#define QSO_DEV_NQ_GT_FILL 16
#define QSO_DEV_PREFILL 64

/* ------------------------------------------------------------------ fp16 */

/* Exact value of an IEEE binary16 bit pattern. */
double qso_half_to_double(uint16_t h) {
  int sign = h >> 15, e = (h >> 10) & 0x1f, m = h & 0x3ff;
  double v;
  if (e == 0)
    v = ldexp((double)m, -24);
  else if (e == 31)
    v = m ? NAN : INFINITY;
  else
    v = ldexp((double)(m | 0x400), e - 25);
  return sign ? -v : v;
}

/* Round a non-negative double that is an integer-plus-fraction to an integer:
 * mode 0 = nearest, ties to even; mode 1 = toward +inf; mode 2 = toward 0. */
static double round_mode(double n, int mode) {
  double f = floor(n), d = n - f;
  if (mode == 1) return d > 0 ? f + 1 : f;
  if (mode == 2) return f;
  if (d > 0.5) return f + 1;
  if (d < 0.5) return f;
  return fmod(f, 2.0) == 0 ? f : f + 1;
}

/* Encode a finite float as binary16 with the given rounding of the magnitude.
 * Integer-encoding trick: for a >= 2^-14 the bit pattern of the magnitude is
 * (E + 14) * 1024 + n where a = n * 2^(E-10), n in [1024, 2048); below 2^-14
 * it is a / 2^-24.  Both are continuous, so a carry from rounding n up to 2048
 * lands on the next exponent by itself. */
static uint16_t f2h(float f, int to_plus_inf) {
  double x = (double)f; /* exact */
  int neg = signbit(x) != 0;
  double a = fabs(x);
  /* rounding of the magnitude: RN -> nearest-even; RU -> up for positive,
   * toward zero for negative */
  int mode = to_plus_inf ? (neg ? 2 : 1) : 0;
  double hm;
  if (a == 0) {
    hm = 0;
  } else if (a < ldexp(1.0, -14)) {
    hm = round_mode(a / ldexp(1.0, -24), mode);
  } else {
    int ex;
    frexp(a, &ex); /* a = fr * 2^ex, fr in [0.5, 1) -> E = ex - 1 */
    int E = ex - 1;
    double n = a / ldexp(1.0, E - 10);
    hm = (double)(E + 14) * 1024.0 + round_mode(n, mode);
  }
  if (hm >= 0x7C00) hm = (mode == 2) ? 0x7BFF : 0x7C00; /* overflow */
  return (uint16_t)((neg ? 0x8000 : 0) | (uint16_t)hm);
}

uint16_t qso_float_to_half_rn(float f) { return f2h(f, 0); }
uint16_t qso_float_to_half_ru(float f) { return f2h(f, 1); }

/* ------------------------------------------------------------ QS-RN-v1 */

/* Round-half-to-even of a non-negative fp32 value, in fp32 (all steps exact). */
static float rne_f32(float u) {
  float f = floorf(u);
  float d = u - f;
  if (d > 0.5f) return f + 1.0f;
  if (d < 0.5f) return f;
  return (fmodf(f, 2.0f) == 0.0f) ? f : f + 1.0f;
}

/* Quantize one group of n fp16 values x[i * x_stride] to 8-bit codes
 * code[i * code_stride] with one shared scale and zero (convention QS-RN-v1).
 * [P3] Figure 3 / "What carries the argument"; [P1] quantizer section. */
void qso_quantize_group(const uint16_t *x, long x_stride, int n,
                        uint16_t *scale, uint16_t *zero, uint8_t *code,
                        long code_stride) {
  double mn = INFINITY, mx = -INFINITY;
  uint16_t hmn = 0;
  for (int i = 0; i < n; ++i) {
    uint16_t h = x[(long)i * x_stride];
    double v = qso_half_to_double(h);
    if (v < mn) { mn = v; hmn = h; }
    if (v > mx) mx = v;
  }
  if (mn == 0) hmn = 0; /* a zero minimum is stored as +0 */
  float r = (float)mx - (float)mn;
  uint16_t hs = 0;
  if (r != 0.0f) {
    float s32 = r / 255.0f;
    hs = qso_float_to_half_ru(s32);
  }
  *scale = hs;
  *zero = hmn;
  float sf = (float)qso_half_to_double(hs);
  float zf = (float)qso_half_to_double(hmn);
  for (int i = 0; i < n; ++i) {
    uint8_t q = 0;
    if (hs != 0) {
      float xf = (float)qso_half_to_double(x[(long)i * x_stride]);
      float u = (xf - zf) / sf;
      float k = rne_f32(u);
      if (k < 0.0f) k = 0.0f;
      if (k > 255.0f) k = 255.0f;
      q = (uint8_t)k;
    }
    code[(long)i * code_stride] = q;
  }
}

/* Split of an 8-bit code into the two 4-bit levels (truncation, [P1]). */
void qso_split_code(uint8_t q, uint8_t *upper, uint8_t *lower) {
  *upper = (uint8_t)(q >> 4);
  *lower = (uint8_t)(q & 15);
}

/* Dequantized value in fp64: draft_bits = 0, the INT8 code (verify); k in
 * 1..7, the draft's reconstruction from the top k bits (deqK above; k = 4 is
 * 16*C_U + 8). */
double qso_dequant(uint8_t q, uint16_t scale, uint16_t zero, int draft_bits) {
  double s = qso_half_to_double(scale), z = qso_half_to_double(zero);
  double c = (double)q;
  if (draft_bits > 0) {
    int sh = 8 - draft_bits;
    c = (double)((q >> sh) << sh) + (double)(1 << (sh - 1));
  }
  return s * c + z;
}

/* ------------------------------------------------------- cache state */

/* Logical state of one hierarchical cache (all arrays owned by the caller).
 * Codes are stored as full 8-bit values; the two 4-bit levels are q >> 4 and
 * q & 15.  Buffer slot of logical buffer token i is (half_base*G + i) % 2G. */
typedef struct {
  int B, H, D, G, cap;
  uint8_t *kq;       /* [B][H][cap][G tokens][D channels] */
  uint8_t *vq;       /* [B][H][cap][G tokens][D channels] */
  uint16_t *ks, *kz; /* [B][H][cap][D]  per channel */
  uint16_t *vs, *vz; /* [B][H][cap][G]  per token */
  uint16_t *bk, *bv; /* [B][H][2G][D]   fp16 double buffer */
  int32_t *state;    /* [B][QSO_STATE_WORDS] */
} qso_cache;

static long bh(const qso_cache *c, int b, int h) { return (long)b * c->H + h; }

static int32_t *st(const qso_cache *c, int b) {
  return c->state + (long)b * QSO_STATE_WORDS;
}

static long slot_of(const qso_cache *c, int b, int i) {
  return ((long)st(c, b)[QSO_HALF_BASE] * c->G + i) % (2L * c->G);
}

/* Append n_new tokens (k_new, v_new: [B][H][n_new][D] fp16) as pending.
 * [P3] "What carries the argument": new tokens enter the fp16 buffer. */
void qso_append(qso_cache *c, const uint16_t *k_new, const uint16_t *v_new,
                int n_new) {
  for (int b = 0; b < c->B; ++b) {
    int32_t *s = st(c, b);
    if (n_new < 0 || s[QSO_FILL] + n_new > 2 * c->G) {
      s[QSO_ERR] |= QSO_DEV_OVERFLOW;
      continue;
    }
    for (int h = 0; h < c->H; ++h)
      for (int i = 0; i < n_new; ++i) {
        long slot = slot_of(c, b, s[QSO_FILL] + i);
        long dst = (bh(c, b, h) * 2 * c->G + slot) * c->D;
        long src = (bh(c, b, h) * n_new + i) * c->D;
        memcpy(c->bk + dst, k_new + src, sizeof(uint16_t) * c->D);
        memcpy(c->bv + dst, v_new + src, sizeof(uint16_t) * c->D);
      }
    s[QSO_FILL] += n_new;
    s[QSO_PENDING] += n_new;
  }
}

/* Drop the last n_drop[b] pending tokens and commit the rest.
 * [P3]: rejected speculative tokens are dropped before quantization;
 * [P1] "Zero-Overhead Rollback": the quantized cache is never touched. */
void qso_rollback(qso_cache *c, const int32_t *n_drop) {
  for (int b = 0; b < c->B; ++b) {
    int32_t *s = st(c, b);
    int r = n_drop[b];
    if (r < 0 || r > s[QSO_PENDING]) {
      s[QSO_ERR] |= QSO_DEV_OVER_ROLLBACK;
      continue;
    }
    s[QSO_FILL] -= r;
    s[QSO_PENDING] = 0;
  }
}

/* mask[b] = 1 when appending n_next more tokens would overflow 2G. */
void qso_need_flush(const qso_cache *c, int n_next, uint8_t *mask) {
  for (int b = 0; b < c->B; ++b)
    mask[b] = (uint8_t)(st(c, b)[QSO_FILL] + n_next > 2 * c->G);
}

/* Quantize G tokens (kt, vt: [G][D] fp16, token-major) of head h of
 * sequence b into group g: keys per channel over the G tokens, values per
 * token over the D (= G) channels.  [P3] Figure 7 / Appendix D. */
static void quantize_block(qso_cache *c, int b, int h, int g, const uint16_t *kt,
                           const uint16_t *vt) {
  int G = c->G, D = c->D;
  long grp = bh(c, b, h) * c->cap + g;
  uint8_t *kq = c->kq + grp * G * D, *vq = c->vq + grp * G * D;
  for (int d = 0; d < D; ++d) /* keys: one group per channel */
    qso_quantize_group(kt + d, D, G, c->ks + grp * D + d, c->kz + grp * D + d,
                       kq + d, D);
  for (int t = 0; t < G; ++t) /* values: one group per token */
    qso_quantize_group(vt + (long)t * D, 1, D, c->vs + grp * G + t,
                       c->vz + grp * G + t, vq + (long)t * D, 1);
}

/* Quantize the oldest buffer half (G committed tokens) of every masked
 * sequence into group n_groups: keys per channel over the G tokens, values
 * per token over the D (= G) channels.  Then toggle the half and drop G.
 * [P3] "What carries the argument" and Figure 7; [P1] periodic group
 * quantization. */
void qso_flush(qso_cache *c, const uint8_t *mask) {
  int G = c->G, D = c->D;
  for (int b = 0; b < c->B; ++b) {
    if (mask && !mask[b]) continue;
    int32_t *s = st(c, b);
    if (s[QSO_FILL] - s[QSO_PENDING] < G) {
      s[QSO_ERR] |= QSO_DEV_FLUSH_UNCOMMITTED;
      continue;
    }
    if (s[QSO_N_GROUPS] >= c->cap) {
      s[QSO_ERR] |= QSO_DEV_CAPACITY;
      continue;
    }
    int g = s[QSO_N_GROUPS];
    uint16_t *kt = malloc(sizeof(uint16_t) * G * D);
    uint16_t *vt = malloc(sizeof(uint16_t) * G * D);
    for (int h = 0; h < c->H; ++h) {
      /* gather the oldest G logical tokens of the ring */
      for (int i = 0; i < G; ++i) {
        long src = (bh(c, b, h) * 2 * G + slot_of(c, b, i)) * D;
        memcpy(kt + (long)i * D, c->bk + src, sizeof(uint16_t) * D);
        memcpy(vt + (long)i * D, c->bv + src, sizeof(uint16_t) * D);
      }
      quantize_block(c, b, h, g, kt, vt);
    }
    free(kt);
    free(vt);
    s[QSO_N_GROUPS] = g + 1;
    s[QSO_HALF_BASE] ^= 1;
    s[QSO_FILL] -= G;
  }
}

/* Fill empty caches from a prompt in one step.  k, v: [B][H][T][D] fp16;
 * sequence b has len[b] prompt tokens.  The first n_groups * G tokens become
 * groups 0..n_groups-1 (G at a time, in order) and the other fill tokens
 * become committed buffer tokens 0..fill-1 in slots 0..fill-1 (half_base 0),
 * with n_groups = len > 2G ? ceil((len - 2G) / G) : 0, fill = len - G n_groups
 * (so fill is in (G, 2G] once len > 2G).  These are the groups and the logical
 * buffer that appending the prompt in pieces of at most G tokens, with a
 * flush before every append that would overflow 2G, leaves behind.  A
 * sequence whose cache is not empty (n_groups, fill or pending non-zero) or
 * whose length is outside [0, T] gets QSO_DEV_PREFILL and is left unchanged;
 * one that needs more than cap groups gets QSO_DEV_CAPACITY and is left
 * unchanged.  [P1] architectural blueprint (the prefill context is quantized
 * once into the hierarchical cache); [P3] "What carries the argument". */
void qso_prefill(qso_cache *c, const uint16_t *k, const uint16_t *v, int T,
                 const int32_t *len) {
  int G = c->G, D = c->D;
  for (int b = 0; b < c->B; ++b) {
    int32_t *s = st(c, b);
    int L = len[b];
    if (s[QSO_N_GROUPS] != 0 || s[QSO_FILL] != 0 || s[QSO_PENDING] != 0 || L < 0 ||
        L > T) {
      s[QSO_ERR] |= QSO_DEV_PREFILL;
      continue;
    }
    int ng = L > 2 * G ? (L - 2 * G + G - 1) / G : 0;
    if (ng > c->cap) {
      s[QSO_ERR] |= QSO_DEV_CAPACITY;
      continue;
    }
    for (int h = 0; h < c->H; ++h) {
      const uint16_t *kp = k + bh(c, b, h) * T * D, *vp = v + bh(c, b, h) * T * D;
      for (int g = 0; g < ng; ++g)
        quantize_block(c, b, h, g, kp + (long)g * G * D, vp + (long)g * G * D);
      for (int i = 0; i < L - ng * G; ++i) {
        long dst = (bh(c, b, h) * 2 * G + i) * D, src = (long)(ng * G + i) * D;
        memcpy(c->bk + dst, kp + src, sizeof(uint16_t) * D);
        memcpy(c->bv + dst, vp + src, sizeof(uint16_t) * D);
      }
    }
    s[QSO_N_GROUPS] = ng;
    s[QSO_FILL] = L - ng * G;
    s[QSO_PENDING] = 0;
    s[QSO_HALF_BASE] = 0;
  }
}

/* ------------------------------------------------ speculative acceptance */

/* Draw from the distribution proportional to w[0..V-1] (non-negative) by an
 * exponential race: with e_x independent Exp(1) variates, the index of the
 * smallest e_x / w_x over w_x > 0 is distributed as w / sum(w).  Ties go to
 * the smaller index; -1 if every weight is 0.  Each quotient is one IEEE fp32
 * division. */
static int race(const float *w, const float *e, int V) {
  int best = -1;
  float key = 0.0f;
  for (int x = 0; x < V; ++x) {
    if (!(w[x] > 0.0f)) continue;
    float k = e[x] / w[x];
    if (best < 0 || k < key) {
      best = x;
      key = k;
    }
  }
  return best;
}

/* Speculative-sampling verification for B sequences, gamma draft tokens each.
 *   p     [B][gamma+1][V]  target probabilities at the gamma+1 positions
 *   q     [B][gamma][V]    draft probabilities the draft tokens came from
 *   draft [B][gamma]       draft tokens
 *   u     [B][gamma]       uniforms in [0, 1), one per draft token
 *   e     [B][V]           Exp(1) variates for the one draw per sequence
 * Draft token i is accepted when u_i * q_i(x_i) < p_i(x_i) (probability
 * min(1, p_i(x_i) / q_i(x_i))); the first rejection at position a stops the
 * round and the emitted token is drawn from the residual
 * max(0, p_a - q_a) (from p_a if that residual is all zero); with every draft
 * token accepted it is drawn from p_gamma.  A draft token outside [0, V) is
 * rejected.  Outputs: n_accept[b] = a, token[b] (or -1 if the weights are all
 * zero) and n_drop[b] = gamma - a (the rollback count of the synthetic round).
 * Pith review page, referee report on Algorithm 1 (VERIFY / CORRECT as
 * rejection sampling with acceptance min(1, p/q) and residual (p - q)_+);
 * [P1] "The Self-Speculative Verification Loop" (acceptance test, stop at
 * the first rejection). */
void qso_spec_accept(const float *p, const float *q, const int32_t *draft,
                     const float *u, const float *e, int B, int gamma, int V,
                     int32_t *n_accept, int32_t *token, int32_t *n_drop) {
  float *w = malloc(sizeof(float) * (size_t)V);
  for (int b = 0; b < B; ++b) {
    const float *pb = p + (size_t)b * (gamma + 1) * V;
    const float *qb = q + (size_t)b * gamma * V;
    int a = 0;
    while (a < gamma) {
      int x = draft[(size_t)b * gamma + a];
      float pa = (x >= 0 && x < V) ? pb[(size_t)a * V + x] : 0.0f;
      float qa = (x >= 0 && x < V) ? qb[(size_t)a * V + x] : 0.0f;
      if (x < 0 || x >= V || !(u[(size_t)b * gamma + a] * qa < pa)) break;
      ++a;
    }
    const float *eb = e + (size_t)b * V;
    int t;
    if (a < gamma) {
      const float *pr = pb + (size_t)a * V, *qr = qb + (size_t)a * V;
      for (int x = 0; x < V; ++x) {
        float d = pr[x] - qr[x];
        w[x] = d > 0.0f ? d : 0.0f;
      }
      t = race(w, eb, V);
      if (t < 0) t = race(pr, eb, V);
    } else {
      t = race(pb + (size_t)gamma * V, eb, V);
    }
    n_accept[b] = a;
    token[b] = t;
    n_drop[b] = gamma - a;
  }
  free(w);
}

/* -------------------------------------------------------------- attention */

/* Decode attention in fp64 for every (b, h) and each of n_q queries of each
 * of the `group` query heads that share KV head h (grouped-query attention;
 * group = 1 is multi-head): q is [B][H*group][n_q][D] fp16, query head
 * h*group + i reads KV head h.  Keys/values are the dequantized groups
 * (draft_bits = k > 0: draft from the top k bits, deqK; 0: verify, INT8)
 * followed by the fp16
 * buffer tokens.  Query j sits at the position of buffer token
 * fill - n_q + j and sees every token at or before it.  Writes
 * out [B][H*group][n_q][D] and lse [B][H*group][n_q] (natural log of the
 * softmax denominator of the scaled scores).  A sequence with n_q > fill gets
 * QSO_DEV_NQ_GT_FILL, zero output and lse = -inf.
 * [P1] "Hierarchical Two-Level Quantization" (draft loads upper 4 bits,
 * target reconstructs INT8); [P3] "What carries the argument". */
void qso_attn(qso_cache *c, int draft_bits, const uint16_t *q, int n_q, int group,
              double scale, double *out, double *lse) {
  int G = c->G, D = c->D;
  for (int b = 0; b < c->B; ++b)
    if (n_q > st(c, b)[QSO_FILL]) st(c, b)[QSO_ERR] |= QSO_DEV_NQ_GT_FILL;
#pragma omp parallel for collapse(2) schedule(dynamic)
  for (int b = 0; b < c->B; ++b)
    for (int h = 0; h < c->H; ++h) {
      const int32_t *s = st(c, b);
      int ng = s[QSO_N_GROUPS], fill = s[QSO_FILL];
      long Tq = (long)ng * G, T = Tq + fill;
      long o = bh(c, b, h) * group * n_q; /* rows of query heads h*group.. */
      if (n_q > fill) {
        for (int j = 0; j < group * n_q; ++j) {
          for (int d = 0; d < D; ++d) out[(o + j) * D + d] = 0.0;
          lse[o + j] = -INFINITY;
        }
        continue;
      }
      double *K = malloc(sizeof(double) * T * D);
      double *V = malloc(sizeof(double) * T * D);
      for (long t = 0; t < Tq; ++t) {
        long g = t / G, i = t % G;
        long grp = bh(c, b, h) * c->cap + g;
        for (int d = 0; d < D; ++d) {
          K[t * D + d] = qso_dequant(c->kq[(grp * G + i) * D + d],
                                     c->ks[grp * D + d], c->kz[grp * D + d],
                                     draft_bits);
          V[t * D + d] = qso_dequant(c->vq[(grp * G + i) * D + d],
                                     c->vs[grp * G + i], c->vz[grp * G + i],
                                     draft_bits);
        }
      }
      for (int i = 0; i < fill; ++i) {
        long src = (bh(c, b, h) * 2 * G + slot_of(c, b, i)) * D;
        for (int d = 0; d < D; ++d) {
          K[(Tq + i) * D + d] = qso_half_to_double(c->bk[src + d]);
          V[(Tq + i) * D + d] = qso_half_to_double(c->bv[src + d]);
        }
      }
      double *S = malloc(sizeof(double) * T);
      for (int gj = 0; gj < group * n_q; ++gj) {
        int j = gj % n_q; /* query head h*group + gj / n_q, position j */
        const uint16_t *qj = q + (o + gj) * D;
        long last = Tq + fill - n_q + j; /* causal limit */
        double m = -INFINITY;
        for (long t = 0; t <= last; ++t) {
          double acc = 0;
          for (int d = 0; d < D; ++d)
            acc += qso_half_to_double(qj[d]) * K[t * D + d];
          S[t] = scale * acc;
          if (S[t] > m) m = S[t];
        }
        /* softmax weights w_t = exp(S_t - m) / l, then o = sum_t w_t v_t */
        double l = 0;
        for (long t = 0; t <= last; ++t) {
          S[t] = exp(S[t] - m);
          l += S[t];
        }
        double *oj = out + (o + gj) * D;
        for (int d = 0; d < D; ++d) oj[d] = 0.0;
        for (long t = 0; t <= last; ++t)
          for (int d = 0; d < D; ++d) oj[d] += S[t] * V[t * D + d];
        for (int d = 0; d < D; ++d) oj[d] /= l;
        lse[o + gj] = m + log(l);
      }
      free(S);
      free(K);
      free(V);
    }
}

/* Number of OpenMP threads the attention loop uses (1 without OpenMP). */
int qso_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
