// qs_attn.cu -- split-KV decode attention over the hierarchical quantized KV
// cache (draft: C_U only, or C_U2 in the two-bit layout; verify: INT8 =
// 16 C_U + C_L) plus the fp16 buffer, with the log-sum-exp combine of the
// splits in the same kernel.
//
// Sources: "QuantSpec Guide: Self-Speculative Decoding & Quantized KV",
// "1. Hierarchical Two-Level Quantization with Bit-Sharing" (draft loads only
// the upper 4 bits from HBM, target reconstructs INT8 from both) and the
// quantizer listing (draft reconstruction at the nibble midpoint);
// "QuantSpec: Self-Speculative Decoding with Hierarchical Quantized KV Cache"
// (Pith review), "What carries the argument" and Appendix E (the buffer design
// works with Flash Decoding: split-KV partial softmax, then an LSE combine).
//
// Design (GB300):
//  * One persistent CTA of twelve warps per SM (eight for a verify tile of
//    at most 16 rows).  All (sequence, head)
//    segments are laid end to end as units (a quantized group of 128 tokens,
//    or a chunk of fp16 buffer tokens) and every CTA takes an equal
//    contiguous range, so ragged batches balance without a host round trip.
//  * Each unit's contiguous plane blocks arrive by bulk async copies
//    (cp.async.bulk, TMA engine) in a ring of shared-memory stages guarded by
//    mbarriers; draft units copy only the C_U planes (8 KB keys + 8 KB values
//    + 1 KB scales/zeros; 4 + 4 + 1 KB for the two-bit draft).  There is no
//    producer warp: the last warp to finish
//    with a stage (a shared-memory arrival counter) issues its refill, so all
//    twelve warps compute.
//  * Warps claim half-units (64 tokens of a group) from a shared counter, so
//    the SM's warps finish together; per-unit fixed costs amortize over 64
//    tokens.  Codes become subnormal fp16 operands (code * 2^-24) by masks
//    and byte permutes, no conversion instructions, and the dense
//    contractions q.K^T and P.V run on m16n8k16 tensor-core MMAs with fp32
//    accumulation (the 2^-24 returns in the fp32 scales).  Scales are folded:
//    B = q * s_K per channel, P' = p * s_V per token, zero-point terms as
//    per-query biases, so the inner loops touch codes only.
//  * Each warp keeps its own online softmax and writes one partial per piece
//    of a segment it touches.  At the end of its range the CTA merges its
//    warps' partials (log-sum-exp); a segment split across CTAs is
//    finished by whichever of them arrives last on the segment's counter,
//    so the whole call is one kernel launch.
#include <math.h>

#include "qs_common.cuh"

namespace qs {
namespace {

constexpr int kPairs = 6;               // units in compute at once (two half-units each)
constexpr int kMaxR = 24;              // query rows per KV head (three column groups of 8)
constexpr int kWarps = 2 * kPairs;
// A verify tile of at most 16 rows (one or two column groups) runs with
// eight warps: its ring (six stages of 34 KB, all the shared memory) then
// holds four units in compute and two in flight instead of six in compute
// and none in flight, and 256 threads may hold 255 registers each, so the
// five-query tile does not spill (32k: 63 against 71 µs per call; 128k:
// 175 against 192).  Three column groups keep twelve warps (four per group).
constexpr int kVerifyWarps = 8;
// fp16 row stride (bytes) of a buffer tile in shared memory.  Rows padded
// by 16 bytes are read without bank conflicts but take one copy per row;
// unpadded rows arrive in one copy per plane.
template <bool PAD>
constexpr int tail_row() { return PAD ? 272 : 256; }
constexpr int kOffKU = 0, kOffVU = 8192, kOffMeta = 16384, kOffKL = 17408, kOffVL = 25600;

template <int MODE>
struct Cfg;
template <>
struct Cfg<QS_DRAFT_UPPER4> {
  static constexpr int kGroupBytes = 8192 + 8192 + 1024;
  static constexpr int kTailTok = 32;
  static constexpr int kStages = 2 * kPairs;  // about one unit in flight per unit in compute
};
template <>
struct Cfg<QS_VERIFY_INT8> {
  static constexpr int kGroupBytes = 4 * 8192 + 1024;
  static constexpr int kTailTok = 64;
  static constexpr int kStages = kPairs;
};

constexpr int align16(int x) { return (x + 15) & ~15; }

template <int MODE>
struct Layout {
  static constexpr int kTailBytes = Cfg<MODE>::kTailTok * tail_row<true>() * 2;
  static constexpr int kStageBytes =
      Cfg<MODE>::kGroupBytes > kTailBytes ? Cfg<MODE>::kGroupBytes : kTailBytes;
  static constexpr int kBarOff = Cfg<MODE>::kStages * kStageBytes;               // full barriers
  static constexpr int kCntOff = align16(kBarOff + 8 * Cfg<MODE>::kStages);      // release counters
  static constexpr int kIssOff = align16(kCntOff + 4 * Cfg<MODE>::kStages);      // unit per stage
  static constexpr int kZeroOff = align16(kIssOff + 4 * Cfg<MODE>::kStages);     // zero row (ldmatrix)
  static constexpr int kMrgOff = kZeroOff + 32;  // barrier of the finishing merge's copies
  static constexpr int kTabOff = kMrgOff + 16;
  // per-sequence tables: n_groups, fill, half_base, segment length, base
  // unit, first segment ordinal, fill before a fused append
  static constexpr int kSmemBytes = kTabOff + 7 * kMaxB * 4;
  static_assert(kStageBytes % 16 == 0 && kBarOff % 16 == 0 && kZeroOff % 16 == 0,
                "bulk copies and ldmatrix rows need 16-byte aligned shared memory");
};

struct Params {
  qs_cache c;
  const uint16_t *q;
  uint16_t *out;
  float *lse;
  float *ws;
  int n_q;    // query positions (causal, the last n_q buffer tokens)
  int R;      // query rows per KV head: group * n_q (row r: query head r / n_q,
              // position r % n_q)
  int ncg;    // column groups of eight rows, ceil(R / 8): warp w serves group w % ncg
  int P;      // split-kernel grid size (number of contiguous unit ranges)
  float sl2;  // softmax_scale * log2(e)
  uint64_t wait_ns;  // limit on each pipeline wait (kWaitLimitNs outside tests)
  int no_issue;      // test entry only: issue no copy, so that every wait runs out
  // append fused in front of the attention (n_new > 0): fp16 [B][H][n_new][D]
  // tokens that enter the buffer before the queries attend
  const uint16_t *k_new, *v_new;
  int n_new;
  size_t ws_floats;  // workspace size (the checked build bounds its indexing by it)
};

struct Tables {
  int *ng, *fill, *hb, *len, *base;  // base in units, len in units per head
  int *ord0;  // ordinal of (b, head 0) among the segments that have units
  int *fold;  // buffered tokens before a fused append (fill - n_new, or fill)
};

__device__ __forceinline__ Tables tables_at(uint8_t *smem, int off) {
  int *t = reinterpret_cast<int *>(smem + off);
  return Tables{t, t + kMaxB, t + 2 * kMaxB, t + 3 * kMaxB, t + 4 * kMaxB, t + 5 * kMaxB,
                t + 6 * kMaxB};
}

// Warp-cooperative: read counters, segment lengths (units per head), the
// exclusive prefix of units (x H) and the ordinal of each sequence's first
// segment (segments of sequences without units are skipped) into the tables.
// With a fused append of n_new tokens, a sequence whose buffer can take them
// attends over fill + n_new tokens (the others over fill: their append fails,
// as a separate append would).  Returns the total number of units.
template <int TT>
__device__ long long build_tables(const qs_cache &c, int n_q, int n_new, Tables T, int lane) {
  const int per = (c.B + 31) / 32;
  const int b0 = lane * per;
  int local = 0, local_ne = 0;
  for (int i = 0; i < per; ++i) {
    const int b = b0 + i;
    if (b < c.B) {
      const int32_t *st = c.state + (size_t)b * QS_STATE_WORDS;
      // clamped so that no counter value can address outside the arrays
      const int ng = min(max(st[QS_ST_N_GROUPS], 0), c.cap_groups);
      const int fill_raw = st[QS_ST_FILL];
      const int fold = min(max(fill_raw, 0), kRing);
      const int fill = (n_new > 0 && fill_raw >= 0 && fill_raw + n_new <= kRing) ? fold + n_new : fold;
      T.ng[b] = ng;
      T.fill[b] = fill;
      T.fold[b] = fold;
      T.hb[b] = st[QS_ST_HALF_BASE] & 1;
      const int len = (n_q <= fill) ? ng + (fill + TT - 1) / TT : 0;
      T.len[b] = len;
      local += len;
      local_ne += len > 0;
    }
  }
  int incl = local, incl_ne = local_ne;
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    const int v_ne = __shfl_up_sync(0xffffffffu, incl_ne, o);
    if (lane >= o) { incl += v; incl_ne += v_ne; }
  }
  long long run = (long long)(incl - local) * c.H;
  int run_ne = (incl_ne - local_ne) * c.H;
  for (int i = 0; i < per; ++i) {
    const int b = b0 + i;
    if (b < c.B) {
      T.base[b] = (int)run;
      T.ord0[b] = run_ne;
      run += (long long)T.len[b] * c.H;
      run_ne += T.len[b] > 0 ? c.H : 0;
    }
  }
  return (long long)__shfl_sync(0xffffffffu, incl, 31) * c.H;
}

// CTA p owns units [range_lo(p), range_lo(p + 1)): floor(p U / P) onwards
// when there are at least as many units as CTAs, else unit p alone (CTAs
// p >= U idle).  Either way every CTA between a segment's first and last
// owner owns part of it.
__device__ __forceinline__ long long range_lo(int p, long long U, int P) {
  if (U < P) return p < U ? p : U;
  if (U * P < (1ll << 32))  // 32-bit division (p <= P)
    return (long long)((uint32_t)p * (uint32_t)U / (uint32_t)P);
  return (long long)p * U / P;
}
// The CTA whose range holds unit x.
__device__ __forceinline__ int cta_of(long long x, long long U, int P) {
  if (U < P) return (int)x;
  if (U * P < (1ll << 32))  // 32-bit division
    return (int)(((uint32_t)(x + 1) * (uint32_t)P - 1u) / (uint32_t)U);
  return (int)(((x + 1) * P - 1) / U);
}

// Where unit x lies: sequence b, head h, unit u of the (b, h) segment, whose
// first unit is s0 and whose ordinal among the segments with units is ord.
// seek() costs a compare while x stays in the current segment.
struct Seg {
  int b = -1, h = 0, u = 0, s0 = 0, len = 0, ord = 0;
  __device__ void seek(int x, const Tables &T, int B) {
    if (b >= 0 && x >= s0 && x < s0 + len) {
      u = x - s0;
      return;
    }
    int lo = 0, hi = B - 1;  // largest b with base[b] <= x (that one has units)
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (T.base[mid] <= x) lo = mid; else hi = mid - 1;
    }
    b = lo;
    len = T.len[b];
    const int off = x - T.base[b];
    h = off / len;
    s0 = T.base[b] + h * len;
    u = x - s0;
    ord = T.ord0[b] + h;
  }
};

// ---- nibble / byte planes -> exact fp16 operands (half2 per pair) --------
// Pair p of a 32-bit word holds elements (p, p + 4) of its 8 nibbles.  A code
// placed in the low mantissa bits of an fp16 whose exponent field is zero is
// the subnormal code * 2^-24, exactly, so a mask (and a byte permute or one
// shift for the other half of the word) is the whole conversion: no offset
// and no subtraction.  The tensor core multiplies these exactly and sums in
// fp32, where code * 2^-24 * B is a normal number; the 2^-24 comes back in
// the fp32 score and output scales.
//
// Verify: the 8-bit code C_INT8 = 16 C_U + C_L, every element c * 2^-24.
__device__ __forceinline__ void pairs_int8(uint32_t wu, uint32_t wl, uint32_t (&e)[4]) {
  const uint32_t ev = bitsel(wl, wu << 4, 0x0F0F0F0Fu);   // codes 0,2,4,6
  const uint32_t od = bitsel(wl >> 4, wu, 0x0F0F0F0Fu);   // codes 1,3,5,7
  e[0] = prmt(ev, 0u, 0x4240);  // bytes 0 and 2 over zero high bytes
  e[1] = prmt(od, 0u, 0x4240);
  e[2] = prmt(ev, 0u, 0x4341);
  e[3] = prmt(od, 0u, 0x4341);
}

// Draft: the nibble C_U stays where it is.  Even elements (pairs 0 and 2)
// sit in bits 0-3 of their half (C_U * 2^-24), odd ones (pairs 1 and 3) in
// bits 4-7 (16 C_U * 2^-24): one shift and four masks per word.  The factor
// 16 of the odd elements is taken out of their other operand (B = q * s_K / 16
// for keys, P' / 16 for values), so every product is C_U * 2^-24 * B.
__device__ __forceinline__ void pairs_upper(uint32_t w, uint32_t (&e)[4]) {
  const uint32_t t = w >> 8;
  e[0] = w & 0x000F000Fu;
  e[1] = w & 0x00F000F0u;
  e[2] = t & 0x000F000Fu;
  e[3] = t & 0x00F000F0u;
}

// Fixed parts of the dequantized value, in units of the scale, that go into
// the zero-point biases (fp32).  Codes enter the contractions uncentred
// (draft 16 C_U, verify C_INT8).  Values are centred on 128 all the same: an
// MMA of ones against the same fp16 P' the codes are multiplied with takes
// 128 * sum_t P'_t out of the product, so the fp16 rounding of p * s_V acts
// on s * (code - 128), of the size of the data, instead of on the distance
// to the group minimum; the bias then carries 128 + the draft's midpoint 8.
// Keys need no centring (q * s_K is carried hi + lo to ~2^-22): the bias
// carries the midpoint alone.
// UB: the top bits the draft reads (4: 16 C_U + 8; 2: 64 C_U2 + 32).
template <int MODE, int UB = 4>
struct Centre {
  static constexpr bool kDraft = MODE == QS_DRAFT_UPPER4;
  static constexpr float kStep = UB == 2 ? 64.f : 16.f;  // draft code step
  static constexpr float kOff = kDraft ? 128.f + kStep / 2 : 128.f;  // values
  static constexpr float kOffK = kDraft ? kStep / 2 : 0.f;           // keys
  static constexpr float kMid = 128.f;  // taken out of the value product
  // true code sum / tensor-core sum: 2^24 (subnormal codes), times the
  // draft's code step
  static constexpr float kScale = 16777216.f * (kDraft ? kStep : 1.f);
};

template <int MODE>
__device__ __forceinline__ void pairs(uint32_t wu, uint32_t wl, uint32_t (&e)[4]) {
  if (MODE == QS_DRAFT_UPPER4) pairs_upper(wu, e);
  else pairs_int8(wu, wl, e);
}

// Two-bit draft layout (see include/qs.h): word k of the C_U2 plane holds
// the top two bits of nibble j of 4-bit words 2k (bits 4j..4j+1) and 2k+1
// (bits 4j+2..4j+3).  The draft converts them as pairs_upper converts
// nibbles, with C_U2 in place of C_U (field sh = 0 for word 2k, 2 for 2k+1):
// even elements C_U2 * 2^-24, odd ones 16 C_U2 * 2^-24.
template <int SH>
__device__ __forceinline__ void pairs_upper2(uint32_t x, uint32_t (&e)[4]) {
  const uint32_t w = x >> SH, t = x >> (SH + 8);
  e[0] = w & 0x00030003u;
  e[1] = w & 0x00300030u;
  e[2] = t & 0x00030003u;
  e[3] = t & 0x00300030u;
}
__device__ __forceinline__ void pairs_upper2_rt(uint32_t x, int sh, uint32_t (&e)[4]) {
  const uint32_t w = x >> sh, t = w >> 8;
  e[0] = w & 0x00030003u;
  e[1] = w & 0x00300030u;
  e[2] = t & 0x00030003u;
  e[3] = t & 0x00300030u;
}
// Verify: the 4-bit word 2k + sh/2 rebuilt from C_U2 word u and M2 word m
// (C_U = 4 C_U2 + M2).
__device__ __forceinline__ uint32_t upper_from2(uint32_t u, uint32_t m, int sh) {
  return ((u << (2 - sh)) & 0xCCCCCCCCu) | ((m >> sh) & 0x33333333u);
}

__device__ __forceinline__ uint32_t lds32(uint32_t a) {
  if (!chk(smem_in(a, 4), 1)) return 0;
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t a) {
  if (!chk(smem_in(a, 8), 1)) return make_uint2(0, 0);
  uint2 v;
  asm volatile("ld.shared.v2.b32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
  return v;
}
__device__ __forceinline__ uint4 lds128(uint32_t a) {
  if (!chk(smem_in(a, 16), 1)) return make_uint4(0, 0, 0, 0);
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(a));
  return v;
}

// Probabilities are taken as 2^(s - m + kExpShift): values up to 64 keep p * s_V
// in the normal fp16 range for the tensor-core operand (far-down tokens of a
// long, diffuse context would otherwise round as fp16 subnormals) while any
// finite fp16 value scale (< 2^10) stays below the fp16 maximum.  The shift
// cancels in O / l; partials store m - kExpShift.
constexpr float kExpShift = 6.f;

// Per-warp online-softmax state for its two queries (columns 2c, 2c+1).
struct Softmax {
  float m[2], l[2], bv[2];
  // O^T accumulators: rows = channels 16 md + r (+8), cols = queries; in
  // tensor-core units (true O / Centre::kScale), the value bias kept apart
  float o[8][4];
  __device__ void reset() {
#pragma unroll
    for (int i = 0; i < 2; ++i) { m[i] = -INFINITY; l[i] = 0.f; bv[i] = 0.f; }
#pragma unroll
    for (int md = 0; md < 8; ++md)
#pragma unroll
      for (int k = 0; k < 4; ++k) o[md][k] = 0.f;
  }
  // New maximum from this step's warp-wide maxima: rescales l and the value
  // bias, returns the factors a0, a1 for O (applied when the step's P.V is
  // merged) and the offsets u0, u1 to subtract from the scores.
  __device__ void update(float g0, float g1, float &u0, float &u1, float &a0, float &a1) {
    const float n0 = fmaxf(m[0], g0), n1 = fmaxf(m[1], g1);
    a0 = (n0 == -INFINITY) ? 1.f : fast_exp2(m[0] - n0);
    a1 = (n1 == -INFINITY) ? 1.f : fast_exp2(m[1] - n1);
    u0 = (n0 == -INFINITY) ? 0.f : n0 - kExpShift;
    u1 = (n1 == -INFINITY) ? 0.f : n1 - kExpShift;
    m[0] = n0;
    m[1] = n1;
    l[0] *= a0; l[1] *= a1; bv[0] *= a0; bv[1] *= a1;
  }
  // O = a * O + D for one 16-channel tile: each step's P.V starts from a zero
  // accumulator, so no tensor-core accumulation chain spans more than a group.
  __device__ __forceinline__ void merge(int md, const float (&d)[4], float a0, float a1) {
    o[md][0] = fmaf(o[md][0], a0, d[0]);
    o[md][1] = fmaf(o[md][1], a1, d[1]);
    o[md][2] = fmaf(o[md][2], a0, d[2]);
    o[md][3] = fmaf(o[md][3], a1, d[3]);
  }
};

__device__ __forceinline__ float warp_max8(float v) {  // over lanes sharing lane & 3
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
  return v;
}
__device__ __forceinline__ float warp_sum8(float v) {
  v += __shfl_xor_sync(0xffffffffu, v, 4);
  v += __shfl_xor_sync(0xffffffffu, v, 8);
  v += __shfl_xor_sync(0xffffffffu, v, 16);
  return v;
}

// q row of query r as tensor-core B pairs in the key-plane channel order:
// k-block kb, first register {q(ch0), q(ch0+4)}, second {q(ch0+1), q(ch0+5)},
// ch0 = 32c + 8 (kb >> 1) + 2 (kb & 1).
__device__ __forceinline__ void load_q_pairs(const uint16_t *qrow, bool valid, int c,
                                             uint32_t (&q0)[8], uint32_t (&q1)[8]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint4 w = make_uint4(0, 0, 0, 0);
    if (valid) w = __ldg(reinterpret_cast<const uint4 *>(qrow + 32 * c) + i);
    q0[2 * i] = prmt(w.x, w.z, 0x5410);
    q1[2 * i] = prmt(w.x, w.z, 0x7632);
    q0[2 * i + 1] = prmt(w.y, w.w, 0x5410);
    q1[2 * i + 1] = prmt(w.y, w.w, 0x7632);
  }
}

// ------------------------------------------------------------ split kernel

// Issue the bulk copies of one unit into a stage (called by one whole warp).
// A two-bit draft copies only the C_U2 half (4 KB) of each upper plane into
// the stage's upper slots; verify copies both halves (the slots' layout is
// then C_U2 | M2 instead of C_U).
__device__ __forceinline__ uint8_t *prm_smem_base() {
  extern __shared__ __align__(128) uint8_t qs_dyn_smem[];
  return qs_dyn_smem;
}

// With a fused append, buffer rows at or past the old fill come straight
// from the appended tokens (the ring gets them in the same launch, not read
// back here).
template <int MODE, int UB, bool PAD>
__device__ __forceinline__ void issue_unit(const Params &prm, const Tables &T, const Seg &cu,
                                           uint32_t dst, uint32_t bar, int lane) {
  const qs_cache &c = prm.c;
  using C = Cfg<MODE>;
  constexpr int TT = C::kTailTok;
  static_assert(kG % TT == 0 && kRing % TT == 0, "a buffer chunk must not straddle the ring end");
  const size_t bh = (size_t)cu.b * c.H + cu.h;
  const int ng = T.ng[cu.b];
  if (cu.u < ng) {
    if (lane == 0) {
      size_t grp = bh * c.cap_groups + cu.u;
      // checked build: a copy out of bounds reads group 0 (and lands in the
      // stage's start) instead, so its barrier still completes
      if (!chk(in_range(grp, 1, (size_t)c.B * c.H * c.cap_groups), 3)) grp = 0;
      if (!chk(smem_in(dst, C::kGroupBytes), 2)) dst = smem_addr(prm_smem_base());
      const uint64_t pol = l2_evict_first_policy();  // planes are read once per call
      constexpr int kUp = (MODE == QS_DRAFT_UPPER4 && UB == 2) ? 4096 : 8192;
      mbar_arrive_expect_tx(bar, C::kGroupBytes - 2 * (8192 - kUp));
      bulk_g2s_hint(dst + kOffKU, c.k_upper + grp * 8192, kUp, bar, pol);
      bulk_g2s_hint(dst + kOffVU, c.v_upper + grp * 8192, kUp, bar, pol);
      bulk_g2s_hint(dst + kOffMeta, c.meta + grp * 512, 1024, bar, pol);
      if (MODE == QS_VERIFY_INT8) {
        bulk_g2s_hint(dst + kOffKL, c.k_lower + grp * 8192, 8192, bar, pol);
        bulk_g2s_hint(dst + kOffVL, c.v_lower + grp * 8192, 8192, bar, pol);
      }
    }
  } else {
    // A buffer chunk: rows fp16 rows of K, then of V.  The rows before the
    // old fill are consecutive ring slots (a chunk starts at a multiple of
    // its size from the half base, so it wraps to the ring's start whole or
    // not at all); rows from the appended tokens follow.
    constexpr int kRow = tail_row<PAD>();
    const int i0 = (cu.u - ng) * TT;
    const int rows = min(TT, T.fill[cu.b] - i0);
    const int fold = T.fold[cu.b];
    const int slot0 = (T.hb[cu.b] * kG + i0) & (kRing - 1);
    // unpadded: one bulk copy each for the K and V ring rows (the copy
    // engine spends about as long on a 256-byte copy as on an 8 KB one);
    // padded: one copy per row
    const int n_bulk = PAD ? 0 : max(0, min(rows, fold - i0));
    if (lane == 0) {
      mbar_arrive_expect_tx(bar, rows * 2 * kD * 2);
      if (n_bulk > 0) {
        size_t r0 = bh * kRing + slot0;
        // checked build: rows out of the ring read row 0 instead
        if (!chk(in_range(r0, n_bulk, (size_t)c.B * c.H * kRing), 4)) r0 = 0;
        uint32_t dk = dst, dv = dst + TT * kRow;
        if (!chk(smem_in(dv, n_bulk * kRow), 2)) dk = dv = smem_addr(prm_smem_base());
        bulk_g2s(dk, c.buf_k + r0 * kD, n_bulk * kRow, bar);
        bulk_g2s(dv, c.buf_v + r0 * kD, n_bulk * kRow, bar);
      }
    }
    __syncwarp();
    const int n_rest = rows - n_bulk;
    for (int rr = lane; rr < 2 * n_rest; rr += 32) {
      const bool isv = rr >= n_rest;
      const int row = n_bulk + (isv ? rr - n_rest : rr);
      const uint16_t *src;
      if (i0 + row < fold) {
        size_t ri = bh * kRing + slot0 + row;
        if (!chk(in_range(ri, 1, (size_t)c.B * c.H * kRing), 4)) ri = 0;
        src = (isv ? c.buf_v : c.buf_k) + ri * kD;
      } else {
        size_t rn = bh * prm.n_new + (i0 + row - fold);
        if (!chk(in_range(rn, 1, (size_t)c.B * c.H * prm.n_new), 4)) rn = 0;
        src = (isv ? prm.v_new : prm.k_new) + rn * kD;
      }
      uint32_t d = dst + (isv ? TT * kRow : 0) + row * kRow;
      if (!chk(smem_in(d, kD * 2), 2)) d = smem_addr(prm_smem_base());
      bulk_g2s(d, src, kD * 2, bar);
    }
  }
}

// Each merge splits a row's partials over up to QS_MERGE_KS adjacent lanes
// (1: one lane per row and four channels).  Measured on the 32k step: 8
// against 1, 215.0 against 215.9 us per step, isolated draft 45.7 against 47.5.
#ifndef QS_MERGE_KS
#define QS_MERGE_KS 8
#endif

// Device-scope fence: in the rare case where a CTA finishes the segment of
// its shared first piece, between the arrival (made mid-range by one lane)
// and the whole CTA's reads of the other CTAs' partials.
__device__ __forceinline__ void fence_gpu() { __threadfence(); }

// Atomic add with acquire and release semantics at CTA scope (a count of
// the CTA's warps in shared memory).
__device__ __forceinline__ int atom_add_acq_rel_cta(int *p, int v) {
  int old;
  asm volatile("atom.add.acq_rel.cta.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Global memory written through ordinary stores (and acquired) is read next
// by bulk copies.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// ------------------------------------------------------- log-sum-exp merge
// Merge of ns partials of one (sequence, head): partial k < nA starts at
// srcA + k * kstrideA floats, partial k >= nA at srcB + (k - nA) * kstrideB.
// Each holds, for each query j < n_q, the unnormalized O_j[d] at j * 128 + d,
// then m_j (log2 domain) at n_q * 128 + j and l_j at n_q * 128 + 8 + j:
//   M_j = max_k m_kj,  L_j = sum_k 2^(m_kj - M_j) l_kj,
//   O_j = sum_k 2^(m_kj - M_j) O_kj.
// final: out_j = O_j / L_j (fp16) and lse_j = (M_j + log2 L_j) ln 2; else the
// merged partial is written to dst (same layout; dst may be partial 0 of the
// sources).  A partial with m = -inf is empty (its l and O are not read into
// the sums; they may be stale).
struct MergeOut {
  bool final;
  uint16_t *out;  // final: fp16 [n_q][128] of this (sequence, head)
  float *lse;     // final: [n_q] or null
  float *dst;     // partial
};

// Loads of partials through generic addresses (shared memory, or global
// memory written by other CTAs: volatile, so never served from a stale L1 line).
__device__ __forceinline__ float ld_part(const float *p) {
  float v;
  asm volatile("ld.volatile.f32 %0, [%1];" : "=f"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ float4 ld_part4(const float *p) {
  float4 v;
  asm volatile("ld.volatile.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p));
  return v;
}

// Row-parallel merge of ns partials.  An item is (row j, four channels): with
// QS_MERGE_KS > 1 and few rows, the partials of an item are split over ks
// adjacent lanes (as many as the CTA's threads allow, at most QS_MERGE_KS),
// which combine their (M, L, O) by shuffles at the end; with QS_MERGE_KS = 1
// one warp takes a row, its lanes four channels each.  Each lane loads a
// batch of partials (m, l and its four channels of O) at once, all in flight
// before the first is used, and folds them into a running (M, L, O) with one
// rescale per batch: no shared-memory scratch and no barrier.  Row j's
// partials start at srcA + (j / 8) * cgA (and srcB + (j / 8) * cgB): warp
// partials hold only the rows of their warp's column group.  dst never
// overlaps the sources (a CTA partial is made only of a range's last piece,
// whose warp partials are in shared memory).  Not inlined: it runs once or
// twice per launch, at the end, where every instruction is fetched cold, so
// one small shared copy matters more than the call.
// Partials per batch of one lane's loads, and the lanes ks that share an
// item (row j, four channels) of R * 32 items: as many as the CTA's threads
// allow, at most QS_MERGE_KS.
constexpr int kMergeBatch = QS_MERGE_KS > 1 ? 4 : 8;
__device__ __forceinline__ int merge_split(int R) {
  int ks = 1;
  while (ks < QS_MERGE_KS && R * 32 * ks * 2 <= (int)blockDim.x) ks *= 2;
  return ks;
}
// Dependent rounds of loads a merge of ns partials takes: passes over the
// items times batches per lane.
__device__ __forceinline__ int merge_rounds(int R, int ns) {
  const int ks = merge_split(R);
  return (R * 32 * ks + (int)blockDim.x - 1) / (int)blockDim.x *
         ((ns + ks * kMergeBatch - 1) / (ks * kMergeBatch));
}

#if QS_MERGE_KS > 1
__device__ __noinline__ void merge_rows(const float *srcA, int cgA, int kstrideA, int nA,
                                        const float *srcB, int cgB, int kstrideB, int ns, int R,
                                        const MergeOut &mo) {
  // items (row j, four channels c4), the partials of an item split over ks
  // adjacent lanes that combine by shuffles at the end
  constexpr int kBatch = kMergeBatch;
  const int items = R * 32;
  const int ks = merge_split(R);
  const int mo_off = R * kD;
#pragma unroll 1
  for (int base = 0; base < items * ks; base += blockDim.x) {
    const int t = base + threadIdx.x;
    const bool valid = t < items * ks;
    const int item = t / ks, kq = t & (ks - 1);
    const int j = valid ? item >> 5 : 0, c4 = item & 31;
    const float *a0 = srcA + (j >> 3) * cgA, *b0 = srcB + (j >> 3) * cgB;
    float M = -INFINITY, L = 0.f;
    float4 A = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
    for (int kb = kq; valid && kb < ns; kb += ks * kBatch) {
      float ms[kBatch], ls[kBatch];
      float4 os[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int k = kb + u * ks;
        ms[u] = -INFINITY;
        ls[u] = 0.f;
        os[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (k < ns) {
          const float *sk = k < nA ? a0 + k * kstrideA : b0 + (k - nA) * kstrideB;
          ms[u] = ld_part(sk + mo_off + j);
          ls[u] = ld_part(sk + mo_off + kMaxR + j);
          os[u] = ld_part4(sk + j * kD + 4 * c4);
        }
      }
      float mn = M;
#pragma unroll
      for (int u = 0; u < kBatch; ++u) mn = fmaxf(mn, ms[u]);
      if (mn == -INFINITY) continue;
      const float a = (M == -INFINITY) ? 0.f : fast_exp2(M - mn);
      L *= a;
      A.x *= a; A.y *= a; A.z *= a; A.w *= a;
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const bool use = ms[u] > -INFINITY;  // an empty partial's l and O stay out
        const float f = use ? fast_exp2(ms[u] - mn) : 0.f;
        L = fmaf(f, use ? ls[u] : 0.f, L);
        A.x = fmaf(f, use ? os[u].x : 0.f, A.x);
        A.y = fmaf(f, use ? os[u].y : 0.f, A.y);
        A.z = fmaf(f, use ? os[u].z : 0.f, A.z);
        A.w = fmaf(f, use ? os[u].w : 0.f, A.w);
      }
      M = mn;
    }
#pragma unroll 1
    for (int o = 1; o < ks; o <<= 1) {
      const float M2 = __shfl_xor_sync(0xffffffffu, M, o), L2 = __shfl_xor_sync(0xffffffffu, L, o);
      float4 A2;
      A2.x = __shfl_xor_sync(0xffffffffu, A.x, o);
      A2.y = __shfl_xor_sync(0xffffffffu, A.y, o);
      A2.z = __shfl_xor_sync(0xffffffffu, A.z, o);
      A2.w = __shfl_xor_sync(0xffffffffu, A.w, o);
      const float mn = fmaxf(M, M2);
      if (mn != -INFINITY) {
        const float a = M == -INFINITY ? 0.f : fast_exp2(M - mn);
        const float a2 = M2 == -INFINITY ? 0.f : fast_exp2(M2 - mn);
        L = L * a + L2 * a2;
        A.x = A.x * a + A2.x * a2;
        A.y = A.y * a + A2.y * a2;
        A.z = A.z * a + A2.z * a2;
        A.w = A.w * a + A2.w * a2;
        M = mn;
      }
    }
    if (valid && kq == 0) {
      if (mo.final) {
        const float Ld = L > 0.f ? L : 1.f;
        uint2 h;
        h.x = pack_half2(A.x / Ld, A.y / Ld);
        h.y = pack_half2(A.z / Ld, A.w / Ld);
        *reinterpret_cast<uint2 *>(mo.out + j * kD + 4 * c4) = h;
        if (mo.lse && c4 == 0) mo.lse[j] = (M + log2f(L)) * 0.69314718055994531f;
      } else {
        reinterpret_cast<float4 *>(mo.dst + j * kD)[c4] = A;
        if (c4 == 0) {
          mo.dst[mo_off + j] = M;
          mo.dst[mo_off + kMaxR + j] = L;
        }
      }
    }
  }
}
#else
__device__ __noinline__ void merge_rows(const float *srcA, int cgA, int kstrideA, int nA,
                                        const float *srcB, int cgB, int kstrideB, int ns, int R,
                                        const MergeOut &mo) {
  constexpr int kBatch = kMergeBatch;
  const int lane = threadIdx.x & 31;
  const int mo_off = R * kD;
#pragma unroll 1
  for (int idx = threadIdx.x; idx < R * 32; idx += blockDim.x) {
    const int j = idx >> 5;
    const float *a0 = srcA + (j >> 3) * cgA, *b0 = srcB + (j >> 3) * cgB;
    float M = -INFINITY, L = 0.f;
    float4 A = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
    for (int kb = 0; kb < ns; kb += kBatch) {
      float ms[kBatch], ls[kBatch];
      float4 os[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int k = kb + u;
        ms[u] = -INFINITY;
        ls[u] = 0.f;
        os[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (k < ns) {
          const float *sk = k < nA ? a0 + k * kstrideA : b0 + (k - nA) * kstrideB;
          ms[u] = ld_part(sk + mo_off + j);
          ls[u] = ld_part(sk + mo_off + kMaxR + j);
          os[u] = ld_part4(sk + j * kD + 4 * lane);
        }
      }
      float mn = M;
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        if (!(ms[u] > -INFINITY)) {  // empty partial: stale l and O stay out
          ms[u] = -INFINITY;
          ls[u] = 0.f;
          os[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        mn = fmaxf(mn, ms[u]);
      }
      if (mn == -INFINITY) continue;  // nothing visible so far
      const float a = (M == -INFINITY) ? 0.f : fast_exp2(M - mn);
      L *= a;
      A.x *= a; A.y *= a; A.z *= a; A.w *= a;
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const float f = (ms[u] == -INFINITY) ? 0.f : fast_exp2(ms[u] - mn);
        L = fmaf(f, ls[u], L);
        A.x = fmaf(f, os[u].x, A.x);
        A.y = fmaf(f, os[u].y, A.y);
        A.z = fmaf(f, os[u].z, A.z);
        A.w = fmaf(f, os[u].w, A.w);
      }
      M = mn;
    }
    __syncwarp();  // every lane's reads of row j are done before dst is written
    if (mo.final) {
      const float Ld = L > 0.f ? L : 1.f;  // L > 0 whenever a token is visible
      uint2 h;
      h.x = pack_half2(A.x / Ld, A.y / Ld);
      h.y = pack_half2(A.z / Ld, A.w / Ld);
      *reinterpret_cast<uint2 *>(mo.out + j * kD + 4 * lane) = h;
      if (mo.lse && lane == 0) mo.lse[j] = (M + log2f(L)) * 0.69314718055994531f;
    } else {
      // generic stores (the readers load with ld.volatile, so no L1 line of
      // theirs can be stale)
      reinterpret_cast<float4 *>(mo.dst + j * kD)[lane] = A;
      if (lane == 0) {
        mo.dst[mo_off + j] = M;
        mo.dst[mo_off + kMaxR + j] = L;
      }
    }
  }
}
#endif

// One warp's partial of a piece (unnormalized, log2 domain; m = -inf if the
// warp saw no visible token; O as accumulated times oscale, plus the value
// bias) in the layout merge_rows reads: rows
// [8 cg, 8 cg + 8) of R, O at row * 128 + d, m at R * 128 + row, l at
// R * 128 + 24 + row; dst is in global or shared memory.
__device__ __forceinline__ void write_partial(const Softmax &sm, float oscale, float *dst, int R,
                                              int cg, int lane, bool pk) {
  const int r = lane >> 2, cq = lane & 3;
  const float l0 = warp_sum8(sm.l[0]), l1 = warp_sum8(sm.l[1]);
  const float v0 = warp_sum8(sm.bv[0]), v1 = warp_sum8(sm.bv[1]);
  // the thread's columns 2 cq, 2 cq + 1: rows 8 cg + 2 cq and the next, or
  // packed, row cq alone (its hi and lo columns)
  const int j0 = pk ? cq : 8 * cg + 2 * cq, j1 = pk ? R : j0 + 1;
#pragma unroll
  for (int md = 0; md < 8; ++md) {
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int d = 16 * md + r + 8 * hh;
      if (j0 < R) dst[j0 * kD + d] = fmaf(sm.o[md][2 * hh], oscale, v0);
      if (j1 < R) dst[j1 * kD + d] = fmaf(sm.o[md][2 * hh + 1], oscale, v1);
    }
  }
  if (r == 0) {
    const float m0 = sm.m[0] == -INFINITY ? -INFINITY : sm.m[0] - kExpShift;
    const float m1 = sm.m[1] == -INFINITY ? -INFINITY : sm.m[1] - kExpShift;
    if (j0 < R) { dst[R * kD + j0] = m0; dst[R * kD + kMaxR + j0] = l0; }
    if (j1 < R) { dst[R * kD + j1] = m1; dst[R * kD + kMaxR + j1] = l1; }
  }
}

// An empty partial of column group cg (the warp saw none of the piece):
// m = -inf, l = 0 for its rows.
__device__ __forceinline__ void write_empty(float *dst, int R, int cg, int lane) {
  const int j = 8 * cg + lane;
  if (lane < 8 && j < R) {
    dst[R * kD + j] = -INFINITY;
    dst[R * kD + kMaxR + j] = 0.f;
  }
}

// Wait (at most limit_ns) until a stage's copy of unit i has been issued.
__device__ __forceinline__ bool wait_issued(volatile int *issued, int i, uint64_t limit_ns) {
  if (*issued == i) return true;
  const uint64_t t0 = globaltimer_ns();
  while (*issued != i)
    if (globaltimer_ns() - t0 > limit_ns) return false;
  return true;
}

// PK (draft, R <= 4 query rows): the MMA's eight columns hold four query
// rows, column 2j the hi part of B = q * s and column 2j + 1 the lo part of
// row j (B column r = lane / 4 reads row r / 2; thread column pair 2c, 2c + 1
// = row c): one MMA per k-block instead of two, and one softmax column per
// thread.
// NW: warps per CTA (12, or kVerifyWarps for a verify tile of <= 16 rows).
template <int MODE, bool PK, int UB, int NW>
__global__ void __launch_bounds__(NW * 32, 1) split_kernel(const Params prm) {
  using C = Cfg<MODE>;
  using L = Layout<MODE>;
  constexpr int TT = C::kTailTok, S = C::kStages;
  constexpr int kTailTiles = TT / 32;  // 16-token tiles of a buffer chunk per warp
  // buffer tiles padded where several column groups read each tile (the
  // 12-warp multi-row variants); unpadded, one copy per plane, elsewhere
  constexpr bool kPadTail = !PK && NW == 12;
  constexpr int kRow = tail_row<kPadTail>();
  extern __shared__ __align__(128) uint8_t smem[];
  const qs_cache &c = prm.c;
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int r = lane >> 2, cq = lane & 3;
  const uint32_t sbase = smem_addr(smem);
  const uint32_t full0 = sbase + L::kBarOff, zero_row = sbase + L::kZeroOff;
  const uint32_t mrg_bar = sbase + L::kMrgOff;
  int *cnt = reinterpret_cast<int *>(smem + L::kCntOff);            // releases per stage
  volatile int *issued = reinterpret_cast<int *>(smem + L::kIssOff);  // unit copied into a stage
  Tables T = tables_at(smem, L::kTabOff);
  __shared__ long long s_total;
  __shared__ int s_abort, s_left_first, s_first_fin, s_seg[2], s_ord[2], s_need[2], s_last[2];
  __shared__ int s_plo[2], s_raw[2];
  __shared__ int s_next[3];  // claim counter per column group

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full0 + 8 * s, 1);
      cnt[s] = 0;
      issued[s] = -1;
    }
    if (MODE == QS_VERIFY_INT8) mbar_init(mrg_bar, 1);
    fence_mbar_init();
    s_next[0] = s_next[1] = s_next[2] = 0;
    s_abort = 0;
    s_left_first = 0;
    s_first_fin = 0;
  }
  if (threadIdx.x < 8) reinterpret_cast<uint32_t *>(smem + L::kZeroOff)[threadIdx.x] = 0;
  pdl_trigger();
  pdl_wait();  // counters, cache and queries are written by earlier kernels
  if (w == 0) {
    const long long tot = build_tables<TT>(c, prm.n_q, prm.n_new, T, lane);
    if (lane == 0) s_total = tot;
  }
  __syncthreads();
  const long long U = s_total;
  const int p = blockIdx.x;
  const int R = prm.R, ncg = prm.ncg, cg = w % ncg;  // this warp's column group
  const int stride = R * kD + 2 * kMaxR;             // floats per partial

  if (prm.n_new > 0 && w == NW - 1) {
    // The fused append, by a warp that issues no first copy.  Every CTA has
    // read the counters above; the CTA whose ticket comes last commits the
    // appended counters (no CTA of this launch reads them again).  The new
    // tokens enter the ring slots past the old fill, which no CTA of this
    // launch reads (its copies of those rows come from k_new / v_new).
    if (lane == 0 && atom_add_acq_rel_gpu(&c.state[QS_ST_TICKET], 1) == (int)gridDim.x - 1) {
      for (int b = 0; b < c.B; ++b) {
        int32_t *st = c.state + (size_t)b * QS_STATE_WORDS;
        if (T.fill[b] != T.fold[b]) {
          st[QS_ST_FILL] = T.fill[b];
          st[QS_ST_PENDING] += prm.n_new;
        } else {
          st[QS_ST_ERR] |= QS_DEV_OVERFLOW;  // as a separate append would: no-op
        }
      }
      c.state[QS_ST_TICKET] = 0;
    }
    constexpr int kRowVec = kD * 2 / 16;  // uint4 per fp16 row
    for (int j = p; j < c.B * c.H; j += gridDim.x) {
      const int b = j / c.H;
      if (T.fill[b] == T.fold[b]) continue;  // this sequence's append failed
      const int slot0 = T.hb[b] * kG + T.fold[b];
      const uint4 *sk = reinterpret_cast<const uint4 *>(prm.k_new) + (size_t)j * prm.n_new * kRowVec;
      const uint4 *sv = reinterpret_cast<const uint4 *>(prm.v_new) + (size_t)j * prm.n_new * kRowVec;
      uint4 *bk = reinterpret_cast<uint4 *>(c.buf_k) + (size_t)j * kRing * kRowVec;
      uint4 *bv = reinterpret_cast<uint4 *>(c.buf_v) + (size_t)j * kRing * kRowVec;
      for (int e = lane; e < prm.n_new * kRowVec; e += 32) {
        const int slot = (slot0 + e / kRowVec) & (kRing - 1);
        bk[slot * kRowVec + e % kRowVec] = sk[e];
        bv[slot * kRowVec + e % kRowVec] = sv[e];
      }
    }
  }

  // sequences with n_q > fill see no token: zero outputs, lse = -inf, error
  for (int b = p; b < c.B; b += prm.P) {
    if (T.len[b] != 0) continue;
    const size_t nh = (size_t)c.H * R;
    uint4 *o = reinterpret_cast<uint4 *>(prm.out + (size_t)b * nh * kD);
    for (size_t i = threadIdx.x; i < nh * (kD / 8); i += (NW * 32)) o[i] = make_uint4(0, 0, 0, 0);
    if (prm.lse)
      for (size_t i = threadIdx.x; i < nh; i += (NW * 32)) prm.lse[(size_t)b * nh + i] = -INFINITY;
    if (threadIdx.x == 0) atomicOr(&c.state[(size_t)b * QS_STATE_WORDS + QS_ST_ERR], QS_DEV_NQ_GT_FILL);
  }

  const int x0 = (int)range_lo(p, U, prm.P), x1 = (int)range_lo(p + 1, U, prm.P);
  if (x0 >= x1) return;
  const int n = x1 - x0;
  Seg first, lastseg;
  first.seek(x0, T, c.B);
  lastseg.seek(x1 - 1, T, c.B);
  const int ord_first = first.ord, ord_last = lastseg.ord;
  // partial slot of warp ww for the piece of segment ordinal o
  auto slot = [&](int o, int ww) {
    const size_t off = ((size_t)(o + p) * NW + ww) * stride;
    // checked build: a partial out of the workspace is written to slot 0
    return prm.ws + (chk(in_range(off, stride, prm.ws_floats), 7) ? off : 0);
  };
  // checked build: [q, q + n) inside the workspace (the merges' reads)
  auto ws_ok = [&](const float *q, size_t n) {
    return chk(in_range((size_t)(q - prm.ws), n, prm.ws_floats), 8);
  };
  // A segment split across CTAs p_lo..p_hi is finished by whichever CTA
  // arrives last on its counter.  CTAs p_lo..p_hi-1 hold it as their last
  // piece and arrive with one merged CTA partial at the end.  CTA p_hi holds
  // it as its first piece; when its range goes on past the segment it does
  // not merge it at all: the warp that leaves the piece last arrives for the
  // CTA (its NW warp partials are all written and fenced by then), and
  // the finishing CTA reads those partials directly.
  const bool shared_first = ord_first != ord_last && first.s0 < x0;
  auto leave = [&](int o) {
    if (!shared_first || o != ord_first) return;
    // The lanes' partial stores are ordered before lane 0's count
    // (__syncwarp); the count is an acquire-release atomic at CTA scope, so
    // the warp that counts last has acquired every other warp's partial, and
    // its device-scope acquire-release arrival (cumulative) publishes them all.
    __syncwarp();
    if (lane == 0 && atom_add_acq_rel_cta(&s_left_first, 1) == NW - 1) {
      const int seg = first.b * c.H + first.h;
      const int plo = cta_of(first.s0, U, prm.P);  // the segment ends in this range: p_hi = p
      if (atom_add_acq_rel_gpu(&c.arrive[seg], 1) == p - plo) {
        // rare: the CTAs before have all arrived; this CTA finishes the
        // segment at its end
        atomicExch(&c.arrive[seg], 0);  // every other arrival is in
        s_first_fin = 1;
      }
    }
    __syncwarp();
  };

  // the warps reach the range's last segment mid-range: start its queries
  // towards L1 now (two 128-byte lines per row; a copy in shared memory was
  // measured no faster)
  if (ord_last != ord_first && threadIdx.x < 2 * R) {
    const size_t bh = (size_t)lastseg.b * c.H + lastseg.h;
    prefetch_l1(prm.q + (bh * R) * kD + threadIdx.x * 64);
  }

  // units i and i + S share stage i % S; warp 0 issues the first S
  if (w == 0 && !prm.no_issue) {
    Seg a;
    for (int k = 0; k < S && k < n; ++k) {
      a.seek(x0 + k, T, c.B);
      if (lane == 0) issued[k] = k;
      issue_unit<MODE, UB, kPadTail>(prm, T, a, sbase + k * L::kStageBytes, full0 + 8 * k, lane);
    }
  }

  Softmax sm;
  sm.reset();
  uint32_t qp0[8], qp1[8];
  int fill = 0, ng = 0;
  int cur_ord = -1;  // segment ordinal of this warp's softmax state (-1: none yet)
  Seg cur, ahead;
  // Work is claimed in half-units (claim h: unit h / 2, tokens of half h % 2)
  // from one shared counter.  Both halves of a unit go to whichever warps
  // claim them; the stage's release counter joins them again.  Draft claims
  // one ahead, so the atomic's latency hides behind a unit's compute; verify,
  // whose ring holds only as many units as are in compute, claims when free
  // (a claim made ahead would wait on a copy that cannot start yet).
  constexpr bool kAhead = MODE == QS_DRAFT_UPPER4;
  auto claim = [&]() {
    int h = 0;
    if (lane == 0)
      h = *reinterpret_cast<volatile int *>(&s_abort) ? 2 * n : atomicAdd(&s_next[cg], 1);
    return __shfl_sync(0xffffffffu, h, 0);
  };
  int h_next = kAhead ? claim() : 0;
  for (;;) {
    const int hcl = kAhead ? h_next : claim();
    if (hcl >= 2 * n) break;
    if (kAhead) h_next = claim();
    const int i = hcl >> 1, hw = hcl & 1;
    cur.seek(x0 + i, T, c.B);
    if (cur.ord != cur_ord) {
      // a new piece: the finished one's partial (empty ones for pieces this
      // warp skipped), then fresh state and this head's queries
      if (cur_ord >= 0) {
        write_partial(sm, Centre<MODE, UB>::kScale, slot(cur_ord, w), R, cg, lane, PK);
        leave(cur_ord);
      }
      for (int o = cur_ord >= 0 ? cur_ord + 1 : ord_first; o < cur.ord; ++o) {
        write_empty(slot(o, w), R, cg, lane);
        leave(o);
      }
      cur_ord = cur.ord;
      const size_t bh = (size_t)cur.b * c.H + cur.h;
      const int qi = PK ? (r >> 1) : 8 * cg + r;  // the query row in B column r
      const bool q_ok =  // (rows qi >= R are not read)
          qi >= R || chk(in_range((bh * R + qi) * kD, kD, (size_t)c.B * c.H * R * kD), 9);
      load_q_pairs(prm.q + (q_ok ? (bh * R + qi) * kD : 0), qi < R, cq, qp0, qp1);
      sm.reset();
      fill = T.fill[cur.b];
      ng = T.ng[cur.b];
    }
    const int stage = i % S;
    // the stage must hold unit i's copy (not the unit S before it) before its
    // barrier parity means anything
    bool ok = wait_issued(issued + stage, i, prm.wait_ns);
    if (ok) ok = mbar_wait(full0 + 8 * stage, (uint32_t)((i / S) & 1), prm.wait_ns);
    ok = __all_sync(0xffffffffu, ok);  // the tensor-core code below needs the whole warp
    if (!ok) {
      if (lane == 0) {
        atomicOr(&c.state[(size_t)cur.b * QS_STATE_WORDS + QS_ST_ERR], QS_DEV_TIMEOUT);
        s_abort = 1;
      }
    } else {
      const uint32_t st = sbase + stage * L::kStageBytes;

      if (cur.u < ng) {
        // ============================================== quantized group
        // This warp: tokens [64 hw, 64 hw + 64) of the group.  B = q * s_K per
        // channel as an fp16 pair hi + lo (lo = the exactly-rounded residual
        // of the fp16 product, one fused multiply-add): a dominant token's
        // large score would otherwise carry the 2^-11 rounding of q * s.
        // The key bias comes from one MMA per k-block whose A rows 0-7 hold
        // the zero-points and rows 8-15 the scales.  The meta rows are stored
        // in fragment order: one 16-byte load gives k-blocks 2i, 2i+1.  The
        // second B register of a k-block (k 8-15) meets the odd code
        // elements; for the draft those are 16 C_U, so its scales are s / 16
        // (an exact power-of-two step; where s / 16 is subnormal the score
        // moves by less than 2^-20 * |q|).
        uint32_t bh0[8], bh1[8], bl0[8], bl1[8];
        float bacc[4] = {0.f, 0.f, 0.f, 0.f}, bacc2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i4 = 0; i4 < 4; ++i4) {
          const uint4 sw = lds128(st + kOffMeta + QS_META_K_SCALE * 256 + 16 * (4 * i4 + cq));
          const uint4 zw = lds128(st + kOffMeta + QS_META_K_ZERO * 256 + 16 * (4 * i4 + cq));
          const int k0 = 2 * i4, k1 = 2 * i4 + 1;
          uint32_t s1 = sw.y, s3 = sw.w;
          if (MODE == QS_DRAFT_UPPER4) {
            s1 = hmul2_u32(s1, 0x2C002C00u);  // fp16 (1/16, 1/16)
            s3 = hmul2_u32(s3, 0x2C002C00u);
          }
          bh0[k0] = hmul2_u32(qp0[k0], sw.x);
          bh1[k0] = hmul2_u32(qp1[k0], s1);
          bh0[k1] = hmul2_u32(qp0[k1], sw.z);
          bh1[k1] = hmul2_u32(qp1[k1], s3);
          bl0[k0] = hfma2_neg_u32(qp0[k0], sw.x, bh0[k0]);
          bl1[k0] = hfma2_neg_u32(qp1[k0], s1, bh1[k0]);
          bl0[k1] = hfma2_neg_u32(qp0[k1], sw.z, bh0[k1]);
          bl1[k1] = hfma2_neg_u32(qp1[k1], s3, bh1[k1]);
          if (PK && (r & 1)) {  // odd B columns carry the lo part
            bh0[k0] = bl0[k0]; bh1[k0] = bl1[k0]; bh0[k1] = bl0[k1]; bh1[k1] = bl1[k1];
          }
          mma16816(bacc, zw.x, sw.x, zw.y, sw.y, qp0[k0], qp1[k0]);
          mma16816(bacc2, zw.z, sw.z, zw.w, sw.w, qp0[k1], qp1[k1]);
        }
        // key dequant s * code + (z + kOffK s), code = 16 C_U or C_INT8:
        // bias = sum q z + kOffK sum q s; the code part scales by kScale
        const float sl2q = prm.sl2 * Centre<MODE, UB>::kScale;
        const float bk0 =
            fmaf(Centre<MODE, UB>::kOffK, bacc[2] + bacc2[2], bacc[0] + bacc2[0]) * prm.sl2;
        const float bk1 =
            fmaf(Centre<MODE, UB>::kOffK, bacc[3] + bacc2[3], bacc[1] + bacc2[1]) * prm.sl2;

        // raw scores (q.k before scale and bias): four m-tiles of 16 tokens
        float s[4][4];
#pragma unroll
        for (int mt = 0; mt < 4; ++mt) {
          const int t0 = 64 * hw + 16 * mt + r;
          // the lane's four 4-bit words of rows t0 and t0 + 8 (two-bit
          // layout: two C_U2 words each, plus two M2 words for verify)
          uint32_t wu0[4], wu1[4];
          if (UB == 4) {
            const uint4 u0 = lds128(st + kOffKU + t0 * 64 + 16 * cq);
            const uint4 u1 = lds128(st + kOffKU + (t0 + 8) * 64 + 16 * cq);
            wu0[0] = u0.x; wu0[1] = u0.y; wu0[2] = u0.z; wu0[3] = u0.w;
            wu1[0] = u1.x; wu1[1] = u1.y; wu1[2] = u1.z; wu1[3] = u1.w;
          } else {
            const uint2 a0 = lds64(st + kOffKU + t0 * 32 + 8 * cq);
            const uint2 a1 = lds64(st + kOffKU + (t0 + 8) * 32 + 8 * cq);
            if (MODE == QS_VERIFY_INT8) {
              const uint2 m0 = lds64(st + kOffKU + 4096 + t0 * 32 + 8 * cq);
              const uint2 m1 = lds64(st + kOffKU + 4096 + (t0 + 8) * 32 + 8 * cq);
              wu0[0] = upper_from2(a0.x, m0.x, 0); wu0[1] = upper_from2(a0.x, m0.x, 2);
              wu0[2] = upper_from2(a0.y, m0.y, 0); wu0[3] = upper_from2(a0.y, m0.y, 2);
              wu1[0] = upper_from2(a1.x, m1.x, 0); wu1[1] = upper_from2(a1.x, m1.x, 2);
              wu1[2] = upper_from2(a1.y, m1.y, 0); wu1[3] = upper_from2(a1.y, m1.y, 2);
            } else {  // draft: converted straight from the C_U2 words below
              wu0[0] = wu0[1] = a0.x; wu0[2] = wu0[3] = a0.y;
              wu1[0] = wu1[1] = a1.x; wu1[2] = wu1[3] = a1.y;
            }
          }
          uint4 l0 = make_uint4(0, 0, 0, 0), l1 = l0;
          if (MODE == QS_VERIFY_INT8) {
            l0 = lds128(st + kOffKL + t0 * 64 + 16 * cq);
            l1 = lds128(st + kOffKL + (t0 + 8) * 64 + 16 * cq);
          }
          float acc[4] = {0.f, 0.f, 0.f, 0.f}, acc2[4] = {0.f, 0.f, 0.f, 0.f};
          const uint32_t wl0[4] = {l0.x, l0.y, l0.z, l0.w}, wl1[4] = {l1.x, l1.y, l1.z, l1.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {  // two independent MMA chains: even / odd k-blocks
            uint32_t a[4], b8[4];
            if (MODE == QS_DRAFT_UPPER4 && UB == 2) {
              if (j & 1) {
                pairs_upper2<2>(wu0[j], a);
                pairs_upper2<2>(wu1[j], b8);
              } else {
                pairs_upper2<0>(wu0[j], a);
                pairs_upper2<0>(wu1[j], b8);
              }
            } else {
              pairs<MODE>(wu0[j], wl0[j], a);
              pairs<MODE>(wu1[j], wl1[j], b8);
            }
            mma16816(acc, a[0], b8[0], a[1], b8[1], bh0[2 * j], bh1[2 * j]);
            mma16816(acc2, a[2], b8[2], a[3], b8[3], bh0[2 * j + 1], bh1[2 * j + 1]);
            if (!PK) {
              mma16816(acc, a[0], b8[0], a[1], b8[1], bl0[2 * j], bl1[2 * j]);
              mma16816(acc2, a[2], b8[2], a[3], b8[3], bl0[2 * j + 1], bl1[2 * j + 1]);
            }
          }
          if (PK) {  // query c: hi column + lo column, rows r and r + 8
            s[mt][0] = (acc[0] + acc2[0]) + (acc[1] + acc2[1]);
            s[mt][2] = (acc[2] + acc2[2]) + (acc[3] + acc2[3]);
            s[mt][1] = s[mt][3] = -INFINITY;
          } else {
#pragma unroll
            for (int k = 0; k < 4; ++k) s[mt][k] = acc[k] + acc2[k];
          }
        }
        // max of scaled scores = max of raw scores * sl2 + bias (sl2 > 0)
        float g0 = fmaxf(s[0][0], s[0][2]), g1 = fmaxf(s[0][1], s[0][3]);
#pragma unroll
        for (int mt = 1; mt < 4; ++mt) {
          g0 = fmaxf(g0, fmaxf(s[mt][0], s[mt][2]));
          g1 = fmaxf(g1, fmaxf(s[mt][1], s[mt][3]));
        }
        float u0, u1, a0, a1;
        sm.update(fmaf(warp_max8(g0), sl2q, bk0), fmaf(warp_max8(g1), sl2q, bk1), u0, u1, a0, a1);
        const float c0 = bk0 - u0, c1 = bk1 - u1;  // p = 2^(raw * sl2 + c)

        // probabilities with the value scale folded in, value zero-point as a
        // bias; each value row holds a lane's four tokens of a quarter together.
        // The second B register of a k-block (tokens 8-15 of a tile, hh = 1)
        // meets the odd code elements: for the draft P' / 16 there.
        uint32_t bp0[4], bp1[4];
#pragma unroll
        for (int qq = 0; qq < 2; ++qq) {
          const int moff = kOffMeta + 2 * (32 * (2 * hw + qq) + 4 * r);
#if QS_CHECKED
          const uint2 svw = lds64(st + moff + QS_META_V_SCALE * 256);
          const uint2 zvw = lds64(st + moff + QS_META_V_ZERO * 256);
#else
          const uint2 svw =
              *reinterpret_cast<const uint2 *>(smem + (st - sbase) + moff + QS_META_V_SCALE * 256);
          const uint2 zvw =
              *reinterpret_cast<const uint2 *>(smem + (st - sbase) + moff + QS_META_V_ZERO * 256);
#endif
          const float2 sv01 = __half22float2(u32_as_h2(svw.x)), sv23 = __half22float2(u32_as_h2(svw.y));
          const float2 zv01 = __half22float2(u32_as_h2(zvw.x)), zv23 = __half22float2(u32_as_h2(zvw.y));
          const float svs[4] = {sv01.x, sv01.y, sv23.x, sv23.y};
          const float zvs[4] = {zv01.x, zv01.y, zv23.x, zv23.y};
#pragma unroll
          for (int ml = 0; ml < 2; ++ml) {
            const int mt = 2 * qq + ml;
            float pv[4];
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              const float sv = svs[2 * ml + hh];
              const float zv = fmaf(Centre<MODE, UB>::kOff, sv, zvs[2 * ml + hh]);
              const float pa = fast_exp2(fmaf(s[mt][2 * hh], sl2q, c0));
              const float pb = PK ? 0.f : fast_exp2(fmaf(s[mt][2 * hh + 1], sl2q, c1));
              sm.l[0] += pa;
              sm.l[1] += pb;
              sm.bv[0] = fmaf(pa, zv, sm.bv[0]);
              sm.bv[1] = fmaf(pb, zv, sm.bv[1]);
              // PK: P' column 2c holds row c (c < R), column 2c + 1 (the lo
              // column of the scores) stays zero (pb = 0)
              const float svp = (MODE == QS_DRAFT_UPPER4 && hh) ? sv * 0.0625f : sv;
              pv[2 * hh] = (PK && cq >= R) ? 0.f : pa * svp;
              pv[2 * hh + 1] = pb * svp;
            }
            bp0[mt] = movmatrix_trans(pack_half2(pv[0], pv[1]));
            bp1[mt] = movmatrix_trans(pack_half2(pv[2], pv[3]));
          }
        }
        {
          // centre the value codes on 128: take 128 * sum_t P'_t out of the
          // value bias, the sum formed by the tensor core from the same fp16
          // P' it multiplies the codes with (A = 1, and 16 against the
          // draft's P' / 16), so the result equals the centred product
          constexpr uint32_t kOnes = 0x3C003C00u;  // fp16 (1, 1)
          constexpr uint32_t kHi = MODE == QS_DRAFT_UPPER4 ? 0x4C004C00u : kOnes;  // (16, 16)
          float sp[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int mt = 0; mt < 4; ++mt) mma16816(sp, kOnes, kOnes, kHi, kHi, bp0[mt], bp1[mt]);
          // every row of the product holds the column sum, while the value
          // bias is a per-lane partial summed over the eight row lanes later:
          // one lane per column takes it
          if (r == 0) {
            sm.bv[0] = fmaf(-Centre<MODE, UB>::kMid, sp[0], sm.bv[0]);
            sm.bv[1] = fmaf(-Centre<MODE, UB>::kMid, sp[1], sm.bv[1]);
          }
        }
        // O^T = a O^T + V^T P'  (values: quarters 2hw and 2hw+1, channel-major)
#pragma unroll
        for (int md = 0; md < 8; ++md) {
          float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int qq = 0; qq < 2; ++qq) {
            const int vrow = (2 * hw + qq) * 128 + 16 * md + r;  // (quarter, channel) row
            uint32_t vu0, vu1, vl0 = 0, vl1 = 0;
            const int sh = 2 * (cq & 1);  // two-bit layout: the lane's half of a C_U2 word
            const uint32_t ra2 = st + kOffVU + vrow * 8 + 4 * (cq >> 1);
            if (UB == 4) {
              const uint32_t ra = st + kOffVU + vrow * 16 + 4 * cq;
              vu0 = lds32(ra);
              vu1 = lds32(ra + 8 * 16);
            } else {
              vu0 = lds32(ra2);
              vu1 = lds32(ra2 + 8 * 8);
              if (MODE == QS_VERIFY_INT8) {
                vu0 = upper_from2(vu0, lds32(ra2 + 4096), sh);
                vu1 = upper_from2(vu1, lds32(ra2 + 4096 + 8 * 8), sh);
              }
            }
            if (MODE == QS_VERIFY_INT8) {
              const uint32_t rl = st + kOffVL + vrow * 16 + 4 * cq;
              vl0 = lds32(rl);
              vl1 = lds32(rl + 8 * 16);
            }
            uint32_t a[4], b8[4];
            if (MODE == QS_DRAFT_UPPER4 && UB == 2) {
              pairs_upper2_rt(vu0, sh, a);
              pairs_upper2_rt(vu1, sh, b8);
            } else {
              pairs<MODE>(vu0, vl0, a);
              pairs<MODE>(vu1, vl1, b8);
            }
            mma16816(d, a[0], b8[0], a[1], b8[1], bp0[2 * qq], bp1[2 * qq]);
            mma16816(d, a[2], b8[2], a[3], b8[3], bp0[2 * qq + 1], bp1[2 * qq + 1]);
          }
          sm.merge(md, d, a0, a1);
        }
      } else {
        // ============================================== fp16 buffer chunk
        // This warp: 16-token tiles [hw * kTailTiles, (hw + 1) * kTailTiles).
        const int i0 = (cur.u - ng) * TT;
        const int rows = min(TT, fill - i0);
        const int mr0 = 16 * kTailTiles * hw;
        if (mr0 < rows) {
          // key fragments in the same permuted channel order as the quantized
          // path, built from shared memory (16-byte loads + byte permutes), so
          // the register-resident q pairs serve as B: no global loads here
          // last visible buffer index of the thread's two columns: row
          // (PK: c; else 8 cg + 2c and the next) sits at position row % n_q
          const int row0 = PK ? cq : 8 * cg + 2 * cq;
          const int lim0 = fill - prm.n_q + row0 % prm.n_q;
          const int lim1 = fill - prm.n_q + (row0 + 1) % prm.n_q;
          float sv[kTailTiles][4];
          float g0 = -INFINITY, g1 = -INFINITY;
#pragma unroll
          for (int tl = 0; tl < kTailTiles; ++tl) {
            const int mr = mr0 + 16 * tl;
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            uint32_t w0[16], w1[16];  // channels 32c..32c+31 of rows mr+r, mr+r+8
#pragma unroll
            for (int i4 = 0; i4 < 4; ++i4) {
              const int ra = mr + r, rb = mr + r + 8;
              const uint4 x = ra < rows ? lds128(st + ra * kRow + 64 * cq + 16 * i4) : make_uint4(0, 0, 0, 0);
              const uint4 y = rb < rows ? lds128(st + rb * kRow + 64 * cq + 16 * i4) : make_uint4(0, 0, 0, 0);
              w0[4 * i4] = x.x; w0[4 * i4 + 1] = x.y; w0[4 * i4 + 2] = x.z; w0[4 * i4 + 3] = x.w;
              w1[4 * i4] = y.x; w1[4 * i4 + 1] = y.y; w1[4 * i4 + 2] = y.z; w1[4 * i4 + 3] = y.w;
            }
#pragma unroll
            for (int kb = 0; kb < 8; ++kb) {
              const int k0 = 4 * (kb >> 1) + (kb & 1);
              mma16816(acc, prmt(w0[k0], w0[k0 + 2], 0x5410), prmt(w1[k0], w1[k0 + 2], 0x5410),
                       prmt(w0[k0], w0[k0 + 2], 0x7632), prmt(w1[k0], w1[k0 + 2], 0x7632), qp0[kb],
                       qp1[kb]);
            }
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const int tok = mr + r + 8 * (k >> 1);
              const bool vis = tok < rows && (i0 + tok) <= ((k & 1) ? lim1 : lim0) && !(PK && (k & 1));
              sv[tl][k] = vis ? acc[k] * prm.sl2 : -INFINITY;
            }
            g0 = fmaxf(g0, fmaxf(sv[tl][0], sv[tl][2]));
            g1 = fmaxf(g1, fmaxf(sv[tl][1], sv[tl][3]));
          }
          float u0, u1, a0, a1;
          sm.update(warp_max8(g0), warp_max8(g1), u0, u1, a0, a1);
          uint32_t bq0[kTailTiles], bq1[kTailTiles];
#pragma unroll
          for (int tl = 0; tl < kTailTiles; ++tl) {
            float pv[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              pv[k] = (PK && cq >= R) ? 0.f : fast_exp2(sv[tl][k] - ((k & 1) ? u1 : u0));
              sm.l[k & 1] += pv[k];
            }
            bq0[tl] = movmatrix_trans(pack_half2(pv[0], pv[1]));
            bq1[tl] = movmatrix_trans(pack_half2(pv[2], pv[3]));
          }
          const uint32_t vbase = st + TT * kRow;
#pragma unroll
          for (int md = 0; md < 8; ++md) {
            float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int tl = 0; tl < kTailTiles; ++tl) {
              const int mi = lane >> 3;
              const int tok = mr0 + 16 * tl + (lane & 7) + (mi >> 1) * 8;
              const int ch = 16 * md + (mi & 1) * 8;
              uint32_t addr = tok < rows ? vbase + tok * kRow + ch * 2 : zero_row;
              if (!chk(smem_in(addr, 16), 6)) addr = zero_row;
              uint32_t f0, f1, f2, f3;
              ldmatrix_x4_trans(addr, f0, f1, f2, f3);
              mma16816(d, f0, f1, f2, f3, bq0[tl], bq1[tl]);
            }
            // fp16 values: true units, the accumulators hold O / kScale
#pragma unroll
            for (int k = 0; k < 4; ++k) d[k] *= 1.f / Centre<MODE, UB>::kScale;
            sm.merge(md, d, a0, a1);
          }
        }
      }

    }

    // release the stage; the later of the unit's two halves issues the refill
    // (unit i + S) unless its own wait failed
    __syncwarp();
    int last = 0;
    if (lane == 0) last = (atomicAdd(&cnt[stage], 1) == 2 * ncg - 1);
    last = __shfl_sync(0xffffffffu, last, 0);
    if (last) {
      if (lane == 0) cnt[stage] = 0;
      if (ok && i + S < n) {
        ahead.seek(x0 + i + S, T, c.B);
        fence_proxy_async_smem();
        if (lane == 0) issued[stage] = i + S;
        __syncwarp();
        issue_unit<MODE, UB, kPadTail>(prm, T, ahead, sbase + stage * L::kStageBytes, full0 + 8 * stage, lane);
      }
    }
  }
  // this warp's partials for the pieces after its last unit's piece are empty
  // (all but the range's last piece go to the workspace)
  if (cur_ord >= 0 && cur_ord < ord_last) {
    write_partial(sm, Centre<MODE, UB>::kScale, slot(cur_ord, w), R, cg, lane, PK);
    leave(cur_ord);
  }
  for (int o = cur_ord >= 0 ? cur_ord + 1 : ord_first; o < ord_last; ++o) {
    write_empty(slot(o, w), R, cg, lane);
    leave(o);
  }

  __syncthreads();
  // no copy may still be landing in the stage memory reused below: after a
  // timeout, wait for each stage's last copy (otherwise every issued copy
  // has been waited for by the warps that claimed its halves).  If that wait
  // runs out too, s_abort = 2: a copy may still land in the stages, so the
  // CTA writes nothing more into them (its partials and merges are skipped;
  // the arrivals below still return the counters to zero).
  if (s_abort) {  // uniform: read after the barrier above
    if (w == 0) {
      const unsigned long long deadline = globaltimer_ns() + prm.wait_ns;
      bool drained = true;
      for (int s = lane; s < S; s += 32) {
        const int j = issued[s];
        if (j >= 0)
          while (!mbar_try_wait(full0 + 8 * s, (uint32_t)((j / S) & 1)))
            if (globaltimer_ns() >= deadline) {
              drained = false;
              break;
            }
      }
      if (!__all_sync(0xffffffffu, drained) && lane == 0) s_abort = 2;
    }
    __syncthreads();
  }

  // ---- log-sum-exp merge.  Per piece of this CTA's range (but a shared
  // first piece, see above): merge the NW warp partials (the last piece's
  // straight from registers through shared memory); a segment that lies
  // wholly in the range is final here.  A segment shared with other CTAs gets
  // one CTA partial (in warp slot 0) and an arrival on its counter; the CTA
  // that arrives last merges the CTA partials of the whole segment and
  // resets the counter.  Only the first and the last piece of a range can be
  // shared.
  const bool aborted = s_abort != 0;
  float *last_part = reinterpret_cast<float *>(smem);  // NW partials, in stage memory (free now)
  chk(smem_in(smem_addr(last_part), (uint32_t)(NW * stride * 4)), 11);
  if (s_abort != 2) {
    if (cur_ord == ord_last)
      write_partial(sm, Centre<MODE, UB>::kScale, last_part + w * stride, R, cg, lane, PK);
    else
      write_empty(last_part + w * stride, R, cg, lane);
  }
  __syncthreads();
  if (s_first_fin && !aborted) {
    fence_gpu();  // the other CTAs' partials are visible from here on
    const long long seg = (long long)first.b * c.H + first.h;
    const int plo = cta_of(first.s0, U, prm.P);
    const MergeOut fo{true, prm.out + (size_t)seg * R * kD,
                      prm.lse ? prm.lse + (size_t)seg * R : nullptr, nullptr};
    if (ws_ok(prm.ws + (size_t)(ord_first + plo) * NW * stride, (size_t)(p - plo) * NW * stride) &&
        ws_ok(slot(ord_first, 0), (size_t)NW * stride) && chk(seg < (long long)c.B * c.H, 10))
    merge_rows(prm.ws + (size_t)(ord_first + plo) * NW * stride, 0, NW * stride, p - plo,
               slot(ord_first, 0), stride, ncg * stride, p - plo + NW / ncg, R, fo);
  }
  int n_arr = 0;
  {
    Seg pc;
    int x = shared_first ? first.s0 + first.len : x0;  // the first piece is done already
    while (x < x1) {
      pc.seek(x, T, c.B);
      const long long seg = (long long)pc.b * c.H + pc.h;
      const int S0 = pc.s0, E0 = pc.s0 + pc.len;
      const int plo = cta_of(S0, U, prm.P), phi = cta_of(E0 - 1, U, prm.P);
      const MergeOut mo{plo == phi, prm.out + (size_t)seg * R * kD,
                        prm.lse ? prm.lse + (size_t)seg * R : nullptr, slot(pc.ord, 0)};
      if (!aborted && chk(seg < (long long)c.B * c.H, 10) &&
          (pc.ord == ord_last || ws_ok(slot(pc.ord, 0), (size_t)NW * stride)))
        merge_rows(pc.ord == ord_last ? last_part : slot(pc.ord, 0), stride, ncg * stride,
                   NW / ncg, nullptr, 0, 0, NW / ncg, R, mo);
      if (plo != phi) {
        if (threadIdx.x == 0) {
          s_seg[n_arr] = (int)seg;
          s_ord[n_arr] = pc.ord;
          s_need[n_arr] = phi - plo + 1;
          s_plo[n_arr] = plo;
          // CTA p_hi left its NW warp partials if the segment was only the
          // first piece of its range
          s_raw[n_arr] = S0 < range_lo(phi, U, prm.P) && E0 < range_lo(phi + 1, U, prm.P);
        }
        ++n_arr;
      }
      x = E0;
    }
  }
  if (n_arr == 0) return;
  __syncthreads();  // this CTA's partials are written (made visible by the fence below)
  if (threadIdx.x < n_arr) {
    int *ctr = c.arrive + s_seg[threadIdx.x];
    const int last = atom_add_acq_rel_gpu(ctr, 1) == s_need[threadIdx.x] - 1;
    if (last) atomicExch(ctr, 0);  // every other arrival is in: ready for the next call
    s_last[threadIdx.x] = last;
  }
  __syncthreads();
  int n_mrg = 0;  // phases of the merge barrier used
  for (int a = 0; a < n_arr; ++a) {
    if (!s_last[a] || aborted) continue;
    const int seg = s_seg[a], b = seg / c.H;
    const int plo = s_plo[a], phi = plo + s_need[a] - 1;
    const MergeOut mo{true, prm.out + (size_t)seg * R * kD,
                      prm.lse ? prm.lse + (size_t)seg * R : nullptr, nullptr};
    // CTA pp's partial of this segment is in its warp slot 0, except that
    // CTA p_hi left its NW warp partials when the segment was only the
    // first piece of its range
    const bool raw = s_raw[a];
    const float *cta0 = prm.ws + ((size_t)(s_ord[a] + plo) * NW) * stride;
    const float *raw0 = prm.ws + ((size_t)(s_ord[a] + phi) * NW) * stride;
    const int nA = raw ? phi - plo : phi - plo + 1;
    if (!(ws_ok(cta0, (size_t)nA * NW * stride) && (!raw || ws_ok(raw0, (size_t)NW * stride)) &&
          chk(seg < (long long)c.B * c.H, 10)))
      continue;
    // Verify: where a merge straight from L2 would wait on six or more round
    // trips (many rows and partials per lane), the segment's partials are
    // first gathered into the stage memory (free now) by one bulk copy each.
    // Measured: the 20-row grouped-query verify (ten rounds) 58.6 -> 56.4 us;
    // the 5-row verify's four rounds gained nothing.  The drafts' merges
    // take one to three rounds; compiled into them (even when not taken) the
    // gathering cost 1-1.5 us per draft call.
    const float *srcA = cta0, *srcB = raw0;
    int kA = NW * stride;
    const int ns = nA + (raw ? NW / ncg : 0);
    const uint32_t n_st = (uint32_t)(nA + (raw ? NW : 0)) * stride * 4;
    if (MODE == QS_VERIFY_INT8 && merge_rounds(R, ns) >= 6 && n_st <= (uint32_t)L::kBarOff) {
      __syncthreads();  // the previous merge's reads of the stage memory are done
      if (threadIdx.x == 0) {
        fence_proxy_async_global();
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(mrg_bar, n_st);
        for (int k = 0; k < nA; ++k)
          bulk_g2s(sbase + k * stride * 4, cta0 + (size_t)k * NW * stride, stride * 4, mrg_bar);
        if (raw) bulk_g2s(sbase + nA * stride * 4, raw0, NW * stride * 4, mrg_bar);
      }
      const bool ok = __syncthreads_and(mbar_wait(mrg_bar, (uint32_t)(n_mrg & 1), prm.wait_ns));
      ++n_mrg;
      if (!ok) {
        if (threadIdx.x == 0) atomicOr(&c.state[(size_t)b * QS_STATE_WORDS + QS_ST_ERR], QS_DEV_TIMEOUT);
        continue;
      }
      srcA = reinterpret_cast<const float *>(smem);
      srcB = srcA + (size_t)nA * stride;
      kA = stride;
    }
    merge_rows(srcA, 0, kA, nA, srcB, stride, ncg * stride, ns, R, mo);
  }
}

// --------------------------------------------------------------- host side
struct DevInfo {
  int ready[16];
  int grid[16];
};
DevInfo g_dev[64];

// Resident CTAs of one split-kernel variant on a device (set up once).
template <int MODE, bool PK, int UB, int NW>
qs_status grid_for_device(int dev, int &P) {
  DevInfo &di = g_dev[dev];
  constexpr int v = 2 * MODE + (PK ? 1 : 0) + (UB == 2 ? 4 : 0) + (NW == 8 ? 8 : 0);
  if (!__atomic_load_n(&di.ready[v], __ATOMIC_ACQUIRE)) {
    const int smem = Layout<MODE>::kSmemBytes;
    if (cudaFuncSetAttribute(split_kernel<MODE, PK, UB, NW>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem) != cudaSuccess)
      return QS_ERR_CUDA;
    int sms = 0, occ = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return QS_ERR_CUDA;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, split_kernel<MODE, PK, UB, NW>, NW * 32,
                                                      smem) != cudaSuccess)
      return QS_ERR_CUDA;
    if (occ < 1) return QS_ERR_CUDA;
    di.grid[v] = sms * occ;
    __atomic_store_n(&di.ready[v], 1, __ATOMIC_RELEASE);
  }
  P = di.grid[v];
  return QS_OK;
}

template <int UB>
qs_status grid_size_ub(int dev, qs_mode mode, bool packed, int ncg, int &P) {
  if (mode == QS_DRAFT_UPPER4)
    return packed ? grid_for_device<QS_DRAFT_UPPER4, true, UB, kWarps>(dev, P)
                  : grid_for_device<QS_DRAFT_UPPER4, false, UB, kWarps>(dev, P);
  return ncg <= 2 ? grid_for_device<QS_VERIFY_INT8, false, UB, kVerifyWarps>(dev, P)
                  : grid_for_device<QS_VERIFY_INT8, false, UB, kWarps>(dev, P);
}

qs_status grid_size(qs_mode mode, bool packed, int upper_bits, int ncg, int &P) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return QS_ERR_CUDA;
  if (dev < 0 || dev >= 64) return QS_ERR_UNSUPPORTED;
  return upper_bits == 2 ? grid_size_ub<2>(dev, mode, packed, ncg, P)
                         : grid_size_ub<4>(dev, mode, packed, ncg, P);
}

// Workspace: (P + B H) x 12 warp slots of R rows (R = group x n_q); an
// eight-warp launch packs its pieces eight slots apart, inside that size.
size_t ws_bytes(int P, int B, int H, int R) {
  return (size_t)(P + (size_t)B * H) * kWarps * (size_t)(R * kD + 2 * kMaxR) * sizeof(float);
}

template <int MODE, bool PK, int UB, int NW>
qs_status launch(const Params &prm, cudaStream_t s) {
  return launch_pdl(split_kernel<MODE, PK, UB, NW>, dim3(prm.P), dim3(NW * 32),
                    Layout<MODE>::kSmemBytes, s, prm);
}

template <int UB>
qs_status launch_ub(qs_mode mode, bool packed, const Params &prm, cudaStream_t st) {
  if (mode == QS_VERIFY_INT8)
    return prm.ncg <= 2 ? launch<QS_VERIFY_INT8, false, UB, kVerifyWarps>(prm, st)
                        : launch<QS_VERIFY_INT8, false, UB, kWarps>(prm, st);
  return packed ? launch<QS_DRAFT_UPPER4, true, UB, kWarps>(prm, st)
                : launch<QS_DRAFT_UPPER4, false, UB, kWarps>(prm, st);
}

}  // namespace
}  // namespace qs

using namespace qs;

extern "C" {

qs_status qs_attn_workspace_size_gqa(const qs_cache *c, int32_t n_q, int32_t group,
                                     size_t *bytes) {
  qs_status s = check_cache(c);
  if (s != QS_OK) return s;
  if (!bytes || n_q < 1 || n_q > kMaxQ || group < 1 || group * n_q > kMaxR) return QS_ERR_ARG;
  int P0 = 0, P1 = 0, P2 = 0;
  if ((s = grid_size(QS_DRAFT_UPPER4, false, c->upper_bits, 1, P0)) != QS_OK) return s;
  if ((s = grid_size(QS_DRAFT_UPPER4, true, c->upper_bits, 1, P1)) != QS_OK) return s;
  if ((s = grid_size(QS_VERIFY_INT8, false, c->upper_bits, (group * n_q + 7) / 8, P2)) != QS_OK) return s;
  const int P = P0 > P1 ? (P0 > P2 ? P0 : P2) : (P1 > P2 ? P1 : P2);
  *bytes = ws_bytes(P, c->B, c->H, group * n_q);
  return QS_OK;
}

qs_status qs_attn_workspace_size(const qs_cache *c, int32_t n_q, size_t *bytes) {
  return qs_attn_workspace_size_gqa(c, n_q, 1, bytes);
}

}  // extern "C"

namespace {

// Validation, launch configuration and launch shared by the entry points.
qs_status decode(const qs_cache *c, qs_mode mode, const uint16_t *q, int32_t n_q, int32_t group,
                 float softmax_scale, uint16_t *out, float *lse, void *workspace,
                 size_t workspace_bytes, uint64_t wait_ns, int no_issue, const uint16_t *k_new,
                 const uint16_t *v_new, int32_t n_new, qs_stream_t stream) {
  qs_status s = check_cache(c);
  if (s != QS_OK) return s;
  if (!q || !out || n_q < 1 || n_q > kMaxQ || group < 1 || group * n_q > kMaxR) return QS_ERR_ARG;
  if (mode != QS_DRAFT_UPPER4 && mode != QS_VERIFY_INT8) return QS_ERR_ARG;
  if (!(softmax_scale > 0.f) || !isfinite(softmax_scale)) return QS_ERR_ARG;
  if (!aligned16(q) || !aligned16(out) || (lse && !aligned16(lse))) return QS_ERR_ALIGN;
  Params prm;
  prm.c = *c;
  prm.q = q;
  prm.out = out;
  prm.lse = lse;
  prm.n_q = n_q;
  prm.R = group * n_q;
  prm.ncg = (prm.R + 7) / 8;
  prm.sl2 = softmax_scale * 1.4426950408889634f;
  prm.wait_ns = wait_ns;
  prm.no_issue = no_issue;
  prm.k_new = k_new;
  prm.v_new = v_new;
  prm.n_new = n_new;
  prm.ws_floats = workspace_bytes / sizeof(float);
  const bool packed = (mode == QS_DRAFT_UPPER4 && prm.R <= 4);
  if ((s = grid_size(mode, packed, c->upper_bits, prm.ncg, prm.P)) != QS_OK) return s;
  if (!workspace || !aligned16(workspace) ||
      workspace_bytes < ws_bytes(prm.P, c->B, c->H, prm.R))
    return QS_ERR_WORKSPACE;
  prm.ws = static_cast<float *>(workspace);
  cudaStream_t st = (cudaStream_t)stream;
  return c->upper_bits == 2 ? launch_ub<2>(mode, packed, prm, st)
                            : launch_ub<4>(mode, packed, prm, st);
}

}  // namespace

extern "C" {

qs_status qs_attn_decode_gqa(const qs_cache *c, qs_mode mode, const uint16_t *q, int32_t n_q,
                             int32_t group, float softmax_scale, uint16_t *out, float *lse,
                             void *workspace, size_t workspace_bytes, qs_stream_t stream) {
  return decode(c, mode, q, n_q, group, softmax_scale, out, lse, workspace, workspace_bytes,
                kWaitLimitNs, 0, nullptr, nullptr, 0, stream);
}

qs_status qs_attn_decode_append(const qs_cache *c, qs_mode mode, const uint16_t *k_new,
                                const uint16_t *v_new, int32_t n_new, const uint16_t *q,
                                int32_t n_q, int32_t group, float softmax_scale, uint16_t *out,
                                float *lse, void *workspace, size_t workspace_bytes,
                                qs_stream_t stream) {
  if (!k_new || !v_new || n_new < 1 || n_new > kRing) return QS_ERR_ARG;
  if (!aligned16(k_new) || !aligned16(v_new)) return QS_ERR_ALIGN;
  return decode(c, mode, q, n_q, group, softmax_scale, out, lse, workspace, workspace_bytes,
                kWaitLimitNs, 0, k_new, v_new, n_new, stream);
}

qs_status qs_attn_decode(const qs_cache *c, qs_mode mode, const uint16_t *q, int32_t n_q,
                         float softmax_scale, uint16_t *out, float *lse, void *workspace,
                         size_t workspace_bytes, qs_stream_t stream) {
  return qs_attn_decode_gqa(c, mode, q, n_q, 1, softmax_scale, out, lse, workspace,
                            workspace_bytes, stream);
}

// Test entry, not declared in include/qs.h: qs_attn_decode_gqa with every
// pipeline wait limited to wait_ns (1 us .. 100 ms) and no copy ever issued,
// so the first wait of every warp runs out.  It exercises the failure path
// of the kernel without a fault: the sequences get QS_DEV_TIMEOUT, the
// kernel returns within a few multiples of wait_ns, no output is written, and
// the arrival counters end at zero, so the next ordinary call on the cache is
// valid.
qs_status qs_test_attn_decode_timeout(const qs_cache *c, qs_mode mode, const uint16_t *q,
                                      int32_t n_q, int32_t group, float softmax_scale,
                                      uint16_t *out, float *lse, void *workspace,
                                      size_t workspace_bytes, uint64_t wait_ns,
                                      qs_stream_t stream) {
  if (wait_ns < 1000ull || wait_ns > 100000000ull) return QS_ERR_ARG;
  return decode(c, mode, q, n_q, group, softmax_scale, out, lse, workspace, workspace_bytes,
                wait_ns, 1, nullptr, nullptr, 0, stream);
}

}  // extern "C"

#if QS_CHECKED
extern "C" int qs_checked_failures_quantize(unsigned long long *out2, int reset);

// Checked build only (-DQS_CHECKED=1): the number of failed bounds checks of
// the attention and quantization kernels since the last reset, and the tag of
// the first (1 shared-memory load, 2 copy destination, 3 group index, 4 buffer
// row, 6 ldmatrix row, 7 partial slot, 8 merge source, 9 query row, 10 output
// head, 11 tail partials, 20 flush group, 21 metadata position, 22 prefill
// group rows, 23 prefill buffer rows).  reset != 0 zeroes the counts.
// Returns 0, or 1 if a CUDA call failed.
extern "C" int qs_checked_failures(unsigned long long *count, unsigned int *first_tag, int reset) {
  unsigned long long a[2], q[2];
  if (cudaMemcpyFromSymbol(a, g_check_fail, sizeof(a)) != cudaSuccess) return 1;
  if (qs_checked_failures_quantize(q, reset)) return 1;
  if (reset) {
    const unsigned long long z[2] = {0, 0};
    if (cudaMemcpyToSymbol(g_check_fail, z, sizeof(z)) != cudaSuccess) return 1;
  }
  *count = a[0] + q[0];
  *first_tag = (unsigned int)(a[0] ? a[1] : q[1]);
  return 0;
}
#endif
