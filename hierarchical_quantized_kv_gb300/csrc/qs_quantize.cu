// qs_quantize.cu -- quantize-on-flush: one G-token fp16 buffer half becomes
// one hierarchical group (C_U / C_L nibble planes plus fp16 scale and zero).
//
// Source: "QuantSpec: Self-Speculative Decoding with Hierarchical Quantized
// KV Cache" (Pith review), "What carries the argument" (C_INT8 = 2^4 C_U +
// C_L, one shared scale and zero-point, a half is quantized once every G
// steps) and Figure 7 / Appendix D (keys per channel over G tokens, values
// per token over G channels, asymmetric).  "QuantSpec Guide", quantizer
// section: min/max, 255 levels, round, clamp, q >> 4 and q & 15.
//
// Convention QS-RN-v1 (every fp32 step IEEE round-to-nearest-even; this file
// is compiled without fast-math so __fsub_rn / __fdiv_rn are exact IEEE):
//   r = max - min, s = r == 0 ? 0 : fp16_round_up(r / 255), z = min (+0 if 0),
//   q = s == 0 ? 0 : clamp(rne((x - z) / s), 0, 255).
#include "qs_common.cuh"

namespace qs {

namespace {

constexpr int kParts = 4;           // CTAs per (head, sequence)
constexpr int kSlice = kD / kParts;  // key channels / value tokens per CTA
// Warps per CTA: a flush is one wave of small CTAs, so its time is one
// CTA's chain of phases, and sixteen warps halve the per-thread work of
// every phase but the packing (flush 14 -> 11.5 µs); a prefill is many
// waves, where eight warps keep more CTAs resident (379 against 426 µs).
constexpr int kFlushWarps = 16, kPrefillWarps = 8;
// Group quarters per quantizing CTA of a prefill, loads pipelined one ahead.
#ifndef QS_PREFILL_QUARTERS
#define QS_PREFILL_QUARTERS 8
#endif
constexpr int kPrefillQuarters = QS_PREFILL_QUARTERS;

// One CTA owns key channels [32p, 32p+32) (one 16-byte column of every key
// row) and value tokens [32p, 32p+32) (value quarter p).
template <int QW>
struct FlushSmem {
  __half k[kG][kSlice];     // keys of the slice   [token][channel - 32p]
  __half v[kSlice][kD];     // values of the slice [token - 32p][channel]
  uint8_t kc[kG][kSlice];   // key codes
  uint8_t vc[kSlice][kD];   // value codes
  float kmin[QW][kSlice], kmax[QW][kSlice];
  uint16_t ks[kSlice], kz[kSlice], vs[kSlice], vz[kSlice];
  int act, base, g;
};

__device__ __forceinline__ void scale_zero(float mn, float mx, uint16_t &s_bits, uint16_t &z_bits,
                                           float &sf, float &zf) {
  const float r = __fsub_rn(mx, mn);
  __half s = __float2half_ru(__fdiv_rn(r, 255.0f));
  if (r == 0.0f) s = __ushort_as_half(0);
  s_bits = __half_as_ushort(s);
  // exact (mn is an fp16 value); a zero minimum is stored as +0
  z_bits = (mn == 0.0f) ? (uint16_t)0 : __half_as_ushort(__float2half_rn(mn));
  sf = __half2float(s);
  zf = mn;
}

// q = clamp(rne(fl((x - z) / s)), 0, 255) with fl the IEEE fp32 quotient, as
// QS-RN-v1 defines it, without a divide per element: rf = fl(1 / s) is exact
// to 2^-24, so u' = fl((x - z) * rf) is within 2^-14 of fl((x - z) / s) for
// every |u| < 256 (u <= 255 (1 + 2^-23) since s >= r / 255).  Both round to
// the same integer unless u' lies within 2^-12 of a half-integer; there the
// exact quotient decides (about one element in 2^11).  Four elements at a
// time, with one warp vote: the exact quotient is computed only when some
// lane of the warp has an element that close to a tie, and then only for
// those elements.  Rounding, clamping to [0, 255] and conversion are one
// saturating conversion.  A zero scale gives code 0 (then rf is +inf and a
// is 0 or positive: the code is forced).  Called by whole warps.
__device__ __forceinline__ void codes4(const float (&x)[4], const float (&zf)[4],
                                       const float (&sf)[4], const float (&rf)[4],
                                       uint32_t (&q)[4]) {
  float a[4], ue[4];
  bool near[4], any = false;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    a[i] = __fsub_rn(x[i], zf[i]);
    ue[i] = __fmul_rn(a[i], rf[i]);
    near[i] = fabsf(__fsub_rn(ue[i], rintf(ue[i]))) > 0.5f - 0x1p-12f;
    any |= near[i];
  }
  if (__any_sync(0xffffffffu, any)) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (near[i]) ue[i] = __fdiv_rn(a[i], sf[i]);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t v;
    asm("cvt.rni.sat.u8.f32 %0, %1;" : "=r"(v) : "f"(ue[i]));
    q[i] = sf[i] == 0.0f ? 0u : v;
  }
}

// Two 4-bit planes' bytes from four 8-bit codes per word: words a and b hold
// codes 4k..4k+3 and 4k+4..4k+7 (channel pairs 2k, 2k+1, 2k+2, 2k+3); the
// result's byte i holds pair i's two nibbles (the first code's in the low
// nibble): upper nibbles (hi) or lower nibbles (lo) of the codes.
__device__ __forceinline__ uint32_t pair_nibbles(uint32_t a, uint32_t b, bool hi) {
  const uint32_t na = (hi ? a >> 4 : a) & 0x0F0F0F0Fu, nb = (hi ? b >> 4 : b) & 0x0F0F0F0Fu;
  // byte 0 of (n | n >> 4): nibble of byte 0, then of byte 1; byte 2: of bytes 2, 3
  return prmt(na | (na >> 4), nb | (nb >> 4), 0x6420);
}

// Token held by nibble position p of a 16-byte value row (quarter layout).
__device__ __forceinline__ int vperm(int p) {
  return 16 * ((p >> 1) & 1) + 8 * (p & 1) + 2 * (p >> 3) + ((p >> 2) & 1);
}

// Position of channel c in a key scale / zero row (inverse of the header's
// map p -> 32((p>>3)&3) + 8(p>>5) + 2((p>>2)&1) + ((p>>1)&1) + 4(p&1)).
__device__ __forceinline__ int kmeta_pos(int c) {
  return ((c >> 2) & 1) | ((c & 1) << 1) | (((c >> 1) & 1) << 2) | (((c >> 5) & 3) << 3) |
         (((c >> 3) & 3) << 5);
}

// Position of token t in a value scale / zero row (inverse of
// p -> 32(p>>5) + ((p>>2)&7) + 16((p>>1)&1) + 8(p&1)).
__device__ __forceinline__ int vmeta_pos(int t) {
  return ((t >> 3) & 1) | (((t >> 4) & 1) << 1) | ((t & 7) << 2) | ((t >> 5) << 5);
}

// Two-bit draft layout: four consecutive 32-bit words w[0..3] of a 4-bit
// upper plane (nibble C_U = 4 C_U2 + M2) become two words of the group's
// C_U2 plane and two of its M2 plane (second 4 KB of the group's 8 KB).
// Word k of each holds, in nibble position j, the two-bit field of word 2k's
// nibble j in bits 4j..4j+1 and of word 2k+1's nibble j in bits 4j+2..4j+3.
// base: the group's upper plane; off: byte offset of w[0] in the 4-bit plane
// (a multiple of 16), so the two words go to off / 2.
__device__ __forceinline__ void store_upper2(uint8_t *base, size_t off, const uint32_t (&w)[4]) {
  uint2 u, m;
  u.x = ((w[0] >> 2) & 0x33333333u) | (w[1] & 0xCCCCCCCCu);
  u.y = ((w[2] >> 2) & 0x33333333u) | (w[3] & 0xCCCCCCCCu);
  m.x = (w[0] & 0x33333333u) | ((w[1] & 0x33333333u) << 2);
  m.y = (w[2] & 0x33333333u) | ((w[3] & 0x33333333u) << 2);
  *reinterpret_cast<uint2 *>(base + off / 2) = u;
  *reinterpret_cast<uint2 *>(base + (size_t)kG * kD / 4 + off / 2) = m;
}

// Asynchronous 16-byte copy global -> shared through the load/store path
// (cached in L2 only; addresses 16-byte aligned), its commit group, and the
// wait until at most N of the thread's groups are still in flight.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// A CTA's share of a group is a quarter: key channels [32 part, 32 part +
// 32) and value tokens [32 part, 32 part + 32).
// 1. loads of a group quarter into kt / vt: the key column slice (64 B of
// each of 128 rows) and 32 value rows; ASYNC: as cp.async copies, one commit
// group (the caller waits for it before quantize_loaded).
template <int QW, bool ASYNC>
__device__ __forceinline__ void load_part(__half (*kt)[kSlice], __half (*vt)[kD], const __half *gk,
                                          const __half *gv, int part, int tid) {
  constexpr int kQThreads = 32 * QW;
  for (int e = tid; e < kG * 4; e += kQThreads) {  // 4 x 16 B per key row
    const int t = e >> 2, q = e & 3;
    const uint4 *src = reinterpret_cast<const uint4 *>(gk + (size_t)t * kD + part * kSlice) + q;
    if (ASYNC)
      cp_async16(smem_addr(&kt[t][0]) + 16 * q, src);
    else
      reinterpret_cast<uint4 *>(&kt[t][0])[q] = *src;
  }
  for (int e = tid; e < kSlice * kD / 8; e += kQThreads) {
    const uint4 *src = reinterpret_cast<const uint4 *>(gv + (size_t)part * kSlice * kD) + e;
    if (ASYNC)
      cp_async16(smem_addr(&vt[0][0]) + 16 * e, src);
    else
      reinterpret_cast<uint4 *>(&vt[0][0])[e] = *src;
  }
  if (ASYNC) cp_async_commit();
}

// Phases 2-7 of a group quarter whose rows are in kt / vt (all loads landed
// and visible to the CTA).
template <int QW>
__device__ void quantize_loaded(FlushSmem<QW> &S, const __half (*kt)[kSlice],
                                const __half (*vt)[kD], const qs_cache &c, size_t grp, int part,
                                int tid) {
  constexpr int kQWarps = QW, kQThreads = 32 * QW;
  const int warp = tid >> 5, lane = tid & 31;

  // 2. keys: min / max per channel, warp w over tokens kG/kQWarps w onwards
  {
    constexpr int kTw = kG / kQWarps;
    float mn = INFINITY, mx = -INFINITY;
    for (int t = kTw * warp; t < kTw * warp + kTw; ++t) {
      const float x = __half2float(kt[t][lane]);
      mn = fminf(mn, x);
      mx = fmaxf(mx, x);
    }
    S.kmin[warp][lane] = mn;
    S.kmax[warp][lane] = mx;
  }
  // 3. values: one warp per token, min / max over the 128 channels, codes
  for (int t = warp; t < kSlice; t += kQWarps) {
    const __half2 *row = reinterpret_cast<const __half2 *>(&vt[t][4 * lane]);
    const float2 a = __half22float2(row[0]), bb = __half22float2(row[1]);
    float mn = fminf(fminf(a.x, a.y), fminf(bb.x, bb.y));
    float mx = fmaxf(fmaxf(a.x, a.y), fmaxf(bb.x, bb.y));
    for (int o = 16; o > 0; o >>= 1) {
      mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    }
    uint16_t sb, zb;
    float sf, zf;
    scale_zero(mn, mx, sb, zb, sf, zf);
    if (lane == 0) {
      S.vs[t] = sb;
      S.vz[t] = zb;
    }
    const float rf = __frcp_rn(sf);
    uint32_t q[4];
    codes4({a.x, a.y, bb.x, bb.y}, {zf, zf, zf, zf}, {sf, sf, sf, sf}, {rf, rf, rf, rf}, q);
    *reinterpret_cast<uint32_t *>(&S.vc[t][4 * lane]) = q[0] | (q[1] << 8) | (q[2] << 16) | (q[3] << 24);
  }
  __syncthreads();
  if (tid < kSlice) {
    float mn = S.kmin[0][tid], mx = S.kmax[0][tid];
    for (int w = 1; w < kQWarps; ++w) {
      mn = fminf(mn, S.kmin[w][tid]);
      mx = fmaxf(mx, S.kmax[w][tid]);
    }
    uint16_t sb, zb;
    float sf, zf;
    scale_zero(mn, mx, sb, zb, sf, zf);
    S.ks[tid] = sb;
    S.kz[tid] = zb;
  }
  __syncthreads();

  // 4. key codes: thread = channel pair j (16 pairs) x kTc tokens
  {
    constexpr int kTc = kG * 16 / kQThreads;
    const int j = tid & 15, t0 = (tid >> 4) * kTc;
    const float s0 = __half2float(__ushort_as_half(S.ks[2 * j]));
    const float s1 = __half2float(__ushort_as_half(S.ks[2 * j + 1]));
    const float z0 = __half2float(__ushort_as_half(S.kz[2 * j]));
    const float z1 = __half2float(__ushort_as_half(S.kz[2 * j + 1]));
    const float r0 = __frcp_rn(s0), r1 = __frcp_rn(s1);
    static_assert(kTc % 2 == 0, "two tokens per step");
#pragma unroll
    for (int t = t0; t < t0 + kTc; t += 2) {
      const float2 x = __half22float2(*reinterpret_cast<const __half2 *>(&kt[t][2 * j]));
      const float2 y = __half22float2(*reinterpret_cast<const __half2 *>(&kt[t + 1][2 * j]));
      uint32_t q[4];
      codes4({x.x, x.y, y.x, y.y}, {z0, z1, z0, z1}, {s0, s1, s0, s1}, {r0, r1, r0, r1}, q);
      *reinterpret_cast<uint16_t *>(&S.kc[t][2 * j]) = (uint16_t)(q[0] | (q[1] << 8));
      *reinterpret_cast<uint16_t *>(&S.kc[t + 1][2 * j]) = (uint16_t)(q[2] | (q[3] << 8));
    }
  }
  __syncthreads();

  if (tid < kG) {
    // 5. key planes: bytes [16p, 16p+16) of token row tid (channels 2i, 2i+1)
    // the row's 32 codes in two 16-byte loads; word m of a plane row holds
    // channel pairs 4m..4m+3 (codes 8m..8m+7)
    const uint4 ra = *reinterpret_cast<const uint4 *>(&S.kc[tid][0]);
    const uint4 rb = *reinterpret_cast<const uint4 *>(&S.kc[tid][16]);
    const uint32_t cw[8] = {ra.x, ra.y, ra.z, ra.w, rb.x, rb.y, rb.z, rb.w};
    uint32_t wu[4], wl[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      wu[m] = pair_nibbles(cw[2 * m], cw[2 * m + 1], true);
      wl[m] = pair_nibbles(cw[2 * m], cw[2 * m + 1], false);
    }
    if (c.upper_bits == 2)
      store_upper2(c.k_upper + grp * kG * (kD / 2), 16 * (4 * tid + part), wu);
    else
      reinterpret_cast<uint4 *>(c.k_upper + (grp * kG + tid) * (kD / 2))[part] =
          make_uint4(wu[0], wu[1], wu[2], wu[3]);
    reinterpret_cast<uint4 *>(c.k_lower + (grp * kG + tid) * (kD / 2))[part] =
        make_uint4(wl[0], wl[1], wl[2], wl[3]);
  } else if (tid < kG + kD) {
    // 6. value quarter p: row d = 16 bytes, nibble position q holds token vperm(q)
    const int d = tid - kG;
    uint32_t wu[4] = {0, 0, 0, 0}, wl[4] = {0, 0, 0, 0};
#pragma unroll
    for (int q = 0; q < 32; ++q) {
      const uint32_t code = S.vc[vperm(q)][d];
      wu[q >> 3] |= (code >> 4) << (4 * (q & 7));
      wl[q >> 3] |= (code & 15u) << (4 * (q & 7));
    }
    const size_t row = (grp * 4 + part) * kD + d;
    if (c.upper_bits == 2)
      store_upper2(c.v_upper + grp * kG * (kD / 2), 16 * (part * kD + d), wu);
    else
      reinterpret_cast<uint4 *>(c.v_upper)[row] = make_uint4(wu[0], wu[1], wu[2], wu[3]);
    reinterpret_cast<uint4 *>(c.v_lower)[row] = make_uint4(wl[0], wl[1], wl[2], wl[3]);
  }
  // 7. metadata: key scale / zero of the channel slice, value scale / zero of the quarter
  if (tid < kSlice) {
    uint16_t *m = c.meta + grp * 4 * 128;
    int kp = kmeta_pos(part * kSlice + tid), vp = vmeta_pos(part * kSlice + tid);
    if (!chk(kp >= 0 && kp < 128 && vp >= 0 && vp < 128, 21)) kp = vp = 0;
    m[QS_META_K_SCALE * 128 + kp] = S.ks[tid];
    m[QS_META_K_ZERO * 128 + kp] = S.kz[tid];
    m[QS_META_V_SCALE * 128 + vp] = S.vs[tid];
    m[QS_META_V_ZERO * 128 + vp] = S.vz[tid];
  }
}

// One CTA's share of quantizing a group of G tokens whose fp16 key and value
// rows (D channels each, row stride D) start at gk and gv: key channels
// [32 part, 32 part + 32) and value tokens [32 part, 32 part + 32), written
// as group `grp` (index into the [B][H][cap] group arrays).  32 QW threads.
template <int QW>
__device__ void quantize_part(FlushSmem<QW> &S, const __half *gk, const __half *gv,
                              const qs_cache &c, size_t grp, int part, int tid) {
  // checked build: a group index out of the arrays writes nothing (the same
  // for every thread of the CTA)
  if (!chk(in_range(grp, 1, (size_t)c.B * c.H * c.cap_groups), 20)) return;
  load_part<QW, false>(S.k, S.v, gk, gv, part, tid);
  __syncthreads();
  quantize_loaded(S, S.k, S.v, c, grp, part, tid);
}

// The prefill's shared memory: a second pair of row buffers (first, so the
// asynchronous copies stay 16-byte aligned) and the flush's.
template <int QW>
struct PrefillSmem {
  __half k1[kG][kSlice];
  __half v1[kSlice][kD];
  FlushSmem<QW> f;
};

}  // namespace

// n_next >= 0: flush the sequences whose buffer cannot take n_next more
// tokens (qs_need_flush's rule; mask unused); else the masked ones (all
// without a mask).
__global__ void __launch_bounds__(32 * kFlushWarps)
    flush_kernel(qs_cache c, const uint8_t *__restrict__ mask, int n_next) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  FlushSmem<kFlushWarps> &S = *reinterpret_cast<FlushSmem<kFlushWarps> *>(smem_raw);
  const int part = blockIdx.x, h = blockIdx.y, b = blockIdx.z, tid = threadIdx.x;
  pdl_trigger();
  pdl_wait();
  int32_t *st = c.state + (size_t)b * QS_STATE_WORDS;
  if (tid == 0) {
    const int fill = st[QS_ST_FILL], pending = st[QS_ST_PENDING], ng = st[QS_ST_N_GROUPS];
    int act = n_next >= 0 ? (fill + n_next > kRing) : (mask ? (mask[b] != 0) : 1);
    const bool lead = (h == 0 && part == 0);
    if (act && fill - pending < kG) {
      if (lead) atomicOr(&st[QS_ST_ERR], QS_DEV_FLUSH_UNCOMMITTED);
      act = 0;
    } else if (act && (ng < 0 || ng >= c.cap_groups)) {
      if (lead) atomicOr(&st[QS_ST_ERR], QS_DEV_CAPACITY);
      act = 0;
    }
    S.act = act;
    S.base = st[QS_ST_HALF_BASE] & 1;
    S.g = ng;
  }
  __syncthreads();
  if (!S.act) return;
  const int base = S.base, g = S.g;
  const size_t bh = (size_t)b * c.H + h;
  const __half *gk = reinterpret_cast<const __half *>(c.buf_k) + (bh * kRing + base * kG) * kD;
  const __half *gv = reinterpret_cast<const __half *>(c.buf_v) + (bh * kRing + base * kG) * kD;

  quantize_part(S, gk, gv, c, bh * c.cap_groups + g, part, tid);
  __syncthreads();
  // every CTA of the sequence has read the old counters once the ticket
  // reaches kParts H - 1 (the planes are published by the kernel's end)
  if (tid == 0 && atom_add_acq_rel_gpu(&st[QS_ST_TICKET], 1) == kParts * c.H - 1) {
    st[QS_ST_N_GROUPS] = g + 1;
    st[QS_ST_HALF_BASE] = base ^ 1;
    st[QS_ST_FILL] -= kG;
    st[QS_ST_TICKET] = 0;
  }
}

// Bulk prefill of empty caches from a prompt (k, v: fp16 [B][H][T][D]).
// Grid (nq + 2, H, B): block x < nq quantizes group quarters [x Q, x Q + Q)
// of the sequence's head (quarter i: part i % 4 of group i / 4; Q =
// kPrefillQuarters), the next quarter's rows copied into the second buffer
// while the current one is quantized; the last two blocks copy buffer halves
// 0 and 1.  The CTA that arrives last on the sequence's ticket writes the
// counters, so every CTA reads the old (empty) ones first.
__global__ void __launch_bounds__(32 * kPrefillWarps) prefill_kernel(qs_cache c, const uint16_t *__restrict__ k,
                                                     const uint16_t *__restrict__ v, int T,
                                                     const int32_t *__restrict__ len, int nq) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  PrefillSmem<kPrefillWarps> &PS = *reinterpret_cast<PrefillSmem<kPrefillWarps> *>(smem_raw);
  FlushSmem<kPrefillWarps> &S = PS.f;
  const int x = blockIdx.x, h = blockIdx.y, b = blockIdx.z, tid = threadIdx.x;
  pdl_trigger();
  pdl_wait();
  int32_t *st = c.state + (size_t)b * QS_STATE_WORDS;
  if (tid == 0) {
    const int L = len[b];
    const bool lead = (h == 0 && x == 0);
    int act = 1, ng = 0;
    if (st[QS_ST_N_GROUPS] != 0 || st[QS_ST_FILL] != 0 || st[QS_ST_PENDING] != 0 || L < 0 ||
        L > T) {
      if (lead) atomicOr(&st[QS_ST_ERR], QS_DEV_PREFILL);
      act = 0;
    } else {
      ng = L > 2 * kG ? (L - 2 * kG + kG - 1) / kG : 0;
      if (ng > c.cap_groups) {
        if (lead) atomicOr(&st[QS_ST_ERR], QS_DEV_CAPACITY);
        act = 0;
      }
    }
    S.act = act;
    S.g = ng;
    S.base = act ? L - ng * kG : 0;  // fill
  }
  __syncthreads();
  if (!S.act) return;
  const int ng = S.g, fill = S.base;
  const size_t bh = (size_t)b * c.H + h;
  const uint16_t *kp = k + bh * T * kD, *vp = v + bh * T * kD;
  if (x < nq) {
    const int q0 = x * kPrefillQuarters, q1 = min(q0 + kPrefillQuarters, 4 * ng);
    const __half *kh = reinterpret_cast<const __half *>(kp), *vh = reinterpret_cast<const __half *>(vp);
    // the rows of quarter i go to buffer i % 2 (one commit group per quarter:
    // a quarter whose rows fail the checked build's range check commits an
    // empty one, so the waits below keep counting quarters)
    auto load = [&](int i) {
      const int g = i >> 2;
      if (!chk(in_range(((size_t)g + 1) * kG, 0, (size_t)T), 22))
        cp_async_commit();
      else if (i & 1)
        load_part<kPrefillWarps, true>(PS.k1, PS.v1, kh + (size_t)g * kG * kD,
                                       vh + (size_t)g * kG * kD, i & 3, tid);
      else
        load_part<kPrefillWarps, true>(S.k, S.v, kh + (size_t)g * kG * kD,
                                       vh + (size_t)g * kG * kD, i & 3, tid);
    };
    if (q0 < q1) load(q0);
    for (int i = q0; i < q1; ++i) {
      if (i + 1 < q1) {
        load(i + 1);  // into the buffer quarter i - 1 used (free since the barrier below)
        cp_async_wait<1>();
      } else {
        cp_async_wait<0>();
      }
      __syncthreads();  // quarter i's rows, copied by every thread, are visible
      const int g = i >> 2;
      // checked build: the group's prompt rows inside the prompt array
      if (chk(in_range(((size_t)g + 1) * kG, 0, (size_t)T), 22) &&
          chk(in_range(bh * c.cap_groups + g, 1, (size_t)c.B * c.H * c.cap_groups), 20)) {
        if (i & 1)
          quantize_loaded(S, PS.k1, PS.v1, c, bh * c.cap_groups + g, i & 3, tid);
        else
          quantize_loaded(S, S.k, S.v, c, bh * c.cap_groups + g, i & 3, tid);
      }
      __syncthreads();  // the buffer and the scratch are free for the next quarters
    }
  } else {
    // buffer half x - nq: tokens i in [G half, G half + G) that are < fill
    const int i0 = (x - nq) * kG, i1 = min(i0 + kG, fill);
    const uint4 *ks = reinterpret_cast<const uint4 *>(kp + (size_t)ng * kG * kD);
    const uint4 *vs = reinterpret_cast<const uint4 *>(vp + (size_t)ng * kG * kD);
    uint4 *kd = reinterpret_cast<uint4 *>(c.buf_k + bh * kRing * kD);
    uint4 *vd = reinterpret_cast<uint4 *>(c.buf_v + bh * kRing * kD);
    if (chk(i1 <= kRing && (size_t)ng * kG + i1 <= (size_t)T, 23))
      for (int e = i0 * (kD / 8) + tid; e < i1 * (kD / 8); e += 32 * kPrefillWarps) {
        kd[e] = ks[e];
        vd[e] = vs[e];
      }
  }
  __syncthreads();
  if (tid == 0 && atom_add_acq_rel_gpu(&st[QS_ST_TICKET], 1) == (int)gridDim.x * c.H - 1) {
    st[QS_ST_N_GROUPS] = ng;
    st[QS_ST_FILL] = fill;
    st[QS_ST_PENDING] = 0;
    st[QS_ST_HALF_BASE] = 0;
    st[QS_ST_TICKET] = 0;
  }
}

}  // namespace qs

using namespace qs;

namespace {
// Opt the kernels into their dynamic shared memory once per device.
qs_status set_smem_once(const void *kernel, int smem, int *mask) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return QS_ERR_CUDA;
  if (dev >= 32 || !(__atomic_load_n(mask, __ATOMIC_ACQUIRE) & (1 << dev))) {
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
        cudaSuccess)
      return QS_ERR_CUDA;
    if (dev < 32) __atomic_fetch_or(mask, 1 << dev, __ATOMIC_RELEASE);
  }
  return QS_OK;
}
int g_flush_ready = 0, g_prefill_ready = 0;  // one bit per device ordinal below 32
}  // namespace

extern "C" qs_status qs_prefill(const qs_cache *c, const uint16_t *k, const uint16_t *v, int32_t T,
                                const int32_t *d_len, qs_stream_t stream) {
  qs_status s = check_cache(c);
  if (s != QS_OK) return s;
  if (!k || !v || !d_len || T < 0 || T > (1 << 26)) return QS_ERR_ARG;
  if (!aligned16(k) || !aligned16(v)) return QS_ERR_ALIGN;
  const int smem = (int)sizeof(PrefillSmem<kPrefillWarps>);
  if ((s = set_smem_once((const void *)prefill_kernel, smem, &g_prefill_ready)) != QS_OK) return s;
  const int gmax = T > 2 * kG ? (T - 2 * kG + kG - 1) / kG : 0;
  const int nq = (4 * gmax + kPrefillQuarters - 1) / kPrefillQuarters;
  return launch_pdl(prefill_kernel, dim3(nq + 2, c->H, c->B), dim3(32 * kPrefillWarps), smem,
                    (cudaStream_t)stream, *c, k, v, (int)T, d_len, nq);
}

extern "C" qs_status qs_quantize_flush(const qs_cache *c, const uint8_t *d_mask,
                                       qs_stream_t stream) {
  qs_status s = check_cache(c);
  if (s != QS_OK) return s;
  const int smem = (int)sizeof(FlushSmem<kFlushWarps>);
  if ((s = set_smem_once((const void *)flush_kernel, smem, &g_flush_ready)) != QS_OK) return s;
  return launch_pdl(flush_kernel, dim3(kParts, c->H, c->B), dim3(32 * kFlushWarps), smem,
                    (cudaStream_t)stream, *c, d_mask, -1);
}

extern "C" qs_status qs_quantize_flush_due(const qs_cache *c, int32_t n_next, qs_stream_t stream) {
  qs_status s = check_cache(c);
  if (s != QS_OK) return s;
  if (n_next < 0 || n_next > kRing) return QS_ERR_ARG;
  const int smem = (int)sizeof(FlushSmem<kFlushWarps>);
  if ((s = set_smem_once((const void *)flush_kernel, smem, &g_flush_ready)) != QS_OK) return s;
  return launch_pdl(flush_kernel, dim3(kParts, c->H, c->B), dim3(32 * kFlushWarps), smem,
                    (cudaStream_t)stream, *c, static_cast<const uint8_t *>(nullptr), (int)n_next);
}

#if QS_CHECKED
// Checked build only: this file's failure count and first failing tag.
extern "C" int qs_checked_failures_quantize(unsigned long long *out2, int reset) {
  if (cudaMemcpyFromSymbol(out2, g_check_fail, sizeof(g_check_fail)) != cudaSuccess) return 1;
  if (reset) {
    const unsigned long long z[2] = {0, 0};
    if (cudaMemcpyToSymbol(g_check_fail, z, sizeof(z)) != cudaSuccess) return 1;
  }
  return 0;
}
#endif
