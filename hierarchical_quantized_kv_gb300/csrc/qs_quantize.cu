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

struct FlushSmem {
  __half k[kG][kD];      // oldest buffer half, keys  [token][channel]
  __half v[kG][kD];      // values
  uint8_t kc[kG][kD];    // 8-bit key codes   [token][channel]
  uint8_t vc[kG][kD];    // 8-bit value codes [token][channel]
  float kmin[2][kD], kmax[2][kD];
  uint16_t ks[kD], kz[kD], vs[kG], vz[kG];
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

__device__ __forceinline__ uint32_t code_of(float x, float zf, float sf) {
  if (sf == 0.0f) return 0;
  const int q = __float2int_rn(__fdiv_rn(__fsub_rn(x, zf), sf));
  return (uint32_t)min(max(q, 0), 255);
}

// Token held by nibble position p of a 16-byte value row (quarter layout).
__device__ __forceinline__ int vperm(int p) {
  return 16 * ((p >> 1) & 1) + 8 * (p & 1) + 2 * (p >> 3) + ((p >> 2) & 1);
}

}  // namespace

__global__ void __launch_bounds__(256) flush_kernel(qs_cache c, const uint8_t *__restrict__ mask) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  FlushSmem &S = *reinterpret_cast<FlushSmem *>(smem_raw);
  const int h = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
  int32_t *st = c.state + (size_t)b * QS_STATE_WORDS;
  if (tid == 0) {
    int act = mask ? (mask[b] != 0) : 1;
    const int fill = st[QS_ST_FILL], pending = st[QS_ST_PENDING], ng = st[QS_ST_N_GROUPS];
    if (act && fill - pending < kG) {
      if (h == 0) atomicOr(&st[QS_ST_ERR], QS_DEV_FLUSH_UNCOMMITTED);
      act = 0;
    } else if (act && (ng < 0 || ng >= c.cap_groups)) {
      if (h == 0) atomicOr(&st[QS_ST_ERR], QS_DEV_CAPACITY);
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

  // 1. the oldest half: ring slots base*G .. base*G + G - 1 (contiguous)
  {
    const uint4 *gk = reinterpret_cast<const uint4 *>(c.buf_k + (bh * kRing + base * kG) * kD);
    const uint4 *gv = reinterpret_cast<const uint4 *>(c.buf_v + (bh * kRing + base * kG) * kD);
    uint4 *sk = reinterpret_cast<uint4 *>(&S.k[0][0]);
    uint4 *sv = reinterpret_cast<uint4 *>(&S.v[0][0]);
    for (int e = tid; e < kG * kD / 8; e += 256) {
      sk[e] = gk[e];
      sv[e] = gv[e];
    }
  }
  __syncthreads();

  // 2. keys: min / max per channel over the G tokens (two halves of tokens)
  {
    const int d = tid & (kD - 1), part = tid >> 7;
    float mn = INFINITY, mx = -INFINITY;
    for (int t = part * 64; t < part * 64 + 64; ++t) {
      const float x = __half2float(S.k[t][d]);
      mn = fminf(mn, x);
      mx = fmaxf(mx, x);
    }
    S.kmin[part][d] = mn;
    S.kmax[part][d] = mx;
  }
  // 3. values: one warp per token, min / max over the D channels, then codes
  {
    const int warp = tid >> 5, lane = tid & 31;
    for (int t = warp; t < kG; t += 8) {
      const __half2 *row = reinterpret_cast<const __half2 *>(&S.v[t][4 * lane]);
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
      const uint32_t q0 = code_of(a.x, zf, sf), q1 = code_of(a.y, zf, sf);
      const uint32_t q2 = code_of(bb.x, zf, sf), q3 = code_of(bb.y, zf, sf);
      *reinterpret_cast<uint32_t *>(&S.vc[t][4 * lane]) = q0 | (q1 << 8) | (q2 << 16) | (q3 << 24);
    }
  }
  __syncthreads();
  if (tid < kD) {
    uint16_t sb, zb;
    float sf, zf;
    scale_zero(fminf(S.kmin[0][tid], S.kmin[1][tid]), fmaxf(S.kmax[0][tid], S.kmax[1][tid]), sb,
               zb, sf, zf);
    S.ks[tid] = sb;
    S.kz[tid] = zb;
  }
  __syncthreads();

  // 4. key codes: thread = channel pair (2j, 2j+1) x a quarter of the tokens
  {
    const int j = tid & 63, tq = tid >> 6;
    const float s0 = __half2float(__ushort_as_half(S.ks[2 * j]));
    const float s1 = __half2float(__ushort_as_half(S.ks[2 * j + 1]));
    const float z0 = __half2float(__ushort_as_half(S.kz[2 * j]));
    const float z1 = __half2float(__ushort_as_half(S.kz[2 * j + 1]));
    for (int t = tq * 32; t < tq * 32 + 32; ++t) {
      const float2 x = __half22float2(*reinterpret_cast<const __half2 *>(&S.k[t][2 * j]));
      const uint32_t q0 = code_of(x.x, z0, s0), q1 = code_of(x.y, z1, s1);
      *reinterpret_cast<uint16_t *>(&S.kc[t][2 * j]) = (uint16_t)(q0 | (q1 << 8));
    }
  }
  __syncthreads();

  const size_t grp = bh * c.cap_groups + g;
  // 5. key planes, token-major: byte i of a token = channels 2i (low), 2i+1
  {
    const int t = tid >> 1, hb = tid & 1;
    uint8_t u[32], l[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const uint32_t c0 = S.kc[t][64 * hb + 2 * i], c1 = S.kc[t][64 * hb + 2 * i + 1];
      u[i] = (uint8_t)((c0 >> 4) | (c1 & 0xF0u));
      l[i] = (uint8_t)((c0 & 15u) | ((c1 & 15u) << 4));
    }
    uint4 *gu = reinterpret_cast<uint4 *>(c.k_upper + (grp * kG + t) * (kD / 2) + 32 * hb);
    uint4 *gl = reinterpret_cast<uint4 *>(c.k_lower + (grp * kG + t) * (kD / 2) + 32 * hb);
    gu[0] = *reinterpret_cast<uint4 *>(&u[0]);
    gu[1] = *reinterpret_cast<uint4 *>(&u[16]);
    gl[0] = *reinterpret_cast<uint4 *>(&l[0]);
    gl[1] = *reinterpret_cast<uint4 *>(&l[16]);
  }
  // 6. value planes: [quarter][channel][16 B], nibble p holds token vperm(p)
  for (int ri = tid; ri < 4 * kD; ri += 256) {
    const int u4 = ri >> 7, d = ri & (kD - 1);
    uint32_t wu[4] = {0, 0, 0, 0}, wl[4] = {0, 0, 0, 0};
#pragma unroll
    for (int p = 0; p < 32; ++p) {
      const uint32_t q = S.vc[32 * u4 + vperm(p)][d];
      wu[p >> 3] |= (q >> 4) << (4 * (p & 7));
      wl[p >> 3] |= (q & 15u) << (4 * (p & 7));
    }
    reinterpret_cast<uint4 *>(c.v_upper)[grp * 4 * kD + ri] = make_uint4(wu[0], wu[1], wu[2], wu[3]);
    reinterpret_cast<uint4 *>(c.v_lower)[grp * 4 * kD + ri] = make_uint4(wl[0], wl[1], wl[2], wl[3]);
  }
  // 7. metadata rows: key scale, key zero (per channel), value scale, zero
  if (tid < 128) {
    uint16_t *m = c.meta + grp * 4 * 128;
    m[QS_META_K_SCALE * 128 + tid] = S.ks[tid];
    m[QS_META_K_ZERO * 128 + tid] = S.kz[tid];
    m[QS_META_V_SCALE * 128 + tid] = S.vs[tid];
    m[QS_META_V_ZERO * 128 + tid] = S.vz[tid];
  }
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    const int ticket = atomicAdd(&st[QS_ST_TICKET], 1);
    if (ticket == c.H - 1) {  // every head has read the old counters
      st[QS_ST_N_GROUPS] = g + 1;
      st[QS_ST_HALF_BASE] = base ^ 1;
      st[QS_ST_FILL] -= kG;
      st[QS_ST_TICKET] = 0;
      __threadfence();
    }
  }
}

}  // namespace qs

using namespace qs;

extern "C" qs_status qs_quantize_flush(const qs_cache *c, const uint8_t *d_mask,
                                       qs_stream_t stream) {
  qs_status s = check_cache(c);
  if (s != QS_OK) return s;
  const int smem = (int)sizeof(FlushSmem);
  static int configured_mask = 0;  // one bit per device ordinal below 32
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return QS_ERR_CUDA;
  if (dev >= 32 || !(configured_mask & (1 << dev))) {
    if (cudaFuncSetAttribute(flush_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
        cudaSuccess)
      return QS_ERR_CUDA;
    if (dev < 32) __atomic_fetch_or(&configured_mask, 1 << dev, __ATOMIC_RELAXED);
  }
  flush_kernel<<<dim3(c->H, c->B), 256, smem, (cudaStream_t)stream>>>(*c, d_mask);
  return launch_status();
}
