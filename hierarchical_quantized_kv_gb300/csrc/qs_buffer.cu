// qs_buffer.cu -- the fp16 double buffer and the per-sequence counters:
// append, rollback, need_flush, error read-back, sizes.
//
// Source: "QuantSpec: Self-Speculative Decoding with Hierarchical Quantized
// KV Cache" (Pith review), "What carries the argument": a double
// full-precision buffer of two halves of G absorbs new tokens; rejected
// speculative tokens are dropped before quantization.  "QuantSpec Guide",
// "Zero-Overhead Rollback": a rollback never touches the quantized cache.
//
// Counters live on the device so that a speculative round needs no host
// synchronization.  Every head of a sequence reads the same counters; the
// last CTA of a sequence to finish (an arrival ticket, no spinning) writes
// the updated counters.
#include "qs_common.cuh"

namespace qs {

// One CTA per (head, sequence): copy n_new rows of K and V into the ring.
__global__ void __launch_bounds__(256) append_kernel(qs_cache c, const uint4 *__restrict__ k_new,
                                                     const uint4 *__restrict__ v_new, int n_new) {
  const int h = blockIdx.x, b = blockIdx.y;
  pdl_trigger();
  pdl_wait();
  int32_t *st = c.state + (size_t)b * QS_STATE_WORDS;
  __shared__ int s_fill, s_base;
  if (threadIdx.x == 0) {
    s_fill = st[QS_ST_FILL];
    s_base = st[QS_ST_HALF_BASE] & 1;
  }
  __syncthreads();
  const int fill = s_fill, base = s_base;
  if (fill < 0 || fill + n_new > kRing) {
    if (h == 0 && threadIdx.x == 0) atomicOr(&st[QS_ST_ERR], QS_DEV_OVERFLOW);
    return;
  }
  constexpr int kRowVec = kD * 2 / 16;  // uint4 per fp16 row
  const size_t bh = (size_t)b * c.H + h;
  uint4 *bk = reinterpret_cast<uint4 *>(c.buf_k) + bh * kRing * kRowVec;
  uint4 *bv = reinterpret_cast<uint4 *>(c.buf_v) + bh * kRing * kRowVec;
  const uint4 *sk = k_new + bh * n_new * kRowVec;
  const uint4 *sv = v_new + bh * n_new * kRowVec;
  for (int e = threadIdx.x; e < n_new * kRowVec; e += blockDim.x) {
    const int i = e / kRowVec, col = e % kRowVec;
    const int slot = (base * kG + fill + i) & (kRing - 1);
    bk[slot * kRowVec + col] = sk[e];
    bv[slot * kRowVec + col] = sv[e];
  }
  __syncthreads();
  // every head has read the old counters once the ticket reaches H - 1
  if (threadIdx.x == 0 && atom_add_acq_rel_gpu(&st[QS_ST_TICKET], 1) == c.H - 1) {
    st[QS_ST_FILL] = fill + n_new;
    st[QS_ST_PENDING] += n_new;
    st[QS_ST_TICKET] = 0;
  }
}

__global__ void rollback_kernel(qs_cache c, const int32_t *__restrict__ n_drop) {
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= c.B) return;
  int32_t *st = c.state + (size_t)b * QS_STATE_WORDS;
  const int r = n_drop[b];
  if (r < 0 || r > st[QS_ST_PENDING]) {
    st[QS_ST_ERR] |= QS_DEV_OVER_ROLLBACK;
    return;
  }
  st[QS_ST_FILL] -= r;
  st[QS_ST_PENDING] = 0;
}

__global__ void need_flush_kernel(qs_cache c, int n_next, uint8_t *__restrict__ mask) {
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= c.B) return;
  mask[b] = (c.state[(size_t)b * QS_STATE_WORDS + QS_ST_FILL] + n_next > kRing) ? 1 : 0;
}

}  // namespace qs

using namespace qs;

extern "C" {

const char *qs_status_string(qs_status s) {
  switch (s) {
    case QS_OK: return "ok";
    case QS_ERR_ARG: return "invalid argument";
    case QS_ERR_SHAPE: return "inconsistent sizes";
    case QS_ERR_ALIGN: return "device pointer not 16-byte aligned";
    case QS_ERR_CUDA: return "CUDA error";
    case QS_ERR_UNSUPPORTED: return "unsupported size (v1: D = G = 128, B <= 256)";
    case QS_ERR_WORKSPACE: return "workspace missing or too small";
    case QS_ERR_TOO_LARGE: return "problem exceeds the fixed scratch of qs_attn_decode_static_ws";
  }
  return "unknown status";
}

qs_status qs_cache_bytes(int32_t B, int32_t H, int32_t D, int32_t G, int32_t cap,
                         qs_cache_bytes_t *out) {
  if (!out || B <= 0 || H <= 0 || D <= 0 || G <= 0 || cap <= 0) return QS_ERR_ARG;
  if (D != kD || G != kG) return QS_ERR_UNSUPPORTED;
  const size_t bh = (size_t)B * H;
  const size_t plane = bh * cap * G * (D / 2);  // one nibble per element
  out->k_upper = out->k_lower = out->v_upper = out->v_lower = plane;
  out->meta = bh * cap * 4 * 128 * 2;
  out->buf_k = out->buf_v = bh * 2 * G * D * 2;
  out->state = (size_t)B * QS_STATE_WORDS * 4;
  out->arrive = bh * 4;
  return QS_OK;
}

qs_status qs_state_reset(const qs_cache *c, qs_stream_t stream) {
  qs_status s = check_cache(c);
  if (s != QS_OK) return s;
  cudaError_t e = cudaMemsetAsync(c->state, 0, (size_t)c->B * QS_STATE_WORDS * 4,
                                  (cudaStream_t)stream);
  if (e == cudaSuccess)
    e = cudaMemsetAsync(c->arrive, 0, (size_t)c->B * c->H * 4, (cudaStream_t)stream);
  return e == cudaSuccess ? QS_OK : QS_ERR_CUDA;
}

qs_status qs_buffer_append(const qs_cache *c, const uint16_t *k_new, const uint16_t *v_new,
                           int32_t n_new, qs_stream_t stream) {
  qs_status s = check_cache(c);
  if (s != QS_OK) return s;
  if (!k_new || !v_new || n_new < 1 || n_new > kRing) return QS_ERR_ARG;
  if (!aligned16(k_new) || !aligned16(v_new)) return QS_ERR_ALIGN;
  return launch_pdl(append_kernel, dim3(c->H, c->B), dim3(256), 0, (cudaStream_t)stream, *c,
                    reinterpret_cast<const uint4 *>(k_new), reinterpret_cast<const uint4 *>(v_new),
                    (int)n_new);
}

qs_status qs_buffer_rollback(const qs_cache *c, const int32_t *d_n_drop, qs_stream_t stream) {
  qs_status s = check_cache(c);
  if (s != QS_OK) return s;
  if (!d_n_drop) return QS_ERR_ARG;
  return launch_pdl(rollback_kernel, dim3((c->B + 127) / 128), dim3(128), 0, (cudaStream_t)stream,
                    *c, d_n_drop);
}

qs_status qs_need_flush(const qs_cache *c, int32_t n_next, uint8_t *d_mask, qs_stream_t stream) {
  qs_status s = check_cache(c);
  if (s != QS_OK) return s;
  if (!d_mask || n_next < 0) return QS_ERR_ARG;
  return launch_pdl(need_flush_kernel, dim3((c->B + 127) / 128), dim3(128), 0,
                    (cudaStream_t)stream, *c, (int)n_next, d_mask);
}

qs_status qs_get_errors(const qs_cache *c, int32_t *h_err, qs_stream_t stream) {
  qs_status s = check_cache(c);
  if (s != QS_OK) return s;
  if (!h_err) return QS_ERR_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  const size_t pitch = QS_STATE_WORDS * sizeof(int32_t);
  cudaError_t e = cudaMemcpy2DAsync(h_err, sizeof(int32_t), c->state + QS_ST_ERR, pitch,
                                    sizeof(int32_t), c->B, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess)
    e = cudaMemset2DAsync(c->state + QS_ST_ERR, pitch, 0, sizeof(int32_t), c->B, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  return e == cudaSuccess ? QS_OK : QS_ERR_CUDA;
}

}  // extern "C"
