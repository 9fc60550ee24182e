// qs_spec.cu -- speculative-sampling acceptance on the device: which draft
// tokens the target accepts, the token emitted after them, and the rollback
// count, without a host round trip.
//
// Source: "QuantSpec: Self-Speculative Decoding with Hierarchical Quantized
// KV Cache" (Pith review), referee report on Algorithm 1: VERIFY / CORRECT as
// rejection sampling, accepting draft token g_i with probability
// min(1, p_i(g_i) / q_i(g_i)) and, on the first rejection, drawing from the
// residual (p_i - q_i)_+; "QuantSpec Guide", "The Self-Speculative
// Verification Loop" (one acceptance test per draft token, stop at the first
// rejection).
//
// Every decision is made in IEEE fp32 with explicit rounding (__fmul_rn,
// __fsub_rn, __fdiv_rn), and the draw is an exponential race (the smallest
// e_x / w_x over w_x > 0, ties to the smaller index) over Exp(1) variates the
// caller supplies, so the result does not depend on summation order.
#include <cooperative_groups.h>

#include "qs_common.cuh"

namespace cg = cooperative_groups;

namespace qs {
namespace {

constexpr int kSpecThreads = 512;
constexpr int kSpecCluster = 8;  // CTAs per sequence: a cluster splits the vocabulary

// (k1, x1) comes before (k2, x2): smaller key, ties to the smaller index;
// index -1 means "nothing yet".
__device__ __forceinline__ bool before(float k1, int x1, float k2, int x2) {
  if (x1 < 0) return false;
  if (x2 < 0) return true;
  return k1 < k2 || (k1 == k2 && x1 < x2);
}

// This CTA's best (key, index) over x in [x0, x1) of the weights p (minus q
// when q is given, clamped at 0): block reduction into s_key[0], s_idx[0].
__device__ void race_block(const float *__restrict__ wp, const float *__restrict__ wq,
                           const float *__restrict__ eb, int x0, int x1, float *s_key,
                           int *s_idx) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  float key = 0.f;
  int idx = -1;
  for (int x = x0 + tid; x < x1; x += kSpecThreads) {
    float w = wp[x];
    if (wq) {
      const float d = __fsub_rn(w, wq[x]);
      w = d > 0.f ? d : 0.f;
    }
    if (w > 0.f) {
      const float k = __fdiv_rn(eb[x], w);
      if (before(k, x, key, idx)) {
        key = k;
        idx = x;
      }
    }
  }
  for (int o = 16; o > 0; o >>= 1) {
    const float k2 = __shfl_xor_sync(0xffffffffu, key, o);
    const int i2 = __shfl_xor_sync(0xffffffffu, idx, o);
    if (before(k2, i2, key, idx)) {
      key = k2;
      idx = i2;
    }
  }
  __syncthreads();  // s_key / s_idx may still be read from an earlier pass
  if (lane == 0) {
    s_key[warp] = key;
    s_idx[warp] = idx;
  }
  __syncthreads();
  if (tid == 0) {
    for (int w2 = 1; w2 < kSpecThreads / 32; ++w2)
      if (before(s_key[w2], s_idx[w2], key, idx)) {
        key = s_key[w2];
        idx = s_idx[w2];
      }
    s_key[0] = key;
    s_idx[0] = idx;
  }
}

// A cluster of kSpecCluster CTAs per sequence (grid kSpecCluster x B): each
// CTA decides the accepted count (the same few reads, the same result), races
// over its slice of the vocabulary, and the slices' winners meet through
// distributed shared memory.
__global__ void __cluster_dims__(kSpecCluster, 1, 1) __launch_bounds__(kSpecThreads)
    spec_accept_kernel(const float *__restrict__ p, const float *__restrict__ q,
                       const int32_t *__restrict__ draft, const float *__restrict__ u,
                       const float *__restrict__ e, int gamma, int V, int32_t *n_accept,
                       int32_t *token, int32_t *n_drop) {
  __shared__ int s_a;
  __shared__ float s_key[kSpecThreads / 32];
  __shared__ int s_idx[kSpecThreads / 32];
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank(), b = blockIdx.y, tid = threadIdx.x;
  pdl_trigger();
  pdl_wait();
  const float *pb = p + (size_t)b * (gamma + 1) * V;
  const float *qb = q + (size_t)b * gamma * V;
  if (tid < 32) {
    // The accepted count: draft token i is tested by lane i % 32 (its token,
    // p, q and u loaded by all lanes at once, not one after another); the
    // first rejection, the lowest set bit of the vote, ends the run.
    int a = gamma;
    for (int base = 0; base < gamma; base += 32) {
      const int i = base + tid;
      bool reject = false;
      if (i < gamma) {
        const int x = draft[(size_t)b * gamma + i];
        reject = x < 0 || x >= V;  // not a token: rejected
        if (!reject) {
          const float pa = pb[(size_t)i * V + x], qa = qb[(size_t)i * V + x];
          reject = !(__fmul_rn(u[(size_t)b * gamma + i], qa) < pa);
        }
      }
      const unsigned rej = __ballot_sync(0xffffffffu, reject);
      if (rej) {
        a = base + __ffs(rej) - 1;
        break;
      }
    }
    if (tid == 0) s_a = a;
  }
  __syncthreads();
  const int a = s_a;
  const float *eb = e + (size_t)b * V;
  const int chunk = (V + kSpecCluster - 1) / kSpecCluster;
  const int x0 = min(V, rank * chunk), x1 = min(V, x0 + chunk);
  // pass 0: the residual (p_a - q_a)_+ after a rejection, else p_gamma;
  // pass 1 (a residual that is zero everywhere): p_a
  int idx = -1;
  for (int pass = 0; pass < 2; ++pass) {
    const float *wq = (a < gamma && pass == 0) ? qb + (size_t)a * V : nullptr;
    race_block(pb + (size_t)a * V, wq, eb, x0, x1, s_key, s_idx);
    cluster.sync();  // every slice's winner is in its CTA's shared memory
    float key = 0.f;
    idx = -1;
    for (int r = 0; r < kSpecCluster; ++r) {  // in rank order: ties to the smaller index
      const float k2 = *cluster.map_shared_rank(&s_key[0], r);
      const int i2 = *cluster.map_shared_rank(&s_idx[0], r);
      if (before(k2, i2, key, idx)) {
        key = k2;
        idx = i2;
      }
    }
    cluster.sync();  // no CTA overwrites its winner while another still reads it
    if (idx >= 0 || a == gamma) break;
  }
  if (rank == 0 && tid == 0) {
    n_accept[b] = a;
    token[b] = idx;
    n_drop[b] = gamma - a;
  }
}

}  // namespace
}  // namespace qs

using namespace qs;

extern "C" qs_status qs_spec_accept(const float *p, const float *q, const int32_t *draft,
                                    const float *u, const float *e, int32_t B, int32_t gamma,
                                    int32_t V, int32_t *n_accept, int32_t *token, int32_t *n_drop,
                                    qs_stream_t stream) {
  if (!p || !q || !draft || !u || !e || !n_accept || !token || !n_drop) return QS_ERR_ARG;
  if (B < 1 || gamma < 1 || gamma > 64 || V < 1) return QS_ERR_ARG;
  const void *ptrs[] = {p, q, draft, u, e, n_accept, token, n_drop};
  for (const void *x : ptrs)
    if (reinterpret_cast<uintptr_t>(x) % 4) return QS_ERR_ALIGN;
  if (B > 65535) return QS_ERR_ARG;
  return launch_pdl(spec_accept_kernel, dim3(kSpecCluster, B), dim3(kSpecThreads), 0,
                    (cudaStream_t)stream, p, q, draft, u, e, (int)gamma, (int)V, n_accept, token,
                    n_drop);
}
