// qs_common.cuh -- shared device helpers and host validation for libqs.
// Inline PTX wrappers for sm_103a: mbarrier, bulk async copies (TMA engine),
// warp-level tensor-core MMA, ldmatrix / movmatrix; plus argument checks.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "../../include/qs.h"

namespace qs {

constexpr int kD = 128;         // head dimension (v1)
constexpr int kG = 128;         // group size (v1)
constexpr int kRing = 2 * kG;   // double buffer slots
constexpr int kMaxB = 256;      // sequences per call (work partition tables)
constexpr int kMaxQ = 8;        // queries per call (one n8 MMA tile)

// ------------------------------------------------------------------ host

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline qs_status check_cache(const qs_cache *c) {
  if (!c || !c->state || !c->arrive || !c->buf_k || !c->buf_v) return QS_ERR_ARG;
  if (c->B <= 0 || c->H <= 0 || c->cap_groups <= 0) return QS_ERR_SHAPE;
  if (c->D != kD || c->G != kG) return QS_ERR_UNSUPPORTED;
  if (c->B > kMaxB) return QS_ERR_UNSUPPORTED;
  if (c->upper_bits != 4 && c->upper_bits != 2) return QS_ERR_ARG;
  if (!c->k_upper || !c->k_lower || !c->v_upper || !c->v_lower || !c->meta) return QS_ERR_ARG;
  const void *ps[] = {c->k_upper, c->k_lower, c->v_upper, c->v_lower,
                      c->meta,    c->buf_k,   c->buf_v,   c->state, c->arrive};
  for (const void *p : ps)
    if (!aligned16(p)) return QS_ERR_ALIGN;
  return QS_OK;
}

inline qs_status launch_status() {
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? QS_OK : QS_ERR_CUDA;
}

// Launch with programmatic stream serialization: the kernel may be scheduled
// while its predecessor in the stream is still running; it calls pdl_wait()
// before touching memory the predecessor writes, which restores stream order.
template <typename... KArgs, typename... Args>
inline qs_status launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                            cudaStream_t stream, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
  return e == cudaSuccess ? QS_OK : QS_ERR_CUDA;
}

// ---------------------------------------------------------------- device

// Programmatic dependent launch: let the next kernel in the stream start its
// launch now / wait until the previous kernel has completed and its writes
// are visible (returns at once when there is no programmatic predecessor).
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---- checked build (-DQS_CHECKED=1): the kernels check the bounds of their
// shared-memory and global indexing on the device.  A failing access is
// skipped (a load reads zero) and counted with a tag naming it, never
// trapped; the checked library exports qs_checked_failures to read the
// counts.  The ordinary build compiles every check away.
#ifndef QS_CHECKED
#define QS_CHECKED 0
#endif
#if QS_CHECKED
static __device__ unsigned long long g_check_fail[2];  // count, first failing tag (per file)
__device__ __forceinline__ bool chk(bool ok, uint32_t tag) {
  if (!ok && atomicAdd(&g_check_fail[0], 1ull) == 0ull) g_check_fail[1] = tag;
  return ok;
}
// [a, a + n) inside this CTA's dynamic shared memory (shared-window address)
__device__ __forceinline__ bool smem_in(uint32_t a, uint32_t n) {
  extern __shared__ __align__(128) uint8_t qs_dyn_smem[];
  uint32_t dyn;
  asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(dyn));
  const uint32_t lo = static_cast<uint32_t>(__cvta_generic_to_shared(qs_dyn_smem));
  return a >= lo && a + n <= lo + dyn;
}
#else
__device__ __forceinline__ constexpr bool chk(bool, uint32_t) { return true; }
__device__ __forceinline__ constexpr bool smem_in(uint32_t, uint32_t) { return true; }
#endif
// [i, i + n) inside an array of len elements
__device__ __forceinline__ bool in_range(size_t i, size_t n, size_t len) {
  return i <= len && n <= len - i;
}

// Upper bound on any single pipeline wait; a healthy call takes well under a
// millisecond, so running out means a broken pipeline: record and bail out.
constexpr uint64_t kWaitLimitNs = 4000000000ull;

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete; false once limit_ns
// have passed (the caller records QS_DEV_TIMEOUT and stops).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                          uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
}

// Device-scope atomic add with acquire and release semantics: an arrival on
// a counter that publishes what the arriving thread wrote or observed before
// it (a barrier before it covers the whole CTA's writes), and after which the
// writes of the threads that arrived earlier are visible (to the whole CTA
// after a barrier).
__device__ __forceinline__ int atom_add_acq_rel_gpu(int *p, int v) {
  int old;
  asm volatile("atom.add.acq_rel.gpu.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// Bulk async copy global -> shared (TMA engine, no tensor map), completion
// counted in bytes on an mbarrier.  Addresses 16-byte aligned, size % 16 == 0.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// L2 policy for data read once per call (the KV stream): evict first, so the
// stream does not push out lines that are reused (instructions, partials,
// counters).
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// bulk_g2s with an L2 cache policy.
__device__ __forceinline__ void bulk_g2s_hint(uint32_t dst, const void *src, uint32_t bytes,
                                              uint32_t bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], "
      "%2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(pol)
      : "memory");
}

// D += A * B, m16n8k16, fp16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
  return d;
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t &r0, uint32_t &r1,
                                            uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr)
               : "memory");
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t &r0, uint32_t &r1,
                                                  uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr)
               : "memory");
}

// Bit select (a & m) | (b & ~m) in one LOP3.
__device__ __forceinline__ uint32_t bitsel(uint32_t a, uint32_t b, uint32_t m) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xE4;" : "=r"(d) : "r"(a), "r"(b), "r"(m));
  return d;
}

__device__ __forceinline__ void prefetch_l1(const void *p) {
  asm volatile("prefetch.global.L1 [%0];" ::"l"(p));
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

__device__ __forceinline__ uint32_t h2_as_u32(__half2 h) { return *reinterpret_cast<uint32_t *>(&h); }
__device__ __forceinline__ __half2 u32_as_h2(uint32_t u) { return *reinterpret_cast<__half2 *>(&u); }

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
  return h2_as_u32(__hmul2(u32_as_h2(a), u32_as_h2(b)));
}
// Exact residual of an fp16 product, rounded once: a * b - c (fused).
__device__ __forceinline__ uint32_t hfma2_neg_u32(uint32_t a, uint32_t b, uint32_t c) {
  return h2_as_u32(__hfma2(u32_as_h2(a), u32_as_h2(b), __hneg2(u32_as_h2(c))));
}
__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  return h2_as_u32(__floats2half2_rn(lo, hi));
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

}  // namespace qs
