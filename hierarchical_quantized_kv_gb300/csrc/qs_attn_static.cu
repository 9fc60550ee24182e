// qs_attn_static.cu -- decode attention for callers that cannot allocate
// device memory.
//
// qs_attn_decode needs a scratch workspace for its split partials, which the
// caller normally allocates.  Some callers cannot: code running under an
// allocator that must not grow (a serving process whose device memory is
// carved up before it starts), callers in another language runtime without a
// CUDA allocator of their own, or a plug-in that is handed only the input and
// output buffers.  qs_attn_decode_static_ws gives them the same computation
// with the scratch placed in a fixed array that lives inside this library.
#include <mutex>

#include "qs_common.cuh"

namespace {

// The scratch array.  Every GPU that loads libqs holds it until the process
// exits; every call shares it.
constexpr size_t kStaticWsBytes = size_t(QS_STATIC_WS_BYTES);
static __device__ __align__(256) unsigned char g_static_ws[kStaticWsBytes];

// In host code the name g_static_ws is only a host-side stand-in, so its
// device address is looked up once per device, with that device current, and
// cached together with the identity of the CUDA context it belongs to: a
// different context on the same device (after cudaDeviceReset, or a context a
// driver-API caller made current) has its own copy of the array, so a change
// of context looks the address up again instead of using a stale one.
struct WsAddr {
  unsigned long long ctx_id;
  void *addr;
};
WsAddr g_ws_addr[64];
std::mutex g_ws_mu;

// The current context's unique id through the driver entry points (the
// runtime has no call for it; the library does not link libcuda itself).
using CtxGetCurrentFn = int (*)(void **);
using CtxGetIdFn = int (*)(void *, unsigned long long *);

bool current_context_id(unsigned long long *id) {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_ws_mu);
    if (!get_current || !get_id) {
      cudaDriverEntryPointQueryResult q1, q2;
      void *f1 = nullptr, *f2 = nullptr;
      if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 12000, cudaEnableDefault,
                                           &q1) != cudaSuccess ||
          q1 != cudaDriverEntryPointSuccess ||
          cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault, &q2) !=
              cudaSuccess ||
          q2 != cudaDriverEntryPointSuccess || !f1 || !f2)
        return false;
      get_current = reinterpret_cast<CtxGetCurrentFn>(f1);
      get_id = reinterpret_cast<CtxGetIdFn>(f2);
    }
  }
  void *ctx = nullptr;
  if (get_current(&ctx) != 0 || !ctx) return false;
  return get_id(ctx, id) == 0;
}

}  // namespace

using namespace qs;

extern "C" qs_status qs_attn_decode_static_ws(const qs_cache *c, qs_mode mode, const uint16_t *q,
                                              int32_t n_q, float softmax_scale, uint16_t *out,
                                              float *lse, qs_stream_t stream) {
  qs_status s = check_cache(c);
  if (s != QS_OK) return s;
  if (!q || !out || n_q < 1 || n_q > kMaxQ) return QS_ERR_ARG;
  size_t need = 0;
  if ((s = qs_attn_workspace_size(c, n_q, &need)) != QS_OK) return s;
  if (need > kStaticWsBytes) return QS_ERR_TOO_LARGE;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return QS_ERR_CUDA;
  if (dev < 0 || dev >= 64) return QS_ERR_UNSUPPORTED;
  unsigned long long ctx = 0;
  void *ws = nullptr;
  if (current_context_id(&ctx)) {
    std::lock_guard<std::mutex> lock(g_ws_mu);
    if (g_ws_addr[dev].addr && g_ws_addr[dev].ctx_id == ctx) ws = g_ws_addr[dev].addr;
  }
  if (!ws) {
    // set-up on this device and context (the lookup makes the device's
    // primary context current when no context is)
    if (cudaGetSymbolAddress(&ws, g_static_ws) != cudaSuccess || !ws) return QS_ERR_CUDA;
    if (!current_context_id(&ctx)) return QS_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_ws_mu);
    g_ws_addr[dev] = WsAddr{ctx, ws};
  }
  return qs_attn_decode(c, mode, q, n_q, softmax_scale, out, lse, ws, kStaticWsBytes, stream);
}
