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
#include "qs_common.cuh"

namespace {

// The scratch array.  Every GPU that loads libqs holds it until the process
// exits; every call shares it.
constexpr size_t kStaticWsBytes = size_t(QS_STATIC_WS_BYTES);
static __device__ __align__(256) unsigned char g_static_ws[kStaticWsBytes];

// Device address of g_static_ws per device ordinal.  In host code the name
// g_static_ws is only a host-side stand-in, so the real address is looked up
// once per device (with that device current) and cached here.
void *g_ws_addr[64];

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
  void *ws = __atomic_load_n(&g_ws_addr[dev], __ATOMIC_ACQUIRE);
  if (!ws) {
    if (cudaGetSymbolAddress(&ws, g_static_ws) != cudaSuccess || !ws) return QS_ERR_CUDA;
    __atomic_store_n(&g_ws_addr[dev], ws, __ATOMIC_RELEASE);
  }
  return qs_attn_decode(c, mode, q, n_q, softmax_scale, out, lse, ws, kStaticWsBytes, stream);
}
