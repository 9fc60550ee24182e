"""ctypes binding of libqs (include/qs.h): argument marshalling only.

Every function here has the name of the C entry point it calls and does no
arithmetic of its own: each step of the hot path runs in the CUDA library.
PyTorch supplies device memory and the current stream.  If ``libqs.so`` has
not been built this module raises on first use -- there is no fallback.
"""
import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libqs.so")

QS_DRAFT_UPPER4, QS_VERIFY_INT8 = 0, 1
(QS_OK, QS_ERR_ARG, QS_ERR_SHAPE, QS_ERR_ALIGN, QS_ERR_CUDA, QS_ERR_UNSUPPORTED, QS_ERR_WORKSPACE,
 QS_ERR_TOO_LARGE) = range(8)
QS_STATIC_WS_BYTES = 8 << 20
DEV_OVERFLOW, DEV_OVER_ROLLBACK, DEV_FLUSH_UNCOMMITTED, DEV_CAPACITY, DEV_NQ_GT_FILL, DEV_TIMEOUT = (
    1, 2, 4, 8, 16, 32)
DEV_PREFILL = 64
ST_N_GROUPS, ST_FILL, ST_PENDING, ST_HALF_BASE, ST_ERR, ST_TICKET = range(6)
STATE_WORDS = 8
META_K_SCALE, META_K_ZERO, META_V_SCALE, META_V_ZERO = range(4)

_P = ctypes.c_void_p
_I32 = ctypes.c_int32


class QsCacheStruct(ctypes.Structure):
    _fields_ = [("B", _I32), ("H", _I32), ("D", _I32), ("G", _I32), ("cap_groups", _I32),
                ("upper_bits", _I32), ("k_upper", _P), ("k_lower", _P), ("v_upper", _P), ("v_lower", _P),
                ("meta", _P), ("buf_k", _P), ("buf_v", _P), ("state", _P), ("arrive", _P)]


class QsCacheBytes(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in
                ("k_upper", "k_lower", "v_upper", "v_lower", "meta", "buf_k", "buf_v", "state",
                 "arrive")]


class QsError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__("%s failed: %s (%d)" % (fn, status_string(status), status))


_lib = None

# exported entry points and their argument types
_SIGS = {
    "qs_cache_bytes": [_I32, _I32, _I32, _I32, _I32, ctypes.POINTER(QsCacheBytes)],
    "qs_state_reset": [ctypes.POINTER(QsCacheStruct), _P],
    "qs_buffer_append": [ctypes.POINTER(QsCacheStruct), _P, _P, _I32, _P],
    "qs_buffer_rollback": [ctypes.POINTER(QsCacheStruct), _P, _P],
    "qs_need_flush": [ctypes.POINTER(QsCacheStruct), _I32, _P, _P],
    "qs_quantize_flush": [ctypes.POINTER(QsCacheStruct), _P, _P],
    "qs_quantize_flush_due": [ctypes.POINTER(QsCacheStruct), _I32, _P],
    "qs_attn_workspace_size": [ctypes.POINTER(QsCacheStruct), _I32, ctypes.POINTER(ctypes.c_size_t)],
    "qs_attn_decode": [ctypes.POINTER(QsCacheStruct), ctypes.c_int, _P, _I32, ctypes.c_float, _P,
                       _P, _P, ctypes.c_size_t, _P],
    "qs_get_errors": [ctypes.POINTER(QsCacheStruct), _P, _P],
    "qs_attn_workspace_size_gqa": [ctypes.POINTER(QsCacheStruct), _I32, _I32,
                                   ctypes.POINTER(ctypes.c_size_t)],
    "qs_attn_decode_gqa": [ctypes.POINTER(QsCacheStruct), ctypes.c_int, _P, _I32, _I32, ctypes.c_float,
                           _P, _P, _P, ctypes.c_size_t, _P],
    "qs_prefill": [ctypes.POINTER(QsCacheStruct), _P, _P, _I32, _P, _P],
    "qs_spec_accept": [_P, _P, _P, _P, _P, _I32, _I32, _I32, _P, _P, _P, _P],
    "qs_attn_decode_static_ws": [ctypes.POINTER(QsCacheStruct), ctypes.c_int, _P, _I32,
                                 ctypes.c_float, _P, _P, _P],
    "qs_attn_decode_append": [ctypes.POINTER(QsCacheStruct), ctypes.c_int, _P, _P, _I32, _P, _I32,
                              _I32, ctypes.c_float, _P, _P, _P, ctypes.c_size_t, _P],
}


def lib():
    """Load libqs.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libqs.so is not built (run __graft_entry__.build()); "
                               "there is no CPU fallback")
        L = ctypes.CDLL(LIB_PATH)
        for name, args in _SIGS.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = ctypes.c_int
        L.qs_status_string.argtypes = [ctypes.c_int]
        L.qs_status_string.restype = ctypes.c_char_p
        _lib = L
    return _lib


def status_string(s):
    return lib().qs_status_string(int(s)).decode()


def _check(fn, status):
    if status != QS_OK:
        raise QsError(fn, status)


_current_raw_stream = None


def _current_stream_handle():
    """cudaStream_t of torch's current stream on the current device.  Through
    torch._C._cuda_getCurrentRawStream (the lookup torch's own generated code
    makes: about 0.3 us a call, against 3 us for torch.cuda.current_stream()
    on the Grace host) where this torch has it, else the public call."""
    global _current_raw_stream
    if _current_raw_stream is None:
        import torch
        raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
        dev = getattr(torch._C, "_cuda_getDevice", None)
        if raw is not None and dev is not None:
            torch.cuda.init()
            _current_raw_stream = lambda: raw(dev())
        else:
            _current_raw_stream = lambda: torch.cuda.current_stream().cuda_stream
    return _current_raw_stream()


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(_current_stream_handle())
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


# -------------------------------------------------------------------- cache

def qs_cache_bytes(B, H, cap_groups, D=128, G=128):
    out = QsCacheBytes()
    _check("qs_cache_bytes", lib().qs_cache_bytes(B, H, D, G, cap_groups, ctypes.byref(out)))
    return {n: getattr(out, n) for n, _ in QsCacheBytes._fields_}


class Cache:
    """A hierarchical quantized KV cache in torch-owned device memory, laid
    out as include/qs.h describes (shapes below are the C layouts)."""

    def __init__(self, B, H, cap_groups, device="cuda", D=128, G=128, upper_bits=4):
        """upper_bits: the top bits of each 8-bit code the draft reads (4, or
        2 for the two-bit draft layout of include/qs.h)."""
        import torch
        self.B, self.H, self.D, self.G, self.cap = B, H, D, G, cap_groups
        self.upper_bits = upper_bits
        qs_cache_bytes(B, H, cap_groups, D, G)  # validates the sizes
        u8 = dict(dtype=torch.uint8, device=device)
        f16 = dict(dtype=torch.float16, device=device)
        self.k_upper = torch.zeros((B, H, cap_groups, G, D // 2), **u8)
        self.k_lower = torch.zeros((B, H, cap_groups, G, D // 2), **u8)
        self.v_upper = torch.zeros((B, H, cap_groups, G // 32, D, 16), **u8)
        self.v_lower = torch.zeros((B, H, cap_groups, G // 32, D, 16), **u8)
        self.meta = torch.zeros((B, H, cap_groups, 4, 128), **f16)
        self.buf_k = torch.zeros((B, H, 2 * G, D), **f16)
        self.buf_v = torch.zeros((B, H, 2 * G, D), **f16)
        self.state = torch.zeros((B, STATE_WORDS), dtype=torch.int32, device=device)
        self.arrive = torch.zeros((B, H), dtype=torch.int32, device=device)
        self.struct = QsCacheStruct(B, H, D, G, cap_groups, upper_bits,
                                    self.k_upper.data_ptr(), self.k_lower.data_ptr(),
                                    self.v_upper.data_ptr(), self.v_lower.data_ptr(),
                                    self.meta.data_ptr(), self.buf_k.data_ptr(),
                                    self.buf_v.data_ptr(), self.state.data_ptr(),
                                    self.arrive.data_ptr())
        self._ref = ctypes.byref(self.struct)

    def nbytes(self):
        return sum(t.numel() * t.element_size() for t in
                   (self.k_upper, self.k_lower, self.v_upper, self.v_lower, self.meta,
                    self.buf_k, self.buf_v, self.state, self.arrive))


def qs_state_reset(cache, stream=None):
    _check("qs_state_reset", lib().qs_state_reset(cache._ref, _stream(stream)))


def qs_buffer_append(cache, k_new, v_new, stream=None):
    """k_new, v_new: fp16 [B, H, n_new, D] contiguous device tensors."""
    assert k_new.is_contiguous() and v_new.is_contiguous() and k_new.shape == v_new.shape
    n_new = k_new.shape[2]
    _check("qs_buffer_append", lib().qs_buffer_append(cache._ref, _ptr(k_new), _ptr(v_new),
                                                      n_new, _stream(stream)))


def qs_buffer_rollback(cache, n_drop, stream=None):
    """n_drop: int32 [B] device tensor."""
    _check("qs_buffer_rollback", lib().qs_buffer_rollback(cache._ref, _ptr(n_drop), _stream(stream)))


def qs_need_flush(cache, n_next, mask, stream=None):
    """mask: uint8 [B] device tensor (written)."""
    _check("qs_need_flush", lib().qs_need_flush(cache._ref, int(n_next), _ptr(mask), _stream(stream)))


def qs_quantize_flush(cache, mask=None, stream=None):
    """mask: uint8 [B] device tensor or None (every sequence)."""
    _check("qs_quantize_flush", lib().qs_quantize_flush(cache._ref, _ptr(mask), _stream(stream)))


def qs_quantize_flush_due(cache, n_next, stream=None):
    """Flush every sequence whose buffer cannot take n_next more tokens."""
    _check("qs_quantize_flush_due", lib().qs_quantize_flush_due(cache._ref, int(n_next),
                                                                _stream(stream)))


def qs_prefill(cache, k, v, lens, stream=None):
    """k, v: fp16 [B, H, T, D] contiguous device tensors; lens: int32 [B]
    device tensor of prompt lengths."""
    assert k.is_contiguous() and v.is_contiguous() and k.shape == v.shape
    _check("qs_prefill", lib().qs_prefill(cache._ref, _ptr(k), _ptr(v), int(k.shape[2]), _ptr(lens),
                                          _stream(stream)))


def qs_spec_accept(p, q, draft, u, e, n_accept, token, n_drop, stream=None):
    """p [B, g+1, V], q [B, g, V], u [B, g], e [B, V]: float32 device tensors;
    draft [B, g] int32; outputs n_accept, token, n_drop: int32 [B] tensors."""
    B, g1, V = p.shape
    for t in (p, q, draft, u, e):
        assert t.is_contiguous()
    _check("qs_spec_accept", lib().qs_spec_accept(_ptr(p), _ptr(q), _ptr(draft), _ptr(u), _ptr(e), B,
                                                  g1 - 1, V, _ptr(n_accept), _ptr(token),
                                                  _ptr(n_drop), _stream(stream)))


def qs_attn_workspace_size(cache, n_q):
    n = ctypes.c_size_t()
    _check("qs_attn_workspace_size", lib().qs_attn_workspace_size(cache._ref, int(n_q), ctypes.byref(n)))
    return n.value


def qs_attn_decode(cache, mode, q, softmax_scale, out, lse=None, workspace=None, stream=None):
    """q, out: fp16 [B, H, n_q, D]; lse: float32 [B, H, n_q] or None;
    workspace: a uint8 device tensor of at least qs_attn_workspace_size bytes."""
    n_q = q.shape[2]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("qs_attn_decode", lib().qs_attn_decode(
        cache._ref, int(mode), _ptr(q), n_q, float(softmax_scale), _ptr(out), _ptr(lse),
        _ptr(workspace), ws_bytes, _stream(stream)))


def qs_attn_workspace_size_gqa(cache, n_q, group):
    n = ctypes.c_size_t()
    _check("qs_attn_workspace_size_gqa", lib().qs_attn_workspace_size_gqa(
        cache._ref, int(n_q), int(group), ctypes.byref(n)))
    return n.value


def qs_attn_decode_gqa(cache, mode, q, group, softmax_scale, out, lse=None, workspace=None,
                       stream=None):
    """q, out: fp16 [B, H*group, n_q, D]; lse: float32 [B, H*group, n_q] or None."""
    n_q = q.shape[2]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("qs_attn_decode_gqa", lib().qs_attn_decode_gqa(
        cache._ref, int(mode), _ptr(q), n_q, int(group), float(softmax_scale), _ptr(out), _ptr(lse),
        _ptr(workspace), ws_bytes, _stream(stream)))


def qs_attn_decode_static_ws(cache, mode, q, softmax_scale, out, lse=None, stream=None):
    """qs_attn_decode with its scratch in the library's fixed device array
    (for callers that cannot allocate device memory); q, out, lse as for
    qs_attn_decode.  Returns the status instead of raising on
    QS_ERR_TOO_LARGE, so a caller can fall back to the allocating call."""
    n_q = q.shape[2]
    status = lib().qs_attn_decode_static_ws(cache._ref, int(mode), _ptr(q), n_q,
                                            float(softmax_scale), _ptr(out), _ptr(lse),
                                            _stream(stream))
    if status != QS_ERR_TOO_LARGE:
        _check("qs_attn_decode_static_ws", status)
    return status


def qs_attn_decode_append(cache, mode, k_new, v_new, q, softmax_scale, out, lse=None,
                          workspace=None, group=1, stream=None):
    """qs_buffer_append(k_new, v_new) then qs_attn_decode(_gqa), one launch.
    k_new, v_new: fp16 [B, H, n_new, D]; q, out: fp16 [B, H*group, n_q, D]."""
    assert k_new.is_contiguous() and v_new.is_contiguous() and k_new.shape == v_new.shape
    n_q = q.shape[2]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("qs_attn_decode_append", lib().qs_attn_decode_append(
        cache._ref, int(mode), _ptr(k_new), _ptr(v_new), k_new.shape[2], _ptr(q), n_q, int(group),
        float(softmax_scale), _ptr(out), _ptr(lse), _ptr(workspace), ws_bytes, _stream(stream)))


def qs_get_errors(cache, stream=None):
    """Per-sequence error words (numpy int32 [B]); clears them on the device."""
    h = np.zeros(cache.B, np.int32)
    _check("qs_get_errors", lib().qs_get_errors(cache._ref, h.ctypes.data_as(ctypes.c_void_p),
                                                _stream(stream)))
    return h
