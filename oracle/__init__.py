"""CPU oracle for the QuantSpec hierarchical quantized KV cache hot path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package; the product path
(the CUDA library and its binding) never does.

The arithmetic lives in ``qs_oracle.c`` (plain C, fp64 attention, exact fp32
quantization under convention QS-RN-v1); this module is argument marshalling
over ctypes plus numpy storage for the logical cache state:

* key/value codes as full 8-bit values [B, H, cap, G tokens, D channels]
  (upper level = code >> 4, lower level = code & 15);
* key scale/zero per channel [B, H, cap, D], value scale/zero per token
  [B, H, cap, G], all fp16;
* the fp16 double buffer [B, H, 2G, D] and per-sequence counters [B, 8]
  (n_groups, fill, pending, half_base, err, 3 reserved).

Parity pins: see the ``-m "not gpu"`` tests (nibble repack, dequantization
bounds, closed-form groups, history independence, empty-cache attention,
draft == verify when every lower level is 8, causal mask via rollback).
"""
import ctypes
import os

import numpy as np

from . import build as _build

N_GROUPS, FILL, PENDING, HALF_BASE, ERR = 0, 1, 2, 3, 4
STATE_WORDS = 8
DEV_OVERFLOW, DEV_OVER_ROLLBACK, DEV_FLUSH_UNCOMMITTED, DEV_CAPACITY, DEV_NQ_GT_FILL = 1, 2, 4, 8, 16
DEV_PREFILL = 64

_lib = None


class _Cache(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("H", ctypes.c_int), ("D", ctypes.c_int),
                ("G", ctypes.c_int), ("cap", ctypes.c_int),
                ("kq", ctypes.c_void_p), ("vq", ctypes.c_void_p),
                ("ks", ctypes.c_void_p), ("kz", ctypes.c_void_p),
                ("vs", ctypes.c_void_p), ("vz", ctypes.c_void_p),
                ("bk", ctypes.c_void_p), ("bv", ctypes.c_void_p),
                ("state", ctypes.c_void_p)]


def lib():
    """Load (building first if needed) the oracle shared library."""
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        P, I, D_, L_ = ctypes.c_void_p, ctypes.c_int, ctypes.c_double, ctypes.c_long
        L.qso_half_to_double.restype = D_
        L.qso_half_to_double.argtypes = [ctypes.c_uint16]
        L.qso_float_to_half_rn.restype = ctypes.c_uint16
        L.qso_float_to_half_rn.argtypes = [ctypes.c_float]
        L.qso_float_to_half_ru.restype = ctypes.c_uint16
        L.qso_float_to_half_ru.argtypes = [ctypes.c_float]
        L.qso_quantize_group.restype = None
        L.qso_quantize_group.argtypes = [P, L_, I, P, P, P, L_]
        L.qso_dequant.restype = D_
        L.qso_dequant.argtypes = [ctypes.c_uint8, ctypes.c_uint16, ctypes.c_uint16, I]
        L.qso_split_code.restype = None
        L.qso_split_code.argtypes = [ctypes.c_uint8, P, P]
        for name, args in (("qso_append", [P, P, P, I]), ("qso_rollback", [P, P]),
                           ("qso_need_flush", [P, I, P]), ("qso_flush", [P, P]),
                           ("qso_prefill", [P, P, P, I, P]),
                           ("qso_spec_accept", [P, P, P, P, P, I, I, I, P, P, P]),
                           ("qso_attn", [P, I, P, I, I, D_, P, P])):
            f = getattr(L, name)
            f.restype = None
            f.argtypes = args
        L.qso_num_threads.restype = I
        L.qso_num_threads.argtypes = []
        _lib = L
    return _lib


def _ptr(a):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def _as_half_bits(x):
    x = np.ascontiguousarray(x)
    if x.dtype == np.float16:
        return x.view(np.uint16)
    assert x.dtype == np.uint16
    return x


# ------------------------------------------------------------------ scalars

def half_to_double(h):
    return lib().qso_half_to_double(int(h))


def float_to_half_rn(f):
    return lib().qso_float_to_half_rn(float(np.float32(f)))


def float_to_half_ru(f):
    return lib().qso_float_to_half_ru(float(np.float32(f)))


def quantize_group(x):
    """QS-RN-v1 on a 1-D fp16 group -> (scale bits, zero bits, uint8 codes)."""
    x = _as_half_bits(np.asarray(x))
    assert x.ndim == 1
    s = np.zeros(1, np.uint16)
    z = np.zeros(1, np.uint16)
    q = np.zeros(x.shape[0], np.uint8)
    lib().qso_quantize_group(_ptr(x), 1, x.shape[0], _ptr(s), _ptr(z), _ptr(q), 1)
    return int(s[0]), int(z[0]), q


def split_code(q):
    u = ctypes.c_uint8()
    l_ = ctypes.c_uint8()
    lib().qso_split_code(int(q), ctypes.byref(u), ctypes.byref(l_))
    return u.value, l_.value


def dequant(q, scale_bits, zero_bits, upper_only, upper_bits=4):
    """fp64 dequantized value of code q: the INT8 code, or (upper_only) the
    draft's reconstruction from the top upper_bits bits."""
    return lib().qso_dequant(int(q), int(scale_bits), int(zero_bits),
                             int(upper_bits) if upper_only else 0)


def spec_accept(p, q, draft, u, e):
    """Speculative-sampling verification (see qso_spec_accept): p [B, g+1, V],
    q [B, g, V], u [B, g] float32; draft [B, g] int32; e [B, V] float32 Exp(1)
    variates.  Returns (n_accept, token, n_drop), int32 [B] each."""
    p, q, u, e = (np.ascontiguousarray(x, np.float32) for x in (p, q, u, e))
    draft = np.ascontiguousarray(draft, np.int32)
    B, g1, V = p.shape
    g = g1 - 1
    assert q.shape == (B, g, V) and draft.shape == (B, g) and u.shape == (B, g) and e.shape == (B, V)
    na, tok, nd = (np.zeros(B, np.int32) for _ in range(3))
    lib().qso_spec_accept(_ptr(p), _ptr(q), _ptr(draft), _ptr(u), _ptr(e), B, g, V,
                          _ptr(na), _ptr(tok), _ptr(nd))
    return na, tok, nd


def num_threads():
    return lib().qso_num_threads()


# ------------------------------------------------------------------ cache

class OracleCache:
    """Logical cache state held in numpy arrays; every method calls the C
    oracle on them in place."""

    def __init__(self, B, H, D=128, G=128, cap=8):
        self.B, self.H, self.D, self.G, self.cap = B, H, D, G, cap
        self.kq = np.zeros((B, H, cap, G, D), np.uint8)
        self.vq = np.zeros((B, H, cap, G, D), np.uint8)
        self.ks = np.zeros((B, H, cap, D), np.uint16)
        self.kz = np.zeros((B, H, cap, D), np.uint16)
        self.vs = np.zeros((B, H, cap, G), np.uint16)
        self.vz = np.zeros((B, H, cap, G), np.uint16)
        self.bk = np.zeros((B, H, 2 * G, D), np.uint16)
        self.bv = np.zeros((B, H, 2 * G, D), np.uint16)
        self.state = np.zeros((B, STATE_WORDS), np.int32)

    def _c(self):
        return _Cache(self.B, self.H, self.D, self.G, self.cap,
                      _ptr(self.kq).value, _ptr(self.vq).value,
                      _ptr(self.ks).value, _ptr(self.kz).value,
                      _ptr(self.vs).value, _ptr(self.vz).value,
                      _ptr(self.bk).value, _ptr(self.bv).value,
                      _ptr(self.state).value)

    def append(self, k_new, v_new):
        k = _as_half_bits(k_new)
        v = _as_half_bits(v_new)
        assert k.shape == v.shape and k.shape[:2] == (self.B, self.H) and k.shape[3] == self.D
        c = self._c()
        lib().qso_append(ctypes.byref(c), _ptr(k), _ptr(v), k.shape[2])

    def rollback(self, n_drop):
        n = np.ascontiguousarray(np.broadcast_to(np.asarray(n_drop, np.int32), (self.B,)))
        c = self._c()
        lib().qso_rollback(ctypes.byref(c), _ptr(n))

    def need_flush(self, n_next):
        m = np.zeros(self.B, np.uint8)
        c = self._c()
        lib().qso_need_flush(ctypes.byref(c), int(n_next), _ptr(m))
        return m

    def flush(self, mask=None):
        c = self._c()
        if mask is None:
            lib().qso_flush(ctypes.byref(c), None)
        else:
            m = np.ascontiguousarray(np.asarray(mask, np.uint8))
            lib().qso_flush(ctypes.byref(c), _ptr(m))

    def prefill(self, k, v, lens):
        """Fill empty caches from a prompt: k, v [B, H, T, D] fp16, lens [B]."""
        kb = _as_half_bits(k)
        vb = _as_half_bits(v)
        assert kb.shape == vb.shape and kb.shape[:2] == (self.B, self.H) and kb.shape[3] == self.D
        n = np.ascontiguousarray(np.broadcast_to(np.asarray(lens, np.int32), (self.B,)))
        c = self._c()
        lib().qso_prefill(ctypes.byref(c), _ptr(kb), _ptr(vb), kb.shape[2], _ptr(n))

    def attn(self, q, upper_only, scale=None, group=1, upper_bits=4):
        """Decode attention in fp64: q [B, H*group, n_q, D] fp16 ->
        (out [B, H*group, n_q, D] float64, lse [B, H*group, n_q] float64);
        query head h*group + i reads KV head h.  upper_only: the draft, which
        reconstructs each code from its top upper_bits bits."""
        qb = _as_half_bits(q)
        assert qb.shape[1] == self.H * group
        n_q = qb.shape[2]
        if scale is None:
            scale = 1.0 / np.sqrt(self.D)
        scale = float(np.float32(scale))
        out = np.zeros((self.B, self.H * group, n_q, self.D), np.float64)
        lse = np.zeros((self.B, self.H * group, n_q), np.float64)
        c = self._c()
        lib().qso_attn(ctypes.byref(c), int(upper_bits) if upper_only else 0, _ptr(qb), n_q,
                       int(group), scale,
                       _ptr(out), _ptr(lse))
        return out, lse

    # views ------------------------------------------------------------
    def counters(self, b):
        s = self.state[b]
        return dict(n_groups=int(s[N_GROUPS]), fill=int(s[FILL]), pending=int(s[PENDING]),
                    half_base=int(s[HALF_BASE]), err=int(s[ERR]))

    def buffer_tokens(self, b, h):
        """Logical buffer tokens (oldest first): (k, v) fp16 bit arrays [fill, D]."""
        s = self.state[b]
        G = self.G
        idx = (s[HALF_BASE] * G + np.arange(s[FILL])) % (2 * G)
        return self.bk[b, h, idx], self.bv[b, h, idx]


def prefill(oc, tokens, n_groups, fill):
    """Bring an oracle cache to a starting state with the same sequence of
    state-machine operations a device prefill uses: per group append G tokens,
    commit (dropping them for sequences that already hold all their groups),
    flush the sequences that still need groups; then append the buffer tokens
    and commit each sequence's fill level.

    ``tokens(b, t0, n)`` returns that sequence's keys and values for tokens
    [t0, t0 + n) as fp16 arrays [H, n, D]."""
    B, H, D, G = oc.B, oc.H, oc.D, oc.G
    ng = np.asarray(n_groups)
    fl = np.asarray(fill)
    for g in range(int(ng.max(initial=0))):
        k = np.zeros((B, H, G, D), np.float16)
        v = np.zeros_like(k)
        for b in range(B):
            if g < ng[b]:
                k[b], v[b] = tokens(b, g * G, G)
        oc.append(k, v)
        oc.rollback(np.where(g < ng, 0, G).astype(np.int32))
        oc.flush((g < ng).astype(np.uint8))
    fmax = int(fl.max(initial=0))
    if fmax:
        k = np.zeros((B, H, fmax, D), np.float16)
        v = np.zeros_like(k)
        for b in range(B):
            if fl[b]:
                k[b, :, :fl[b]], v[b, :, :fl[b]] = tokens(b, int(ng[b]) * G, int(fl[b]))
        oc.append(k, v)
        oc.rollback((fmax - fl).astype(np.int32))
