"""Test-side model of the device cache layout, written from include/qs.h.

It converts the oracle's logical state (8-bit codes, scales, zeros, buffer,
counters) to the byte layout the header specifies and back, so tests can
compare device arrays bit for bit or load oracle state into a device cache.
It shares no code with the CUDA library.
"""
import numpy as np

import oracle


def vperm(p):
    """Token (within a 32-token quarter) stored at nibble position p of a
    16-byte value row: 32u + 16((p>>1)&1) + 8(p&1) + 2(p>>3) + ((p>>2)&1)."""
    p = np.asarray(p)
    return 16 * ((p >> 1) & 1) + 8 * (p & 1) + 2 * (p >> 3) + ((p >> 2) & 1)


def _nibbles_to_bytes(n):
    return (n[..., 0::2] | (n[..., 1::2] << 4)).astype(np.uint8)


def pack_k(kq):
    """codes [..., G, D] -> (upper, lower) planes [..., G, D/2]."""
    return _nibbles_to_bytes(kq >> 4), _nibbles_to_bytes(kq & 15)


def pack_v(vq):
    """codes [..., G tokens, D] -> planes [..., G/32, D, 16]."""
    G, D = vq.shape[-2], vq.shape[-1]
    tok = (32 * np.arange(G // 32)[:, None] + vperm(np.arange(32))[None, :])  # [4, 32]
    perm = vq[..., tok, :]                    # [..., 4, 32, D]
    perm = np.swapaxes(perm, -1, -2)          # [..., 4, D, 32]
    return _nibbles_to_bytes(perm >> 4), _nibbles_to_bytes(perm & 15)


def unpack_k(upper, lower):
    u = np.stack([upper & 15, upper >> 4], -1).reshape(*upper.shape[:-1], -1)
    l_ = np.stack([lower & 15, lower >> 4], -1).reshape(*lower.shape[:-1], -1)
    return (u << 4 | l_).astype(np.uint8)


def kmeta_perm(p):
    """Channel stored at position p of a key scale / zero row."""
    p = np.asarray(p)
    return 32 * ((p >> 3) & 3) + 8 * (p >> 5) + 2 * ((p >> 2) & 1) + ((p >> 1) & 1) + 4 * (p & 1)


def vmeta_perm(p):
    """Token stored at position p of a value scale / zero row."""
    p = np.asarray(p)
    return 32 * (p >> 5) + ((p >> 2) & 7) + 16 * ((p >> 1) & 1) + 8 * (p & 1)


def meta(ks, kz, vs, vz):
    """fp16 bit arrays [..., 128] x4 -> [..., 4, 128] (rows: K scale, K zero,
    V scale, V zero), each row in the header's position order."""
    kp, vp = kmeta_perm(np.arange(128)), vmeta_perm(np.arange(128))
    return np.stack([ks[..., kp], kz[..., kp], vs[..., vp], vz[..., vp]], axis=-2).astype(np.uint16)


def repack_upper2(plane):
    """A 4-bit upper plane (8 KB per group, any group shape) in the two-bit
    draft layout of include/qs.h: per group, words 2k and 2k+1 of the nibble
    plane give word k of the C_U2 plane (first 4 KB) and of the M2 plane
    (second 4 KB); nibble j of word k holds word 2k's field in bits 0-1 and
    word 2k+1's in bits 2-3 (C_U = 4 C_U2 + M2)."""
    shp = plane.shape
    w = np.ascontiguousarray(plane).reshape(-1, 2048).view(np.uint8)
    w = w.reshape(-1, 8192).copy().view("<u4")  # [groups, 2048] words
    a, b = w[:, 0::2], w[:, 1::2]
    u2 = ((a >> 2) & 0x33333333) | (b & 0xCCCCCCCC)
    m2 = (a & 0x33333333) | ((b & 0x33333333) << 2)
    out = np.concatenate([u2, m2], axis=1).astype("<u4")
    return out.view(np.uint8).reshape(shp)


def device_arrays(oc: oracle.OracleCache, upper_bits=4):
    """The oracle state in the device layout (numpy); upper_bits = 2 gives the
    two-bit draft layout of the upper planes."""
    ku, kl = pack_k(oc.kq)
    vu, vl = pack_v(oc.vq)
    if upper_bits == 2:
        ku, vu = repack_upper2(ku), repack_upper2(vu)
    return dict(k_upper=ku, k_lower=kl, v_upper=vu, v_lower=vl,
                meta=meta(oc.ks, oc.kz, oc.vs, oc.vz),
                buf_k=oc.bk, buf_v=oc.bv, state=oc.state)


def load_into(cache, oc: oracle.OracleCache):
    """Copy the oracle's state into a device cache (qs.Cache)."""
    import torch
    arrs = device_arrays(oc, getattr(cache, "upper_bits", 4))
    for name, a in arrs.items():
        t = getattr(cache, name)
        src = torch.from_numpy(np.ascontiguousarray(a))
        if t.dtype == torch.float16:
            src = src.view(torch.int16).view(torch.float16)
        t.copy_(src.reshape(t.shape))


def read_device(cache):
    """Device cache arrays as numpy (fp16 as uint16 bits)."""
    import torch
    out = {}
    for name in ("k_upper", "k_lower", "v_upper", "v_lower", "meta", "buf_k", "buf_v", "state"):
        t = getattr(cache, name).detach().cpu()
        if t.dtype == torch.float16:
            t = t.view(torch.int16)
        a = t.numpy()
        out[name] = a.view(np.uint16) if a.dtype == np.int16 else a
    return out
