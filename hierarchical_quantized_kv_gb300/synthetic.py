"""Seeded synthetic inputs for the decode-attention workloads.

This module only draws random numbers; it holds none of the method's
arithmetic, so both the CUDA path and the CPU oracle can be fed from it.

Value recipe (Llama-2-7B attention shapes: head_dim 128, MHA):
  * K, V, Q ~ N(0, 1), cast to fp16 with round-to-nearest;
  * per (sequence, head) a random subset of key channels is scaled by a
    factor (outlier channels: 4 x 10 on the tiny case, round(0.02*128) = 3 x 8
    elsewhere);
  * ragged batches draw per-sequence context lengths and buffer fill levels
    uniformly.

Every draw comes from numpy's PCG64 keyed by a ``SeedSequence`` of
(seed, stream tag, indices), so a token chunk's values do not depend on how
many other chunks were drawn before it.
"""
from dataclasses import dataclass, field

import numpy as np

TAG_KV, TAG_Q, TAG_OUTLIER, TAG_LEN, TAG_ACCEPT = 1, 2, 3, 4, 5
CHUNK = 128  # tokens per generated chunk


def _rng(*key):
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(list(key))))


@dataclass(frozen=True)
class Workload:
    """One synthetic decode-attention workload (all sizes in tokens)."""
    name: str
    B: int
    H: int
    D: int = 128
    G: int = 128
    context: tuple = ()          # per-sequence total context (quantized + buffer)
    fill: tuple = ()             # per-sequence buffer fill at start
    n_outlier: int = 3
    outlier_factor: float = 8.0
    gamma: int = 4
    seed: int = 0
    group: int = 1               # query heads per KV head (H counts KV heads)
    extra: dict = field(default_factory=dict)

    @property
    def quantized(self):
        return tuple(c - f for c, f in zip(self.context, self.fill))

    @property
    def n_groups(self):
        return tuple(t // self.G for t in self.quantized)


def tiny(seed=0):
    return Workload("tiny_b1_h2_ctx1024", B=1, H=2, context=(1024,), fill=(256,),
                    n_outlier=4, outlier_factor=10.0, seed=seed)


def llama_32k(seed=0):
    return Workload("llama2_7b_b1_h32_ctx32768", B=1, H=32, context=(32768,), fill=(256,),
                    seed=seed)


def llama31_8b_32k(seed=0):
    """Llama-3.1-8B attention shape: 32 query heads on 8 KV heads (group 4)."""
    return Workload("llama31_8b_b1_kv8_q32_ctx32768", B=1, H=8, context=(32768,), fill=(256,),
                    seed=seed, group=4)


def ctx_128k(seed=0):
    return Workload("b1_h32_ctx131072", B=1, H=32, context=(131072,), fill=(256,), seed=seed)


def batched_32k(seed=0):
    return Workload("batched_b8_h32_ctx32768", B=8, H=32, context=(32768,) * 8,
                    fill=(256,) * 8, seed=seed)


def ragged(seed=0, B=16, lo=4096, hi=65536):
    """Context L_b ~ U[lo, hi], fill f_b ~ U[1, 256]; the quantized part is
    128 * floor((L_b - f_b) / 128), so the actual context is within 127
    tokens of L_b and stays a whole number of groups."""
    r = _rng(seed, TAG_LEN)
    L = r.integers(lo, hi, endpoint=True, size=B)
    f = r.integers(1, 256, endpoint=True, size=B)
    q = 128 * ((L - f) // 128)
    return Workload("ragged_b%d_h32_ctx%d_%d" % (B, lo, hi), B=B, H=32,
                    context=tuple(int(a + b) for a, b in zip(q, f)),
                    fill=tuple(int(x) for x in f), seed=seed)


CONFIGS = {"tiny": tiny, "32k": llama_32k, "128k": ctx_128k,
           "batched32k": batched_32k, "ragged": ragged, "gqa32k": llama31_8b_32k}


def outlier_channels(w: Workload, b: int):
    """[H, n_outlier] distinct key-channel indices for sequence b."""
    r = _rng(w.seed, TAG_OUTLIER, b)
    return np.stack([r.choice(w.D, size=w.n_outlier, replace=False) for _ in range(w.H)])


def kv_chunk(w: Workload, b: int, chunk: int, n: int = CHUNK):
    """Keys and values for tokens [chunk*128, chunk*128 + n) of sequence b:
    two fp16 arrays [H, n, D] (n <= 128)."""
    assert 0 < n <= CHUNK
    r = _rng(w.seed, TAG_KV, b, chunk)
    k = r.standard_normal((w.H, CHUNK, w.D), dtype=np.float32)
    v = r.standard_normal((w.H, CHUNK, w.D), dtype=np.float32)
    if w.n_outlier:
        idx = outlier_channels(w, b)
        for h in range(w.H):
            k[h, :, idx[h]] *= np.float32(w.outlier_factor)
    return k[:, :n].astype(np.float16), v[:, :n].astype(np.float16)


def kv_tokens(w: Workload, b: int, t0: int, n: int):
    """Keys and values for tokens [t0, t0 + n) of sequence b: fp16 [H, n, D]."""
    ks, vs = [], []
    t = t0
    while t < t0 + n:
        c = t // CHUNK
        lo = t - c * CHUNK
        hi = min(CHUNK, t0 + n - c * CHUNK)
        k, v = kv_chunk(w, b, c, hi)
        ks.append(k[:, lo:hi])
        vs.append(v[:, lo:hi])
        t = c * CHUNK + hi
    if not ks:
        z = np.zeros((w.H, 0, w.D), np.float16)
        return z, z.copy()
    return np.concatenate(ks, axis=1), np.concatenate(vs, axis=1)


def queries(w: Workload, call: int, n_q: int):
    """Queries for decode call number ``call``: fp16 [B, H * group, n_q, D]."""
    r = _rng(w.seed, TAG_Q, call)
    return r.standard_normal((w.B, w.H * w.group, n_q, w.D), dtype=np.float32).astype(np.float16)


def accepted_counts(w: Workload, step: int):
    """Seeded accepted-draft counts a_b in 0..gamma for speculative round ``step``."""
    r = _rng(w.seed, TAG_ACCEPT, step)
    return r.integers(0, w.gamma, endpoint=True, size=w.B).astype(np.int32)
