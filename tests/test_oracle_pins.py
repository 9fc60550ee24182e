"""Pins of the CPU oracle against facts fixed by the pages and by mathematics.

Each test checks the oracle against something other than itself: library
routines (numpy fp16), hand-derived closed forms (tests/golden), bounds that
follow from the quantizer's definition, invariants of the buffer state
machine, and textbook softmax attention in special cases that reduce to it.
"""
import os

import numpy as np
import pytest

import oracle
from hierarchical_quantized_kv_gb300 import synthetic

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "qs_rn_v1_closed_form.txt")


def h(x):
    return np.asarray(x, np.float16)


def hbits(x):
    return h(x).view(np.uint16)


def f16(bits):
    return np.asarray(bits, np.uint16).view(np.float16).astype(np.float64)


# ----------------------------------------------------------------- fp16

def test_half_decode_matches_numpy_for_every_pattern():
    bits = np.arange(65536, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.half_to_double(b) for b in bits])
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite], ref[finite])
    assert np.array_equal(np.isinf(got), np.isinf(ref))
    assert np.array_equal(np.isnan(got), np.isnan(ref))


def test_float_to_half_round_nearest_matches_numpy():
    r = np.random.default_rng(1)
    xs = np.concatenate([
        r.standard_normal(4000).astype(np.float32) * np.float32(10) ** r.integers(-9, 5, 4000),
        np.float32([0.0, -0.0, 65504, 65519.99, 65520, -65520, 1e-8, 2.98e-8, 5.96e-8, 6.1e-5]),
        # exact ties between fp16 neighbours
        (np.arange(1, 200, dtype=np.float32) + np.float32(0.5)) * np.float32(2.0 ** -10),
    ]).astype(np.float32)
    with np.errstate(over="ignore"):
        ref = xs.astype(np.float16).view(np.uint16)
    got = np.array([oracle.float_to_half_rn(x) for x in xs], np.uint16)
    assert np.array_equal(got, ref)


def test_float_to_half_round_up_is_smallest_not_below():
    r = np.random.default_rng(2)
    xs = (r.random(3000).astype(np.float32) * np.float32(2.0) ** r.integers(-26, 15, 3000)).astype(np.float32)
    xs = np.concatenate([xs, np.float32([1.0, 0.5, 2.0 ** -24, 3 * 2.0 ** -25, 1 / 255.0])])
    for x in xs:
        b = oracle.float_to_half_ru(x)
        v = float(np.uint16(b).view(np.float16))
        assert v >= float(x)
        below = float(np.nextafter(np.float16(v), np.float16(-np.inf)))
        assert below < float(x)


# ------------------------------------------------- quantizer closed forms

def _golden_cases():
    cases = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, xs, s, z, q = [p.strip() for p in line.split("|")]
            cases.append((name, [float(v) for v in xs.split()], int(s, 16), int(z, 16),
                          [int(v) for v in q.split()]))
    return cases


@pytest.mark.parametrize("case", _golden_cases(), ids=lambda c: c[0])
def test_golden_closed_form(case):
    name, xs, s, z, q = case
    gs, gz, gq = oracle.quantize_group(h(xs))
    assert (gs, gz) == (s, z), name
    assert gq.tolist() == q, name


def test_nibble_repack_exhaustive():
    # x = 0..255 has r = 255, s = 1, z = 0, so code i is exactly i
    s, z, q = oracle.quantize_group(h(np.arange(256)))
    assert (s, z) == (0x3C00, 0)
    assert q.tolist() == list(range(256))
    for c in range(256):
        u, l_ = oracle.split_code(c)
        assert 0 <= u < 16 and 0 <= l_ < 16
        assert 16 * u + l_ == c


@pytest.mark.parametrize("seed", range(6))
def test_grid_aligned_group_is_lossless(seed):
    # x = z + s*k with k in 0..255 (0 and 255 present), s a power of two:
    # every step of QS-RN-v1 is exact, so the codes are k and deq8 == x.
    r = np.random.default_rng(seed)
    e = int(r.integers(-8, -1))
    s = 2.0 ** e
    z = float(r.integers(-1000, 1000)) * s   # |x| / s < 2048: exact in fp16
    k = r.integers(0, 256, 128)
    k[3], k[77] = 0, 255
    x = z + s * k
    assert np.array_equal(h(x).astype(np.float64), x)
    gs, gz, gq = oracle.quantize_group(h(x))
    assert f16(gs) == s and f16(gz) == z
    assert np.array_equal(gq, k)
    for i in range(0, 128, 7):
        assert oracle.dequant(gq[i], gs, gz, False) == x[i]


def test_constant_and_two_valued_groups():
    for v in (0.0, -2.5, 3.0e4, 1e-7):
        s, z, q = oracle.quantize_group(h([v] * 128))
        assert s == 0 and np.all(q == 0)
        assert oracle.dequant(0, s, z, False) == float(np.float16(v))
        assert oracle.dequant(0, s, z, True) == float(np.float16(v))
    r = np.random.default_rng(3)
    for _ in range(200):
        a, b = np.sort(h(r.standard_normal(2) * 10.0 ** r.integers(-3, 3)))
        if float(b) - float(a) < 255 * 2.0 ** -14:
            continue  # subnormal fp16 scale: rounding it up may cost more than a code
        x = np.where(r.random(128) < 0.5, a, b).astype(np.float16)
        x[0], x[1] = a, b
        s, z, q = oracle.quantize_group(x)
        assert set(q.tolist()) <= {0, 255}
        assert np.all((q == 255) == (x == b))


@pytest.mark.parametrize("scale_exp", [-6, 0, 4])
def test_dequant_error_bounds(scale_exp):
    # |x - deq8| <= s (1/2 + eps), |x - deqU| <= s (8.5 + eps), eps covers the
    # two fp32 roundings inside u (about 255 * 2 * 2^-24 < 2^-13).
    r = np.random.default_rng(10 + scale_exp)
    worst8, worstU = 0.0, 0.0
    for _ in range(300):
        x = h(r.standard_normal(128) * 2.0 ** scale_exp + r.uniform(-3, 3) * 2.0 ** scale_exp)
        s, z, q = oracle.quantize_group(x)
        sv = f16(s)
        xd = x.astype(np.float64)
        d8 = np.array([oracle.dequant(c, s, z, False) for c in q])
        dU = np.array([oracle.dequant(c, s, z, True) for c in q])
        e8 = np.max(np.abs(xd - d8)) / sv
        eU = np.max(np.abs(xd - dU)) / sv
        assert e8 <= 0.5 + 2.0 ** -13
        assert eU <= 8.5 + 2.0 ** -13
        worst8, worstU = max(worst8, e8), max(worstU, eU)
    # the bounds are approached, so they are the right ones
    assert worst8 > 0.49 and worstU > 8.3


@pytest.mark.parametrize("scale_exp", [-6, 0, 4])
def test_two_bit_draft_error_bound(scale_exp):
    """Top-2-bit draft (a k-bit draft in general, the pages show k = 4 only):
    the reconstruction sits at the middle of the 64 codes sharing the top two
    bits, so |x - deq2| <= s (32.5 + eps), and the bound is reached."""
    r = np.random.default_rng(30 + scale_exp)
    worst = 0.0
    for _ in range(300):
        x = h(r.standard_normal(128) * 2.0 ** scale_exp + r.uniform(-3, 3) * 2.0 ** scale_exp)
        s, z, q = oracle.quantize_group(x)
        d2 = np.array([oracle.dequant(c, s, z, True, upper_bits=2) for c in q])
        e = np.max(np.abs(x.astype(np.float64) - d2)) / f16(s)
        assert e <= 32.5 + 2.0 ** -13
        worst = max(worst, e)
    assert worst > 31.5


def test_k_bit_draft_is_the_int8_code_at_the_bucket_middle():
    """For every code, the k-bit draft value is the INT8 value of the code
    with the same top k bits and the low bits at the middle (k = 4: | 0x08;
    k = 2: | 0x20), and the draft reads no bit below the top k."""
    s, z = int(hbits(0.0625)), int(hbits(-3.0))
    for q in range(256):
        assert oracle.dequant(q, s, z, True, 4) == oracle.dequant((q & 0xF0) | 0x08, s, z, False)
        assert oracle.dequant(q, s, z, True, 2) == oracle.dequant((q & 0xC0) | 0x20, s, z, False)
        assert oracle.dequant(q, s, z, True, 2) == oracle.dequant(q & 0xC0, s, z, True, 2)


def test_codes_stay_in_range_for_extreme_groups():
    for x in ([-65504.0, 65504.0] + [0.0] * 126, [-1e-3, 6e4] * 64):
        s, z, q = oracle.quantize_group(h(x))
        assert q.min() == 0 and q.max() == 255
    # a range of two subnormal steps: the scale is a subnormal fp16, the top
    # code falls short of 255 but every code stays a valid byte
    s, z, q = oracle.quantize_group(h([6e-8, 1.8e-7] * 64))
    assert q.min() == 0 and 0 < q.max() <= 255


# ------------------------------------------------- buffer state machine

def _stream(rng, H, n, D=128):
    return (h(rng.standard_normal((1, H, n, D))), h(rng.standard_normal((1, H, n, D))))


@pytest.mark.parametrize("seed", range(4))
def test_history_independence_and_rollback(seed):
    """After random append / rollback / flush sequences the quantized groups
    equal QS-RN-v1 applied to the committed token stream in consecutive
    G-chunks, the buffer holds the stream's tail, and a rollback never
    changes an existing group."""
    rng = np.random.default_rng(100 + seed)
    H, G, D = 2, 128, 128
    c = oracle.OracleCache(1, H, D, G, cap=8)
    committed_k, committed_v = [], []   # plain list model of the stream
    pending_k, pending_v = [], []
    for step in range(520):
        if c.need_flush(5)[0]:
            c.flush()
            cnt = c.counters(0)
            assert cnt["err"] == 0
        n_new = int(rng.integers(1, 6))
        k, v = _stream(rng, H, n_new)
        c.append(k, v)
        pending_k += [k[0, :, i] for i in range(n_new)]
        pending_v += [v[0, :, i] for i in range(n_new)]
        drop = int(rng.integers(0, n_new + 1))
        groups_before = (c.kq.copy(), c.vq.copy(), c.ks.copy(), c.vs.copy())
        c.rollback([drop])
        for a, b in zip(groups_before, (c.kq, c.vq, c.ks, c.vs)):
            assert np.array_equal(a, b)
        keep = len(pending_k) - drop
        committed_k += pending_k[:keep]
        committed_v += pending_v[:keep]
        pending_k, pending_v = [], []
    cnt = c.counters(0)
    assert cnt["err"] == 0 and cnt["pending"] == 0
    ng = cnt["n_groups"]
    assert ng >= 3
    assert ng * G + cnt["fill"] == len(committed_k)
    K = np.stack(committed_k, axis=1)  # [H, T, D]
    V = np.stack(committed_v, axis=1)
    for hh in range(H):
        for g in range(ng):
            kt = K[hh, g * G:(g + 1) * G]
            vt = V[hh, g * G:(g + 1) * G]
            for d in range(0, D, 5):
                s, z, q = oracle.quantize_group(np.ascontiguousarray(kt[:, d]))
                assert c.ks[0, hh, g, d] == s and c.kz[0, hh, g, d] == z
                assert np.array_equal(c.kq[0, hh, g, :, d], q)
            for t in range(0, G, 5):
                s, z, q = oracle.quantize_group(np.ascontiguousarray(vt[t]))
                assert c.vs[0, hh, g, t] == s and c.vz[0, hh, g, t] == z
                assert np.array_equal(c.vq[0, hh, g, t], q)
        bk, bv = c.buffer_tokens(0, hh)
        assert np.array_equal(bk, K[hh, ng * G:].view(np.uint16))
        assert np.array_equal(bv, V[hh, ng * G:].view(np.uint16))


def test_error_paths_are_flagged_and_no_ops():
    rng = np.random.default_rng(7)
    c = oracle.OracleCache(2, 1, 128, 128, cap=1)
    k, v = rng.standard_normal((2, 1, 200, 128)), rng.standard_normal((2, 1, 200, 128))
    c.append(h(k), h(v))
    snap = c.state.copy()
    c.append(h(k[:, :, :57]), h(v[:, :, :57]))           # 257 > 256
    assert np.all(c.state[:, oracle.ERR] & oracle.DEV_OVERFLOW)
    assert np.array_equal(c.state[:, :4], snap[:, :4])
    c.state[:, oracle.ERR] = 0
    c.flush()                                             # 0 committed
    assert np.all(c.state[:, oracle.ERR] == oracle.DEV_FLUSH_UNCOMMITTED)
    c.state[:, oracle.ERR] = 0
    c.rollback([201, 10])                                 # seq 0 drops more than pending
    assert c.state[0, oracle.ERR] == oracle.DEV_OVER_ROLLBACK and c.state[1, oracle.ERR] == 0
    assert c.counters(0)["fill"] == 200 and c.counters(1)["fill"] == 190
    c.state[:, oracle.ERR] = 0
    c.rollback([0, 0])
    c.flush([1, 1])
    assert np.all(c.state[:, oracle.N_GROUPS] == 1)
    c.append(h(k[:, :, :70]), h(v[:, :, :70]))
    c.rollback([0, 0])
    c.flush([0, 1])                                       # capacity 1 reached
    assert c.state[0, oracle.ERR] == 0 and c.state[1, oracle.ERR] == oracle.DEV_CAPACITY
    q = h(rng.standard_normal((2, 1, 3, 128)))
    c2 = oracle.OracleCache(1, 1, 128, 128, cap=1)
    c2.append(h(k[:1, :, :2]), h(v[:1, :, :2]))
    out, lse = c2.attn(q[:1], upper_only=False)
    assert c2.state[0, oracle.ERR] == oracle.DEV_NQ_GT_FILL
    assert np.all(out == 0) and np.all(np.isneginf(lse))


# ------------------------------------------------------------- attention

def naive_attention(q, K, V, scale):
    """Textbook softmax attention in fp64 for one query row."""
    s = scale * (K @ q)
    w = np.exp(s - s.max())
    return (w[:, None] * V).sum(0) / w.sum(), s.max() + np.log(w.sum())


@pytest.mark.parametrize("fill", [1, 5, 130, 256])
def test_empty_quantized_region_is_plain_softmax_attention(fill):
    rng = np.random.default_rng(fill)
    B, H, D = 2, 3, 128
    c = oracle.OracleCache(B, H, D, 128, cap=2)
    k = h(rng.standard_normal((B, H, fill, D)) * 2)
    v = h(rng.standard_normal((B, H, fill, D)))
    c.append(k, v)
    n_q = min(5, fill)
    q = h(rng.standard_normal((B, H, n_q, D)))
    scale = 1 / np.sqrt(D)
    for upper in (False, True):
        out, lse = c.attn(q, upper_only=upper, scale=scale)
        for b in range(B):
            for hh in range(H):
                for j in range(n_q):
                    last = fill - n_q + j
                    ref, rl = naive_attention(q[b, hh, j].astype(np.float64),
                                              k[b, hh, :last + 1].astype(np.float64),
                                              v[b, hh, :last + 1].astype(np.float64),
                                              float(np.float32(scale)))
                    np.testing.assert_allclose(out[b, hh, j], ref, rtol=1e-12, atol=1e-12)
                    assert abs(lse[b, hh, j] - rl) < 1e-11


def _grid_tokens(rng, H, n, D, G):
    """Tokens whose every key channel group (G tokens) and value token group
    (D channels) lies on a power-of-two grid with both ends present, so the
    quantization is lossless (see test_grid_aligned_group_is_lossless)."""
    k = np.zeros((H, n, D))
    v = np.zeros((H, n, D))
    for hh in range(H):
        for g in range(n // G):
            sk = 2.0 ** rng.integers(-7, -3, D)
            zk = rng.integers(-40, 40, D) * sk
            code = rng.integers(0, 256, (G, D))
            code[0], code[1] = 0, 255
            k[hh, g * G:(g + 1) * G] = zk + sk * code
            sv = 2.0 ** rng.integers(-7, -3, G)
            zv = rng.integers(-40, 40, G) * sv
            code = rng.integers(0, 256, (G, D))
            code[:, 0], code[:, 1] = 0, 255
            v[hh, g * G:(g + 1) * G] = zv[:, None] + sv[:, None] * code
    assert np.array_equal(h(k).astype(np.float64), k) and np.array_equal(h(v).astype(np.float64), v)
    return h(k), h(v)


def test_verify_attention_on_lossless_groups_equals_plain_attention():
    rng = np.random.default_rng(11)
    H, D, G = 2, 128, 128
    c = oracle.OracleCache(1, H, D, G, cap=4)
    kq, vq = _grid_tokens(rng, H, 3 * G, D, G)
    for g in range(3):
        c.append(kq[None, :, g * G:(g + 1) * G], vq[None, :, g * G:(g + 1) * G])
        c.rollback([0])
        c.flush()
    kb = h(rng.standard_normal((1, H, 40, D)))
    vb = h(rng.standard_normal((1, H, 40, D)))
    c.append(kb, vb)
    assert c.counters(0)["n_groups"] == 3 and c.counters(0)["fill"] == 40
    q = h(rng.standard_normal((1, H, 5, D)))
    out, lse = c.attn(q, upper_only=False)
    K = np.concatenate([kq, kb[0]], axis=1).astype(np.float64)
    V = np.concatenate([vq, vb[0]], axis=1).astype(np.float64)
    for hh in range(H):
        for j in range(5):
            last = 3 * G + 40 - 5 + j
            ref, rl = naive_attention(q[0, hh, j].astype(np.float64), K[hh, :last + 1],
                                      V[hh, :last + 1], float(np.float32(1 / np.sqrt(D))))
            np.testing.assert_allclose(out[0, hh, j], ref, rtol=1e-11, atol=1e-12)


def _dequantized_context(c, b, hh, upper_bits):
    """Brute force, from the stored arrays alone: every quantized group
    dequantized as s * code + z in fp64 (keys: scale and zero per channel;
    values: per token), followed by the logical buffer tokens.  upper_bits:
    None for the INT8 code, k for the k-bit draft (top k bits, low bits at
    their middle)."""
    ng = c.counters(b)["n_groups"]
    ks, kz = f16(c.ks[b, hh, :ng]), f16(c.kz[b, hh, :ng])     # [ng, D]
    vs, vz = f16(c.vs[b, hh, :ng]), f16(c.vz[b, hh, :ng])     # [ng, G]
    kq = c.kq[b, hh, :ng].astype(np.int64)                   # [ng, G, D]
    vq = c.vq[b, hh, :ng].astype(np.int64)
    if upper_bits is not None:
        low = 8 - upper_bits
        kq = ((kq >> low) << low) + (1 << (low - 1))
        vq = ((vq >> low) << low) + (1 << (low - 1))
    K = ks[:, None, :] * kq + kz[:, None, :]
    V = vs[:, :, None] * vq + vz[:, :, None]
    bk, bv = c.buffer_tokens(b, hh)
    K = np.concatenate([K.reshape(-1, c.D), f16(bk)])
    V = np.concatenate([V.reshape(-1, c.D), f16(bv)])
    return K, V


@pytest.mark.parametrize("group", [1, 2])
def test_attention_equals_brute_force_over_dequantized_groups(group):
    """Random (lossy) groups: both modes, n_q of 1 and 5, ragged sequences and
    a grouped-query layout, against textbook attention over the brute-force
    dequantized context, with query j of n_q seeing the context up to its own
    position."""
    rng = np.random.default_rng(17 + group)
    B, H, D, G = 2, 2, 128, 128
    c = oracle.OracleCache(B, H, D, G, cap=4)
    for n in (G, G, G, 77):
        k = h(rng.standard_normal((B, H, n, D)) * rng.uniform(0.2, 3, (B, H, 1, D))
              + rng.uniform(-2, 2, (B, H, 1, D)))
        v = h(rng.standard_normal((B, H, n, D)))
        c.flush(c.need_flush(n))
        c.append(k, v)
        c.rollback([0, n // 2])     # sequence 1 keeps half of each piece
    c.flush([1, 0])                 # ragged: sequence 0 gains one more group
    assert [c.counters(b)["n_groups"] for b in range(B)] == [3, 1]
    assert [c.counters(b)["fill"] for b in range(B)] == [77, 103]
    assert not c.state[:, oracle.ERR].any()
    scale = 1 / np.sqrt(D)
    for n_q in (1, 5):
        q = h(rng.standard_normal((B, H * group, n_q, D)))
        for ub in (None, 4, 2):
            out, lse = c.attn(q, upper_only=ub is not None, scale=scale, group=group,
                              upper_bits=ub or 4)
            for b in range(B):
                for qh in range(H * group):
                    K, V = _dequantized_context(c, b, qh // group, ub)
                    for j in range(n_q):
                        last = len(K) - n_q + j
                        ref, rl = naive_attention(q[b, qh, j].astype(np.float64), K[:last + 1],
                                                  V[:last + 1], float(np.float32(scale)))
                        np.testing.assert_allclose(out[b, qh, j], ref, rtol=1e-10, atol=1e-12)
                        assert abs(lse[b, qh, j] - rl) < 1e-10


def test_draft_equals_verify_when_every_lower_level_is_eight():
    rng = np.random.default_rng(12)
    H, D, G = 2, 128, 128
    c = oracle.OracleCache(1, H, D, G, cap=3)
    c.append(h(rng.standard_normal((1, H, 20, D))), h(rng.standard_normal((1, H, 20, D))))
    c.state[0, oracle.N_GROUPS] = 3
    c.kq[:] = (rng.integers(0, 16, c.kq.shape) * 16 + 8).astype(np.uint8)
    c.vq[:] = (rng.integers(0, 16, c.vq.shape) * 16 + 8).astype(np.uint8)
    for a in (c.ks, c.vs):
        a[:] = hbits(2.0 ** rng.integers(-8, -3, a.shape))
    for a in (c.kz, c.vz):
        a[:] = hbits(rng.uniform(-2, 2, a.shape))
    q = h(rng.standard_normal((1, H, 4, D)))
    o_d, l_d = c.attn(q, upper_only=True)
    o_v, l_v = c.attn(q, upper_only=False)
    assert np.array_equal(o_d, o_v) and np.array_equal(l_d, l_v)
    # and with the lower levels set to 0 the draft does differ
    c.kq[:] &= 0xF0
    o_v2, _ = c.attn(q, upper_only=False)
    o_d2, _ = c.attn(q, upper_only=True)
    assert np.array_equal(o_d2, o_d) and not np.allclose(o_v2, o_d)


def test_two_bit_draft_equals_verify_when_the_low_six_bits_are_32():
    rng = np.random.default_rng(13)
    H, D, G = 2, 128, 128
    c = oracle.OracleCache(1, H, D, G, cap=3)
    c.append(h(rng.standard_normal((1, H, 20, D))), h(rng.standard_normal((1, H, 20, D))))
    c.state[0, oracle.N_GROUPS] = 3
    c.kq[:] = (rng.integers(0, 4, c.kq.shape) * 64 + 32).astype(np.uint8)
    c.vq[:] = (rng.integers(0, 4, c.vq.shape) * 64 + 32).astype(np.uint8)
    for a in (c.ks, c.vs):
        a[:] = hbits(2.0 ** rng.integers(-8, -3, a.shape))
    for a in (c.kz, c.vz):
        a[:] = hbits(rng.uniform(-2, 2, a.shape))
    q = h(rng.standard_normal((1, H, 4, D)))
    o_d, l_d = c.attn(q, upper_only=True, upper_bits=2)
    o_v, l_v = c.attn(q, upper_only=False)
    assert np.array_equal(o_d, o_v) and np.array_equal(l_d, l_v)
    # codes with other low bits move the verify result but not the draft's
    c.kq[:] ^= (rng.integers(0, 32, c.kq.shape)).astype(np.uint8)
    o_d2, _ = c.attn(q, upper_only=True, upper_bits=2)
    o_v2, _ = c.attn(q, upper_only=False)
    o_d4, _ = c.attn(q, upper_only=True, upper_bits=4)
    assert np.array_equal(o_d2, o_d) and not np.allclose(o_v2, o_d) and not np.allclose(o_d4, o_d)


def test_causal_mask_matches_single_query_after_rollback():
    """Query j of an n_q-query call sees exactly what a single query sees
    after the last n_q-1-j pending tokens are rolled back."""
    w = synthetic.tiny()
    rng = np.random.default_rng(13)
    c = oracle.OracleCache(1, w.H, w.D, w.G, cap=4)
    k, v = synthetic.kv_tokens(w, 0, 0, 2 * w.G + 60)
    c.append(k[None, :, :w.G], v[None, :, :w.G])
    c.append(k[None, :, w.G:2 * w.G], v[None, :, w.G:2 * w.G])
    c.rollback([0])
    c.flush()
    c.append(k[None, :, 2 * w.G:], v[None, :, 2 * w.G:])
    c.rollback([0])
    n_q = 5
    kn = h(rng.standard_normal((1, w.H, n_q, w.D)))
    vn = h(rng.standard_normal((1, w.H, n_q, w.D)))
    c.append(kn, vn)
    q = h(rng.standard_normal((1, w.H, n_q, w.D)))
    for upper in (False, True):
        out, lse = c.attn(q, upper_only=upper)
        for j in range(n_q):
            c2 = oracle.OracleCache(1, w.H, w.D, w.G, cap=4)
            for name in ("kq", "vq", "ks", "kz", "vs", "vz", "bk", "bv", "state"):
                getattr(c2, name)[:] = getattr(c, name)
            c2.rollback([n_q - 1 - j])
            o1, l1 = c2.attn(q[:, :, j:j + 1], upper_only=upper)
            np.testing.assert_allclose(o1[:, :, 0], out[:, :, j], rtol=1e-13, atol=1e-14)
            np.testing.assert_allclose(l1[:, :, 0], lse[:, :, j], rtol=1e-13, atol=1e-14)


def test_single_visible_token_returns_its_value():
    rng = np.random.default_rng(14)
    c = oracle.OracleCache(1, 2, 128, 128, cap=1)
    k = h(rng.standard_normal((1, 2, 1, 128)))
    v = h(rng.standard_normal((1, 2, 1, 128)))
    c.append(k, v)
    out, lse = c.attn(h(rng.standard_normal((1, 2, 1, 128))), upper_only=True)
    assert np.array_equal(out[0, :, 0], v[0, :, 0].astype(np.float64))


def test_quantized_attention_error_is_bounded_by_dequant_error():
    """Attention over the quantized cache stays close to attention over the
    original fp16 tokens: verify (INT8) much closer than draft (upper 4)."""
    w = synthetic.tiny()
    c = oracle.OracleCache(1, w.H, w.D, w.G, cap=8)
    T = 6 * w.G
    k, v = synthetic.kv_tokens(w, 0, 0, T + 100)
    for g in range(6):
        c.append(k[None, :, g * w.G:(g + 1) * w.G], v[None, :, g * w.G:(g + 1) * w.G])
        c.rollback([0])
        c.flush()
    c.append(k[None, :, T:], v[None, :, T:])
    q = synthetic.queries(w, 0, 1)
    o8, _ = c.attn(q, upper_only=False)
    oU, _ = c.attn(q, upper_only=True)
    K, V = k.astype(np.float64), v.astype(np.float64)
    for hh in range(w.H):
        ref, _ = naive_attention(q[0, hh, 0].astype(np.float64), K[hh], V[hh],
                                 float(np.float32(1 / np.sqrt(w.D))))
        e8 = np.abs(o8[0, hh, 0] - ref).max()
        eU = np.abs(oU[0, hh, 0] - ref).max()
        assert e8 < 0.02 and e8 < eU


# --------------------------------------------------------------- bulk prefill

def _appended_prompt(rng, K, V, L, cap):
    """The state-machine path for a prompt: append its first L tokens in
    pieces of 1..G, committing each, with a flush before every append that
    would overflow the 2G buffer."""
    H, D = K.shape[1], K.shape[3]
    c = oracle.OracleCache(1, H, D, 128, cap)
    t = 0
    while t < L:
        n = min(int(rng.integers(1, 129)), L - t)
        if c.need_flush(n)[0]:
            c.flush()
        c.append(np.ascontiguousarray(K[:, :, t:t + n]), np.ascontiguousarray(V[:, :, t:t + n]))
        c.rollback([0])
        t += n
    return c


@pytest.mark.parametrize("L", [0, 1, 127, 128, 255, 256, 257, 383, 384, 385, 700, 1000])
def test_prefill_equals_appending_the_prompt(L):
    """A one-step prefill leaves the same groups, counters and logical buffer
    as appending the prompt piece by piece through the state machine (whose
    groups are pinned to QS-RN-v1 of the committed stream above)."""
    rng = np.random.default_rng(500 + L)
    H, G = 2, 128
    K, V = _stream(rng, H, L + 7)  # the prompt array is longer than the prompt
    ref = _appended_prompt(rng, K, V, L, cap=8)
    pre = oracle.OracleCache(1, H, 128, G, cap=8)
    pre.prefill(K, V, [L])
    cr, cp = ref.counters(0), pre.counters(0)
    assert cp["err"] == 0 and cr["err"] == 0 and cp["half_base"] == 0
    ng = 0 if L <= 2 * G else -(-(L - 2 * G) // G)
    assert cp["n_groups"] == cr["n_groups"] == ng
    assert cp["fill"] == cr["fill"] == L - ng * G and cp["pending"] == cr["pending"] == 0
    if L > 2 * G:
        assert G < cp["fill"] <= 2 * G
    for name in ("kq", "vq", "ks", "kz", "vs", "vz"):
        a, b = getattr(ref, name), getattr(pre, name)
        assert np.array_equal(a[:, :, :ng], b[:, :, :ng]), name
        assert not b[:, :, ng:].any(), name  # groups past n_groups untouched
    for hh in range(H):
        for x, y in zip(ref.buffer_tokens(0, hh), pre.buffer_tokens(0, hh)):
            assert np.array_equal(x, y)
        # slots 0..fill-1 in order (half_base 0)
        assert np.array_equal(pre.bk[0, hh, :cp["fill"]], K[0, hh, ng * G:L].view(np.uint16))


def test_prefill_error_paths_are_flagged_and_no_ops():
    rng = np.random.default_rng(7)
    H, T = 1, 400
    k1, v1 = _stream(rng, H, T)
    K, V = np.concatenate([k1] * 4), np.concatenate([v1] * 4)
    c = oracle.OracleCache(4, H, 128, 128, cap=1)
    # ok (no group) / needs 2 groups with cap 1 / longer than T / negative
    c.prefill(K, V, [200, 400, 401, -1])
    assert c.counters(0) == dict(n_groups=0, fill=200, pending=0, half_base=0, err=0)
    assert c.state[1, oracle.ERR] == oracle.DEV_CAPACITY
    assert c.state[2, oracle.ERR] == oracle.DEV_PREFILL and c.state[3, oracle.ERR] == oracle.DEV_PREFILL
    assert not c.state[1:, :oracle.ERR].any() and not c.bk[1:].any() and not c.kq.any()
    # a second prefill of a non-empty cache changes nothing
    snap = (c.state.copy(), c.bk.copy(), c.bv.copy())
    c.prefill(K, V, [300, 0, 0, 0])
    assert c.state[0, oracle.ERR] == oracle.DEV_PREFILL
    assert np.array_equal(c.state[0, :oracle.ERR], snap[0][0, :oracle.ERR])
    assert np.array_equal(c.bk, snap[1]) and np.array_equal(c.bv, snap[2])
    # cap 1 fits exactly one group: 257..384 tokens
    c2 = oracle.OracleCache(1, H, 128, 128, cap=1)
    c2.prefill(k1, v1, [384])
    assert c2.counters(0)["n_groups"] == 1 and c2.counters(0)["fill"] == 256


# ------------------------------------------------ speculative acceptance

def _spec_inputs(rng, p, q, N):
    """N independent rounds with the same p, q rows: draft tokens drawn from q
    (inverse CDF), acceptance uniforms and Exp(1) variates."""
    g = q.shape[0]
    V = p.shape[1]
    draft = np.empty((N, g), np.int32)
    for i in range(g):
        cdf = np.cumsum(q[i].astype(np.float64))
        draft[:, i] = np.minimum(np.searchsorted(cdf, rng.random(N) * cdf[-1], side="right"), V - 1)
    u = rng.random((N, g)).astype(np.float32)
    e = rng.exponential(size=(N, V)).astype(np.float32)
    P = np.ascontiguousarray(np.broadcast_to(p, (N,) + p.shape))
    Q = np.ascontiguousarray(np.broadcast_to(q, (N,) + q.shape))
    return P, Q, draft, u, e


def _z(count, n, prob):
    return abs(count - n * prob) / np.sqrt(max(n * prob * (1 - prob), 1e-12))


def test_spec_accept_preserves_the_target_distribution():
    """Speculative sampling's defining property, checked by simulation (fixed
    seed, 5-sigma bounds): the first emitted token is distributed as p_0 (the
    draft token when accepted, else the residual draw), the first token is
    accepted with probability sum_x min(p_0, q_0), the token after an accepted
    one is distributed as p_1, and the bonus token after gamma acceptances as
    p_gamma.  A wrong acceptance ratio, a draw from p instead of (p - q)_+, or
    a shifted position all fail it."""
    rng = np.random.default_rng(2024)
    V, g, N = 5, 3, 200000
    p = np.array([[0.40, 0.10, 0.20, 0.05, 0.25],
                  [0.05, 0.50, 0.15, 0.20, 0.10],
                  [0.30, 0.30, 0.10, 0.10, 0.20],
                  [0.10, 0.10, 0.10, 0.60, 0.10]], np.float32)
    q = np.array([[0.10, 0.40, 0.20, 0.25, 0.05],
                  [0.30, 0.20, 0.20, 0.10, 0.20],
                  [0.20, 0.20, 0.20, 0.20, 0.20]], np.float32)
    P, Q, draft, u, e = _spec_inputs(rng, p, q, N)
    na, tok, nd = oracle.spec_accept(P, Q, draft, u, e)
    assert np.array_equal(nd, g - na) and na.min() >= 0 and na.max() <= g
    y0 = np.where(na >= 1, draft[:, 0], tok)
    for x in range(V):
        assert _z((y0 == x).sum(), N, p[0, x]) < 5, ("y0", x)
    acc = float(np.minimum(p[0], q[0]).sum())
    assert _z((na >= 1).sum(), N, acc) < 5
    sel = na >= 1
    y1 = np.where(na[sel] >= 2, draft[sel, 1], tok[sel])
    for x in range(V):
        assert _z((y1 == x).sum(), sel.sum(), p[1, x]) < 5, ("y1", x)
    allacc = na == g
    assert allacc.sum() > 1000
    for x in range(V):
        assert _z((tok[allacc] == x).sum(), allacc.sum(), p[g, x]) < 5, ("bonus", x)


def test_spec_accept_special_cases():
    V, g = 6, 4
    rng = np.random.default_rng(3)
    p = rng.dirichlet(np.ones(V), g + 1).astype(np.float32)
    q = p[:g].copy()
    draft = np.array([[1, 2, 3, 4]], np.int32)
    u = np.full((1, g), 0.999, np.float32)
    e = np.array([[3.0, 0.5, 2.0, 1.0, 0.25, 4.0]], np.float32)
    # q == p: every draft token is accepted; the bonus comes from p_gamma
    na, tok, nd = oracle.spec_accept(p[None], q[None], draft, u, e)
    assert na[0] == g and nd[0] == 0
    assert tok[0] == int(np.argmin(e[0] / p[g]))
    # a draft token the target gives probability 0 is rejected there, and the
    # draw excludes every token where p <= q
    p2 = p.copy()
    p2[2, 0] += p2[2, 3]  # the mass of token 3 moves to token 0
    p2[2, 3] = 0.0
    na, tok, nd = oracle.spec_accept(p2[None], q[None], draft, u, e)
    assert na[0] == 2 and nd[0] == 2
    assert tok[0] == 0  # the only token with p > q at position 2
    # a draft token outside [0, V) is rejected
    na, _, _ = oracle.spec_accept(p[None], q[None], np.array([[1, 2, V, 4]], np.int32), u, e)
    assert na[0] == 2
    # all-zero weights: token -1
    z = np.zeros((1, g + 1, V), np.float32)
    na, tok, nd = oracle.spec_accept(z, np.zeros((1, g, V), np.float32), draft, u, e)
    assert na[0] == 0 and tok[0] == -1 and nd[0] == g


# ------------------------------------------------ grouped-query attention

@pytest.mark.parametrize("group,n_q", [(1, 5), (4, 1), (4, 5), (3, 8)])
def test_grouped_query_attention_equals_replicated_heads(group, n_q):
    """Query head h*g + i of grouped-query attention attends KV head h: the
    result equals multi-head attention on a cache whose KV heads are each
    repeated g times (same fp64 arithmetic, so bit for bit), in both modes."""
    rng = np.random.default_rng(40 + group * 10 + n_q)
    B, H, T = 2, 2, 700
    k = h(rng.standard_normal((B, H, T, 128)) * 2)
    v = h(rng.standard_normal((B, H, T, 128)))
    oc = oracle.OracleCache(B, H, 128, 128, cap=4)
    oc.prefill(k, v, [T, 300])
    rep = oracle.OracleCache(B, H * group, 128, 128, cap=4)
    for name in ("kq", "vq", "ks", "kz", "vs", "vz", "bk", "bv"):
        setattr(rep, name, np.ascontiguousarray(np.repeat(getattr(oc, name), group, axis=1)))
    rep.state = oc.state.copy()
    q = h(rng.standard_normal((B, H * group, n_q, 128)))
    for upper in (True, False):
        o1, l1 = oc.attn(q, upper, group=group)
        o2, l2 = rep.attn(q, upper)
        assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    # and the rows differ across the query heads of one KV head
    assert not np.array_equal(o1[:, 0], o1[:, group - 1]) or group == 1
