"""GPU parity: libqs (through the C ABI) against the CPU oracle.

Bit-exact: codes (as packed planes), scales, zeros, buffer contents, counters
and error words.  Attention outputs: max-abs <= 1e-2 and relative RMS <=
2e-3 against the oracle's fp64 result on the same seeded inputs; the
log-sum-exp within 5e-3 (bounded by the fp16 rounding of q * s_K, about
2^-11 of sum_d |q_d k_d| * softmax_scale, far below this on these inputs).
"""
import os

import numpy as np
import pytest

import oracle
from hierarchical_quantized_kv_gb300 import driver, qs, synthetic
from tests import layout

pytestmark = pytest.mark.gpu

ATOL, RRMS, LSE_TOL = 1e-2, 2e-3, 5e-3
DRAFT, VERIFY = qs.QS_DRAFT_UPPER4, qs.QS_VERIFY_INT8


@pytest.fixture(scope="module")
def torch():
    import torch as t
    assert t.cuda.is_available(), "GPU tests need CUDA"
    import __graft_entry__
    __graft_entry__.build()
    return t


def h16(rng, shape, scale=1.0):
    return (rng.standard_normal(shape) * scale).astype(np.float16)


def to_dev(torch, a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def assert_state_equal(cache, oc, what=""):
    got = layout.read_device(cache)
    want = layout.device_arrays(oc, cache.upper_bits)
    for name in want:
        g, w_ = got[name], want[name]
        if name == "state":
            w_ = w_.copy()
            w_[:, oracle.ERR] = g[:, oracle.ERR]  # error words are compared separately
        assert np.array_equal(g.reshape(w_.shape), w_), "%s: %s differs" % (what, name)


def run_attn(torch, cache, mode, q, scale=None, lse=True):
    B, H, n_q, D = q.shape
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    qd = to_dev(torch, q)
    out = torch.full_like(qd, float("nan"))
    l_ = torch.full((B, H, n_q), float("nan"), dtype=torch.float32, device="cuda") if lse else None
    ws = torch.empty(qs.qs_attn_workspace_size(cache, n_q), dtype=torch.uint8, device="cuda")
    qs.qs_attn_decode(cache, mode, qd, scale, out, l_, ws)
    torch.cuda.synchronize()
    assert int(cache.arrive.abs().sum().item()) == 0, "segment counters not back at zero"
    return out.double().cpu().numpy(), (l_.double().cpu().numpy() if lse else None)


def assert_close(got, ref, got_lse=None, ref_lse=None, what=""):
    assert np.all(np.isfinite(got)), what
    err = np.abs(got - ref).max()
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
    log = os.environ.get("QS_PARITY_LOG")
    if log:
        with open(log, "a") as f:
            f.write("%s\t%s\tmax_abs=%.3g\trel_rms=%.3g\n"
                    % (os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0], what, err, rel))
    assert err <= ATOL and rel <= RRMS, "%s: max-abs %.3g rel-rms %.3g" % (what, err, rel)
    if got_lse is not None:
        fin = np.isfinite(ref_lse)
        assert np.array_equal(np.isfinite(got_lse), fin), what
        assert np.abs(got_lse[fin] - ref_lse[fin]).max() <= LSE_TOL, what
    return err, rel


# ---------------------------------------------------------- bookkeeping

@pytest.mark.parametrize("seed", [0, 1])
def test_buffer_and_flush_bit_exact(torch, seed):
    """Random append / rollback / flush sequences, including failing
    preconditions, give bit-identical device and oracle state."""
    rng = np.random.default_rng(seed)
    B, H, cap = 3, 4, 5
    cache = qs.Cache(B, H, cap)
    oc = oracle.OracleCache(B, H, 128, 128, cap)
    qs.qs_state_reset(cache)
    mask_d = torch.zeros(B, dtype=torch.uint8, device="cuda")
    for step in range(260):
        op = rng.random()
        if op < 0.06:   # a flush with a random mask, may fail per sequence
            m = rng.integers(0, 2, B).astype(np.uint8)
            qs.qs_quantize_flush(cache, to_dev(torch, m))
            oc.flush(m)
        elif op < 0.08:  # rollback that may exceed the pending tokens
            r = rng.integers(0, 8, B).astype(np.int32)
            qs.qs_buffer_rollback(cache, to_dev(torch, r))
            oc.rollback(r)
        else:
            qs.qs_need_flush(cache, 6, mask_d)
            m = oc.need_flush(6)
            assert np.array_equal(mask_d.cpu().numpy(), m)
            qs.qs_quantize_flush(cache, mask_d)
            oc.flush(m)
            n = int(rng.integers(1, 7))
            k, v = h16(rng, (B, H, n, 128), 3.0), h16(rng, (B, H, n, 128))
            qs.qs_buffer_append(cache, to_dev(torch, k), to_dev(torch, v))
            oc.append(k, v)
            r = np.array([rng.integers(0, n + 1) for _ in range(B)], np.int32)
            qs.qs_buffer_rollback(cache, to_dev(torch, r))
            oc.rollback(r)
        if step % 20 == 0 or step == 259:
            assert_state_equal(cache, oc, "step %d" % step)
            errs = qs.qs_get_errors(cache)
            assert np.array_equal(errs, oc.state[:, oracle.ERR]), step
            oc.state[:, oracle.ERR] = 0
    assert oc.state[:, oracle.N_GROUPS].sum() >= 4


def _degenerate_line(p, n, rng, extreme):
    """n fp16 values of pattern p: the groups QS-RN-v1 treats specially
    (constant, signed zeros, two-valued, a range that gives a subnormal
    scale, fp16 subnormal inputs, exact ties, the fp16 extremes, a single
    outlier) and a few plain ones."""
    E = 65504.0 if extreme else 3.0       # moderate: value rows stay O(1), so the
    C = 60000.0 if extreme else 10.0      # fp16 rounding of p * s_V stays far inside 1e-2
    W = 1e3 if extreme else 3.0
    x = np.zeros(n)
    if p == 0:
        x[:] = 1.5
    elif p == 1:
        x[:] = 0.0
    elif p == 2:
        x[:] = -0.0
    elif p == 3:
        x[:] = np.where(np.arange(n) % 2 == 0, 0.0, -0.0)
    elif p == 4:
        x[:] = np.where(np.arange(n) % 2 == 0, -3.0, 7.0)
    elif p == 5:
        x[:] = np.where(np.arange(n) % 2 == 0, 1.0, 1.0 + 2.0 ** -10)
    elif p == 6:
        x[:] = rng.uniform(-E, E, n)
        x[0], x[1] = -E, E
    elif p == 7:
        x[:] = rng.integers(-100, 101, n) * 2.0 ** -24
    elif p == 8:   # s = 2^-6 exactly, every other code an exact tie
        x[:] = (rng.integers(0, 255, n) + 0.5) * 2.0 ** -6
        x[0], x[1] = 0.0, 255 * 2.0 ** -6
    elif p == 9:
        x[:] = C
        x[5] = -C
    elif p == 10:
        x[17 % n] = 2.5
    elif p == 11:
        x[:] = rng.standard_normal(n) * 1e-3
    elif p == 12:
        x[:] = rng.standard_normal(n) * W
    elif p == 13:
        x[:] = rng.standard_normal(n) + 100.0
    elif p == 14:
        x[:] = rng.integers(0, 256, n) * 0.125
        x[0], x[1] = 0.0, 255 * 0.125
    else:
        x[:] = rng.standard_normal(n)
    return x.astype(np.float16)


def _degenerate_tokens(rng, H, extreme):
    """[1, H, 128, 128] keys and values whose groups are the degenerate
    patterns: key channel d follows pattern d mod 16 over the 128 tokens,
    value token t follows pattern t mod 16 over the 128 channels; head 1
    negates head 0 (+0 becomes -0)."""
    k = np.zeros((1, H, 128, 128), np.float16)
    v = np.zeros_like(k)
    for d in range(128):
        k[0, 0, :, d] = _degenerate_line(d % 16, 128, rng, extreme)
    for t in range(128):
        v[0, 0, t, :] = _degenerate_line(t % 16, 128, rng, extreme)
    for hh in range(1, H):
        k[0, hh], v[0, hh] = -k[0, 0], -v[0, 0]
    return k, v


@pytest.mark.parametrize("extreme", [False, True])
@pytest.mark.parametrize("ub", [4, 2])
def test_degenerate_groups_bit_exact(torch, extreme, ub):
    """Groups QS-RN-v1 treats specially, quantized by the flush (16-warp
    CTAs) and by the prefill (8-warp CTAs): planes, scales and zeros bit for
    bit against the oracle in both plane layouts; then attention over them
    with moderate ranges.  With the fp16 extremes only the bytes are
    compared: the value path rounds p * s_V to fp16, an absolute error that
    grows with the value range, while the attention tolerance is absolute."""
    rng = np.random.default_rng(41 + extreme)
    H = 2
    kd, vd = _degenerate_tokens(rng, H, extreme)
    knew, vnew = h16(rng, (1, H, 256, 128), 2.0), h16(rng, (1, H, 256, 128))
    k = np.concatenate([kd, knew], axis=2)
    v = np.concatenate([vd, vnew], axis=2)
    # flush path: the 128 degenerate tokens are the oldest half
    cache = qs.Cache(1, H, 2, upper_bits=ub)
    qs.qs_state_reset(cache)
    oc = oracle.OracleCache(1, H, 128, 128, 2)
    qs.qs_buffer_append(cache, to_dev(torch, k[:, :, :256]), to_dev(torch, v[:, :, :256]))
    oc.append(k[:, :, :256], v[:, :, :256])
    zero = to_dev(torch, np.zeros(1, np.int32))
    qs.qs_buffer_rollback(cache, zero)
    oc.rollback([0])
    qs.qs_quantize_flush(cache, None)
    oc.flush()
    torch.cuda.synchronize()
    assert oc.counters(0)["n_groups"] == 1
    assert_state_equal(cache, oc, "flush of degenerate groups")
    # the patterns do reach the special cases: zero scales and subnormal scales
    ks = oc.ks[0, 0, 0].view(np.float16).astype(np.float64)
    assert np.any(ks == 0) and np.any((ks > 0) & (ks < 2.0 ** -14))
    # prefill path: 384 prompt tokens, group 0 is the degenerate half
    pc = qs.Cache(1, H, 2, upper_bits=ub)
    qs.qs_state_reset(pc)
    op = oracle.OracleCache(1, H, 128, 128, 2)
    lens = np.array([384], np.int32)
    qs.qs_prefill(pc, to_dev(torch, k), to_dev(torch, v), to_dev(torch, lens))
    op.prefill(k, v, lens)
    torch.cuda.synchronize()
    assert op.counters(0)["n_groups"] == 1
    assert_state_equal(pc, op, "prefill of degenerate groups")
    assert np.all(qs.qs_get_errors(cache) == 0) and np.all(qs.qs_get_errors(pc) == 0)
    assert not oc.state[:, oracle.ERR].any() and not op.state[:, oracle.ERR].any()
    if extreme:
        return
    for mode, n_q in ((DRAFT, 1), (VERIFY, 5)):
        q = h16(rng, (1, H, n_q, 128))
        got, gl = run_attn(torch, cache, mode, q)
        ref, rl = oc.attn(q, upper_only=(mode == DRAFT), upper_bits=ub)
        assert_close(got, ref, gl, rl, "degenerate groups, mode %d" % mode)


def test_append_overflow_is_a_no_op(torch):
    rng = np.random.default_rng(5)
    cache = qs.Cache(2, 2, 2)
    oc = oracle.OracleCache(2, 2, 128, 128, 2)
    qs.qs_state_reset(cache)
    k, v = h16(rng, (2, 2, 200, 128)), h16(rng, (2, 2, 200, 128))
    for c in (cache,):
        qs.qs_buffer_append(c, to_dev(torch, k), to_dev(torch, v))
    oc.append(k, v)
    qs.qs_buffer_append(cache, to_dev(torch, k[:, :, :57]), to_dev(torch, v[:, :, :57]))
    oc.append(k[:, :, :57], v[:, :, :57])
    assert_state_equal(cache, oc)
    assert np.all(qs.qs_get_errors(cache) == qs.DEV_OVERFLOW)
    assert np.all(qs.qs_get_errors(cache) == 0)  # read-back clears


def test_corrupted_counters_written_from_the_host(torch):
    """Host-side fault injection: counters past every limit (negative, past
    the capacity, past the ring, an odd half base) written straight into the
    state.  Every call stays in bounds (device counters are validated or
    clamped before they index anything): no CUDA error, each sequence's
    error word flags it, attention outputs are finite, the segment counters
    end at zero, and after qs_state_reset a normal round works again."""
    rng = np.random.default_rng(91)
    B, H, cap = 4, 2, 3
    cache = qs.Cache(B, H, cap)
    qs.qs_state_reset(cache)
    bad = np.zeros((B, qs.STATE_WORDS), np.int32)
    bad[:, :4] = [[-5, 300, -2, 7], [99, -1, 5, 1], [2, 1000, 1000, 0], [1 << 30, 128, -3, 3]]
    cache.state.copy_(torch.from_numpy(bad))
    mask = torch.zeros(B, dtype=torch.uint8, device="cuda")
    qs.qs_need_flush(cache, 1, mask)
    qs.qs_quantize_flush(cache, mask)
    k1, v1 = h16(rng, (B, H, 1, 128)), h16(rng, (B, H, 1, 128))
    qs.qs_buffer_append(cache, to_dev(torch, k1), to_dev(torch, v1))
    qs.qs_buffer_rollback(cache, to_dev(torch, np.zeros(B, np.int32)))
    q = h16(rng, (B, H, 1, 128))
    for mode in (DRAFT, VERIFY):
        got, gl = run_attn(torch, cache, mode, q)  # also checks the segment counters
        assert np.all(np.isfinite(got))
    errs = qs.qs_get_errors(cache)
    assert np.all(errs != 0), errs
    assert errs[0] & qs.DEV_OVERFLOW and errs[1] & qs.DEV_NQ_GT_FILL
    assert errs[2] & qs.DEV_FLUSH_UNCOMMITTED and errs[3] & qs.DEV_OVER_ROLLBACK
    # recovery: an emptied cache runs a normal append + attention
    qs.qs_state_reset(cache)
    oc = oracle.OracleCache(B, H, 128, 128, cap)
    k, v = h16(rng, (B, H, 40, 128)), h16(rng, (B, H, 40, 128))
    qs.qs_buffer_append(cache, to_dev(torch, k), to_dev(torch, v))
    oc.append(k, v)
    got, gl = run_attn(torch, cache, VERIFY, q)
    ref, rl = oc.attn(q, upper_only=False)
    assert_close(got, ref, gl, rl, "after reset")
    assert np.all(qs.qs_get_errors(cache) == 0)


def test_host_argument_errors(torch):
    cache = qs.Cache(1, 1, 1)
    with pytest.raises(qs.QsError) as e:
        qs.qs_buffer_append(cache, torch.zeros((1, 1, 0, 128), dtype=torch.float16, device="cuda"),
                            torch.zeros((1, 1, 0, 128), dtype=torch.float16, device="cuda"))
    assert e.value.status == qs.QS_ERR_ARG
    q = torch.zeros((1, 1, 9, 128), dtype=torch.float16, device="cuda")
    with pytest.raises(qs.QsError) as e:
        qs.qs_attn_decode(cache, DRAFT, q, 0.1, torch.empty_like(q), None, None)
    assert e.value.status == qs.QS_ERR_ARG
    q = q[:, :, :2].contiguous()
    with pytest.raises(qs.QsError) as e:
        qs.qs_attn_decode(cache, DRAFT, q, 0.1, torch.empty_like(q), None, None)
    assert e.value.status == qs.QS_ERR_WORKSPACE


# ----------------------------------------------------------- tiny config

def test_tiny_config_round(torch):
    """The tiny workload: 768 quantized + 256 buffer tokens, 4 outlier key
    channels x10.  Draft 1 query, verify 5 queries, flush one half, then a
    5-token round that rolls back 3 rejected tokens; state bit-exact and
    outputs within tolerance at every step."""
    w = synthetic.tiny()
    cache = qs.Cache(w.B, w.H, 8)
    driver.prefill(cache, w)
    oc = oracle.OracleCache(w.B, w.H, w.D, w.G, 8)
    oracle.prefill(oc, lambda b, t0, n: synthetic.kv_tokens(w, b, t0, n), w.n_groups, w.fill)
    assert_state_equal(cache, oc, "prefill")
    assert oc.counters(0)["n_groups"] == 6 and oc.counters(0)["fill"] == 256

    def both(mode, q, what):
        got, gl = run_attn(torch, cache, mode, q)
        ref, rl = oc.attn(q, upper_only=(mode == DRAFT))
        assert_close(got, ref, gl, rl, what)

    both(DRAFT, synthetic.queries(w, 0, 1), "draft")
    both(VERIFY, synthetic.queries(w, 1, 5), "verify")
    qs.qs_quantize_flush(cache)
    oc.flush()
    assert_state_equal(cache, oc, "flush")
    k, v = synthetic.kv_tokens(w, 0, 1024, 5)
    qs.qs_buffer_append(cache, to_dev(torch, k[None]), to_dev(torch, v[None]))
    oc.append(k[None], v[None])
    both(VERIFY, synthetic.queries(w, 2, 5), "verify after flush")
    both(DRAFT, synthetic.queries(w, 3, 1), "draft with pending")
    qs.qs_buffer_rollback(cache, to_dev(torch, np.array([3], np.int32)))
    oc.rollback([3])
    assert_state_equal(cache, oc, "rollback")
    both(DRAFT, synthetic.queries(w, 4, 1), "draft after rollback")
    both(VERIFY, synthetic.queries(w, 5, 2), "verify after rollback")
    assert np.all(qs.qs_get_errors(cache) == 0)


# ------------------------------------------- injected state, edge cases

def _oracle_state(rng, B, H, n_groups, fill, cap, k_scale=2.0):
    oc = oracle.OracleCache(B, H, 128, 128, cap)
    toks = {}

    def tokens(b, t0, n):
        key = (b, t0, n)
        if key not in toks:
            r = np.random.default_rng([int(rng.integers(1 << 30)), b, t0])
            k = (r.standard_normal((H, n, 128)) * k_scale)
            k[:, :, :3] *= 8
            toks[key] = (k.astype(np.float16), r.standard_normal((H, n, 128)).astype(np.float16))
        return toks[key]

    oracle.prefill(oc, tokens, n_groups, fill)
    return oc


@pytest.mark.parametrize("n_groups,fill", [(0, 1), (0, 8), (0, 31), (1, 32), (1, 33), (2, 64),
                                           (3, 65), (0, 127), (2, 128), (1, 200), (5, 255),
                                           (4, 256)])
@pytest.mark.parametrize("n_q", [1, 2, 5, 8])
def test_attn_edge_cases(torch, n_groups, fill, n_q):
    if n_q > fill:
        pytest.skip("n_q > fill is the error case")
    rng = np.random.default_rng(1000 * n_groups + fill + 7 * n_q)
    B, H = 2, 3
    oc = _oracle_state(rng, B, H, [n_groups, n_groups], [fill, fill], cap=max(n_groups, 1))
    cache = qs.Cache(B, H, max(n_groups, 1))
    layout.load_into(cache, oc)
    q = h16(rng, (B, H, n_q, 128))
    for mode in (DRAFT, VERIFY):
        got, gl = run_attn(torch, cache, mode, q)
        ref, rl = oc.attn(q, upper_only=(mode == DRAFT))
        assert_close(got, ref, gl, rl, "mode %d" % mode)


def test_attn_ragged_small(torch):
    rng = np.random.default_rng(77)
    ng = [0, 5, 1, 3, 0, 2, 7]
    fl = [3, 256, 1, 129, 64, 33, 200]
    B, H = len(ng), 3
    oc = _oracle_state(rng, B, H, ng, fl, cap=8)
    cache = qs.Cache(B, H, 8)
    layout.load_into(cache, oc)
    for n_q in (1, 3):
        q = h16(rng, (B, H, n_q, 128))
        for mode in (DRAFT, VERIFY):
            got, gl = run_attn(torch, cache, mode, q)
            ref, rl = oc.attn(q, upper_only=(mode == DRAFT))
            assert_close(got, ref, gl, rl, "n_q %d mode %d" % (n_q, mode))
        # sequences with fill < n_q are flagged on both sides
        assert np.array_equal(qs.qs_get_errors(cache), oc.state[:, oracle.ERR])
        oc.state[:, oracle.ERR] = 0


@pytest.mark.parametrize("H,n_groups,fill", [(1, 100, 70), (2, 300, 129), (8, 130, 5),
                                              (40, 30, 250)])
def test_attn_split_spans(torch, H, n_groups, fill):
    """Segments split over few and over many CTAs (fewer units than CTAs;
    about 76, 19 and 4 CTAs per segment), with 1, 2 and 5 query rows: both
    ways of finishing a split segment (from every warp's partial, or from
    one partial per CTA), each call twice (the segment counters must be back
    at zero for the next call)."""
    rng = np.random.default_rng(H * 1000 + n_groups)
    B = 1
    oc = _oracle_state(rng, B, H, [n_groups], [fill], cap=n_groups)
    cache = qs.Cache(B, H, n_groups)
    layout.load_into(cache, oc)
    for n_q in (1, 2, 5):
        q = h16(rng, (B, H, n_q, 128))
        for mode in (DRAFT, VERIFY):
            ref, rl = oc.attn(q, upper_only=(mode == DRAFT))
            for rep in range(2):
                got, gl = run_attn(torch, cache, mode, q)
                assert_close(got, ref, gl, rl, "n_q %d mode %d call %d" % (n_q, mode, rep))


@pytest.mark.parametrize("B,H,n_groups,fill", [(1, 32, 40, 253), (3, 8, 60, 252)])
def test_chained_round_no_host_sync(torch, B, H, n_groups, fill):
    """A speculative round launched back to back on one stream, as a serving
    loop runs it (flush mask, flush, then append + draft four times,
    rollback, append five, verify), with no host synchronization in between:
    kernels overlap through programmatic dependent launch, and attention
    starts copying quantized groups before its grid dependency wait.  Every
    output equals the oracle's for the state at its point in the round."""
    rng = np.random.default_rng(B * 100 + H)
    oc = _oracle_state(rng, B, H, [n_groups] * B, [fill] * B, cap=n_groups + 2)
    cache = qs.Cache(B, H, n_groups + 2)
    layout.load_into(cache, oc)
    g = 4
    kd = [h16(rng, (B, H, 1, 128), 2.0) for _ in range(g)]
    vd = [h16(rng, (B, H, 1, 128)) for _ in range(g)]
    qd = [h16(rng, (B, H, 1, 128)) for _ in range(g)]
    kt, vt = h16(rng, (B, H, g + 1, 128), 2.0), h16(rng, (B, H, g + 1, 128))
    qv = h16(rng, (B, H, g + 1, 128))
    drop = np.full(B, g, np.int32)
    dev = [to_dev(torch, a) for a in kd + vd + qd + [kt, vt, qv, drop]]
    kdd, vdd, qdd = dev[:g], dev[g:2 * g], dev[2 * g:3 * g]
    ktd, vtd, qvd, dropd = dev[3 * g:]
    outs = [torch.full_like(q, float("nan")) for q in qdd]
    outv = torch.full_like(qvd, float("nan"))
    lse = torch.full((B, H, g + 1), float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.empty(qs.qs_attn_workspace_size(cache, g + 1), dtype=torch.uint8, device="cuda")
    mask = torch.zeros(B, dtype=torch.uint8, device="cuda")
    scale = 1.0 / np.sqrt(128)
    torch.cuda.synchronize()
    qs.qs_need_flush(cache, g + 1, mask)
    qs.qs_quantize_flush(cache, mask)
    for i in range(g):
        qs.qs_buffer_append(cache, kdd[i], vdd[i])
        qs.qs_attn_decode(cache, DRAFT, qdd[i], scale, outs[i], None, ws)
    qs.qs_buffer_rollback(cache, dropd)
    qs.qs_buffer_append(cache, ktd, vtd)
    qs.qs_attn_decode(cache, VERIFY, qvd, scale, outv, lse, ws)
    torch.cuda.synchronize()

    m = oc.need_flush(g + 1)
    assert m.all() and np.array_equal(mask.cpu().numpy(), m)  # fill + 5 > 256: a flush
    oc.flush(m)
    for i in range(g):
        oc.append(kd[i], vd[i])
        ref, _ = oc.attn(qd[i], upper_only=True)
        assert_close(outs[i].double().cpu().numpy(), ref, what="draft %d" % i)
    oc.rollback(drop)
    oc.append(kt, vt)
    ref, rl = oc.attn(qv, upper_only=False)
    assert_close(outv.double().cpu().numpy(), ref, lse.double().cpu().numpy(), rl, "verify")
    assert np.array_equal(cache.state.cpu().numpy()[:, :4], oc.state[:, :4])
    assert int(cache.arrive.abs().sum().item()) == 0
    assert np.all(qs.qs_get_errors(cache) == 0)


@pytest.mark.parametrize("mode", [DRAFT, VERIFY])
def test_peaked_attention(torch, mode):
    """One key far above the rest (a large score on a quantized token): the
    softmax is dominated by it, so the score's own rounding shows directly
    in the output."""
    rng = np.random.default_rng(21)
    B, H, ng, fill = 1, 2, 6, 40
    oc = oracle.OracleCache(B, H, 128, 128, ng)
    q = h16(rng, (B, H, 2, 128))

    def tokens(b, t0, n):
        k = rng.standard_normal((H, n, 128))
        k[:, :, :3] *= 8
        if t0 <= 300 < t0 + n:  # token 300: aligned with the queries
            k[:, 300 - t0] = 2.5 * q[0, :, 0].astype(np.float64)
        return k.astype(np.float16), rng.standard_normal((H, n, 128)).astype(np.float16)

    oracle.prefill(oc, tokens, [ng], [fill])
    cache = qs.Cache(B, H, ng)
    layout.load_into(cache, oc)
    got, gl = run_attn(torch, cache, mode, q)
    ref, rl = oc.attn(q, upper_only=(mode == DRAFT))
    assert_close(got, ref, gl, rl, "peaked mode %d" % mode)


def test_attn_nq_greater_than_fill(torch):
    rng = np.random.default_rng(3)
    oc = _oracle_state(rng, 3, 2, [2, 0, 1], [4, 2, 40], cap=2)
    cache = qs.Cache(3, 2, 2)
    layout.load_into(cache, oc)
    q = h16(rng, (3, 2, 3, 128))
    got, gl = run_attn(torch, cache, VERIFY, q)
    ref, rl = oc.attn(q, upper_only=False)
    assert np.all(got[1] == 0) and np.all(np.isneginf(gl[1]))
    assert_close(got, ref, gl, rl)
    errs = qs.qs_get_errors(cache)
    assert errs.tolist() == [0, qs.DEV_NQ_GT_FILL, 0]


def test_draft_equals_verify_when_lower_is_eight(torch):
    """Crafted codes with every C_L = 8: draft and verify must agree (the
    oracle pins this exactly; on the device both take the same inputs to
    the same kernels up to the code extraction)."""
    rng = np.random.default_rng(9)
    oc = _oracle_state(rng, 1, 2, [3], [20], cap=3)
    oc.kq[:] = (oc.kq & 0xF0) | 8
    oc.vq[:] = (oc.vq & 0xF0) | 8
    cache = qs.Cache(1, 2, 3)
    layout.load_into(cache, oc)
    q = h16(rng, (1, 2, 4, 128))
    gd, _ = run_attn(torch, cache, DRAFT, q)
    gv, _ = run_attn(torch, cache, VERIFY, q)
    ref, _ = oc.attn(q, upper_only=False)
    assert_close(gd, ref)
    assert_close(gv, ref)
    assert np.abs(gd - gv).max() < 2e-3


# ------------------------------------------------------------- bulk prefill

def _prompt(rng, B, H, T):
    return h16(rng, (B, H, T, 128), 2.0), h16(rng, (B, H, T, 128))


def test_prefill_bit_exact_then_decode(torch):
    """qs_prefill against the oracle's prefill (itself pinned to the append /
    flush path): every array bit for bit for prompt lengths around the group
    and buffer boundaries; then attention, a flush and an append on top."""
    rng = np.random.default_rng(31)
    B, H, T, cap = 6, 2, 700, 5
    lens = np.array([0, 1, 256, 257, 385, 700], np.int32)
    k, v = _prompt(rng, B, H, T)
    cache = qs.Cache(B, H, cap)
    qs.qs_prefill(cache, to_dev(torch, k), to_dev(torch, v), to_dev(torch, lens))
    oc = oracle.OracleCache(B, H, 128, 128, cap)
    oc.prefill(k, v, lens)
    assert_state_equal(cache, oc, "prefill")
    assert np.all(qs.qs_get_errors(cache) == 0) and np.all(oc.state[:, oracle.ERR] == 0)
    for mode, n_q in ((DRAFT, 1), (VERIFY, 5)):
        q = h16(rng, (B, H, n_q, 128))
        got, gl = run_attn(torch, cache, mode, q)
        ref, rl = oc.attn(q, upper_only=(mode == DRAFT))
        assert_close(got, ref, gl, rl, "after prefill, mode %d" % mode)
    assert np.array_equal(qs.qs_get_errors(cache), oc.state[:, oracle.ERR])
    oc.state[:, oracle.ERR] = 0
    mask = torch.zeros(B, dtype=torch.uint8, device="cuda")
    qs.qs_need_flush(cache, 5, mask)
    qs.qs_quantize_flush(cache, mask)
    oc.flush(oc.need_flush(5))
    k5, v5 = _prompt(rng, B, H, 5)
    qs.qs_buffer_append(cache, to_dev(torch, k5), to_dev(torch, v5))
    oc.append(k5, v5)
    assert_state_equal(cache, oc, "flush + append after prefill")
    assert np.all(qs.qs_get_errors(cache) == 0)


def test_two_bit_draft_layout(torch):
    """upper_bits = 2 (a draft from the top two bits of each code): prefill
    and flush write the C_U2 / M2 planes bit for bit; draft (one query and
    three) and verify attention match the oracle, before and after a flush
    and an append; the same cache read with the 4-bit draft differs."""
    rng = np.random.default_rng(37)
    B, H, T, cap = 3, 2, 700, 6
    lens = np.array([300, 129, 700], np.int32)
    k, v = _prompt(rng, B, H, T)
    cache = qs.Cache(B, H, cap, upper_bits=2)
    qs.qs_prefill(cache, to_dev(torch, k), to_dev(torch, v), to_dev(torch, lens))
    oc = oracle.OracleCache(B, H, 128, 128, cap)
    oc.prefill(k, v, lens)
    assert_state_equal(cache, oc, "two-bit prefill")

    def both(what):
        for mode, n_q in ((DRAFT, 1), (DRAFT, 3), (VERIFY, 5)):
            q = h16(rng, (B, H, n_q, 128))
            got, gl = run_attn(torch, cache, mode, q)
            ref, rl = oc.attn(q, upper_only=(mode == DRAFT), upper_bits=2)
            assert_close(got, ref, gl, rl, "%s, mode %d, n_q %d" % (what, mode, n_q))
            if mode == DRAFT:
                ref4, _ = oc.attn(q, upper_only=True, upper_bits=4)
                assert np.abs(got - ref4).max() > 10 * ATOL
    both("after prefill")
    mask = torch.zeros(B, dtype=torch.uint8, device="cuda")
    qs.qs_need_flush(cache, 130, mask)
    qs.qs_quantize_flush(cache, mask)
    oc.flush(oc.need_flush(130))
    k5, v5 = _prompt(rng, B, H, 5)
    qs.qs_buffer_append(cache, to_dev(torch, k5), to_dev(torch, v5))
    oc.append(k5, v5)
    assert_state_equal(cache, oc, "two-bit flush + append")
    both("after flush")
    assert np.all(qs.qs_get_errors(cache) == 0)


@pytest.mark.parametrize("n_groups,fill,n_q", [(0, 8, 1), (1, 33, 5), (2, 128, 2), (5, 255, 8),
                                               (3, 65, 1)])
def test_two_bit_attn_edge_cases(torch, n_groups, fill, n_q):
    rng = np.random.default_rng(500 + 10 * n_groups + n_q)
    B, H = 2, 3
    oc = _oracle_state(rng, B, H, [n_groups, n_groups], [fill, fill], cap=max(n_groups, 1))
    cache = qs.Cache(B, H, max(n_groups, 1), upper_bits=2)
    layout.load_into(cache, oc)
    q = h16(rng, (B, H, n_q, 128))
    for mode in (DRAFT, VERIFY):
        got, gl = run_attn(torch, cache, mode, q)
        ref, rl = oc.attn(q, upper_only=(mode == DRAFT), upper_bits=2)
        assert_close(got, ref, gl, rl, "mode %d" % mode)


def test_prefill_error_paths(torch):
    rng = np.random.default_rng(7)
    H, T = 1, 400
    k, v = _prompt(rng, 4, H, T)
    cache = qs.Cache(4, H, 1)
    oc = oracle.OracleCache(4, H, 128, 128, 1)
    lens = np.array([200, 400, 401, -1], np.int32)  # ok / needs 2 groups / > T / < 0
    qs.qs_prefill(cache, to_dev(torch, k), to_dev(torch, v), to_dev(torch, lens))
    oc.prefill(k, v, lens)
    assert_state_equal(cache, oc, "errors")
    errs = qs.qs_get_errors(cache)
    assert np.array_equal(errs, oc.state[:, oracle.ERR])
    assert list(errs) == [0, qs.DEV_CAPACITY, qs.DEV_PREFILL, qs.DEV_PREFILL]
    oc.state[:, oracle.ERR] = 0
    lens2 = np.array([300, 0, 0, 0], np.int32)  # sequence 0 is no longer empty
    qs.qs_prefill(cache, to_dev(torch, k), to_dev(torch, v), to_dev(torch, lens2))
    oc.prefill(k, v, lens2)
    assert_state_equal(cache, oc, "non-empty")
    assert list(qs.qs_get_errors(cache)) == [qs.DEV_PREFILL, 0, 0, 0]
    with pytest.raises(qs.QsError) as e:
        qs.qs_prefill(cache, to_dev(torch, k[:, :, :0]), to_dev(torch, v[:, :, :0]), None)
    assert e.value.status == qs.QS_ERR_ARG


def test_prefill_full_size_32k(torch):
    """The 32k workload's whole prompt in one call (254 groups + 256 buffer
    tokens per head, 32 heads) equals the oracle bit for bit, and equals the
    state the append / flush path builds (logical content)."""
    w = synthetic.llama_32k()
    T = w.context[0]
    k, v = synthetic.kv_tokens(w, 0, 0, T)
    cap = w.n_groups[0] + 1
    cache = qs.Cache(1, w.H, cap)
    qs.qs_prefill(cache, to_dev(torch, k[None]), to_dev(torch, v[None]),
                  to_dev(torch, np.array([T], np.int32)))
    oc = oracle.OracleCache(1, w.H, w.D, w.G, cap)
    oc.prefill(k[None], v[None], [T])
    assert oc.counters(0)["n_groups"] == w.n_groups[0] and oc.counters(0)["fill"] == w.fill[0]
    assert_state_equal(cache, oc, "32k prefill")
    ref = qs.Cache(1, w.H, cap)
    driver.prefill(ref, w)
    a, b = layout.read_device(cache), layout.read_device(ref)
    for name in ("k_upper", "k_lower", "v_upper", "v_lower", "meta"):
        assert np.array_equal(a[name], b[name]), name
    assert np.array_equal(a["state"][0, :3], b["state"][0, :3])
    hb = int(b["state"][0, 3])
    slots = (hb * w.G + np.arange(w.fill[0])) % (2 * w.G)
    assert np.array_equal(a["buf_k"][0][:, :w.fill[0]], b["buf_k"][0][:, slots])
    assert np.all(qs.qs_get_errors(cache) == 0)


# ------------------------------------------------------------ full sizes

def _sampled_oracle(w, bs, hs):
    cap = max(w.n_groups) + 1
    oc = oracle.OracleCache(len(bs), len(hs), w.D, w.G, cap)

    def tokens(i, t0, n):
        k, v = synthetic.kv_tokens(w, bs[i], t0, n)
        return k[hs], v[hs]

    oracle.prefill(oc, tokens, [w.n_groups[b] for b in bs], [w.fill[b] for b in bs])
    return oc


@pytest.mark.parametrize("cfg,bs,hs,ub", [
    ("32k", [0], list(range(32)), 4),
    ("128k", [0], [0, 7, 19, 31], 4),
    ("batched32k", [0, 5, 7], [1, 30], 4),
    ("ragged", [0, 3, 9, 15], [2, 17], 4),
    ("32k", [0], [0, 13, 31], 2),
])
def test_full_size_sampled(torch, cfg, bs, hs, ub):
    """Full-size workloads in the launch configuration the benchmark times;
    the oracle recomputes the sampled (sequence, head) pairs.  ub: the top
    bits the draft reads (2: the two-bit draft layout)."""
    w = synthetic.CONFIGS[cfg]()
    cap = max(w.n_groups) + 1
    cache = qs.Cache(w.B, w.H, cap, upper_bits=ub)
    driver.prefill(cache, w)
    oc = _sampled_oracle(w, bs, hs)
    # quantized planes of the sampled heads, bit for bit
    dev = layout.read_device(cache)
    want = layout.device_arrays(oc, ub)
    for name in ("k_upper", "k_lower", "v_upper", "v_lower", "meta"):
        g = dev[name][np.ix_(bs, hs)]
        assert np.array_equal(g[:, :, :oc.cap], want[name]), name
    assert np.array_equal(dev["state"][bs, :5], want["state"][:, :5])

    def both(call, mode, n_q):
        q = synthetic.queries(w, call, n_q)
        got, gl = run_attn(torch, cache, mode, q)
        ref, rl = oc.attn(np.ascontiguousarray(q[np.ix_(bs, hs)]), upper_only=(mode == DRAFT),
                          upper_bits=ub)
        assert_close(got[np.ix_(bs, hs)], ref, gl[np.ix_(bs, hs)], rl, "%s mode %d" % (cfg, mode))

    both(0, DRAFT, 1)
    # a verify round: flush where the 5 target tokens would overflow, append
    # them, then 5 causal queries (every sequence then has fill >= 5)
    mask = torch.zeros(w.B, dtype=torch.uint8, device="cuda")
    qs.qs_need_flush(cache, 5, mask)
    qs.qs_quantize_flush(cache, mask)
    m = oc.need_flush(5)
    assert np.array_equal(mask.cpu().numpy()[bs], m)
    oc.flush(m)
    k = np.zeros((w.B, w.H, 5, w.D), np.float16)
    v = np.zeros_like(k)
    for b in range(w.B):
        k[b], v[b] = synthetic.kv_tokens(w, b, w.context[b], 5)
    qs.qs_buffer_append(cache, to_dev(torch, k), to_dev(torch, v))
    oc.append(np.ascontiguousarray(k[np.ix_(bs, hs)]), np.ascontiguousarray(v[np.ix_(bs, hs)]))
    dev = layout.read_device(cache)
    want = layout.device_arrays(oc, ub)
    for name in ("k_upper", "v_lower", "meta"):
        g = dev[name][np.ix_(bs, hs)]
        assert np.array_equal(g[:, :, :want[name].shape[2]], want[name]), name
    # the logical buffer tokens (ring slots past fill may hold different
    # dropped tokens: the device prefill appended the batch-wide maximum fill)
    for i, b in enumerate(bs):
        st = dev["state"][b]
        assert np.array_equal(st[:4], oc.state[i, :4])
        slots = (st[3] * w.G + np.arange(st[1])) % (2 * w.G)
        for name, ref in (("buf_k", oc.bk), ("buf_v", oc.bv)):
            assert np.array_equal(dev[name][b][hs][:, slots], ref[i][:, slots]), name
    both(1, VERIFY, 5)
    both(2, DRAFT, 1)
    assert np.all(qs.qs_get_errors(cache) == 0)


# ------------------------------------------------- grouped-query attention

def run_attn_gqa(torch, cache, mode, q, group):
    B, HQ, n_q, D = q.shape
    qd = to_dev(torch, q)
    out = torch.full_like(qd, float("nan"))
    lse = torch.full((B, HQ, n_q), float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.empty(qs.qs_attn_workspace_size_gqa(cache, n_q, group), dtype=torch.uint8,
                     device="cuda")
    qs.qs_attn_decode_gqa(cache, mode, qd, group, 1.0 / np.sqrt(D), out, lse, ws)
    torch.cuda.synchronize()
    assert int(cache.arrive.abs().sum().item()) == 0, "segment counters not back at zero"
    return out.double().cpu().numpy(), lse.double().cpu().numpy()


@pytest.mark.parametrize("group,n_q,ub", [(4, 1, 4), (8, 1, 4), (4, 5, 4), (2, 5, 4), (3, 8, 4),
                                          (1, 5, 4), (5, 4, 4), (24, 1, 4), (4, 1, 2), (4, 5, 2),
                                          (3, 8, 2)])
def test_gqa_attention(torch, group, n_q, ub):
    """Grouped-query attention (query head h*g + i on KV head h) against the
    oracle for 1, 2 and 3 column groups of query rows (up to 24 rows per KV
    head), ragged prompts, both modes, 4- and 2-bit drafts."""
    rng = np.random.default_rng(70 + 10 * group + n_q)
    B, H, T, cap = 3, 2, 2200, 17
    lens = np.array([1000, 333, 2200], np.int32)
    k, v = h16(rng, (B, H, T, 128), 2.0), h16(rng, (B, H, T, 128))
    cache = qs.Cache(B, H, cap, upper_bits=ub)
    qs.qs_prefill(cache, to_dev(torch, k), to_dev(torch, v), to_dev(torch, lens))
    oc = oracle.OracleCache(B, H, 128, 128, cap)
    oc.prefill(k, v, lens)
    for mode in (DRAFT, VERIFY):
        q = h16(rng, (B, H * group, n_q, 128))
        got, gl = run_attn_gqa(torch, cache, mode, q, group)
        ref, rl = oc.attn(q, upper_only=(mode == DRAFT), group=group, upper_bits=ub)
        assert_close(got, ref, gl, rl, "gqa g=%d n_q=%d mode %d" % (group, n_q, mode))
    assert np.all(qs.qs_get_errors(cache) == 0)


def test_gqa_full_size_llama31_8b(torch):
    """Llama-3.1-8B attention shape at 32k (8 KV heads, 32 query heads): the
    draft call (4 rows per KV head) and the 5-query verify call (20 rows, three
    column groups), every head against the oracle."""
    w = synthetic.llama31_8b_32k()
    T = w.context[0]
    k, v = synthetic.kv_tokens(w, 0, 0, T)
    cap = w.n_groups[0] + 1
    cache = qs.Cache(1, w.H, cap)
    qs.qs_prefill(cache, to_dev(torch, k[None]), to_dev(torch, v[None]),
                  to_dev(torch, np.array([T], np.int32)))
    oc = oracle.OracleCache(1, w.H, w.D, w.G, cap)
    oc.prefill(k[None], v[None], [T])
    for call, (mode, n_q) in enumerate(((DRAFT, 1), (VERIFY, 5))):
        q = synthetic.queries(w, call, n_q)
        got, gl = run_attn_gqa(torch, cache, mode, q, w.group)
        ref, rl = oc.attn(q, upper_only=(mode == DRAFT), group=w.group)
        assert_close(got, ref, gl, rl, "llama31 8b mode %d" % mode)
    assert np.all(qs.qs_get_errors(cache) == 0)
