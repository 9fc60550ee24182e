"""qs_attn_decode_append (append, then decode attention, in one launch)
against the oracle running the two operations one after the other.

The attention output must be within the parity tolerance of the other tests;
the buffer, the counters and the error words bit-exact: a sequence whose buffer
cannot take the tokens is flagged QS_DEV_OVERFLOW and attends over its buffer as
it was, exactly as a separate append followed by the attention would do.
"""
import numpy as np
import pytest

import oracle
from tests import layout
from tests.test_gpu_qs import (DRAFT, VERIFY, _oracle_state, assert_close, assert_state_equal,
                               h16, to_dev)
from hierarchical_quantized_kv_gb300 import qs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    import torch as t
    assert t.cuda.is_available(), "GPU tests need CUDA"
    import __graft_entry__
    __graft_entry__.build()
    return t


def fused(torch, cache, mode, k, v, q, group=1, lse=True):
    kd, vd, qd = to_dev(torch, k), to_dev(torch, v), to_dev(torch, q)
    out = torch.full_like(qd, float("nan"))
    l_ = torch.full(q.shape[:3], float("nan"), dtype=torch.float32, device="cuda") if lse else None
    ws = torch.empty(qs.qs_attn_workspace_size_gqa(cache, q.shape[2], group), dtype=torch.uint8,
                     device="cuda")
    qs.qs_attn_decode_append(cache, mode, kd, vd, qd, 1.0 / np.sqrt(128), out, l_, ws, group)
    torch.cuda.synchronize()
    assert int(cache.arrive.abs().sum().item()) == 0, "segment counters not back at zero"
    return out.double().cpu().numpy(), (l_.double().cpu().numpy() if lse else None)


@pytest.mark.parametrize("B,H,n_groups,fill", [(1, 32, 40, 253), (3, 8, 60, 130), (2, 2, 3, 40)])
def test_fused_round_matches_separate_calls(torch, B, H, n_groups, fill):
    """A speculative round with the appends fused into the attention calls:
    four (append 1 draft token, draft), rollback, (append 5, verify), rollback;
    outputs against the oracle at each point, state bit-exact at the end."""
    rng = np.random.default_rng(B * 100 + H + fill)
    cap = n_groups + 2
    oc = _oracle_state(rng, B, H, [n_groups] * B, [fill] * B, cap=cap)
    cache = qs.Cache(B, H, cap)
    layout.load_into(cache, oc)
    g = 4
    m = oc.need_flush(g + 1)
    qs.qs_quantize_flush(cache, to_dev(torch, m))
    oc.flush(m)
    for i in range(g):
        k, v, q = h16(rng, (B, H, 1, 128), 2.0), h16(rng, (B, H, 1, 128)), h16(rng, (B, H, 1, 128))
        got, gl = fused(torch, cache, DRAFT, k, v, q)
        oc.append(k, v)
        ref, rl = oc.attn(q, upper_only=True)
        assert_close(got, ref, gl, rl, "draft %d" % i)
    drop = np.full(B, g, np.int32)
    qs.qs_buffer_rollback(cache, to_dev(torch, drop))
    oc.rollback(drop)
    k, v, q = h16(rng, (B, H, g + 1, 128), 2.0), h16(rng, (B, H, g + 1, 128)), h16(rng, (B, H, g + 1, 128))
    got, gl = fused(torch, cache, VERIFY, k, v, q)
    oc.append(k, v)
    ref, rl = oc.attn(q, upper_only=False)
    assert_close(got, ref, gl, rl, "verify")
    r = rng.integers(0, g + 1, B).astype(np.int32)
    qs.qs_buffer_rollback(cache, to_dev(torch, r))
    oc.rollback(r)
    assert_state_equal(cache, oc, "after the round")
    assert np.all(qs.qs_get_errors(cache) == 0)


def test_overflow_and_short_buffers_in_one_batch(torch):
    """Four sequences: one whose buffer cannot take the tokens (flagged, it
    attends over its old buffer), one with an empty quantized region, one that
    has fewer buffered tokens than queries even after the append (flagged,
    zero output, lse -inf) and an ordinary one."""
    rng = np.random.default_rng(5)
    B, H, cap = 4, 3, 6
    oc = _oracle_state(rng, B, H, [4, 0, 0, 5], [254, 20, 1, 100], cap=cap)
    cache = qs.Cache(B, H, cap)
    layout.load_into(cache, oc)
    n_new, n_q = 3, 5
    k, v, q = h16(rng, (B, H, n_new, 128), 2.0), h16(rng, (B, H, n_new, 128)), h16(rng, (B, H, n_q, 128))
    got, gl = fused(torch, cache, VERIFY, k, v, q)
    oc.append(k, v)
    ref, rl = oc.attn(q, upper_only=False)
    errs = qs.qs_get_errors(cache)
    want = np.array([qs.DEV_OVERFLOW, 0, qs.DEV_NQ_GT_FILL, 0], np.int32)
    assert np.array_equal(errs, want), errs
    ok = np.array([0, 1, 3])
    assert_close(got[ok], ref[ok], gl[ok], rl[ok], "verify")
    assert np.all(got[2] == 0) and np.all(np.isneginf(gl[2]))
    oc.state[:, oracle.ERR] = 0
    assert_state_equal(cache, oc, "after the fused call")


@pytest.mark.parametrize("mode,n_new,n_q", [(DRAFT, 1, 1), (VERIFY, 5, 5)])
def test_grouped_query_fused(torch, mode, n_new, n_q):
    """Grouped-query heads (4 query heads per KV head): the appended tokens
    are the KV heads' and every query head of the group sees them."""
    rng = np.random.default_rng(11 + n_q)
    B, H, group, cap = 2, 4, 4, 5
    oc = _oracle_state(rng, B, H, [3, 1], [120, 7], cap=cap)
    cache = qs.Cache(B, H, cap)
    layout.load_into(cache, oc)
    k, v = h16(rng, (B, H, n_new, 128), 2.0), h16(rng, (B, H, n_new, 128))
    q = h16(rng, (B, H * group, n_q, 128))
    got, gl = fused(torch, cache, mode, k, v, q, group=group)
    oc.append(k, v)
    ref, rl = oc.attn(q, upper_only=(mode == DRAFT), group=group)
    assert_close(got, ref, gl, rl, "grouped-query")
    assert_state_equal(cache, oc, "after the fused call")
    assert np.all(qs.qs_get_errors(cache) == 0)


def test_host_validation(torch):
    cache = qs.Cache(1, 2, 2)
    k = torch.zeros((1, 2, 1, 128), dtype=torch.float16, device="cuda")
    q = torch.zeros((1, 2, 1, 128), dtype=torch.float16, device="cuda")
    ws = torch.empty(qs.qs_attn_workspace_size(cache, 1), dtype=torch.uint8, device="cuda")
    L = qs.lib()
    args = lambda kk, vv, n: (cache._ref, DRAFT, qs._ptr(kk), qs._ptr(vv), n, qs._ptr(q), 1, 1, 0.1,
                              qs._ptr(q), None, qs._ptr(ws), ws.numel(), None)
    assert L.qs_attn_decode_append(*args(None, k, 1)) == qs.QS_ERR_ARG
    assert L.qs_attn_decode_append(*args(k, k, 0)) == qs.QS_ERR_ARG
    assert L.qs_attn_decode_append(*args(k, k, 257)) == qs.QS_ERR_ARG
    kv = k.view(-1)[1:]  # a 2-byte offset: not 16-byte aligned
    assert L.qs_attn_decode_append(*args(kv, k, 1)) == qs.QS_ERR_ALIGN


@pytest.mark.parametrize("n_next", [0, 5, 60, 130])
def test_flush_due_equals_need_flush_then_flush(torch, n_next):
    """qs_quantize_flush_due(n_next): the sequences whose buffer cannot take
    n_next more tokens are flushed, bit for bit as qs_need_flush + the masked
    qs_quantize_flush; among them, at some n_next, one at capacity and one
    whose oldest half still holds pending tokens, both flagged and left
    unchanged."""
    rng = np.random.default_rng(40 + n_next)
    B, H = 6, 3
    ng, fill = [2, 0, 3, 1, 4, 2], [250, 200, 130, 125, 250, 140]
    cap = 4  # sequence 4 is at capacity
    oc = _oracle_state(rng, B, H, ng, fill, cap=cap)
    cache = qs.Cache(B, H, cap)
    layout.load_into(cache, oc)
    # four pending tokens everywhere: sequence 3 then has 125 committed
    k, v = h16(rng, (B, H, 4, 128), 2.0), h16(rng, (B, H, 4, 128))
    oc.append(k, v)
    qs.qs_buffer_append(cache, to_dev(torch, k), to_dev(torch, v))
    qs.qs_quantize_flush_due(cache, n_next)
    oc.flush(oc.need_flush(n_next))
    torch.cuda.synchronize()
    assert_state_equal(cache, oc, "flush_due(%d)" % n_next)
    errs = qs.qs_get_errors(cache)
    assert np.array_equal(errs, oc.state[:, oracle.ERR]), (errs, oc.state[:, oracle.ERR])
    if n_next == 130:
        assert errs[3] == qs.DEV_FLUSH_UNCOMMITTED and errs[4] == qs.DEV_CAPACITY


def test_flush_due_host_validation(torch):
    cache = qs.Cache(1, 2, 2)
    for bad in (-1, 257):
        assert qs.lib().qs_quantize_flush_due(cache._ref, bad, None) == qs.QS_ERR_ARG
