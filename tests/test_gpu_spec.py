"""GPU parity of qs_spec_accept (speculative-sampling acceptance) against the
oracle: accepted counts, emitted tokens and rollback counts bit for bit (every
decision is an IEEE fp32 operation on both sides), and the rollback count
feeding qs_buffer_rollback on the device."""
import numpy as np
import pytest

import oracle
from hierarchical_quantized_kv_gb300 import qs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    import torch as t
    assert t.cuda.is_available(), "GPU tests need CUDA"
    import __graft_entry__
    __graft_entry__.build()
    return t


def softmax_rows(rng, shape, temp):
    z = rng.standard_normal(shape) * temp
    z = np.exp(z - z.max(axis=-1, keepdims=True))
    return (z / z.sum(axis=-1, keepdims=True)).astype(np.float32)


def draw(rng, q):
    """Draft tokens sampled from q [B, g, V] (inverse CDF)."""
    B, g, V = q.shape
    cdf = np.cumsum(q.astype(np.float64), axis=-1)
    r = rng.random((B, g, 1)) * cdf[..., -1:]
    return np.minimum((cdf < r).sum(axis=-1), V - 1).astype(np.int32)


def run(torch, p, q, draft, u, e):
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    B = p.shape[0]
    outs = [torch.full((B,), -7, dtype=torch.int32, device="cuda") for _ in range(3)]
    qs.qs_spec_accept(dev(p), dev(q), dev(draft), dev(u), dev(e), *outs)
    torch.cuda.synchronize()
    return [o.cpu().numpy() for o in outs]


@pytest.mark.parametrize("B,g,V,temp", [(64, 4, 32000, 3.0), (37, 4, 32000, 0.3), (8, 8, 1000, 1.0),
                                        (5, 1, 1, 1.0), (16, 3, 513, 6.0)])
def test_spec_accept_matches_oracle(torch, B, g, V, temp):
    rng = np.random.default_rng(B * 1000 + V)
    p = softmax_rows(rng, (B, g + 1, V), temp)
    # drafts close to the target (as a quantized draft is), with some far off
    q = softmax_rows(rng, (B, g, V), temp) if temp > 2 else \
        (0.8 * p[:, :g] + 0.2 * softmax_rows(rng, (B, g, V), temp)).astype(np.float32)
    draft = draw(rng, q)
    u = rng.random((B, g)).astype(np.float32)
    e = rng.exponential(size=(B, V)).astype(np.float32)
    got = run(torch, p, q, draft, u, e)
    want = oracle.spec_accept(p, q, draft, u, e)
    for gname, gv, wv in zip(("n_accept", "token", "n_drop"), got, want):
        assert np.array_equal(gv, wv), gname
    assert np.all(got[1] >= 0)


def test_spec_accept_edge_cases(torch):
    rng = np.random.default_rng(11)
    B, g, V = 6, 4, 700
    p = softmax_rows(rng, (B, g + 1, V), 1.0)
    q = p[:, :g].copy()
    draft = draw(rng, q)
    u = rng.random((B, g)).astype(np.float32)
    e = rng.exponential(size=(B, V)).astype(np.float32)
    draft[1, 2] = V        # not a token: rejected at 2
    draft[2, 0] = -3       # rejected at 0
    p[3] = 0.0             # all-zero target: rejected at 0, token -1
    q[4, 1] = 0.0          # a zero residual nowhere positive: fallback to p_1
    p[4, 1] = 0.0
    p[4, 1, 5] = 1.0
    draft[4, 1] = 6        # p = 0 there: rejected at 1, residual = token 5
    got = run(torch, p, q, draft, u, e)
    want = oracle.spec_accept(p, q, draft, u, e)
    for gv, wv in zip(got, want):
        assert np.array_equal(gv, wv)
    assert got[0][0] == g and got[0][1] == 2 and got[0][2] == 0 and got[1][3] == -1
    assert got[0][4] == 1 and got[1][4] == 5


def test_rollback_count_feeds_the_buffer_on_the_device(torch):
    """A round of the speculative loop without a host round trip: append the
    gamma + 1 target tokens, decide acceptance on the device, and roll back
    the device-side n_drop; the cache state equals the oracle's."""
    rng = np.random.default_rng(5)
    B, H, g, V = 4, 2, 4, 2000
    cache = qs.Cache(B, H, 2)
    oc = oracle.OracleCache(B, H, 128, 128, 2)
    qs.qs_state_reset(cache)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    k = rng.standard_normal((B, H, 20, 128)).astype(np.float16)
    qs.qs_buffer_append(cache, dev(k), dev(k))
    oc.append(k, k)
    qs.qs_buffer_rollback(cache, dev(np.zeros(B, np.int32)))
    oc.rollback(np.zeros(B, np.int32))
    kt = rng.standard_normal((B, H, g + 1, 128)).astype(np.float16)
    qs.qs_buffer_append(cache, dev(kt), dev(kt))
    oc.append(kt, kt)
    p = softmax_rows(rng, (B, g + 1, V), 1.0)
    q = (0.7 * p[:, :g] + 0.3 * softmax_rows(rng, (B, g, V), 1.0)).astype(np.float32)
    draft = draw(rng, q)
    u = rng.random((B, g)).astype(np.float32)
    e = rng.exponential(size=(B, V)).astype(np.float32)
    na, tok, nd = (torch.zeros(B, dtype=torch.int32, device="cuda") for _ in range(3))
    qs.qs_spec_accept(dev(p), dev(q), dev(draft), dev(u), dev(e), na, tok, nd)
    qs.qs_buffer_rollback(cache, nd)  # straight from the device
    wa, wt, wd = oracle.spec_accept(p, q, draft, u, e)
    oc.rollback(wd)
    torch.cuda.synchronize()
    assert np.array_equal(nd.cpu().numpy(), wd)
    st = cache.state.cpu().numpy()
    assert np.array_equal(st[:, :4], oc.state[:, :4])
    assert np.all(qs.qs_get_errors(cache) == 0)
