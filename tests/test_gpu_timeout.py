"""The bounded waits of the attention kernel, made to run out on purpose.

Every pipeline wait of the split-KV kernel gives up after a time limit,
records QS_DEV_TIMEOUT in the sequence's error word and lets the kernel
finish (no trap, no endless loop).  The library's test entry
qs_test_attn_decode_timeout (not part of include/qs.h) runs the ordinary
kernel with a 1 ms limit and without issuing any copy, so the word each warp
waits on is never written and every wait runs out.  The test checks that the
call returns, that every sequence is flagged, that no output is written, that
the arrival counters are back at zero, and that ordinary calls on the same
cache and context afterwards match the oracle.
"""
import ctypes
import time

import numpy as np
import pytest

import oracle
from hierarchical_quantized_kv_gb300 import driver, qs, synthetic

pytestmark = pytest.mark.gpu

ATOL, RRMS = 1e-2, 2e-3
WAIT_NS = 1_000_000  # 1 ms per wait


@pytest.fixture(scope="module")
def torch():
    import torch as t
    assert t.cuda.is_available(), "GPU tests need CUDA"
    import __graft_entry__
    __graft_entry__.build()
    return t


def _timeout_call(torch, cache, mode, q, group, scale, out, lse, ws):
    f = qs.lib().qs_test_attn_decode_timeout
    f.argtypes = [ctypes.POINTER(qs.QsCacheStruct), ctypes.c_int, ctypes.c_void_p, ctypes.c_int32,
                  ctypes.c_int32, ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p,
                  ctypes.c_void_p, ctypes.c_size_t, ctypes.c_uint64, ctypes.c_void_p]
    f.restype = ctypes.c_int
    return f(cache._ref, mode, ctypes.c_void_p(q.data_ptr()), q.shape[2], group,
             ctypes.c_float(scale), ctypes.c_void_p(out.data_ptr()),
             None if lse is None else ctypes.c_void_p(lse.data_ptr()),
             ctypes.c_void_p(ws.data_ptr()), ws.numel(), WAIT_NS,
             ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _check_close(got, ref):
    err = np.abs(got - ref).max()
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert err <= ATOL and rel <= RRMS, (err, rel)


def _prompt_cache(torch, w, T):
    """A one-sequence cache prefilled with the first T tokens of workload w,
    and the oracle's copy of it."""
    k, v = synthetic.kv_tokens(w, 0, 0, T)
    ng = -(-(T - 2 * w.G) // w.G) if T > 2 * w.G else 0
    cache = qs.Cache(1, w.H, ng + 1)
    qs.qs_prefill(cache, torch.from_numpy(k[None]).cuda(), torch.from_numpy(v[None]).cuda(),
                  torch.tensor([T], dtype=torch.int32, device="cuda"))
    oc = oracle.OracleCache(1, w.H, w.D, w.G, cap=ng + 1)
    oracle.prefill(oc, lambda b, t0, n: synthetic.kv_tokens(w, 0, t0, n), [ng], [T - ng * w.G])
    return cache, oc


@pytest.mark.parametrize("case", ["tiny", "4096_tokens_32_heads"])
def test_waits_run_out_and_the_cache_stays_usable(torch, case):
    if case == "tiny":
        w = synthetic.tiny()
        cache = qs.Cache(w.B, w.H, 8)
        driver.prefill(cache, w)
        oc = oracle.OracleCache(w.B, w.H, w.D, w.G, cap=8)
        oracle.prefill(oc, lambda b, t0, n: synthetic.kv_tokens(w, b, t0, n), w.n_groups, w.fill)
    else:  # ~30 units per head over 152 CTAs: shared segments, arrivals
        w = synthetic.llama_32k()
        cache, oc = _prompt_cache(torch, w, 4096)
    scale = 1.0 / np.sqrt(w.D)
    for call, (mode, n_q) in enumerate(((qs.QS_DRAFT_UPPER4, 1), (qs.QS_VERIFY_INT8, 5))):
        q_np = synthetic.queries(w, call, n_q)
        q = torch.from_numpy(q_np).cuda()
        ws = torch.empty(qs.qs_attn_workspace_size(cache, n_q), dtype=torch.uint8, device="cuda")
        out = torch.full_like(q, float("nan"))
        lse = torch.full(q.shape[:3], float("nan"), dtype=torch.float32, device="cuda")
        t0 = time.perf_counter()
        assert _timeout_call(torch, cache, mode, q, 1, scale, out, lse, ws) == qs.QS_OK
        torch.cuda.synchronize()
        assert time.perf_counter() - t0 < 5.0  # a few 1 ms waits, not the 4 s default
        errs = qs.qs_get_errors(cache)
        assert np.all(errs == qs.DEV_TIMEOUT), errs
        assert int(cache.arrive.abs().sum()) == 0          # ready for the next call
        assert bool(torch.isnan(out).all()) and bool(torch.isnan(lse).all())  # nothing written
        # the same cache and context: ordinary calls are valid again
        qs.qs_attn_decode(cache, mode, q, scale, out, lse, ws)
        torch.cuda.synchronize()
        ref, ref_lse = oc.attn(q_np, upper_only=(mode == qs.QS_DRAFT_UPPER4), scale=scale)
        _check_close(out.double().cpu().numpy(), ref)
        assert np.abs(lse.double().cpu().numpy() - ref_lse).max() < 5e-3
        assert np.all(qs.qs_get_errors(cache) == 0)
        assert int(cache.arrive.abs().sum()) == 0


def test_wait_limit_outside_its_range_is_rejected(torch):
    w = synthetic.tiny()
    cache = qs.Cache(w.B, w.H, 8)
    q = torch.zeros((1, 2, 1, 128), dtype=torch.float16, device="cuda")
    ws = torch.empty(qs.qs_attn_workspace_size(cache, 1), dtype=torch.uint8, device="cuda")
    f = qs.lib().qs_test_attn_decode_timeout
    f.argtypes = [ctypes.POINTER(qs.QsCacheStruct), ctypes.c_int, ctypes.c_void_p, ctypes.c_int32,
                  ctypes.c_int32, ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p,
                  ctypes.c_void_p, ctypes.c_size_t, ctypes.c_uint64, ctypes.c_void_p]
    f.restype = ctypes.c_int
    for limit in (0, 999, 100_000_001):
        assert f(cache._ref, 0, ctypes.c_void_p(q.data_ptr()), 1, 1, ctypes.c_float(0.1),
                 ctypes.c_void_p(q.data_ptr()), None, ctypes.c_void_p(ws.data_ptr()), ws.numel(),
                 limit, None) == qs.QS_ERR_ARG
