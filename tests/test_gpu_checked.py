"""The bounds-checked build (-DQS_CHECKED=1, libqs_checked.so) over the
small workloads and the edge cases: every shared-memory load, copy
destination and source, workspace slot, query row and output head of the
attention kernel, and every group, metadata position and prompt row of the
flush and prefill kernels, is checked on the device; a failing check is
counted (never trapped) and read back through qs_checked_failures.  The runs
must count no failure, and their results still match the oracle.
"""
import ctypes

import numpy as np
import pytest

import oracle
from hierarchical_quantized_kv_gb300 import build as qs_build
from hierarchical_quantized_kv_gb300 import driver, qs, synthetic
from tests import layout
from tests.test_gpu_qs import DRAFT, VERIFY, _oracle_state, assert_close, h16, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def checked():
    """The binding pointed at the checked library for this module's tests
    (restored afterwards)."""
    import torch
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    path = qs_build.build(checked=True)
    saved = qs.LIB_PATH, qs._lib
    qs.LIB_PATH, qs._lib = path, None
    L = qs.lib()
    L.qs_checked_failures.argtypes = [ctypes.POINTER(ctypes.c_ulonglong),
                                      ctypes.POINTER(ctypes.c_uint), ctypes.c_int]
    L.qs_checked_failures.restype = ctypes.c_int

    def failures(reset=True):
        n, tag = ctypes.c_ulonglong(), ctypes.c_uint()
        torch.cuda.synchronize()
        assert L.qs_checked_failures(ctypes.byref(n), ctypes.byref(tag), int(reset)) == 0
        return n.value, tag.value
    failures()
    yield torch, failures
    qs.LIB_PATH, qs._lib = saved


def _attn(torch, cache, mode, q, group=1):
    qd = to_dev(torch, q)
    out = torch.full_like(qd, float("nan"))
    lse = torch.full(q.shape[:3], float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.empty(qs.qs_attn_workspace_size_gqa(cache, q.shape[2], group), dtype=torch.uint8,
                     device="cuda")
    qs.qs_attn_decode_gqa(cache, mode, qd, group, 1.0 / np.sqrt(128), out, lse, ws)
    torch.cuda.synchronize()
    return out.double().cpu().numpy(), lse.double().cpu().numpy()


def test_tiny_workload_through_the_checked_build(checked):
    torch, failures = checked
    w = synthetic.tiny()
    cache = qs.Cache(w.B, w.H, 8)
    driver.prefill(cache, w)   # appends, rollbacks and flushes
    oc = oracle.OracleCache(w.B, w.H, w.D, w.G, cap=8)
    oracle.prefill(oc, lambda b, t0, n: synthetic.kv_tokens(w, b, t0, n), w.n_groups, w.fill)
    for call, (mode, n_q) in enumerate(((DRAFT, 1), (VERIFY, 5))):
        q = synthetic.queries(w, call, n_q)
        got, gl = _attn(torch, cache, mode, q)
        ref, rl = oc.attn(q, upper_only=(mode == DRAFT))
        assert_close(got, ref, gl, rl, "tiny mode %d" % mode)
    assert failures() == (0, 0)


@pytest.mark.parametrize("n_groups,fill", [(0, 1), (0, 31), (1, 33), (3, 65), (2, 128), (5, 255),
                                           (4, 256)])
@pytest.mark.parametrize("n_q,group", [(1, 1), (5, 1), (8, 1), (5, 4), (1, 4)])
def test_edge_cases_through_the_checked_build(checked, n_groups, fill, n_q, group):
    torch, failures = checked
    rng = np.random.default_rng(1000 * n_groups + fill + 7 * n_q + group)
    B, H = 2, 3
    oc = _oracle_state(rng, B, H, [n_groups, max(n_groups - 1, 0)], [fill, max(fill // 2, 1)],
                       cap=n_groups + 1)
    cache = qs.Cache(B, H, n_groups + 1)
    layout.load_into(cache, oc)
    q = h16(rng, (B, H * group, n_q, 128))
    for mode in (DRAFT, VERIFY):
        got, gl = _attn(torch, cache, mode, q, group)
        ref, rl = oc.attn(q, upper_only=(mode == DRAFT), group=group)
        ok = [b for b in range(B) if n_q <= oc.counters(b)["fill"]]
        if ok:  # (sequences with fewer buffered tokens than queries are flagged)
            assert_close(got[ok], ref[ok], gl[ok], rl[ok], "mode %d" % mode)
    qs.qs_get_errors(cache)
    assert failures() == (0, 0)


def test_prefill_flush_and_fused_append_through_the_checked_build(checked):
    torch, failures = checked
    rng = np.random.default_rng(3)
    B, H, T = 2, 4, 700
    k, v = h16(rng, (B, H, T, 128), 2.0), h16(rng, (B, H, T, 128))
    lens = np.array([700, 300], np.int32)
    cache = qs.Cache(B, H, 6)
    qs.qs_prefill(cache, to_dev(torch, k), to_dev(torch, v), to_dev(torch, lens))
    oc = oracle.OracleCache(B, H, 128, 128, cap=6)
    oc.prefill(k, v, lens)
    qs.qs_quantize_flush_due(cache, 5)
    oc.flush(oc.need_flush(5))
    kn, vn, q = h16(rng, (B, H, 5, 128), 2.0), h16(rng, (B, H, 5, 128)), h16(rng, (B, H, 5, 128))
    out = torch.full((B, H, 5, 128), float("nan"), dtype=torch.float16, device="cuda")
    ws = torch.empty(qs.qs_attn_workspace_size(cache, 5), dtype=torch.uint8, device="cuda")
    qs.qs_attn_decode_append(cache, VERIFY, to_dev(torch, kn), to_dev(torch, vn), to_dev(torch, q),
                             1.0 / np.sqrt(128), out, None, ws)
    torch.cuda.synchronize()
    oc.append(kn, vn)
    ref, _ = oc.attn(q, upper_only=False)
    assert_close(out.double().cpu().numpy(), ref, what="prefill, flush, fused verify")
    assert np.all(qs.qs_get_errors(cache) == 0)
    assert failures() == (0, 0)
