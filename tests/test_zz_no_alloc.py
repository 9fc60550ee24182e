"""qs_attn_decode_static_ws: decode attention for callers that cannot
allocate device memory.

Such callers (a serving process whose device memory is fixed up front, a
foreign runtime without a CUDA allocator, a plug-in handed only its input and
output buffers) cannot provide the scratch workspace qs_attn_decode needs.
This entry point keeps that scratch in a fixed array inside the library.  The
test calls it through the C ABI, twice in a row, and checks each result
against qs_attn_decode on the same inputs, within the parity tolerance of the
other tests.  This file is named to be collected last.
"""
import numpy as np
import pytest

from hierarchical_quantized_kv_gb300 import driver, qs, synthetic

pytestmark = pytest.mark.gpu

ATOL, RRMS = 1e-2, 2e-3


@pytest.fixture(scope="module")
def torch():
    import torch as t
    assert t.cuda.is_available(), "GPU tests need CUDA"
    import __graft_entry__
    __graft_entry__.build()
    return t


def _static_call(torch, cache, mode, q, scale, out, lse):
    # through the C ABI (ctypes marshalling in the binding); returns the status
    return qs.qs_attn_decode_static_ws(cache, mode, q, scale, out, lse)


def test_static_workspace_matches_allocating_call(torch):
    w = synthetic.tiny()
    cache = qs.Cache(w.B, w.H, 8)
    driver.prefill(cache, w)
    scale = 1.0 / np.sqrt(w.D)
    for call, (mode, n_q) in enumerate(((qs.QS_DRAFT_UPPER4, 1), (qs.QS_VERIFY_INT8, 5))):
        q = torch.from_numpy(synthetic.queries(w, call, n_q)).cuda()
        ref = torch.empty_like(q)
        ref_lse = torch.empty((w.B, w.H, n_q), dtype=torch.float32, device="cuda")
        ws = torch.empty(qs.qs_attn_workspace_size(cache, n_q), dtype=torch.uint8, device="cuda")
        qs.qs_attn_decode(cache, mode, q, scale, ref, ref_lse, ws)
        for rep in range(2):  # two calls in a row share the static scratch
            out = torch.full_like(q, float("nan"))
            lse = torch.full((w.B, w.H, n_q), float("nan"), dtype=torch.float32, device="cuda")
            status = _static_call(torch, cache, mode, q, scale, out, lse)
            assert status == qs.QS_OK, qs.status_string(status)
            torch.cuda.synchronize()
            g, r = out.double().cpu().numpy(), ref.double().cpu().numpy()
            assert np.all(np.isfinite(g))
            err = np.abs(g - r).max()
            rel = np.linalg.norm(g - r) / np.linalg.norm(r)
            assert err <= ATOL and rel <= RRMS, (mode, rep, err, rel)
            assert np.abs(lse.cpu().numpy() - ref_lse.cpu().numpy()).max() < 1e-3
    assert np.all(qs.qs_get_errors(cache) == 0)


def test_static_workspace_rejects_sizes_beyond_its_limit(torch):
    # 64 sequences x 32 heads x 8 queries need more scratch than the fixed array
    cache = qs.Cache(64, 32, 1)
    q = torch.zeros((64, 32, 8, 128), dtype=torch.float16, device="cuda")
    out = torch.empty_like(q)
    assert qs.qs_attn_workspace_size(cache, 8) > qs.QS_STATIC_WS_BYTES
    status = _static_call(torch, cache, qs.QS_VERIFY_INT8, q, 0.1, out, None)
    assert status == qs.QS_ERR_TOO_LARGE
