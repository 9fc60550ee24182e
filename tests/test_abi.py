"""The C-ABI library builds, loads on a machine without a GPU, exports every
entry point include/qs.h declares, and validates arguments on the host
before touching CUDA."""
import ctypes
import os
import re

import numpy as np
import pytest

import __graft_entry__
from hierarchical_quantized_kv_gb300 import qs
from tests import layout

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "qs.h")


@pytest.fixture(scope="module")
def L():
    __graft_entry__.build()
    return qs.lib()


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"^(?:qs_status|const char \*)\s*(qs_\w+)\s*\(", text, flags=re.M)


def test_every_declared_symbol_is_exported(L):
    names = declared_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(L, n), n


def test_cache_bytes_and_unsupported_sizes(L):
    b = qs.qs_cache_bytes(2, 3, 5)
    assert b["k_upper"] == 2 * 3 * 5 * 128 * 64 == b["v_lower"]
    assert b["meta"] == 2 * 3 * 5 * 4 * 128 * 2
    assert b["buf_k"] == 2 * 3 * 256 * 128 * 2
    assert b["state"] == 2 * 8 * 4
    assert b["arrive"] == 2 * 3 * 4
    out = qs.QsCacheBytes()
    assert L.qs_cache_bytes(1, 1, 64, 128, 1, ctypes.byref(out)) == qs.QS_ERR_UNSUPPORTED
    assert L.qs_cache_bytes(0, 1, 128, 128, 1, ctypes.byref(out)) == qs.QS_ERR_ARG


def _fake_cache(**kw):
    c = qs.QsCacheStruct(1, 2, 128, 128, 4, 4, *([0x10000] * 9))
    for k, v in kw.items():
        setattr(c, k, v)
    return c


def test_host_validation_before_any_cuda_call(L):
    assert L.qs_state_reset(None, None) == qs.QS_ERR_ARG
    c = _fake_cache(state=0x10008)
    assert L.qs_state_reset(ctypes.byref(c), None) == qs.QS_ERR_ALIGN
    c = _fake_cache(arrive=0x10004)
    assert L.qs_state_reset(ctypes.byref(c), None) == qs.QS_ERR_ALIGN
    c = _fake_cache(arrive=None)
    assert L.qs_state_reset(ctypes.byref(c), None) == qs.QS_ERR_ARG
    c = _fake_cache(D=96)
    assert L.qs_state_reset(ctypes.byref(c), None) == qs.QS_ERR_UNSUPPORTED
    for ub in (0, 1, 3, 8):
        c = _fake_cache(upper_bits=ub)
        assert L.qs_state_reset(ctypes.byref(c), None) == qs.QS_ERR_ARG
    c = _fake_cache(B=300)
    assert L.qs_quantize_flush(ctypes.byref(c), None, None) == qs.QS_ERR_UNSUPPORTED
    c = _fake_cache()
    p = ctypes.c_void_p(0x20000)
    assert L.qs_buffer_append(ctypes.byref(c), p, p, 0, None) == qs.QS_ERR_ARG
    assert L.qs_buffer_append(ctypes.byref(c), p, p, 257, None) == qs.QS_ERR_ARG
    assert L.qs_buffer_rollback(ctypes.byref(c), None, None) == qs.QS_ERR_ARG
    for n_q in (0, 9):
        assert L.qs_attn_decode(ctypes.byref(c), 0, p, n_q, ctypes.c_float(0.1), p, None, p,
                                1 << 20, None) == qs.QS_ERR_ARG
    assert L.qs_attn_decode(ctypes.byref(c), 2, p, 1, ctypes.c_float(0.1), p, None, p, 1 << 20,
                            None) == qs.QS_ERR_ARG
    assert L.qs_attn_decode(ctypes.byref(c), 0, ctypes.c_void_p(0x20004), 1, ctypes.c_float(0.1),
                            p, None, p, 1 << 20, None) == qs.QS_ERR_ALIGN
    for s in range(8):
        assert qs.status_string(s)


def test_layout_permutations_are_bijections():
    assert sorted(layout.vperm(np.arange(32)).tolist()) == list(range(32))
    assert sorted(layout.kmeta_perm(np.arange(128)).tolist()) == list(range(128))
    assert sorted(layout.vmeta_perm(np.arange(128)).tolist()) == list(range(128))


def test_pack_unpack_roundtrip():
    rng = np.random.default_rng(0)
    kq = rng.integers(0, 256, (2, 3, 128, 128)).astype(np.uint8)
    u, l_ = layout.pack_k(kq)
    assert u.shape == (2, 3, 128, 64)
    assert np.array_equal(layout.unpack_k(u, l_), kq)
    vu, vl = layout.pack_v(kq)
    assert vu.shape == (2, 3, 4, 128, 16)
    # token 32u + vperm(p) of channel d sits at nibble p of row (u, d)
    for _ in range(50):
        a, b2, uu, d, p = (rng.integers(2), rng.integers(3), rng.integers(4), rng.integers(128),
                           rng.integers(32))
        byte = vu[a, b2, uu, d, p // 2]
        nib = (byte >> (4 * (p % 2))) & 15
        assert nib == kq[a, b2, 32 * uu + layout.vperm(p), d] >> 4


def test_gqa_host_validation(L):
    c = _fake_cache()
    p = ctypes.c_void_p(0x20000)
    n = ctypes.c_size_t()
    for n_q, g in ((1, 0), (5, 5), (8, 4), (0, 1), (9, 1)):
        assert L.qs_attn_workspace_size_gqa(ctypes.byref(c), n_q, g, ctypes.byref(n)) == qs.QS_ERR_ARG
        assert L.qs_attn_decode_gqa(ctypes.byref(c), 0, p, n_q, g, ctypes.c_float(0.1), p, None, p,
                                    1 << 20, None) == qs.QS_ERR_ARG


def test_prefill_and_spec_accept_host_validation(L):
    c = _fake_cache()
    p = ctypes.c_void_p(0x20000)
    assert L.qs_prefill(ctypes.byref(c), None, p, 10, p, None) == qs.QS_ERR_ARG
    assert L.qs_prefill(ctypes.byref(c), p, p, -1, p, None) == qs.QS_ERR_ARG
    assert L.qs_prefill(ctypes.byref(c), ctypes.c_void_p(0x20008), p, 10, p, None) == qs.QS_ERR_ALIGN
    f = L.qs_spec_accept
    args = [p] * 5 + [4, 4, 100] + [p] * 3 + [None]  # valid shape: not launched here
    for i, bad in ((0, None), (5, 0), (6, 0), (6, 65), (7, 0), (9, None)):
        a = list(args)
        a[i] = bad
        assert f(*a) == qs.QS_ERR_ARG, (i, bad)
    a = list(args)
    a[3] = ctypes.c_void_p(0x20002)
    assert f(*a) == qs.QS_ERR_ALIGN


def test_header_is_plain_c_and_links(L, tmp_path):
    """include/qs.h compiled as C11 by gcc; the program links against the
    library and calls its pure host functions (no GPU needed)."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    libdir = os.path.dirname(qs.LIB_PATH)
    exe = str(tmp_path / "abi_check")
    subprocess.run([gcc, "-std=c11", "-Wall", "-Werror", "-pedantic",
                    "-I" + os.path.join(root, "include"),
                    os.path.join(root, "tests", "abi_check.c"), "-L" + libdir, "-lqs",
                    "-Wl,-rpath," + libdir, "-o", exe], check=True)
    out = subprocess.run([exe], capture_output=True, text=True)
    assert out.returncode == 0 and out.stdout.strip() == "abi ok", (out.returncode, out.stdout)
