"""The C-ABI library loads and exports every symbol include/msa.h declares
(no compute calls: this runs without a GPU)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
LIB = os.path.join(ROOT, "block_sparse_long_proxy_gb300", "libmsa.so")
HDR = os.path.join(ROOT, "include", "msa.h")


def declared_functions():
    text = open(HDR).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(msa_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(LIB):
        import __graft_entry__
        __graft_entry__.build()
    return ctypes.CDLL(LIB)


def test_header_declares_the_hot_path():
    names = declared_functions()
    for n in ["msa_plan", "msa_proxy_maxscore", "msa_topk_select", "msa_sparse_attn", "msa_sparse_attn_bwd",
              "msa_check_errors", "msa_last_error", "msa_plan_destroy"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_covers_every_declared_symbol(lib):
    from block_sparse_long_proxy_gb300 import msa
    assert sorted(msa.SIGNATURES) == declared_functions()


def test_host_validation_without_gpu(lib):
    """Argument checks run before any device work, so they answer on a
    machine without a GPU."""
    from block_sparse_long_proxy_gb300 import msa
    f = msa._lib
    assert f.msa_topk_select(None, 1, 1, 1, 1, None, None, None) == 1
    ql = (ctypes.c_int32 * 1)(10)
    kl = (ctypes.c_int32 * 1)(5)      # qo_len > kv_len
    h = ctypes.c_void_p()
    assert f.msa_plan(ql, kl, 1, 8, 2, 2, 64, 32, 128, 4, 16, 0, 0, None, ctypes.byref(h)) == 1
    assert b"qo_len <= kv_len" in f.msa_last_error()
    kl[0] = 100
    assert f.msa_plan(ql, kl, 1, 8, 2, 2, 96, 32, 128, 4, 16, 0, 0, None, ctypes.byref(h)) == 2   # head_dim 96
    assert f.msa_plan(ql, kl, 1, 8, 2, 3, 64, 32, 128, 4, 16, 0, 0, None, ctypes.byref(h)) == 2   # Hp % Hkv != 0
    assert f.msa_plan(ql, kl, 1, 8, 2, 16, 64, 32, 128, 4, 16, 0, 0, None, ctypes.byref(h)) == 2  # Hp does not divide Hq
    assert f.msa_plan(ql, kl, 1, 8, 2, 1, 64, 32, 128, 4, 16, 0, 0, None, ctypes.byref(h)) == 2   # Hp < Hkv
    assert f.msa_plan(ql, kl, 1, 8, 3, 3, 64, 32, 128, 4, 16, 0, 0, None, ctypes.byref(h)) == 1   # Hq % Hkv
    assert f.msa_plan(ql, kl, 1, 8, 2, 2, 64, 32, 64, 4, 16, 0, 0, None, ctypes.byref(h)) == 2    # page 64
    # sequence lengths: a negative qo_len, an empty kv_len and a batch without query rows are refused
    ql2 = (ctypes.c_int32 * 2)(0, 0)
    kl2 = (ctypes.c_int32 * 2)(100, 300)
    assert f.msa_plan(ql2, kl2, 2, 8, 2, 2, 64, 32, 128, 4, 16, 0, 0, None, ctypes.byref(h)) == 1
    assert b"no query rows" in f.msa_last_error()
    ql2[1] = -1
    assert f.msa_plan(ql2, kl2, 2, 8, 2, 2, 64, 32, 128, 4, 16, 0, 0, None, ctypes.byref(h)) == 1
    ql2[1], kl2[1] = 0, 0
    assert f.msa_plan(ql2, kl2, 2, 8, 2, 2, 64, 32, 128, 4, 16, 0, 0, None, ctypes.byref(h)) == 1
    assert f.msa_version() == b"0.1.0"
