"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every function include/dsaidx.h declares, and rejects bad arguments before
touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HDR = os.path.join(ROOT, "include", "dsaidx.h")


def _declared():
    txt = open(HDR).read()
    return sorted(set(re.findall(r"\b(dsa_[a-z_]+)\s*\(", txt)))


@pytest.fixture(scope="module")
def L():
    from dsa_sparse_attention_store_gb300 import dsaidx
    if not os.path.exists(dsaidx.LIB_PATH):
        import __graft_entry__
        __graft_entry__.build()
    return dsaidx.lib()


def test_exports_every_declared_symbol(L):
    names = _declared()
    assert "dsa_index_store" in names and "dsa_index_topk" in names
    for n in names:
        assert hasattr(L, n), n


def test_status_strings_and_page_bytes(L):
    from dsa_sparse_attention_store_gb300 import dsaidx
    for s in range(7):
        assert dsaidx.status_str(s)
    assert L.dsa_cache_page_bytes(0) == 16384
    assert L.dsa_cache_page_bytes(1) == 8448
    assert L.dsa_cache_page_bytes(2) == 4352    # 64 x (64 code bytes + 4-byte scale)
    assert L.dsa_cache_page_bytes(7) == 0


def test_invalid_arguments_rejected_without_device(L):
    P = ctypes.c_void_p
    fake = P(0x1000)      # never dereferenced: every case below fails validation first
    good = P(0x100000)
    # null context
    assert L.dsa_index_store(None, good, good, good, good, 1, 1, 1, good, 1, 0, None) == 1
    # unknown format
    assert L.dsa_index_store(fake, good, good, good, good, 1, 1, 1, good, 1, 3, None) == 2
    # negative token count / zero pages
    assert L.dsa_index_store(fake, good, good, good, good, -1, 1, 1, good, 1, 0, None) == 1
    assert L.dsa_index_store(fake, good, good, good, good, 1, 1, 1, good, 0, 0, None) == 1
    # null pointer
    assert L.dsa_index_store(fake, None, good, good, good, 1, 1, 1, good, 1, 0, None) == 1
    # misaligned k_raw / cache
    assert L.dsa_index_store(fake, P(0x100008), good, good, good, 1, 1, 1, good, 1, 0, None) == 1
    assert L.dsa_index_store(fake, good, good, good, good, 1, 1, 1, P(0x100010), 1, 0, None) == 1
    # T == 0 is a no-op
    assert L.dsa_index_store(fake, None, None, None, None, 0, 1, 1, None, 1, 0, None) == 0
    # and so is Tq == 0 (no buffer is needed, every format)
    for f in (0, 1, 2):
        empty = [None, None, None, 1, f, None, 1, None, None, 1, 0, 1]
        assert L.dsa_index_topk(fake, *empty, 512, None, None, None, 0, None) == 0
    args = [good, good, good, 1, 0, good, 1, good, good, 1, 4, 1]
    # k above 2048
    assert L.dsa_index_topk(fake, *args, 2049, good, good, good, 1 << 30, None) == 2
    assert L.dsa_index_topk(None, *args, 512, good, good, good, 1 << 30, None) == 1
    # unknown format
    bad = list(args)
    bad[4] = 5
    assert L.dsa_index_topk(fake, *bad, 512, good, good, good, 1 << 30, None) == 2
    # null output
    assert L.dsa_index_topk(fake, *args, 512, None, good, good, 1 << 30, None) == 1
    # misaligned workspace
    assert L.dsa_index_topk(fake, *args, 512, good, good, P(0x100040), 1 << 30, None) == 1
    # workspace size query rejects bad k / format / null ctx
    assert L.dsa_index_topk_workspace_size(fake, 4, 1, 0, 0) == 0
    assert L.dsa_index_topk_workspace_size(None, 4, 1, 512, 0) == 0
    assert L.dsa_index_topk_workspace_size(fake, 4, 1, 512, 9) == 0
    # settings on a null context
    assert L.dsa_ctx_set_hadamard(None, 1) == 1
    assert L.dsa_ctx_set_slot_output(None, 1) == 1
    assert L.dsa_selftest_bounded_wait(None, None) == 1
    # k outside 1 .. 2048
    assert L.dsa_index_topk(fake, *args, 0, good, good, good, 1 << 30, None) == 2
    assert L.dsa_index_topk(fake, *args, 2049, good, good, good, 1 << 30, None) == 2
    assert L.dsa_index_topk_workspace_size(fake, 4, 1, 2049, 0) == 0


def test_context_creation_without_gpu_fails_cleanly(L):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    h = ctypes.c_void_p()
    st = L.dsa_ctx_create(ctypes.byref(h), ctypes.c_float(10000.0), ctypes.c_float(1e-6), 64, None)
    assert st in (2, 3) and not h.value
    assert L.dsa_ctx_create(ctypes.byref(h), ctypes.c_float(-1.0), ctypes.c_float(1e-6), 64, None) == 1


def test_device_is_checked_before_the_context_is_read(L):
    # With every argument valid, the next step is the check that the current
    # device is the context's. Without a GPU it cannot pass (no device to
    # query), so the call returns DSA_ERR_CUDA before the fake context below
    # is ever dereferenced or anything is enqueued.
    import torch
    if torch.cuda.is_available():
        pytest.skip("needs a machine without a GPU (the context pointer is fake)")
    P = ctypes.c_void_p
    fake = P(0x1000)
    good = P(0x100000)
    assert L.dsa_index_store(fake, good, good, good, good, 1, 1, 1, good, 1, 0, None) == 3
    args = [good, good, good, 1, 0, good, 1, good, good, 1, 4, 1]
    assert L.dsa_index_topk(fake, *args, 512, good, good, good, 1 << 30, None) == 3
    assert L.dsa_index_topk_static(fake, *args, 512, good, good, None) == 3
    assert L.dsa_get_device_status(fake, None) == 3
    assert L.dsa_selftest_bounded_wait(fake, None) == 3
