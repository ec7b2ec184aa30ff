"""Python binding of libdsaidx: argument marshalling only.

Every step of the indexer runs in the library's CUDA kernels; this module
checks tensor shapes/dtypes, passes device pointers and the current CUDA
stream through the C ABI declared in include/dsaidx.h, and raises on a
non-zero status. There is no fallback: without the built library every call
raises.
"""
from __future__ import annotations

import ctypes
import os

FMT_BF16 = 0
FMT_FP8 = 1
FMT_FP4 = 2
KERNEL_KINDS = ("store", "plan", "score_bf16", "score_fp8", "score_fp4")
HEADS = 64
HEAD_DIM = 128
PAGE_SIZE = 64

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdsaidx.so")
_lib = None

_c_int = ctypes.c_int32
_c_ptr = ctypes.c_void_p
_c_size = ctypes.c_size_t


class DsaError(RuntimeError):
    def __init__(self, where: str, status: int):
        super().__init__(f"{where}: {status_str(status)} (status {status})")
        self.status = status


def lib() -> ctypes.CDLL:
    """Load libdsaidx.so (built in-tree); raises if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built: run __graft_entry__.build()")
        L = ctypes.CDLL(LIB_PATH)
        L.dsa_ctx_create.argtypes = [ctypes.POINTER(_c_ptr), ctypes.c_float, ctypes.c_float, _c_int, _c_ptr]
        L.dsa_ctx_create.restype = ctypes.c_int
        L.dsa_ctx_destroy.argtypes = [_c_ptr]
        L.dsa_ctx_destroy.restype = ctypes.c_int
        L.dsa_cache_page_bytes.argtypes = [ctypes.c_int]
        L.dsa_cache_page_bytes.restype = _c_size
        L.dsa_index_store.argtypes = [_c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_int, _c_int, _c_int,
                                      _c_ptr, _c_int, ctypes.c_int, _c_ptr]
        L.dsa_index_store.restype = ctypes.c_int
        L.dsa_index_topk_workspace_size.argtypes = [_c_ptr, _c_int, _c_int, _c_int, ctypes.c_int]
        L.dsa_index_topk_workspace_size.restype = _c_size
        L.dsa_index_topk.argtypes = [_c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_int, ctypes.c_int, _c_ptr, _c_int,
                                     _c_ptr, _c_ptr, _c_int, _c_int, _c_int, _c_int, _c_ptr, _c_ptr,
                                     _c_ptr, _c_size, _c_ptr]
        L.dsa_index_topk.restype = ctypes.c_int
        L.dsa_index_topk_static.argtypes = [_c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_int, ctypes.c_int, _c_ptr,
                                            _c_int, _c_ptr, _c_ptr, _c_int, _c_int, _c_int, _c_int,
                                            _c_ptr, _c_ptr, _c_ptr]
        L.dsa_index_topk_static.restype = ctypes.c_int
        L.dsa_get_device_status.argtypes = [_c_ptr, _c_ptr]
        L.dsa_get_device_status.restype = ctypes.c_int
        L.dsa_selftest_bounded_wait.argtypes = [_c_ptr, _c_ptr]
        L.dsa_selftest_bounded_wait.restype = ctypes.c_int
        L.dsa_ctx_set_slot_output.argtypes = [_c_ptr, _c_int]
        L.dsa_ctx_set_slot_output.restype = ctypes.c_int
        L.dsa_ctx_set_hadamard.argtypes = [_c_ptr, _c_int]
        L.dsa_ctx_set_hadamard.restype = ctypes.c_int
        L.dsa_profile_enable.argtypes = [_c_ptr, ctypes.c_int]
        L.dsa_profile_enable.restype = ctypes.c_int
        L.dsa_profile_read.argtypes = [_c_ptr, ctypes.POINTER(ctypes.c_float), ctypes.POINTER(_c_int)]
        L.dsa_profile_read.restype = ctypes.c_int
        L.dsa_status_str.argtypes = [ctypes.c_int]
        L.dsa_status_str.restype = ctypes.c_char_p
        _lib = L
    return _lib


def status_str(s: int) -> str:
    try:
        return lib().dsa_status_str(int(s)).decode()
    except RuntimeError:
        return f"status {s}"


def page_bytes(fmt: int) -> int:
    return int(lib().dsa_cache_page_bytes(int(fmt)))


def _stream_ptr(stream):
    if stream is None:
        import torch
        return _c_ptr(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return _c_ptr(stream)
    return _c_ptr(stream.cuda_stream)


def _dev(t, dtype, shape=None, name="tensor"):
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return _c_ptr(t.data_ptr())


class Context:
    """A library context on the current CUDA device (RoPE table, gamma,
    device status word)."""

    def __init__(self, theta: float = 10000.0, eps: float = 1e-6, max_pos: int = 131072,
                 gamma_bf16=None):
        self.theta = float(theta)
        self.eps = float(eps)
        self.max_pos = int(max_pos)
        h = _c_ptr()
        g = None
        if gamma_bf16 is not None:
            import numpy as np
            garr = np.ascontiguousarray(gamma_bf16, dtype=np.uint16)
            if garr.shape != (128,):
                raise ValueError("gamma_bf16 must be 128 bf16 bit patterns")
            self._gamma = garr
            g = _c_ptr(garr.ctypes.data)
        st = lib().dsa_ctx_create(ctypes.byref(h), ctypes.c_float(theta), ctypes.c_float(eps),
                                  _c_int(max_pos), g)
        if st != 0:
            raise DsaError("dsa_ctx_create", st)
        self._h = h

    @property
    def handle(self):
        return self._h

    def close(self):
        if getattr(self, "_h", None):
            lib().dsa_ctx_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def store(self, k_raw, rope_pos, seq_id, page_table, cache, num_pages: int, fmt: int,
              stream=None):
        """dsa_index_store: write RMSNorm+RoPE'd index keys into the paged cache."""
        import torch
        T = int(k_raw.shape[0]) if k_raw.dim() == 2 else -1
        B, max_pages = int(page_table.shape[0]), int(page_table.shape[1])
        st = lib().dsa_index_store(
            self._h, _dev(k_raw, torch.bfloat16, (T, HEAD_DIM), "k_raw"),
            _dev(rope_pos, torch.int32, (T,), "rope_pos"), _dev(seq_id, torch.int32, (T,), "seq_id"),
            _dev(page_table, torch.int32, None, "page_table"), _c_int(T), _c_int(B), _c_int(max_pages),
            _dev(cache, torch.uint8, None, "cache"), _c_int(num_pages), int(fmt), _stream_ptr(stream))
        if st != 0:
            raise DsaError("dsa_index_store", st)

    def topk_workspace_size(self, Tq: int, B: int, k: int, fmt: int) -> int:
        return int(lib().dsa_index_topk_workspace_size(self._h, _c_int(Tq), _c_int(B), _c_int(k), int(fmt)))

    def topk(self, q, head_w, cache, num_pages: int, fmt: int, page_table, seq_lens, cu_q,
             causal: bool, k: int, out_idx, out_score, workspace, stream=None):
        """dsa_index_topk: per-query top-k key positions and scores."""
        import torch
        Tq = int(q.shape[0])
        B, max_pages = int(page_table.shape[0]), int(page_table.shape[1])
        st = lib().dsa_index_topk(
            self._h, _dev(q, torch.bfloat16, (Tq, HEADS, HEAD_DIM), "q"),
            _dev(head_w, torch.float32, (Tq, HEADS), "head_w"), _dev(cache, torch.uint8, None, "cache"),
            _c_int(num_pages), int(fmt), _dev(page_table, torch.int32, None, "page_table"),
            _c_int(max_pages), _dev(seq_lens, torch.int32, (B,), "seq_lens"),
            _dev(cu_q, torch.int32, (B + 1,), "cu_q"), _c_int(B), _c_int(Tq), _c_int(1 if causal else 0),
            _c_int(k), _dev(out_idx, torch.int32, (Tq, k), "out_idx"),
            _dev(out_score, torch.float32, (Tq, k), "out_score"),
            _dev(workspace, torch.uint8, None, "workspace"), _c_size(workspace.numel()),
            _stream_ptr(stream))
        if st != 0:
            raise DsaError("dsa_index_topk", st)

    def topk_static(self, q, head_w, cache, num_pages: int, fmt: int, page_table, seq_lens, cu_q,
                    causal: bool, k: int, out_idx, out_score, stream=None):
        """dsa_index_topk_static: as topk(), with the library's fixed scratch
        array instead of a caller workspace (allocates nothing)."""
        import torch
        Tq = int(q.shape[0])
        B, max_pages = int(page_table.shape[0]), int(page_table.shape[1])
        st = lib().dsa_index_topk_static(
            self._h, _dev(q, torch.bfloat16, (Tq, HEADS, HEAD_DIM), "q"),
            _dev(head_w, torch.float32, (Tq, HEADS), "head_w"), _dev(cache, torch.uint8, None, "cache"),
            _c_int(num_pages), int(fmt), _dev(page_table, torch.int32, None, "page_table"),
            _c_int(max_pages), _dev(seq_lens, torch.int32, (B,), "seq_lens"),
            _dev(cu_q, torch.int32, (B + 1,), "cu_q"), _c_int(B), _c_int(Tq), _c_int(1 if causal else 0),
            _c_int(k), _dev(out_idx, torch.int32, (Tq, k), "out_idx"),
            _dev(out_score, torch.float32, (Tq, k), "out_score"), _stream_ptr(stream))
        if st != 0:
            raise DsaError("dsa_index_topk_static", st)

    def set_hadamard(self, on: bool = True):
        """Store keys (and rotate queries) with the 128-point Walsh-Hadamard transform."""
        st = lib().dsa_ctx_set_hadamard(self._h, 1 if on else 0)
        if st != 0:
            raise DsaError("dsa_ctx_set_hadamard", st)

    def selftest_bounded_wait(self, stream=None):
        """Enqueue the bounded-wait self-test (records a timeout in the status)."""
        st = lib().dsa_selftest_bounded_wait(self._h, _stream_ptr(stream))
        if st != 0:
            raise DsaError("dsa_selftest_bounded_wait", st)

    def set_slot_output(self, on: bool = True):
        """Top-k returns cache slots (page * 64 + offset) instead of positions."""
        st = lib().dsa_ctx_set_slot_output(self._h, 1 if on else 0)
        if st != 0:
            raise DsaError("dsa_ctx_set_slot_output", st)

    def profile_enable(self, on: bool = True):
        st = lib().dsa_profile_enable(self._h, 1 if on else 0)
        if st != 0:
            raise DsaError("dsa_profile_enable", st)

    def profile_read(self):
        """{kind: (total ms, launches)} since the previous read (synchronises)."""
        ms = (ctypes.c_float * len(KERNEL_KINDS))()
        n = (_c_int * len(KERNEL_KINDS))()
        st = lib().dsa_profile_read(self._h, ms, n)
        if st != 0:
            raise DsaError("dsa_profile_read", st)
        return {k: (float(ms[i]), int(n[i])) for i, k in enumerate(KERNEL_KINDS)}

    def device_status(self, stream=None) -> int:
        """Synchronise the stream; read and clear the device status word."""
        return int(lib().dsa_get_device_status(self._h, _stream_ptr(stream)))
