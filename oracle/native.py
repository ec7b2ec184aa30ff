"""The C++17 oracle (oracle/cpp/dsa_oracle.cpp) through ctypes.

Test infrastructure, not the product: only tests/, __graft_entry__ (which
builds it and whose smoke() may call it) and bench.py's CPU-baseline and
reference legs use it. It computes the same definitions as oracle.store and
oracle.indexer, written a second time in C++ with std::thread so that
full-size workloads can be checked row by row, and shares no code with the
GPU library. The functions below take and return the same arrays as their
numpy counterparts.

Built with g++ (C++17, -ffp-contract=off so that no fp32 multiply-add of the
store is fused) into oracle/_build/<machine>/libdsaoracle.so on first use.
"""
from __future__ import annotations

import ctypes
import os
import platform
import shutil
import subprocess

import numpy as np

from . import store as S

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "cpp", "dsa_oracle.cpp")
BUILD = os.path.join(HERE, "_build", platform.machine())
LIB = os.path.join(BUILD, "libdsaoracle.so")
FLAGS = ["-O3", "-std=c++17", "-ffp-contract=off", "-fPIC", "-shared", "-pthread"]

_lib = None


def build(force: bool = False) -> str:
    """Compile the C++ oracle (if its source is newer than the library)."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    cxx = shutil.which("g++") or shutil.which("c++")
    if not cxx:
        raise RuntimeError("no C++ compiler for the oracle")
    tmp = LIB + f".{os.getpid()}.tmp"
    r = subprocess.run([cxx, *FLAGS, "-o", tmp, SRC], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"oracle build failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i32, i64 = ctypes.c_int, ctypes.c_longlong
        L.dso_hardware_threads.restype = i32
        L.dso_store.argtypes = [P, i32, i32, P, P, P, i64, P, i32, i32, ctypes.c_float, ctypes.c_float,
                                P, i32, i32]
        L.dso_store.restype = i32
        L.dso_topk.argtypes = [P, i32, P, i32, i32, P, P, P, P, i32, i32, i32, P, i64, P, P, P, P, i32]
        L.dso_topk.restype = i32
        _lib = L
    return _lib


def threads() -> int:
    """Threads the oracle runs on by default: std::thread::hardware_concurrency()."""
    return int(lib().dso_hardware_threads())


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a, ctypes.c_void_p(a.ctypes.data)


def store(cache: np.ndarray, fmt: int, k_raw_bits, pos, seq, page_table, num_pages: int,
          theta: float = 10000.0, eps: float = 1e-6, gamma_bits=None, hadamard: bool = False,
          nthreads: int | None = None) -> None:
    """Write the tokens' index keys into the byte image of the paged cache
    (in place, like oracle.store.store)."""
    T = len(pos)
    if T == 0:
        return
    assert cache.dtype == np.uint8 and cache.flags.c_contiguous
    kr, kp = _c(k_raw_bits, np.uint16)
    ps, pp = _c(pos, np.int32)
    sq, sp = _c(seq, np.int32)
    pt, ptp = _c(page_table, np.int32)
    g = None
    if gamma_bits is not None:
        ga, g = _c(gamma_bits, np.uint16)
    st = lib().dso_store(ctypes.c_void_p(cache.ctypes.data), num_pages, fmt, kp, pp, sp, T, ptp,
                         pt.shape[0], pt.shape[1], theta, eps, g, 1 if hadamard else 0,
                         nthreads or threads())
    if st != 0:
        raise ValueError("sequence, position or page id out of range")


def visible_counts(cu_q, seq_lens, rows, causal: bool) -> np.ndarray:
    cu_q = np.asarray(cu_q, dtype=np.int64)
    seq_lens = np.asarray(seq_lens, dtype=np.int64)
    rows = np.asarray(rows, dtype=np.int64)
    b = np.searchsorted(cu_q, rows, side="right") - 1
    nq = cu_q[b + 1] - cu_q[b]
    qpos = seq_lens[b] - nq + (rows - cu_q[b])
    return qpos + 1 if causal else seq_lens[b]


def index_topk(cache, fmt, page_table, seq_lens, cu_q, q_bits, head_w, causal: bool, k: int,
               rows=None, return_scores: bool = False, hadamard: bool = False,
               nthreads: int | None = None):
    """Top-k positions and fp32 scores for the given query rows (all by
    default), like oracle.indexer.index_topk: (idx [n, k] int32, score [n, k]
    float32) and, when return_scores, a dict row -> float64 scores over the
    row's visible keys."""
    Tq = q_bits.shape[0]
    rows = np.arange(Tq, dtype=np.int64) if rows is None else np.asarray(rows, dtype=np.int64)
    n = len(rows)
    out_i = np.empty((n, k), dtype=np.int32)
    out_s = np.empty((n, k), dtype=np.float32)
    cnt = visible_counts(cu_q, seq_lens, rows, causal)
    full = off = None
    fp = op = None
    if return_scores:
        off = np.zeros(n, dtype=np.int64)
        off[1:] = np.cumsum(cnt)[:-1]
        full = np.empty(int(cnt.sum()), dtype=np.float64)
        fp = ctypes.c_void_p(full.ctypes.data)
        op = ctypes.c_void_p(off.ctypes.data)
    ca = np.ascontiguousarray(cache, dtype=np.uint8)
    pt, ptp = _c(page_table, np.int32)
    # every page a row reads must exist in the cache image
    num_pages = ca.size // S.PAGE_BYTES[fmt]
    b = np.searchsorted(np.asarray(cu_q, dtype=np.int64), rows, side="right") - 1
    for bb in np.unique(b):
        need = int(cnt[b == bb].max(initial=0) + S.PAGE - 1) // S.PAGE
        ids = pt[bb, :need]
        if need > pt.shape[1] or np.any((ids < 0) | (ids >= num_pages)):
            raise ValueError("page id out of range")
    sl, slp = _c(seq_lens, np.int32)
    cq, cqp = _c(cu_q, np.int32)
    qb, qbp = _c(q_bits, np.uint16)
    hw, hwp = _c(head_w, np.float32)
    rr, rrp = _c(rows, np.int64)
    st = lib().dso_topk(ctypes.c_void_p(ca.ctypes.data), fmt, ptp, pt.shape[0], pt.shape[1], slp, cqp, qbp,
                        hwp, 1 if causal else 0, k, 1 if hadamard else 0, rrp, n,
                        ctypes.c_void_p(out_i.ctypes.data), ctypes.c_void_p(out_s.ctypes.data), fp, op,
                        nthreads or threads())
    if st != 0:
        raise ValueError("bad format or k")
    if return_scores:
        d = {int(r): full[off[i]:off[i] + cnt[i]] for i, r in enumerate(rows.tolist())}
        return out_i, out_s, d
    return out_i, out_s


def new_cache(num_pages: int, fmt: int) -> np.ndarray:
    return S.new_cache(num_pages, fmt)
