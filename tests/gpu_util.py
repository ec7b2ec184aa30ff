"""Helpers for the GPU tests: move a synthetic workload to the device, run the
library through its binding, and run the oracle on the same inputs (the C++
oracle for speed; the numpy oracle on request)."""
from __future__ import annotations

import numpy as np

from oracle import indexer as X
from oracle import native as N
from oracle import store as S


def t_bf16(bits: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)


def device_workload(wl, fmt, ctx, store_fill=True, store_new=True):
    """Upload wl, allocate a cache, run the store for fill then new tokens."""
    import torch
    from dsa_sparse_attention_store_gb300 import page_bytes
    dev = torch.device("cuda")
    d = {
        "page_table": torch.from_numpy(wl.page_table).to(dev),
        "seq_lens": torch.from_numpy(wl.seq_lens).to(dev),
        "cu_q": torch.from_numpy(wl.cu_q).to(dev),
        "q": t_bf16(wl.q).to(dev),
        "head_w": torch.from_numpy(wl.head_w).to(dev),
        "cache": torch.zeros(wl.num_pages * page_bytes(fmt), dtype=torch.uint8, device=dev),
    }
    for tag in ("fill", "new"):
        if (tag == "fill" and not store_fill) or (tag == "new" and not store_new):
            continue
        k = getattr(wl, f"{tag}_k")
        if k.shape[0] == 0:
            continue
        d[f"{tag}_k"] = t_bf16(k).to(dev)
        d[f"{tag}_pos"] = torch.from_numpy(getattr(wl, f"{tag}_pos")).to(dev)
        d[f"{tag}_seq"] = torch.from_numpy(getattr(wl, f"{tag}_seq")).to(dev)
        ctx.store(d[f"{tag}_k"], d[f"{tag}_pos"], d[f"{tag}_seq"], d["page_table"], d["cache"],
                  wl.num_pages, fmt)
    return d


def run_topk(wl, fmt, ctx, d, k=None):
    import torch
    k = wl.k if k is None else k
    dev = torch.device("cuda")
    Tq = wl.Tq
    out_i = torch.empty((Tq, k), dtype=torch.int32, device=dev)
    out_s = torch.empty((Tq, k), dtype=torch.float32, device=dev)
    ws = torch.empty(ctx.topk_workspace_size(Tq, wl.B, k, fmt), dtype=torch.uint8, device=dev)
    ctx.topk(d["q"], d["head_w"], d["cache"], wl.num_pages, fmt, d["page_table"], d["seq_lens"],
             d["cu_q"], wl.causal, k, out_i, out_s, ws)
    torch.cuda.synchronize()
    return out_i.cpu().numpy(), out_s.cpu().numpy()


def oracle_cache(wl, fmt, native=True):
    """The oracle's byte image of the cache after the workload's stores (the
    C++ oracle by default; its bytes equal the numpy oracle's, which
    tests/test_oracle_native.py pins)."""
    c = S.new_cache(wl.num_pages, fmt)
    st = N.store if native else S.store
    st(c, fmt, wl.fill_k, wl.fill_pos, wl.fill_seq, wl.page_table, wl.num_pages, wl.theta, wl.eps)
    st(c, fmt, wl.new_k, wl.new_pos, wl.new_seq, wl.page_table, wl.num_pages, wl.theta, wl.eps)
    return c


def oracle_topk(wl, fmt, cache, rows, k=None, native=True, hadamard=False):
    """Oracle top-k of the given rows with their full score vectors (the C++
    oracle by default)."""
    k = wl.k if k is None else k
    f = N.index_topk if native else X.index_topk
    return f(cache, fmt, wl.page_table, wl.seq_lens, wl.cu_q, wl.q, wl.head_w, wl.causal, k,
             rows=rows, return_scores=True, hadamard=hadamard)


def compare_all_rows(wl, fmt, cache, gi, gs, rows=None, k=None, block=1024, hadamard=False):
    """Compare the GPU's rows with the C++ oracle block by block (so the full
    score vectors of a long prefill never sit in memory at once). Returns
    (ok, summary over all rows)."""
    from tests import parity as P
    k = wl.k if k is None else k
    rows = np.arange(wl.Tq) if rows is None else np.asarray(rows)
    bad, n, swaps, err = [], 0, 0, 0.0
    for i0 in range(0, len(rows), block):
        rr = rows[i0:i0 + block]
        oi, os_, full = oracle_topk(wl, fmt, cache, rr, k, hadamard=hadamard)
        ok, reps = P.compare(rr, gi[rr], gs[rr], oi, os_, full, k, fmt)
        n += len(reps)
        swaps += sum(r.swaps for r in reps)
        err = max(err, max((r.logit_err for r in reps), default=0.0))
        bad += [r for r in reps if not r.ok]
    summ = {"rows": n, "failed": len(bad), "swaps": int(swaps), "max_logit_err": err,
            "first_failure": None if not bad else f"row {bad[0].row}: {bad[0].why}"}
    return not bad, summ


def slot_bytes(cache_np: np.ndarray, fmt: int, wl, pos, seq):
    """Bytes of the given tokens' slots (codes + scale for fp8 / fp4), [n, token_bytes]."""
    page, off = S.slots(pos, seq, wl.page_table, wl.num_pages)
    pb = S.PAGE_BYTES[fmt]
    if fmt == S.FMT_BF16:
        base = page * pb + off * 256
        return cache_np[base[:, None] + np.arange(256)[None, :]]
    cb = S.CODE_BYTES[fmt]
    base = page * pb + off * cb
    data = cache_np[base[:, None] + np.arange(cb)[None, :]]
    sb = page * pb + 64 * cb + off * 4
    sc = cache_np[sb[:, None] + np.arange(4)[None, :]]
    return np.concatenate([data, sc], axis=1)
