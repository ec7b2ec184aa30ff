"""Helpers for the GPU tests: move a synthetic workload to the device, run the
library through its binding, and run the oracle on the same inputs."""
from __future__ import annotations

import numpy as np

from oracle import indexer as X
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


def oracle_cache(wl, fmt):
    c = S.new_cache(wl.num_pages, fmt)
    S.store(c, fmt, wl.fill_k, wl.fill_pos, wl.fill_seq, wl.page_table, wl.num_pages, wl.theta, wl.eps)
    S.store(c, fmt, wl.new_k, wl.new_pos, wl.new_seq, wl.page_table, wl.num_pages, wl.theta, wl.eps)
    return c


def oracle_topk(wl, fmt, cache, rows, k=None):
    k = wl.k if k is None else k
    return X.index_topk(cache, fmt, wl.page_table, wl.seq_lens, wl.cu_q, wl.q, wl.head_w,
                        wl.causal, k, rows=rows, return_scores=True)


def slot_bytes(cache_np: np.ndarray, fmt: int, wl, pos, seq):
    """Bytes of the given tokens' slots (data + scale for fp8), [n, token_bytes]."""
    page, off = S.slots(pos, seq, wl.page_table, wl.num_pages)
    pb = S.PAGE_BYTES[fmt]
    if fmt == S.FMT_BF16:
        base = page * pb + off * 256
        return cache_np[base[:, None] + np.arange(256)[None, :]]
    base = page * pb + off * 128
    data = cache_np[base[:, None] + np.arange(128)[None, :]]
    sb = page * pb + 8192 + off * 4
    sc = cache_np[sb[:, None] + np.arange(4)[None, :]]
    return np.concatenate([data, sc], axis=1)
