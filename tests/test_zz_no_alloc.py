"""GPU test of dsa_index_topk_static, the top-k entry point for callers that
cannot allocate device memory (an engine that has already split all free
memory into its own pools, or a latency-critical path where cudaMalloc is not
allowed). It must give the same results as dsa_index_topk with a caller
workspace and pass the oracle comparison, on two calls in a row that share
its fixed scratch array, leave the device's free memory unchanged, and
reject sizes beyond that array without launching.

This file is collected last so that a run stopping at the first failure has
already run every other test.
"""
import ctypes

import numpy as np
import pytest

from synth import inputs as I
from tests import gpu_util as U
from tests import parity as P

pytestmark = pytest.mark.gpu


def _call_static(ctx, wl, fmt, d, k, out_i, out_s):
    from dsa_sparse_attention_store_gb300 import dsaidx
    import torch
    L = dsaidx.lib()
    P = ctypes.c_void_p
    st = L.dsa_index_topk_static(
        ctx.handle, P(d["q"].data_ptr()), P(d["head_w"].data_ptr()), P(d["cache"].data_ptr()),
        wl.num_pages, fmt, P(d["page_table"].data_ptr()), wl.max_pages, P(d["seq_lens"].data_ptr()),
        P(d["cu_q"].data_ptr()), wl.B, wl.Tq, 1 if wl.causal else 0, k, P(out_i.data_ptr()),
        P(out_s.data_ptr()), P(torch.cuda.current_stream().cuda_stream))
    return st


@pytest.mark.parametrize("fmt", [0, 1, 2])
def test_static_scratch_matches_workspace_path(fmt):
    import torch
    from dsa_sparse_attention_store_gb300 import Context
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    ctx = Context(theta=10000.0, eps=1e-6, max_pos=20000)
    try:
        for n, wl in enumerate([I.make_workload("na", [5000, 300, 12000], [1, 1, 1], [1, 1, 1], True, 512,
                                                seed=41, wid=40),
                                I.make_workload("nb", [2500, 700], [8, 8], [2500, 700], True, 1024,
                                                seed=42, wid=41)]):
            d = U.device_workload(wl, fmt, ctx)
            ref_i, ref_s = U.run_topk(wl, fmt, ctx, d)
            outs = [(torch.full((wl.Tq, wl.k), 7, dtype=torch.int32, device="cuda"),
                     torch.full((wl.Tq, wl.k), 7.0, dtype=torch.float32, device="cuda")) for _ in range(2)]
            # a first call looks up the scratch array (it may load the module);
            # after it, the calls must not change the device's free memory
            assert _call_static(ctx, wl, fmt, d, wl.k, *outs[0]) == 0
            torch.cuda.synchronize()
            free0 = torch.cuda.mem_get_info()[0]
            for call in range(2):   # two calls in a row share the static scratch
                out_i, out_s = outs[call]
                out_i.fill_(7)
                out_s.fill_(7.0)
                st = _call_static(ctx, wl, fmt, d, wl.k, out_i, out_s)
                assert st == 0, f"workload {n} call {call}: status {st}"
            torch.cuda.synchronize()
            assert torch.cuda.mem_get_info()[0] == free0, "the static entry point allocated device memory"
            assert ctx.device_status() == 0
            cache = U.oracle_cache(wl, fmt)
            rows = np.arange(wl.Tq)
            o_i, o_s, full = U.oracle_topk(wl, fmt, cache, rows)
            for call in range(2):
                gi, gs = outs[call][0].cpu().numpy(), outs[call][1].cpu().numpy()
                # same kernels and inputs as the workspace path: positions equal,
                # scores within the bf16 logit tolerance of its scores
                assert np.array_equal(gi, ref_i), f"workload {n} call {call}: positions differ"
                fin = np.isfinite(ref_s)
                assert np.array_equal(fin, np.isfinite(gs))
                assert np.allclose(gs[fin], ref_s[fin], rtol=2e-3, atol=0)
                # and against the oracle, with the rules every other top-k test uses
                ok, reps = P.compare(rows, gi, gs, o_i, o_s, full, wl.k, fmt)
                assert ok, P.summary(reps)
    finally:
        ctx.close()


def test_static_scratch_rejects_oversized_request():
    # the smallest batch whose workspace exceeds the fixed array: one
    # sequence, k = 1024. Every buffer is allocated at its true size (about
    # 27 GB on the device), so the call could not read outside them even if
    # it were not refused; it must be refused before anything is launched.
    import torch
    from dsa_sparse_attention_store_gb300 import Context
    ctx = Context(theta=10000.0, eps=1e-6, max_pos=4096)
    try:
        lo, hi = 1, 1 << 22
        while lo < hi:                                   # largest Tq that fits
            mid = (lo + hi + 1) // 2
            if ctx.topk_workspace_size(mid, 1, 1024, 1) <= (32 << 20):
                lo = mid
            else:
                hi = mid - 1
        Tq = lo + 1
        assert ctx.topk_workspace_size(Tq, 1, 1024, 1) > (32 << 20)
        npg = (Tq + 63) // 64
        d = {
            "q": torch.empty((Tq, 64, 128), dtype=torch.bfloat16, device="cuda"),
            "head_w": torch.empty((Tq, 64), dtype=torch.float32, device="cuda"),
            "cache": torch.zeros(npg * 8448, dtype=torch.uint8, device="cuda"),
            "page_table": torch.arange(npg, dtype=torch.int32, device="cuda").view(1, npg),
            "seq_lens": torch.tensor([Tq], dtype=torch.int32, device="cuda"),
            "cu_q": torch.tensor([0, Tq], dtype=torch.int32, device="cuda"),
        }

        class W:  # the call's sizes
            num_pages, max_pages, B, causal = npg, npg, 1, True
        W.Tq = Tq
        out_i = torch.zeros((Tq, 1024), dtype=torch.int32, device="cuda")
        out_s = torch.zeros((Tq, 1024), dtype=torch.float32, device="cuda")
        assert _call_static(ctx, W, 1, d, 1024, out_i, out_s) == 6     # DSA_ERR_WORKSPACE
        torch.cuda.synchronize()
        assert int(out_i[:64].abs().sum()) == 0 and int(out_i[-64:].abs().sum()) == 0   # nothing ran
        del d, out_i, out_s
        torch.cuda.empty_cache()
    finally:
        ctx.close()
