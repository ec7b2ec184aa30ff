"""Failure detection on the GPU without a GPU fault: a bounded wait that runs
out is reported through the status word and leaves the context usable; an
out-of-range page id in the page table the scorer reads is reported and its
page skipped (the store's own check is in test_gpu_store.py); a call made
with another device current is refused before anything is enqueued; and no
call writes outside its output, workspace or cache buffers (canary bytes
around each)."""
import numpy as np
import pytest

from oracle import store as S
from synth import inputs as I
from tests import gpu_util as U
from tests import parity as P

pytestmark = pytest.mark.gpu

CANARY = 0x5A
PAD = 4096


@pytest.fixture(scope="module")
def ctx():
    import torch
    from dsa_sparse_attention_store_gb300 import Context
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    c = Context(theta=10000.0, eps=1e-6, max_pos=131072)
    yield c
    c.close()


def _padded(nbytes, dev):
    """A device byte buffer with PAD canary bytes before and after the
    nbytes-long interior (interior zeroed); returns (whole, interior)."""
    import torch
    whole = torch.full((nbytes + 2 * PAD,), CANARY, dtype=torch.uint8, device=dev)
    inner = whole[PAD:PAD + nbytes]
    inner.zero_()
    return whole, inner


def _canaries_intact(whole):
    h = whole.cpu().numpy()
    return bool(np.all(h[:PAD] == CANARY) and np.all(h[-PAD:] == CANARY))


def test_bounded_wait_reports_timeout_and_context_stays_usable(ctx):
    import torch
    assert ctx.device_status() == 0
    ctx.selftest_bounded_wait()
    from dsa_sparse_attention_store_gb300 import dsaidx
    st = ctx.device_status()
    assert st == 5, dsaidx.status_str(st)          # DSA_ERR_TIMEOUT
    assert ctx.device_status() == 0                # read and cleared
    # the context and the device still work: a small top-k passes parity
    wl = I.make_workload("ft", [700, 300], [2, 1], [700, 300], True, 512, seed=51, wid=51)
    d = U.device_workload(wl, S.FMT_BF16, ctx)
    gi, gs = U.run_topk(wl, S.FMT_BF16, ctx, d)
    assert ctx.device_status() == 0
    cache = U.oracle_cache(wl, S.FMT_BF16)
    rows = np.arange(wl.Tq)
    oi, os_, full = U.oracle_topk(wl, S.FMT_BF16, cache, rows)
    ok, reps = P.compare(rows, gi, gs, oi, os_, full, wl.k, S.FMT_BF16)
    assert ok, P.summary(reps)
    torch.cuda.synchronize()


@pytest.mark.parametrize("fmt", [S.FMT_BF16, S.FMT_FP8, S.FMT_FP4])
@pytest.mark.parametrize("shape", ["decode", "prefill"])
def test_no_writes_outside_buffers(ctx, fmt, shape):
    import torch
    from dsa_sparse_attention_store_gb300 import page_bytes
    dev = torch.device("cuda")
    if shape == "decode":
        wl = I.make_workload("cd", [3000, 900, 5000, 64], [1] * 4, [1] * 4, True, 512, seed=52, wid=52)
    else:
        wl = I.make_workload("cp", [1100, 200], [300, 200], [1100, 200], True, 512, seed=53, wid=53)
    # cache with canaries around it
    cw, cache = _padded(wl.num_pages * page_bytes(fmt), dev)
    d = U.device_workload(wl, fmt, ctx, store_fill=False, store_new=False)
    d["cache"] = cache
    for tag in ("fill", "new"):
        k = getattr(wl, f"{tag}_k")
        if k.shape[0]:
            ctx.store(U.t_bf16(k).to(dev), torch.from_numpy(getattr(wl, f"{tag}_pos")).to(dev),
                      torch.from_numpy(getattr(wl, f"{tag}_seq")).to(dev), d["page_table"], cache,
                      wl.num_pages, fmt)
    k = wl.k
    iw, oi_b = _padded(wl.Tq * k * 4, dev)
    sw, os_b = _padded(wl.Tq * k * 4, dev)
    wsz = ctx.topk_workspace_size(wl.Tq, wl.B, k, fmt)
    ww, ws = _padded(wsz, dev)
    # interiors must keep the alignment the API asks for (PAD is 4096)
    oi = oi_b.view(torch.int32).view(wl.Tq, k)
    os_ = os_b.view(torch.float32).view(wl.Tq, k)
    ctx.topk(d["q"], d["head_w"], cache, wl.num_pages, fmt, d["page_table"], d["seq_lens"], d["cu_q"],
             wl.causal, k, oi, os_, ws)
    torch.cuda.synchronize()
    assert ctx.device_status() == 0
    for name, w in (("cache", cw), ("out_idx", iw), ("out_score", sw), ("workspace", ww)):
        assert _canaries_intact(w), f"write outside {name}"
    # and the result is still right
    ocache = U.oracle_cache(wl, fmt)
    rows = np.arange(wl.Tq) if wl.Tq <= 200 else np.linspace(0, wl.Tq - 1, 200).astype(np.int64)
    o_i, o_s, full = U.oracle_topk(wl, fmt, ocache, rows)
    ok, reps = P.compare(rows, oi.cpu().numpy()[rows], os_.cpu().numpy()[rows], o_i, o_s, full, k, fmt)
    assert ok, P.summary(reps)


def test_wrong_device_rejected_without_launch():
    # a context made on device 0, called with device 1 current: the call must
    # be refused before anything is enqueued (the kernels would run on device
    # 1 but read device 0's table and status word)
    import torch
    from dsa_sparse_attention_store_gb300 import Context, dsaidx
    if torch.cuda.device_count() < 2:
        pytest.skip("needs two GPUs")
    torch.cuda.set_device(0)
    c = Context(theta=10000.0, eps=1e-6, max_pos=4096)
    try:
        wl = I.make_workload("wd", [300], [2], [300], True, 512, seed=54, wid=54)
        torch.cuda.set_device(1)
        d = U.device_workload(wl, S.FMT_BF16, c, store_fill=False, store_new=False)
        k = U.t_bf16(wl.new_k).cuda()
        pos = torch.from_numpy(wl.new_pos).cuda()
        seq = torch.from_numpy(wl.new_seq).cuda()
        with pytest.raises(dsaidx.DsaError) as e:
            c.store(k, pos, seq, d["page_table"], d["cache"], wl.num_pages, S.FMT_BF16)
        assert e.value.status == 1
        torch.cuda.synchronize()
        assert int(d["cache"].sum()) == 0
    finally:
        torch.cuda.set_device(0)
        c.close()


@pytest.mark.parametrize("fmt", [S.FMT_BF16, S.FMT_FP8, S.FMT_FP4])
@pytest.mark.parametrize("shape", ["decode", "prefill"])
def test_scorer_skips_out_of_range_page(ctx, fmt, shape):
    # the keys are stored through a valid page table; top-k then reads a copy
    # in which one page id of sequence 0 (positions 192..255) points past the
    # cache. The scorer skips that page (no copy is issued for it, its keys
    # score -inf), records DSA_ERR_DEVICE_BOUNDS and carries on; rows that
    # never see positions 192..255 must still match the oracle.
    import torch
    if shape == "decode":
        wl = I.make_workload("bd", [3000, 900, 5000], [1, 1, 1], [1, 1, 1], True, 512, seed=55, wid=55)
        rows = np.array([1, 2])                      # sequence 0's query sees the bad page
    else:
        wl = I.make_workload("bf", [700, 300], [700, 300], [700, 300], True, 512, seed=56, wid=56)
        rows = np.concatenate([np.arange(0, 192), np.arange(700, 1000)])
    d = U.device_workload(wl, fmt, ctx)
    assert ctx.device_status() == 0
    bad_pt = d["page_table"].clone()
    bad_pt[0, 3] = wl.num_pages + 7
    k = wl.k
    oi = torch.empty((wl.Tq, k), dtype=torch.int32, device="cuda")
    os_ = torch.empty((wl.Tq, k), dtype=torch.float32, device="cuda")
    ws = torch.empty(ctx.topk_workspace_size(wl.Tq, wl.B, k, fmt), dtype=torch.uint8, device="cuda")
    ctx.topk(d["q"], d["head_w"], d["cache"], wl.num_pages, fmt, bad_pt, d["seq_lens"], d["cu_q"],
             wl.causal, k, oi, os_, ws)
    assert ctx.device_status() == 4                   # DSA_ERR_DEVICE_BOUNDS, no trap
    assert ctx.device_status() == 0                   # read and cleared
    gi, gs = oi.cpu().numpy(), os_.cpu().numpy()
    # no row selects a position of the skipped page
    b = np.searchsorted(wl.cu_q, np.arange(wl.Tq), side="right") - 1
    in_bad = (b[:, None] == 0) & (gi >= 192) & (gi < 256)
    assert not in_bad.any()
    cache = U.oracle_cache(wl, fmt)
    o_i, o_s, full = U.oracle_topk(wl, fmt, cache, rows)
    ok, reps = P.compare(rows, gi[rows], gs[rows], o_i, o_s, full, k, fmt)
    assert ok, P.summary(reps)
