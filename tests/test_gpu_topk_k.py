"""GPU parity of top-k for any k up to 2048 and of the cache-slot output
(the selected tokens feed the sparse attention: "The Crash That Changed
Direction", section "The Experiment: Why fp32?")."""
import numpy as np
import pytest

from oracle import store as S
from synth import inputs as I
from tests import gpu_util as U
from tests import parity as P

pytestmark = pytest.mark.gpu


def _ctx(**opts):
    import torch
    from dsa_sparse_attention_store_gb300 import Context
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    c = Context(theta=10000.0, eps=1e-6, max_pos=131072)
    if opts.get("slots"):
        c.set_slot_output(True)
    return c


@pytest.fixture(scope="module")
def ctx():
    c = _ctx()
    yield c
    c.close()


@pytest.fixture(scope="module")
def ctx_slots():
    c = _ctx(slots=True)
    yield c
    c.close()


def _decode():
    rng = np.random.default_rng(41)
    L = [int(v) for v in rng.integers(300, 7000, 20)] + [20000, 15000]
    return I.make_workload("kd", L, [1] * len(L), [1] * len(L), True, 512, seed=42, wid=41)


def _prefill():
    return I.make_workload("kp", [3300, 260], [260, 120], [3300, 260], True, 512, seed=43, wid=42)


@pytest.mark.parametrize("k,fmt", [(1, S.FMT_BF16), (100, S.FMT_FP8), (700, S.FMT_FP4), (1500, S.FMT_FP8),
                                   (2048, S.FMT_BF16), (2048, S.FMT_FP4)])
@pytest.mark.parametrize("shape", ["decode", "prefill"])
def test_any_k(ctx, shape, k, fmt):
    # k above 1024 runs the top-2048 selection (in one-query tiles, for the
    # prefill shape too); the contexts here are long enough that 2048 of the
    # visible keys are selected, not all of them
    wl = _decode() if shape == "decode" else _prefill()
    d = U.device_workload(wl, fmt, ctx)
    gi, gs = U.run_topk(wl, fmt, ctx, d, k)
    assert ctx.device_status() == 0
    assert gi.shape == (wl.Tq, k)
    cache = U.oracle_cache(wl, fmt)
    rows = np.arange(wl.Tq) if wl.Tq <= 200 else np.linspace(0, wl.Tq - 1, 200).astype(np.int64)
    oi, os_, full = U.oracle_topk(wl, fmt, cache, rows, k)
    ok, reps = P.compare(rows, gi[rows], gs[rows], oi, os_, full, k, fmt)
    assert ok, P.summary(reps)


@pytest.mark.parametrize("fmt", [S.FMT_BF16, S.FMT_FP8, S.FMT_FP4])
@pytest.mark.parametrize("shape", ["decode", "prefill"])
def test_slot_output(ctx, ctx_slots, shape, fmt):
    wl = _decode() if shape == "decode" else _prefill()
    d = U.device_workload(wl, fmt, ctx)
    pi, ps = U.run_topk(wl, fmt, ctx, d)
    si, ss = U.run_topk(wl, fmt, ctx_slots, d)
    assert ctx.device_status() == 0 and ctx_slots.device_status() == 0
    # same selection and scores; each slot is page_table[b][pos / 64] * 64 + pos % 64
    assert np.array_equal(ps, ss)
    b = np.searchsorted(wl.cu_q, np.arange(wl.Tq), side="right") - 1
    pt = wl.page_table.astype(np.int64)
    want = np.where(pi >= 0, pt[b[:, None], np.maximum(pi, 0) // 64] * 64 + np.maximum(pi, 0) % 64, -1)
    assert np.array_equal(si, want)
