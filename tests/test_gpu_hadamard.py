"""GPU parity of the Hadamard-rotated store and the matching query rotation
(the rotation between RoPE and the store: "The Moment of Validation",
section "Input Knowledge Required to Understand This Message"; queries and
keys in the same order: "The Fused Kernel Decision", section "Assumptions and
Their Validity"): stored bytes bit-exact, top-k within the parity rules."""
import numpy as np
import pytest

from oracle import indexer as X
from oracle import store as S
from synth import inputs as I
from tests import gpu_util as U
from tests import parity as P

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ctx():
    import torch
    from dsa_sparse_attention_store_gb300 import Context
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    c = Context(theta=10000.0, eps=1e-6, max_pos=131072)
    c.set_hadamard(True)
    yield c
    c.close()


def _oracle_cache(wl, fmt):
    c = S.new_cache(wl.num_pages, fmt)
    for k, p, q in ((wl.fill_k, wl.fill_pos, wl.fill_seq), (wl.new_k, wl.new_pos, wl.new_seq)):
        S.store(c, fmt, k, p, q, wl.page_table, wl.num_pages, wl.theta, wl.eps, hadamard=True)
    return c


@pytest.mark.parametrize("fmt", [S.FMT_BF16, S.FMT_FP8, S.FMT_FP4])
def test_rotated_store_bitexact(ctx, fmt):
    rng = np.random.default_rng(31)
    T = 700
    x = rng.standard_normal((T, 128)) * np.exp(rng.uniform(-12, 12, (T, 1)))
    x[0] = 0.0
    x[1, :] = 1e-3
    x[1, 40] = 2e3
    wl = I.make_workload("hs", [T], [1], [T], True, 512, seed=32, wid=31)
    wl.new_k = I.to_bf16_bits(x.astype(np.float32))
    d = U.device_workload(wl, fmt, ctx, store_fill=False)
    assert ctx.device_status() == 0
    got = d["cache"].cpu().numpy()
    want = S.new_cache(wl.num_pages, fmt)
    S.store(want, fmt, wl.new_k, wl.new_pos, wl.new_seq, wl.page_table, wl.num_pages, wl.theta,
            wl.eps, hadamard=True)
    gb = U.slot_bytes(got, fmt, wl, wl.new_pos, wl.new_seq)
    wb = U.slot_bytes(want, fmt, wl, wl.new_pos, wl.new_seq)
    bad = np.nonzero(np.any(gb != wb, axis=1))[0]
    assert len(bad) == 0, f"{len(bad)} tokens differ, first at token {bad[0]}"


@pytest.mark.parametrize("fmt", [S.FMT_BF16, S.FMT_FP8, S.FMT_FP4])
@pytest.mark.parametrize("case", ["prefill", "decode"])
def test_rotated_topk_parity(ctx, fmt, case):
    if case == "prefill":
        wl = I.make_workload("hp", [1500, 700, 90], [300, 200, 90], [1500, 700, 90], True, 512,
                             seed=33, wid=32)
    else:
        rng = np.random.default_rng(34)
        L = [int(v) for v in rng.integers(600, 9000, 24)]
        wl = I.make_workload("hd", L, [1] * 24, [1] * 24, True, 512, seed=35, wid=33)
    d = U.device_workload(wl, fmt, ctx)
    gi, gs = U.run_topk(wl, fmt, ctx, d)
    assert ctx.device_status() == 0
    cache = _oracle_cache(wl, fmt)
    rows = np.arange(wl.Tq) if wl.Tq <= 300 else np.linspace(0, wl.Tq - 1, 300).astype(np.int64)
    oi, os_, full = X.index_topk(cache, fmt, wl.page_table, wl.seq_lens, wl.cu_q, wl.q, wl.head_w,
                                 wl.causal, wl.k, rows=rows, return_scores=True, hadamard=True)
    ok, reps = P.compare(rows, gi[rows], gs[rows], oi, os_, full, wl.k, fmt)
    assert ok, P.summary(reps)
