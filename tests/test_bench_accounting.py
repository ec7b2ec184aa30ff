"""The bench's roofline accounting: algorithmic bytes and flops per scorer
launch, checked against the workloads' shapes computed independently."""
import importlib.util
import os

import numpy as np

from synth import inputs as I

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench", os.path.join(ROOT, "bench.py"))
    b = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(b)
    return b


def test_long_prefill_flops_is_the_causal_triangle():
    b = _bench()
    wl = I.long_prefill()
    _, flops = b.scorer_algorithmic(wl, 0)
    L = 22528
    assert flops == L * (L + 1) // 2 * 2 * 64 * 128       # 4.158 TFLOP
    assert abs(flops / 1e12 - 4.158) < 1e-3


def test_batched_decode_bytes_per_format():
    b = _bench()
    wl = I.batched_decode()
    keys = int(wl.seq_lens.astype(np.int64).sum())
    pages = int(np.sum((wl.seq_lens.astype(np.int64) + 63) // 64))
    fixed = 64 * (64 * 128 * 2 + 64 * 4) + 4 * pages + 64 * 512 * 8
    for fmt, per_key in ((0, 256), (1, 128 + 4)):
        nbytes, flops = b.scorer_algorithmic(wl, fmt)
        assert nbytes == keys * per_key + fixed
        assert flops == keys * 2 * 64 * 128             # one query per sequence sees all its keys
    # the fp8 launch moves a bit over half the bf16 bytes
    r = b.scorer_algorithmic(wl, 1)[0] / b.scorer_algorithmic(wl, 0)[0]
    assert 0.51 < r < 0.53


def test_whole_job_rate_weak_scaling():
    b = _bench()
    assert b.whole_job_rate(1000, 10, 1, 5.0) == 1000 * 10 / 0.005
    assert b.whole_job_rate(1000, 10, 4, 5.0) == 4 * b.whole_job_rate(1000, 10, 1, 5.0)


def test_needles_selected_counts_each_needle_per_query():
    # three needle queries (rows 1, 2, 3 of four) and two needles at
    # positions 10 and 20: row 1 selected both, row 2 only the first, row 3
    # neither; row 0 is not a needle query and is ignored
    b = _bench()

    class W:
        needle_queries = (1, 2, 3)
        needles = (10, 20)

    out = np.array([[10, 20, 30], [20, 5, 10], [10, 7, -1], [1, 2, 3]], dtype=np.int32)
    rep = b.needles_selected(W(), out)
    assert rep == {"selected_per_needle": [2, 1], "selected": 3, "of": 6}
