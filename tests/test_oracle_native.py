"""Pins for the C++17 oracle (oracle/cpp/dsa_oracle.cpp): its stored bytes
equal the numpy oracle's bit for bit, its scores equal the numpy oracle's to
float64 rounding and a pure-Python brute force on tiny inputs, its top-k is
the full sort of those scores, and the Hadamard query rotation is exact."""
import numpy as np
import pytest

from oracle import formats as F
from oracle import indexer as X
from oracle import native as N
from oracle import store as S
from synth import inputs as I


def _both_caches(wl, fmt, hadamard=False, gamma=None):
    a = S.new_cache(wl.num_pages, fmt)
    b = S.new_cache(wl.num_pages, fmt)
    for k, p, q in ((wl.fill_k, wl.fill_pos, wl.fill_seq), (wl.new_k, wl.new_pos, wl.new_seq)):
        S.store(a, fmt, k, p, q, wl.page_table, wl.num_pages, wl.theta, wl.eps, gamma, hadamard)
        N.store(b, fmt, k, p, q, wl.page_table, wl.num_pages, wl.theta, wl.eps, gamma, hadamard)
    return a, b


@pytest.mark.parametrize("hadamard", [False, True])
@pytest.mark.parametrize("fmt", [S.FMT_BF16, S.FMT_FP8, S.FMT_FP4])
def test_store_bytes_equal_numpy_oracle(fmt, hadamard):
    rng = np.random.default_rng(11)
    T = 1500
    x = rng.standard_normal((T, 128)) * np.exp(rng.uniform(-20, 20, (T, 1)))
    x[0] = 0.0
    x[1] = 1e-38
    x[2, :] = 1e-3
    x[2, 17] = 3e4
    x[3] = rng.standard_normal(128) * np.exp(rng.uniform(-30, 30, 128))
    # the key of the sum-of-squares order golden
    x[4] = 0.0
    x[4, [0, 2, 4, 77, 103, 121]] = [4096, 1, 1, 1, 1, 1]
    wl = I.make_workload("nst", [T, 700], [1, 1], [T, 700], True, 512, seed=12, wid=12)
    wl.new_k[:T] = I.to_bf16_bits(x.astype(np.float32))
    gamma = I.to_bf16_bits(rng.uniform(0.5, 2.0, 128).astype(np.float32))
    a, b = _both_caches(wl, fmt, hadamard, gamma)
    assert np.array_equal(a, b)


def test_store_bytes_equal_numpy_oracle_long_positions():
    wl = I.make_workload("nsl", [131072] * 2, [1] * 2, [300] * 2, True, 1024, seed=0, wid=4)
    wl.fill_pos = wl.fill_pos[:0]
    wl.fill_seq = wl.fill_seq[:0]
    wl.fill_k = wl.fill_k[:0]
    for fmt in (S.FMT_BF16, S.FMT_FP8, S.FMT_FP4):
        a, b = _both_caches(wl, fmt)
        assert np.array_equal(a, b)


def test_store_rejects_bad_page():
    pt = np.array([[0, 5]], np.int32)
    cache = S.new_cache(2, S.FMT_BF16)
    with pytest.raises(ValueError):
        N.store(cache, S.FMT_BF16, F.f32_to_bf16(np.ones((1, 128), np.float32)), np.array([64]),
                np.array([0]), pt, 2)


def _compare_topk(wl, fmt, hadamard=False, k=None):
    k = wl.k if k is None else k
    a, b = _both_caches(wl, fmt, hadamard)
    assert np.array_equal(a, b)
    oi, os_, full = X.index_topk(a, fmt, wl.page_table, wl.seq_lens, wl.cu_q, wl.q, wl.head_w,
                                 wl.causal, k, return_scores=True, hadamard=hadamard)
    ni, ns, nfull = N.index_topk(b, fmt, wl.page_table, wl.seq_lens, wl.cu_q, wl.q, wl.head_w,
                                 wl.causal, k, return_scores=True, hadamard=hadamard)
    assert np.array_equal(oi, ni)
    fin = np.isfinite(os_)
    assert np.array_equal(fin, np.isfinite(ns))
    assert np.allclose(ns[fin], os_[fin], rtol=1e-6, atol=0)     # fp32-rounded copies
    for r, s in full.items():
        m = max(np.abs(s).max(initial=0.0), 1e-300)
        assert nfull[r].shape == s.shape
        assert np.all(np.abs(nfull[r] - s) <= 1e-12 * m)


@pytest.mark.parametrize("fmt", [S.FMT_BF16, S.FMT_FP8, S.FMT_FP4])
def test_topk_equals_numpy_oracle_prefill(fmt):
    wl = I.make_workload("ntp", [300, 777, 129], [300, 40, 129], [300, 777, 129], True, 128,
                         seed=13, wid=13)
    _compare_topk(wl, fmt)


@pytest.mark.parametrize("fmt", [S.FMT_BF16, S.FMT_FP8, S.FMT_FP4])
def test_topk_equals_numpy_oracle_decode_non_causal(fmt):
    wl = I.make_workload("ntd", [2000, 700, 64], [1, 3, 2], [1, 3, 2], False, 512, seed=14, wid=14)
    _compare_topk(wl, fmt)


@pytest.mark.parametrize("fmt", [S.FMT_BF16, S.FMT_FP8, S.FMT_FP4])
def test_topk_equals_numpy_oracle_hadamard(fmt):
    wl = I.make_workload("nth", [600, 200], [5, 3], [600, 200], True, 64, seed=15, wid=15)
    _compare_topk(wl, fmt, hadamard=True)


def test_topk_ties_broken_by_position():
    wl = I.make_workload("ntz", [900], [3], [900], True, 512, seed=16, wid=16)
    wl.q[:] = 0
    cache = N.new_cache(wl.num_pages, 0)
    N.store(cache, 0, wl.new_k, wl.new_pos, wl.new_seq, wl.page_table, wl.num_pages)
    ni, ns = N.index_topk(cache, 0, wl.page_table, wl.seq_lens, wl.cu_q, wl.q, wl.head_w, True, 512)
    assert np.array_equal(ni, np.tile(np.arange(512, dtype=np.int32), (3, 1)))
    assert np.all(ns == 0)


def test_bruteforce_tiny():
    # pure-Python scores and a full sort, on 70 keys and 3 queries (signed w)
    wl = I.make_workload("ntb", [70], [3], [70], True, 16, seed=17, wid=17)
    for fmt in (S.FMT_BF16, S.FMT_FP8, S.FMT_FP4):
        cache = N.new_cache(wl.num_pages, fmt)
        N.store(cache, fmt, wl.new_k, wl.new_pos, wl.new_seq, wl.page_table, wl.num_pages)
        ni, ns, full = N.index_topk(cache, fmt, wl.page_table, wl.seq_lens, wl.cu_q, wl.q, wl.head_w,
                                    True, 16, return_scores=True)
        keys = S.read_keys(cache, fmt, wl.page_table[0], 70).tolist()
        for r in range(3):
            qpos = 67 + r
            qv = F.bf16_to_f64(wl.q[r]).tolist()
            w = [float(v) for v in wl.head_w[r]]
            sc = []
            for p in range(qpos + 1):
                tot = 0.0
                for h in range(64):
                    d = sum(qv[h][i] * keys[p][i] for i in range(128))
                    tot += w[h] * max(d, 0.0)
                sc.append(tot)
            assert np.allclose(full[r], sc, rtol=0, atol=1e-12 * max(abs(v) for v in sc))
            order = sorted(range(qpos + 1), key=lambda i: (-sc[i], i))[:16]
            assert [int(v) for v in ni[r]] == order


def test_hadamard_rotation_exact_on_exact_keys():
    # a bf16 cache holding v (entries -1, 0, 1) and one holding H v (integers
    # of magnitude <= 128, exact in bf16): the rotated scores of the second
    # equal the plain scores of the first to float64 rounding
    rng = np.random.default_rng(18)
    L = 100
    v = rng.integers(-1, 2, (L, 128)).astype(np.float64)
    hv = v @ X.sylvester().T
    wl = I.make_workload("nhx", [L], [4], [L], True, 32, seed=18, wid=18)
    pt = wl.page_table[0]

    def cache_of(vals):
        c = N.new_cache(wl.num_pages, 0)
        view = c.reshape(-1, 64, 256)
        for p in range(L):
            view[pt[p // 64], p % 64] = F.f32_to_bf16(vals[p].astype(np.float32)).view(np.uint8)
        return c
    _, _, plain = N.index_topk(cache_of(v), 0, wl.page_table, wl.seq_lens, wl.cu_q, wl.q, wl.head_w,
                               True, 32, return_scores=True)
    _, _, rot = N.index_topk(cache_of(hv), 0, wl.page_table, wl.seq_lens, wl.cu_q, wl.q, wl.head_w,
                             True, 32, return_scores=True, hadamard=True)
    for r in plain:
        m = np.abs(plain[r]).max()
        assert np.all(np.abs(rot[r] - plain[r]) <= 1e-12 * m)


def test_threads_reported():
    assert N.threads() >= 1
