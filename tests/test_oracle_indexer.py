"""Pins for the oracle's scoring and top-k: pure-Python brute force on tiny
inputs, a GEMV special case, full-sort selection with ties, invariants
(weight scaling, page-table permutation, causality, short contexts), the
planted-needle property, and checks that the comparison rules reject
planted mistakes."""
import numpy as np
import pytest

from oracle import formats as F
from oracle import indexer as X
from oracle import store as S
from synth import inputs as I
from tests import parity as P


def _store(wl, fmt):
    cache = S.new_cache(wl.num_pages, fmt)
    S.store(cache, fmt, wl.fill_k, wl.fill_pos, wl.fill_seq, wl.page_table, wl.num_pages,
            wl.theta, wl.eps)
    S.store(cache, fmt, wl.new_k, wl.new_pos, wl.new_seq, wl.page_table, wl.num_pages,
            wl.theta, wl.eps)
    return cache


def _decode_key_by_hand(cache, fmt, page, off):
    if fmt == S.FMT_BF16:
        base = page * 16384 + off * 256
        bits = cache[base:base + 256].view(np.uint16)
        return [float(v) for v in F.bf16_to_f64(bits)]
    if fmt == S.FMT_FP8:
        base = page * 8448 + off * 128
        sc = float(cache[page * 8448 + 8192 + off * 4: page * 8448 + 8196 + off * 4].view("<f4")[0])
        return [float(v) * sc for v in F.e4m3_to_f64(cache[base:base + 128])]
    # fp4: 64 bytes of code pairs (even dimension in the low nibble), then the
    # page's 64 scales; the E2M1 magnitudes written out by hand
    mag = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    base = page * 4352 + off * 64
    sc = float(cache[page * 4352 + 4096 + off * 4: page * 4352 + 4100 + off * 4].view("<f4")[0])
    out = []
    for byte in cache[base:base + 64].tolist():
        for c in (byte & 0xF, byte >> 4):
            out.append((-1.0 if c & 8 else 1.0) * mag[c & 7] * sc)
    return out


@pytest.mark.parametrize("fmt", [S.FMT_BF16, S.FMT_FP8, S.FMT_FP4])
@pytest.mark.parametrize("causal", [True, False])
def test_bruteforce_tiny(fmt, causal):
    wl = I.make_workload("bf", [70, 40], [3, 2], [70, 40], causal, 16, seed=3, wid=11)
    cache = _store(wl, fmt)
    oi, os_ = X.index_topk(cache, fmt, wl.page_table, wl.seq_lens, wl.cu_q, wl.q, wl.head_w,
                           causal, 16)
    for r in range(wl.Tq):
        b = 0 if r < 3 else 1
        nq = 3 if b == 0 else 2
        L = int(wl.seq_lens[b])
        qpos = L - nq + (r - int(wl.cu_q[b]))
        nvis = qpos + 1 if causal else L
        qv = F.bf16_to_f64(wl.q[r]).tolist()
        w = [float(v) for v in wl.head_w[r]]
        sc = []
        for p in range(nvis):
            kv = _decode_key_by_hand(cache, fmt, int(wl.page_table[b, p // 64]), p % 64)
            tot = 0.0
            for h in range(64):
                d = 0.0
                for j in range(128):
                    d += qv[h][j] * kv[j]
                tot += w[h] * max(d, 0.0)
            sc.append(tot)
        order = sorted(range(nvis), key=lambda i: (-sc[i], i))[:16]
        got = [int(v) for v in oi[r] if v >= 0]
        assert got == order
        assert np.allclose(os_[r, :len(order)], [sc[i] for i in order], rtol=1e-6, atol=1e-6)
        assert np.all(oi[r, len(order):] == -1) and np.all(np.isneginf(os_[r, len(order):]))


def test_gemv_special_case():
    # one head with weight 1, positive query and keys: score = K q (a GEMV)
    rng = np.random.default_rng(9)
    n = 50
    keys = np.abs(F.bf16_to_f64(F.f32_to_bf16(rng.standard_normal((n, 128)).astype(np.float32))))
    q = np.zeros((1, 64, 128), np.float32)
    q[0, 5] = np.abs(rng.standard_normal(128))
    qb = F.f32_to_bf16(q)
    w = np.zeros((1, 64), np.float32)
    w[0, 5] = 1.0
    s = X.scores(keys, qb, w)[0]
    qv = F.bf16_to_f64(qb[0, 5])
    want = [sum(float(keys[i, j]) * float(qv[j]) for j in range(128)) for i in range(n)]
    assert np.allclose(s, want, rtol=1e-12)


def test_select_topk_full_sort_with_ties():
    rng = np.random.default_rng(10)
    for n, k in [(0, 4), (3, 4), (4, 4), (100, 7), (1000, 512), (600, 512)]:
        s = rng.integers(-5, 6, n).astype(np.float64)
        idx, val = X.select_topk(s, k)
        want = sorted(range(n), key=lambda i: (-s[i], i))[:k]
        assert idx[:len(want)].tolist() == want
        assert np.all(idx[len(want):] == -1)
        assert np.array_equal(val[:len(want)], s[want])


@pytest.mark.parametrize("fmt", [S.FMT_BF16, S.FMT_FP8, S.FMT_FP4])
def test_invariants(fmt):
    wl = I.make_workload("inv", [700, 333], [40, 9], [700, 333], True, 64, seed=5, wid=12)
    cache = _store(wl, fmt)
    oi, os_ = X.index_topk(cache, fmt, wl.page_table, wl.seq_lens, wl.cu_q, wl.q, wl.head_w,
                           True, 64)
    # scaling w by 4 (exact) scales scores by 4 and keeps the positions
    oi2, os2 = X.index_topk(cache, fmt, wl.page_table, wl.seq_lens, wl.cu_q, wl.q,
                            wl.head_w * np.float32(4), True, 64)
    assert np.array_equal(oi, oi2)
    fin = np.isfinite(os_)
    assert np.array_equal(os2[fin], os_[fin] * 4)
    # permuting the pages (same tokens, another page table) changes nothing
    perm = I.permutation(wl.num_pages, 99, 1)
    pt2 = np.where(wl.page_table >= 0, perm[np.maximum(wl.page_table, 0)], -1).astype(np.int32)
    cache2 = S.new_cache(wl.num_pages, fmt)
    S.store(cache2, fmt, wl.new_k, wl.new_pos, wl.new_seq, pt2, wl.num_pages)
    oi3, os3 = X.index_topk(cache2, fmt, pt2, wl.seq_lens, wl.cu_q, wl.q, wl.head_w, True, 64)
    assert np.array_equal(oi, oi3) and np.array_equal(os_, os3)
    # causal: no selected position beyond the query's own; short contexts take all
    for r in range(wl.Tq):
        qpos = X.query_position(wl.cu_q, wl.seq_lens, r)
        sel = oi[r][oi[r] >= 0]
        assert sel.max() <= qpos
        assert len(sel) == min(64, qpos + 1)
        if qpos + 1 <= 64:
            assert set(sel.tolist()) == set(range(qpos + 1))


def test_non_causal_sees_whole_sequence():
    wl = I.make_workload("nc", [200], [5], [200], False, 8, seed=6, wid=13)
    cache = _store(wl, S.FMT_BF16)
    oi, _, full = X.index_topk(cache, 0, wl.page_table, wl.seq_lens, wl.cu_q, wl.q, wl.head_w,
                               False, 8, return_scores=True)
    for r in range(wl.Tq):
        assert full[r].shape[0] == 200


@pytest.mark.parametrize("fmt", [S.FMT_BF16, S.FMT_FP8])
def test_needle_recall_full_size(fmt):
    # planted needles must be in the top-k of every query that carries u
    wl = I.needle()
    cache = _store(wl, fmt)
    rows = np.array(wl.needle_queries)
    oi, _ = X.index_topk(cache, fmt, wl.page_table, wl.seq_lens, wl.cu_q, wl.q, wl.head_w,
                         True, wl.k, rows=rows)
    for t in range(len(rows)):
        for p in wl.needles:
            assert p in set(oi[t].tolist())


def test_comparator_accepts_identity_and_rejects_mistakes():
    wl = I.make_workload("cmp", [900], [30], [900], True, 64, seed=8, wid=14)
    cache = _store(wl, S.FMT_BF16)
    rows = np.arange(wl.Tq)
    oi, os_, full = X.index_topk(cache, 0, wl.page_table, wl.seq_lens, wl.cu_q, wl.q,
                                 wl.head_w, True, 64, return_scores=True)
    ok, _ = P.compare(rows, oi, os_, oi, os_, full, 64, 0)
    assert ok
    # a dropped head term (a mistake planted in an oracle re-run) is caught
    w2 = wl.head_w.copy()
    w2[:, 7] = 0
    bi, bs = X.index_topk(cache, 0, wl.page_table, wl.seq_lens, wl.cu_q, wl.q, w2, True, 64)
    ok, _ = P.compare(rows, bi, bs, oi, os_, full, 64, 0)
    assert not ok
    # an off-by-one causal mask is caught
    bad = oi.copy()
    for r in range(wl.Tq):
        qpos = X.query_position(wl.cu_q, wl.seq_lens, r)
        bad[r, -1] = qpos + 1
    ok, _ = P.compare(rows, bad, os_, oi, os_, full, 64, 0)
    assert not ok
    # a wrong order is caught
    sw = oi.copy()
    sw[:, [0, 1]] = sw[:, [1, 0]]
    ss = os_.copy()
    ss[:, [0, 1]] = ss[:, [1, 0]]
    ok, _ = P.compare(rows, sw, ss, oi, os_, full, 64, 0)
    assert not ok
