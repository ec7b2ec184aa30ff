"""Pins for the Hadamard-rotated store and the matching query rotation in
the oracle (the rotation between RoPE and the store: "The Moment of
Validation", section "Input Knowledge Required to Understand This Message";
queries and keys in the same order: "The Fused Kernel Decision", section
"Assumptions and Their Validity")."""
import numpy as np
import pytest

from oracle import formats as F
from oracle import indexer as X
from oracle import store as S
from synth import inputs as I


def _bf16(x):
    return F.f32_to_bf16(np.asarray(x, dtype=np.float32))


def test_sylvester_is_the_parity_formula_and_orthogonal():
    # entry (i, j) of the Sylvester matrix is (-1)^popcount(i & j)
    H = X.sylvester()
    i = np.arange(128)
    want = 1.0 - 2.0 * (np.vectorize(lambda v: bin(v).count("1"))(i[:, None] & i[None, :]) % 2)
    assert np.array_equal(H, want)
    assert np.array_equal(H @ H.T, 128.0 * np.eye(128))


def test_butterfly_equals_matrix_exactly_on_small_integers():
    # |x| <= 8: every partial sum is an integer below 2^11, exact in fp32
    rng = np.random.default_rng(1)
    x = rng.integers(-8, 9, (64, 128)).astype(np.float32)
    got = S.wht_f32(x).astype(np.float64)
    assert np.array_equal(got, x.astype(np.float64) @ X.sylvester().T)
    # applying it twice multiplies by 128
    assert np.array_equal(S.wht_f32(S.wht_f32(x)).astype(np.float64), 128.0 * x)


def test_butterfly_one_hot_is_a_matrix_row():
    for j in (0, 1, 5, 64, 127):
        e = np.zeros((1, 128), dtype=np.float32)
        e[0, j] = 3.0
        assert np.array_equal(S.wht_f32(e)[0], 3.0 * X.sylvester()[:, j])


def test_butterfly_rounding_within_fp32_bound():
    # 7 stages of rounded sums: |error| <= 7 * 2^-24 * 128 * max|x| (loose)
    rng = np.random.default_rng(2)
    x = (rng.standard_normal((200, 128)) * np.exp(rng.uniform(-4, 4, (200, 1)))).astype(np.float32)
    got = S.wht_f32(x).astype(np.float64)
    want = x.astype(np.float64) @ X.sylvester().T
    bound = 7 * 2.0 ** -24 * 128 * np.abs(x).max(axis=1, keepdims=True)
    assert np.all(np.abs(got - want) <= bound)


def _store_both(wl, fmt, hadamard):
    cache = S.new_cache(wl.num_pages, fmt)
    for k, p, q in ((wl.fill_k, wl.fill_pos, wl.fill_seq), (wl.new_k, wl.new_pos, wl.new_seq)):
        S.store(cache, fmt, k, p, q, wl.page_table, wl.num_pages, wl.theta, wl.eps, hadamard=hadamard)
    return cache


def test_rotated_store_holds_the_transform_of_the_plain_key():
    wl = I.make_workload("h", [300], [4], [300], True, 16, seed=5, wid=21)
    plain = _store_both(wl, S.FMT_BF16, False)
    rot = _store_both(wl, S.FMT_BF16, True)
    kp = S.read_keys(plain, S.FMT_BF16, wl.page_table[0], 300)
    kr = S.read_keys(rot, S.FMT_BF16, wl.page_table[0], 300)
    # H k within the bf16 rounding of both stores (the plain key rounded to
    # bf16 before the transform, the rotated key after it)
    want = kp @ X.sylvester().T
    tol = 2.0 ** -8 * np.abs(kp).sum(axis=1, keepdims=True) + 2.0 ** -8 * np.abs(want)
    assert np.all(np.abs(kr - want) <= tol)


@pytest.mark.parametrize("fmt", [S.FMT_BF16, S.FMT_FP8])
def test_scores_invariant_under_rotation(fmt):
    # (H q) . (H k) / 128 = q . k: rotated scores equal the plain ones up to
    # the two stores' rounding (bf16: 2^-8 per element; e4m3: 2^-4)
    wl = I.make_workload("h2", [400, 180], [3, 2], [400, 180], True, 32, seed=6, wid=22)
    plain = _store_both(wl, fmt, False)
    rot = _store_both(wl, fmt, True)
    _, _, sp = X.index_topk(plain, fmt, wl.page_table, wl.seq_lens, wl.cu_q, wl.q, wl.head_w,
                            True, 32, return_scores=True)
    _, _, sr = X.index_topk(rot, fmt, wl.page_table, wl.seq_lens, wl.cu_q, wl.q, wl.head_w,
                            True, 32, return_scores=True, hadamard=True)
    rel = 2e-2 if fmt == S.FMT_BF16 else 2.5e-1
    for r in sp:
        m = np.abs(sp[r]).max()
        assert np.abs(sp[r] - sr[r]).max() <= rel * m


def test_bruteforce_tiny_rotated():
    wl = I.make_workload("h3", [90], [3], [90], True, 8, seed=8, wid=23)
    cache = _store_both(wl, S.FMT_BF16, True)
    oi, os_ = X.index_topk(cache, S.FMT_BF16, wl.page_table, wl.seq_lens, wl.cu_q, wl.q,
                           wl.head_w, True, 8, hadamard=True)
    keys = S.read_keys(cache, S.FMT_BF16, wl.page_table[0], 90).tolist()
    Hm = X.sylvester().tolist()
    for r in range(wl.Tq):
        qpos = 90 - 3 + r
        qv = F.bf16_to_f64(wl.q[r]).tolist()
        w = [float(v) for v in wl.head_w[r]]
        # the query heads rotated by the explicit matrix, one head at a time
        qr = [[sum(Hm[i][j] * qv[h][j] for j in range(128)) for i in range(128)] for h in range(64)]
        sc = []
        for p in range(qpos + 1):
            tot = 0.0
            for h in range(64):
                d = 0.0
                for i in range(128):
                    d += qr[h][i] * keys[p][i]
                tot += w[h] * max(d / 128.0, 0.0)
            sc.append(tot)
        order = sorted(range(qpos + 1), key=lambda i: (-sc[i], i))[:8]
        assert [int(v) for v in oi[r] if v >= 0] == order
        assert np.allclose(os_[r, :8], [sc[i] for i in order], rtol=1e-6, atol=1e-6)


def test_rotated_scores_equal_plain_scores_on_exact_keys():
    # keys that are exactly H v (small integers v: every entry of H v is an
    # integer below 2^11, exact in float64): with the query rotated exactly,
    # (H q) . (H v) / 128 = q . v, so the rotated scores equal the plain
    # scores of v to float64 rounding. A query rotation rounded to bf16 (8
    # significant bits) would miss by about 1e-3 of the scores.
    rng = np.random.default_rng(9)
    v = rng.integers(-4, 5, (40, 128)).astype(np.float64)
    keys_rot = v @ X.sylvester().T
    q_bits = I.to_bf16_bits(rng.standard_normal((5, 64, 128)).astype(np.float32))
    w = (rng.standard_normal((5, 64)) / 8).astype(np.float32)
    plain = X.scores(v, q_bits, w)
    rot = X.scores(keys_rot, q_bits, w, hadamard=True)
    scale = np.abs(plain).max(axis=1, keepdims=True)
    assert np.all(np.abs(rot - plain) <= 1e-12 * scale)
