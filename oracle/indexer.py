"""Oracle for the indexer's scoring and top-k selection.

What is computed ("The Crash That Changed Direction", sections "The
Experiment: Why fp32?" and "Assumptions Made and Broken": the indexer scores
every cached index key against the query's index heads with a batched matrix
product, applies a ReLU, and keeps the top-K key positions, K = 512 or 1024):

  s[q, key] = sum_h  w[q, h] * max(0, sum_d q[q, h, d] * k[key, d])

with k the stored key value (bf16, or the e4m3 or e2m1 code times the token's fp32
scale, decoded exactly). The head-weighted sum and the causal rule are the
plainest reading the pages leave open: a query at position p sees keys
0..p of its own sequence (all keys 0..L-1 when not causal). Queries of
sequence b are the last n_q(b) positions: q_pos = L_b - n_q(b) + j.

The contraction is one float64 matrix product (exact bf16 x bf16 products,
float64 sums), the ReLU and head sum are float64, and the result is selected
on those float64 values. Top-k = the first min(k, visible) keys in the order
(score descending, position ascending); unused slots hold -1 / -inf. Scores
are reported rounded to fp32.

With a Hadamard-rotated cache (see oracle.store) the stored key is H k; each
query head is rotated by the same matrix H, exactly (a float64 product with
the +-1 Sylvester matrix: sums of 128 bf16 values), and the dot products are
divided by 128 (exact). The pages require only that queries and keys use the
same order ("The Fused Kernel Decision", section "Assumptions and Their
Validity"); they round nothing on the query side, so the rotated query is
not rounded here either and (H q) . (H k) / 128 = q . k holds up to the
store's rounding of k.
"""
from __future__ import annotations

import numpy as np

from . import formats as F
from . import store as S

H = 64


def sequence_of_rows(cu_q: np.ndarray, rows) -> np.ndarray:
    cu_q = np.asarray(cu_q, dtype=np.int64)
    return np.searchsorted(cu_q, np.asarray(rows, dtype=np.int64), side="right") - 1


def query_position(cu_q, seq_lens, row: int) -> int:
    b = int(sequence_of_rows(cu_q, [row])[0])
    nq = int(cu_q[b + 1] - cu_q[b])
    return int(seq_lens[b]) - nq + (row - int(cu_q[b]))


def visible_count(cu_q, seq_lens, row: int, causal: bool) -> int:
    b = int(sequence_of_rows(cu_q, [row])[0])
    return query_position(cu_q, seq_lens, row) + 1 if causal else int(seq_lens[b])


def sylvester(n: int = S.D) -> np.ndarray:
    """Sylvester Hadamard matrix of order n (entries +-1), float64."""
    h = np.ones((1, 1))
    while h.shape[0] < n:
        h = np.block([[h, h], [h, -h]])
    return h


def scores(keys: np.ndarray, q_bits: np.ndarray, w: np.ndarray, hadamard: bool = False) -> np.ndarray:
    """float64 scores of keys [n,128] for queries q_bits [m,64,128], w [m,64] -> [m,n]."""
    m = q_bits.shape[0]
    qf = F.bf16_to_f64(q_bits).reshape(m * H, S.D)
    if hadamard:
        qf = (qf @ sylvester().T) / 128.0
    dots = keys @ qf.T                                   # [n, m*64]
    dots = np.maximum(dots, 0.0).reshape(keys.shape[0], m, H)
    return np.einsum("nmh,mh->mn", dots, np.asarray(w, dtype=np.float64))


def select_topk(s: np.ndarray, k: int):
    """Positions of the k best (score desc, position asc) and their scores."""
    n = s.shape[0]
    kk = min(k, n)
    idx = np.full(k, -1, dtype=np.int32)
    val = np.full(k, -np.inf, dtype=np.float64)
    if kk == 0:
        return idx, val
    if kk < n:
        kth = np.partition(s, n - kk)[n - kk]
        cand = np.nonzero(s >= kth)[0]
    else:
        cand = np.arange(n)
    order = np.lexsort((cand, -s[cand]))[:kk]
    sel = cand[order]
    idx[:kk] = sel
    val[:kk] = s[sel]
    return idx, val


def index_topk(cache, fmt, page_table, seq_lens, cu_q, q_bits, head_w, causal: bool,
               k: int, rows=None, block: int = 16, return_scores: bool = False,
               hadamard: bool = False):
    """Top-k positions and fp32 scores for the given query rows (all by default).

    Returns (idx [n, k] int32, score [n, k] float32) and, when return_scores,
    a dict row -> float64 score vector over the row's visible keys.
    """
    Tq = q_bits.shape[0]
    rows = np.arange(Tq) if rows is None else np.asarray(rows, dtype=np.int64)
    out_i = np.full((len(rows), k), -1, dtype=np.int32)
    out_s = np.full((len(rows), k), -np.inf, dtype=np.float32)
    full = {}
    seqs = sequence_of_rows(cu_q, rows)
    for b in np.unique(seqs):
        L = int(seq_lens[b])
        keys = S.read_keys(cache, fmt, page_table[b], L)
        mine = np.nonzero(seqs == b)[0]
        for c0 in range(0, len(mine), block):
            blk = mine[c0:c0 + block]
            rr = rows[blk]
            sc = scores(keys, q_bits[rr], head_w[rr], hadamard)
            for t, r in enumerate(rr.tolist()):
                n = visible_count(cu_q, seq_lens, r, causal)
                sv = sc[t, :n]
                i, v = select_topk(sv, k)
                out_i[blk[t]] = i
                out_s[blk[t]] = v.astype(np.float32)
                if return_scores:
                    full[r] = sv.copy()
    if return_scores:
        return out_i, out_s, full
    return out_i, out_s
