"""Seeded synthetic inputs for the DSA indexer workloads.

This module is shared by the tests, the bench and the oracle harness. It
draws random numbers and lays them out in the shapes the indexer consumes;
it holds none of the indexer's own arithmetic (no normalisation, no
quantisation, no scoring, and neither side calls it to compute a result).
The one rotation here is the needle workload's: to plant a key that points
along a chosen direction after the store, the raw row is that direction
turned back by its RoPE angle (an input construction in float64).
Everything is counter-based, so the same (seed, stream, index) gives the
same value on any machine.

Generator: SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014): state_i = base + (i + 1) * 0x9E3779B97F4A7C15,
output = mix(state_i) with the published 30/27/31 xor-shift multipliers.
Normals use the Box-Muller transform on two 53-bit uniforms.

Workloads follow the shapes the pages describe (head_dim 128 index keys,
64 index heads, 64-token pages, top-k 512 or 1024; contexts of about 2K to
16K tokens for decode, 10498 and 22528 tokens for prefill, 131072 for long
decode). Values are N(0, 1) unless stated.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
M1 = np.uint64(0xBF58476D1CE4E5B9)
M2 = np.uint64(0x94D049BB133111EB)

D = 128          # index head_dim
H = 64           # index heads
PAGE = 64        # tokens per cache page

# tensor stream ids (mixed with the workload id)
S_KFILL, S_KNEW, S_Q, S_W, S_CTX, S_PERM, S_U, S_NOISE, S_GAMMA = range(1, 10)


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * M1
    z = (z ^ (z >> np.uint64(27))) * M2
    return z ^ (z >> np.uint64(31))


def _base(seed: int, stream: int) -> np.uint64:
    s = np.array([(seed & 0xFFFFFFFF) << 32 | (stream & 0xFFFFFFFF)], dtype=np.uint64)
    return _mix(s + GOLDEN)[0]


def raw_u64(n: int, seed: int, stream: int, offset: int = 0) -> np.ndarray:
    """n SplitMix64 outputs of stream (seed, stream), starting at counter offset."""
    with np.errstate(over="ignore"):
        i = np.arange(offset + 1, offset + n + 1, dtype=np.uint64)
        return _mix(_base(seed, stream) + i * GOLDEN)


def uniform(n: int, seed: int, stream: int, offset: int = 0) -> np.ndarray:
    """Uniform float64 in [0, 1) from the top 53 bits."""
    return (raw_u64(n, seed, stream, offset) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def normal(n: int, seed: int, stream: int, chunk: int = 1 << 23) -> np.ndarray:
    """n N(0,1) float32 values (Box-Muller; pair i uses counters 2i and 2i+1)."""
    out = np.empty(n, dtype=np.float32)
    npairs = (n + 1) // 2
    for p0 in range(0, npairs, chunk):
        p1 = min(npairs, p0 + chunk)
        u = uniform(2 * (p1 - p0), seed, stream, offset=2 * p0)
        u1 = 1.0 - u[0::2]                      # (0, 1]
        u2 = u[1::2]
        r = np.sqrt(-2.0 * np.log(u1))
        z = np.empty(2 * (p1 - p0), dtype=np.float64)
        z[0::2] = r * np.cos(2.0 * math.pi * u2)
        z[1::2] = r * np.sin(2.0 * math.pi * u2)
        lo = 2 * p0
        hi = min(n, 2 * p1)
        out[lo:hi] = z[: hi - lo]
    return out


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (round to nearest even); input packing only."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def permutation(n: int, seed: int, stream: int) -> np.ndarray:
    return np.argsort(raw_u64(n, seed, stream), kind="stable").astype(np.int64)


def randint(n: int, lo: int, hi: int, seed: int, stream: int) -> np.ndarray:
    """Integers uniform in [lo, hi] inclusive."""
    return (lo + np.floor(uniform(n, seed, stream) * (hi - lo + 1))).astype(np.int64)


@dataclasses.dataclass
class Workload:
    """One synthetic indexer workload, host arrays only.

    Cache:  num_pages pages of 64 token slots; page_table[b, j] is the page
            holding positions 64j..64j+63 of sequence b (-1 when unused).
    Store:  fill_* tokens are written before the timed step; new_* tokens are
            written by the step itself. k_raw rows are bf16 bit patterns.
    Query:  q [Tq, 64, 128] bf16 bits, head_w [Tq, 64] float32; the queries of
            sequence b are rows cu_q[b]..cu_q[b+1]-1, at positions
            seq_lens[b] - n_q(b) + j.
    """
    name: str
    seq_lens: np.ndarray          # [B] int32, context length after the step's store
    cu_q: np.ndarray              # [B+1] int32
    page_table: np.ndarray        # [B, max_pages] int32
    num_pages: int
    fill_k: np.ndarray            # [Tf, 128] uint16 (bf16 bits)
    fill_pos: np.ndarray          # [Tf] int32
    fill_seq: np.ndarray          # [Tf] int32
    new_k: np.ndarray             # [Tn, 128] uint16
    new_pos: np.ndarray           # [Tn] int32
    new_seq: np.ndarray           # [Tn] int32
    q: np.ndarray                 # [Tq, 64, 128] uint16
    head_w: np.ndarray            # [Tq, 64] float32
    causal: bool
    k: int
    theta: float = 10000.0
    eps: float = 1e-6
    needles: tuple = ()           # positions of planted needle keys
    needle_queries: tuple = ()    # query rows that carry the needle direction

    @property
    def B(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def Tq(self) -> int:
        return int(self.q.shape[0])

    @property
    def max_pages(self) -> int:
        return int(self.page_table.shape[1])

    @property
    def max_pos(self) -> int:
        return int(self.seq_lens.max())

    def key_scores(self) -> int:
        """Sum over queries of the number of visible keys."""
        tot = 0
        for b in range(self.B):
            nq = int(self.cu_q[b + 1] - self.cu_q[b])
            L = int(self.seq_lens[b])
            if self.causal:
                tot += sum(L - nq + j + 1 for j in range(nq))
            else:
                tot += nq * L
        return tot


def _paging(seq_lens: np.ndarray, seed: int, wid: int, spare: int = 0):
    npg = [(int(L) + PAGE - 1) // PAGE for L in seq_lens]
    num_pages = sum(npg) + spare
    perm = permutation(num_pages, seed, wid * 16 + S_PERM)
    max_pages = max(npg)
    pt = np.full((len(seq_lens), max_pages), -1, dtype=np.int32)
    c = 0
    for b, n in enumerate(npg):
        pt[b, :n] = perm[c:c + n]
        c += n
    return pt, num_pages


def _tokens(seq_lens, starts, ends):
    pos, seq = [], []
    for b in range(len(seq_lens)):
        p = np.arange(starts[b], ends[b], dtype=np.int32)
        pos.append(p)
        seq.append(np.full(p.shape, b, dtype=np.int32))
    if not pos:
        return np.zeros(0, np.int32), np.zeros(0, np.int32)
    return np.concatenate(pos), np.concatenate(seq)


def make_workload(name: str, seq_lens, n_q, n_new, causal: bool, k: int,
                  seed: int = 0, wid: int = 0, w_abs: bool = False) -> Workload:
    """Generic workload: sequence b has seq_lens[b] tokens after the step, the
    last n_new[b] of which are stored by the step; its last n_q[b] tokens are
    queries. head_w ~ N(0,1)/8 (|N(0,1)|/8 when w_abs)."""
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    n_q = np.asarray(n_q, dtype=np.int32)
    n_new = np.asarray(n_new, dtype=np.int32)
    B = len(seq_lens)
    pt, num_pages = _paging(seq_lens, seed, wid)
    fill_pos, fill_seq = _tokens(seq_lens, np.zeros(B, np.int64), seq_lens - n_new)
    new_pos, new_seq = _tokens(seq_lens, seq_lens - n_new, seq_lens)
    Tf, Tn = fill_pos.shape[0], new_pos.shape[0]
    fill_k = to_bf16_bits(normal(Tf * D, seed, wid * 16 + S_KFILL)).reshape(Tf, D)
    new_k = to_bf16_bits(normal(Tn * D, seed, wid * 16 + S_KNEW)).reshape(Tn, D)
    Tq = int(n_q.sum())
    q = to_bf16_bits(normal(Tq * H * D, seed, wid * 16 + S_Q)).reshape(Tq, H, D)
    w = normal(Tq * H, seed, wid * 16 + S_W).reshape(Tq, H)
    if w_abs:
        w = np.abs(w)
    w = (w / np.float32(8.0)).astype(np.float32)
    cu_q = np.zeros(B + 1, dtype=np.int32)
    cu_q[1:] = np.cumsum(n_q)
    return Workload(name=name, seq_lens=seq_lens, cu_q=cu_q, page_table=pt,
                    num_pages=num_pages, fill_k=fill_k, fill_pos=fill_pos,
                    fill_seq=fill_seq, new_k=new_k, new_pos=new_pos,
                    new_seq=new_seq, q=q, head_w=w, causal=causal, k=k)


# ---------------------------------------------------------------- the five workloads

def tiny_prefill(L: int = 1024, k: int = 512, seed: int = 0) -> Workload:
    """1 sequence of L tokens, all stored by the step, all scored causally."""
    return make_workload(f"tiny_prefill_L{L}", [L], [L], [L], True, k, seed, wid=0)


def batched_decode(B: int = 64, lo: int = 2048, hi: int = 16384, k: int = 512,
                   seed: int = 0) -> Workload:
    """B sequences, one query each; context uniform in [lo, hi]; the step
    stores the query token's key (the last position) and scores it."""
    ctx = randint(B, lo, hi, seed, 1 * 16 + S_CTX).astype(np.int32)
    return make_workload(f"batched_decode_B{B}", ctx, np.ones(B), np.ones(B), True, k,
                         seed, wid=1)


def long_prefill(L: int = 22528, k: int = 512, seed: int = 0) -> Workload:
    return make_workload(f"long_prefill_L{L}", [L], [L], [L], True, k, seed, wid=2)


def long_decode(B: int = 8, L: int = 131072, n_new: int = 256, n_q: int = 8,
                k: int = 1024, seed: int = 0) -> Workload:
    """B sequences at L tokens; the step appends n_new tokens per sequence and
    scores the last n_q tokens of each."""
    return make_workload(f"long_decode_B{B}_L{L}", [L] * B, [n_q] * B, [n_new] * B,
                         True, k, seed, wid=4)


NEEDLE_NORM = 11.3
NEEDLE_DEPTHS = (0.05, 0.25, 0.50, 0.75, 0.95)


def needle_direction(seed: int = 0) -> np.ndarray:
    """The fixed random direction u (float64 [128], norm 11.3)."""
    g = normal(D, seed, 3 * 16 + S_U).astype(np.float64)
    return g * (NEEDLE_NORM / np.linalg.norm(g))


def needle(L: int = 10498, n_last: int = 64, k: int = 512, seed: int = 0,
           w_abs: bool = True) -> Workload:
    """Needle recall: Q and K ~ N(0,1); at depths 5/25/50/75/95 % a key is
    replaced so that its stored (normalised, rotated) value points along
    0.8 u + 0.2 xi; the last n_last queries get +u on every head.

    The needle is defined in the stored key space. Because the store rotates
    each key by its position, the raw row is the needle vector rotated back
    by that position (RoPE's pairing: dims i and i+64, angle pos*theta^(-i/64)),
    so that after the store it points along the needle direction again.
    """
    wl = make_workload(f"needle_L{L}", [L], [L], [L], True, k, seed, wid=3, w_abs=w_abs)
    u = needle_direction(seed)
    depths = tuple(int(math.floor(f * L)) for f in NEEDLE_DEPTHS)
    noise = normal(len(depths) * D, seed, 3 * 16 + S_NOISE).astype(np.float64).reshape(-1, D)
    kf = bf16_bits_to_f32(wl.new_k).astype(np.float64)
    half = D // 2
    for n, pos in enumerate(depths):
        v = 0.8 * u + 0.2 * noise[n]
        ang = np.array([pos * math.pow(wl.theta, -(2.0 * i) / D) for i in range(half)])
        c, s = np.cos(ang), np.sin(ang)
        a, b = v[:half], v[half:]
        # inverse rotation (angle -ang)
        kf[pos, :half] = a * c + b * s
        kf[pos, half:] = b * c - a * s
    wl.new_k = to_bf16_bits(kf.astype(np.float32))
    qf = bf16_bits_to_f32(wl.q).astype(np.float64)
    rows = tuple(range(L - n_last, L))
    qf[L - n_last:, :, :] += u[None, None, :]
    wl.q = to_bf16_bits(qf.astype(np.float32)).reshape(wl.q.shape)
    wl.needles = depths
    wl.needle_queries = rows
    return wl


WORKLOADS = {
    "tiny_prefill": tiny_prefill,
    "batched_decode": batched_decode,
    "long_prefill": long_prefill,
    "needle": needle,
    "long_decode": long_decode,
}
