// The DSA indexer's scorer: configuration, device code and launch template,
// shared by the translation units that instantiate it (topk.cu for bf16
// caches, topk_fp8.cu and topk_fp4.cu), so that the kernel variants of the
// three cache formats compile in parallel. What it computes and how is
// described at the top of topk.cu.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <algorithm>

#include "internal.cuh"
#include "ptx.cuh"

namespace dsa {
namespace sc {

constexpr int kH = 64;
constexpr int kD = 128;
constexpr int kTile = 128;  // keys per MMA tile = 2 pages
constexpr int kPageBytesFp8 = 64 * 128 + 64 * 4;
constexpr int kPageBytesFp4 = 64 * 64 + 64 * 4;
// a query tile split over at most this many CTAs merges its pieces' sorted
// lists pairwise; one split over more (selecting more than 512 keys) selects
// once over their union
constexpr int kFewPieces = 4;

// The work is split evenly in units: a query tile with n key tiles costs
// n + ovh units, ovh standing for its fixed costs (query load, final merge
// or selection and sort), so CTAs that get many short query tiles get fewer.
struct PlanHdr {
  int qtot;         // query tiles
  int Ge;           // CTAs with work: min(grid, total units)
  long long total;  // units over all query tiles
  int ovh;          // units charged per query tile on top of its key tiles
};

// Per query tile: {b, row0, nrows, ntile} and {L, qpos0, 0, 0} where qpos0 is
// the position of the tile's first query.
struct WsLayout {
  size_t hdr, meta, prefix, counters, rec, partials, gthr, total;
  int QT, G, qtmax, NG;
};

inline size_t up256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

constexpr int kMaxGrid = 1024;  // most CTAs of the scorer (one per SM)

// Tiles of several queries of one sequence when the queries outnumber the
// sequences: four, or two when the query carries one more term (the
// Hadamard rotation), whose larger query tile only fits beside the operand
// ring at half the width; one-query tiles for decode and for selections of
// 2048 keys, whose candidate buffer only fits there.
inline int pick_qt(int Tq, int B, bool hadamard, int ksel) {
  if (ksel > 1024 || Tq < 2 * B) return 1;
  if (hadamard) return Tq >= 2 ? 2 : 1;
  return Tq >= 4 ? 4 : 1;
}
// selection size (the sorting networks' K) for an output of k entries
inline int select_size(int k) { return k <= 512 ? 512 : (k <= 1024 ? 1024 : 2048); }

inline WsLayout ws_layout(int num_sms, int Tq, int B, int k, bool hadamard) {
  WsLayout L{};
  L.QT = pick_qt(Tq, B, hadamard, k);
  L.NG = L.QT;  // top-k groups (one per query): merge counters per (query tile, group)
  L.G = std::min(num_sms, kMaxGrid);
  L.qtmax = (Tq + L.QT - 1) / L.QT + B;
  size_t o = 0;
  L.hdr = o;
  o += 256;
  L.meta = o;
  o = up256(o + static_cast<size_t>(L.qtmax) * 32);
  L.prefix = o;
  o = up256(o + static_cast<size_t>(L.qtmax + 1) * 8);
  L.counters = o;
  o = up256(o + static_cast<size_t>(L.qtmax) * L.NG * 4);
  L.rec = o;
  o = up256(o + static_cast<size_t>(L.G) * 4);
  L.partials = o;
  o = up256(o + static_cast<size_t>(2) * L.G * L.QT * k * 8);
  L.gthr = o;  // per query row: the largest running k-th key published by its pieces
  o = up256(o + static_cast<size_t>(Tq) * 8);
  L.total = o;
  return L;
}

// ------------------------------------------------------------------ ordering keys
// 64-bit key: ordered fp32 score in the high word, ~position in the low word,
// so that a larger key means (higher score, then lower position). Key 0 is
// below every real key and marks an empty slot.
__device__ __forceinline__ uint64_t make_key(float s, int pos) {
  const uint32_t u = __float_as_uint(s + 0.0f);  // -0 -> +0
  const uint32_t o = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return (static_cast<uint64_t>(o) << 32) | static_cast<uint32_t>(~static_cast<uint32_t>(pos));
}
__device__ __forceinline__ float key_score(uint64_t key) {
  const uint32_t o = static_cast<uint32_t>(key >> 32);
  const uint32_t u = (o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o;
  return __uint_as_float(u);
}
__device__ __forceinline__ int key_pos(uint64_t key) {
  return static_cast<int>(~static_cast<uint32_t>(key));
}

// ------------------------------------------------------------------ block scans (1024 threads)
template <typename T>
__device__ T block_excl_scan(T v, T* sm, T& total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  T x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const T y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sm[w] = x;
  __syncthreads();
  if (w == 0) {
    T s = sm[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const T y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    sm[lane] = s;
  }
  __syncthreads();
  const T excl = x - v + (w > 0 ? sm[w - 1] : T(0));
  total = sm[31];
  __syncthreads();
  return excl;
}

__device__ __forceinline__ long long range_start(int c, long long total, int G) {
  return static_cast<long long>(c) * total / G;
}

__device__ __forceinline__ int owner_of(long long gtile, long long total, int G) {
  int c = static_cast<int>(gtile * G / total);
  while (c + 1 < G && range_start(c + 1, total, G) <= gtile) ++c;
  while (c > 0 && range_start(c, total, G) > gtile) --c;
  return c;
}
// A CTA keeps at most two partial lists: slot 2c for the query tile its
// range starts in, 2c+1 for the one it ends in.
__device__ __forceinline__ int partial_slot(int c, long long qt_start, long long total, int G) {
  return range_start(c, total, G) >= qt_start ? 2 * c : 2 * c + 1;
}

// One CTA. Per-sequence sizes and query-tile offsets live in shared memory
// (B <= kMaxSeqs), so the only global round trips are the input loads and
// the final writes.
constexpr int kMaxSeqs = 16384;

// ------------------------------------------------------------------ query preparation
// The query tile arrives in shared memory as the caller's bf16 rows (two
// 64-column halves of N rows, 128-byte swizzle). Where it is not used as it
// is, one warp turns a (query, head) row of 128 values into its tensor-core
// terms in place, each lane taking 4 consecutive values:
//
// fp8 and fp4 caches: the e4m3 keys (stored, or widened from e2m1) go to the
// tensor cores as they are (kind::f8f6f4, e4m3 x e4m3, both operands of one
// type), so the row is
// split into e4m3 terms whose sum is the query: a power-of-two scale 2^e
// puts the row's largest magnitude in [2^7, 2^8); t1 = e4m3(2^e q),
// t2 = e4m3(2^e q - t1) (t3 likewise), each difference exact in fp32. A
// bf16 value has 8 significant bits and an e4m3 normal 4, so two terms give
// 2^e q exactly whenever the remainder is not below e4m3's subnormal step,
// i.e. for every value at least 2^-10 of the row's maximum; smaller ones
// keep an absolute error of at most 2^-10 (scaled units). Products of e4m3
// operands are exact in the fp32 accumulator, and the row's head weight
// w' = w * 2^-e undoes the scale after the ReLU (relu(2^e x) = 2^e relu(x)).
//
// With the Hadamard rotation on, the row is first rotated by the same
// unnormalised Walsh-Hadamard transform as the stored keys (fp32 butterflies
// in the store's order: h = 1, 2 inside a lane's 4 values, h = 4 .. 64
// between lanes l and l ^ (h/4)); the rotated values are sums of up to 128
// bf16 values and carry more bits than one bf16 or two e4m3 terms hold, so
// bf16 caches take hi = bf16(x) and lo = bf16(x - hi) (16 significant bits)
// and fp8 and fp4 caches three e4m3 terms (12 significant bits); w' carries a
// further 2^-7 (the transform's gain 128 on the dot product).
//
// Terms follow one another in shared memory: a bf16 term as two 64-column
// halves, an e4m3 term as one 128-byte row, all of N rows. The first two
// e4m3 terms of row r, and the hi term, take the same two 128-byte lines as
// the row's bf16 values, so a warp converts its row in place once every
// lane has read it.
template <bool E4M3, bool HAD, int N, int NQ>
__device__ __forceinline__ void prep_row(uint8_t* sQ, int r, float* sw, int lane) {
  const int half = lane >> 4, chunk = (lane & 15) >> 1;  // values 4l..4l+3
  const int in_off = r * 128 + ((chunk ^ (r & 7)) << 4) + (lane & 1) * 8;
  const uint2 v = *reinterpret_cast<const uint2*>(sQ + half * (N * 128) + in_off);
  float x[4] = {__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xFFFF0000u),
                __uint_as_float(v.y << 16), __uint_as_float(v.y & 0xFFFF0000u)};
  if constexpr (HAD) {
#pragma unroll
    for (int h = 1; h < 4; h <<= 1) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if ((e & h) == 0) {
          const float a = x[e], b = x[e + h];
          x[e] = __fadd_rn(a, b);
          x[e + h] = __fsub_rn(a, b);
        }
      }
    }
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float p = __shfl_xor_sync(0xffffffffu, x[e], m);
        x[e] = (lane & m) ? __fsub_rn(p, x[e]) : __fadd_rn(x[e], p);
      }
    }
  }
  constexpr int kGain = HAD ? 7 : 0;  // log2 of the rotation's gain on q . k
  if constexpr (!E4M3) {
    // bf16 caches (only with the rotation): hi in place, lo as the next term
    const __nv_bfloat162 h0 = __floats2bfloat162_rn(x[0], x[1]);
    const __nv_bfloat162 h1 = __floats2bfloat162_rn(x[2], x[3]);
    const float2 f0 = __bfloat1622float2(h0), f1 = __bfloat1622float2(h1);
    const __nv_bfloat162 l0 = __floats2bfloat162_rn(__fsub_rn(x[0], f0.x), __fsub_rn(x[1], f0.y));
    const __nv_bfloat162 l1 = __floats2bfloat162_rn(__fsub_rn(x[2], f1.x), __fsub_rn(x[3], f1.y));
    uint2 hi2, lo2;
    hi2.x = *reinterpret_cast<const uint32_t*>(&h0);
    hi2.y = *reinterpret_cast<const uint32_t*>(&h1);
    lo2.x = *reinterpret_cast<const uint32_t*>(&l0);
    lo2.y = *reinterpret_cast<const uint32_t*>(&l1);
    __syncwarp();
    *reinterpret_cast<uint2*>(sQ + half * (N * 128) + in_off) = hi2;
    *reinterpret_cast<uint2*>(sQ + 2 * (N * 128) + half * (N * 128) + in_off) = lo2;
    if (lane == 0) sw[r] = sw[r] * (1.0f / (1 << kGain));
  } else {
    float m = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    // e such that m * 2^e lies in [2^7, 2^8): from m's exponent field (a
    // subnormal or zero row takes the largest e kept normal, 126); both 2^e
    // and 2^-e are exact fp32 powers of two built from their bits
    const int be = (__float_as_int(m) >> 23) & 0xFF;
    const int e = be == 0 ? 126 : min(134 - be, 126);
    const float up = __int_as_float((127 + e) << 23);
    const float down = __int_as_float(max(127 - e - kGain, 1) << 23);  // 2^-(e + gain), at least 2^-126
    uint32_t t[NQ] = {};
#pragma unroll
    for (int p = 0; p < 2; ++p) {
      float y0 = x[2 * p] * up, y1 = x[2 * p + 1] * up;
#pragma unroll
      for (int term = 0; term < NQ; ++term) {
        const __nv_fp8x2_storage_t q2 = __nv_cvt_float2_to_fp8x2(make_float2(y0, y1), __NV_SATFINITE, __NV_E4M3);
        t[term] |= static_cast<uint32_t>(q2) << (16 * p);
        const __half2_raw qh = __nv_cvt_fp8x2_to_halfraw2(q2, __NV_E4M3);
        y0 = __fsub_rn(y0, __half2float(__ushort_as_half(qh.x)));  // exact: the remainder
        y1 = __fsub_rn(y1, __half2float(__ushort_as_half(qh.y)));
      }
    }
    __syncwarp();  // the row's bf16 values are read by every lane before the terms replace them
    const int out_off = r * 128 + (((lane >> 2) ^ (r & 7)) << 4) + (lane & 3) * 4;
#pragma unroll
    for (int term = 0; term < NQ; ++term) *reinterpret_cast<uint32_t*>(sQ + term * (N * 128) + out_off) = t[term];
    if (lane == 0) sw[r] = sw[r] * down;
  }
}

// ------------------------------------------------------------------ fp4 keys
// Eight e2m1 codes (a 32-bit word, code i in bits 4i .. 4i+3: sign, two
// exponent bits with bias 1, one mantissa bit) to eight e4m3 bytes, code i
// in byte i of lo (i < 4) or hi. Every e2m1 value is an e4m3 value, so this
// is a table: magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6 are the e4m3 codes
// 0x00, 0x30, 0x38, 0x3C, 0x40, 0x44, 0x48, 0x4C (bias 7: 0.5 = 2^-1 is
// exponent field 6), looked up by byte permutation on the low three bits of
// each code; the sign moves from bit 3 of the code to bit 7 of the byte.
__device__ __forceinline__ void e2m1x8_to_e4m3(uint32_t w, uint32_t& lo, uint32_t& hi) {
  constexpr uint32_t kMag0 = 0x3C383000u, kMag1 = 0x4C484440u;
  // a selector nibble's fourth bit is ignored: each picks byte (nibble & 7)
  const uint32_t s = (w >> 3) & 0x11111111u;  // code i's sign at bit 4i
  lo = __byte_perm(kMag0, kMag1, w) | __byte_perm(0x8000u, 0u, s);
  hi = __byte_perm(kMag0, kMag1, w >> 16) | __byte_perm(0x8000u, 0u, s >> 16);
}

// ------------------------------------------------------------------ scorer configuration
template <int QT, int FMT, int KSEL, int NQ>
struct Cfg {
  static constexpr int N = 64 * QT;                      // MMA N: queries x heads
  static constexpr int QSW = QT == 4 ? 2 : 1;            // queries per score warp
  static constexpr int NSW = 4 * QT / QSW;               // score warps (4 cover the 128 lanes)
  // top-k groups of 4 warps: one per query, except for one-query tiles,
  // where two groups take alternate query tiles so that one group's final
  // selection overlaps the other's filtering of the next tile's keys
  static constexpr bool ALT = QT == 1;
  static constexpr int NTK = ALT ? 2 : QT;
  static constexpr int QPT = ALT ? 1 : QT / NTK;         // queries per top-k group
  static constexpr int NBUF = ALT ? 2 : QT;              // running top-k buffers
  // key-tile operand stages (32 KB bf16, 16 KB e4m3): enough bytes in flight
  // per SM to cover the HBM latency of a streaming one-query tile; the
  // four-query tiles of a prefill read their keys from L2 and keep two bf16
  // stages (a third measured 1 % slower on the 22528-token prefill) or three
  // e4m3 ones (six measured 2 % slower)
  // fp4 keys: the tile's e2m1 codes land in a ring of their own (NR slots
  // of 8 KB, the bytes in flight) and the converter warps widen them into
  // an operand stage, which then only has to cover the conversion and MMA
  static constexpr bool FP4 = FMT == DSA_FMT_FP4;
  static constexpr bool E8 = FMT != DSA_FMT_BF16;        // e4m3 operands (fp8, or widened fp4)
  static constexpr int S = FP4 ? (QT == 4 ? 2 : 3)
                               : QT == 4 ? (FMT == DSA_FMT_BF16 ? 2 : 3)
                                         : (FMT == DSA_FMT_BF16 ? (QT == 2 ? 3 : 4) : 6);
  static constexpr int NR = FP4 ? (QT == 4 ? 3 : 6) : 0;  // raw fp4 tile slots
  static constexpr int RAW_BYTES = kTile * 64;
  static constexpr int NCV = FP4 ? 2 : 0;                 // converter warps
  static constexpr int NST = QT == 4 ? 6 : 16;           // score staging slots (tiles)
  // alternating groups each read their own ring of staging slots: a group
  // that skips the other's query tile must not wait on a slot phase that
  // the score warps have not reached yet
  static constexpr int NRING = ALT ? 2 : 1;
  static constexpr int RS = NST / NRING;                 // slots per ring
  // candidate keys of one query's running top-k, cut back to KSEL by radix
  // select when full: one-query tiles get a buffer large enough that a
  // CTA's piece of a decode query usually needs one selection, at its end
  static constexpr int TK = ALT ? (FMT == DSA_FMT_BF16 && NQ == 2 ? 3072 : 4096) : (KSEL > 512 ? 2304 : 1280);
  // a selection keeps KSEL keys and the cut aims below TK - 2 tiles: both
  // must leave room for one more tile, and the merge of a split query's
  // lists for four 128-key chunks
  static_assert(TK >= KSEL + 4 * 128, "candidate buffer too small for the selection and the merge");
  static constexpr int W_SCORE = 2;                      // first score warp
  static constexpr int W_TOPK = W_SCORE + NSW;           // first top-k warp
  static constexpr int W_CONV = W_TOPK + 4 * NTK;          // first converter warp
  static constexpr int NWARPS = W_CONV + NCV;
  static constexpr int NTHREADS = 32 * NWARPS;
  // TMEM accumulator buffers: the MMA of a tile waits for the score warps
  // to have read the buffer it reuses, so a deeper ring hides that round
  // trip; four-query tiles fill the 512 columns with two
  static constexpr int NTB = QT == 4 ? 2 : 4;
  static constexpr int TMEM_COLS = NTB * N;
  static constexpr int TERM_BYTES = N * 128 * (FMT == DSA_FMT_BF16 ? 2 : 1);  // one query term
  // a page: its key codes, then its 64 fp32 scales (e4m3 / e2m1 keys)
  static constexpr int PAGE_BYTES = FMT == DSA_FMT_FP8 ? kPageBytesFp8 : kPageBytesFp4;
  static constexpr int SC_OFF = FMT == DSA_FMT_FP8 ? 64 * 128 : 64 * 64;
  static_assert(PAGE_BYTES % 16 == 0 && SC_OFF % 16 == 0, "bulk copies start on 16-byte boundaries");
  static constexpr int Q_BYTES = NQ * TERM_BYTES;
  // the query tile arrives as the caller's bf16 rows (N x 256 bytes) and,
  // unless it is used as it is (bf16 cache, no rotation), the score warps
  // turn it into its terms in place
  static constexpr bool PREP = E8 || NQ > 1;
  static constexpr bool HAD = FMT == DSA_FMT_BF16 ? NQ == 2 : NQ == 3;
  static_assert(!HAD || PREP, "the rotation is applied by the conversion");
  static constexpr int OP_BYTES = kTile * (FMT == DSA_FMT_BF16 ? 256 : 128);
  static constexpr int ST_BYTES = QT * kTile * 4;        // one staged tile of scores
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_OP = OFF_Q + Q_BYTES;
  static constexpr int OFF_TOPK = OFF_OP + S * OP_BYTES;
  static constexpr int OFF_ST = OFF_TOPK + NBUF * TK * 8;
  static constexpr int OFF_W = OFF_ST + NST * ST_BYTES;
  static constexpr int OFF_HIST = OFF_W + 2 * QT * 64 * 4;   // head weights, double-buffered
  // fp8 / fp4 key scales of one-query tiles: the 2 x 64 fp32 scales of a
  // tile's two pages come into a ring of their own by bulk copy beside the
  // codes (the score warps read them after the MMA has released the operand
  // stage); four-query tiles load them from global memory a tile ahead (a
  // ring for them measured no faster)
  static constexpr bool SCALE_RING = E8 && QT == 1;
  static constexpr int NSC = SCALE_RING ? 16 : 0;          // scale slots (tiles)
  static constexpr int OFF_SC = OFF_HIST + NTK * 512 * 4;  // after the radix-select histograms
  static constexpr int OFF_RAW = OFF_SC + NSC * kTile * 4;
  static constexpr int OFF_MISC = OFF_RAW + NR * RAW_BYTES;
  static constexpr int MISC_BYTES = 2048;
  static constexpr int SMEM = OFF_MISC + MISC_BYTES + 1024;
  static_assert(SMEM <= 232448, "shared memory budget");
  static_assert(TK % 128 == 0 && TK >= KSEL + 128, "candidate buffer");
  static_assert(NTHREADS <= 1024, "block size");
};

struct Misc {
  uint64_t op_full[8], op_empty[8];
  uint64_t tm_full[4], tm_empty[4], q_full, q_empty, fin, w_full[2], w_empty[2];
  uint64_t st_full[16], st_empty[16];
  uint64_t sc_full[16], sc_empty[16];
  uint64_t raw_full[8], raw_empty[8];  // fp4 code slots
  uint64_t prep[2];  // the query tile of a weight buffer has been turned into its terms
  uint32_t tmem_base;
  int abort;
  int cnt[4];
  unsigned long long thr[4];
  int gok[4], glast[4], gdigit[4], gabove[4], gcd[4];  // per top-k group
  int wsum[4][2][4];
  unsigned long long gmin[4][4], gmax[4][4];
  unsigned int hmax[4];  // per top-k group: largest candidate score word, for a cut
};
static_assert(sizeof(Misc) <= 2048, "misc");

struct ScoreArgs {
  const int32_t* page_table;
  int max_pages;
  int causal;
  const uint8_t* cache;
  int num_pages;
  const float* w;  // head weights (prepared queries: with their scales folded in)
  long long qrows;  // (query, head) rows
  const char* ws;
  WsLayout L;
  int32_t* out_idx;
  float* out_score;
  int kout;         // entries per output row (<= the selection size KSEL)
  int slots;        // output cache slots instead of positions
  unsigned int* status;
};

struct Seg {
  int qt, b, row0, nrows, ntile, t0, t1, L, qpos0;
  long long qstart, qend;  // the query tile's range in the flattened work
  bool whole;
};

// Contiguous, equal share of the flattened (query tile, key tile) work.
struct SegIter {
  long long g, gbeg, gend;
  int qt, ovh;
  const long long* prefix;
  const int4* meta;
  __device__ void init(const long long* p, const int4* m, const int* rec, long long total, int c,
                       int Ge, int ovh_units) {
    prefix = p;
    meta = m;
    ovh = ovh_units;
    if (total <= 0 || c >= Ge) {
      g = gbeg = gend = 0;
      qt = 0;
      return;
    }
    gbeg = range_start(c, total, Ge);
    gend = range_start(c + 1, total, Ge);
    g = gbeg;
    qt = rec[c];
  }
  // Next query tile with key tiles inside this CTA's range. A query tile
  // occupies units [p0, p1): ovh overhead units, then one unit per key tile.
  __device__ bool next(Seg& s) {
    while (g < gend) {
      const long long p0 = prefix[qt], p1 = prefix[qt + 1];
      if (p1 <= g) {
        ++qt;
        continue;
      }
      const long long tb = p0 + ovh;  // unit of key tile 0
      const int4 m = meta[2 * qt];
      const long long t0 = g > tb ? g - tb : 0;
      const long long t1 = min(static_cast<long long>(m.w), gend - tb);
      g = min(p1, gend);
      if (t1 <= t0) continue;
      const int4 m1 = meta[2 * qt + 1];
      s.qt = qt;
      s.b = m.x;
      s.row0 = m.y;
      s.nrows = m.z;
      s.ntile = m.w;
      s.L = m1.x;
      s.qpos0 = m1.y;
      s.qstart = p0;
      s.qend = p1;
      s.t0 = static_cast<int>(t0);
      s.t1 = static_cast<int>(t1);
      s.whole = (t0 == 0 && t1 == m.w);
      return true;
    }
    return false;
  }
};

// ------------------------------------------------------------------ running top-k (one group of 128 threads)
// Keys above a query's threshold are appended to a shared-memory candidate
// buffer as tiles arrive. A full buffer is cut back: the first time to its K
// largest keys by an exact radix select, whose K-th key becomes the
// threshold, later by a two-pass cut that keeps the score bins holding the
// K largest and raises the threshold to their lower edge; at the end of the
// query tile one exact selection leaves the K keys, which are sorted. The
// buffer is large next to K, so the selections are few: one-query tiles
// (decode) have one 3072- or 4096-key buffer per group and a CTA's piece of
// a decode query usually needs one or two selections.
//
// The sorting networks run in registers over K slots held by the group's 4
// warps: slot x = w*PW + lane*E + e is register e of lane `lane` of warp w
// (PW = K/4, E = K/128). Strides below E stay inside a thread, strides up
// to PW use shuffles, larger ones (between warps) go through a K-key
// shared-memory exchange buffer.

__device__ __forceinline__ void push_key(bool pass, uint64_t key, uint64_t* buf, int* cnt, int cap,
                                         unsigned int* status, int lane) {
  const unsigned m = __ballot_sync(0xffffffffu, pass);
  if (m) {
    const int leader = __ffs(m) - 1;
    int base = 0;
    if (lane == leader) base = atomicAdd(cnt, __popc(m));
    base = __shfl_sync(0xffffffffu, base, leader);
    // the callers make room before every push; a key that would still land
    // past the buffer is dropped and the overflow recorded, never written
    if (lane == leader && base + __popc(m) > cap) atomicOr(status, DSA_DEV_BOUNDS);
    const int idx = base + __popc(m & ((1u << lane) - 1u));
    if (pass && idx < cap) buf[idx] = key;
  }
}

// Keep exactly the K largest keys of buf[0..cnt) (when cnt > K). Radix
// select of the K-th largest key: a min/max pass finds the highest bit where
// the keys differ, then each pass histograms the next (up to) 8 bits of the
// keys that still match the selected prefix. Each warp counts into its own
// 256 bins (16-bit counters packed two per word, plain shared atomics, four
// keys in flight per thread). The kept keys (those >= the prefix) are
// compacted in place, four per thread per round. The filter threshold
// becomes the selected prefix minus one. hist: 4 x 128 words.
__device__ inline void group_compact(uint64_t* buf, int* cnt, unsigned long long* thr, int K,
                              uint32_t* hist, Misc* ms, int g, int gt, int barid) {
  const int n = *cnt;
  if (n <= K) return;
  const int w = gt >> 5, lane = gt & 31;
  // ---- min / max of the keys
  uint64_t mn = ~0ull, mx = 0ull;
  for (int i = gt; i < n; i += 128) {
    const uint64_t key = buf[i];
    mn = key < mn ? key : mn;
    mx = key > mx ? key : mx;
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    const uint64_t a = __shfl_xor_sync(0xffffffffu, mn, o);
    const uint64_t b = __shfl_xor_sync(0xffffffffu, mx, o);
    mn = a < mn ? a : mn;
    mx = b > mx ? b : mx;
  }
  if (lane == 0) {
    ms->gmin[g][w] = mn;
    ms->gmax[g][w] = mx;
  }
  named_bar(barid, 128);
#pragma unroll
  for (int x = 0; x < 4; ++x) {
    const uint64_t a = ms->gmin[g][x], b = ms->gmax[g][x];
    mn = a < mn ? a : mn;
    mx = b > mx ? b : mx;
  }
  // bits above hb are common to every key
  int hb = 63 - __clzll(static_cast<long long>(mn ^ mx));
  uint64_t mask = hb >= 63 ? 0ull : ~((2ull << hb) - 1ull);
  uint64_t prefix = mn & mask;
  int remaining = K;
  uint32_t* hw = hist + w * 128;
  while (hb >= 0) {
    const int lo = hb >= 7 ? hb - 7 : 0;
    const int width = hb - lo + 1;
    const uint64_t dmask = (1ull << width) - 1ull;
    for (int i = gt; i < 512; i += 128) hist[i] = 0;
    named_bar(barid, 128);
    for (int r0 = 0; r0 < n; r0 += 512) {
      uint64_t kv[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int i = r0 + e * 128 + gt;
        kv[e] = i < n ? buf[i] : 0ull;
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int i = r0 + e * 128 + gt;
        if (i < n && (kv[e] & mask) == prefix) {
          const uint32_t d = static_cast<uint32_t>((kv[e] >> lo) & dmask);
          atomicAdd(&hw[d >> 1], (d & 1u) ? 0x10000u : 1u);
        }
      }
    }
    named_bar(barid, 128);
    if (gt < 32) {
      // lane l holds bins 255-8l .. 248-8l (descending digits), summed over warps
      int c[8];
      int sum = 0;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int bin = 255 - 8 * gt - e;
        const int sh = (bin & 1) * 16;
        int v = 0;
#pragma unroll
        for (int x = 0; x < 4; ++x) v += static_cast<int>((hist[x * 128 + (bin >> 1)] >> sh) & 0xFFFFu);
        c[e] = v;
        sum += v;
      }
      int incl = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (gt >= o) incl += y;
      }
      const int excl = incl - sum;
      if (excl < remaining && remaining <= incl) {
        int acc = excl;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          if (acc + c[e] >= remaining) {
            ms->gdigit[g] = 255 - 8 * gt - e;
            ms->gabove[g] = acc;
            ms->gcd[g] = c[e];
            break;
          }
          acc += c[e];
        }
      }
    }
    named_bar(barid, 128);
    const int d = ms->gdigit[g];
    remaining -= ms->gabove[g];
    const int cd = ms->gcd[g];
    prefix |= static_cast<uint64_t>(d) << lo;
    mask |= dmask << lo;
    hb = lo - 1;
    if (cd == remaining) break;
  }
  // ---- keep keys >= prefix, in place (writes never pass the current round)
  int base = 0;
  for (int r0 = 0; r0 < n; r0 += 512) {
    uint64_t kv[4];
    int keep = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int i = r0 + e * 128 + gt;
      kv[e] = i < n ? buf[i] : 0ull;
      keep += (i < n && kv[e] >= prefix) ? 1 : 0;
    }
    int incl = keep;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const int par = (r0 >> 9) & 1;
    if (lane == 31) ms->wsum[g][par][w] = incl;
    named_bar(barid, 128);
    int off = base + incl - keep, tot = 0;
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      const int v = ms->wsum[g][par][x];
      if (x < w) off += v;
      tot += v;
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int i = r0 + e * 128 + gt;
      if (i < n && kv[e] >= prefix) buf[off++] = kv[e];
    }
    base += tot;
  }
  named_bar(barid, 128);
  if (gt == 0) {
    *cnt = base;
    *thr = prefix > 0 ? prefix - 1 : 0;
  }
  named_bar(barid, 128);
}

// Cut buf[0..n) back, cheaply, to the keys of the top score bins holding at
// least K keys, once a threshold is known: every key lies above the current
// threshold, so the high words (ordered scores) span thr_hi .. hmax (the
// largest, found by a first pass); 256 bins of a power-of-two width cover
// that span, one histogram finds the bin B that holds the K-th largest key,
// and the keys of bins >= B stay: K .. K + |B| of them. The threshold rises
// to just below bin B's lower edge, which is at most the K-th largest key,
// so no key of the top K is lost. Three passes over the buffer (maximum,
// histogram, compaction) where the exact radix select takes six to eight. Returns false, leaving the buffer as it is,
// when the cut would keep more than `room` keys. hist: 256 words.
__device__ inline bool group_cut(uint64_t* buf, int* cnt, unsigned long long* thr, int K, int room,
                          uint32_t* hist, Misc* ms, int g, int gt, int barid) {
  const int n = *cnt;
  if (n <= K) return true;
  const int w = gt >> 5, lane = gt & 31;
  const uint32_t lo = static_cast<uint32_t>(*thr >> 32);
  // the largest candidate's score word bounds the bins from above
  if (gt == 0) ms->hmax[g] = 0u;
  for (int i = gt; i < 256; i += 128) hist[i] = 0u;
  uint32_t hm = 0u;
  for (int i = gt; i < n; i += 128) {
    const uint32_t h = static_cast<uint32_t>(buf[i] >> 32);
    hm = h > hm ? h : hm;
  }
  hm = __reduce_max_sync(0xffffffffu, hm);
  named_bar(barid, 128);
  if (lane == 0) atomicMax(&ms->hmax[g], hm);
  named_bar(barid, 128);
  const uint32_t hmax = ms->hmax[g];
  if (hmax < lo) return false;
  const uint64_t span1 = static_cast<uint64_t>(hmax - lo);  // span - 1
  const int sh = span1 >= 256 ? (64 - __clzll(static_cast<long long>(span1))) - 8 : 0;
  for (int i = gt; i < n; i += 128) {
    const uint32_t h = static_cast<uint32_t>(buf[i] >> 32);
    atomicAdd(&hist[(h - lo) >> sh], 1u);
  }
  named_bar(barid, 128);
  if (gt < 32) {
    // lane l holds bins 255-8l .. 248-8l (descending)
    int c[8], sum = 0;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      c[e] = static_cast<int>(hist[255 - 8 * gt - e]);
      sum += c[e];
    }
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (gt >= o) incl += y;
    }
    const int excl = incl - sum;
    if (excl < K && K <= incl) {
      int acc = excl;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        acc += c[e];
        if (acc >= K) {
          ms->gdigit[g] = 255 - 8 * gt - e;  // bin B
          ms->gabove[g] = acc;               // keys kept
          break;
        }
      }
    }
  }
  named_bar(barid, 128);
  const int B = ms->gdigit[g];
  const int kept = ms->gabove[g];
  if (kept > room) return false;
  const uint32_t edge = lo + (static_cast<uint32_t>(B) << sh);
  int base = 0;
  for (int r0 = 0; r0 < n; r0 += 512) {
    uint64_t kv[4];
    int keep = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int i = r0 + e * 128 + gt;
      kv[e] = i < n ? buf[i] : 0ull;
      keep += (i < n && static_cast<uint32_t>(kv[e] >> 32) >= edge) ? 1 : 0;
    }
    int incl = keep;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const int par = (r0 >> 9) & 1;
    if (lane == 31) ms->wsum[g][par][w] = incl;
    named_bar(barid, 128);
    int off = base + incl - keep, tot = 0;
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      const int v = ms->wsum[g][par][x];
      if (x < w) off += v;
      tot += v;
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int i = r0 + e * 128 + gt;
      if (i < n && static_cast<uint32_t>(kv[e] >> 32) >= edge) buf[off++] = kv[e];
    }
    base += tot;
  }
  named_bar(barid, 128);
  if (gt == 0) {
    *cnt = base;
    const unsigned long long t = (static_cast<unsigned long long>(edge) << 32) - 1ull;
    if (t > *thr) *thr = t;
  }
  named_bar(barid, 128);
  return true;
}

// Compare-exchange of registers e and e ^ S (stride S < E) of each thread;
// descending where (x & size) == 0.
template <int K, int S>
__device__ __forceinline__ void net_reg_stage(uint64_t (&v)[K / 128], int size, int w, int lane) {
  constexpr int PW = K / 4, E = PW / 32;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    if ((e ^ S) > e) {
      const int x = w * PW + lane * E + e;
      const bool desc = (x & size) == 0;
      const uint64_t a = v[e], b = v[e ^ S];
      const bool sw = (a < b) == desc;
      v[e] = sw ? b : a;
      v[e ^ S] = sw ? a : b;
    }
  }
}

// One stage of a bitonic network: slot x is compared with slot x ^ stride,
// the lower slot keeps the larger key where (x & size) == 0 (descending
// run) and the smaller one elsewhere.
template <int K>
__device__ __forceinline__ void net_stage(uint64_t (&v)[K / 128], int size, int stride, uint64_t* xbuf,
                                          int w, int lane, int barid) {
  constexpr int PW = K / 4, E = PW / 32;
  if (stride >= PW) {
    const bool lower = ((w * PW) & stride) == 0;
    const bool desc = ((w * PW) & size) == 0;
    const bool tmax = lower == desc;
    const int x0 = w * PW + lane * E;
    named_bar(barid, 128);
#pragma unroll
    for (int e = 0; e < E; ++e) xbuf[x0 + e] = v[e];
    named_bar(barid, 128);
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const uint64_t o = xbuf[(x0 + e) ^ stride];
      v[e] = ((v[e] > o) == tmax) ? v[e] : o;
    }
  } else if (stride >= E) {
    const int ls = stride / E;
    const bool lower = (lane & ls) == 0;
    const bool desc = ((w * PW + lane * E) & size) == 0;
    const bool tmax = lower == desc;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const uint64_t o = __shfl_xor_sync(0xffffffffu, v[e], ls);
      v[e] = ((v[e] > o) == tmax) ? v[e] : o;
    }
  } else {
    // register index must be a compile-time constant: one branch per stride
    if constexpr (E > 1) if (stride == 1) net_reg_stage<K, 1>(v, size, w, lane);
    if constexpr (E > 2) if (stride == 2) net_reg_stage<K, 2>(v, size, w, lane);
    if constexpr (E > 4) if (stride == 4) net_reg_stage<K, 4>(v, size, w, lane);
    if constexpr (E > 8) if (stride == 8) net_reg_stage<K, 8>(v, size, w, lane);
    static_assert(E <= 16, "register strides above 8");
  }
}

// Sort the K slots descending.
template <int K>
__device__ __forceinline__ void net_sort(uint64_t (&v)[K / 128], uint64_t* xbuf, int w, int lane, int barid) {
#pragma unroll
  for (int size = 2; size <= K; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) net_stage<K>(v, size, stride, xbuf, w, lane, barid);
  }
}


// Sort buf[0..n) (n <= K, distinct keys) into buf[0..K) descending, 0 in
// the slots past n. buf (at least K keys) is the exchange buffer.
template <int K>
__device__ __forceinline__ void sort_list(uint64_t* buf, int n, int gt, int barid) {
  constexpr int PW = K / 4, E = PW / 32;
  const int w = gt >> 5, lane = gt & 31;
  uint64_t v[E];
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int x = w * PW + e * 32 + lane;
    v[e] = x < n ? buf[x] : 0ull;
  }
  net_sort<K>(v, buf, w, lane, barid);
  named_bar(barid, 128);  // every read of buf is done
#pragma unroll
  for (int e = 0; e < E; ++e) buf[w * PW + lane * E + e] = v[e];
  named_bar(barid, 128);
}

// Sort a bitonic sequence of K slots descending.
template <int K>
__device__ __forceinline__ void net_merge(uint64_t (&v)[K / 128], uint64_t* xbuf, int w, int lane, int barid) {
#pragma unroll
  for (int stride = K >> 1; stride > 0; stride >>= 1) net_stage<K>(v, 2 * K, stride, xbuf, w, lane, barid);
}

// L := the K largest keys of the sorted lists src(c), c = c0..c1 (global
// memory, K keys each, descending, written by other CTAs). xbuf (K keys)
// may be L itself.
template <int K, typename SrcOf>
__device__ __forceinline__ void merge_lists(SrcOf src_of, int c0, int c1, uint64_t* L, uint64_t* xbuf, int gt,
                                            int barid) {
  constexpr int PW = K / 4, E = PW / 32;
  const int w = gt >> 5, lane = gt & 31;
  const int x0 = w * PW + lane * E;
  uint64_t v[E];
  const unsigned long long* s0 = src_of(c0);
#pragma unroll
  for (int e = 0; e < E; ++e) v[e] = __ldcg(s0 + x0 + e);
  for (int c = c0 + 1; c <= c1; ++c) {
    const unsigned long long* sc = src_of(c);
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const uint64_t o = __ldcg(sc + (K - 1 - x0 - e));
      v[e] = v[e] > o ? v[e] : o;
    }
    net_merge<K>(v, xbuf, w, lane, barid);
  }
  named_bar(barid, 128);  // every read of xbuf is done
#pragma unroll
  for (int e = 0; e < E; ++e) L[x0 + e] = v[e];
  named_bar(barid, 128);
}

// One output row from a sorted list: its first kout entries, positions (or
// cache slots, page_table[pos / 64] * 64 + pos % 64, when pt_row is given)
// and scores, -1 / -inf for empty slots.
template <int K>
__device__ __forceinline__ void write_row(const uint64_t* L, int32_t* oi, float* os, int kout,
                                          const int32_t* pt_row, int gt) {
#pragma unroll
  for (int i = 0; i < K / 128; ++i) {
    const int x = i * 128 + gt;
    if (x < kout) {
      const uint64_t key = L[x];
      int id = -1;
      if (key) {
        const int pos = key_pos(key);
        id = pt_row ? pt_row[pos >> 6] * 64 + (pos & 63) : pos;
      }
      oi[x] = id;
      os[x] = key ? key_score(key) : -__int_as_float(0x7f800000);
    }
  }
}

// ------------------------------------------------------------------ the scorer
template <int QT, int FMT, int KSEL, int NQ>
__global__ void __launch_bounds__(Cfg<QT, FMT, KSEL, NQ>::NTHREADS, 1)
    score_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const ScoreArgs a) {
  using C = Cfg<QT, FMT, KSEL, NQ>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t* sQ = sm + C::OFF_Q;
  uint8_t* sOp = sm + C::OFF_OP;
  uint64_t* sTopk = reinterpret_cast<uint64_t*>(sm + C::OFF_TOPK);
  float* sW = reinterpret_cast<float*>(sm + C::OFF_W);
  float* sSt = reinterpret_cast<float*>(sm + C::OFF_ST);
  float* sSc = reinterpret_cast<float*>(sm + C::OFF_SC);
  uint32_t* sHist = reinterpret_cast<uint32_t*>(sm + C::OFF_HIST);
  uint8_t* sRaw = sm + C::OFF_RAW;
  Misc* ms = reinterpret_cast<Misc*>(sm + C::OFF_MISC);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cta = blockIdx.x;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::S; ++i) {
      // filled by the TMA (one arrival with the bytes) or, for fp4 keys, by
      // every converter thread
      mbar_init(&ms->op_full[i], C::FP4 ? 32 * C::NCV : 1);
      mbar_init(&ms->op_empty[i], 1);
    }
    for (int i = 0; i < C::NR; ++i) {
      mbar_init(&ms->raw_full[i], 1);
      mbar_init(&ms->raw_empty[i], 32 * C::NCV);
    }
    for (int i = 0; i < C::NTB; ++i) {
      mbar_init(&ms->tm_full[i], 1);
      mbar_init(&ms->tm_empty[i], C::NSW);
    }
    for (int i = 0; i < C::NST; ++i) {
      mbar_init(&ms->st_full[i], C::NSW);
      mbar_init(&ms->st_empty[i], C::ALT ? 4 : 4 * C::NTK);
    }
    for (int i = 0; i < C::NSC; ++i) {
      mbar_init(&ms->sc_full[i], 1);
      mbar_init(&ms->sc_empty[i], C::NSW);
    }
    mbar_init(&ms->q_full, 1);
    mbar_init(&ms->q_empty, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&ms->w_full[i], 1);
      mbar_init(&ms->w_empty[i], C::NSW);
      mbar_init(&ms->prep[i], C::NSW);
    }
    mbar_init(&ms->fin, 1);
    ms->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&ms->tmem_base, C::TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = ms->tmem_base;

  // everything above is local set-up; global inputs are read only after the
  // previous kernel on the stream has completed
  pdl_wait();
  pdl_trigger();
  const PlanHdr* hdr = reinterpret_cast<const PlanHdr*>(a.ws + a.L.hdr);
  const int4* meta = reinterpret_cast<const int4*>(a.ws + a.L.meta);
  const long long* prefix = reinterpret_cast<const long long*>(a.ws + a.L.prefix);
  const int* rec = reinterpret_cast<const int*>(a.ws + a.L.rec);
  const long long total = hdr->total;
  const int Ge = hdr->Ge;
  const int ovh = hdr->ovh;
  SegIter it;
  it.init(prefix, meta, rec, total, cta, Ge, ovh);
  volatile int* abort_flag = &ms->abort;

  if (warp == 0) {
    // ---------------------------------------------------------- producer
    int tile_seq = 0, seg_i = 0;
    Seg s;
    bool stop = false;
    while (!stop && it.next(s)) {
      const int npg = (s.L + 63) >> 6;
      const int32_t* pt = a.page_table + static_cast<long long>(s.b) * a.max_pages;
      int pid0 = -1, pid1 = -1;
      {  // page ids of the first 32 tiles, before waiting for the Q buffer
        const int tt = s.t0 + lane;
        if (tt < s.t1) {
          if (2 * tt < npg) pid0 = pt[2 * tt];
          if (2 * tt + 1 < npg) pid1 = pt[2 * tt + 1];
        }
      }
      if (lane == 0) {
        if (!mbar_wait(&ms->q_empty, (seg_i & 1) ^ 1)) {
          atomicOr(a.status, DSA_DEV_TIMEOUT);
          *abort_flag = 1;
        } else {
          // the caller's bf16 rows, as two 64-column halves
          mbar_arrive_expect_tx(&ms->q_full, C::N * 256);
          tma_load_2d(sQ, &tm_q, 0, s.row0 * kH, &ms->q_full);
          tma_load_2d(sQ + C::N * 128, &tm_q, 64, s.row0 * kH, &ms->q_full);
        }
        // the tile's head-weight rows into the weight buffer the epilogue
        // released two query tiles ago (each buffer has its own barriers, so
        // the producer can never run two tiles ahead of the epilogue on it)
        const int wb = seg_i & 1, wu = seg_i >> 1;
        if (!*abort_flag) {
          if (!mbar_wait(&ms->w_empty[wb], (wu & 1) ^ 1)) {
            atomicOr(a.status, DSA_DEV_TIMEOUT);
            *abort_flag = 1;
          } else {
            mbar_arrive_expect_tx(&ms->w_full[wb], s.nrows * kH * 4);
            bulk_load(sW + wb * (QT * 64), a.w + static_cast<long long>(s.row0) * kH,
                      s.nrows * kH * 4, &ms->w_full[wb]);
          }
        }
      }
      for (int t = s.t0; t < s.t1; ++t) {
        if (__shfl_sync(0xffffffffu, *abort_flag, 0)) {
          stop = true;
          break;
        }
        const int rel = (t - s.t0) & 31;
        if (rel == 0 && t > s.t0) {
          const int tt = t + lane;
          pid0 = -1;
          pid1 = -1;
          if (tt < s.t1) {
            if (2 * tt < npg) pid0 = pt[2 * tt];
            if (2 * tt + 1 < npg) pid1 = pt[2 * tt + 1];
          }
        }
        const int p0 = __shfl_sync(0xffffffffu, pid0, rel);
        const int p1 = __shfl_sync(0xffffffffu, pid1, rel);
        if (lane == 0) {
          const bool v0 = p0 >= 0 && p0 < a.num_pages;
          const bool v1 = p1 >= 0 && p1 < a.num_pages;
          if ((2 * t < npg && !v0) || (2 * t + 1 < npg && !v1)) atomicOr(a.status, DSA_DEV_BOUNDS);
          const int slot = tile_seq % C::S, u = tile_seq / C::S;
          const int rs = C::FP4 ? tile_seq % C::NR : 0, ur = C::FP4 ? tile_seq / C::NR : 0;
          if (!(C::FP4 ? mbar_wait(&ms->raw_empty[rs], (ur & 1) ^ 1) : mbar_wait(&ms->op_empty[slot], (u & 1) ^ 1))) {
            atomicOr(a.status, DSA_DEV_TIMEOUT);
            *abort_flag = 1;
          } else {
            uint8_t* dst = sOp + slot * C::OP_BYTES;
            if constexpr (C::FP4) {
              // a page's 64 x 64 code bytes are contiguous: one bulk copy each
              // into the raw slot, widened by the converter warps
              uint8_t* rdst = sRaw + rs * C::RAW_BYTES;
              mbar_arrive_expect_tx(&ms->raw_full[rs], (v0 + v1) * 4096);
              if (v0) bulk_load(rdst, a.cache + static_cast<long long>(p0) * C::PAGE_BYTES, 4096, &ms->raw_full[rs]);
              if (v1) bulk_load(rdst + 4096, a.cache + static_cast<long long>(p1) * C::PAGE_BYTES, 4096, &ms->raw_full[rs]);
            } else if constexpr (FMT == DSA_FMT_BF16) {
              // a page = two 64-column halves of 64 keys (128 B rows each)
              mbar_arrive_expect_tx(&ms->op_full[slot], (v0 + v1) * 16384);
              if (v0) {
                tma_load_2d(dst, &tm_k, 0, p0 * 64, &ms->op_full[slot]);
                tma_load_2d(dst + 16384, &tm_k, 64, p0 * 64, &ms->op_full[slot]);
              }
              if (v1) {
                tma_load_2d(dst + 8192, &tm_k, 0, p1 * 64, &ms->op_full[slot]);
                tma_load_2d(dst + 16384 + 8192, &tm_k, 64, p1 * 64, &ms->op_full[slot]);
              }
            } else {
              // a page = 64 keys x 128 e4m3 bytes (its 64 scales follow it)
              mbar_arrive_expect_tx(&ms->op_full[slot], (v0 + v1) * 8192);
              if (v0) tma_load_3d(dst, &tm_k, 0, 0, p0, &ms->op_full[slot]);
              if (v1) tma_load_3d(dst + 8192, &tm_k, 0, 0, p1, &ms->op_full[slot]);
            }
          }
          if constexpr (C::SCALE_RING) {
            // the two pages' 256-byte scale blocks into the tile's scale slot
            const int ss = tile_seq % C::NSC, us = tile_seq / C::NSC;
            if (!*abort_flag && !mbar_wait(&ms->sc_empty[ss], (us & 1) ^ 1)) {
              atomicOr(a.status, DSA_DEV_TIMEOUT);
              *abort_flag = 1;
            }
            if (!*abort_flag) {
              mbar_arrive_expect_tx(&ms->sc_full[ss], (v0 + v1) * 256);
              const uint8_t* sb = a.cache + C::SC_OFF;
              if (v0) bulk_load(sSc + ss * kTile, sb + static_cast<long long>(p0) * C::PAGE_BYTES, 256, &ms->sc_full[ss]);
              if (v1) bulk_load(sSc + ss * kTile + 64, sb + static_cast<long long>(p1) * C::PAGE_BYTES, 256, &ms->sc_full[ss]);
            }
          }
        }
        ++tile_seq;
      }
      ++seg_i;
    }
    // on abort, let this CTA's copies in flight land before the CTA exits
    if (lane == 0 && *abort_flag) {
      if constexpr (C::FP4) {
        for (int i = 1; i <= C::NR && tile_seq - i >= 0; ++i) {
          const int ts = tile_seq - i;
          mbar_wait(&ms->raw_full[ts % C::NR], (ts / C::NR) & 1, 20000000LL);
        }
      } else {
        for (int i = 1; i <= C::S && tile_seq - i >= 0; ++i) {
          const int ts = tile_seq - i;
          mbar_wait(&ms->op_full[ts % C::S], (ts / C::S) & 1, 20000000LL);
        }
      }
      if constexpr (C::SCALE_RING) {
        for (int i = 1; i <= C::NSC && tile_seq - i >= 0; ++i) {
          const int ts = tile_seq - i;
          mbar_wait(&ms->sc_full[ts % C::NSC], (ts / C::NSC) & 1, 20000000LL);
        }
      }
      mbar_wait(&ms->q_full, (seg_i - 1) & 1, 20000000LL);
      if (seg_i > 0) mbar_wait(&ms->w_full[(seg_i - 1) & 1], ((seg_i - 1) >> 1) & 1, 20000000LL);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f16(128, C::N, FMT == DSA_FMT_BF16);
      int tile_seq = 0, seg_i = 0;
      Seg s;
      bool stop = false;
      while (!stop && it.next(s)) {
        const bool qok = C::PREP ? mbar_wait(&ms->prep[seg_i & 1], (seg_i >> 1) & 1)
                                 : mbar_wait(&ms->q_full, seg_i & 1);
        if (!qok) {
          atomicOr(a.status, DSA_DEV_TIMEOUT);
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        for (int t = s.t0; t < s.t1; ++t) {
          const int slot = tile_seq % C::S, u = tile_seq / C::S;
          const int buf = tile_seq % C::NTB, ub = tile_seq / C::NTB;
          if (*abort_flag || !mbar_wait(&ms->op_full[slot], u & 1) ||
              !mbar_wait(&ms->tm_empty[buf], (ub & 1) ^ 1)) {
            if (!*abort_flag) atomicOr(a.status, DSA_DEV_TIMEOUT);
            *abort_flag = 1;
            stop = true;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(sOp + slot * C::OP_BYTES);
          const uint32_t b0 = smem_u32(sQ);
          const uint32_t d = tbase + static_cast<uint32_t>(buf * C::N);
          // the query terms accumulate into the same scores; the B operand's
          // 128-byte-row blocks (N rows each) follow one another: bf16 terms
          // as two 64-column halves, e4m3 terms as one 128-byte row
#pragma unroll
          for (int kk = 0; kk < (FMT == DSA_FMT_BF16 ? 8 : 4) * NQ; ++kk) {
            const uint64_t bd = sw128_desc(b0 + (kk >> 2) * (C::N * 128) + (kk & 3) * 32);
            if constexpr (FMT == DSA_FMT_BF16) {
              // K = 16 per step: the key tile's two 64-column halves of 4 steps (32 B each)
              const uint64_t ad = sw128_desc(a0 + ((kk >> 2) & 1) * 16384 + (kk & 3) * 32);
              tc_mma_f16(d, ad, bd, idesc, kk > 0 ? 1u : 0u);
            } else {
              // K = 32 per step over one 128-byte row
              const uint64_t ad = sw128_desc(a0 + (kk & 3) * 32);
              tc_mma_e4m3(d, ad, bd, idesc, kk > 0 ? 1u : 0u);
            }
          }
          tc_commit(&ms->op_empty[slot]);
          tc_commit(&ms->tm_full[buf]);
          ++tile_seq;
        }
        tc_commit(&ms->q_empty);
        ++seg_i;
      }
      // every MMA this thread issued has completed before TMEM is released
      tc_commit(&ms->fin);
      mbar_wait(&ms->fin, 0, 200000000LL);
    }
    __syncwarp();
  } else if (warp < C::W_TOPK) {
    // ---------------------------------------------------------- score warps
    // Warp w reads its 32 TMEM lanes (keys) of query j's 64 columns, frees
    // the accumulator as soon as they are in registers, reduces them to
    // one score per key (ReLU, head weights, fp8 / fp4 key scale) and stages the
    // scores, -inf for keys that are masked or in an invalid page.
    const int j0 = ((warp - C::W_SCORE) >> 2) * C::QSW;  // this warp's first query
    const int q4 = warp & 3;
    const int row = q4 * 32 + lane;
    int tile_seq = 0, seg_i = 0, rq0 = 0, rq1 = 0;
    Seg s;
    bool stop = false;
    while (!stop && it.next(s)) {
      const int32_t* pt = a.page_table + static_cast<long long>(s.b) * a.max_pages;
      if (!__all_sync(0xffffffffu, mbar_wait(&ms->w_full[seg_i & 1], (seg_i >> 1) & 1) &&
                                       (!C::PREP || mbar_wait(&ms->q_full, seg_i & 1)))) {
        if (lane == 0) {
          atomicOr(a.status, DSA_DEV_TIMEOUT);
          *abort_flag = 1;
        }
        break;
      }
      if constexpr (C::PREP) {
        // this warp's rows of the query tile into their terms (and the rows'
        // head weights rescaled), then wait until every row is done: the MMA
        // needs all of them and this warp reads every head weight of its
        // queries
        float* sWp = sW + (seg_i & 1) * (QT * 64);
        for (int r = warp - C::W_SCORE; r < C::N; r += C::NSW)
          prep_row<C::E8, C::HAD, C::N, NQ>(sQ, r, sWp, lane);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ms->prep[seg_i & 1]);
        if (!__all_sync(0xffffffffu, mbar_wait(&ms->prep[seg_i & 1], (seg_i >> 1) & 1))) {
          if (lane == 0) {
            atomicOr(a.status, DSA_DEV_TIMEOUT);
            *abort_flag = 1;
          }
          break;
        }
      }
      const float* sWs = sW + (seg_i & 1) * (QT * 64);
      const int ring = C::ALT ? (seg_i & 1) : 0;
      int rq = ring ? rq1 : rq0;  // tiles staged so far in this ring
      // page id of this thread's key in tile tt (-1: past the sequence or
      // out of range), and the fp8 / fp4 key's scale; issued ahead of use so the
      // global-memory latency overlaps earlier tiles (page ids two tiles
      // ahead, scales one tile ahead)
      auto page_of = [&](int tt) -> int {
        const int p = tt * kTile + row;
        if (tt >= s.t1 || p >= s.L) return -1;
        const int v = pt[p >> 6];
        return (v < 0 || v >= a.num_pages) ? -1 : v;
      };
      auto scale_of = [&](int id, int tt) -> float {
        if constexpr (C::E8 && !C::SCALE_RING) {
          if (id >= 0)
            return __ldg(reinterpret_cast<const float*>(a.cache + static_cast<long long>(id) * C::PAGE_BYTES +
                                                        C::SC_OFF + ((tt * kTile + row) & 63) * 4));
        }
        return 1.f;
      };
      int pid_n1 = page_of(s.t0);
      int pid_n2 = page_of(s.t0 + 1);
      float scale_n1 = scale_of(pid_n1, s.t0);
      for (int t = s.t0; t < s.t1; ++t) {
        const int pos = t * kTile + row;
        const int pid = pid_n1;
        const float kscale = scale_n1;
        pid_n1 = pid_n2;
        pid_n2 = page_of(t + 2);
        scale_n1 = scale_of(pid_n1, t + 1);
        const int buf = tile_seq % C::NTB, ub = tile_seq / C::NTB;
        const int sq = C::ALT ? rq : tile_seq;
        const int st = ring * C::RS + sq % C::RS, us = sq / C::RS;
        if (!__all_sync(0xffffffffu, mbar_wait(&ms->tm_full[buf], ub & 1))) {
          if (lane == 0) {
            atomicOr(a.status, DSA_DEV_TIMEOUT);
            *abort_flag = 1;
          }
          stop = true;
          break;
        }
        tc_fence_after();
        float rscale = 1.f;  // this key's scale (fp8 / fp4), from the scale ring
        if constexpr (C::SCALE_RING) {
          const int ss = tile_seq % C::NSC, uss = tile_seq / C::NSC;
          if (!__all_sync(0xffffffffu, mbar_wait(&ms->sc_full[ss], uss & 1))) {
            if (lane == 0) {
              atomicOr(a.status, DSA_DEV_TIMEOUT);
              *abort_flag = 1;
            }
            stop = true;
            break;
          }
          rscale = sSc[ss * kTile + row];
          __syncwarp();
          if (lane == 0) mbar_arrive(&ms->sc_empty[ss]);
        }
        float scs[C::QSW];
#pragma unroll
        for (int jj = 0; jj < C::QSW; ++jj) {
          const int j = j0 + jj;
          const uint32_t tl = tbase + (static_cast<uint32_t>(q4 * 32) << 16) +
                              static_cast<uint32_t>(buf * C::N + j * 64);
          const float4* w4 = reinterpret_cast<const float4*>(sWs + j * 64);
          // four quarters of 16 columns through one register buffer (32-column
          // halves made the fp8 four-query scorer spill: 7 % slower)
          float v[16];
          unsigned long long a2[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
          for (int qc = 0; qc < 4; ++qc) {
            tmem_ld16(tl + qc * 16, v);
            tmem_ld_wait_regs(v);
            if (jj == C::QSW - 1 && qc == 3) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(&ms->tm_empty[buf]);  // accumulators are in registers
            }
#pragma unroll
            for (int h4 = 0; h4 < 4; ++h4) {
              const float4 ww = w4[qc * 4 + h4];
              const int b = (h4 & 1) * 2;
              a2[b + 0] = ffma2(ww.x, ww.y, fmaxf(v[4 * h4 + 0], 0.f), fmaxf(v[4 * h4 + 1], 0.f), a2[b + 0]);
              a2[b + 1] = ffma2(ww.z, ww.w, fmaxf(v[4 * h4 + 2], 0.f), fmaxf(v[4 * h4 + 3], 0.f), a2[b + 1]);
            }
          }
          float acc[8];
#pragma unroll
          for (int i = 0; i < 4; ++i) unpack2(a2[i], acc[2 * i], acc[2 * i + 1]);
          float sc = ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
          if constexpr (C::E8) sc *= C::SCALE_RING ? rscale : kscale;
          const int lim = j < s.nrows ? (a.causal ? s.qpos0 + j + 1 : s.L) : 0;
          if (pid < 0 || pos >= lim) sc = -__int_as_float(0x7f800000);
          scs[jj] = sc;
        }
        if (!__all_sync(0xffffffffu, mbar_wait(&ms->st_empty[st], (us & 1) ^ 1))) {
          if (lane == 0) {
            atomicOr(a.status, DSA_DEV_TIMEOUT);
            *abort_flag = 1;
          }
          stop = true;
          break;
        }
#pragma unroll
        for (int jj = 0; jj < C::QSW; ++jj) sSt[st * (QT * kTile) + (j0 + jj) * kTile + row] = scs[jj];
        __syncwarp();
        if (lane == 0) mbar_arrive(&ms->st_full[st]);
        ++tile_seq;
        ++rq;
      }
      if constexpr (C::ALT) {
        if (ring) rq1 = rq; else rq0 = rq;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&ms->w_empty[seg_i & 1]);  // this warp is done with the weights
      ++seg_i;
    }
  } else if (warp >= C::W_CONV) {
    // ---------------------------------------------------------- fp4 converters
    // Each thread widens 16-byte chunks of the tile (16 dims of one key row)
    // from the raw slot's e2m1 pairs into the operand stage's e4m3 bytes,
    // in the 128-byte swizzle the MMA reads (chunk c of row r at chunk
    // c ^ (r & 7)); consecutive threads take consecutive chunks, so a warp
    // reads and writes whole rows without bank conflicts.
    if constexpr (C::FP4) {
      const int ct = threadIdx.x - 32 * C::W_CONV;
      int tile_seq = 0;
      Seg s;
      bool stop = false;
      while (!stop && it.next(s)) {
        for (int t = s.t0; t < s.t1; ++t) {
          if (__shfl_sync(0xffffffffu, *abort_flag, 0)) {
            stop = true;
            break;
          }
          const int rs = tile_seq % C::NR, ur = tile_seq / C::NR;
          const int slot = tile_seq % C::S, u = tile_seq / C::S;
          if (!__all_sync(0xffffffffu, mbar_wait(&ms->raw_full[rs], ur & 1) &&
                                           mbar_wait(&ms->op_empty[slot], (u & 1) ^ 1))) {
            if (lane == 0) {
              atomicOr(a.status, DSA_DEV_TIMEOUT);
              *abort_flag = 1;
            }
            stop = true;
            break;
          }
          // chunk i = ct + 64 j (j < 16): row r = ct / 8 + 8 j, chunk column
          // c = ct % 8, so the swizzled column and the row phase are this
          // thread's constants and every address is a fixed offset; all
          // sixteen loads go out before the first conversion
          constexpr int PER = kTile * 8 / (32 * C::NCV);
          const uint2* src = reinterpret_cast<const uint2*>(sRaw + rs * C::RAW_BYTES) + ct;
          uint8_t* dst = sOp + slot * C::OP_BYTES + (ct >> 3) * 128 + (((ct & 7) ^ ((ct >> 3) & 7)) << 4);
          uint2 w[PER];
#pragma unroll
          for (int jj = 0; jj < PER; ++jj) w[jj] = src[jj * 32 * C::NCV];
#pragma unroll
          for (int jj = 0; jj < PER; ++jj) {
            uint4 o;
            e2m1x8_to_e4m3(w[jj].x, o.x, o.y);
            e2m1x8_to_e4m3(w[jj].y, o.z, o.w);
            *reinterpret_cast<uint4*>(dst + jj * (32 * C::NCV / 8) * 128) = o;
          }
          // the stage is read by the tensor cores (async proxy)
          fence_proxy_async_smem();
          mbar_arrive(&ms->op_full[slot]);
          mbar_arrive(&ms->raw_empty[rs]);
          ++tile_seq;
        }
      }
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------- top-k groups
    // Group tg owns queries tg*QPT .. tg*QPT+QPT-1 of each query tile (of
    // every other query tile, query 0, when the tiles hold one query): it
    // filters the staged scores against each query's threshold into its
    // candidate buffer, bounds the buffer (radix select), and
    // at the end of the query tile leaves the sorted top-k in the first KSEL
    // slots and writes the row (or publishes the top-k of its piece of the
    // keys and, if it is the last piece to finish, merges all pieces).
    const int tg = (warp - C::W_TOPK) >> 2;
    const int gt = threadIdx.x - 32 * (C::W_TOPK + 4 * tg);
    const int barid = 1 + tg;
    uint32_t* hist = sHist + tg * 512;
    int tile_seq = 0, seg_i = 0;
    Seg s;
    bool stop = false;
    int* counters = reinterpret_cast<int*>(const_cast<char*>(a.ws) + a.L.counters);
    unsigned long long* gthr = reinterpret_cast<unsigned long long*>(const_cast<char*>(a.ws) + a.L.gthr);
    unsigned long long* partials =
        reinterpret_cast<unsigned long long*>(const_cast<char*>(a.ws) + a.L.partials);
    // query jj of this group in the tile, its running top-k and where its
    // candidates go (the batch after the sorted list, or the whole buffer)
    auto qrow = [&](int jj) { return C::ALT ? jj : tg * C::QPT + jj; };
    auto qlist = [&](int jj) { return sTopk + (C::ALT ? tg : tg * C::QPT + jj) * C::TK; };
    auto qbuf = [&](int jj) { return C::ALT ? tg : tg * C::QPT + jj; };
    // page-table row for slot output (null: positions)
    auto out_pt = [&](const Seg& sg) -> const int32_t* {
      return a.slots ? a.page_table + static_cast<long long>(sg.b) * a.max_pages : nullptr;
    };
    while (!stop && it.next(s)) {
      if (C::ALT && (seg_i++ & 1) != tg) continue;  // the other group's query tile
      // A query tile whose keys are split over several CTAs shares one
      // threshold per query: each piece publishes its running k-th key
      // (atomicMax) and filters against the largest one published. A key
      // below another piece's k-th key has k keys above it already, so it
      // cannot be in the query's top-k; the pieces' lists still hold every
      // key that is. The shared word is touched only when a piece's own
      // threshold has changed (after a selection), never per tile: other
      // pieces hammer the same word.
      const bool share = !s.whole;
      unsigned long long thr[C::QPT];
      int nsel[C::QPT];  // selections so far
#pragma unroll
      for (int jj = 0; jj < C::QPT; ++jj) {
        const int jb = qbuf(jj);
        if (gt == 0) {
          ms->cnt[jb] = 0;
          ms->thr[jb] = 0;
        }
        thr[jj] = 0;
        nsel[jj] = 0;
      }
      if (gt == 0) ms->gok[tg] = 1;
      named_bar(barid, 128);
      for (int t = s.t0; t < s.t1; ++t) {
        const int pos = t * kTile + gt;
        // this group's ring (the only ring unless the groups alternate)
        const int st = (C::ALT ? tg : 0) * C::RS + tile_seq % C::RS, us = tile_seq / C::RS;
        const bool ok = __all_sync(0xffffffffu, mbar_wait(&ms->st_full[st], us & 1));
        if (ok) {
#pragma unroll
          for (int jj = 0; jj < C::QPT; ++jj) {
            const int j = qrow(jj), jb = qbuf(jj);
            const float sc = sSt[st * (QT * kTile) + j * kTile + gt];
            const uint64_t key = make_key(sc, pos);
            const bool pass = __float_as_uint(sc) != 0xff800000u && key > thr[jj];
            push_key(pass, key, qlist(jj), &ms->cnt[jb], C::TK, a.status, lane);
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&ms->st_empty[st]);
        } else if (lane == 0) {
          atomicOr(a.status, DSA_DEV_TIMEOUT);
          *abort_flag = 1;
          ms->gok[tg] = 0;
        }
        named_bar(barid, 128);
        if (!ms->gok[tg]) {
          stop = true;
          break;
        }
#pragma unroll
        for (int jj = 0; jj < C::QPT; ++jj) {
          const int jb = qbuf(jj);
          // make room before the next tile could overflow the buffer; the
          // first selection of a one-query tile comes at 2 KSEL candidates,
          // early enough that its threshold keeps the buffer (and the
          // piece's last selection) small
          constexpr int kFirst = 2 * KSEL < C::TK ? 2 * KSEL : C::TK;
          const int limit = (C::ALT && nsel[jj] == 0) ? kFirst : C::TK;
          if (ms->cnt[jb] > C::TK) {  // only after a recorded overflow: the dropped keys are gone
            named_bar(barid, 128);
            if (gt == 0) ms->cnt[jb] = C::TK;
            named_bar(barid, 128);
          }
          if (ms->cnt[jb] > limit - kTile) {
            // after the first (exact) selection the threshold bounds the
            // scores from below and the cheap cut usually suffices
            if (nsel[jj] == 0 || !group_cut(qlist(jj), &ms->cnt[jb], &ms->thr[jb], KSEL, limit - 2 * kTile,
                                            hist, ms, tg, gt, barid))
              group_compact(qlist(jj), &ms->cnt[jb], &ms->thr[jb], KSEL, hist, ms, tg, gt, barid);
            ++nsel[jj];
            unsigned long long t_new = ms->thr[jb];
            const int j = qrow(jj);
            if (share && j < s.nrows) {
              unsigned long long* g = gthr + s.row0 + j;
              if (gt == 0) atomicMax(g, t_new);
              const unsigned long long gv = __ldcg(g);
              t_new = gv > t_new ? gv : t_new;
            }
            thr[jj] = t_new > thr[jj] ? t_new : thr[jj];
          }
        }
        ++tile_seq;
      }
      if (stop) break;

      // ------------------------------------------------ finish the segment
      // a split query tile's pieces: CTAs cf .. cl. With a few, each sorts
      // its top-k and the last merges the sorted lists pairwise; with many,
      // the last streams the unsorted lists through its filter and selects
      // and sorts once (the pairwise merges would cost one merge per piece)
      // (selections of 512 keys always merge pairwise: their merges are
      // cheap, and a decode kernel is better off without the second path's
      // code, which runs cold once per CTA)
      const int cf = s.whole ? cta : owner_of(s.qstart + ovh, total, Ge);  // owner of key tile 0
      const int cl = s.whole ? cta : owner_of(s.qend - 1, total, Ge);
      const bool many = KSEL > 512 && cl - cf + 1 > kFewPieces;
#pragma unroll
      for (int jj = 0; jj < C::QPT; ++jj) {
        const int jb = qbuf(jj);
        group_compact(qlist(jj), &ms->cnt[jb], &ms->thr[jb], KSEL, hist, ms, tg, gt, barid);
        if (share && gt == 0 && qrow(jj) < s.nrows) atomicMax(gthr + s.row0 + qrow(jj), ms->thr[jb]);
        // a whole query tile, or a piece of one split in few pieces, is
        // sorted here (the few sorted lists are merged); the pieces of a
        // query tile split in many go out unsorted
        if ((s.whole || !many) && qrow(jj) < s.nrows)
          sort_list<KSEL>(qlist(jj), min(ms->cnt[jb], KSEL), gt, barid);
      }
      if (s.whole) {
#pragma unroll
        for (int jj = 0; jj < C::QPT; ++jj) {
          const int j = qrow(jj);
          if (j < s.nrows) {
            const long long o = static_cast<long long>(s.row0 + j) * a.kout;
            write_row<KSEL>(qlist(jj), a.out_idx + o, a.out_score + o, a.kout, out_pt(s), gt);
          }
        }
      } else {
        // this CTA holds one piece of the query tile's keys: publish its
        // top-k (sorted or not, 0 in the slots past its count); the last
        // piece to finish merges all of them
        const int slot = partial_slot(cta, s.qstart, total, Ge);
#pragma unroll
        for (int jj = 0; jj < C::QPT; ++jj) {
          const int j = qrow(jj);
          if (j < s.nrows) {
            const uint64_t* L = qlist(jj);
            const int n = ms->cnt[qbuf(jj)];
            unsigned long long* dst = partials + (static_cast<long long>(slot) * QT + j) * KSEL;
#pragma unroll
            for (int i = 0; i < KSEL / 128; ++i) {
              const int x = i * 128 + gt;
              dst[x] = x < n ? L[x] : 0ull;
            }
          }
        }
        __threadfence();
        named_bar(barid, 128);
        if (gt == 0) {
          // one counter per query tile and group (per query tile when the
          // groups alternate: its pieces may sit in either group)
          const int old = atomicAdd(&counters[s.qt * QT + (C::ALT ? 0 : tg)], 1);
          ms->glast[tg] = (old == cl - cf);
          __threadfence();
        }
        named_bar(barid, 128);
        if (ms->glast[tg] && !many) {
#pragma unroll
          for (int jj = 0; jj < C::QPT; ++jj) {
            const int j = qrow(jj);
            if (j < s.nrows) {
              auto src_of = [&](int c) {
                return partials + (static_cast<long long>(partial_slot(c, s.qstart, total, Ge)) * QT + j) * KSEL;
              };
              uint64_t* L = qlist(jj);
              merge_lists<KSEL>(src_of, cf, cl, L, L, gt, barid);
              const long long o = static_cast<long long>(s.row0 + j) * a.kout;
              write_row<KSEL>(L, a.out_idx + o, a.out_score + o, a.kout, out_pt(s), gt);
            }
          }
        } else if (KSEL > 512 && ms->glast[tg]) {
          // The pieces' lists stream through the running top-k once more,
          // filtered from the start by the shared threshold: it is at least
          // every piece's k-th key, so each key of the query's top k is
          // above it, and most of the pieces' keys are not. One selection
          // and one sort follow.
#pragma unroll
          for (int jj = 0; jj < C::QPT; ++jj) {
            const int j = qrow(jj), jb = qbuf(jj);
            if (j < s.nrows) {
              uint64_t* L = qlist(jj);
              if (gt == 0) {
                ms->cnt[jb] = 0;
                ms->thr[jb] = __ldcg(gthr + s.row0 + j);
              }
              named_bar(barid, 128);
              // four 128-key chunks at a time, with room for them made first
              const int nchunk = (cl - cf + 1) * (KSEL / 512);
#pragma unroll 1
              for (int q = 0; q < nchunk; ++q) {
                const int c = cf + q / (KSEL / 512), i0 = (q % (KSEL / 512)) * 4;
                const unsigned long long* src =
                    partials + (static_cast<long long>(partial_slot(c, s.qstart, total, Ge)) * QT + j) * KSEL;
                uint64_t kv[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) kv[e] = __ldcg(src + (i0 + e) * 128 + gt);
                // the threshold is a true lower bound from the start, so the
                // cheap cut serves until the final exact selection
                if (ms->cnt[jb] > C::TK - 4 * kTile &&
                    !group_cut(L, &ms->cnt[jb], &ms->thr[jb], KSEL, C::TK - 5 * kTile, hist, ms, tg, gt, barid))
                  group_compact(L, &ms->cnt[jb], &ms->thr[jb], KSEL, hist, ms, tg, gt, barid);
                const unsigned long long th = ms->thr[jb];
#pragma unroll
                for (int e = 0; e < 4; ++e) push_key(kv[e] > th, kv[e], L, &ms->cnt[jb], C::TK, a.status, lane);
                named_bar(barid, 128);
                if (ms->cnt[jb] > C::TK) {  // only after a recorded overflow
                  if (gt == 0) ms->cnt[jb] = C::TK;
                  named_bar(barid, 128);
                }
              }
              group_compact(L, &ms->cnt[jb], &ms->thr[jb], KSEL, hist, ms, tg, gt, barid);
              sort_list<KSEL>(L, min(ms->cnt[jb], KSEL), gt, barid);
              const long long o = static_cast<long long>(s.row0 + j) * a.kout;
              write_row<KSEL>(L, a.out_idx + o, a.out_score + o, a.kout, out_pt(s), gt);
            }
          }
        }
      }
      named_bar(barid, 128);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, C::TMEM_COLS);
  }
}

// ------------------------------------------------------------------ host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

template <int QT, int FMT, int KSEL, int NQ>
dsa_status run_score(dsa_ctx* ctx, const CUtensorMap& tq, const CUtensorMap& tk,
                     const ScoreArgs& args, int G, cudaStream_t stream) {
  using C = Cfg<QT, FMT, KSEL, NQ>;
  auto kern = score_kernel<QT, FMT, KSEL, NQ>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
    return DSA_ERR_CUDA;
  LaunchScope scope(ctx, FMT == DSA_FMT_BF16 ? DSA_K_SCORE_BF16 : FMT == DSA_FMT_FP8 ? DSA_K_SCORE_FP8 : DSA_K_SCORE_FP4,
                    stream);
  const cudaError_t e = launch_pdl(kern, dim3(G), dim3(C::NTHREADS), C::SMEM, stream, tq, tk, args);
  return e == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

template <int QT, int FMT, int NQ>
dsa_status run_score_k(dsa_ctx* ctx, int k, const CUtensorMap& tq, const CUtensorMap& tk,
                       const ScoreArgs& args, int G, cudaStream_t stream) {
  if (k == 512) return run_score<QT, FMT, 512, NQ>(ctx, tq, tk, args, G, stream);
  if constexpr (QT == 1) {  // 2048-key selections run in one-query tiles only
    if (k == 2048) return run_score<QT, FMT, 2048, NQ>(ctx, tq, tk, args, G, stream);
  }
  return run_score<QT, FMT, 1024, NQ>(ctx, tq, tk, args, G, stream);
}

// One format's scorer launch: the variant for one- or four-query tiles
// (qt), the number of query terms (nq) and the selection size (ksel).
// Defined in topk.cu (bf16), topk_fp8.cu and topk_fp4.cu.
dsa_status score_bf16(dsa_ctx* ctx, int qt, int nq, int ksel, const CUtensorMap& tq, const CUtensorMap& tk,
                      const ScoreArgs& args, int G, cudaStream_t stream);
dsa_status score_fp8(dsa_ctx* ctx, int qt, int nq, int ksel, const CUtensorMap& tq, const CUtensorMap& tk,
                     const ScoreArgs& args, int G, cudaStream_t stream);
dsa_status score_fp4(dsa_ctx* ctx, int qt, int nq, int ksel, const CUtensorMap& tq, const CUtensorMap& tk,
                     const ScoreArgs& args, int G, cudaStream_t stream);

}  // namespace sc
}  // namespace dsa
