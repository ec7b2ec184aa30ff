// C++17 oracle for the DSA indexer: test infrastructure, not the product.
//
// A plain CPU restatement of what the indexer computes, multithreaded with
// std::thread, sharing no code with the GPU library. It is the same
// definition as the numpy oracle beside it (oracle/store.py,
// oracle/indexer.py), written a second time so that full-size workloads can
// be checked row by row; the tests pin the two against each other (stored
// bytes bit for bit, scores to float64 rounding) and against brute force.
//
// Sources (web pages on the bf16 index-K fix in the DSA indexer):
//  * "The Moment of Validation: Diagnosing an OOM Crash in the bf16 Index-K
//    Fix for DeepSeek V4 Sparse Attention", section "Input Knowledge Required
//    to Understand This Message": the fused store normalises each index key,
//    applies RoPE and writes it as 128 e4m3 bytes plus a 4-byte scale
//    (132 B/token) or as 128 bf16 values (256 B/token); a Hadamard transform
//    may come between RoPE and the store.
//  * "The Fused Kernel Decision: Precision Archaeology in the CUDA Sparse
//    Attention Indexer", section "The Message": 64-token pages, a token maps
//    to a page and an offset; section "Assumptions and Their Validity":
//    queries and keys must use one element order.
//  * "The Crash That Changed Direction", sections "The Experiment: Why fp32?"
//    and "Assumptions Made and Broken": scores come from a batched product of
//    queries and keys followed by a ReLU; fp8 keys are up-converted exactly;
//    the top-512 (or 1024) positions are kept.
//
// Store, per token (every fp32 operation rounded to nearest, none fused;
// build with -ffp-contract=off):
//   ss   = sum of squares: 16 partials over dims 8g..8g+7 in dim order, then
//          pairwise (g, g+8), (g, g+4), (g, g+2), (g, g+1)
//   r    = 1 / sqrt(ss * (1/128) + eps);  y_d = (x_d * r) * gamma_d
//   RoPE = dims i and i+64 rotated by pos * theta^(-2i/128), cos and sin
//          evaluated in double and rounded once to fp32:
//          y'_i = y_i c - y_{i+64} s,  y'_{i+64} = y_{i+64} c + y_i s
//   optional Hadamard: fp32 butterflies h = 1, 2, ..., 64, (a, b) -> (a+b, a-b)
//   bf16 = round to nearest even; fp8: scale = max(max|y'|, 1e-4) / 448,
//          code = e4m3(y' * (1/scale)) rounded to nearest even, saturating;
//   fp4  = the same with 6 and e2m1 (OCP MX v1.0 FP4 element: bias 1, one
//          mantissa bit, largest 6), two codes per byte, the even dimension
//          in the low nibble (64 B + 4 B scale per token). The pages name an
//          fp4 variant ("The Fused Kernel Decision", section "The Message: A
//          Blueprint for Kernel Modification") without a layout: this is the
//          fp8 key with e2m1 elements.
// Scores: s = sum_h w_h * max(0, q_h . k) in double, k the stored key exactly
// (bf16 value, or e4m3 / e2m1 value times its scale); with the Hadamard rotation the
// query heads are rotated exactly by the +-1 Sylvester matrix and the dot
// products divided by 128. Each dot product is summed over d in order.
// Top-k: the visible keys sorted by (score desc, position asc), the first
// min(k, visible) kept; unused slots -1 / -inf.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <thread>
#include <vector>

namespace {

constexpr int D = 128;
constexpr int HALF = 64;
constexpr int H = 64;
constexpr int PAGE = 64;
constexpr int FMT_BF16 = 0;
constexpr int FMT_FP8 = 1;
constexpr int FMT_FP4 = 2;
constexpr long long kPageBytes[3] = {PAGE * D * 2, PAGE * D + PAGE * 4, PAGE * D / 2 + PAGE * 4};
constexpr long long kCodeBytes[3] = {0, D, D / 2};  // per token, before the page's scales

float f32_of_bits(uint32_t b) {
  float f;
  std::memcpy(&f, &b, 4);
  return f;
}
uint32_t bits_of_f32(float f) {
  uint32_t b;
  std::memcpy(&b, &f, 4);
  return b;
}

float bf16_value(uint16_t b) { return f32_of_bits(static_cast<uint32_t>(b) << 16); }

// binary32 -> bf16, round to nearest, ties to even (quiet NaN for NaN)
uint16_t bf16_round(float x) {
  const uint32_t u = bits_of_f32(x);
  if (std::isnan(x)) return static_cast<uint16_t>((u >> 16) | 0x40);
  const uint32_t hi = u >> 16, lo = u & 0xFFFFu;
  const bool up = lo > 0x8000u || (lo == 0x8000u && (hi & 1u));
  return static_cast<uint16_t>(hi + (up ? 1u : 0u));
}

// OCP E4M3 code -> value: bias 7, 3 mantissa bits; S.1111.111 is NaN
double e4m3_value(uint8_t c) {
  const int e = (c >> 3) & 0xF, m = c & 7;
  double v;
  if (e == 15 && m == 7) return std::numeric_limits<double>::quiet_NaN();
  if (e == 0)
    v = std::ldexp(static_cast<double>(m), -9);  // 2^-6 * m/8
  else
    v = std::ldexp(1.0 + m / 8.0, e - 7);
  return (c & 0x80) ? -v : v;
}

// binary32 -> E4M3 code, nearest with ties to even, saturating at +-448.
// Below 448 the result is the nearest multiple of the binade's spacing
// (2^(E-3) in [2^E, 2^(E+1)), 2^-9 below 2^-6), which is representable.
uint8_t e4m3_round(float xf) {
  if (std::isnan(xf)) return 0x7F;
  const double x = xf;
  const bool neg = std::signbit(x);
  const double a = std::fabs(x);
  double v;
  if (a >= 448.0) {
    v = 448.0;
  } else {
    int ex = 0;
    std::frexp(a, &ex);  // a = f * 2^ex, f in [0.5, 1)
    int E = a == 0.0 ? -6 : std::max(ex - 1, -6);
    const double q = std::ldexp(1.0, E - 3);
    v = std::nearbyint(a / q) * q;  // default rounding mode: ties to even
    v = std::min(v, 448.0);
  }
  uint8_t code;
  if (v < std::ldexp(1.0, -6)) {
    code = static_cast<uint8_t>(std::lrint(v / std::ldexp(1.0, -9)));
  } else {
    int ev = 0;
    std::frexp(v, &ev);
    const int Ev = ev - 1;
    const int m = static_cast<int>(std::lrint((v / std::ldexp(1.0, Ev) - 1.0) * 8.0));
    code = static_cast<uint8_t>(((Ev + 7) << 3) | m);
  }
  return neg ? static_cast<uint8_t>(code | 0x80) : code;
}

// OCP E2M1 code (low 4 bits) -> value: bias 1, one mantissa bit, no NaN
double e2m1_value(uint8_t c) {
  const int e = (c >> 1) & 3, m = c & 1;
  const double v = e == 0 ? 0.5 * m : std::ldexp(1.0 + 0.5 * m, e - 1);
  return (c & 8) ? -v : v;
}

// binary32 -> E2M1 code, nearest with ties to even, saturating at +-6. The
// representable magnitudes are the multiples of 0.5 up to 2, of 1 up to 4
// and of 2 up to 6; a tie goes to the even multiple, which is the even code.
uint8_t e2m1_round(float xf) {
  const double x = xf;
  const bool neg = std::signbit(x);
  const double a = std::fabs(x);
  const double q = a < 2.0 ? 0.5 : (a < 4.0 ? 1.0 : 2.0);
  const double v = std::min(std::nearbyint(a / q) * q, 6.0);
  uint8_t code;
  if (v < 1.0)
    code = static_cast<uint8_t>(v * 2.0);  // 0 or 0.5: subnormal codes 0, 1
  else {
    int ev = 0;
    std::frexp(v, &ev);  // v = f * 2^ev, f in [0.5, 1)
    const int E = ev - 1;
    const int m = static_cast<int>(std::lrint((v / std::ldexp(1.0, E) - 1.0) * 2.0));
    code = static_cast<uint8_t>(((E + 1) << 1) | m);
  }
  return neg ? static_cast<uint8_t>(code | 8) : code;
}

// Run f(i) for i in [0, n) on nthreads threads (dynamic, in chunks).
template <typename F>
void parallel_for(long long n, int nthreads, long long chunk, F f) {
  if (nthreads <= 1 || n <= chunk) {
    for (long long i = 0; i < n; ++i) f(i);
    return;
  }
  std::atomic<long long> next(0);
  std::vector<std::thread> th;
  for (int t = 0; t < nthreads; ++t)
    th.emplace_back([&] {
      while (true) {
        const long long b = next.fetch_add(chunk);
        if (b >= n) break;
        const long long e = std::min(n, b + chunk);
        for (long long i = b; i < e; ++i) f(i);
      }
    });
  for (auto& t : th) t.join();
}

// ------------------------------------------------------------------ store
void store_token(uint8_t* cache, int fmt, const uint16_t* kr, int pos, long long page,
                 float theta, float eps, const float* gamma, bool hadamard) {
  float x[D], y[D], o[D];
  for (int d = 0; d < D; ++d) x[d] = bf16_value(kr[d]);
  float p[16];
  for (int g = 0; g < 16; ++g) {
    float acc = 0.0f;
    for (int e = 0; e < 8; ++e) acc = acc + x[8 * g + e] * x[8 * g + e];  // products exact
    p[g] = acc;
  }
  for (int n = 8; n >= 1; n >>= 1)
    for (int g = 0; g < n; ++g) p[g] = p[g] + p[g + n];
  const float ss = p[0];
  const float ms = ss * (1.0f / 128.0f);
  const float r = 1.0f / std::sqrt(ms + eps);
  for (int d = 0; d < D; ++d) y[d] = (x[d] * r) * gamma[d];
  const double th = static_cast<double>(theta);
  for (int i = 0; i < HALF; ++i) {
    const double f = std::pow(th, -(2.0 * i) / 128.0);
    const double ang = static_cast<double>(pos) * f;
    const float c = static_cast<float>(std::cos(ang));
    const float s = static_cast<float>(std::sin(ang));
    const float a = y[i], b = y[i + HALF];
    const float ac = a * c, bs = b * s, bc = b * c, as = a * s;
    o[i] = ac - bs;
    o[i + HALF] = bc + as;
  }
  if (hadamard) {
    for (int h = 1; h < D; h <<= 1)
      for (int i = 0; i < D; ++i)
        if ((i & h) == 0) {
          const float a = o[i], b = o[i + h];
          o[i] = a + b;
          o[i + h] = a - b;
        }
  }
  const int off = pos % PAGE;
  uint8_t* pg = cache + page * kPageBytes[fmt];
  if (fmt == FMT_BF16) {
    uint16_t* dst = reinterpret_cast<uint16_t*>(pg + static_cast<long long>(off) * D * 2);
    for (int d = 0; d < D; ++d) dst[d] = bf16_round(o[d]);
  } else {
    float amax = 0.0f;
    for (int d = 0; d < D; ++d) amax = std::max(amax, std::fabs(o[d]));
    amax = std::max(amax, 1e-4f);
    const float scale = amax / (fmt == FMT_FP8 ? 448.0f : 6.0f);
    const float inv = 1.0f / scale;
    const long long cb = kCodeBytes[fmt];
    uint8_t* dst = pg + static_cast<long long>(off) * cb;
    if (fmt == FMT_FP8)
      for (int d = 0; d < D; ++d) dst[d] = e4m3_round(o[d] * inv);
    else
      for (int d = 0; d < D; d += 2)
        dst[d / 2] = static_cast<uint8_t>(e2m1_round(o[d] * inv) | (e2m1_round(o[d + 1] * inv) << 4));
    std::memcpy(pg + PAGE * cb + off * 4, &scale, 4);
  }
}

// ------------------------------------------------------------------ scores
struct TopkArgs {
  const uint8_t* cache;
  int fmt;
  const int32_t* page_table;
  int max_pages;
  const int32_t* seq_lens;
  const int32_t* cu_q;
  int B;
  const uint16_t* q;
  const float* w;
  int causal;
  int k;
  int hadamard;
};

int sequence_of(const TopkArgs& a, long long row) {
  // the b with cu_q[b] <= row < cu_q[b+1]
  const int32_t* it = std::upper_bound(a.cu_q, a.cu_q + a.B + 1, static_cast<int32_t>(row));
  return static_cast<int>(it - a.cu_q) - 1;
}

// Visible keys of a query row: positions 0..qpos (causal) or 0..L-1.
long long visible(const TopkArgs& a, long long row) {
  const int b = sequence_of(a, row);
  const int nq = a.cu_q[b + 1] - a.cu_q[b];
  const long long L = a.seq_lens[b];
  const long long qpos = L - nq + (row - a.cu_q[b]);
  return a.causal ? qpos + 1 : L;
}

// Exact value of the stored key at position p of sequence b.
void read_key(const TopkArgs& a, int b, long long p, double* k) {
  const long long page = a.page_table[static_cast<long long>(b) * a.max_pages + p / PAGE];
  const int off = static_cast<int>(p % PAGE);
  const uint8_t* pg = a.cache + page * kPageBytes[a.fmt];
  if (a.fmt == FMT_BF16) {
    const uint16_t* src = reinterpret_cast<const uint16_t*>(pg + static_cast<long long>(off) * D * 2);
    for (int d = 0; d < D; ++d) k[d] = bf16_value(src[d]);
  } else if (a.fmt == FMT_FP8) {
    static const std::vector<double> table = [] {  // every code's exact value
      std::vector<double> t(256);
      for (int c = 0; c < 256; ++c) t[c] = e4m3_value(static_cast<uint8_t>(c));
      return t;
    }();
    float scale;
    std::memcpy(&scale, pg + PAGE * D + off * 4, 4);
    const uint8_t* src = pg + static_cast<long long>(off) * D;
    for (int d = 0; d < D; ++d) k[d] = table[src[d]] * static_cast<double>(scale);
  } else {
    float scale;
    std::memcpy(&scale, pg + PAGE * (D / 2) + off * 4, 4);
    const uint8_t* src = pg + static_cast<long long>(off) * (D / 2);
    for (int d = 0; d < D; d += 2) {
      k[d] = e2m1_value(src[d / 2] & 0xF) * static_cast<double>(scale);
      k[d + 1] = e2m1_value(src[d / 2] >> 4) * static_cast<double>(scale);
    }
  }
}

// Sylvester Hadamard matrix entry: (-1)^popcount(i & j)
double sylvester(int i, int j) { return (__builtin_popcount(i & j) & 1) ? -1.0 : 1.0; }

// The one matrix product of the score: C[h][j] = sum_d Q[h][d] * Kt[d][j]
// for the 64 heads and a block of KB keys (Kt holds the keys transposed),
// every entry summed over d in order d = 0, 1, ..., 127. Holding a 4 x KB
// block of entries while d advances is only a loop order: no entry's sum is
// split or reassociated. v2d is two doubles (a GCC vector type); its + and *
// are the elementwise IEEE double operations.
typedef double v2d __attribute__((vector_size(16)));
constexpr int KB = 8;
constexpr int HB = 4;
void qk_block(const double* Q, const double* Kt, double* C) {
  constexpr int NV = KB / 2;
  for (int h0 = 0; h0 < H; h0 += HB) {
    v2d acc[HB][NV];
    for (int hh = 0; hh < HB; ++hh)
      for (int j = 0; j < NV; ++j) acc[hh][j] = v2d{0.0, 0.0};
    for (int d = 0; d < D; ++d) {
      v2d kv[NV];
      for (int j = 0; j < NV; ++j) kv[j] = v2d{Kt[d * KB + 2 * j], Kt[d * KB + 2 * j + 1]};
      for (int hh = 0; hh < HB; ++hh) {
        const double qs = Q[(h0 + hh) * D + d];
        const v2d qv = v2d{qs, qs};
        for (int j = 0; j < NV; ++j) acc[hh][j] = acc[hh][j] + qv * kv[j];
      }
    }
    for (int hh = 0; hh < HB; ++hh)
      for (int j = 0; j < NV; ++j) {
        C[(h0 + hh) * KB + 2 * j] = acc[hh][j][0];
        C[(h0 + hh) * KB + 2 * j + 1] = acc[hh][j][1];
      }
  }
}

// Scores of one query row over its n visible keys, into s[0..n).
void score_row(const TopkArgs& a, long long row, long long n, double* s) {
  const int b = sequence_of(a, row);
  // the query heads, exactly (rotated by the Sylvester matrix and divided by
  // 128 when the cache holds Hadamard-rotated keys)
  std::vector<double> Q(static_cast<size_t>(H) * D);
  const uint16_t* qr = a.q + row * H * D;
  for (int h = 0; h < H; ++h) {
    if (a.hadamard) {
      for (int i = 0; i < D; ++i) {
        double acc = 0.0;
        for (int j = 0; j < D; ++j) acc += sylvester(i, j) * static_cast<double>(bf16_value(qr[h * D + j]));
        Q[static_cast<size_t>(h) * D + i] = acc / 128.0;
      }
    } else {
      for (int d = 0; d < D; ++d) Q[static_cast<size_t>(h) * D + d] = bf16_value(qr[h * D + d]);
    }
  }
  double w[H];
  for (int h = 0; h < H; ++h) w[h] = a.w[row * H + h];
  double k[D], Kt[D * KB], C[H * KB];
  for (long long p0 = 0; p0 < n; p0 += KB) {
    const int nb = static_cast<int>(std::min<long long>(KB, n - p0));
    for (int j = 0; j < KB; ++j) {
      if (j < nb)
        read_key(a, b, p0 + j, k);
      else
        for (int d = 0; d < D; ++d) k[d] = 0.0;
      for (int d = 0; d < D; ++d) Kt[d * KB + j] = k[d];
    }
    qk_block(Q.data(), Kt, C);
    for (int j = 0; j < nb; ++j) {
      double tot = 0.0;  // heads in order h = 0 .. 63
      for (int h = 0; h < H; ++h) tot += w[h] * std::max(C[h * KB + j], 0.0);
      s[p0 + j] = tot;
    }
  }
}

// Top-k of one row from its scores: (score desc, position asc).
void select_row(const double* s, long long n, int k, int32_t* oi, float* os) {
  const long long kk = std::min<long long>(k, n);
  std::vector<int32_t> idx(static_cast<size_t>(n));
  for (long long p = 0; p < n; ++p) idx[p] = static_cast<int32_t>(p);
  auto better = [s](int32_t x, int32_t y) { return s[x] > s[y] || (s[x] == s[y] && x < y); };
  std::partial_sort(idx.begin(), idx.begin() + kk, idx.end(), better);
  for (long long i = 0; i < k; ++i) {
    if (i < kk) {
      oi[i] = idx[i];
      os[i] = static_cast<float>(s[idx[i]]);
    } else {
      oi[i] = -1;
      os[i] = -std::numeric_limits<float>::infinity();
    }
  }
}

}  // namespace

extern "C" {

int dso_hardware_threads() {
  const unsigned n = std::thread::hardware_concurrency();
  return n ? static_cast<int>(n) : 1;
}

// Write T tokens into the byte image of a paged cache. Returns 0, or -1 if a
// sequence, position or page id is out of range (nothing is written then).
int dso_store(uint8_t* cache, int num_pages, int fmt, const uint16_t* k_raw, const int32_t* pos,
              const int32_t* seq, long long T, const int32_t* page_table, int B, int max_pages,
              float theta, float eps, const uint16_t* gamma_bf16, int hadamard, int nthreads) {
  if (fmt != FMT_BF16 && fmt != FMT_FP8 && fmt != FMT_FP4) return -1;
  std::vector<long long> page(static_cast<size_t>(T));
  for (long long t = 0; t < T; ++t) {
    if (seq[t] < 0 || seq[t] >= B || pos[t] < 0 || pos[t] >= static_cast<long long>(max_pages) * PAGE)
      return -1;
    const long long pg = page_table[static_cast<long long>(seq[t]) * max_pages + pos[t] / PAGE];
    if (pg < 0 || pg >= num_pages) return -1;
    page[t] = pg;
  }
  float gamma[D];
  for (int d = 0; d < D; ++d) gamma[d] = gamma_bf16 ? bf16_value(gamma_bf16[d]) : 1.0f;
  parallel_for(T, nthreads, 256, [&](long long t) {
    store_token(cache, fmt, k_raw + t * D, pos[t], page[t], theta, eps, gamma, hadamard != 0);
  });
  return 0;
}

// Top-k for nrows query rows. out_idx / out_score: [nrows][k]. full (may be
// null): every row's scores over its visible keys, row i at full_off[i].
int dso_topk(const uint8_t* cache, int fmt, const int32_t* page_table, int B, int max_pages,
             const int32_t* seq_lens, const int32_t* cu_q, const uint16_t* q, const float* w,
             int causal, int k, int hadamard, const long long* rows, long long nrows,
             int32_t* out_idx, float* out_score, double* full, const long long* full_off,
             int nthreads) {
  if ((fmt != FMT_BF16 && fmt != FMT_FP8 && fmt != FMT_FP4) || k < 1) return -1;
  TopkArgs a{cache, fmt, page_table, max_pages, seq_lens, cu_q, B, q, w, causal, k, hadamard};
  parallel_for(nrows, nthreads, 1, [&](long long i) {
    const long long row = rows[i];
    const long long n = visible(a, row);
    std::vector<double> own;
    double* s;
    if (full) {
      s = full + full_off[i];
    } else {
      own.resize(static_cast<size_t>(std::max<long long>(n, 1)));
      s = own.data();
    }
    score_row(a, row, n, s);
    select_row(s, n, k, out_idx + i * k, out_score + i * k);
  });
  return 0;
}

}  // extern "C"
