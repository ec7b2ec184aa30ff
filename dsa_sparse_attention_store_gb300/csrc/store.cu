// Index-key store kernel: RMSNorm + RoPE + (e4m3 or e2m1 with a per-token
// scale | bf16) written into a 64-token paged cache.
//
// What it computes follows "The Moment of Validation: Diagnosing an OOM Crash
// in the bf16 Index-K Fix for DeepSeek V4 Sparse Attention" (section "Input
// Knowledge Required to Understand This Message": normalisation, RoPE and
// the store fused in one kernel; 132 B/token fp8, 256 B/token bf16) and "The
// Fused Kernel Decision" (section "The Message": 64-token pages, a token goes
// to a page and an offset, a bf16 page is [64*128]).
//
// Mapping: one token per half-warp. Lane l (0..15) owns dims 8l..8l+7 and
// moves them with one 16-byte load and one 16-byte (bf16), 8-byte (fp8) or
// 4-byte (fp4) store, so a warp reads 512 contiguous bytes per instruction. The sum of
// squares is 8 sequential fused multiply-adds per lane (exact products of
// bf16 inputs) followed by a xor butterfly over the half-warp (8, 4, 2, 1):
// this order is the store's definition, which is what makes the bytes
// reproducible. RoPE pairs dim i (lane l < 8) with dim i+64 (lane l+8), one
// shuffle. Every fp32 step uses the round-to-nearest intrinsics so no
// multiply-add is contracted.
//
// Strided RoPE loads made the kernel bound by the L1 data pipe (wavefronts),
// so the context keeps its RoPE table and gamma in lane-interleaved layouts
// (after which the dependent load latency bounds it): lane j = l & 7 needs
// the (cos, sin) pairs 8j..8j+7 of its position, as four 16-byte chunks,
// and chunk v of every lane sits in one contiguous 128-byte block of the
// row (float4 8v + j), so each of the four loads touches one line per token
// instead of four; gamma's two float4 per lane are stored as [16 first
// halves][16 second halves] likewise. Values and arithmetic are unchanged.
//
// Optional Hadamard rotation (same pages: the fused kernel applies a Hadamard
// transform before the store): the unnormalised 128-point Walsh-Hadamard
// transform in natural order, as butterflies h = 1, 2, 4 inside a lane's 8
// dims and h = 8, 16, 32, 64 between lanes l and l ^ (h/8), each pair
// (i, i+h) becoming (a + b, a - b) in fp32.
#include <cuda_bf16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>

#include "internal.cuh"

namespace dsa {
namespace {

constexpr int kD = 128;
constexpr int kPage = 64;

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// The kernel is latency-bound (two dependent rounds of loads per token), so
// it is compiled for 12 resident CTAs per SM (96 tokens in flight; 40
// registers, with 16-24 bytes per thread spilled to L1): 6 % faster on the
// 1.05M-token fill than the 10 CTAs its 47 registers allowed, in both
// formats; 16 CTAs (32 registers) were 27 % slower.
template <int FMT, bool HAD>
__global__ void __launch_bounds__(128, 12) store_kernel(
    const uint4* __restrict__ k_raw, const int32_t* __restrict__ rope_pos,
    const int32_t* __restrict__ seq_id, const int32_t* __restrict__ page_table, int T, int B,
    int max_pages, uint8_t* __restrict__ cache, int num_pages, const float4* __restrict__ rope,
    int max_pos, const float* __restrict__ gamma, float eps, unsigned int* status, int R, int Cr) {
  pdl_wait();
  pdl_trigger();
  // chunk of 8 tokens: CTA b takes chunk j = b / R of region r = b % R, the
  // token array being cut into R regions of Cr chunks
  const long long chunk = static_cast<long long>(blockIdx.x % R) * Cr + blockIdx.x / R;
  const long long tok_l = chunk * 8 + (threadIdx.x >> 4);
  const int tok = tok_l < T ? static_cast<int>(tok_l) : T;
  const int l = threadIdx.x & 15;
  const bool live = tok < T;

  // Loads in two dependent rounds: the token's raw key, position, sequence
  // and this lane's gamma first (independent), then its page id and RoPE
  // row (which need the position and sequence).
  int pos = 0, page = -1;
  bool ok = false;
  uint4 raw = make_uint4(0, 0, 0, 0);
  float4 g0 = make_float4(0.f, 0.f, 0.f, 0.f), g1 = g0;
  int s = -1;
  if (live) {
    // the raw keys and the cache writes stream through L2 once (evict-first),
    // so that the RoPE table rows, shared by every sequence at a position,
    // stay in L2
    raw = __ldcs(k_raw + static_cast<long long>(tok) * 16 + l);
    pos = rope_pos[tok];
    s = seq_id[tok];
  }
  g0 = __ldg(reinterpret_cast<const float4*>(gamma) + l);
  g1 = __ldg(reinterpret_cast<const float4*>(gamma) + 16 + l);
  if (live) {
    ok = s >= 0 && s < B && pos >= 0 && pos < max_pos && pos < max_pages * kPage;
    if (ok) {
      page = page_table[static_cast<long long>(s) * max_pages + pos / kPage];
      ok = page >= 0 && page < num_pages;
    }
    if (!ok && l == 0) atomicOr(status, DSA_DEV_BOUNDS);
  }
  const bool pos_ok = live && pos >= 0 && pos < max_pos;  // the RoPE row may be read
  const float4* cs4 = rope + static_cast<long long>(pos_ok ? pos : 0) * 32 + (l & 7);
  float4 cst[4];
#pragma unroll
  for (int v = 0; v < 4; ++v) cst[v] = __ldg(cs4 + 8 * v);

  float x[8] = {bf16_lo(raw.x), bf16_hi(raw.x), bf16_lo(raw.y), bf16_hi(raw.y),
                bf16_lo(raw.z), bf16_hi(raw.z), bf16_lo(raw.w), bf16_hi(raw.w)};

  // sum of squares: sequential in dim order within the lane, then a butterfly
  float ss = 0.f;
#pragma unroll
  for (int e = 0; e < 8; ++e) ss = __fmaf_rn(x[e], x[e], ss);
#pragma unroll
  for (int m = 8; m >= 1; m >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, m));
  const float ms = __fmul_rn(ss, 0.0078125f);
  const float r = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, eps)));

  const float gm[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
  float y[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) y[e] = __fmul_rn(__fmul_rn(x[e], r), gm[e]);

  // RoPE, dims i and i+64 (lanes l and l^8)
  float py[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) py[e] = __shfl_xor_sync(0xffffffffu, y[e], 8);
  float c[8], sn[8];
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    const float4 t = ok ? cst[v] : make_float4(1.f, 0.f, 1.f, 0.f);
    c[2 * v] = t.x;
    sn[2 * v] = t.y;
    c[2 * v + 1] = t.z;
    sn[2 * v + 1] = t.w;
  }
  float o[8];
  if (l < 8) {
#pragma unroll
    for (int e = 0; e < 8; ++e) o[e] = __fsub_rn(__fmul_rn(y[e], c[e]), __fmul_rn(py[e], sn[e]));
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) o[e] = __fadd_rn(__fmul_rn(y[e], c[e]), __fmul_rn(py[e], sn[e]));
  }

  if constexpr (HAD) {
#pragma unroll
    for (int h = 1; h < 8; h <<= 1) {
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        if ((e & h) == 0) {
          const float a = o[e], b = o[e + h];
          o[e] = __fadd_rn(a, b);
          o[e + h] = __fsub_rn(a, b);
        }
      }
    }
#pragma unroll
    for (int m = 1; m < 16; m <<= 1) {
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float p = __shfl_xor_sync(0xffffffffu, o[e], m);
        o[e] = (l & m) ? __fsub_rn(p, o[e]) : __fadd_rn(o[e], p);
      }
    }
  }

  const int off = pos & (kPage - 1);
  if constexpr (FMT == DSA_FMT_BF16) {
    if (ok) {
      uint32_t w[4];
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        const __nv_bfloat162 p = __floats2bfloat162_rn(o[2 * v], o[2 * v + 1]);
        w[v] = *reinterpret_cast<const uint32_t*>(&p);
      }
      uint4* dst = reinterpret_cast<uint4*>(cache + static_cast<long long>(page) * (kPage * kD * 2) +
                                            off * (kD * 2)) + l;
      __stcs(dst, make_uint4(w[0], w[1], w[2], w[3]));
    }
  } else {
    float amax = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(o[e]));
#pragma unroll
    for (int m = 8; m >= 1; m >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, m));
    amax = fmaxf(amax, 1e-4f);
    constexpr bool E4M3 = FMT == DSA_FMT_FP8;
    const float scale = __fdiv_rn(amax, E4M3 ? 448.0f : 6.0f);
    const float inv = __fdiv_rn(1.0f, scale);
    if (!E4M3 && ok) {
      // fp4: 8 e2m1 codes in one word, dimension 8l + 2v in the low nibble
      // of byte v (round to nearest even, saturating at 6)
      uint32_t w = 0;
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        const __nv_fp4x2_storage_t p = __nv_cvt_float2_to_fp4x2(
            make_float2(__fmul_rn(o[2 * v], inv), __fmul_rn(o[2 * v + 1], inv)), __NV_E2M1,
            cudaRoundNearest);
        w |= static_cast<uint32_t>(p) << (8 * v);
      }
      uint8_t* pg = cache + static_cast<long long>(page) * (kPage * kD / 2 + kPage * 4);
      __stcs(reinterpret_cast<unsigned int*>(pg + off * (kD / 2) + 4 * l), w);
      if (l == 0) __stcs(reinterpret_cast<float*>(pg + kPage * kD / 2 + off * 4), scale);
    }
    if (E4M3 && ok) {
      uint32_t w[2];
#pragma unroll
      for (int v = 0; v < 2; ++v) {
        const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(
            make_float2(__fmul_rn(o[4 * v], inv), __fmul_rn(o[4 * v + 1], inv)), __NV_SATFINITE,
            __NV_E4M3);
        const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(
            make_float2(__fmul_rn(o[4 * v + 2], inv), __fmul_rn(o[4 * v + 3], inv)),
            __NV_SATFINITE, __NV_E4M3);
        w[v] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
      }
      uint8_t* pg = cache + static_cast<long long>(page) * (kPage * kD + kPage * 4);
      __stcs(reinterpret_cast<uint2*>(pg + off * kD + 8 * l), make_uint2(w[0], w[1]));
      if (l == 0) __stcs(reinterpret_cast<float*>(pg + kPage * kD + off * 4), scale);
    }
  }
}

}  // namespace

dsa_status launch_store(dsa_ctx* ctx, const void* k_raw, const int32_t* pos, const int32_t* seq,
                        const int32_t* page_table, int32_t T, int32_t B, int32_t max_pages,
                        void* cache, int32_t num_pages, dsa_fmt fmt, cudaStream_t stream) {
  if (T == 0) return DSA_OK;
  // 128-thread blocks (8 tokens): 4 % faster than 256 on the 1.05M-token fill,
  // 512 were 23 % slower
  const long long chunks = (static_cast<long long>(T) + 7) / 8;
  // The CTAs visit the token array in R interleaved regions (consecutive
  // CTAs take the same chunk index of different regions). A batch of R (or a
  // multiple of R) equal-length sequences stored one after another then has
  // its R tokens of one position in flight together, so their shared RoPE
  // table row comes from DRAM once instead of once per sequence; for any
  // other layout the order is immaterial. Each region is still a contiguous
  // stream of 2 KB chunks.
  const int R = B >= 8 ? 8 : (B >= 1 ? B : 1);
  const long long Cr = (chunks + R - 1) / R;
  const unsigned blocks = static_cast<unsigned>(Cr * R);
  LaunchScope scope(ctx, DSA_K_STORE, stream);
  auto kern = fmt == DSA_FMT_BF16 ? (ctx->hadamard ? store_kernel<DSA_FMT_BF16, true> : store_kernel<DSA_FMT_BF16, false>)
               : fmt == DSA_FMT_FP8 ? (ctx->hadamard ? store_kernel<DSA_FMT_FP8, true> : store_kernel<DSA_FMT_FP8, false>)
                                    : (ctx->hadamard ? store_kernel<DSA_FMT_FP4, true> : store_kernel<DSA_FMT_FP4, false>);
  const cudaError_t e = launch_pdl(kern, dim3(blocks), dim3(128), 0, stream,
                                   static_cast<const uint4*>(k_raw), pos, seq, page_table, T, B,
                                   max_pages, static_cast<uint8_t*>(cache), num_pages,
                                   ctx->rope, ctx->max_pos,
                                   static_cast<const float*>(ctx->gamma), ctx->eps, ctx->status, R,
                                   static_cast<int>(Cr));
  return e == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

}  // namespace dsa
