// Score + top-k selection of the DSA indexer on sm_103a.
//
// What is computed ("The Crash That Changed Direction", sections "The
// Experiment: Why fp32?" and "Assumptions Made and Broken"): every query's
// 64 index heads are multiplied against all cached index keys (a batched
// matrix product), each head's dot product goes through a ReLU, the heads are
// combined with per-head weights into one score per key, keys after the
// query's position are masked, and the top-k positions are kept (k = 512 or
// 1024 on the pages; any k up to 2048 here). Fp8 keys enter the product as
// stored (e4m3 tensor-core operands), fp4 keys widened to e4m3 on chip.
//
// Files: scorer.cuh holds the scorer (configuration, device code, launch
// template); this file the plan kernel, the bf16 variants and the launch
// sequence; topk_fp8.cu and topk_fp4.cu the other formats' variants.
//
// Why it streams ("When the Fused Kernel Isn't Enough", section "The
// Message: Validation and Discovery"): materialising the [q_len x ctx]
// logits ran out of memory at 22K tokens. Here every score lives only in
// registers; key tiles stream through a per-query running top-k in shared
// memory. Scratch is the schedule, at most two partial top-k lists per CTA
// (when a query tile's context is split across CTAs) and one shared
// threshold per query: O(#SMs x k + Tq), whatever the context length.
//
// Kernels, in launch order (all with programmatic dependent launch):
//   plan    one CTA: query tiles (QT queries of one sequence), a prefix sum
//           of their key-tile counts, and each CTA's first query tile, so the
//           CTAs split the total work evenly with one dependent load.
//   score   persistent, one CTA per SM, warp-specialised:
//             warp 0      producer: page-table lookups, TMA of 64-token pages
//                         (fp4: bulk copies of the pages' codes into a raw
//                         ring; fp8 and fp4 one-query tiles: a bulk copy of
//                         the pages' scales into a ring of their own)
//             warp 1      MMA issuer: tcgen05.mma M=128 keys x N=QT*64 heads
//                         x K=128 into a ring of TMEM accumulators (4 for
//                         one-query tiles, 2 for four-query tiles)
//             fp4 only   two converter warps widen the raw codes to e4m3 in
//                         the operand stage
//             score warps at the start of a query tile, for e4m3 caches or
//                         the Hadamard rotation: the tile's bf16 query rows
//                         rotated (if on) and turned into tensor-core terms
//                         in place (e4m3 terms with a power-of-two scale per
//                         row, folded into the head weight); then per key
//                         tile tcgen05.ld, ReLU, head-weighted sum, fp8 key
//                         scale, mask; one score per key staged in a ring of
//                         shared-memory slots
//             top-k groups of 4 warps: threshold filter of the staged scores
//                         into a candidate buffer per query, cut back by
//                         radix select when full and at the end, then sorted
//                         (one-query tiles: two groups on alternate query
//                         tiles; four-query tiles: one group per query);
//                         then output (or, for a query tile split across
//                         CTAs, a partial top-k per piece, merged by the
//                         piece that finishes last: pairwise from sorted
//                         lists when the pieces are few, else by streaming
//                         the lists through its filter and selecting once;
//                         the pieces share a running threshold per query)
//           Keys sit on the MMA's M dimension so each score thread owns one
//           key (one TMEM lane) and reduces over heads in its own registers.
#include "scorer.cuh"

namespace dsa {
namespace sc {

// ------------------------------------------------------------------ plan

__global__ void __launch_bounds__(1024) plan_kernel(const int32_t* __restrict__ seq_lens,
                                                    const int32_t* __restrict__ cu_q, int B, int Tq,
                                                    int QT, int NG, int causal, int max_pages, int k,
                                                    int ovh, char* ws, WsLayout L, int32_t* out_idx,
                                                    float* out_score, unsigned int* status, int prefix_in_smem) {
  __shared__ int smi[32];
  __shared__ long long sml[32];
  __shared__ long long s_rs[kMaxGrid + 1];  // each CTA's range start in the flattened work
  extern __shared__ long long plan_sm[];
  long long* s_pre = plan_sm;                                         // [qtmax + 1] when prefix_in_smem
  int* s_cq = reinterpret_cast<int*>(s_pre + (prefix_in_smem ? L.qtmax + 1 : 0));  // [B + 1]
  int* s_len = s_cq + (B + 1);   // [B]
  int* s_qoff = s_len + B;       // [B + 1]
  pdl_wait();
  pdl_trigger();
  PlanHdr* hdr = reinterpret_cast<PlanHdr*>(ws + L.hdr);
  int4* meta = reinterpret_cast<int4*>(ws + L.meta);
  long long* prefix = reinterpret_cast<long long*>(ws + L.prefix);
  int* cnt = reinterpret_cast<int*>(ws + L.counters);
  int* rec = reinterpret_cast<int*>(ws + L.rec);
  unsigned long long* gthr = reinterpret_cast<unsigned long long*>(ws + L.gthr);

  for (int i = threadIdx.x; i <= B; i += 1024) {
    s_cq[i] = cu_q[i];
    if (i < B) s_len[i] = seq_lens[i];
  }
  __syncthreads();

  int carry = 0;
  for (int base = 0; base < B; base += 1024) {
    const int b = base + threadIdx.x;
    int v = 0;
    if (b < B) {
      const int q0 = s_cq[b], q1 = s_cq[b + 1], Ls = s_len[b];
      const int nq = q1 - q0;
      const bool ok = q0 >= 0 && nq >= 0 && q1 <= Tq && Ls >= nq &&
                      static_cast<long long>(Ls) <= static_cast<long long>(max_pages) * 64;
      if (!ok) atomicOr(status, DSA_DEV_BOUNDS);
      v = ok ? (nq + QT - 1) / QT : 0;
    }
    int tot;
    const int ex = block_excl_scan<int>(v, smi, tot);
    if (b < B) s_qoff[b] = carry + ex;
    carry += tot;
  }
  if (threadIdx.x == 0) s_qoff[B] = carry;
  __syncthreads();
  const int qtot = carry;
  // the merge counters and the shared thresholds start at zero (coalesced)
  for (int i = threadIdx.x; i < qtot * NG; i += 1024) cnt[i] = 0;
  for (int i = threadIdx.x; i < Tq; i += 1024) gthr[i] = 0ull;
  // query tile qt: its sequence b (the last with s_qoff[b] <= qt), index t
  // in b, first row, rows, first query position
  auto tile_of = [&](int qt, int& b, int& row0, int& nrows, int& qpos0) {
    int lo = 0, hi = B - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_qoff[mid] <= qt) lo = mid; else hi = mid - 1;
    }
    b = lo;
    const int t = qt - s_qoff[b];
    const int q0 = s_cq[b], nq = s_cq[b + 1] - q0;
    row0 = q0 + t * QT;
    nrows = min(QT, nq - t * QT);
    qpos0 = s_len[b] - nq + t * QT;
  };

  long long lcarry = 0;
  for (int base = 0; base < qtot; base += 1024) {
    const int qt = base + threadIdx.x;
    long long cost = 0;
    int4 m = make_int4(0, 0, 0, 0);
    if (qt < qtot) {
      int b, row0, nrows, qpos0;
      tile_of(qt, b, row0, nrows, qpos0);
      const int kend = causal ? (qpos0 + nrows) : s_len[b];
      const int ntile = kend > 0 ? (kend + kTile - 1) / kTile : 0;
      m = make_int4(b, row0, nrows, ntile);
      meta[2 * qt] = m;
      cost = ntile > 0 ? ntile + ovh : 0;
    }
    long long tot;
    const long long ex = block_excl_scan<long long>(cost, sml, tot);
    if (qt < qtot) {
      prefix[qt] = lcarry + ex;
      if (prefix_in_smem) s_pre[qt] = lcarry + ex;
      if (m.w == 0) {  // no visible keys: the rows are all padding
        for (int r = 0; r < m.z; ++r)
          for (int i = 0; i < k; ++i) {
            out_idx[static_cast<long long>(m.y + r) * k + i] = -1;
            out_score[static_cast<long long>(m.y + r) * k + i] = -__int_as_float(0x7f800000);
          }
      }
    }
    lcarry += tot;
  }
  const long long total = lcarry;
  const int Ge = total < L.G ? static_cast<int>(total) : L.G;
  if (threadIdx.x == 0) {
    prefix[qtot] = total;
    if (prefix_in_smem) s_pre[qtot] = total;
    hdr->qtot = qtot;
    hdr->Ge = Ge;
    hdr->total = total;
    hdr->ovh = ovh;
  }
  if (Ge > 0)
    for (int c = threadIdx.x; c <= Ge; c += 1024) s_rs[c] = range_start(c, total, Ge);
  __syncthreads();
  // the CTA whose range holds unit u: the last c < Ge with s_rs[c] <= u
  auto owner = [&](long long u) {
    int lo = 0, hi = Ge - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_rs[mid] <= u) lo = mid; else hi = mid - 1;
    }
    return lo;
  };
  // first query tile of each CTA: the non-empty tile holding its range start;
  // and each query tile's first and last CTA with key tiles of it
  for (int qt = threadIdx.x; qt < qtot; qt += 1024) {
    const long long p0 = prefix_in_smem ? s_pre[qt] : prefix[qt];
    const long long p1 = prefix_in_smem ? s_pre[qt + 1] : prefix[qt + 1];
    int b, row0, nrows, qpos0;
    tile_of(qt, b, row0, nrows, qpos0);
    const bool work = p1 > p0;
    meta[2 * qt + 1] = make_int4(s_len[b], qpos0, work ? owner(p0 + ovh) : -1, work ? owner(p1 - 1) : -1);
    if (!work) continue;
    for (int c = owner(p0); c < Ge && s_rs[c] < p1; ++c)
      if (s_rs[c] >= p0) rec[c] = qt;
  }
}

dsa_status score_bf16(dsa_ctx* ctx, int qt, int nq, int ksel, const CUtensorMap& tq, const CUtensorMap& tk,
                      const ScoreArgs& args, int G, cudaStream_t stream) {
  if (nq == 2)
    return qt == 2 ? run_score_k<2, DSA_FMT_BF16, 2>(ctx, ksel, tq, tk, args, G, stream)
                   : run_score_k<1, DSA_FMT_BF16, 2>(ctx, ksel, tq, tk, args, G, stream);
  if (qt == 4) return run_score_k<4, DSA_FMT_BF16, 1>(ctx, ksel, tq, tk, args, G, stream);
  return run_score_k<1, DSA_FMT_BF16, 1>(ctx, ksel, tq, tk, args, G, stream);
}

}  // namespace sc

using namespace sc;

int max_sequences() { return kMaxSeqs; }

size_t topk_workspace(const dsa_ctx* ctx, int32_t Tq, int32_t B, int32_t k, dsa_fmt fmt) {
  (void)fmt;  // the same for every cache format
  return ws_layout(ctx->num_sms, Tq, B, select_size(k), ctx->hadamard != 0).total;
}

dsa_status launch_topk(dsa_ctx* ctx, const void* q, const float* head_w, const void* cache,
                       int32_t num_pages, dsa_fmt fmt, const int32_t* page_table,
                       int32_t max_pages, const int32_t* seq_lens, const int32_t* cu_q,
                       int32_t B, int32_t Tq, int32_t causal, int32_t k, int32_t* out_idx,
                       float* out_score, void* workspace, size_t ws_bytes, cudaStream_t stream) {
  (void)ws_bytes;
  // tensor-map row coordinates are 32-bit: the (query, head) rows must stay
  // below 2^31
  if (static_cast<long long>(Tq) * kH > 0x7FFFFFFFLL) return DSA_ERR_UNSUPPORTED;
  // any k <= 2048 runs the top-512, top-1024 or top-2048 selection and
  // writes the first k entries of each sorted row
  const int ksel = select_size(k);
  const WsLayout L = ws_layout(ctx->num_sms, Tq, B, ksel, ctx->hadamard != 0);
  char* ws = static_cast<char*>(workspace);
  {
    LaunchScope scope(ctx, DSA_K_PLAN, stream);
    // the fixed cost of a query tile, in key tiles (query load, final
    // selection, sort and output); for four-query tiles swept on GB300 over
    // 8..20: 14 balances the 22528- and 10498-token prefills (the longer one
    // prefers more, the shorter less)
    const int ovh = L.QT == 4 ? 14 : (L.QT == 2 ? 8 : 4);
    // the prefix of the query tiles' costs stays in shared memory when it fits
    const size_t base = static_cast<size_t>(3 * B + 2) * sizeof(int);
    const size_t pre = static_cast<size_t>(L.qtmax + 1) * sizeof(long long);
    const int in_smem = base + pre <= 160 * 1024 ? 1 : 0;
    const size_t psm = base + (in_smem ? pre : 0);
    if (cudaFuncSetAttribute(plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(psm)) != cudaSuccess)
      return DSA_ERR_CUDA;
    if (launch_pdl(plan_kernel, dim3(1), dim3(1024), psm, stream, seq_lens, cu_q, B, Tq, L.QT, L.NG,
                   causal, max_pages, k, ovh, ws, L, out_idx, out_score, ctx->status, in_smem) != cudaSuccess)
      return DSA_ERR_CUDA;
  }

  const long long rows = static_cast<long long>(Tq) * kH;

  EncodeTiledFn enc = reinterpret_cast<EncodeTiledFn>(ctx->encode_tiled);
  CUtensorMap tq, tk;
  {  // the caller's queries: [rows x 128] bf16, boxes of 64 columns x the tile's rows
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kD * 2)};
    const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(64 * L.QT)};
    const cuuint32_t estr[2] = {1, 1};
    if (enc(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(q), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return DSA_ERR_CUDA;
  }
  if (fmt == DSA_FMT_BF16) {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(num_pages) * 64};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kD * 2)};
    const cuuint32_t box[2] = {64, 64};
    const cuuint32_t estr[2] = {1, 1};
    if (enc(&tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(cache), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return DSA_ERR_CUDA;
  } else if (fmt == DSA_FMT_FP4) {
    tk = tq;  // fp4 codes come by plain bulk copies: no tensor map (the argument goes unused)
  } else {
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kD), 64, static_cast<cuuint64_t>(num_pages)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(kPageBytesFp8)};
    const cuuint32_t box[3] = {128, 64, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    if (enc(&tk, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(cache), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return DSA_ERR_CUDA;
  }

  ScoreArgs args;
  args.page_table = page_table;
  args.max_pages = max_pages;
  args.causal = causal;
  args.qrows = rows;
  args.cache = static_cast<const uint8_t*>(cache);
  args.num_pages = num_pages;
  args.w = head_w;
  args.ws = ws;
  args.L = L;
  args.out_idx = out_idx;
  args.kout = k;
  args.slots = ctx->slot_output;
  args.out_score = out_score;
  args.status = ctx->status;
  const int G = L.G;
  dsa_status st;
  // one-query tiles (pick_qt) with one more query term under the rotation;
  // bf16 queries are one term unrotated, e4m3 queries two
  const int nq = (fmt == DSA_FMT_BF16 ? 1 : 2) + (ctx->hadamard ? 1 : 0);
  if (fmt == DSA_FMT_BF16) st = score_bf16(ctx, L.QT, nq, ksel, tq, tk, args, G, stream);
  else if (fmt == DSA_FMT_FP8) st = score_fp8(ctx, L.QT, nq, ksel, tq, tk, args, G, stream);
  else st = score_fp4(ctx, L.QT, nq, ksel, tq, tk, args, G, stream);
  return st;
}

}  // namespace dsa
