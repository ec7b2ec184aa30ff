// The scorer's fp4 kernel variants (see scorer.cuh and topk.cu).
#include "scorer.cuh"

namespace dsa {
namespace sc {

dsa_status score_fp4(dsa_ctx* ctx, int qt, int nq, int ksel, const CUtensorMap& tq, const CUtensorMap& tk,
                     const ScoreArgs& args, int G, cudaStream_t stream) {
  if (nq == 3)
    return qt == 2 ? run_score_k<2, DSA_FMT_FP4, 3>(ctx, ksel, tq, tk, args, G, stream)
                   : run_score_k<1, DSA_FMT_FP4, 3>(ctx, ksel, tq, tk, args, G, stream);
  if (qt == 4) return run_score_k<4, DSA_FMT_FP4, 2>(ctx, ksel, tq, tk, args, G, stream);
  return run_score_k<1, DSA_FMT_FP4, 2>(ctx, ksel, tq, tk, args, G, stream);
}

}  // namespace sc
}  // namespace dsa
