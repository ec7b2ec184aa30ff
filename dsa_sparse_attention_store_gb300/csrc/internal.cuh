// Internal declarations shared by the library's translation units.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/dsaidx.h"

// device status word bits
#define DSA_DEV_BOUNDS 1u
#define DSA_DEV_TIMEOUT 2u

struct dsa_ctx {
  int device;
  int num_sms;
  float theta;
  float eps;
  int max_pos;
  float2* rope;          // [max_pos][64] (cos, sin), fp32
  float* gamma;          // [128]
  unsigned int* status;  // device status word
  void* encode_tiled;    // cuTensorMapEncodeTiled entry point
};

namespace dsa {

dsa_status launch_store(dsa_ctx* ctx, const void* k_raw, const int32_t* pos, const int32_t* seq,
                        const int32_t* page_table, int32_t T, int32_t B, int32_t max_pages,
                        void* cache, int32_t num_pages, dsa_fmt fmt, cudaStream_t stream);

size_t topk_workspace(const dsa_ctx* ctx, int32_t Tq, int32_t B, int32_t k, dsa_fmt fmt);

dsa_status launch_topk(dsa_ctx* ctx, const void* q, const float* head_w, const void* cache,
                       int32_t num_pages, dsa_fmt fmt, const int32_t* page_table,
                       int32_t max_pages, const int32_t* seq_lens, const int32_t* cu_q,
                       int32_t B, int32_t Tq, int32_t causal, int32_t k, int32_t* out_idx,
                       float* out_score, void* workspace, size_t ws_bytes, cudaStream_t stream);

}  // namespace dsa
