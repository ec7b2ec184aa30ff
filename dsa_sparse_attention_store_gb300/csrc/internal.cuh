// Internal declarations shared by the library's translation units.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <utility>

#include "../../include/dsaidx.h"

// device status word bits
#define DSA_DEV_BOUNDS 1u
#define DSA_DEV_TIMEOUT 2u

struct dsa_prof_rec {
  int kind;
  cudaEvent_t ev0, ev1;
};

struct dsa_ctx {
  int device;
  int num_sms;
  float theta;
  float eps;
  int max_pos;
  // RoPE (cos, sin) in fp32, [max_pos][32] float4, lane-interleaved: float4
  // 8v + j of a row holds pairs 8j + 2v and 8j + 2v + 1 (j < 8, v < 4)
  float4* rope;
  int hadamard;          // store keys rotated by the 128-point Walsh-Hadamard transform
  int slot_output;       // top-k returns cache slots instead of positions
  float* gamma;          // [128]
  unsigned int* status;  // device status word
  void* encode_tiled;    // cuTensorMapEncodeTiled entry point
  // kernel timing (dsa_profile_*)
  int prof_on;
  int prof_n;                    // records in use
  dsa_prof_rec* prof;            // kProfCap records, events created on enable
  long long launches[DSA_K_COUNT];
};

namespace dsa {
constexpr int kProfCap = 8192;

// Every call that enqueues work first checks that the calling thread's
// current device is the context's: the kernels launch on the current device
// but read the context's device memory (table, gamma, status word), so a
// call made with another device current is rejected before anything is
// enqueued. Returns DSA_ERR_CUDA when no device can be queried.
inline dsa_status check_device(const dsa_ctx* ctx) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return DSA_ERR_CUDA;
  return dev == ctx->device ? DSA_OK : DSA_ERR_INVALID_ARG;
}
// Record the start/end of one kernel launch of kind `kind` on `stream`.
struct LaunchScope {
  dsa_ctx* ctx;
  int kind;
  dsa_prof_rec* rec;
  cudaStream_t stream;
  LaunchScope(dsa_ctx* c, int k, cudaStream_t s) : ctx(c), kind(k), rec(nullptr), stream(s) {
    ctx->launches[kind] += 1;
    if (ctx->prof_on && ctx->prof_n < kProfCap) {
      rec = &ctx->prof[ctx->prof_n++];
      rec->kind = kind;
      cudaEventRecord(rec->ev0, stream);
    }
  }
  ~LaunchScope() {
    if (rec) cudaEventRecord(rec->ev1, stream);
  }
};

// Launch with programmatic dependent launch allowed: the kernel may start
// while the previous kernel on the stream is still running, so every kernel
// launched this way executes griddepcontrol.wait before it reads global
// memory that a predecessor may write.
template <typename... Kargs, typename... Args>
cudaError_t launch_pdl(void (*kern)(Kargs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
}  // namespace dsa

namespace dsa {

dsa_status launch_store(dsa_ctx* ctx, const void* k_raw, const int32_t* pos, const int32_t* seq,
                        const int32_t* page_table, int32_t T, int32_t B, int32_t max_pages,
                        void* cache, int32_t num_pages, dsa_fmt fmt, cudaStream_t stream);

size_t topk_workspace(const dsa_ctx* ctx, int32_t Tq, int32_t B, int32_t k, dsa_fmt fmt);
int max_sequences();  // largest B dsa_index_topk accepts

dsa_status launch_topk(dsa_ctx* ctx, const void* q, const float* head_w, const void* cache,
                       int32_t num_pages, dsa_fmt fmt, const int32_t* page_table,
                       int32_t max_pages, const int32_t* seq_lens, const int32_t* cu_q,
                       int32_t B, int32_t Tq, int32_t causal, int32_t k, int32_t* out_idx,
                       float* out_score, void* workspace, size_t ws_bytes, cudaStream_t stream);

}  // namespace dsa
