// C ABI of libdsaidx: context set-up (RoPE table, gamma, status word),
// argument validation, and dispatch to the store and top-k launchers.
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <new>
#include <vector>

#include "internal.cuh"
#include "ptx.cuh"

namespace {

// Self-test of the bounded waits: thread 0 waits on a shared-memory
// mbarrier that nothing ever arrives at, with the scorer's wait and a budget
// of `budget` clock cycles, then records DSA_DEV_TIMEOUT the way the scorer
// does when a pipeline wait runs out, and the kernel returns.
__global__ void bounded_wait_probe(unsigned int* status, long long budget) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    dsa::mbar_init(&bar, 1);
    dsa::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !dsa::mbar_wait(&bar, 0, budget)) atomicOr(status, DSA_DEV_TIMEOUT);
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

cudaStream_t as_stream(dsa_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

}  // namespace

extern "C" {

const char* dsa_status_str(dsa_status s) {
  switch (s) {
    case DSA_OK: return "ok";
    case DSA_ERR_INVALID_ARG: return "invalid argument";
    case DSA_ERR_UNSUPPORTED: return "unsupported";
    case DSA_ERR_CUDA: return "CUDA error";
    case DSA_ERR_DEVICE_BOUNDS: return "device saw an out-of-range page id, position or sequence";
    case DSA_ERR_TIMEOUT: return "a bounded device wait ran out";
    case DSA_ERR_WORKSPACE: return "workspace too small";
  }
  return "unknown status";
}

size_t dsa_cache_page_bytes(dsa_fmt fmt) {
  if (fmt == DSA_FMT_BF16) return DSA_PAGE_SIZE * DSA_HEAD_DIM * 2;
  if (fmt == DSA_FMT_FP8) return DSA_PAGE_SIZE * DSA_HEAD_DIM + DSA_PAGE_SIZE * 4;
  if (fmt == DSA_FMT_FP4) return DSA_PAGE_SIZE * DSA_HEAD_DIM / 2 + DSA_PAGE_SIZE * 4;
  return 0;
}

dsa_status dsa_ctx_create(dsa_ctx** out, float rope_theta, float rms_eps, int32_t max_pos,
                          const uint16_t* gamma_bf16) {
  if (!out || !(rope_theta > 0.f) || !(rms_eps >= 0.f) || max_pos <= 0) return DSA_ERR_INVALID_ARG;
  *out = nullptr;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DSA_ERR_CUDA;
  int major = 0, minor = 0, sms = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return DSA_ERR_CUDA;
  if (major != 10 || minor != 3) return DSA_ERR_UNSUPPORTED;

  void* fn = nullptr;
  cudaDriverEntryPointQueryResult qres;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &qres) != cudaSuccess ||
      qres != cudaDriverEntryPointSuccess || !fn)
    return DSA_ERR_CUDA;

  // RoPE table: angle pos * theta^(-2i/128) in double, cos/sin rounded once
  // to fp32, stored lane-interleaved for the store kernel: float4 8v + j of a
  // row holds pairs 8j + 2v and 8j + 2v + 1
  const size_t n = static_cast<size_t>(max_pos) * 32;
  std::vector<float4> tab(n);
  double freq[64];
  for (int i = 0; i < 64; ++i) freq[i] = std::pow(static_cast<double>(rope_theta), -(2.0 * i) / 128.0);
  for (int32_t p = 0; p < max_pos; ++p) {
    float cs[128];
    for (int i = 0; i < 64; ++i) {
      const double a = static_cast<double>(p) * freq[i];
      cs[2 * i] = static_cast<float>(std::cos(a));
      cs[2 * i + 1] = static_cast<float>(std::sin(a));
    }
    for (int j = 0; j < 8; ++j)
      for (int v = 0; v < 4; ++v) {
        const float* q = cs + 2 * (8 * j + 2 * v);
        tab[static_cast<size_t>(p) * 32 + 8 * v + j] = make_float4(q[0], q[1], q[2], q[3]);
      }
  }
  // gamma (fp32), interleaved the same way: float4 l holds dims 8l..8l+3 and
  // float4 16 + l dims 8l+4..8l+7
  float gl[128];
  for (int d = 0; d < 128; ++d) {
    if (gamma_bf16) {
      const uint32_t b = static_cast<uint32_t>(gamma_bf16[d]) << 16;
      std::memcpy(&gl[d], &b, 4);
    } else {
      gl[d] = 1.0f;
    }
  }
  float g[128];
  for (int l = 0; l < 16; ++l)
    for (int e = 0; e < 4; ++e) {
      g[4 * l + e] = gl[8 * l + e];
      g[64 + 4 * l + e] = gl[8 * l + 4 + e];
    }

  dsa_ctx* c = new (std::nothrow) dsa_ctx();
  if (!c) return DSA_ERR_CUDA;
  c->device = dev;
  c->num_sms = sms;
  c->theta = rope_theta;
  c->eps = rms_eps;
  c->max_pos = max_pos;
  c->encode_tiled = fn;
  bool okk = cudaMalloc(&c->rope, n * sizeof(float4)) == cudaSuccess &&
             cudaMalloc(&c->gamma, 128 * sizeof(float)) == cudaSuccess &&
             cudaMalloc(&c->status, sizeof(unsigned int)) == cudaSuccess &&
             cudaMemcpy(c->rope, tab.data(), n * sizeof(float4), cudaMemcpyHostToDevice) == cudaSuccess &&
             cudaMemcpy(c->gamma, g, sizeof(g), cudaMemcpyHostToDevice) == cudaSuccess &&
             cudaMemset(c->status, 0, sizeof(unsigned int)) == cudaSuccess;
  if (!okk) {
    cudaFree(c->rope);
    cudaFree(c->gamma);
    cudaFree(c->status);
    delete c;
    return DSA_ERR_CUDA;
  }
  *out = c;
  return DSA_OK;
}

dsa_status dsa_ctx_destroy(dsa_ctx* ctx) {
  if (!ctx) return DSA_ERR_INVALID_ARG;
  // free on the context's device, whichever device is current, and restore it
  int cur = -1;
  const bool have_cur = cudaGetDevice(&cur) == cudaSuccess;
  if (have_cur && cur != ctx->device) cudaSetDevice(ctx->device);
  cudaDeviceSynchronize();
  cudaFree(ctx->rope);
  cudaFree(ctx->gamma);
  cudaFree(ctx->status);
  if (ctx->prof) {
    for (int i = 0; i < dsa::kProfCap; ++i) {
      cudaEventDestroy(ctx->prof[i].ev0);
      cudaEventDestroy(ctx->prof[i].ev1);
    }
    delete[] ctx->prof;
  }
  delete ctx;
  if (have_cur && cur >= 0) cudaSetDevice(cur);
  return DSA_OK;
}

dsa_status dsa_ctx_set_hadamard(dsa_ctx* ctx, int32_t on) {
  if (!ctx) return DSA_ERR_INVALID_ARG;
  ctx->hadamard = on ? 1 : 0;
  return DSA_OK;
}

dsa_status dsa_ctx_set_slot_output(dsa_ctx* ctx, int32_t on) {
  if (!ctx) return DSA_ERR_INVALID_ARG;
  ctx->slot_output = on ? 1 : 0;
  return DSA_OK;
}

dsa_status dsa_profile_enable(dsa_ctx* ctx, int on) {
  if (!ctx) return DSA_ERR_INVALID_ARG;
  if (on && !ctx->prof) {
    ctx->prof = new (std::nothrow) dsa_prof_rec[dsa::kProfCap];
    if (!ctx->prof) return DSA_ERR_CUDA;
    for (int i = 0; i < dsa::kProfCap; ++i) {
      if (cudaEventCreate(&ctx->prof[i].ev0) != cudaSuccess ||
          cudaEventCreate(&ctx->prof[i].ev1) != cudaSuccess)
        return DSA_ERR_CUDA;
    }
  }
  ctx->prof_on = on ? 1 : 0;
  return DSA_OK;
}

dsa_status dsa_profile_read(dsa_ctx* ctx, float* ms, int32_t* launches) {
  if (!ctx || !ms || !launches) return DSA_ERR_INVALID_ARG;
  if (const dsa_status d = dsa::check_device(ctx)) return d;
  for (int k = 0; k < DSA_K_COUNT; ++k) {
    ms[k] = 0.f;
    launches[k] = static_cast<int32_t>(ctx->launches[k]);
    ctx->launches[k] = 0;
  }
  if (cudaDeviceSynchronize() != cudaSuccess) return DSA_ERR_CUDA;
  for (int i = 0; i < ctx->prof_n; ++i) {
    float t = 0.f;
    if (cudaEventElapsedTime(&t, ctx->prof[i].ev0, ctx->prof[i].ev1) != cudaSuccess) return DSA_ERR_CUDA;
    ms[ctx->prof[i].kind] += t;
  }
  ctx->prof_n = 0;
  return DSA_OK;
}

dsa_status dsa_selftest_bounded_wait(dsa_ctx* ctx, dsa_stream_t stream) {
  if (!ctx) return DSA_ERR_INVALID_ARG;
  if (const dsa_status d = dsa::check_device(ctx)) return d;
  bounded_wait_probe<<<1, 32, 0, as_stream(stream)>>>(ctx->status, 2000000LL);  // about 1 ms
  return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

dsa_status dsa_get_device_status(dsa_ctx* ctx, dsa_stream_t stream) {
  if (!ctx) return DSA_ERR_INVALID_ARG;
  if (const dsa_status d = dsa::check_device(ctx)) return d;
  unsigned int w = 0;
  if (cudaStreamSynchronize(as_stream(stream)) != cudaSuccess) return DSA_ERR_CUDA;
  if (cudaMemcpy(&w, ctx->status, sizeof(w), cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemset(ctx->status, 0, sizeof(w)) != cudaSuccess)
    return DSA_ERR_CUDA;
  if (w & DSA_DEV_BOUNDS) return DSA_ERR_DEVICE_BOUNDS;
  if (w & DSA_DEV_TIMEOUT) return DSA_ERR_TIMEOUT;
  return DSA_OK;
}

dsa_status dsa_index_store(dsa_ctx* ctx, const void* k_raw, const int32_t* rope_pos,
                           const int32_t* seq_id, const int32_t* page_table, int32_t T,
                           int32_t B, int32_t max_pages, void* cache, int32_t num_pages,
                           dsa_fmt fmt, dsa_stream_t stream) {
  if (!ctx) return DSA_ERR_INVALID_ARG;
  if (fmt != DSA_FMT_BF16 && fmt != DSA_FMT_FP8 && fmt != DSA_FMT_FP4) return DSA_ERR_UNSUPPORTED;
  if (T < 0 || B <= 0 || max_pages <= 0 || num_pages <= 0) return DSA_ERR_INVALID_ARG;
  if (T == 0) return DSA_OK;
  if (!k_raw || !rope_pos || !seq_id || !page_table || !cache) return DSA_ERR_INVALID_ARG;
  if (!aligned(k_raw, 16) || !aligned(cache, 256) || !aligned(rope_pos, 4) || !aligned(seq_id, 4) ||
      !aligned(page_table, 4))
    return DSA_ERR_INVALID_ARG;
  if (const dsa_status d = dsa::check_device(ctx)) return d;
  return dsa::launch_store(ctx, k_raw, rope_pos, seq_id, page_table, T, B, max_pages, cache,
                           num_pages, fmt, as_stream(stream));
}

size_t dsa_index_topk_workspace_size(const dsa_ctx* ctx, int32_t Tq, int32_t B, int32_t k,
                                     dsa_fmt fmt) {
  if (!ctx || Tq < 0 || B <= 0 || k < 1 || k > 2048) return 0;
  if (fmt != DSA_FMT_BF16 && fmt != DSA_FMT_FP8 && fmt != DSA_FMT_FP4) return 0;
  return dsa::topk_workspace(ctx, Tq, B, k, fmt);
}

dsa_status dsa_index_topk(dsa_ctx* ctx, const void* q, const float* head_w, const void* cache,
                          int32_t num_pages, dsa_fmt fmt, const int32_t* page_table,
                          int32_t max_pages, const int32_t* seq_lens, const int32_t* cu_q,
                          int32_t B, int32_t Tq, int32_t causal, int32_t k, int32_t* out_idx,
                          float* out_score, void* workspace, size_t ws_bytes,
                          dsa_stream_t stream) {
  if (!ctx) return DSA_ERR_INVALID_ARG;
  if (fmt != DSA_FMT_BF16 && fmt != DSA_FMT_FP8 && fmt != DSA_FMT_FP4) return DSA_ERR_UNSUPPORTED;
  if (k < 1 || k > 2048) return DSA_ERR_UNSUPPORTED;
  if (Tq < 0 || B <= 0 || max_pages <= 0 || num_pages <= 0) return DSA_ERR_INVALID_ARG;
  if (static_cast<long long>(num_pages) * 64 > 0x7FFFFFFFLL) return DSA_ERR_UNSUPPORTED;
  if (B > dsa::max_sequences()) return DSA_ERR_UNSUPPORTED;
  if (Tq == 0) return DSA_OK;
  if (!q || !head_w || !cache || !page_table || !seq_lens || !cu_q || !out_idx || !out_score ||
      !workspace)
    return DSA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(cache, 256) || !aligned(workspace, 256) || !aligned(head_w, 16) ||
      !aligned(out_idx, 4) || !aligned(out_score, 4))
    return DSA_ERR_INVALID_ARG;
  if (const dsa_status d = dsa::check_device(ctx)) return d;
  if (ws_bytes < dsa::topk_workspace(ctx, Tq, B, k, fmt)) return DSA_ERR_WORKSPACE;
  return dsa::launch_topk(ctx, q, head_w, cache, num_pages, fmt, page_table, max_pages, seq_lens,
                          cu_q, B, Tq, causal ? 1 : 0, k, out_idx, out_score, workspace, ws_bytes,
                          as_stream(stream));
}

}  // extern "C"
