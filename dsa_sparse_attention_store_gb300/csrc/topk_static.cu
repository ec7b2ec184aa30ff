// dsa_index_topk_static: dsa_index_topk for callers that cannot allocate
// device memory.
//
// Some callers cannot hand this library a workspace: a serving engine that
// has already carved all free device memory into its own pools (KV cache,
// activations) and forbids allocations outside them, or a caller on a
// latency-critical path where cudaMalloc/cudaFree would add implicit device
// synchronisation or could fail under memory pressure. This entry point runs
// the same kernels as dsa_index_topk but takes its scratch from a fixed
// array that is part of the library's device image, so the call allocates
// nothing.
//
// The array is a file-scope __device__ variable of DSA_STATIC_WORKSPACE_BYTES:
// every GPU that loads the library holds it until the process exits. Host
// code cannot use the array's name as a device address, so the address is
// looked up with cudaGetSymbolAddress once per device, on the first call made
// with that device current (make that first call before any stream capture),
// and again if the device's CUDA context has changed since (after a device
// reset the module is loaded anew and the array may have moved).
// All calls share the array and it keeps the last call's contents: calls that
// overlap on the GPU (different streams, or different threads without
// ordering) race on it. Nothing in it needs clearing between calls: the
// schedule kernel that starts every call rewrites the only fields that must
// start at zero (the split-merge counters), and every other field is written
// before it is read within the call.
#include <mutex>

#include "internal.cuh"

static __device__ __align__(256) unsigned char g_dsa_static_ws[DSA_STATIC_WORKSPACE_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_ptr[kMaxDevices] = {};
CUcontext g_owner[kMaxDevices] = {};  // the CUDA context the cached address belongs to

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);

// The calling thread's current CUDA context (null if it cannot be read).
CUcontext current_context() {
  static CtxGetCurrentFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<CtxGetCurrentFn>(nullptr);
    return reinterpret_cast<CtxGetCurrentFn>(p);
  }();
  CUcontext c = nullptr;
  if (!fn || fn(&c) != CUDA_SUCCESS) return nullptr;
  return c;
}

// Device address of the scratch array for the current device. Looked up
// once per device and CUDA context: after a device reset the runtime loads
// the module again in a new context, where the array may sit elsewhere, so a
// changed context triggers a new lookup.
dsa_status static_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DSA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return DSA_ERR_UNSUPPORTED;
  const CUcontext cur = current_context();
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_ptr[dev] || !cur || g_owner[dev] != cur) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_dsa_static_ws) != cudaSuccess || !p) return DSA_ERR_CUDA;
    g_ptr[dev] = p;
    g_owner[dev] = current_context();  // the lookup made the device's context current
  }
  *out = g_ptr[dev];
  return DSA_OK;
}

bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3) == 0; }

}  // namespace

extern "C" dsa_status dsa_index_topk_static(dsa_ctx* ctx, const void* q, const float* head_w,
                                            const void* cache, int32_t num_pages, dsa_fmt fmt,
                                            const int32_t* page_table, int32_t max_pages,
                                            const int32_t* seq_lens, const int32_t* cu_q,
                                            int32_t B, int32_t Tq, int32_t causal, int32_t k,
                                            int32_t* out_idx, float* out_score,
                                            dsa_stream_t stream) {
  if (!ctx) return DSA_ERR_INVALID_ARG;
  if (fmt != DSA_FMT_BF16 && fmt != DSA_FMT_FP8 && fmt != DSA_FMT_FP4) return DSA_ERR_UNSUPPORTED;
  if (k < 1 || k > 2048) return DSA_ERR_UNSUPPORTED;
  if (Tq < 0 || B <= 0 || max_pages <= 0 || num_pages <= 0) return DSA_ERR_INVALID_ARG;
  if (static_cast<long long>(num_pages) * 64 > 0x7FFFFFFFLL) return DSA_ERR_UNSUPPORTED;
  if (B > dsa::max_sequences()) return DSA_ERR_UNSUPPORTED;
  if (Tq == 0) return DSA_OK;
  if (!q || !head_w || !cache || !page_table || !seq_lens || !cu_q || !out_idx || !out_score)
    return DSA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(q) & 15) || (reinterpret_cast<uintptr_t>(cache) & 255) ||
      (reinterpret_cast<uintptr_t>(head_w) & 15) || !aligned4(out_idx) || !aligned4(out_score))
    return DSA_ERR_INVALID_ARG;
  if (const dsa_status d = dsa::check_device(ctx)) return d;
  // the sizes must fit the fixed scratch array; nothing is allocated instead
  if (dsa::topk_workspace(ctx, Tq, B, k, fmt) > static_cast<size_t>(DSA_STATIC_WORKSPACE_BYTES))
    return DSA_ERR_WORKSPACE;
  void* ws = nullptr;
  const dsa_status st = static_scratch(&ws);
  if (st != DSA_OK) return st;
  return dsa::launch_topk(ctx, q, head_w, cache, num_pages, fmt, page_table, max_pages, seq_lens,
                          cu_q, B, Tq, causal ? 1 : 0, k, out_idx, out_score, ws,
                          static_cast<size_t>(DSA_STATIC_WORKSPACE_BYTES),
                          reinterpret_cast<cudaStream_t>(stream));
}
