/*
 * libdsaidx -- the DeepSeek Sparse Attention (DSA) indexer hot path on one
 * GB300 GPU: the index-key store and the score + top-k selection.
 *
 * Sources (web pages on the bf16 index-K fix in the DSA indexer):
 *  [VAL] "The Moment of Validation: Diagnosing an OOM Crash in the bf16 Index-K
 *        Fix for DeepSeek V4 Sparse Attention", section "Input Knowledge
 *        Required to Understand This Message": fp8 index keys take 128 bytes of
 *        data plus a 4-byte scale (132 B/token), bf16 keys 128 x 2 = 256
 *        B/token; the fused store normalises, applies RoPE and stores in one
 *        kernel call.
 *  [DEC] "The Fused Kernel Decision: Precision Archaeology in the CUDA Sparse
 *        Attention Indexer", section "The Message": the indexer buffer is
 *        paged, page_size = 64, [npages, 64*128] bf16; each token maps to a
 *        page and an offset and its 128 values are written there.
 *  [CRA] "The Crash That Changed Direction", sections "The Experiment: Why
 *        fp32?" and "Assumptions Made and Broken": scores come from a batched
 *        matrix product of queries and index keys followed by a ReLU; the
 *        pages up-convert fp8 keys exactly before the product (this library
 *        gives them to the tensor cores as stored, see dsa_index_topk); the
 *        top-512 (or 1024) key positions are kept.
 *  [WFK] "When the Fused Kernel Isn't Enough", section "The Message:
 *        Validation and Discovery": materialising the logits over the whole
 *        context ran out of memory at about 22K tokens. This library never
 *        materialises the [q_len x ctx] logits: key tiles stream through a
 *        running per-query top-k.
 *
 * Conventions for every call:
 *  - Pointers marked (device) are CUDA device pointers owned by the caller;
 *    pointers marked (host) are host memory. The library keeps no pointer
 *    after a call returns.
 *  - Work is enqueued on `stream` and is asynchronous; argument errors are
 *    returned before anything is enqueued. Calls that enqueue work must be
 *    made with the context's device current (the one current at
 *    dsa_ctx_create); otherwise they return DSA_ERR_INVALID_ARG and enqueue
 *    nothing. A launch failure returns
 *    DSA_ERR_CUDA. Errors found on the device (a page id out of range, a
 *    bounded wait that ran out) do not trap: the kernel skips the access,
 *    records the error in a status word of the context and carries on;
 *    dsa_get_device_status() reads and clears it.
 *  - Sizes are int32 element counts; the byte layouts are stated per call.
 *  - Index heads H = 64 and head_dim D = 128 are fixed. Page size is 64.
 */
#ifndef DSAIDX_H
#define DSAIDX_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* dsa_stream_t; /* a cudaStream_t; NULL = legacy default stream */

typedef enum {
  DSA_OK = 0,
  DSA_ERR_INVALID_ARG = 1,   /* null pointer, negative size, misaligned pointer ... */
  DSA_ERR_UNSUPPORTED = 2,   /* k not in 1..2048, unknown format, no sm_103 device */
  DSA_ERR_CUDA = 3,          /* a CUDA runtime/driver call failed */
  DSA_ERR_DEVICE_BOUNDS = 4, /* device saw a page id / position / sequence out of range (or a
                                top-k candidate buffer would have overflowed: the keys are
                                dropped, never written past the buffer) */
  DSA_ERR_TIMEOUT = 5,       /* a bounded device-side wait ran out */
  DSA_ERR_WORKSPACE = 6      /* workspace too small */
} dsa_status;

typedef enum {
  DSA_FMT_BF16 = 0, /* 128 bf16 per token = 256 B; page = [64][128] bf16 = 16384 B      [DEC] */
  DSA_FMT_FP8 = 1,  /* 128 e4m3 + 1 fp32 scale = 132 B per token; page = [64][128] e4m3
                       followed by [64] fp32 scales = 8448 B                            [VAL] */
  DSA_FMT_FP4 = 2   /* 128 e2m1 (OCP MX FP4: 1 sign, 2 exponent bits with bias 1, 1
                       mantissa bit; magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6) packed two
                       per byte, the even dimension in the low nibble, + 1 fp32 scale
                       = 68 B per token; page = [64][64] code bytes followed by [64]
                       fp32 scales = 4352 B. [DEC], section "The Message: A Blueprint
                       for Kernel Modification", names an fp4 variant of the indexer
                       kernel for more aggressive compression without a layout; this
                       one is the fp8 key with its element type narrowed to e2m1. */
} dsa_fmt;

enum { DSA_HEADS = 64, DSA_HEAD_DIM = 128, DSA_PAGE_SIZE = 64 };

typedef struct dsa_ctx dsa_ctx; /* opaque; one per device */

/* Create a context on the current CUDA device.
 *  rope_theta  RoPE base theta (> 0); frequency of pair i is theta^(-2i/128).
 *  rms_eps     RMSNorm epsilon (>= 0).
 *  max_pos     positions the store accepts are 0 .. max_pos-1 (> 0). The
 *              context holds a cos/sin table of max_pos x 64 x 8 bytes built
 *              on the host in double precision and rounded to fp32.
 *  gamma_bf16  (host) 128 bf16 RMSNorm weights, or NULL for all ones.
 * Allocates device memory (the table, gamma, a status word). Returns
 * DSA_ERR_UNSUPPORTED if the device is not compute capability 10.3. */
dsa_status dsa_ctx_create(dsa_ctx** out, float rope_theta, float rms_eps, int32_t max_pos,
                          const uint16_t* gamma_bf16);

/* Free the context's device memory. Synchronises the device first. */
dsa_status dsa_ctx_destroy(dsa_ctx* ctx);

/* Bytes per cache page for a format (16384, 8448 or 4352); 0 for an unknown format. */
size_t dsa_cache_page_bytes(dsa_fmt fmt);

/* Index-key store ([VAL], [DEC]): for each token t,
 *   y  = RMSNorm(k_raw[t]) * gamma            (fp32, eps = rms_eps)
 *   y' = RoPE(y, rope_pos[t])                 (dims i and i+64 rotated together)
 *   written to page page_table[seq_id[t]][rope_pos[t] / 64], slot rope_pos[t] % 64:
 *   bf16: round-to-nearest-even of y'; fp8: scale = max(max|y'|, 1e-4) / 448,
 *   e4m3 (round to nearest even, saturating) of y' * (1/scale), and the scale;
 *   fp4: the same with 6 for 448 and e2m1 for e4m3.
 * The fp32 operations follow one fixed order, so the stored bytes are
 * reproducible bit for bit (sum of squares: 16 sequential partials over 8
 * consecutive dims, then a pairwise tree; every product and sum of the
 * rotation rounded separately).
 *  k_raw       (device) [T][128] bf16, 16-byte aligned rows.
 *  rope_pos    (device) [T] int32: the token's position in its sequence; also
 *              its cache position. Must be in [0, min(max_pos, 64*max_pages)).
 *  seq_id      (device) [T] int32 in [0, B).
 *  page_table  (device) [B][max_pages] int32 page ids in [0, num_pages).
 *  cache       (device) num_pages * dsa_cache_page_bytes(fmt) bytes, 256-byte aligned.
 * Tokens must not share a slot within one call. Out-of-range seq/pos/page on
 * the device: the token is skipped and DSA_ERR_DEVICE_BOUNDS is recorded. */
dsa_status dsa_index_store(dsa_ctx* ctx, const void* k_raw, const int32_t* rope_pos,
                           const int32_t* seq_id, const int32_t* page_table, int32_t T,
                           int32_t B, int32_t max_pages, void* cache, int32_t num_pages,
                           dsa_fmt fmt, dsa_stream_t stream);

/* Hadamard rotation ("The Moment of Validation", section "Input Knowledge
 * Required to Understand This Message": the fused store applies a Hadamard
 * transform between RoPE and quantisation; "The Fused Kernel Decision",
 * section "Assumptions and Their Validity": queries and keys must use the
 * same order). When on, dsa_index_store writes H y' instead of y', H the
 * unnormalised 128-point Walsh-Hadamard transform in natural (Sylvester)
 * order (entries +-1, fp32 butterflies h = 1, 2, ..., 64, each pair
 * (i, i+h) -> (a + b, a - b)), and dsa_index_topk rotates every query head by
 * the same H and divides the dot products by 128, so scores keep their
 * meaning: (H q) . (H k) / 128 = q . k. The query is rotated exactly, as far
 * as the scores can tell: the fp32 rotation is carried as two bf16 terms
 * (hi + lo, 16 significant bits) for bf16 caches and three e4m3 terms (12
 * bits) for fp8 and fp4 caches, each term its own pass of the tensor cores,
 * and the queries run in tiles of two queries of one sequence (one for a
 * decode batch, one query per sequence) instead of four.
 * A cache must be written and read with the same setting. Off by default;
 * applies to the calls made after it, and changes the size
 * dsa_index_topk_workspace_size reports. */
dsa_status dsa_ctx_set_hadamard(dsa_ctx* ctx, int32_t on);

/* Slot output: when on, dsa_index_topk writes into out_idx the cache slot of
 * each selected key, page_table[b][pos / 64] * 64 + pos % 64 (the row the
 * sparse attention gathers), instead of its position pos; padding stays -1.
 * The pages feed the selected tokens to the attention ("The Crash That
 * Changed Direction", section "The Experiment: Why fp32?"); the slot is what
 * a paged gather needs. Off by default; applies to the calls made after it. */
dsa_status dsa_ctx_set_slot_output(dsa_ctx* ctx, int32_t on);

/* Upper bound of the workspace bytes dsa_index_topk needs for these sizes.
 * It does not grow with the context length: it holds the schedule
 * (O(Tq + B)), split-context partial lists (O(#SMs * k)) and one shared
 * threshold per query (8 bytes). The same for both cache formats: the
 * queries are turned into their tensor-core terms inside the scorer, in
 * shared memory. */
size_t dsa_index_topk_workspace_size(const dsa_ctx* ctx, int32_t Tq, int32_t B, int32_t k,
                                     dsa_fmt fmt);

/* Score + top-k ([CRA]): for each query row r of sequence b (rows
 * cu_q[b] .. cu_q[b+1]-1, position p = seq_lens[b] - n_q(b) + j for the j-th),
 *   s[r, key] = sum_h head_w[r][h] * max(0, sum_d q[r][h][d] * k[key][d])
 * over the visible keys of sequence b: positions 0..p when causal, else
 * 0..seq_lens[b]-1; k is the stored key (fp8 / fp4: e4m3 / e2m1 value times
 * its scale).
 * Output row r holds the positions (within the sequence) and fp32 scores of
 * the min(k, visible) best keys, ordered by (score desc, position asc);
 * unused slots are -1 / -inf. Products accumulate in fp32. For fp8 caches
 * the stored e4m3 keys enter the tensor cores as they are and each query row
 * (one head) as two e4m3 terms under a power-of-two scale: exact for every
 * query value of at least 2^-10 of its row's largest magnitude, smaller
 * values off by at most 2^-17 of that magnitude. fp4 caches take the same
 * path: the scorer widens each tile's e2m1 codes to e4m3 in shared memory
 * (exact: every e2m1 value is an e4m3 value), so only the bytes read from
 * memory shrink.
 *  q           (device) [Tq][64][128] bf16, 16-byte aligned.
 *  head_w      (device) [Tq][64] fp32, 16-byte aligned.
 *  cache       (device) as written by dsa_index_store, num_pages pages of fmt.
 *  page_table  (device) [B][max_pages] int32; entries past a sequence's last
 *              page are not read.
 *  seq_lens    (device) [B] int32, n_q(b) <= seq_lens[b] <= 64*max_pages.
 *  cu_q        (device) [B+1] int32, cu_q[0] = 0, non-decreasing, cu_q[B] = Tq.
 *  k           1 .. 2048 (the pages use 512 and 1024, and a downstream
 *              gather may take 2048; other k run the top-512, top-1024 or
 *              top-2048 selection and keep the first k of each sorted row;
 *              k > 1024 runs in one-query tiles, the decode kernel, whatever
 *              the batch: a 2048-key candidate buffer only fits there).
 *              B <= 16384 and Tq < 2^25, else DSA_ERR_UNSUPPORTED.
 *  out_idx     (device) [Tq][k] int32;  out_score (device) [Tq][k] fp32.
 *  workspace   (device) >= dsa_index_topk_workspace_size(...) bytes, 256-byte
 *              aligned; contents need not be initialised and are scratch.
 * Scratch memory is O(#SMs * tile) + O(Tq * k): the logits are never stored. */
dsa_status dsa_index_topk(dsa_ctx* ctx, const void* q, const float* head_w, const void* cache,
                          int32_t num_pages, dsa_fmt fmt, const int32_t* page_table,
                          int32_t max_pages, const int32_t* seq_lens, const int32_t* cu_q,
                          int32_t B, int32_t Tq, int32_t causal, int32_t k, int32_t* out_idx,
                          float* out_score, void* workspace, size_t ws_bytes,
                          dsa_stream_t stream);

/* Allocation-free top-k, for callers that cannot allocate device memory
 * (an engine whose memory is already carved into its own pools, or a
 * latency-critical path that must not call cudaMalloc). The pages have no
 * counterpart; it is an addition of this library.
 * Same arguments and results as dsa_index_topk, without the workspace: the
 * scratch is a fixed array of DSA_STATIC_WORKSPACE_BYTES in the library's
 * device image, held by every GPU that loads the library until exit. The
 * call allocates nothing. Its first call on a device looks up the array's
 * device address (cudaGetSymbolAddress); make that first call before any
 * stream capture. A device reset (cudaDeviceReset) invalidates that address:
 * the next call notices the new CUDA context and looks it up again, so make
 * it, too, outside a capture. All calls share the array: calls that overlap on the GPU
 * race. Nothing in it needs clearing; each call rewrites what must start at
 * zero. Returns DSA_ERR_WORKSPACE, without launching anything, when
 * dsa_index_topk_workspace_size(ctx, Tq, B, k, fmt) exceeds
 * DSA_STATIC_WORKSPACE_BYTES (on a 152-SM GB300 with one sequence: batches
 * up to about 1.29M queries with k <= 512 and 1.07M with 512 < k <= 1024,
 * any cache format; with the Hadamard rotation on, about 970K and 892K;
 * with k > 1024, about 549K, rotation on or off). */
#define DSA_STATIC_WORKSPACE_BYTES (32u << 20)
dsa_status dsa_index_topk_static(dsa_ctx* ctx, const void* q, const float* head_w,
                                 const void* cache, int32_t num_pages, dsa_fmt fmt,
                                 const int32_t* page_table, int32_t max_pages,
                                 const int32_t* seq_lens, const int32_t* cu_q, int32_t B,
                                 int32_t Tq, int32_t causal, int32_t k, int32_t* out_idx,
                                 float* out_score, dsa_stream_t stream);

/* Kernel timing, for benchmarks and profiling. While enabled, the library
 * records a CUDA event pair on the launch stream around each kernel it
 * launches (at most 8192 pairs between reads; later launches are counted but
 * not timed). dsa_profile_read synchronises the device, writes per-kind total
 * milliseconds and launch counts since the previous read (launches are
 * counted whether or not timing is on), and resets both. */
typedef enum {
  DSA_K_STORE = 0,      /* dsa_index_store */
  DSA_K_PLAN = 1,       /* dsa_index_topk: schedule */
  DSA_K_SCORE_BF16 = 2, /* dsa_index_topk: tensor-core scorer + running top-k, bf16 cache */
  DSA_K_SCORE_FP8 = 3,  /* the same, fp8 cache */
  DSA_K_SCORE_FP4 = 4,  /* the same, fp4 cache */
  DSA_K_COUNT = 5
} dsa_kernel_kind;
dsa_status dsa_profile_enable(dsa_ctx* ctx, int on);
dsa_status dsa_profile_read(dsa_ctx* ctx, float* ms /* [DSA_K_COUNT] */,
                            int32_t* launches /* [DSA_K_COUNT] */);

/* Synchronise `stream`, then read and clear the context's device status
 * word. Returns DSA_OK or the first device-side error recorded. */
dsa_status dsa_get_device_status(dsa_ctx* ctx, dsa_stream_t stream);

/* Failure-detection self-test: enqueues a one-CTA kernel that waits, with
 * the scorer's bounded mbarrier wait, on a barrier nothing ever signals;
 * after about a millisecond the wait gives up, DSA_ERR_TIMEOUT is recorded
 * in the status word (read it with dsa_get_device_status) and the kernel
 * returns, leaving the context usable. Exercises the error path of a stalled
 * pipeline without faulting or hanging the GPU. */
dsa_status dsa_selftest_bounded_wait(dsa_ctx* ctx, dsa_stream_t stream);

/* Static string for a status code. */
const char* dsa_status_str(dsa_status s);

#ifdef __cplusplus
}
#endif
#endif /* DSAIDX_H */
