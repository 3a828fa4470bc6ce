/*
 * dsa.h -- C ABI of libdsa.so: the GLM-5 DSA attention hot path on one
 * NVIDIA GB300 (sm_103a).
 *
 * The path has three steps, each an entry point below, plus one call that
 * runs all three:
 *
 *   1. dsa_indexer_scores -- lightning indexer.  For query position t and
 *      every causal history position s <= t
 *          I[t,s] = sum_{h<32} w[t,h] * ReLU( sum_{d<128} q_idx[t,h,d] * k_idx[s,d] )
 *      ("GLM-5.1 架构深度拆解", section 3.2 "Indexer 公式" Steps 4-5 and
 *      section 3.6 Step 5; the GLM-5 explainer page: 32 index queries of
 *      128 dims, one 128-dim index key per position, ReLU, 32 weights).
 *      Products and sums are fp32 (the pages cast both operands to fp32).
 *      Any positive softmax_scale factors out of the ReLU; fold it into w.
 *   2. dsa_topk -- causal top-k (section 3.6 Steps 6-7: positions s > t are
 *      masked, min(index_topk, length) positions are kept; section 3.4: the
 *      selection must be deterministic; explainer page: a query that sees
 *      fewer than 2048 positions keeps all of them).
 *   3. dsa_sparse_mla_fwd -- 64-head softmax attention over the selected
 *      rows of the latent cache, absorbed form: each cached row is
 *      [512 latent || 64 RoPE key] (section 2.5, section 4.2: the RoPE key
 *      is one stream shared by all heads), QK runs over all 576 columns and
 *      V is the first 512 (explainer page: the top-2048 ids only drive the
 *      gather; section 3.1 step 2: exact attention on the selected tokens).
 *   4. dsa_forward -- 1 -> 2 -> 3 for prefill, chunked prefill and decode.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - bf16 tensors are passed as their 16-bit patterns (uint16_t).
 *  - Every tensor pointer is a DEVICE pointer unless stated otherwise, and
 *    must be 16-byte aligned.  The caller owns every buffer; the library
 *    allocates nothing and keeps no pointer after a call returns.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls
 *    are stream-ordered and asynchronous; none synchronises except
 *    dsa_read_device_status.  Calls on different streams that share a
 *    workspace race.
 *  - Query rows of all sequences are packed: row r of sequence b is
 *    q_off[b] + i, i in [0, n_b), n_b = q_off[b+1] - q_off[b], and sits at
 *    position t = ctx_len[b] - n_b + i.  The caches hold sequence b's
 *    positions at rows b * cache_stride + s.  The caller appends the new
 *    tokens' cache rows before the call (the pages append the new index key
 *    before scoring it), so ctx_len counts them.
 *  - Host-side argument errors return DSA_ERR_INVALID_ARG and launch
 *    nothing.  Errors only the device can see (a q_off/ctx_len that breaks
 *    the bounds below, an index outside [-1, t]) skip the offending row,
 *    leave its outputs unwritten, and latch a code in the workspace's status
 *    word, read back by dsa_read_device_status.  Kernels never trap.
 */
#ifndef DSA_H
#define DSA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define DSA_API __attribute__((visibility("default")))
#else
#define DSA_API
#endif

#define DSA_INDEX_HEADS 32   /* index_n_heads */
#define DSA_INDEX_DIM 128    /* index_head_dim */
#define DSA_HEADS 64         /* num_attention_heads */
#define DSA_QK_DIM 576       /* kv_lora_rank 512 + qk_rope_head_dim 64 */
#define DSA_V_DIM 512        /* kv_lora_rank */
#define DSA_MAX_TOPK 2048    /* index_topk */
#define DSA_NOPE_DIM 192     /* qk_nope_head_dim */
#define DSA_ROPE_DIM 64      /* qk_rope_head_dim */
#define DSA_V_HEAD_DIM 256   /* v_head_dim */
#define DSA_KVB_ROWS 448     /* kv_b_proj output rows per head: 192 nope key + 256 value */
#define DSA_HIDDEN 6144      /* hidden size (o_proj output) */

typedef enum dsa_status {
    DSA_OK = 0,
    DSA_ERR_INVALID_ARG = 1, /* host-side argument check failed; nothing launched */
    DSA_ERR_UNSUPPORTED = 2, /* a shape or mode this build does not implement */
    DSA_ERR_WORKSPACE = 3,   /* ws is NULL or ws_bytes < dsa_workspace_size() */
    DSA_ERR_CUDA = 4,        /* a CUDA launch or runtime call failed */
    DSA_ERR_TIMEOUT = 5,     /* device: a bounded wait inside a kernel expired */
    DSA_ERR_BAD_BATCH = 6,   /* device: q_off / ctx_len outside the host bounds */
    DSA_ERR_BAD_INDEX = 7,   /* device: a selected index outside [-1, t] */
    DSA_ERR_INTERNAL = 8     /* device: an internal consistency check failed (a bug); the write was skipped */
} dsa_status;

/* One call's batch.  q_off and ctx_len are DEVICE int32 arrays, read by the
 * kernels: the lengths may change on the device between calls that keep the
 * same host arguments; the host only gives upper bounds, used to size grids.  Device-side requirements, checked
 * by the kernels (DSA_ERR_BAD_BATCH): q_off[0] = 0, q_off[batch] = total_q,
 * 0 <= n_b <= max_q, n_b <= ctx_len[b] <= max_ctx. */
typedef struct dsa_batch {
    int32_t batch;            /* B >= 1 sequences */
    int32_t total_q;          /* packed query rows, >= 0 */
    int32_t max_q;            /* bound on n_b */
    int32_t max_ctx;          /* bound on ctx_len[b]; <= cache_stride */
    int64_t cache_stride;     /* cache rows per sequence */
    const int32_t* q_off;     /* device [B+1] */
    const int32_t* ctx_len;   /* device [B] */
} dsa_batch;

/* Human-readable name of a status code (static storage, never NULL). */
DSA_API const char* dsa_status_string(int status);

/* Bytes of workspace that every call below needs for `batch` and top-k `k`
 * (the largest of them).  Host only; launches nothing. */
DSA_API dsa_status dsa_workspace_size(const dsa_batch* batch, int k, size_t* bytes);

/* Clears the device status word of a workspace (stream-ordered memset).
 * A fresh workspace must be cleared once before its first use. */
DSA_API dsa_status dsa_reset_device_status(void* ws, void* stream);

/* Synchronises `stream`, then copies the workspace's status word to *out
 * (DSA_OK if no kernel latched an error since the last reset). */
DSA_API dsa_status dsa_read_device_status(const void* ws, void* stream, dsa_status* out);

/* Text of the last CUDA error behind a DSA_ERR_CUDA returned to this host
 * thread ("no error" if none).  Thread-local, static storage. */
DSA_API const char* dsa_last_cuda_error(void);

/* Number of kernels this library has launched in this process so far (all
 * devices, all streams).  Instrumentation for benchmarks; host only. */
DSA_API uint64_t dsa_kernel_launch_count(void);

/* Diagnostic for the failure path: launches one CTA whose thread waits on a
 * barrier phase that nothing completes, bounded by limit_us (1 .. 10^6
 * microseconds).  The wait gives up, latches DSA_ERR_TIMEOUT in the status
 * word of ws (as every kernel of the path does when one of its bounded waits
 * expires) and the kernel returns normally: no trap, no hang, the context
 * stays usable.  Read the result with dsa_read_device_status. */
DSA_API dsa_status dsa_selftest_wait_timeout(void* ws, uint32_t limit_us, void* stream);

/* Step 1: lightning-indexer scores.
 *   q_idx  bf16 [total_q, 32, 128]  post-RoPE index queries
 *   w      fp32 [total_q, 32]       head weights
 *   k_idx  bf16 [batch * cache_stride, 128]  index-key cache
 *   scores fp32 [total_q, ld]       out: scores[r*ld + s] = I[t,s] for s <= t;
 *                                   entries s > t are not written
 * ld >= max_ctx, ld % 4 == 0.  Uses only the status word of ws. */
DSA_API dsa_status dsa_indexer_scores(const dsa_batch* batch, const uint16_t* q_idx, const float* w,
                              const uint16_t* k_idx, float* scores, int64_t ld, void* ws,
                              size_t ws_bytes, void* stream);

/* Step 2: causal top-k of score rows (as written by step 1).
 *   idx int32 [total_q, k]  out: the min(k, t+1) positions s <= t with the
 *       largest scores, ascending; entries past them are -1.  Scores are
 *       compared as fp32 values (-0.0 == +0.0); of equal scores the lower
 *       position wins.  Deterministic and bit-exact.  NaN scores are outside
 *       the contract.
 * 1 <= k <= 2048, ld >= max_ctx, ld % 4 == 0. */
DSA_API dsa_status dsa_topk(const dsa_batch* batch, const float* scores, int64_t ld, int k, int32_t* idx,
                    void* ws, size_t ws_bytes, void* stream);

/* Step 3: sparse MLA attention, absorbed form.
 *   q   bf16 [total_q, 64, 576]            absorbed queries
 *   kv  bf16 [batch * cache_stride, 576]   latent cache ([512 latent || 64 rope])
 *   idx int32 [total_q, k]                 selected positions, -1 = none
 *   out bf16 [total_q, 64, 512]            softmax(sm_scale * q.kv) @ kv[:, :512]
 *   lse fp32 [total_q, 64] or NULL         natural-log sum-exp of the logits
 * A row with no valid index gets out = 0 and lse = -inf.  Entries outside
 * [-1, t] latch DSA_ERR_BAD_INDEX and are skipped.
 * IndexShare ("GLM-5.2 架构 QA", Q2.1-Q2.2): a "shared" layer skips the
 * indexer and the top-k and reuses the indices of the last "full" layer;
 * it is this call with that layer's idx (dsa_forward's idx_out) and the
 * shared layer's own q and latent cache. */
DSA_API dsa_status dsa_sparse_mla_fwd(const dsa_batch* batch, const uint16_t* q, const uint16_t* kv,
                              const int32_t* idx, int k, float sm_scale, uint16_t* out, float* lse,
                              void* ws, size_t ws_bytes, void* stream);

/* Step 3 for callers that cannot allocate device memory.  The pages have no
 * counterpart to this call; it exists for integration.  Some callers cannot
 * allocate at the point where attention runs: serving loops that budget
 * every byte of device memory in advance and treat any allocation as a
 * failure, or embedders whose allocator is not reachable from the calling
 * thread.  This
 * call computes exactly what dsa_sparse_mla_fwd computes (same kernels, same
 * split of each query's selected list, so the same bits), but it takes no
 * workspace: its split-K partials live in a 32 MiB array of static device
 * memory owned by the library, which every GPU that loads the library holds
 * until the process exits.  It calls no cudaMalloc or cudaFree.
 *   device_status  optional DEVICE int32 (caller-owned, cleared by the
 *                  caller); device-side errors (indices outside [-1, t], a
 *                  batch outside its bounds) are latched there; NULL = not
 *                  reported.
 * Returns DSA_ERR_WORKSPACE, before launching anything, when the call's
 * partials would not fit in the 32 MiB array: each partial (one split of one
 * query row) takes 131,328 bytes, so at most 255 fit.  Rows split 2, 4 or 8
 * ways merge inside a CTA cluster and need no partials (64 decode rows at
 * k = 2048, 8 rows at k = 2048); 40 rows x 3 splits (k = 2048) take 15.8 MB;
 * 100 rows x 3 splits (k = 2047) do not fit.
 * The first call on a device looks up the array's device address (once per
 * device); make that first call before any stream capture.  The address
 * stays cached for the process: after cudaDeviceReset this call must not be
 * used again.  A launch failure returns DSA_ERR_CUDA and is reported by
 * dsa_last_cuda_error, like every other call.  Every call on a
 * device shares the one array, so calls whose kernels overlap on the GPU
 * (different streams, or different host threads) race and corrupt each
 * other's results: order them on one stream. */
DSA_API dsa_status dsa_sparse_mla_fwd_noalloc(const dsa_batch* batch, const uint16_t* q, const uint16_t* kv,
                                              const int32_t* idx, int k, float sm_scale, uint16_t* out,
                                              float* lse, int32_t* device_status, void* stream);

/* Steps 1-3 in one call (prefill, one chunk of a chunked prefill, or a
 * decode step).  idx_out [total_q, k] and scores_out [total_q, ld] are
 * optional (NULL = keep them in the workspace only); ld is ignored when
 * scores_out is NULL.  Steps 1-2 run over chunks of query rows whose scores
 * fit in 512 MiB of the workspace; step 3 then runs once over every row.
 * Results equal steps 1-3 called one by one, bit for bit. */
DSA_API dsa_status dsa_forward(const dsa_batch* batch, const uint16_t* q_idx, const float* w,
                       const uint16_t* k_idx, const uint16_t* q, const uint16_t* kv, int k,
                       float sm_scale, uint16_t* out, float* lse, int32_t* idx_out,
                       float* scores_out, int64_t ld, void* ws, size_t ws_bytes, void* stream);

/* ---- MLA around the path ("GLM-5.1 架构深度拆解", section 4.5 Steps 1-4
 * and 7-8; section 4.1).  kv_b_proj's weight w_kv_b [64 * 448, 512] holds,
 * per head h, W_UK[h] (rows h*448 .. h*448+191: k_nope = W_UK[h] c) and
 * W_UV[h] (rows h*448+192 .. h*448+447: v = W_UV[h] c) for the 512-dim
 * cached latent c.  Because q_nope . (W_UK c) = (W_UK^T q_nope) . c and
 * sum_s p_s W_UV c_s = W_UV sum_s p_s c_s, the attention runs on the cached
 * rows directly: absorb the query before it, apply W_UV and o_proj after. */

/* The absorbed query: q_out[t, h, 0:512] = W_UK[h]^T q_nope[t, h],
 * q_out[t, h, 512:576] = q_pe[t, h] (bf16, fp32 accumulation, rounded to
 * nearest even).  Layouts (row-major, DEVICE, bf16 bits, 16-byte aligned):
 *   q_nope  [total_q, 64, 192]   post-projection query, nope part
 *   q_pe    [total_q, 64, 64]    post-RoPE query, rope part
 *   w_kv_b  [64 * 448, 512]      kv_b_proj weight (nn.Linear layout)
 *   q_out   [total_q, 64, 576]   the q of dsa_sparse_mla_fwd / dsa_forward
 * ws: any workspace of at least 256 bytes (its status word receives
 * device-side timeouts).  total_q = 0 is a no-op.  Errors: null or
 * misaligned pointers, total_q < 0 or >= 2^26 -> DSA_ERR_INVALID_ARG;
 * launch failures -> DSA_ERR_CUDA. */
DSA_API dsa_status dsa_mla_absorb_q(int32_t total_q, const uint16_t* q_nope, const uint16_t* q_pe,
                                    const uint16_t* w_kv_b, uint16_t* q_out, void* ws, size_t ws_bytes,
                                    void* stream);

/* Bytes of workspace dsa_mla_output needs for total_q rows: the 256-byte
 * status header plus, when few rows leave the tensor cores idle, the fp32
 * partial sums of a split of the K dimension (summed in a fixed order, so
 * results do not depend on timing).  Errors: NULL bytes or total_q outside
 * [0, 2^26) -> DSA_ERR_INVALID_ARG. */
DSA_API dsa_status dsa_mla_workspace_size(int32_t total_q, size_t* bytes);

/* The layer output from the attention's latent output:
 *   o_mid[t, h*256 + e] = (W_UV[h] o_lat[t, h])[e]     (bf16)
 *   y[t, n] = sum_c w_o[n, c] o_mid[t, c]              (bf16)
 * fp32 accumulation, each result rounded to bf16 (o_mid is rounded before
 * o_proj reads it).  Layouts (row-major, DEVICE, bf16 bits, 16-byte aligned):
 *   o_lat   [total_q, 64, 512]   `out` of dsa_sparse_mla_fwd / dsa_forward
 *   w_kv_b  [64 * 448, 512]      kv_b_proj weight
 *   w_o     [6144, 64 * 256]     o_proj weight (nn.Linear layout)
 *   o_mid   [total_q, 64 * 256]  caller-owned intermediate
 *   y       [total_q, 6144]
 * ws: at least dsa_mla_workspace_size(total_q) bytes, else
 * DSA_ERR_WORKSPACE; other errors as dsa_mla_absorb_q. */
DSA_API dsa_status dsa_mla_output(int32_t total_q, const uint16_t* o_lat, const uint16_t* w_kv_b,
                                  const uint16_t* w_o, uint16_t* o_mid, uint16_t* y, void* ws, size_t ws_bytes,
                                  void* stream);

/* ---- The index-key producer ("GLM-5.1 架构深度拆解", section 3.6 Steps 2-4):
 * the step before the indexer, for the new tokens of a call.  For the new
 * token at packed row r (sequence b, position t = ctx_len[b] - n_b + i):
 *   k = LayerNorm(wk x[r])            over 128 dims: mean, biased variance,
 *                                     (v - mean) / sqrt(var + eps) * gamma + beta
 *   k[i] = k[i] cos[r,i] - k[i+32] sin[r,i],  k[i+32] = k[i+32] cos[r,i+32]
 *          + k[i] sin[r,i+32]  for i < 32 (rotate-half RoPE on dims 0..63)
 *   k_idx[b * cache_stride + t] = bf16(k)     (the cache append)
 *   w_out[r, h] = (w_proj x[r])[h] * 32^-1/2  (the w of dsa_indexer_scores)
 * fp32 accumulation and arithmetic; k rounded to bf16 (nearest even).  The
 * pages fix neither the rotary base nor the pairing: the caller passes the
 * rows of its rotary table (cos / sin of the token's position, fp32 [64]),
 * the pairing is the rotate-half one.
 * Layouts (row-major, DEVICE, 16-byte aligned):
 *   x       bf16 [total_q, 6144]   hidden states of the new tokens
 *   wk      bf16 [128, 6144]       indexer key projection (nn.Linear layout)
 *   gamma, beta fp32 [128]         k_norm affine parameters
 *   cos, sin fp32 [total_q, 64]    rotary rows of each token's position
 *   w_proj  bf16 [32, 6144]        indexer weights_proj
 *   k_idx   bf16 [batch * cache_stride, 128]   index-key cache (only the new
 *                                  tokens' rows are written)
 *   w_out   fp32 [total_q, 32]
 * ws: at least dsa_index_key_workspace_size(total_q) bytes (status header
 * plus fp32 partial sums), else DSA_ERR_WORKSPACE.  Errors: bad batch,
 * null or misaligned pointers, eps not positive and finite ->
 * DSA_ERR_INVALID_ARG; rows the device-side q_off / ctx_len leave
 * inconsistent are skipped and DSA_ERR_BAD_BATCH is latched. */
DSA_API dsa_status dsa_index_key_workspace_size(int32_t total_q, size_t* bytes);
DSA_API dsa_status dsa_index_key_producer(const dsa_batch* batch, const uint16_t* x, const uint16_t* wk,
                                          const float* gamma, const float* beta, float eps, const float* cos,
                                          const float* sin, const uint16_t* w_proj, uint16_t* k_idx, float* w_out,
                                          void* ws, size_t ws_bytes, void* stream);

/* ---- Reduced-precision index keys.  The pages give no FP8 recipe for the
 * indexer (only that weights_proj stays in fp32 / bf16); this library's
 * reading: E4M3 (the OCP 8-bit format: 4 exponent bits, bias 7, 3 mantissa
 * bits, largest finite 448) with one fp32 scale per 128-value row --
 * amax / 448 (1 for an all-zero row) -- per cached index key and per
 * (token, head) of the indexer queries.  Both scales are positive, so
 *   I[t,s] = ks[s] * sum_h (w[t,h] qs[t,h]) ReLU(q8[t,h] . k8[s])
 * with exact E4M3 products accumulated in fp32 on the tensor cores.  The
 * index-key cache then takes 132 bytes per token instead of 256. */

/* codes[r, :] = E4M3(in[r, :] / scale[r]), scale[r] = amax_r / 448 (fp32;
 * quotients in fp32, round to nearest even, saturating at +-448).
 *   in     bf16 [rows, 128] (DEVICE)    index keys or indexer queries
 *   codes  uint8 [rows, 128] (DEVICE)   scale fp32 [rows] (DEVICE)
 * 16-byte aligned pointers; rows < 0 -> DSA_ERR_INVALID_ARG. */
DSA_API dsa_status dsa_quantize_fp8(int64_t rows, const uint16_t* in, uint8_t* codes, float* scale, void* stream);

/* Step 1 on E4M3 queries and keys:
 *   q8 uint8 [total_q, 32, 128], qs fp32 [total_q, 32]   (dsa_quantize_fp8 of q_idx)
 *   k8 uint8 [batch * cache_stride, 128], ks fp32 [batch * cache_stride]
 *   w, scores, ld, ws: as dsa_indexer_scores. */
DSA_API dsa_status dsa_indexer_scores_fp8(const dsa_batch* batch, const uint8_t* q8, const float* qs,
                                          const float* w, const uint8_t* k8, const float* ks, float* scores,
                                          int64_t ld, void* ws, size_t ws_bytes, void* stream);

/* Steps 1-3 with E4M3 index keys (inputs of step 1 as
 * dsa_indexer_scores_fp8, the rest as dsa_forward). */
DSA_API dsa_status dsa_forward_fp8(const dsa_batch* batch, const uint8_t* q8, const float* qs, const float* w,
                                   const uint8_t* k8, const float* ks, const uint16_t* q, const uint16_t* kv, int k,
                                   float sm_scale, uint16_t* out, float* lse, int32_t* idx_out, float* scores_out,
                                   int64_t ld, void* ws, size_t ws_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DSA_H */
