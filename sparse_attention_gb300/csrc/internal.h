// internal.h -- definitions shared by the CUDA translation units of libdsa.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "../../include/dsa.h"

namespace dsa {

constexpr int kHIdx = DSA_INDEX_HEADS;   // 32 indexer heads
constexpr int kDIdx = DSA_INDEX_DIM;     // 128 dims per indexer head / key
constexpr int kH = DSA_HEADS;            // 64 attention heads
constexpr int kDQK = DSA_QK_DIM;         // 576 = 512 latent + 64 rope
constexpr int kDV = DSA_V_DIM;           // 512
constexpr int kMaxTopk = DSA_MAX_TOPK;   // 2048
constexpr int kDefaultSMs = 152;         // GB300: used when no device can be queried

// Upper bound on any single in-kernel wait (a phase of an mbarrier).  A wait
// that exceeds it latches DSA_ERR_TIMEOUT and the kernel winds down.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// The first 256 bytes of every workspace: the device status word.
constexpr size_t kWsHeaderBytes = 256;

// Device view of dsa_batch.
struct BatchDev {
    int32_t B, total_q, max_q, max_ctx;
    int64_t stride;
    const int32_t* q_off;
    const int32_t* ctx_len;
};

// The local query indices [i0, i1) of every sequence that one launch
// processes.  A per-row buffer is either addressed by the packed row
// q_off[b] + i ("global") or, for chunk-sized scratch, by
// b * (i1 - i0) + (i - i0) ("local").
struct RowRange {
    int32_t i0, i1;
};

struct SeqInfo {
    int32_t q0, nq, ctx;
};

__device__ __forceinline__ void latch_status(int32_t* status, int code) {
    if (status) atomicCAS(status, 0, code);
}

// Loads and checks sequence b; false (and a latched DSA_ERR_BAD_BATCH) if
// its q_off / ctx_len break the host bounds.
__device__ __forceinline__ bool load_seq(const BatchDev& bd, int b, int32_t* status, SeqInfo& s) {
    s.q0 = __ldg(bd.q_off + b);
    const int32_t q1 = __ldg(bd.q_off + b + 1);
    s.nq = q1 - s.q0;
    s.ctx = __ldg(bd.ctx_len + b);
    const bool ok = s.q0 >= 0 && q1 <= bd.total_q && s.nq >= 0 && s.nq <= bd.max_q && s.nq <= s.ctx &&
                    s.ctx <= bd.max_ctx;
    if (!ok) latch_status(status, DSA_ERR_BAD_BATCH);
    return ok;
}

__device__ __forceinline__ int64_t buf_row(bool local, const SeqInfo& s, int b, int32_t i, RowRange rr) {
    return local ? (int64_t)b * (rr.i1 - rr.i0) + (i - rr.i0) : (int64_t)s.q0 + i;
}

// Tensor map of a row-major 2-D bf16 tensor [rows, inner] (row stride inner*2
// bytes), 128-byte swizzle, box {box_inner, box_rows}.  False if the driver
// entry point is unavailable or rejects the arguments.
bool make_tmap_bf16_2d(CUtensorMap* tm, const void* base, uint64_t inner, uint64_t rows, uint32_t box_inner,
                       uint32_t box_rows);

// The same for a 2-D tensor of bytes (row stride inner bytes).
bool make_tmap_u8_2d(CUtensorMap* tm, const void* base, uint64_t inner, uint64_t rows, uint32_t box_inner,
                     uint32_t box_rows);

// Streaming multiprocessors of the current device (cudaDevAttrMultiProcessorCount,
// read once per device); kDefaultSMs when no device can be queried.
int num_sms();

// Adds n to the process-wide count of kernels launched by this library.
void count_launches(int n);

// DSA_OK for cudaSuccess; otherwise records e as this thread's last CUDA
// error (dsa_last_cuda_error), clears a non-sticky launch error and returns
// DSA_ERR_CUDA.
dsa_status cuda_status(cudaError_t e);

// ------------------------------------------------------------ launchers --

cudaError_t launch_indexer(const BatchDev& bd, RowRange rr, const uint16_t* q_idx, const float* w,
                           const uint16_t* k_idx, float* scores, int64_t ld, bool scores_local,
                           int32_t* status, cudaStream_t stream);

// FP8 (E4M3) index keys: scores from quantized queries / keys (qs per
// (token, head), ks per cached key), and the row quantizer.
cudaError_t launch_indexer_fp8(const BatchDev& bd, RowRange rr, const uint8_t* q8, const float* qs, const float* w,
                               const uint8_t* k8, const float* ks, float* scores, int64_t ld, bool scores_local,
                               int32_t* status, cudaStream_t stream);
cudaError_t launch_quantize_fp8(int64_t rows, const uint16_t* in, uint8_t* codes, float* scale, cudaStream_t stream);

// after_previous: launched as a programmatic dependent of the previous
// kernel in the stream (its CTAs may become resident while that kernel
// finishes, and wait for it before reading anything).
cudaError_t launch_topk(const BatchDev& bd, RowRange rr, const float* scores, int64_t ld,
                        bool scores_local, int k, int32_t* idx, bool idx_local, int32_t* status,
                        cudaStream_t stream, bool after_previous = false);

// Bytes of scratch the attention launch needs for `rows` query rows.
size_t sparse_mla_scratch_bytes(const BatchDev& bd, int64_t rows, int k);

cudaError_t launch_sparse_mla(const BatchDev& bd, RowRange rr, const uint16_t* q, const uint16_t* kv,
                              const int32_t* idx, bool idx_local, int k, float sm_scale,
                              uint16_t* out, float* lse, void* scratch, size_t scratch_bytes,
                              int32_t* status, cudaStream_t stream, bool after_previous = false);

cudaError_t launch_mla_absorb_q(int32_t total_q, const uint16_t* q_nope, const uint16_t* q_pe,
                                const uint16_t* w_kvb, uint16_t* q_out, int32_t* status, cudaStream_t stream);
cudaError_t launch_mla_output(int32_t total_q, const uint16_t* o_lat, const uint16_t* w_kvb, const uint16_t* w_o,
                              uint16_t* o_mid, uint16_t* y, float* part, int32_t* status, cudaStream_t stream);
// Bytes of split-K partials dsa_mla_output needs for total_q rows (0: none).
size_t mla_partial_bytes(int32_t total_q);

// C = A . B^T for a K-major A [M, K] and K-major B [N, K] (tensor maps with
// boxes {64, 128} and {64, 256}), fp32 results part[s][m][n] of `splits`
// equal K splits (their sum is the product); K a multiple of 64.
cudaError_t launch_gemm_f32_parts(const CUtensorMap& tm_a, const CUtensorMap& tm_b, int32_t M, int32_t N, int32_t K,
                                  int32_t splits, float* part, int32_t* status, cudaStream_t stream);
// The K splits launch_gemm_f32_parts should use for an M x N x K product.
int gemm_k_splits(int32_t M, int32_t N, int32_t K);

// The index-key producer: workspace bytes past the status header, launch.
size_t index_key_partial_bytes(int32_t total_q);
cudaError_t launch_index_key(const BatchDev& bd, const uint16_t* x, const uint16_t* wk, const float* gamma,
                             const float* beta, float eps, const float* cos_t, const float* sin_t,
                             const uint16_t* w_proj, uint16_t* k_idx, float* w_out, float* part, int32_t* status,
                             cudaStream_t stream);

}  // namespace dsa
