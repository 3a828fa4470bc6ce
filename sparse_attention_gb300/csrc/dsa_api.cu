// dsa_api.cu -- the extern "C" entry points of libdsa.so (declared and
// documented in include/dsa.h): host-side argument checks, workspace
// layout, and the launch sequence of dsa_forward.
#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstdio>

#include "internal.h"

namespace dsa {

static std::atomic<uint64_t> g_launches{0};
void count_launches(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

namespace {

// Scores of one dsa_forward chunk (the workspace holds one chunk).  Fewer,
// larger chunks cost fewer wave tails of the indexer and top-k launches than
// keeping each chunk in L2 saves (measured: 16,384-token prefill 9.13 ms with
// 64 MiB chunks, 8.83 ms with 512 MiB; 65,536 tokens in 8,192-token calls
// 60.6 ms and 53.0 ms).
constexpr size_t kScoreChunkBytes = size_t(512) << 20;

// Inside dsa_forward the top-k and attention launches of decode-sized
// batches (fewer query rows than SMs) are programmatic dependents of the
// launch before them: their CTAs become resident while that kernel drains,
// and wait for it before reading its results (64 x 32,768 decode step
// 154.6 -> 151.2 us; 8 x 202,752, whose rows the top-k and the attention
// split over clusters, 104.8 -> 99.7 us).  Many-row prefills ran slightly
// slower chained (7.72 -> 7.74 ms), so they launch plainly.
bool chain_launches(const dsa_batch* b) {
    return (int64_t)b->batch * b->max_q < num_sms();
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

dsa_status check_batch(const dsa_batch* b) {
    if (!b) return DSA_ERR_INVALID_ARG;
    if (b->batch < 1 || b->batch > 65535) return DSA_ERR_INVALID_ARG;
    if (b->total_q < 0 || b->max_q < 0 || b->max_ctx < 0) return DSA_ERR_INVALID_ARG;
    if (b->max_q > (1 << 19)) return DSA_ERR_UNSUPPORTED;            // grid limits
    if (b->total_q >= (1 << 26)) return DSA_ERR_UNSUPPORTED;         // TMA row coordinates
    if (b->cache_stride < b->max_ctx || b->cache_stride < 0) return DSA_ERR_INVALID_ARG;
    if ((int64_t)b->batch * b->cache_stride >= (int64_t(1) << 31)) return DSA_ERR_UNSUPPORTED;
    if (!b->q_off || !b->ctx_len) return DSA_ERR_INVALID_ARG;
    return DSA_OK;
}

BatchDev to_dev(const dsa_batch* b) {
    return BatchDev{b->batch, b->total_q, b->max_q, b->max_ctx, b->cache_stride, b->q_off, b->ctx_len};
}

struct WsLayout {
    int32_t chunk_rows;     // local query rows per dsa_forward chunk
    int64_t ld_s;           // row stride of the scratch score rows
    size_t off_scores, off_idx, off_attn, attn_bytes, total;
};

WsLayout ws_layout(const dsa_batch* b, int k) {
    WsLayout L{};
    const BatchDev bd = to_dev(b);
    L.ld_s = std::max<int64_t>(4, ((int64_t)b->max_ctx + 3) / 4 * 4);
    const size_t row_bytes = (size_t)b->batch * L.ld_s * sizeof(float);
    int64_t rows = (int64_t)(kScoreChunkBytes / std::max<size_t>(row_bytes, 1));
    rows = std::max<int64_t>(1, std::min<int64_t>(rows, std::max(b->max_q, 1)));
    L.chunk_rows = (int32_t)rows;
    size_t off = kWsHeaderBytes;
    L.off_scores = off;
    off = round_up(off + (size_t)b->batch * rows * L.ld_s * sizeof(float), 256);
    // indices of every query row: the attention runs once after all chunks
    L.off_idx = off;
    off = round_up(off + (size_t)b->batch * std::max(b->max_q, 1) * k * sizeof(int32_t), 256);
    L.off_attn = off;
    // attention scratch for a whole-batch launch
    L.attn_bytes = sparse_mla_scratch_bytes(bd, b->max_q, k);
    off = round_up(off + L.attn_bytes, 256);
    L.total = off;
    return L;
}

dsa_status check_ws(const dsa_batch* b, int k, void* ws, size_t ws_bytes) {
    if (!ws || !aligned16(ws)) return DSA_ERR_WORKSPACE;
    if (ws_bytes < ws_layout(b, k).total) return DSA_ERR_WORKSPACE;
    return DSA_OK;
}

}  // namespace

thread_local cudaError_t t_last_error = cudaSuccess;

int num_sms() {
    constexpr int kMaxDevices = 64;
    static std::atomic<int> cache[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return kDefaultSMs;
    }
    const int v = cache[dev].load(std::memory_order_relaxed);
    if (v > 0) return v;
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
        cudaGetLastError();
        return kDefaultSMs;
    }
    cache[dev].store(n, std::memory_order_relaxed);
    return n;
}

dsa_status cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return DSA_OK;
    t_last_error = e;
    cudaGetLastError();  // clear a non-sticky launch error of this thread
    return DSA_ERR_CUDA;
}

}  // namespace dsa

using namespace dsa;

namespace {

// Steps 1-3: `score(rr, scores, ld, local)` runs the indexer over the local
// query rows rr (bf16 or E4M3 keys); the rest is shared.
template <typename ScoreFn>
dsa_status forward_impl(const dsa_batch* batch, ScoreFn score, const uint16_t* q, const uint16_t* kv, int k,
                        float sm_scale, uint16_t* out, float* lse, int32_t* idx_out, float* scores_out, int64_t ld,
                        void* ws, cudaStream_t s) {
    const BatchDev bd = to_dev(batch);
    const WsLayout L = ws_layout(batch, k);
    uint8_t* base = static_cast<uint8_t*>(ws);
    int32_t* status = static_cast<int32_t*>(ws);
    float* sc = scores_out ? scores_out : reinterpret_cast<float*>(base + L.off_scores);
    const int64_t sc_ld = scores_out ? ld : L.ld_s;
    // indices by packed row (idx_out, or the workspace buffer of every row)
    int32_t* ix = idx_out ? idx_out : reinterpret_cast<int32_t*>(base + L.off_idx);
    const bool chain = chain_launches(batch);
    // scores and top-k chunk by chunk, then one attention launch over every
    // row (no per-chunk wave tails)
    for (int32_t i0 = 0; i0 < batch->max_q; i0 += L.chunk_rows) {
        const RowRange rr{i0, std::min(i0 + L.chunk_rows, batch->max_q)};
        cudaError_t e = score(rr, sc, sc_ld, scores_out == nullptr);
        if (e == cudaSuccess)
            e = launch_topk(bd, rr, sc, sc_ld, scores_out == nullptr, k, ix, false, status, s, chain);
        if (e != cudaSuccess) return cuda_status(e);
    }
    return cuda_status(launch_sparse_mla(bd, RowRange{0, batch->max_q}, q, kv, ix, false, k, sm_scale, out, lse,
                                         base + L.off_attn, L.attn_bytes, status, s, chain));
}

// Host checks shared by the forward calls (everything but the indexer inputs).
dsa_status check_forward(const dsa_batch* batch, const uint16_t* q, const uint16_t* kv, int k, float sm_scale,
                         const uint16_t* out, const float* lse, const int32_t* idx_out, const float* scores_out,
                         int64_t ld, void* ws, size_t ws_bytes) {
    dsa_status st = check_batch(batch);
    if (st != DSA_OK) return st;
    if (k < 1 || k > kMaxTopk) return DSA_ERR_INVALID_ARG;
    if ((st = check_ws(batch, k, ws, ws_bytes)) != DSA_OK) return st;
    if (batch->total_q == 0 || batch->max_q == 0) return DSA_OK;
    if (!q || !kv || !out) return DSA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(kv) || !aligned16(out) || (lse && !aligned16(lse)) ||
        (idx_out && !aligned16(idx_out)) || (scores_out && !aligned16(scores_out)))
        return DSA_ERR_INVALID_ARG;
    if (scores_out && (ld < batch->max_ctx || ld % 4 != 0)) return DSA_ERR_INVALID_ARG;
    if (!(sm_scale > 0.f) || sm_scale == INFINITY) return DSA_ERR_INVALID_ARG;
    return DSA_OK;
}

}  // namespace

extern "C" {

const char* dsa_status_string(int s) {
    switch (s) {
        case DSA_OK: return "DSA_OK";
        case DSA_ERR_INVALID_ARG: return "DSA_ERR_INVALID_ARG: an argument failed the host-side check";
        case DSA_ERR_UNSUPPORTED: return "DSA_ERR_UNSUPPORTED: shape or mode not implemented";
        case DSA_ERR_WORKSPACE: return "DSA_ERR_WORKSPACE: workspace missing, misaligned or too small";
        case DSA_ERR_CUDA: return "DSA_ERR_CUDA: a CUDA launch or runtime call failed";
        case DSA_ERR_TIMEOUT: return "DSA_ERR_TIMEOUT: a bounded in-kernel wait expired";
        case DSA_ERR_BAD_BATCH: return "DSA_ERR_BAD_BATCH: q_off/ctx_len outside the host bounds";
        case DSA_ERR_BAD_INDEX: return "DSA_ERR_BAD_INDEX: a selected index outside [-1, t]";
        case DSA_ERR_INTERNAL: return "DSA_ERR_INTERNAL: an internal consistency check failed in a kernel";
        default: return "unknown dsa_status";
    }
}

const char* dsa_last_cuda_error(void) { return cudaGetErrorString(t_last_error); }

uint64_t dsa_kernel_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

dsa_status dsa_workspace_size(const dsa_batch* batch, int k, size_t* bytes) {
    if (!bytes) return DSA_ERR_INVALID_ARG;
    dsa_status st = check_batch(batch);
    if (st != DSA_OK) return st;
    if (k < 1 || k > kMaxTopk) return DSA_ERR_INVALID_ARG;
    *bytes = ws_layout(batch, k).total;
    return DSA_OK;
}

dsa_status dsa_reset_device_status(void* ws, void* stream) {
    if (!ws || !aligned16(ws)) return DSA_ERR_WORKSPACE;
    return cuda_status(cudaMemsetAsync(ws, 0, kWsHeaderBytes, static_cast<cudaStream_t>(stream)));
}

dsa_status dsa_read_device_status(const void* ws, void* stream, dsa_status* out) {
    if (!ws || !out) return DSA_ERR_INVALID_ARG;
    int32_t v = 0;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(&v, ws, sizeof v, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_status(e);
    *out = static_cast<dsa_status>(v);
    return DSA_OK;
}

dsa_status dsa_indexer_scores(const dsa_batch* batch, const uint16_t* q_idx, const float* w, const uint16_t* k_idx,
                              float* scores, int64_t ld, void* ws, size_t ws_bytes, void* stream) {
    dsa_status st = check_batch(batch);
    if (st != DSA_OK) return st;
    if (!ws || !aligned16(ws) || ws_bytes < kWsHeaderBytes) return DSA_ERR_WORKSPACE;
    if (batch->total_q == 0 || batch->max_q == 0) return DSA_OK;
    if (!q_idx || !w || !k_idx || !scores) return DSA_ERR_INVALID_ARG;
    if (!aligned16(q_idx) || !aligned16(w) || !aligned16(k_idx) || !aligned16(scores)) return DSA_ERR_INVALID_ARG;
    if (ld < batch->max_ctx || ld % 4 != 0) return DSA_ERR_INVALID_ARG;
    const BatchDev bd = to_dev(batch);
    return cuda_status(launch_indexer(bd, RowRange{0, batch->max_q}, q_idx, w, k_idx, scores, ld, false,
                                      static_cast<int32_t*>(ws), static_cast<cudaStream_t>(stream)));
}

dsa_status dsa_topk(const dsa_batch* batch, const float* scores, int64_t ld, int k, int32_t* idx, void* ws,
                    size_t ws_bytes, void* stream) {
    dsa_status st = check_batch(batch);
    if (st != DSA_OK) return st;
    if (k < 1 || k > kMaxTopk) return DSA_ERR_INVALID_ARG;
    if (!ws || !aligned16(ws) || ws_bytes < kWsHeaderBytes) return DSA_ERR_WORKSPACE;
    if (batch->total_q == 0 || batch->max_q == 0) return DSA_OK;
    if (!scores || !idx || !aligned16(scores) || !aligned16(idx)) return DSA_ERR_INVALID_ARG;
    if (ld < batch->max_ctx || ld % 4 != 0) return DSA_ERR_INVALID_ARG;
    const BatchDev bd = to_dev(batch);
    return cuda_status(launch_topk(bd, RowRange{0, batch->max_q}, scores, ld, false, k, idx, false,
                                   static_cast<int32_t*>(ws), static_cast<cudaStream_t>(stream)));
}

dsa_status dsa_sparse_mla_fwd(const dsa_batch* batch, const uint16_t* q, const uint16_t* kv, const int32_t* idx,
                              int k, float sm_scale, uint16_t* out, float* lse, void* ws, size_t ws_bytes,
                              void* stream) {
    dsa_status st = check_batch(batch);
    if (st != DSA_OK) return st;
    if (k < 1 || k > kMaxTopk) return DSA_ERR_INVALID_ARG;
    if ((st = check_ws(batch, k, ws, ws_bytes)) != DSA_OK) return st;
    if (batch->total_q == 0 || batch->max_q == 0) return DSA_OK;
    if (!q || !kv || !idx || !out) return DSA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(kv) || !aligned16(idx) || !aligned16(out) || (lse && !aligned16(lse)))
        return DSA_ERR_INVALID_ARG;
    if (!(sm_scale > 0.f) || sm_scale == INFINITY) return DSA_ERR_INVALID_ARG;
    const BatchDev bd = to_dev(batch);
    const WsLayout L = ws_layout(batch, k);
    uint8_t* base = static_cast<uint8_t*>(ws);
    return cuda_status(launch_sparse_mla(bd, RowRange{0, batch->max_q}, q, kv, idx, false, k, sm_scale, out, lse,
                                         base + L.off_attn, L.attn_bytes, static_cast<int32_t*>(ws),
                                         static_cast<cudaStream_t>(stream)));
}

dsa_status dsa_forward(const dsa_batch* batch, const uint16_t* q_idx, const float* w, const uint16_t* k_idx,
                       const uint16_t* q, const uint16_t* kv, int k, float sm_scale, uint16_t* out, float* lse,
                       int32_t* idx_out, float* scores_out, int64_t ld, void* ws, size_t ws_bytes, void* stream) {
    dsa_status st = check_forward(batch, q, kv, k, sm_scale, out, lse, idx_out, scores_out, ld, ws, ws_bytes);
    if (st != DSA_OK || batch->total_q == 0 || batch->max_q == 0) return st;
    if (!q_idx || !w || !k_idx || !aligned16(q_idx) || !aligned16(w) || !aligned16(k_idx)) return DSA_ERR_INVALID_ARG;
    const BatchDev bd = to_dev(batch);
    int32_t* status = static_cast<int32_t*>(ws);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return forward_impl(
        batch,
        [&](RowRange rr, float* sc, int64_t sld, bool local) {
            return launch_indexer(bd, rr, q_idx, w, k_idx, sc, sld, local, status, s);
        },
        q, kv, k, sm_scale, out, lse, idx_out, scores_out, ld, ws, s);
}

dsa_status dsa_forward_fp8(const dsa_batch* batch, const uint8_t* q8, const float* qs, const float* w,
                           const uint8_t* k8, const float* ks, const uint16_t* q, const uint16_t* kv, int k,
                           float sm_scale, uint16_t* out, float* lse, int32_t* idx_out, float* scores_out, int64_t ld,
                           void* ws, size_t ws_bytes, void* stream) {
    dsa_status st = check_forward(batch, q, kv, k, sm_scale, out, lse, idx_out, scores_out, ld, ws, ws_bytes);
    if (st != DSA_OK || batch->total_q == 0 || batch->max_q == 0) return st;
    if (!q8 || !qs || !w || !k8 || !ks || !aligned16(q8) || !aligned16(qs) || !aligned16(w) || !aligned16(k8) ||
        !aligned16(ks))
        return DSA_ERR_INVALID_ARG;
    const BatchDev bd = to_dev(batch);
    int32_t* status = static_cast<int32_t*>(ws);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return forward_impl(
        batch,
        [&](RowRange rr, float* sc, int64_t sld, bool local) {
            return launch_indexer_fp8(bd, rr, q8, qs, w, k8, ks, sc, sld, local, status, s);
        },
        q, kv, k, sm_scale, out, lse, idx_out, scores_out, ld, ws, s);
}

dsa_status dsa_indexer_scores_fp8(const dsa_batch* batch, const uint8_t* q8, const float* qs, const float* w,
                                  const uint8_t* k8, const float* ks, float* scores, int64_t ld, void* ws,
                                  size_t ws_bytes, void* stream) {
    dsa_status st = check_batch(batch);
    if (st != DSA_OK) return st;
    if (!ws || !aligned16(ws) || ws_bytes < kWsHeaderBytes) return DSA_ERR_WORKSPACE;
    if (batch->total_q == 0 || batch->max_q == 0) return DSA_OK;
    if (!q8 || !qs || !w || !k8 || !ks || !scores) return DSA_ERR_INVALID_ARG;
    if (!aligned16(q8) || !aligned16(qs) || !aligned16(w) || !aligned16(k8) || !aligned16(ks) || !aligned16(scores))
        return DSA_ERR_INVALID_ARG;
    if (ld < batch->max_ctx || ld % 4 != 0) return DSA_ERR_INVALID_ARG;
    return cuda_status(launch_indexer_fp8(to_dev(batch), RowRange{0, batch->max_q}, q8, qs, w, k8, ks, scores, ld,
                                          false, static_cast<int32_t*>(ws), static_cast<cudaStream_t>(stream)));
}

dsa_status dsa_quantize_fp8(int64_t rows, const uint16_t* in, uint8_t* codes, float* scale, void* stream) {
    if (rows < 0) return DSA_ERR_INVALID_ARG;
    if (rows == 0) return DSA_OK;
    if (!in || !codes || !scale || !aligned16(in) || !aligned16(codes) || !aligned16(scale))
        return DSA_ERR_INVALID_ARG;
    return cuda_status(launch_quantize_fp8(rows, in, codes, scale, static_cast<cudaStream_t>(stream)));
}

dsa_status dsa_mla_absorb_q(int32_t total_q, const uint16_t* q_nope, const uint16_t* q_pe, const uint16_t* w_kv_b,
                            uint16_t* q_out, void* ws, size_t ws_bytes, void* stream) {
    if (total_q < 0 || total_q >= (1 << 26)) return DSA_ERR_INVALID_ARG;
    if (!ws || !aligned16(ws) || ws_bytes < kWsHeaderBytes) return DSA_ERR_WORKSPACE;
    if (total_q == 0) return DSA_OK;
    if (!q_nope || !q_pe || !w_kv_b || !q_out) return DSA_ERR_INVALID_ARG;
    if (!aligned16(q_nope) || !aligned16(q_pe) || !aligned16(w_kv_b) || !aligned16(q_out)) return DSA_ERR_INVALID_ARG;
    return cuda_status(launch_mla_absorb_q(total_q, q_nope, q_pe, w_kv_b, q_out, static_cast<int32_t*>(ws),
                                           static_cast<cudaStream_t>(stream)));
}

dsa_status dsa_mla_workspace_size(int32_t total_q, size_t* bytes) {
    if (!bytes || total_q < 0 || total_q >= (1 << 26)) return DSA_ERR_INVALID_ARG;
    *bytes = round_up(kWsHeaderBytes + mla_partial_bytes(total_q), 256);
    return DSA_OK;
}

dsa_status dsa_mla_output(int32_t total_q, const uint16_t* o_lat, const uint16_t* w_kv_b, const uint16_t* w_o,
                          uint16_t* o_mid, uint16_t* y, void* ws, size_t ws_bytes, void* stream) {
    if (total_q < 0 || total_q >= (1 << 26)) return DSA_ERR_INVALID_ARG;
    if (!ws || !aligned16(ws) || ws_bytes < kWsHeaderBytes + mla_partial_bytes(total_q)) return DSA_ERR_WORKSPACE;
    if (total_q == 0) return DSA_OK;
    if (!o_lat || !w_kv_b || !w_o || !o_mid || !y) return DSA_ERR_INVALID_ARG;
    if (!aligned16(o_lat) || !aligned16(w_kv_b) || !aligned16(w_o) || !aligned16(o_mid) || !aligned16(y))
        return DSA_ERR_INVALID_ARG;
    float* part = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + kWsHeaderBytes);
    return cuda_status(launch_mla_output(total_q, o_lat, w_kv_b, w_o, o_mid, y, part, static_cast<int32_t*>(ws),
                                         static_cast<cudaStream_t>(stream)));
}

dsa_status dsa_index_key_workspace_size(int32_t total_q, size_t* bytes) {
    if (!bytes || total_q < 0 || total_q >= (1 << 26)) return DSA_ERR_INVALID_ARG;
    *bytes = round_up(kWsHeaderBytes + index_key_partial_bytes(total_q), 256);
    return DSA_OK;
}

dsa_status dsa_index_key_producer(const dsa_batch* batch, const uint16_t* x, const uint16_t* wk, const float* gamma,
                                  const float* beta, float eps, const float* cos_t, const float* sin_t,
                                  const uint16_t* w_proj, uint16_t* k_idx, float* w_out, void* ws, size_t ws_bytes,
                                  void* stream) {
    dsa_status st = check_batch(batch);
    if (st != DSA_OK) return st;
    if (!ws || !aligned16(ws) || ws_bytes < kWsHeaderBytes + index_key_partial_bytes(batch->total_q))
        return DSA_ERR_WORKSPACE;
    if (batch->total_q == 0) return DSA_OK;
    if (!x || !wk || !gamma || !beta || !cos_t || !sin_t || !w_proj || !k_idx || !w_out) return DSA_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(wk) || !aligned16(gamma) || !aligned16(beta) || !aligned16(cos_t) ||
        !aligned16(sin_t) || !aligned16(w_proj) || !aligned16(k_idx) || !aligned16(w_out))
        return DSA_ERR_INVALID_ARG;
    if (!(eps > 0.f) || eps == INFINITY) return DSA_ERR_INVALID_ARG;
    float* part = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + kWsHeaderBytes);
    return cuda_status(launch_index_key(to_dev(batch), x, wk, gamma, beta, eps, cos_t, sin_t, w_proj, k_idx, w_out,
                                        part, static_cast<int32_t*>(ws), static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
