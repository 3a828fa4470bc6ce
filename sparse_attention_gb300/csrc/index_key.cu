// index_key.cu -- the index-key producer: the step before the lightning
// indexer, for the new tokens of a call.
//
// ("GLM-5.1 架构深度拆解", section 3.6 Steps 2-4.)  For a new token with
// hidden state x (6144):
//   k = k_norm(wk x)                  LayerNorm over 128 dims (mean, biased
//                                     variance, eps, gamma, beta)
//   k[0:64] = RoPE(k[0:64])           rotate-half form, pairs (i, i + 32),
//                                     with the token's cos / sin rows
//   k[64:128] unchanged               (the pages split rope-first)
//   w = (weights_proj x) * 32^-1/2    the 32 indexer head weights
// k is written, as bf16, into the index-key cache at the token's position
// (row b * cache_stride + t); w is written as fp32 [total_q, 32], the w of
// dsa_indexer_scores / dsa_forward.
//
// Two tensor-core GEMMs (wk and weights_proj against the hidden states,
// split over K when few tokens leave SMs idle) write fp32 partial sums; one
// warp per token then sums the splits in order, normalises, rotates and
// stores (lane l holds dims l, l + 32, l + 64, l + 96, so both members of
// every RoPE pair sit in one lane).
#include <cuda_bf16.h>

#include <algorithm>
#include <cmath>

#include "internal.h"
#include "ptx.cuh"

namespace dsa {
namespace {

constexpr int kHidden = 6144;
constexpr int kRope = 64;

struct SplitPlan {
    int sk, sw;         // K splits of the wk and weights_proj products
    size_t off_w;       // float offset of the weights_proj partials
    size_t floats;      // partial floats in all
};

SplitPlan plan(int32_t total_q) {
    SplitPlan p{};
    p.sk = gemm_k_splits(total_q, kDIdx, kHidden);
    p.sw = gemm_k_splits(total_q, kHIdx, kHidden);
    p.off_w = (size_t)p.sk * total_q * kDIdx;
    p.floats = p.off_w + (size_t)p.sw * total_q * kHIdx;
    return p;
}

__global__ void __launch_bounds__(256)
    index_key_finish_kernel(const BatchDev bd, const float* __restrict__ part_k, int sk,
                            const float* __restrict__ part_w, int sw, const float* __restrict__ gamma,
                            const float* __restrict__ beta, float eps, const float* __restrict__ cos_t,
                            const float* __restrict__ sin_t, uint16_t* __restrict__ k_idx, float* __restrict__ w_out,
                            int32_t* status) {
    const int lane = threadIdx.x & 31;
    const int64_t r = (int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);   // packed token row
    if (r >= bd.total_q) return;
    // the sequence of row r: the last b with q_off[b] <= r
    int lo = 0, hi = bd.B - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(bd.q_off + mid) <= r) lo = mid;
        else hi = mid - 1;
    }
    SeqInfo sq;
    if (!load_seq(bd, lo, status, sq)) return;
    const int32_t i = (int32_t)(r - sq.q0);
    if (i < 0 || i >= sq.nq) {
        latch_status(status, DSA_ERR_BAD_BATCH);   // rows not covered by q_off
        return;
    }
    const int64_t t = (int64_t)sq.ctx - sq.nq + i;

    // k: the four dims of this lane, splits summed in order (loads of four
    // splits in flight at a time)
    float v[4] = {0.f, 0.f, 0.f, 0.f};
    int s = 0;
    for (; s + 4 <= sk; s += 4) {
        float t4[4][4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
            for (int j = 0; j < 4; ++j) t4[u][j] = part_k[((int64_t)(s + u) * bd.total_q + r) * kDIdx + lane + 32 * j];
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
            for (int j = 0; j < 4; ++j) v[j] += t4[u][j];
    }
    for (; s < sk; ++s)
#pragma unroll
        for (int j = 0; j < 4; ++j) v[j] += part_k[((int64_t)s * bd.total_q + r) * kDIdx + lane + 32 * j];
    float sum = (v[0] + v[1]) + (v[2] + v[3]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    const float mean = sum * (1.f / kDIdx);
    float sq_dev = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) sq_dev += (v[j] - mean) * (v[j] - mean);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sq_dev += __shfl_xor_sync(0xffffffffu, sq_dev, o);
    const float rstd = rsqrtf(sq_dev * (1.f / kDIdx) + eps);
    float z[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int d = lane + 32 * j;
        z[j] = (v[j] - mean) * rstd * __ldg(gamma + d) + __ldg(beta + d);
    }
    // RoPE on dims [0, 64): (z0, z1) = dims (lane, lane + 32) rotate together
    const float* cr = cos_t + r * kRope;
    const float* sr = sin_t + r * kRope;
    const float k0 = z[0] * __ldg(cr + lane) - z[1] * __ldg(sr + lane);
    const float k1 = z[1] * __ldg(cr + lane + 32) + z[0] * __ldg(sr + lane + 32);
    uint16_t* krow = k_idx + ((int64_t)lo * bd.stride + t) * kDIdx;
    const float outv[4] = {k0, k1, z[2], z[3]};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const __nv_bfloat16 bv = __float2bfloat16_rn(outv[j]);
        krow[lane + 32 * j] = *reinterpret_cast<const uint16_t*>(&bv);
    }
    // w: one head per lane (eight splits' loads in flight at a time)
    float acc = 0.f;
    int s2 = 0;
    for (; s2 + 8 <= sw; s2 += 8) {
        float t8[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) t8[u] = part_w[((int64_t)(s2 + u) * bd.total_q + r) * kHIdx + lane];
#pragma unroll
        for (int u = 0; u < 8; ++u) acc += t8[u];
    }
    for (; s2 < sw; ++s2) acc += part_w[((int64_t)s2 * bd.total_q + r) * kHIdx + lane];
    w_out[r * kHIdx + lane] = acc * rsqrtf((float)kHIdx);
}

}  // namespace

size_t index_key_partial_bytes(int32_t total_q) { return plan(total_q).floats * sizeof(float); }

cudaError_t launch_index_key(const BatchDev& bd, const uint16_t* x, const uint16_t* wk, const float* gamma,
                             const float* beta, float eps, const float* cos_t, const float* sin_t,
                             const uint16_t* w_proj, uint16_t* k_idx, float* w_out, float* part, int32_t* status,
                             cudaStream_t stream) {
    const int32_t T = bd.total_q;
    if (T <= 0) return cudaSuccess;
    const SplitPlan p = plan(T);
    CUtensorMap tm_x, tm_k, tm_w;
    if (!make_tmap_bf16_2d(&tm_x, x, kHidden, (uint64_t)T, 64, 128) ||
        !make_tmap_bf16_2d(&tm_k, wk, kHidden, kDIdx, 64, 256) ||
        !make_tmap_bf16_2d(&tm_w, w_proj, kHidden, kHIdx, 64, 256))
        return cudaErrorInvalidValue;
    cudaError_t e = launch_gemm_f32_parts(tm_x, tm_k, T, kDIdx, kHidden, p.sk, part, status, stream);
    if (e != cudaSuccess) return e;
    e = launch_gemm_f32_parts(tm_x, tm_w, T, kHIdx, kHidden, p.sw, part + p.off_w, status, stream);
    if (e != cudaSuccess) return e;
    const int warps = 8;
    index_key_finish_kernel<<<(unsigned)((T + warps - 1) / warps), 32 * warps, 0, stream>>>(
        bd, part, p.sk, part + p.off_w, p.sw, gamma, beta, eps, cos_t, sin_t, k_idx, w_out, status);
    e = cudaGetLastError();
    if (e == cudaSuccess) count_launches(1);
    return e;
}

}  // namespace dsa
