// sparse_mla.cu -- sparse MLA attention over the selected latent rows,
// absorbed form.
//
// For query row t and head h, over the selected positions s_j = idx[t, j]:
//   l_j   = sm_scale * q[t,h,:] . kv[s_j, :]          (576 = 512 latent + 64 rope)
//   out   = sum_j softmax_j(l) * kv[s_j, 0:512]
//   lse   = log sum_j exp(l_j)
// ("GLM-5.1 架构深度拆解", section 3.1 step 2 and section 4.2: the RoPE key
// is one stream shared by all heads; section 2.5: 576-wide cached rows; the
// GLM-5 explainer page: the top-2048 ids only drive the gather.)
//
// This file holds the CUDA-core path: one CTA per (query row, split of the
// selected list) with the 64-head query block resident in shared memory;
// selected rows are gathered 32 at a time with 16-byte loads, logits and
// the running softmax are fp32, and the output accumulates in registers.
// When a query's selected list is split over several CTAs, each writes an
// fp32 partial (normalised output and lse) to scratch and a merge kernel
// combines them with log-sum-exp weights.
#include <cuda_bf16.h>

#include <algorithm>
#include <cmath>

#include "internal.h"

namespace dsa {
namespace {

constexpr int kThreads = 256;
constexpr int kRows = 32;                       // selected rows per block
constexpr int kQStride = kDQK + 8;              // padded bf16 row stride (bank spread)
constexpr int kKVStride = kDQK + 8;
constexpr int kPStride = kRows + 1;

struct AttnSmem {
    __nv_bfloat16 q[kH * kQStride];
    __nv_bfloat16 kv[kRows * kKVStride];
    float p[kH * kPStride];
    float m[kH], l[kH], alpha[kH];
    int32_t sel[kRows];
};

__device__ __forceinline__ float2 bf2_to_f2(uint32_t v) {
    return make_float2(__uint_as_float(v << 16), __uint_as_float(v & 0xFFFF0000u));
}

__global__ void __launch_bounds__(kThreads, 1)
    sparse_mla_simt_kernel(const BatchDev bd, const RowRange rr, const uint16_t* __restrict__ q,
                           const uint16_t* __restrict__ kv, const int32_t* __restrict__ idx, const int idx_local,
                           const int k, const int rows_per_seq, const int splits, const int per_split,
                           const float sm_scale,
                           uint16_t* __restrict__ out, float* __restrict__ lse, float* __restrict__ part_o,
                           float* __restrict__ part_lse, int32_t* status) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    AttnSmem& S = *reinterpret_cast<AttnSmem*>(smem_raw);
    const int b = blockIdx.y;
    SeqInfo sq;
    if (!load_seq(bd, b, status, sq)) return;
    const int32_t i = rr.i0 + (int32_t)(blockIdx.x / splits);
    const int sp = (int)(blockIdx.x % splits);
    if (i >= min(rr.i1, sq.nq)) return;
    const int32_t t = sq.ctx - sq.nq + i;
    const int64_t grow = (int64_t)sq.q0 + i;                       // packed query row
    const int32_t* sel_row = idx + buf_row(idx_local, sq, b, i, rr) * (int64_t)k;
    const int j_begin = sp * per_split, j_end = min(k, j_begin + per_split);
    const uint16_t* kv_seq = kv + (int64_t)b * bd.stride * kDQK;
    const int tid = threadIdx.x;

    // query block -> shared memory
    {
        const uint4* src = reinterpret_cast<const uint4*>(q + grow * kH * kDQK);
        for (int e = tid; e < kH * kDQK / 8; e += kThreads) {
            const int h = e / (kDQK / 8), c = e % (kDQK / 8);
            *reinterpret_cast<uint4*>(&S.q[h * kQStride + c * 8]) = __ldg(src + e);
        }
    }
    if (tid < kH) {
        S.m[tid] = -INFINITY;
        S.l[tid] = 0.f;
    }
    // thread roles
    const int qk_h = tid >> 2, qk_r = tid & 3;    // QK: head, row phase
    const int pv_h = tid >> 2, pv_c = tid & 3;    // PV: head, column phase
    float acc[128];
#pragma unroll
    for (int c = 0; c < 128; ++c) acc[c] = 0.f;

    for (int jb = j_begin; jb < j_end; jb += kRows) {
        __syncthreads();
        if (tid < kRows) {
            const int j = jb + tid;
            int32_t s = (j < j_end) ? __ldg(sel_row + j) : -1;
            if (s < -1 || s > t) {
                latch_status(status, DSA_ERR_BAD_INDEX);
                s = -1;
            }
            S.sel[tid] = s;
        }
        __syncthreads();
        // gather the selected rows (16 B per load)
        for (int e = tid; e < kRows * (kDQK / 8); e += kThreads) {
            const int r = e / (kDQK / 8), c = e % (kDQK / 8);
            const int32_t s = S.sel[r];
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (s >= 0) v = __ldg(reinterpret_cast<const uint4*>(kv_seq + (int64_t)s * kDQK) + c);
            *reinterpret_cast<uint4*>(&S.kv[r * kKVStride + c * 8]) = v;
        }
        __syncthreads();
        // logits: head qk_h against rows qk_r + 4u
        {
            float dot[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) dot[u] = 0.f;
            const uint32_t* qrow = reinterpret_cast<const uint32_t*>(&S.q[qk_h * kQStride]);
            for (int d2 = 0; d2 < kDQK / 2; ++d2) {
                const float2 qv = bf2_to_f2(qrow[d2]);
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const float2 kvv =
                        bf2_to_f2(reinterpret_cast<const uint32_t*>(&S.kv[(qk_r + 4 * u) * kKVStride])[d2]);
                    dot[u] = fmaf(qv.x, kvv.x, dot[u]);
                    dot[u] = fmaf(qv.y, kvv.y, dot[u]);
                }
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int r = qk_r + 4 * u;
                S.p[qk_h * kPStride + r] = (S.sel[r] >= 0) ? dot[u] * sm_scale : -INFINITY;
            }
        }
        __syncthreads();
        // online softmax, one thread per head
        if (tid < kH) {
            float mx = S.m[tid];
            for (int r = 0; r < kRows; ++r) mx = fmaxf(mx, S.p[tid * kPStride + r]);
            const float alpha = (mx == -INFINITY) ? 1.f : expf(S.m[tid] - mx);
            float sum = 0.f;
            for (int r = 0; r < kRows; ++r) {
                const float lg = S.p[tid * kPStride + r];
                const float pr = (lg == -INFINITY) ? 0.f : expf(lg - mx);
                S.p[tid * kPStride + r] = pr;
                sum += pr;
            }
            S.l[tid] = S.l[tid] * alpha + sum;
            S.m[tid] = mx;
            S.alpha[tid] = alpha;
        }
        __syncthreads();
        // O[h, :] = alpha * O + P @ V  (columns 2*(pv_c + 4c), +1)
        {
            const float alpha = S.alpha[pv_h];
#pragma unroll
            for (int c = 0; c < 128; ++c) acc[c] *= alpha;
            for (int r = 0; r < kRows; ++r) {
                const float pr = S.p[pv_h * kPStride + r];
                const uint32_t* vrow = reinterpret_cast<const uint32_t*>(&S.kv[r * kKVStride]);
#pragma unroll
                for (int c = 0; c < 64; ++c) {
                    const float2 v = bf2_to_f2(vrow[pv_c + 4 * c]);
                    acc[2 * c] = fmaf(pr, v.x, acc[2 * c]);
                    acc[2 * c + 1] = fmaf(pr, v.y, acc[2 * c + 1]);
                }
            }
        }
    }
    __syncthreads();
    const float l = S.l[pv_h], m = S.m[pv_h];
    const float inv = l > 0.f ? 1.f / l : 0.f;
    const float row_lse = l > 0.f ? m + logf(l) : -INFINITY;
    if (splits == 1) {
        uint32_t* o = reinterpret_cast<uint32_t*>(out + (grow * kH + pv_h) * kDV);
#pragma unroll
        for (int c = 0; c < 64; ++c) {
            const __nv_bfloat162 v = __floats2bfloat162_rn(acc[2 * c] * inv, acc[2 * c + 1] * inv);
            o[pv_c + 4 * c] = *reinterpret_cast<const uint32_t*>(&v);
        }
        if (lse && pv_c == 0) lse[grow * kH + pv_h] = row_lse;
    } else {
        const int64_t prow = ((int64_t)b * rows_per_seq + (i - rr.i0)) * splits + sp;
        float2* o = reinterpret_cast<float2*>(part_o + (prow * kH + pv_h) * kDV);
#pragma unroll
        for (int c = 0; c < 64; ++c) o[pv_c + 4 * c] = make_float2(acc[2 * c] * inv, acc[2 * c + 1] * inv);
        if (pv_c == 0) part_lse[prow * kH + pv_h] = row_lse;
    }
}

// out = sum_s exp(lse_s - L) * o_s, L = log sum_s exp(lse_s)
__global__ void __launch_bounds__(256)
    merge_kernel(const BatchDev bd, const RowRange rr, const int rows_per_seq, const int splits,
                 const float* __restrict__ part_o,
                 const float* __restrict__ part_lse, uint16_t* __restrict__ out, float* __restrict__ lse,
                 int32_t* status) {
    const int b = blockIdx.y;
    SeqInfo sq;
    if (!load_seq(bd, b, status, sq)) return;
    const int32_t i = rr.i0 + (int32_t)blockIdx.x;
    if (i >= min(rr.i1, sq.nq)) return;
    const int64_t grow = (int64_t)sq.q0 + i;
    const int64_t prow0 = ((int64_t)b * rows_per_seq + (i - rr.i0)) * splits;
    const int h = threadIdx.x >> 2, part = threadIdx.x & 3;   // 64 heads x 4 column quarters
    float mx = -INFINITY;
    for (int s = 0; s < splits; ++s) mx = fmaxf(mx, part_lse[(prow0 + s) * kH + h]);
    float wsum = 0.f;
    float acc[128];
#pragma unroll
    for (int c = 0; c < 128; ++c) acc[c] = 0.f;
    if (mx > -INFINITY) {
        for (int s = 0; s < splits; ++s) {
            const float ls = part_lse[(prow0 + s) * kH + h];
            if (ls == -INFINITY) continue;
            const float wgt = expf(ls - mx);
            wsum += wgt;
            const float4* o = reinterpret_cast<const float4*>(part_o + ((prow0 + s) * kH + h) * kDV + part * 128);
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                const float4 v = o[c];
                acc[4 * c] = fmaf(wgt, v.x, acc[4 * c]);
                acc[4 * c + 1] = fmaf(wgt, v.y, acc[4 * c + 1]);
                acc[4 * c + 2] = fmaf(wgt, v.z, acc[4 * c + 2]);
                acc[4 * c + 3] = fmaf(wgt, v.w, acc[4 * c + 3]);
            }
        }
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    uint2* o = reinterpret_cast<uint2*>(out + (grow * kH + h) * kDV + part * 128);
#pragma unroll
    for (int c = 0; c < 32; ++c) {
        const __nv_bfloat162 v0 = __floats2bfloat162_rn(acc[4 * c] * inv, acc[4 * c + 1] * inv);
        const __nv_bfloat162 v1 = __floats2bfloat162_rn(acc[4 * c + 2] * inv, acc[4 * c + 3] * inv);
        o[c] = make_uint2(*reinterpret_cast<const uint32_t*>(&v0), *reinterpret_cast<const uint32_t*>(&v1));
    }
    if (lse && part == 0) lse[grow * kH + h] = wsum > 0.f ? mx + logf(wsum) : -INFINITY;
}

// number of CTAs per query row: enough to give ~2 CTAs per SM
int choose_splits(int64_t rows, int k) {
    if (rows <= 0) return 1;
    const int64_t want = (2 * kNumSMs + rows - 1) / rows;
    const int max_by_k = std::max(1, k / 64);
    return (int)std::min<int64_t>(std::max<int64_t>(1, want), std::min(32, max_by_k));
}

}  // namespace

// The split count depends only on the batch bounds, never on how many rows
// one launch covers, so a row's arithmetic is the same in every call.
size_t sparse_mla_scratch_bytes(const BatchDev& bd, int64_t rows_per_seq, int k) {
    const int64_t rows = rows_per_seq * bd.B;
    const int splits = choose_splits((int64_t)bd.B * bd.max_q, k);
    if (splits <= 1) return 0;
    return (size_t)rows * splits * kH * (kDV + 1) * sizeof(float);
}

cudaError_t launch_sparse_mla(const BatchDev& bd, RowRange rr, const uint16_t* q, const uint16_t* kv,
                              const int32_t* idx, bool idx_local, int k, float sm_scale, uint16_t* out,
                              float* lse, void* scratch, size_t scratch_bytes, int32_t* status,
                              cudaStream_t stream) {
    const int32_t rows_per_seq = min(rr.i1, bd.max_q) - rr.i0;
    if (rows_per_seq <= 0) return cudaSuccess;
    const int64_t rows = (int64_t)rows_per_seq * bd.B;
    const int splits = choose_splits((int64_t)bd.B * bd.max_q, k);
    const int per_split = ((k + splits - 1) / splits + kRows - 1) / kRows * kRows;
    float* part_o = nullptr;
    float* part_lse = nullptr;
    if (splits > 1) {
        const size_t need = sparse_mla_scratch_bytes(bd, rows_per_seq, k);
        if (!scratch || scratch_bytes < need) return cudaErrorInvalidValue;
        part_o = static_cast<float*>(scratch);
        part_lse = part_o + (size_t)rows * splits * kH * kDV;
    }
    const size_t smem = sizeof(AttnSmem);
    cudaError_t e =
        cudaFuncSetAttribute(sparse_mla_simt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)(rows_per_seq * splits), bd.B);
    sparse_mla_simt_kernel<<<grid, kThreads, smem, stream>>>(bd, rr, q, kv, idx, idx_local ? 1 : 0, k,
                                                             rows_per_seq, splits, per_split, sm_scale, out,
                                                             lse, part_o, part_lse, status);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    count_launches(1);
    if (splits == 1) return e;
    merge_kernel<<<dim3(rows_per_seq, bd.B), 256, 0, stream>>>(bd, rr, rows_per_seq, splits, part_o, part_lse,
                                                              out, lse, status);
    e = cudaGetLastError();
    if (e == cudaSuccess) count_launches(1);
    return e;
}

}  // namespace dsa
