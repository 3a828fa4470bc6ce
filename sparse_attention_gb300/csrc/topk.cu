// topk.cu -- deterministic causal top-k of indexer score rows.
//
// ("GLM-5.1 架构深度拆解", section 3.6 Steps 6-7: positions s > t are masked
// and min(index_topk, length) positions are kept; section 3.4: the
// selection must be deterministic; the GLM-5 explainer page: a query that
// sees fewer than 2048 positions keeps all of them.)
//
// One CTA per query row.  Scores are mapped to order-preserving 32-bit keys
// (-0.0 folded onto +0.0) and the k-th largest key tau is found by a radix
// select over three digits (11 + 11 + 10 bits), each a shared-memory
// histogram restricted to the keys that match the digits found so far.
// The output is then written by one ordered pass over the row: a key above
// tau is taken, a key equal to tau is taken while fewer than `need` equal
// keys have been taken before it (so ties go to the lower position), and
// each taken position is written at its rank in position order, found by
// block-wide prefix sums.  Positions come out ascending; no atomics decide
// anything but the (order-free) histogram counts, so the result is the same
// bit for bit on every run.  A row short enough to fit in shared memory is
// read from global memory once; a longer row is re-read per pass (from L2
// when it was just written).
#include "internal.h"

namespace dsa {
namespace {

constexpr int kThreads = 1024;
constexpr int kBins = 2048;
constexpr int kMaxSmemKeys = 40960;   // 160 KiB of keys

__device__ __forceinline__ uint32_t order_key(float f) {
    uint32_t u = __float_as_uint(f);
    if (u == 0x80000000u) u = 0u;     // -0.0 compares equal to +0.0
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Inclusive block-wide scan of one 32-bit value per thread.
__device__ __forceinline__ uint32_t block_inclusive_scan(uint32_t v, uint32_t* warp_sums) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t n = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += n;
    }
    if (lane == 31) warp_sums[warp] = v;
    __syncthreads();
    if (warp == 0) {
        uint32_t s = warp_sums[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t n = __shfl_up_sync(0xffffffffu, s, o);
            if (lane >= o) s += n;
        }
        warp_sums[lane] = s;      // inclusive warp prefix
    }
    __syncthreads();
    const uint32_t add = warp ? warp_sums[warp - 1] : 0u;
    const uint32_t res = v + add;
    __syncthreads();              // warp_sums may be reused right after
    return res;
}

struct TopkSmem {
    uint32_t hist[kBins];
    uint32_t warp_sums[32];
    uint32_t sel_digit, sel_above, total, chunk_total;
};

__global__ void __launch_bounds__(kThreads, 1)
    topk_kernel(const BatchDev bd, const RowRange rr, const float* __restrict__ scores, const int64_t ld,
                const int scores_local, const int k, int32_t* __restrict__ idx, const int idx_local,
                const int smem_keys, int32_t* status) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    TopkSmem& S = *reinterpret_cast<TopkSmem*>(smem_raw);
    uint32_t* keys = reinterpret_cast<uint32_t*>(smem_raw + sizeof(TopkSmem));

    const int b = blockIdx.y;
    SeqInfo sq;
    if (!load_seq(bd, b, status, sq)) return;
    const int32_t i = rr.i0 + (int32_t)blockIdx.x;
    if (i >= min(rr.i1, sq.nq)) return;
    const int32_t t = sq.ctx - sq.nq + i;
    const int32_t n = t + 1;
    const float* row = scores + buf_row(scores_local, sq, b, i, rr) * ld;
    int32_t* out = idx + buf_row(idx_local, sq, b, i, rr) * (int64_t)k;
    const int tid = threadIdx.x;

    if (n <= k) {  // every causal position is selected
        for (int j = tid; j < k; j += kThreads) out[j] = j < n ? j : -1;
        return;
    }

    const int32_t n4 = (n + 3) & ~3;          // rows are padded to ld, ld % 4 == 0
    const bool in_smem = n4 <= smem_keys;
    if (in_smem) {
        const float4* r4 = reinterpret_cast<const float4*>(row);
        for (int j = tid; j < n4 / 4; j += kThreads) {
            const float4 v = __ldg(r4 + j);
            reinterpret_cast<uint4*>(keys)[j] =
                make_uint4(order_key(v.x), order_key(v.y), order_key(v.z), order_key(v.w));
        }
    }
    auto key_at = [&](int32_t j) -> uint32_t { return in_smem ? keys[j] : order_key(__ldg(row + j)); };

    // ---------------------------------------------------- radix select
    uint32_t prefix = 0u, pmask = 0u;
    uint32_t need = (uint32_t)k;
    const int shifts[3] = {21, 10, 0};
    const uint32_t widths[3] = {11u, 11u, 10u};
#pragma unroll 1
    for (int p = 0; p < 3; ++p) {
        const int sh = shifts[p];
        const uint32_t dmask = (1u << widths[p]) - 1u;
        for (int e = tid; e < kBins; e += kThreads) S.hist[e] = 0u;
        __syncthreads();
        for (int32_t j = tid; j < n; j += kThreads) {
            const uint32_t key = key_at(j);
            if ((key & pmask) == prefix) atomicAdd(&S.hist[(key >> sh) & dmask], 1u);
        }
        __syncthreads();
        // thread tid owns bins 2*tid and 2*tid+1; the count of keys in bins
        // above them is the block total minus an inclusive scan in bin order
        const uint32_t c0 = S.hist[2 * tid], c1 = S.hist[2 * tid + 1];
        const uint32_t incl = block_inclusive_scan(c0 + c1, S.warp_sums);
        if (tid == kThreads - 1) S.total = incl;
        __syncthreads();
        const uint32_t total = S.total;
        const uint32_t above1 = total - incl;          // bins > 2*tid+1
        const uint32_t above0 = above1 + c1;           // bins > 2*tid
        if (above1 < need && need <= above1 + c1) {
            S.sel_digit = 2u * tid + 1u;
            S.sel_above = above1;
        }
        if (above0 < need && need <= above0 + c0) {
            S.sel_digit = 2u * tid;
            S.sel_above = above0;
        }
        __syncthreads();
        const uint32_t d = S.sel_digit;
        need -= S.sel_above;
        prefix |= d << sh;
        pmask |= dmask << sh;
        __syncthreads();
    }
    const uint32_t tau = prefix;      // the k-th largest key; `need` keys equal to it are taken

    // ------------------------------------------------ ordered compaction
    uint32_t gt_run = 0u, eq_run = 0u;
    constexpr int kE = 4;
#pragma unroll 1
    for (int32_t base = 0; base < n; base += kThreads * kE) {
        const int32_t j0 = base + tid * kE;
        uint32_t kk[kE] = {0u, 0u, 0u, 0u};
        if (in_smem) {
            if (j0 < n4) {
                const uint4 v = reinterpret_cast<const uint4*>(keys)[j0 / 4];
                kk[0] = v.x; kk[1] = v.y; kk[2] = v.z; kk[3] = v.w;
            }
        } else if (j0 < n4) {
            const float4 v = __ldg(reinterpret_cast<const float4*>(row) + j0 / 4);
            kk[0] = order_key(v.x); kk[1] = order_key(v.y); kk[2] = order_key(v.z); kk[3] = order_key(v.w);
        }
        uint32_t gt = 0u, eq = 0u;
#pragma unroll
        for (int e = 0; e < kE; ++e) {
            if (j0 + e < n) {
                gt += kk[e] > tau;
                eq += kk[e] == tau;
            }
        }
        const uint32_t packed = block_inclusive_scan(gt | (eq << 16), S.warp_sums);
        if (tid == kThreads - 1) S.chunk_total = packed;
        uint32_t gtb = gt_run + (packed & 0xFFFFu) - gt;
        uint32_t eqb = eq_run + (packed >> 16) - eq;
#pragma unroll
        for (int e = 0; e < kE; ++e) {
            if (j0 + e < n) {
                if (kk[e] > tau) {
                    out[gtb + min(eqb, need)] = j0 + e;
                    ++gtb;
                } else if (kk[e] == tau) {
                    if (eqb < need) out[gtb + eqb] = j0 + e;
                    ++eqb;
                }
            }
        }
        __syncthreads();
        gt_run += S.chunk_total & 0xFFFFu;
        eq_run += S.chunk_total >> 16;
        __syncthreads();
    }
}

}  // namespace

cudaError_t launch_topk(const BatchDev& bd, RowRange rr, const float* scores, int64_t ld, bool scores_local,
                        int k, int32_t* idx, bool idx_local, int32_t* status, cudaStream_t stream) {
    const int32_t rows_per_seq = min(rr.i1, bd.max_q) - rr.i0;
    if (rows_per_seq <= 0) return cudaSuccess;
    const int32_t max_n4 = (bd.max_ctx + 3) & ~3;
    const int smem_keys = max_n4 <= kMaxSmemKeys ? max_n4 : 0;
    const size_t smem = sizeof(TopkSmem) + (size_t)smem_keys * 4;
    cudaError_t e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid(rows_per_seq, bd.B);
    topk_kernel<<<grid, kThreads, smem, stream>>>(bd, rr, scores, ld, scores_local ? 1 : 0, k, idx,
                                                  idx_local ? 1 : 0, smem_keys, status);
    const cudaError_t err = cudaGetLastError();
    if (err == cudaSuccess) count_launches(1);
    return err;
}

}  // namespace dsa
