// indexer.cu -- lightning-indexer scores on the 5th-generation tensor cores.
//
//   I[t,s] = sum_{h<32} w[t,h] * ReLU( q_idx[t,h,:] . k_idx[s,:] )
//
// ("GLM-5.1 架构深度拆解", section 3.2 Steps 4-5 and section 3.6 Step 5;
// the GLM-5 explainer page, indexer paragraph.)
//
// The contraction over the 128 index dims is a dense GEMM: keys are the M
// side (128 keys per tile, one TMEM lane per key) and a group of NQ
// consecutive queries of one sequence times their 32 heads is the N side
// (N = 32 * NQ).  One CTA owns one query group and a contiguous range of
// key tiles; roles are split by warp:
//   warp 0      TMA producer: the query block once, then key tiles through
//               a ring of shared-memory stages (128B-swizzled boxes)
//   warp 1      TMEM allocator and MMA issuer (tcgen05.mma kind::f16,
//               bf16 x bf16 -> fp32), double-buffered accumulators
//   warps 2..    epilogue (8 warps for query groups, two per TMEM lane
//               quarter each taking half of the queries; 4 for a single
//               query): tcgen05.ld one key row per thread (two queries'
//               accumulators per wait), then the ReLU and the
//               head-weighted sum in registers (fp32, four partial sums
//               over the heads in a fixed order), and a coalesced store of
//               one fp32 score per (query, key) with s <= t.
// Scores of positions s > t are never written.
#include <cuda.h>

#include <algorithm>
#include <cstdio>

#include "internal.h"
#include "ptx.cuh"

namespace dsa {
namespace {

// NQ queries per group; kFp8: E4M3 queries and keys with scales (else bf16).
template <int NQ, bool kFp8 = false>
struct IdxCfg {
    static constexpr int kN = NQ * kHIdx;            // MMA N: queries x heads
    static constexpr int kBM = 128;                  // keys per tile: MMA M
    static constexpr int kStages = (NQ == 1) ? 3 : 4;
    // a key row is 128 dims: two 64-element boxes of bf16 or one 128-element
    // box of E4M3, 128 bytes per row either way
    static constexpr int kBoxes = kFp8 ? 1 : 2;
    static constexpr int kBoxElems = kFp8 ? 128 : 64;
    static constexpr int kABoxBytes = kBM * 128;     // 16 KiB
    static constexpr int kABytes = kBoxes * kABoxBytes;
    static constexpr int kBBoxBytes = kN * 128;
    static constexpr int kBBytes = kBoxes * kBBoxBytes;
    static constexpr int kAcc = 2;                   // TMEM accumulator buffers
    static constexpr int kTmemCols = (kN * kAcc < 32) ? 32 : kN * kAcc;
    // epilogue warps: two per TMEM lane quarter (each half of the queries)
    // for query groups, one per quarter for a single query
    static constexpr int kEpiWarps = (NQ >= 8) ? 8 : 4;
    static constexpr int kThreads = 64 + 32 * kEpiWarps;
    static constexpr int kQPerWarp = NQ * 4 / kEpiWarps;  // queries of one epilogue warp
    static constexpr int kEpiQ = (kQPerWarp >= 2) ? 2 : 1;    // queries read from TMEM per wait
    static constexpr int kOffA = 0;
    static constexpr int kOffB = kOffA + kStages * kABytes;
    static constexpr int kOffW = kOffB + kBBytes;
    static constexpr int kOffBar = kOffW + NQ * kHIdx * 4;
    static constexpr int kNumBars = 2 * kStages + 1 + 2 * kAcc + 1;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;
    static constexpr int kSmemBytes = kOffMisc + 16 + 1024;  // + slack for 1 KiB alignment
    static_assert(kTmemCols == 32 || kTmemCols == 64 || kTmemCols == 128 || kTmemCols == 256 ||
                      kTmemCols == 512,
                  "TMEM allocation must be a power of two >= 32");
    static_assert(kN % 16 == 0 && kN >= 16 && kN <= 256, "invalid MMA N for M = 128");
};

template <int NQ, bool kFp8>
__global__ void __launch_bounds__(IdxCfg<NQ, kFp8>::kThreads, 1)
    indexer_kernel(const BatchDev bd, const RowRange rr, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_q, const float* __restrict__ w,
                   const float* __restrict__ qscale, const float* __restrict__ kscale,
                   float* __restrict__ scores, const int64_t ld, const int scores_local,
                   const int tiles_per_split, int32_t* status) {
    using C = IdxCfg<NQ, kFp8>;
    constexpr int kEpiQ = C::kEpiQ;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    pdl_launch_dependents();     // a dependent top-k may start launching
    const int b = blockIdx.z;
    SeqInfo sq;
    if (!load_seq(bd, b, status, sq)) return;
    // query groups in reverse: the longest causal key ranges start first,
    // which shortens the launch's tail (16,384-token prefill: 0.99 -> 0.95 ms)
    const int32_t qlo = rr.i0 + (int32_t)(gridDim.y - 1 - blockIdx.y) * NQ;   // local query indices [qlo, qhi)
    const int32_t qhi = min(min(qlo + NQ, rr.i1), sq.nq);
    if (qlo >= qhi) return;
    const int32_t pos0 = sq.ctx - sq.nq;                             // position of local query 0
    const int32_t ntiles = (pos0 + qhi - 1) / C::kBM + 1;
    const int32_t j0 = (int32_t)blockIdx.x * tiles_per_split;
    const int32_t j1 = min(j0 + tiles_per_split, ntiles);
    if (j0 >= j1) return;
    const int niter = j1 - j0;

    const uint32_t sA = smem_u32(smem + C::kOffA);
    const uint32_t sB = smem_u32(smem + C::kOffB);
    float* w_s = reinterpret_cast<float*>(smem + C::kOffW);
    const uint32_t bar0 = smem_u32(smem + C::kOffBar);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (C::kStages + s); };
    const uint32_t bfull_bar = bar0 + 8u * (2 * C::kStages);
    auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * C::kStages + 1 + a); };
    auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * C::kStages + 1 + C::kAcc + a); };
    const uint32_t drain_bar = bar0 + 8u * (2 * C::kStages + 1 + 2 * C::kAcc);
    volatile uint32_t* misc = reinterpret_cast<volatile uint32_t*>(smem + C::kOffMisc);

    const uint32_t warp = warp_id(), lane = lane_id();

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        mbar_init(bfull_bar, 1);
        for (int a = 0; a < C::kAcc; ++a) {
            mbar_init(tfull_bar(a), 1);
            mbar_init(tempty_bar(a), 32 * C::kEpiWarps);
        }
        mbar_init(drain_bar, 1);
        misc[1] = 0;  // abort flag
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(smem + C::kOffMisc), C::kTmemCols);
        tmem_relinquish();
    }
    if (warp >= 2) {
        // head weights of the group (0 for rows past the group's end)
        for (int e = threadIdx.x - 64; e < NQ * kHIdx; e += 32 * C::kEpiWarps) {
            const int qi = e / kHIdx;
            const int64_t wi = ((int64_t)sq.q0 + qlo + qi) * kHIdx + (e % kHIdx);
            // E4M3 queries: the positive scale of each (token, head) passes
            // through the ReLU and folds into the head weight
            w_s[e] = (qlo + qi < qhi) ? __ldg(w + wi) * (kFp8 ? __ldg(qscale + wi) : 1.f) : 0.f;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = misc[0];

    if (warp == 0) {
        // ---------------------------------------------------- TMA producer
        if (elect_one()) {
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_q);
            const int32_t qrow = (sq.q0 + qlo) * kHIdx;
            mbar_arrive_expect_tx(bfull_bar, C::kBBytes);
#pragma unroll
            for (int bx = 0; bx < C::kBoxes; ++bx)
                tma_load_2d(sB + bx * C::kBBoxBytes, &tm_q, bfull_bar, bx * C::kBoxElems, qrow);
            // one query group per sequence: every key is read by one CTA only,
            // so the stream is marked evict-first and the scores produced
            // from it stay in L2 for the top-k
            const bool once = bd.max_q <= NQ;
            const uint64_t pol = l2_evict_first_policy();
            int issued = 0;
            for (int it = 0; it < niter; ++it) {
                const int s = it % C::kStages;
                const uint32_t ph = (it / C::kStages) & 1u;
                if (misc[1] || !mbar_wait(empty_bar(s), ph ^ 1u)) {
                    latch_status(status, DSA_ERR_TIMEOUT);
                    misc[1] = 1;
                    break;
                }
                const int32_t krow = (int32_t)((int64_t)b * bd.stride + (int64_t)(j0 + it) * C::kBM);
                mbar_arrive_expect_tx(full_bar(s), C::kABytes);
#pragma unroll
                for (int bx = 0; bx < C::kBoxes; ++bx) {
                    const uint32_t dst = sA + s * C::kABytes + bx * C::kABoxBytes;
                    if (once) tma_load_2d_hint(dst, &tm_k, full_bar(s), bx * C::kBoxElems, krow, pol);
                    else tma_load_2d(dst, &tm_k, full_bar(s), bx * C::kBoxElems, krow);
                }
                ++issued;
            }
            if (misc[1]) {
                // wind down: let every copy this thread started land first
                for (int it = max(0, issued - C::kStages); it < issued; ++it)
                    mbar_wait(full_bar(it % C::kStages), (it / C::kStages) & 1u);
                mbar_wait(bfull_bar, 0);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------ MMA issuer
        if (elect_one()) {
            constexpr uint32_t idesc = kFp8 ? idesc_e4m3_f32(C::kBM, C::kN) : idesc_bf16_f32(C::kBM, C::kN);
            bool ok = mbar_wait(bfull_bar, 0);
            tc_fence_after();
            for (int it = 0; ok && it < niter; ++it) {
                const int s = it % C::kStages;
                const int a = it & 1;
                if (misc[1] || !mbar_wait(full_bar(s), (it / C::kStages) & 1u) ||
                    !mbar_wait(tempty_bar(a), ((it >> 1) & 1u) ^ 1u)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem_base + (uint32_t)(a * C::kN);
#pragma unroll
                for (int kb = 0; kb < C::kBoxes; ++kb) {
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks) {       // 32 bytes of K per instruction
                        const uint64_t ad =
                            sdesc_sw128(sA + s * C::kABytes + kb * C::kABoxBytes + ks * 32, 16, 1024);
                        const uint64_t bdsc = sdesc_sw128(sB + kb * C::kBBoxBytes + ks * 32, 16, 1024);
                        if (kFp8) mma_f8_ss(d, ad, bdsc, idesc, (kb | ks) != 0);
                        else mma_bf16_ss(d, ad, bdsc, idesc, (kb | ks) != 0);
                    }
                }
                mma_commit(empty_bar(s));
                mma_commit(tfull_bar(a));
            }
            if (!ok) {
                latch_status(status, DSA_ERR_TIMEOUT);
                misc[1] = 1;
            }
            // every MMA this thread issued has finished once drain completes
            mma_commit(drain_bar);
            mbar_wait(drain_bar, 0);
        }
        __syncwarp();
    } else {
        // -------------------------------------------------------- epilogue
        const uint32_t lq = warp & 3u;                     // TMEM lane quarter of this warp
        const int32_t row = (int32_t)(lq * 32 + lane);     // key row within the tile
        const int q_first = (int)((warp - 2) >> 2) * C::kQPerWarp;   // this warp's queries
        for (int it = 0; it < niter; ++it) {
            const int a = it & 1;
            bool ok = !misc[1] && mbar_wait(tfull_bar(a), (it >> 1) & 1u);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) {
                latch_status(status, DSA_ERR_TIMEOUT);
                misc[1] = 1;
                break;
            }
            tc_fence_after();
            const int32_t s = (j0 + it) * C::kBM + row;
            const uint32_t tq = tmem_base + ((lq * 32u) << 16) + (uint32_t)(a * C::kN);
            // E4M3 keys: the key's positive scale multiplies its whole score
            const float kmul = kFp8 && s <= pos0 + qhi - 1 ? __ldg(kscale + (int64_t)b * bd.stride + s) : 1.f;
#pragma unroll 1
            for (int q0 = q_first; q0 < q_first + C::kQPerWarp; q0 += kEpiQ) {
                // kEpiQ queries' accumulators in flight before one wait
                uint32_t r[kEpiQ][32];
#pragma unroll
                for (int u = 0; u < kEpiQ; ++u) tmem_ld_32x32b_x32(tq + (uint32_t)((q0 + u) * 32), r[u]);
                tmem_ld_wait();
#pragma unroll
                for (int u = 0; u < kEpiQ; ++u) {
                    const int32_t i = qlo + q0 + u;
                    const float4* wq = reinterpret_cast<const float4*>(w_s + (q0 + u) * kHIdx);
                    // four partial sums over heads h = 4m + j, m in order, then (a0 + a1) + (a2 + a3)
                    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int m = 0; m < kHIdx / 4; ++m) {
                        const float4 wv = wq[m];
                        acc[0] = fmaf(wv.x, fmaxf(__uint_as_float(r[u][4 * m]), 0.f), acc[0]);
                        acc[1] = fmaf(wv.y, fmaxf(__uint_as_float(r[u][4 * m + 1]), 0.f), acc[1]);
                        acc[2] = fmaf(wv.z, fmaxf(__uint_as_float(r[u][4 * m + 2]), 0.f), acc[2]);
                        acc[3] = fmaf(wv.w, fmaxf(__uint_as_float(r[u][4 * m + 3]), 0.f), acc[3]);
                    }
                    const float v = ((acc[0] + acc[1]) + (acc[2] + acc[3])) * kmul;
                    if (i < qhi && s <= pos0 + i) scores[buf_row(scores_local, sq, b, i, rr) * ld + s] = v;
                }
            }
            tc_fence_before();
            mbar_arrive(tempty_bar(a));
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, C::kTmemCols);
    }
}

template <int NQ, bool kFp8>
cudaError_t launch_nq(const BatchDev& bd, RowRange rr, const void* q_idx, const float* qs, const float* w,
                      const void* k_idx, const float* ks, float* scores, int64_t ld, bool scores_local,
                      int32_t* status, cudaStream_t stream) {
    using C = IdxCfg<NQ, kFp8>;
    const int32_t rows_per_seq = min(rr.i1, bd.max_q) - rr.i0;
    if (rows_per_seq <= 0 || bd.max_ctx <= 0) return cudaSuccess;
    const int32_t groups = (rows_per_seq + NQ - 1) / NQ;
    const int32_t tiles = (bd.max_ctx + C::kBM - 1) / C::kBM;
    int tps;
    if (NQ > 1) {
        // query groups: long key ranges per CTA amortise its setup (TMEM,
        // barriers, the query block) -- measured 1.10 ms at 16 tiles, 0.99 ms
        // at 64 for a 16,384-token prefill
        tps = 64;
    } else {
        // decode-like: spread every sequence's key stream over enough CTAs
        // for ~4 CTAs per SM in total
        const int64_t total = (int64_t)tiles * groups * bd.B;
        const int64_t nsm = num_sms();
        tps = (int)std::max<int64_t>(4, (total + 4 * nsm - 1) / (4 * nsm));
    }
    const int32_t splits = (tiles + tps - 1) / tps;
    CUtensorMap tm_k, tm_q;
    const uint64_t krows = (uint64_t)bd.B * (uint64_t)bd.stride, qrows = (uint64_t)bd.total_q * kHIdx;
    const bool ok = kFp8 ? make_tmap_u8_2d(&tm_k, k_idx, kDIdx, krows, C::kBoxElems, C::kBM) &&
                               make_tmap_u8_2d(&tm_q, q_idx, kDIdx, qrows, C::kBoxElems, C::kN)
                         : make_tmap_bf16_2d(&tm_k, k_idx, kDIdx, krows, C::kBoxElems, C::kBM) &&
                               make_tmap_bf16_2d(&tm_q, q_idx, kDIdx, qrows, C::kBoxElems, C::kN);
    if (!ok) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(indexer_kernel<NQ, kFp8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::kSmemBytes);
    if (e != cudaSuccess) return e;
    dim3 grid(splits, groups, bd.B);
    indexer_kernel<NQ, kFp8><<<grid, C::kThreads, C::kSmemBytes, stream>>>(
        bd, rr, tm_k, tm_q, w, qs, ks, scores, ld, scores_local ? 1 : 0, tps, status);
    const cudaError_t err = cudaGetLastError();
    if (err == cudaSuccess) count_launches(1);
    return err;
}

}  // namespace

cudaError_t launch_indexer(const BatchDev& bd, RowRange rr, const uint16_t* q_idx, const float* w,
                           const uint16_t* k_idx, float* scores, int64_t ld, bool scores_local,
                           int32_t* status, cudaStream_t stream) {
    if (bd.max_q >= 16)
        return launch_nq<8, false>(bd, rr, q_idx, nullptr, w, k_idx, nullptr, scores, ld, scores_local, status,
                                   stream);
    return launch_nq<1, false>(bd, rr, q_idx, nullptr, w, k_idx, nullptr, scores, ld, scores_local, status, stream);
}

cudaError_t launch_indexer_fp8(const BatchDev& bd, RowRange rr, const uint8_t* q8, const float* qs, const float* w,
                               const uint8_t* k8, const float* ks, float* scores, int64_t ld, bool scores_local,
                               int32_t* status, cudaStream_t stream) {
    if (bd.max_q >= 16)
        return launch_nq<8, true>(bd, rr, q8, qs, w, k8, ks, scores, ld, scores_local, status, stream);
    return launch_nq<1, true>(bd, rr, q8, qs, w, k8, ks, scores, ld, scores_local, status, stream);
}

// One warp per row of 128 values: amax -> scale = amax / 448 (1 for a zero
// row), codes = E4M3(v / scale) by the hardware's round-to-nearest-even
// conversion with saturation to +-448.
__global__ void __launch_bounds__(256) quantize_fp8_kernel(int64_t rows, const uint16_t* __restrict__ in,
                                                           uint8_t* __restrict__ codes, float* __restrict__ scale) {
    const int lane = threadIdx.x & 31;
    const int64_t r = (int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
    if (r >= rows) return;
    const uint2 raw = reinterpret_cast<const uint2*>(in + r * kDIdx)[lane];     // 4 bf16 values
    float v[4] = {__uint_as_float(raw.x << 16), __uint_as_float(raw.x & 0xFFFF0000u),
                  __uint_as_float(raw.y << 16), __uint_as_float(raw.y & 0xFFFF0000u)};
    float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float sc = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
    uint16_t lo, hi;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(__fdiv_rn(v[1], sc)), "f"(__fdiv_rn(v[0], sc)));
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(__fdiv_rn(v[3], sc)), "f"(__fdiv_rn(v[2], sc)));
    reinterpret_cast<uint32_t*>(codes + r * kDIdx)[lane] = (uint32_t)lo | ((uint32_t)hi << 16);
    if (lane == 0) scale[r] = sc;
}

cudaError_t launch_quantize_fp8(int64_t rows, const uint16_t* in, uint8_t* codes, float* scale, cudaStream_t stream) {
    if (rows <= 0) return cudaSuccess;
    const int warps = 8;
    quantize_fp8_kernel<<<(unsigned)((rows + warps - 1) / warps), 32 * warps, 0, stream>>>(rows, in, codes, scale);
    const cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) count_launches(1);
    return e;
}

}  // namespace dsa
