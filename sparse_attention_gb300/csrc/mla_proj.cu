// mla_proj.cu -- the MLA projections on either side of the sparse attention,
// in absorbed form, on the 5th-generation tensor cores.
//
// ("GLM-5.1 架构深度拆解", section 4.5 Steps 1-4 and 7-8: kv_b_proj expands
// the 512-dim compressed KV to 64 heads x (192 nope key + 256 value), o_proj
// maps the 64 x 256 head outputs to the 6144-dim hidden state; section 4.1
// and section 2.5: the cache keeps the 512 + 64 compressed row.)  With
// W_UK[h] = rows h*448 .. +191 and W_UV[h] = rows h*448+192 .. +447 of
// kv_b_proj's weight [64*448, 512]:
//   q[t,h] . (W_UK[h] c) = (W_UK[h]^T q[t,h]) . c    -> absorb_q before the attention
//   sum_s p_s (W_UV[h] c_s) = W_UV[h] (sum_s p_s c_s) -> W_UV after it, then o_proj
// so the attention runs on the cached 576-wide rows directly.
//
// All three products are one bf16 GEMM kernel, C = A . B (fp32 accumulation
// in TMEM, bf16 out), batched over heads by shifting A's column, B's row and
// C's column per batch index:
//   absorb_q : A = q_nope[:, h, :] [T, 192], B = W_UK[h] as [K=192, N=512] (N-major)
//   W_UV     : A = o_lat[:, h, :]  [T, 512], B = W_UV[h] as [N=256, K=512] (K-major)
//   o_proj   : A = o [T, 16384],             B = W_o [N=6144, K=16384]     (K-major)
// Tiles of 128 x 256 with K steps of 64; persistent CTAs walk the tiles in
// groups of m-tiles (operand reuse in L2).  Roles by warp:
//   warp 0      TMA producer: A and B boxes through a 4-stage ring
//   warp 1      TMEM owner and MMA issuer (tcgen05.mma kind::f16), two
//               256-column accumulators so a tile's epilogue overlaps the
//               next tile's MMAs
//   warps 2..5  epilogue: tcgen05.ld one output row per thread, round to
//               bf16, store.
#include <algorithm>

#include "internal.h"
#include "ptx.cuh"

namespace dsa {
namespace {

constexpr int kBM = 128, kBN = 256, kBK = 64;
constexpr int kStages = 4;
constexpr int kABytes = kBM * kBK * 2;      // 16 KiB
constexpr int kBBytes = kBN * kBK * 2;      // 32 KiB
constexpr int kBBoxMnBytes = kBK * 64 * 2;  // one 64 (k) x 64 (n) box of an N-major B: 8 KiB
constexpr int kThreads = 192;
constexpr int kTmemCols = 2 * kBN;
constexpr int kGroupM = 16;                 // m-tiles per raster group
constexpr int kOffA = 0;
constexpr int kOffB = kOffA + kStages * kABytes;
constexpr int kOffBar = kOffB + kStages * kBBytes;
constexpr int kNumBars = 2 * kStages + 4 + 1;
constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kSmemBytes = kOffMisc + 16 + 1024;

constexpr int kDNope = 192, kDRope = 64, kDVh = 256, kKvbRows = 448, kHidden = 6144;

struct GemmArgs {
    int32_t M, N, K, batches;
    int32_t a_col0, a_col_step;   // A column of k = 0 for batch b: a_col0 + b * a_col_step
    int32_t b_row0, b_row_step;   // B row of n = 0 (K-major) or of k = 0 (N-major) for batch b
    uint16_t* C;
    int64_t ldc, c_col0, c_col_step;
    int32_t tiles_m, tiles_n;
    // split-K: splits > 1 writes fp32 partials part[s][m][ldc] (same column
    // layout as C); reduce_kernel then sums them in split order into C.
    // out_fp32: the partials are the result (no bf16 C, no reduce).
    int32_t splits;
    float* part;
    int32_t out_fp32;
};

// Tile `tile` -> batch b, m-tile, n-tile and K split ks (K splits outermost).
__device__ __forceinline__ void tile_coords(const GemmArgs& g, int32_t tile, int32_t& b, int32_t& mt, int32_t& nt,
                                            int32_t& ks) {
    const int32_t per_batch = g.tiles_m * g.tiles_n;
    const int32_t per_split = per_batch * g.batches;
    ks = tile / per_split;
    tile -= ks * per_split;
    b = tile / per_batch;
    const int32_t r = tile - b * per_batch;
    // groups of kGroupM m-tiles: within a group m moves fastest
    const int32_t group = r / (kGroupM * g.tiles_n);
    const int32_t first_m = group * kGroupM;
    const int32_t gm = min(g.tiles_m - first_m, kGroupM);
    const int32_t in_group = r - group * kGroupM * g.tiles_n;
    mt = first_m + in_group % gm;
    nt = in_group / gm;
}

template <bool kBMn>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_bf16_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                     const GemmArgs g, int32_t* status) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sA = smem_u32(smem + kOffA);
    const uint32_t sB = smem_u32(smem + kOffB);
    const uint32_t bar0 = smem_u32(smem + kOffBar);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (kStages + s); };
    auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * kStages + a); };
    auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * kStages + 2 + a); };
    const uint32_t drain_bar = bar0 + 8u * (2 * kStages + 4);
    volatile uint32_t* misc = reinterpret_cast<volatile uint32_t*>(smem + kOffMisc);
    const uint32_t warp = warp_id(), lane = lane_id();

    const int32_t total_tiles = g.tiles_m * g.tiles_n * g.batches * g.splits;
    const int32_t nk = g.K / kBK;
    // k-tiles [k_lo(ks), k_lo(ks + 1)) belong to split ks
    auto k_lo = [&](int32_t ks) { return (int32_t)(((int64_t)nk * ks) / g.splits); };

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull_bar(a), 1);
            mbar_init(tempty_bar(a), 128);
        }
        mbar_init(drain_bar, 1);
        misc[1] = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(smem + kOffMisc), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = misc[0];

    if (warp == 0) {
        // ---------------------------------------------------- TMA producer
        if (elect_one()) {
            prefetch_tmap(&tm_a);
            prefetch_tmap(&tm_b);
            int it = 0;
            bool ok = true;
            for (int32_t tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x) {
                int32_t b, mt, nt, ks;
                tile_coords(g, tile, b, mt, nt, ks);
                const int32_t ax = g.a_col0 + b * g.a_col_step;
                const int32_t brow = g.b_row0 + b * g.b_row_step;
                for (int kt = k_lo(ks); kt < k_lo(ks + 1); ++kt, ++it) {
                    const int s = it % kStages;
                    if (misc[1] || !mbar_wait(empty_bar(s), ((it / kStages) & 1u) ^ 1u)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(full_bar(s), kABytes + kBBytes);
                    tma_load_2d(sA + s * kABytes, &tm_a, full_bar(s), ax + kt * kBK, mt * kBM);
                    if (kBMn) {
#pragma unroll
                        for (int j = 0; j < kBN / 64; ++j)
                            tma_load_2d(sB + s * kBBytes + j * kBBoxMnBytes, &tm_b, full_bar(s), nt * kBN + j * 64,
                                        brow + kt * kBK);
                    } else {
                        tma_load_2d(sB + s * kBBytes, &tm_b, full_bar(s), kt * kBK, brow + nt * kBN);
                    }
                }
            }
            if (!ok) {
                latch_status(status, DSA_ERR_TIMEOUT);
                misc[1] = 1;
                // wind down: let the copies of the last stages land
                for (int j = max(0, it - kStages); j < it; ++j) mbar_wait(full_bar(j % kStages), (j / kStages) & 1u);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------ MMA issuer
        if (elect_one()) {
            constexpr uint32_t idesc = idesc_bf16_f32(kBM, kBN, false, kBMn);
            int it = 0, lt = 0;
            bool ok = true;
            for (int32_t tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x, ++lt) {
                const int a = lt & 1;
                if (misc[1] || !mbar_wait(tempty_bar(a), ((lt >> 1) & 1u) ^ 1u)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem_base + (uint32_t)(a * kBN);
                int32_t b, mt, nt, ks;
                tile_coords(g, tile, b, mt, nt, ks);
                const int32_t kt0 = k_lo(ks);
                for (int kt = kt0; kt < k_lo(ks + 1); ++kt, ++it) {
                    const int s = it % kStages;
                    if (misc[1] || !mbar_wait(full_bar(s), (it / kStages) & 1u)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk) {
                        const uint64_t ad = sdesc_sw128(sA + s * kABytes + kk * 32, 16, 1024);
                        const uint64_t bd = kBMn ? sdesc_sw128(sB + s * kBBytes + kk * 2048, kBBoxMnBytes, 1024)
                                                 : sdesc_sw128(sB + s * kBBytes + kk * 32, 16, 1024);
                        mma_bf16_ss(d, ad, bd, idesc, kt != kt0 || kk != 0);
                    }
                    mma_commit(empty_bar(s));
                }
                if (!ok) break;
                mma_commit(tfull_bar(a));
            }
            if (!ok) {
                latch_status(status, DSA_ERR_TIMEOUT);
                misc[1] = 1;
            }
            mma_commit(drain_bar);
            mbar_wait(drain_bar, 0);
        }
        __syncwarp();
    } else {
        // -------------------------------------------------------- epilogue
        const uint32_t lq = warp & 3u;
        const int32_t row = (int32_t)(lq * 32 + lane);
        int lt = 0;
        for (int32_t tile = blockIdx.x; tile < total_tiles; tile += gridDim.x, ++lt) {
            const int a = lt & 1;
            bool ok = !misc[1] && mbar_wait(tfull_bar(a), (lt >> 1) & 1u);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) {
                latch_status(status, DSA_ERR_TIMEOUT);
                misc[1] = 1;
                break;
            }
            tc_fence_after();
            int32_t b, mt, nt, ks;
            tile_coords(g, tile, b, mt, nt, ks);
            const int32_t m = mt * kBM + row;
            const int64_t col = g.c_col0 + (int64_t)b * g.c_col_step + (int64_t)nt * kBN;
            uint16_t* crow = g.C + (int64_t)m * g.ldc + col;
            float* prow = g.part + ((int64_t)ks * g.M + m) * g.ldc + col;
            const uint32_t taddr = tmem_base + ((lq * 32u) << 16) + (uint32_t)(a * kBN);
#pragma unroll 1
            for (int c = 0; c < kBN / 32; ++c) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(taddr + (uint32_t)(c * 32), r);
                tmem_ld_wait();
                if (m < g.M && nt * kBN + c * 32 < g.N && (g.splits > 1 || g.out_fp32)) {
                    float4* dst = reinterpret_cast<float4*>(prow + c * 32);
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        dst[q] = make_float4(__uint_as_float(r[4 * q]), __uint_as_float(r[4 * q + 1]),
                                             __uint_as_float(r[4 * q + 2]), __uint_as_float(r[4 * q + 3]));
                } else if (m < g.M && nt * kBN + c * 32 < g.N) {
                    uint4* dst = reinterpret_cast<uint4*>(crow + c * 32);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        uint4 pk;
                        pk.x = pack_bf16x2(__uint_as_float(r[8 * q]), __uint_as_float(r[8 * q + 1]));
                        pk.y = pack_bf16x2(__uint_as_float(r[8 * q + 2]), __uint_as_float(r[8 * q + 3]));
                        pk.z = pack_bf16x2(__uint_as_float(r[8 * q + 4]), __uint_as_float(r[8 * q + 5]));
                        pk.w = pack_bf16x2(__uint_as_float(r[8 * q + 6]), __uint_as_float(r[8 * q + 7]));
                        dst[q] = pk;
                    }
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
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

// C[m, c] = bf16(sum over splits s, in order, of part[s][m][c]) for the
// whole [M, ldc] footprint; 8 columns per thread.
__global__ void reduce_kernel(int64_t M, int64_t ldc, int splits, const float* __restrict__ part,
                              uint16_t* __restrict__ C) {
    const int64_t n8 = M * ldc / 8;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += (int64_t)gridDim.x * blockDim.x) {
        float acc[8];
        const float4* p0 = reinterpret_cast<const float4*>(part) + 2 * i;
        float4 a = p0[0], b = p0[1];
        acc[0] = a.x; acc[1] = a.y; acc[2] = a.z; acc[3] = a.w;
        acc[4] = b.x; acc[5] = b.y; acc[6] = b.z; acc[7] = b.w;
        for (int s = 1; s < splits; ++s) {
            const float4* ps = reinterpret_cast<const float4*>(part + (int64_t)s * M * ldc) + 2 * i;
            a = ps[0];
            b = ps[1];
            acc[0] += a.x; acc[1] += a.y; acc[2] += a.z; acc[3] += a.w;
            acc[4] += b.x; acc[5] += b.y; acc[6] += b.z; acc[7] += b.w;
        }
        uint4 pk;
        pk.x = pack_bf16x2(acc[0], acc[1]);
        pk.y = pack_bf16x2(acc[2], acc[3]);
        pk.z = pack_bf16x2(acc[4], acc[5]);
        pk.w = pack_bf16x2(acc[6], acc[7]);
        reinterpret_cast<uint4*>(C)[i] = pk;
    }
}

// q_out[t, h, 512 + d] = q_pe[t, h, d]: one 16-byte piece per thread.
__global__ void copy_rope_kernel(int64_t rows, const uint4* __restrict__ q_pe, uint16_t* __restrict__ q_out) {
    const int64_t n = rows * (kDRope * 2 / 16);
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = i / 8, p = i % 8;
        reinterpret_cast<uint4*>(q_out + r * kDQK + kDV)[p] = q_pe[i];
    }
}

// K splits of a GEMM whose output tiles fill few SMs: enough CTAs for about
// one wave, each with at least 8 k-tiles (fewer made the split-sum pass
// cost more than the extra CTAs saved: 64-token W_UV is not split, 64-token
// index-key products split 12 ways).  Depends only on the shape.
int choose_k_splits(int32_t M, int32_t N, int32_t K, int32_t batches) {
    const int64_t tiles = (int64_t)((M + kBM - 1) / kBM) * ((N + kBN - 1) / kBN) * batches;
    const int32_t nk = K / kBK;
    if (tiles == 0 || tiles * 2 > num_sms()) return 1;
    return (int)std::max<int64_t>(1, std::min<int64_t>(nk / 8, num_sms() / tiles));
}

template <bool kBMn>
cudaError_t launch_gemm(const CUtensorMap& tm_a, const CUtensorMap& tm_b, GemmArgs g, int32_t* status,
                        cudaStream_t stream) {
    g.tiles_m = (g.M + kBM - 1) / kBM;
    g.tiles_n = (g.N + kBN - 1) / kBN;
    if (g.splits < 1) g.splits = 1;
    const int64_t tiles = (int64_t)g.tiles_m * g.tiles_n * g.batches * g.splits;
    if (tiles == 0) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(gemm_bf16_kernel<kBMn>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kSmemBytes);
    if (e != cudaSuccess) return e;
    const int grid = (int)std::min<int64_t>(tiles, num_sms());
    gemm_bf16_kernel<kBMn><<<grid, kThreads, kSmemBytes, stream>>>(tm_a, tm_b, g, status);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    count_launches(1);
    if (g.splits == 1 || g.out_fp32) return cudaSuccess;
    const int64_t n8 = (int64_t)g.M * g.ldc / 8;
    const int blocks = (int)std::min<int64_t>((n8 + 255) / 256, 8 * num_sms());
    reduce_kernel<<<blocks, 256, 0, stream>>>(g.M, g.ldc, g.splits, g.part, g.C);
    e = cudaGetLastError();
    if (e == cudaSuccess) count_launches(1);
    return e;
}

}  // namespace

cudaError_t launch_gemm_f32_parts(const CUtensorMap& tm_a, const CUtensorMap& tm_b, int32_t M, int32_t N, int32_t K,
                                  int32_t splits, float* part, int32_t* status, cudaStream_t stream) {
    GemmArgs g{};
    g.M = M;
    g.N = N;
    g.K = K;
    g.batches = 1;
    g.ldc = N;
    g.splits = splits;
    g.part = part;
    g.out_fp32 = 1;
    return launch_gemm<false>(tm_a, tm_b, g, status, stream);
}

int gemm_k_splits(int32_t M, int32_t N, int32_t K) { return choose_k_splits(M, N, K, 1); }

// Split-K partials of dsa_mla_output for total_q rows (the W_UV and o_proj
// products run one after the other and share the buffer).
size_t mla_partial_bytes(int32_t total_q) {
    const size_t uv = (size_t)choose_k_splits(total_q, kDVh, kDV, kH) * total_q * kH * kDVh;
    const size_t op = (size_t)choose_k_splits(total_q, kHidden, kH * kDVh, 1) * total_q * kHidden;
    const size_t a = std::max(uv > (size_t)total_q * kH * kDVh ? uv : 0, op > (size_t)total_q * kHidden ? op : 0);
    return a * sizeof(float);
}

cudaError_t launch_mla_absorb_q(int32_t total_q, const uint16_t* q_nope, const uint16_t* q_pe,
                                const uint16_t* w_kvb, uint16_t* q_out, int32_t* status, cudaStream_t stream) {
    if (total_q <= 0) return cudaSuccess;
    CUtensorMap tm_a, tm_b;
    if (!make_tmap_bf16_2d(&tm_a, q_nope, (uint64_t)kH * kDNope, (uint64_t)total_q, kBK, kBM) ||
        !make_tmap_bf16_2d(&tm_b, w_kvb, kDV, (uint64_t)kH * kKvbRows, 64, kBK))
        return cudaErrorInvalidValue;
    GemmArgs g{};
    g.M = total_q;
    g.N = kDV;
    g.K = kDNope;
    g.batches = kH;
    g.a_col0 = 0;
    g.a_col_step = kDNope;
    g.b_row0 = 0;
    g.b_row_step = kKvbRows;
    g.C = q_out;
    g.ldc = (int64_t)kH * kDQK;
    g.c_col0 = 0;
    g.c_col_step = kDQK;
    g.splits = 1;                 // the rope columns of q_out are not the GEMM's: no split-K

    cudaError_t e = launch_gemm<true>(tm_a, tm_b, g, status, stream);
    if (e != cudaSuccess) return e;
    const int64_t pieces = (int64_t)total_q * kH * 8;
    const int blocks = (int)std::min<int64_t>((pieces + 255) / 256, 16 * num_sms());
    copy_rope_kernel<<<blocks, 256, 0, stream>>>((int64_t)total_q * kH, reinterpret_cast<const uint4*>(q_pe), q_out);
    e = cudaGetLastError();
    if (e == cudaSuccess) count_launches(1);
    return e;
}

cudaError_t launch_mla_output(int32_t total_q, const uint16_t* o_lat, const uint16_t* w_kvb, const uint16_t* w_o,
                              uint16_t* o_mid, uint16_t* y, float* part, int32_t* status, cudaStream_t stream) {
    if (total_q <= 0) return cudaSuccess;
    CUtensorMap tm_a, tm_b;
    // o_mid[:, h, :] = o_lat[:, h, :] . W_UV[h]^T
    if (!make_tmap_bf16_2d(&tm_a, o_lat, (uint64_t)kH * kDV, (uint64_t)total_q, kBK, kBM) ||
        !make_tmap_bf16_2d(&tm_b, w_kvb, kDV, (uint64_t)kH * kKvbRows, kBK, kBN))
        return cudaErrorInvalidValue;
    GemmArgs g{};
    g.M = total_q;
    g.N = kDVh;
    g.K = kDV;
    g.batches = kH;
    g.a_col0 = 0;
    g.a_col_step = kDV;
    g.b_row0 = kDNope;
    g.b_row_step = kKvbRows;
    g.C = o_mid;
    g.ldc = (int64_t)kH * kDVh;
    g.c_col0 = 0;
    g.c_col_step = kDVh;
    g.splits = choose_k_splits(g.M, g.N, g.K, g.batches);    // partials cover all of o_mid
    g.part = part;
    cudaError_t e = launch_gemm<false>(tm_a, tm_b, g, status, stream);
    if (e != cudaSuccess) return e;
    // y = o_mid . W_o^T
    if (!make_tmap_bf16_2d(&tm_a, o_mid, (uint64_t)kH * kDVh, (uint64_t)total_q, kBK, kBM) ||
        !make_tmap_bf16_2d(&tm_b, w_o, (uint64_t)kH * kDVh, kHidden, kBK, kBN))
        return cudaErrorInvalidValue;
    GemmArgs g2{};
    g2.M = total_q;
    g2.N = kHidden;
    g2.K = kH * kDVh;
    g2.batches = 1;
    g2.C = y;
    g2.ldc = kHidden;
    g2.splits = choose_k_splits(g2.M, g2.N, g2.K, 1);
    g2.part = part;
    return launch_gemm<false>(tm_a, tm_b, g2, status, stream);
}

}  // namespace dsa
