// sparse_mla.cu -- sparse MLA attention over the selected latent rows,
// absorbed form, on the 5th-generation tensor cores.
//
// For query row t and head h, over the selected positions s_j = idx[t, j]:
//   l_j   = sm_scale * q[t,h,:] . kv[s_j, :]          (576 = 512 latent + 64 rope)
//   out   = sum_j softmax_j(l) * kv[s_j, 0:512]
//   lse   = log sum_j exp(l_j)
// ("GLM-5.1 架构深度拆解", section 3.1 step 2 and section 4.2: the RoPE key
// is one stream shared by all heads; section 2.5: 576-wide cached rows; the
// GLM-5 explainer page: the top-2048 ids only drive the gather.)
//
// One CTA per (query row, segment of its selected list).  With only 64
// heads, a heads-as-M MMA would run at M = 64, half the tensor rate; so the
// products are taken transposed, with the 128 gathered rows of a block on
// the M = 128 side:
//   S^T[128 rows, 64 heads] = KV_blk[128, 576] . Q^T           (K-major A and B)
//   O^T[512, 64]           += V_blk^T[512, 128] . P^T[128, 64]  (MN-major A and B)
// V_blk is the first 512 columns of the same gathered tile, so every row is
// read from memory once.  Roles by warp:
//   warps 0, 1  producers: validate the block's indices and gather the
//               576-wide rows with 16-byte cp.async copies (8 lanes per
//               128-byte row piece, coalesced; 8 rows per instruction pair)
//               into nine 64-column chunks laid out 128B-swizzled.  When
//               the caches do not stay in L2, the rows of the next block are
//               prefetched into L2 (the first block's during the index
//               scan), so that a gather waits on L2 rather than on HBM
//   warp 2      TMEM owner; loads Q once by TMA; MMA issuer
//   warps 3..10 softmax: thread = one gathered row and 32 of the heads (two
//               warps per TMEM lane quarter).  The running per-head max m
//               only moves when some score exceeds it by more than 2^8 (a
//               vote over the block); only then is the exact block max
//               taken (warp max by redux.sync, then across lane quarters)
//               and O^T rescaled in TMEM.  p = 2^(s*c - m) in fp32, written
//               as bf16 P^T over the RoPE chunk (free once S^T is done);
//               final normalisation straight from TMEM into the output (or
//               a split's fp32 partial), one column per thread
// A single 144 KiB row tile fits next to Q (72 KiB); it is refilled chunk
// by chunk as soon as the MMAs that read each chunk have completed.
// Split-K partials (for few query rows): with 2 or 4 splits the CTAs of a
// row form a cluster; each rank merges a share of the heads from its own
// TMEM and the other ranks' weighted contributions, which arrive by one
// bulk copy per peer (no scratch memory).  More splits write fp32 partials
// that merge_kernel combines.
#include <cooperative_groups.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <type_traits>
#include <cmath>

#include "internal.h"
#include "ptx.cuh"

namespace cg = cooperative_groups;

namespace dsa {
namespace {

constexpr int kBlk = 128;                    // gathered rows per block (MMA M)
constexpr int kChunks = kDQK / 64;           // 9 column chunks of 64
constexpr int kVChunks = kDV / 64;           // the first 8 hold V
constexpr int kKVChunkBytes = kBlk * 128;    // 16 KiB
constexpr int kQChunkBytes = kH * 128;       // 8 KiB
#ifndef DSA_ATTN_PRODUCER_WARPS
#define DSA_ATTN_PRODUCER_WARPS 2
#endif
#ifndef DSA_ATTN_SOFTMAX_WARPS
#define DSA_ATTN_SOFTMAX_WARPS 8
#endif
constexpr int kProducerWarps = DSA_ATTN_PRODUCER_WARPS;

constexpr int kProducerRows = kBlk / (4 * kProducerWarps);   // rows of a block per producer lane
constexpr int kMmaWarp = kProducerWarps;                  // warp 2
constexpr int kSoftmaxWarp0 = kMmaWarp + 1;               // warps 3..10
constexpr int kSoftmaxWarps = DSA_ATTN_SOFTMAX_WARPS;     // two (or four) per TMEM lane quarter
constexpr int kHPT = kH * 4 / kSoftmaxWarps;              // heads per softmax thread: 32
constexpr int kSoftmaxThreads = 32 * kSoftmaxWarps;
constexpr int kThreads = 32 * kSoftmaxWarp0 + kSoftmaxThreads;   // 352
static_assert(kHPT == 16 || kHPT == 32, "the softmax loads S^T and O^T 16 or 32 columns at a time");

// kHPT TMEM columns of this thread's lane from taddr
__device__ __forceinline__ void tmem_ld_hpt(uint32_t taddr, uint32_t (&r)[32]) { tmem_ld_32x32b_x32(taddr, r); }
__device__ __forceinline__ void tmem_ld_hpt(uint32_t taddr, uint32_t (&r)[16]) { tmem_ld_32x32b_x16(taddr, r); }
constexpr int64_t kL2PrefetchBytes = int64_t(128) << 20;  // cache bytes above which rows are prefetched
constexpr int kPrefetchAhead = 1;                         // blocks prefetched ahead of the gather
constexpr int kMaxClusterMerge = 4;                       // most splits merged inside a cluster
constexpr float kRescaleLog2 = 8.0f;         // rescale O only when a max grows by > 2^8
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// shared memory layout (offsets from a 1024-aligned base)
constexpr int kOffKV = 0;
constexpr int kOffQ = kOffKV + kChunks * kKVChunkBytes;       // 147456
constexpr int kOffIdx = kOffQ + kChunks * kQChunkBytes;       // int32 [2][128]
constexpr int kOffWmax = kOffIdx + 2 * kBlk * 4;              // float [4][64]
constexpr int kOffM = kOffWmax + 4 * kH * 4;                  // float m_use[64]
constexpr int kOffAlpha = kOffM + kH * 4;                     // float alpha[64]
constexpr int kOffThr = kOffAlpha + kH * 4;                   // float thr[64]: the vote's bound in raw score units
constexpr int kOffL = kOffThr + kH * 4;                       // float [4][64], l_tot[64], 1 / l_tot[64], lse[64]
constexpr int kOffMisc = kOffL + 7 * kH * 4;                  // u32: tmem base, abort, rows staged
constexpr int kOffBar = kOffMisc + 16;
constexpr int kBarQ = 0;
constexpr int kBarKV = 1;                                     // [9]: chunk c landed
constexpr int kBarPair = kBarKV + kChunks;                    // [4]: chunks 2i, 2i+1 consumed
constexpr int kBarS = kBarPair + 4;                           // S^T ready
constexpr int kBarP = kBarS + 1;                              // P^T written (one arrival per softmax warp)
constexpr int kBarO = kBarP + 1;                              // PV of a block done (chunk 8 free)
constexpr int kBarIdx = kBarO + 1;                            // [2]: indices of a block published
constexpr int kBarDrain = kBarIdx + 2;
constexpr int kBarRecv = kBarDrain + 1;                       // cluster merge: the peers' contributions landed
constexpr int kNumBars = kBarRecv + 1;
constexpr int kSmemBytes = kOffBar + kNumBars * 8 + 1024;
static_assert(kSmemBytes <= 232448, "shared memory budget");
// epilogue staging tiles (one per softmax warp, 32 rows x 32 columns of
// fp32 at most) in the row tile, after the 64 KiB a cluster merge sends from
constexpr int kStageOff = 65536;
constexpr int kStageBytes = 32 * 32 * 4;
static_assert(kStageOff + kSoftmaxWarps * kStageBytes <= kChunks * kKVChunkBytes, "staging fits in the row tile");
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0;                                // O^T: 4 blocks x 64 columns
constexpr uint32_t kTmemS = 256;                              // S^T: 64 columns

// A warp's results for NX rows of a row-major destination, one column per
// lane (columns d0 .. d0 + 31 of row x at dst + x * row_stride): staged in
// the warp's own shared-memory tile, then written back with 16-byte stores
// (a 2-byte store per lane and row cost ~16 cycles per warp instruction).
// dst and row_stride keep every row 16-byte aligned.
template <typename T, int NX>
__device__ __forceinline__ void store_warp_tile(T* stage, const T (&v)[NX], T* dst, int64_t row_stride,
                                                uint32_t lane) {
#pragma unroll
    for (int x = 0; x < NX; ++x) stage[x * 32 + lane] = v[x];
    __syncwarp();
    constexpr int kVec = 16 / (int)sizeof(T);         // elements per 16 bytes
    constexpr int kPerRow = 32 / kVec;                // 16-byte pieces of a row's 32 columns
#pragma unroll
    for (int c = (int)lane; c < NX * kPerRow; c += 32) {
        const int x = c / kPerRow, q = c % kPerRow;
        *reinterpret_cast<uint4*>(dst + x * row_stride + q * kVec) =
            *reinterpret_cast<const uint4*>(stage + x * 32 + q * kVec);
    }
    __syncwarp();
}

__global__ void __launch_bounds__(kThreads, 1)
    sparse_mla_tc_kernel(const BatchDev bd, const RowRange rr, const __grid_constant__ CUtensorMap tm_q,
                         const uint16_t* __restrict__ kv, const int32_t* __restrict__ idx, const int idx_local,
                         const int k, const int rows_per_seq, const int splits, const int per_split,
                         const int l2_prefetch, const int cluster_merge, const float sm_scale,
                         uint16_t* __restrict__ out,
                         float* __restrict__ lse,
                         float* __restrict__ part_o, float* __restrict__ part_lse, int32_t* status) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    pdl_wait();                  // the indices of the previous launch are complete
    const int b = blockIdx.y;
    SeqInfo sq;
    if (!load_seq(bd, b, status, sq)) return;
    const int32_t i = rr.i0 + (int32_t)(blockIdx.x / splits);
    const int sp = (int)(blockIdx.x % splits);
    if (i >= min(rr.i1, sq.nq)) return;
    const int32_t t = sq.ctx - sq.nq + i;
    const int64_t grow = (int64_t)sq.q0 + i;
    const int32_t* sel = idx + buf_row(idx_local, sq, b, i, rr) * (int64_t)k;
    const int j_begin = sp * per_split;
    const int j_end = min(k, j_begin + per_split);
    const int64_t prow = ((int64_t)b * rows_per_seq + (i - rr.i0)) * splits + sp;   // split partial row

    const uint32_t sKV = smem_u32(smem + kOffKV);
    const uint32_t sQ = smem_u32(smem + kOffQ);
    int32_t* s_idx = reinterpret_cast<int32_t*>(smem + kOffIdx);
    float* s_wmax = reinterpret_cast<float*>(smem + kOffWmax);
    float* s_m = reinterpret_cast<float*>(smem + kOffM);
    float* s_alpha = reinterpret_cast<float*>(smem + kOffAlpha);
    float* s_thr = reinterpret_cast<float*>(smem + kOffThr);
    float* s_l = reinterpret_cast<float*>(smem + kOffL);
    volatile uint32_t* misc = reinterpret_cast<volatile uint32_t*>(smem + kOffMisc);
    const uint32_t bar0 = smem_u32(smem + kOffBar);
    auto bar = [&](int n) { return bar0 + 8u * (uint32_t)n; };
    const uint32_t warp = warp_id(), lane = lane_id();

    // blocks of this segment: up to its last valid entry.  Every thread
    // scans a few entries (16-byte loads when the rows are 16-byte aligned),
    // so the scan costs one memory round trip; the per-warp maxima meet in
    // shared memory (the block-max scratch, unused until the first block).
    // With L2 prefetching on, the rows of the first kPrefetchAhead blocks
    // are prefetched as their indices are seen.
    const uint8_t* kv_seq = reinterpret_cast<const uint8_t*>(kv) + (int64_t)b * bd.stride * (kDQK * 2);
    auto prefetch_row = [&](int j, int32_t sv) {
        if (l2_prefetch && j < j_begin + kPrefetchAhead * kBlk && sv >= 0 && sv <= t)
            prefetch_l2_bulk(kv_seq + (int64_t)sv * (kDQK * 2), kDQK * 2);
    };
    {
        int last = -1;
        if ((k & 3) == 0) {
            const int4* sel4 = reinterpret_cast<const int4*>(sel + j_begin);   // j_begin is a multiple of 128
            for (int q = (int)threadIdx.x; q < (j_end - j_begin) >> 2; q += kThreads) {
                const int4 v = __ldg(sel4 + q);
                const int j = j_begin + 4 * q;
                if (v.x >= 0) last = j;
                if (v.y >= 0) last = j + 1;
                if (v.z >= 0) last = j + 2;
                if (v.w >= 0) last = j + 3;
                prefetch_row(j, v.x);
                prefetch_row(j + 1, v.y);
                prefetch_row(j + 2, v.z);
                prefetch_row(j + 3, v.w);
            }
        } else {
            for (int j = j_begin + (int)threadIdx.x; j < j_end; j += kThreads) {
                const int32_t sv = __ldg(sel + j);
                if (sv >= 0) last = j;
                prefetch_row(j, sv);
            }
        }
        last = __reduce_max_sync(0xffffffffu, last);
        if (lane == 0) reinterpret_cast<int*>(s_wmax)[warp] = last;
    }
    if (threadIdx.x == 32 * kMmaWarp) prefetch_tmap(&tm_q);
    if (threadIdx.x == 0) {
        for (int n = 0; n < kNumBars; ++n) mbar_init(bar(n), 1);
        mbar_init(bar(kBarP), kSoftmaxThreads / 32);
        mbar_init(bar(kBarIdx), 1);
        mbar_init(bar(kBarIdx + 1), 1);
        // a row merged in a cluster receives, from every other split, its
        // contribution to the heads this CTA merges (bf16, kH / splits heads)
        if (cluster_merge)
            mbar_arrive_expect_tx(bar(kBarRecv), (uint32_t)((splits - 1) * (kH / splits) * kDV * 2));
        for (int c = 0; c < kChunks; ++c) mbar_init(bar(kBarKV + c), 32 * kProducerWarps);
        misc[1] = 0;
        misc[2] = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_u32(smem + kOffMisc), kTmemCols);
        tmem_relinquish();
    }
    if (threadIdx.x >= 32 * kSoftmaxWarp0 && threadIdx.x < 32 * kSoftmaxWarp0 + kH) {
        s_m[threadIdx.x - 32 * kSoftmaxWarp0] = -INFINITY;
        s_thr[threadIdx.x - 32 * kSoftmaxWarp0] = -INFINITY;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];
    int nblk;
    {
        int last = -1;
        for (int w = 0; w < kThreads / 32; ++w) last = max(last, reinterpret_cast<const int*>(s_wmax)[w]);
        nblk = last < j_begin ? 0 : (last - j_begin) / kBlk + 1;
    }
    named_bar_sync(6, kThreads);     // every thread has read the maxima before the block-max scratch is reused
    const float c2 = sm_scale * kLog2e;      // logits in log2 units

    if (warp < kProducerWarps) {
        // ----------------------------------------------------------- producers
        // producer lane gl = (rq, piece): rows 16n + rq of the block, 16-byte
        // piece `piece` of each 128-byte row chunk; 8 lanes cover one row
        // chunk (coalesced) and row r % 8 == rq % 8 fixes the swizzle
        const int gl = (int)threadIdx.x;
        const int rq = gl >> 3, piece = gl & 7;
        const uint32_t dpat = (uint32_t)(rq * 128 + ((piece ^ (rq & 7)) << 4));
        bool ok = true;
        for (int jb = 0; jb < nblk; ++jb) {
            const uint32_t ph = (uint32_t)jb & 1u;
            int32_t* ib = s_idx + (jb & 1) * kBlk;
            // this block's indices (warp 0) are loaded before the prefetch
            // below, so that the two round trips overlap
            int32_t v[4];
            if (warp == 0) {
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int j = j_begin + jb * kBlk + u * 32 + (int)lane;
                    v[u] = (j < j_end) ? __ldg(sel + j) : -1;
                }
            }
            if (l2_prefetch && jb + kPrefetchAhead < nblk) {
                // the rows of block jb + kPrefetchAhead (valid indices only),
                // one 1152-byte bulk prefetch each
                for (int u = gl; u < kBlk; u += 32 * kProducerWarps) {
                    const int j = j_begin + (jb + kPrefetchAhead) * kBlk + u;
                    const int32_t sv = j < j_end ? __ldg(sel + j) : -1;
                    if (sv >= 0 && sv <= t) prefetch_l2_bulk(kv_seq + (int64_t)sv * (kDQK * 2), kDQK * 2);
                }
            }
            if (warp == 0) {
                // indices of this block: validated, -1 where invalid or past the segment
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    if (v[u] < -1 || v[u] > t) {
                        latch_status(status, DSA_ERR_BAD_INDEX);
                        v[u] = -1;
                    }
                }
                // buffer jb & 1 was last read by the softmax of block jb - 2,
                // which finished before PV(jb - 2) started; these warps have
                // already waited for PV(jb - 2) to complete (before refilling
                // chunk 8 in block jb - 1), so the buffer is free and the
                // block's indices and row offsets are ready before PV(jb - 1)
                ok = __all_sync(0xffffffffu, !misc[1]);
                if (ok) {
#pragma unroll
                    for (int u = 0; u < 4; ++u) ib[u * 32 + lane] = v[u];
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(kBarIdx + (jb & 1)));
                } else {
                    misc[1] = 1;
                }
            }
            named_bar_sync(4, 32 * kProducerWarps);     // the block's indices are in shared memory
            if (misc[1]) {
                ok = false;
                break;
            }
            uint32_t soff[kProducerRows];   // byte offset of each of this lane's rows (+ piece)
#pragma unroll
            for (int n = 0; n < kProducerRows; ++n) {
                const int32_t sv = ib[4 * kProducerWarps * n + rq];
                soff[n] = (uint32_t)(sv >= 0 ? sv : 0) * (uint32_t)(kDQK * 2) + (uint32_t)(piece * 16);
            }
            for (int c = 0; c < kChunks; ++c) {
                // chunk c of the previous block must have been consumed: chunks
                // 2i and 2i + 1 are freed together (one wait per pair)
                if (jb > 0 && (c == kVChunks || (c & 1) == 0)) {
                    const uint32_t fb = c < kVChunks ? bar(kBarPair + c / 2) : bar(kBarO);
                    ok = mbar_wait(fb, ph ^ 1u);
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) break;
                }
                const uint8_t* src = kv_seq + c * 128;
                const uint32_t dst = sKV + c * kKVChunkBytes + dpat;
#pragma unroll
                for (int n = 0; n < kProducerRows; ++n)
                    cp_async_16(dst + (uint32_t)(512 * kProducerWarps) * n, src + soff[n]);
                cp_async_arrive(bar(kBarKV + c));
            }
            // both producer warps agree before either starts the next block
            if (named_bar_or(5, 32 * kProducerWarps, !ok)) {
                ok = false;
                misc[1] = 1;
                break;
            }
        }
        if (!ok) latch_status(status, DSA_ERR_TIMEOUT);
        if (misc[1]) {
            // wind down: let every copy this warp started land first
            asm volatile("cp.async.wait_all;" ::: "memory");
        }
        __syncwarp();
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------- MMA
        if (elect_one()) {
            constexpr uint32_t idesc_s = idesc_bf16_f32(kBlk, kH, false, false);
            constexpr uint32_t idesc_o = idesc_bf16_f32(kBlk, kH, true, true);
            // Q by TMA (this warp is idle until it lands; the producers go
            // straight to the first block's indices)
            if (nblk > 0) {
                mbar_arrive_expect_tx(bar(kBarQ), kChunks * kQChunkBytes);
                for (int c = 0; c < kChunks; ++c)
                    tma_load_2d(sQ + c * kQChunkBytes, &tm_q, bar(kBarQ), c * 64, (int32_t)(grow * kH));
            }
            bool ok = nblk == 0 || mbar_wait(bar(kBarQ), 0);
            const bool q_landed = ok;
            tc_fence_after();
            for (int jb = 0; ok && jb < nblk; ++jb) {
                const uint32_t ph = (uint32_t)jb & 1u;
                // S^T = KV_blk . Q^T over the 9 chunks of 64 columns
                for (int c = 0; c < kChunks; ++c) {
                    if (misc[1] || !mbar_wait(bar(kBarKV + c), ph)) {
                        ok = false;
                        break;
                    }
                    fence_proxy_async_smem();      // cp.async data -> tensor-core reads
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t ad = sdesc_sw128(sKV + c * kKVChunkBytes + kk * 32, 16, 1024);
                        const uint64_t bdsc = sdesc_sw128(sQ + c * kQChunkBytes + kk * 32, 16, 1024);
                        mma_bf16_ss(tmem + kTmemS, ad, bdsc, idesc_s, (c | kk) != 0);
                    }
                }
                if (!ok) break;
                mma_commit(bar(kBarS));
                // O^T += V^T . P^T once the softmax has written P^T
                if (misc[1] || !mbar_wait(bar(kBarP), ph)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t sP = sKV + kVChunks * kKVChunkBytes;
                for (int dv = 0; dv < 4; ++dv) {
#pragma unroll
                    for (int kk = 0; kk < kBlk / 16; ++kk) {
                        const uint64_t ad =
                            sdesc_sw128(sKV + (2 * dv) * kKVChunkBytes + kk * 2048, kKVChunkBytes, 1024);
                        const uint64_t bdsc = sdesc_sw128(sP + kk * 2048, 1024, 1024);
                        mma_bf16_ss(tmem + kTmemO + dv * kH, ad, bdsc, idesc_o, (jb | kk) != 0);
                    }
                    mma_commit(bar(kBarPair + dv));
                }
                mma_commit(bar(kBarO));
            }
            if (!ok) {
                latch_status(status, DSA_ERR_TIMEOUT);
                misc[1] = 1;
            }
            // every MMA this thread issued has finished once drain completes
            mma_commit(bar(kBarDrain));
            mbar_wait(bar(kBarDrain), 0);
            if (!q_landed) mbar_wait(bar(kBarQ), 0);    // Q's copy must land before the CTA exits
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------- softmax
        // warp w: TMEM lane quarter w % 4 (rows), head group (w - 5) / 4 of
        // kHPT heads
        const uint32_t lq = warp & 3u;
        const int h0 = ((int)(warp - kSoftmaxWarp0) >> 2) * kHPT;
        const int r = (int)(lq * 32 + lane);           // row of the block
        const int st = (int)threadIdx.x - 32 * kSoftmaxWarp0;   // 0..511 among the softmax threads
        const uint32_t lane_base = (lq * 32u) << 16;
        float lsum[kHPT];
#pragma unroll
        for (int x = 0; x < kHPT; ++x) lsum[x] = 0.f;
        bool ok = true;
        for (int jb = 0; jb < nblk; ++jb) {
            const uint32_t ph = (uint32_t)jb & 1u;
            const bool got = !misc[1] && mbar_wait(bar(kBarIdx + (jb & 1)), ((uint32_t)jb >> 1) & 1u) &&
                             mbar_wait(bar(kBarS), ph);
            tc_fence_after();
            const bool valid = s_idx[(jb & 1) * kBlk + r] >= 0;
            // the running max moves only when a score exceeds it by 2^8; the
            // vote compares raw scores with (m + 8) / c2 per head (a trigger
            // only: the exact block max below decides whether m moves).  The
            // bounds are read while the TMEM load is in flight.
            float s[kHPT];
            bool exceed = false;
            {
                uint32_t u[kHPT];
                tmem_ld_hpt(tmem + lane_base + kTmemS + h0, u);
                float4 tv[kHPT / 4];
#pragma unroll
                for (int x = 0; x < kHPT; x += 4) tv[x / 4] = *reinterpret_cast<const float4*>(s_thr + h0 + x);
                tmem_ld_wait();
#pragma unroll
                for (int x = 0; x < kHPT; ++x) s[x] = valid ? __uint_as_float(u[x]) : -INFINITY;
#pragma unroll
                for (int x = 0; x < kHPT; x += 4) {
                    exceed |= s[x] > tv[x / 4].x;
                    exceed |= s[x + 1] > tv[x / 4].y;
                    exceed |= s[x + 2] > tv[x / 4].z;
                    exceed |= s[x + 3] > tv[x / 4].w;
                }
            }
            // a thread whose wait failed (abort or time-out) joins the vote
            // with the slow path, where every softmax thread learns of it
            // after the same barrier and all stop together: no named barrier
            // is ever left waiting
            if (named_bar_or(2, kSoftmaxThreads, exceed || !got)) {
                volatile int* s_abort = reinterpret_cast<volatile int*>(s_l);   // [softmax warp], unused until the epilogue
                const bool wabort = __any_sync(0xffffffffu, !got);
                if (lane == 0) s_abort[warp - kSoftmaxWarp0] = wabort ? 1 : 0;
                // exact per-head block max: warp max, then across lane quarters
#pragma unroll
                for (int x = 0; x < kHPT; ++x) {
                    const float mx = warp_max_f32(s[x]);
                    if (lane == 0) s_wmax[lq * kH + h0 + x] = mx;
                }
                named_bar_sync(1, kSoftmaxThreads);
                bool any_abort = false;
#pragma unroll
                for (int w2 = 0; w2 < kSoftmaxWarps; ++w2) any_abort |= s_abort[w2] != 0;
                if (any_abort) {
                    ok = false;
                    break;
                }
                bool need = false;
                if (st < kH) {
                    const float mb = fmaxf(fmaxf(s_wmax[st], s_wmax[kH + st]),
                                           fmaxf(s_wmax[2 * kH + st], s_wmax[3 * kH + st]));
                    const float mold = s_m[st];
                    const float mnew = mb * c2;
                    float alpha = 1.f;
                    if (mb > -INFINITY && (mold == -INFINITY || mnew > mold + kRescaleLog2)) {
                        alpha = exp2f(mold - mnew);          // 0 when nothing was seen yet
                        s_m[st] = mnew;
                        s_thr[st] = (mnew + kRescaleLog2) / c2;
                        need = true;
                    }
                    s_alpha[st] = alpha;
                }
                if (named_bar_or(2, kSoftmaxThreads, need)) {
                    // O^T holds the blocks before jb once PV(jb - 1) has completed
                    const bool w = jb == 0 || mbar_wait(bar(kBarO), ph ^ 1u);
                    if (named_bar_or(3, kSoftmaxThreads, !w)) {
                        ok = false;
                        break;
                    }
                    if (jb > 0) {
                        tc_fence_after();
#pragma unroll 1
                        for (int piece = 0; piece < 4 * (kHPT / 16); ++piece) {   // 4 dv blocks x kHPT heads
                            uint32_t u[16];
                            const int hx = (piece % (kHPT / 16)) * 16;
                            const uint32_t ta = tmem + lane_base + kTmemO + (piece / (kHPT / 16)) * kH + h0 + hx;
                            tmem_ld_32x32b_x16(ta, u);
                            tmem_ld_wait();
#pragma unroll
                            for (int x = 0; x < 16; ++x)
                                u[x] = __float_as_uint(__uint_as_float(u[x]) * s_alpha[h0 + hx + x]);
                            tmem_st_32x32b_x16(ta, u);
                        }
                        tmem_st_wait();
                    }
#pragma unroll
                    for (int x = 0; x < kHPT; ++x) lsum[x] *= s_alpha[h0 + x];
                }
            }
            // P^T row r, heads h0..h0+15: 2 swizzled 16-byte pieces (MN-major B)
            uint8_t* p_row = smem + kOffKV + kVChunks * kKVChunkBytes + r * 128;
#pragma unroll
            for (int e4 = 0; e4 < kHPT / 8; ++e4) {
                const float4 ma = *reinterpret_cast<const float4*>(s_m + h0 + e4 * 8);
                const float4 mb = *reinterpret_cast<const float4*>(s_m + h0 + e4 * 8 + 4);
                const float mm[8] = {ma.x, ma.y, ma.z, ma.w, mb.x, mb.y, mb.z, mb.w};
                float p[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int x = e4 * 8 + e;
                    p[e] = valid ? ex2_approx(fmaf(s[x], c2, -mm[e])) : 0.f;
                    lsum[x] += p[e];
                }
                uint4 pk;
                pk.x = pack_bf16x2(p[0], p[1]);
                pk.y = pack_bf16x2(p[2], p[3]);
                pk.z = pack_bf16x2(p[4], p[5]);
                pk.w = pack_bf16x2(p[6], p[7]);
                const int c8 = (h0 >> 3) + e4;
                *reinterpret_cast<uint4*>(p_row + ((c8 ^ (r & 7)) << 4)) = pk;
            }
            // one arrival per warp once all its lanes' P^T writes are fenced
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(kBarP));
        }
        if (!ok) {
            latch_status(status, DSA_ERR_TIMEOUT);
            misc[1] = 1;
        }
        // ------------------------------------------------------- epilogue
        // l: the per-thread partial sums reduced over the 128 rows
#pragma unroll
        for (int x = 0; x < kHPT; ++x) {
            float v = lsum[x];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
            if (lane == 0) s_l[lq * kH + h0 + x] = v;
        }
        const bool got_o = ok && (nblk == 0 || mbar_wait(bar(kBarO), ((uint32_t)nblk - 1u) & 1u));
        // agreed by every softmax thread: the staging below has a named barrier
        const bool w = !named_bar_or(3, kSoftmaxThreads, !got_o);
        if (st < kH) {
            const float lt = s_l[st] + s_l[kH + st] + s_l[2 * kH + st] + s_l[3 * kH + st];
            s_l[4 * kH + st] = lt;
            s_l[5 * kH + st] = lt > 0.f ? 1.f / lt : 0.f;
            const float ls = lt > 0.f ? (s_m[st] + log2f(lt)) * kLn2 : -INFINITY;
            if (splits == 1) {
                if (lse) lse[grow * kH + st] = ls;
            } else if (cluster_merge) {
                s_l[6 * kH + st] = ls;
            } else {
                part_lse[prow * kH + st] = ls;
            }
        }
        named_bar_sync(1, kSoftmaxThreads);
        if (w && !cluster_merge) {
            // every MMA has completed (PV of the last block): each thread
            // stores its output column d of its heads straight from TMEM
            // (per head a warp writes 32 consecutive columns: 64 bytes of
            // bf16 output or 128 bytes of an fp32 split partial)
            tc_fence_after();
            float inv[kHPT];                                  // 1 / l of this thread's heads
#pragma unroll
            for (int x = 0; x < kHPT; x += 4) {
                const float4 v = *reinterpret_cast<const float4*>(s_l + 5 * kH + h0 + x);
                inv[x] = v.x;
                inv[x + 1] = v.y;
                inv[x + 2] = v.z;
                inv[x + 3] = v.w;
            }
            // the warp's staging tile: the row tile is free once every PV is done
            uint8_t* stage = smem + kOffKV + kStageOff + (warp - kSoftmaxWarp0) * kStageBytes;
            for (int dv = 0; dv < 4; ++dv) {
                const int d0 = dv * 128 + (int)(lq * 32);      // the warp's 32 output columns
                uint32_t u[kHPT];
                if (nblk > 0) {
                    tmem_ld_hpt(tmem + lane_base + kTmemO + dv * kH + h0, u);
                    tmem_ld_wait();
                } else {
#pragma unroll
                    for (int x = 0; x < kHPT; ++x) u[x] = 0u;
                }
                if (splits == 1) {
                    uint16_t o16[kHPT];
#pragma unroll
                    for (int x = 0; x < kHPT; ++x) {
                        const __nv_bfloat16 b16 = __float2bfloat16_rn(__uint_as_float(u[x]) * inv[x]);
                        o16[x] = *reinterpret_cast<const uint16_t*>(&b16);
                    }
                    store_warp_tile(reinterpret_cast<uint16_t*>(stage), o16, out + (grow * kH + h0) * kDV + d0,
                                    kDV, lane);
                } else {
                    float o32[kHPT];
#pragma unroll
                    for (int x = 0; x < kHPT; ++x) o32[x] = __uint_as_float(u[x]) * inv[x];
                    store_warp_tile(reinterpret_cast<float*>(stage), o32, part_o + (prow * kH + h0) * kDV + d0,
                                    kDV, lane);
                }
            }
        }
    }

    if (cluster_merge) {
        // The row's splits are the CTAs of this cluster, rank = split; rank
        // sp merges the heads h = sp (mod splits):
        //   out[h] = sum_s f_s[h] o_s[h],  f_s = exp(lse_s - m) / sum_s' exp(lse_s' - m),
        // o_s the split's normalised output, m = max_s lse_s, summed in split
        // order.  Distributed shared memory moves ~14 bytes per clock, so
        // only the lse values and, for each peer, its heads of this split's
        // weighted contribution f_s o_s in bf16 cross the cluster (one bulk
        // copy per peer into its then free Q region); a CTA's own term is
        // taken in fp32 straight from TMEM.
        cg::cluster_group cluster = cg::this_cluster();
        cluster.sync();                      // every split's lse is staged, its Q region free
        if (warp >= kSoftmaxWarp0) {
            const int st = (int)threadIdx.x - 32 * kSoftmaxWarp0;
            const uint32_t lq = warp & 3u;
            const int h0 = ((int)(warp - kSoftmaxWarp0) >> 2) * kHPT;
            const int r = (int)(lq * 32 + lane);
            const uint32_t lane_base = (lq * 32u) << 16;
            float* s_g = s_wmax;                              // g[h] = f_sp[h] / l[h] (free by now)
            if (st < kH) {
                const int h = st;
                float ls[kMaxClusterMerge];
                float mx = -INFINITY;
#pragma unroll
                for (int s2 = 0; s2 < kMaxClusterMerge; ++s2) {
                    ls[s2] = s2 < splits ? *cluster.map_shared_rank(s_l + 6 * kH + h, (unsigned)s2) : -INFINITY;
                    mx = fmaxf(mx, ls[s2]);
                }
                float wsum = 0.f;
#pragma unroll
                for (int s2 = 0; s2 < kMaxClusterMerge; ++s2)
                    if (mx > -INFINITY && s2 < splits && ls[s2] != -INFINITY) wsum += expf(ls[s2] - mx);
                const float f = wsum > 0.f && ls[sp] != -INFINITY ? expf(ls[sp] - mx) / wsum : 0.f;
                s_g[h] = f * s_l[5 * kH + h];
                if (lse && h % splits == sp) lse[grow * kH + h] = wsum > 0.f ? mx + logf(wsum) : -INFINITY;
            }
            named_bar_sync(1, kSoftmaxThreads);
            // the head arithmetic below is specialised on the split count
            // (2 or 4, a divisor of the 32 heads of a thread), so it folds
            auto merge_heads = [&](auto splits_c) {
                constexpr int S = decltype(splits_c)::value;
                constexpr int hsS = kH / S;
                constexpr uint32_t slotS = (uint32_t)(hsS * kDV * 2);
                // this split's contribution to every other rank's heads, bf16,
                // rank q's heads h = q + S k at [q][k][d] in the (free) row tile
                tc_fence_after();
                uint16_t* send = reinterpret_cast<uint16_t*>(smem + kOffKV);
                for (int dv = 0; dv < 4; ++dv) {
                    const int d = dv * 128 + r;
                    uint32_t u[kHPT];
                    if (nblk > 0) {
                        tmem_ld_hpt(tmem + lane_base + kTmemO + dv * kH + h0, u);
                        tmem_ld_wait();
                    } else {
#pragma unroll
                        for (int x = 0; x < kHPT; ++x) u[x] = 0u;
                    }
#pragma unroll
                    for (int x = 0; x < kHPT; ++x) {
                        const int q = x % S;                   // h0 is a multiple of kHPT
                        if (q == sp) continue;
                        const int h = h0 + x;
                        const __nv_bfloat16 b16 = __float2bfloat16_rn(__uint_as_float(u[x]) * s_g[h]);
                        send[(q * hsS + h0 / S + x / S) * kDV + d] = *reinterpret_cast<const uint16_t*>(&b16);
                    }
                }
                fence_proxy_async_smem();    // the generic-proxy stores, before the bulk copies read them
                named_bar_sync(1, kSoftmaxThreads);
                if (st == 0) {
                    for (int q = 0; q < S; ++q) {
                        if (q == sp) continue;
                        const uint32_t dst =
                            map_to_cluster_rank(smem_u32(smem + kOffQ) + (uint32_t)sp * slotS, (uint32_t)q);
                        bulk_copy_to_peer(dst, smem_u32(smem + kOffKV) + (uint32_t)q * slotS, slotS,
                                          map_to_cluster_rank(bar(kBarRecv), (uint32_t)q));
                    }
                }
                // every other split's contribution to this rank's heads
                const bool got = !named_bar_or(3, kSoftmaxThreads, !mbar_wait(bar(kBarRecv), 0));
                if (!got) {
                    latch_status(status, DSA_ERR_TIMEOUT);
                    return;
                }
                const uint16_t* recv = reinterpret_cast<const uint16_t*>(smem + kOffQ);
                tc_fence_after();
                uint16_t* stage =
                    reinterpret_cast<uint16_t*>(smem + kOffKV + kStageOff + (warp - kSoftmaxWarp0) * kStageBytes);
                for (int dv = 0; dv < 4; ++dv) {
                    const int d = dv * 128 + r;
                    uint32_t u[kHPT];
                    if (nblk > 0) {
                        tmem_ld_hpt(tmem + lane_base + kTmemO + dv * kH + h0, u);
                        tmem_ld_wait();
                    } else {
#pragma unroll
                        for (int x = 0; x < kHPT; ++x) u[x] = 0u;
                    }
                    // this rank's heads of the thread: x = sp + S j
                    uint16_t o16[kHPT / S];
#pragma unroll
                    for (int j = 0; j < kHPT / S; ++j) {
                        const int h = h0 + sp + S * j;
                        const int k = h0 / S + j;
                        // u[sp + S j] with sp < S chosen by selects (no local-memory indexing)
                        uint32_t uv = u[S * j];
#pragma unroll
                        for (int q = 1; q < S; ++q)
                            if (sp == q) uv = u[S * j + q];
                        float acc = 0.f;
#pragma unroll
                        for (int s2 = 0; s2 < S; ++s2) {
                            const float c = s2 == sp ? __uint_as_float(uv) * s_g[h]
                                                     : __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(
                                                           recv + (s2 * hsS + k) * kDV + d));
                            acc += c;
                        }
                        const __nv_bfloat16 b16 = __float2bfloat16_rn(acc);
                        o16[j] = *reinterpret_cast<const uint16_t*>(&b16);
                    }
                    store_warp_tile(stage, o16, out + (grow * kH + h0 + sp) * kDV + dv * 128 + (int)(lq * 32),
                                    (int64_t)S * kDV, lane);
                }
            };
            if (splits == 2) merge_heads(std::integral_constant<int, 2>{});
            else merge_heads(std::integral_constant<int, 4>{});
        }
        // a CTA's row tile is the source of its bulk copies and its Q region
        // their destination: none exits before every copy has landed
        cluster.sync();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// out = sum_s exp(lse_s - L) * o_s, L = log sum_s exp(lse_s).  One CTA per
// (query row, 8 heads); warp = head, lane = 16 output columns.
__global__ void __launch_bounds__(256)
    merge_kernel(const BatchDev bd, const RowRange rr, const int rows_per_seq, const int splits,
                 const float* __restrict__ part_o, const float* __restrict__ part_lse, uint16_t* __restrict__ out,
                 float* __restrict__ lse, int32_t* status) {
    const int b = blockIdx.y;
    SeqInfo sq;
    if (!load_seq(bd, b, status, sq)) return;
    const int32_t i = rr.i0 + (int32_t)(blockIdx.x >> 3);
    if (i >= min(rr.i1, sq.nq)) return;
    const int64_t grow = (int64_t)sq.q0 + i;
    const int64_t prow0 = ((int64_t)b * rows_per_seq + (i - rr.i0)) * splits;
    const int h = (int)(blockIdx.x & 7) * 8 + (int)(threadIdx.x >> 5);
    const int c0 = (int)(threadIdx.x & 31) * 16;
    float mx = -INFINITY;
    for (int s = 0; s < splits; ++s) mx = fmaxf(mx, part_lse[(prow0 + s) * kH + h]);
    float wsum = 0.f;
    float acc[16];
#pragma unroll
    for (int c = 0; c < 16; ++c) acc[c] = 0.f;
    if (mx > -INFINITY) {
        for (int s = 0; s < splits; ++s) {
            const float ls = part_lse[(prow0 + s) * kH + h];
            if (ls == -INFINITY) continue;
            const float wgt = expf(ls - mx);
            wsum += wgt;
            const float4* o = reinterpret_cast<const float4*>(part_o + ((prow0 + s) * kH + h) * kDV + c0);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const float4 v = o[c];
                acc[4 * c] = fmaf(wgt, v.x, acc[4 * c]);
                acc[4 * c + 1] = fmaf(wgt, v.y, acc[4 * c + 1]);
                acc[4 * c + 2] = fmaf(wgt, v.z, acc[4 * c + 2]);
                acc[4 * c + 3] = fmaf(wgt, v.w, acc[4 * c + 3]);
            }
        }
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    uint4* o = reinterpret_cast<uint4*>(out + (grow * kH + h) * kDV + c0);
#pragma unroll
    for (int c = 0; c < 2; ++c) {
        uint4 pk;
        pk.x = pack_bf16x2(acc[8 * c] * inv, acc[8 * c + 1] * inv);
        pk.y = pack_bf16x2(acc[8 * c + 2] * inv, acc[8 * c + 3] * inv);
        pk.z = pack_bf16x2(acc[8 * c + 4] * inv, acc[8 * c + 5] * inv);
        pk.w = pack_bf16x2(acc[8 * c + 6] * inv, acc[8 * c + 7] * inv);
        o[c] = pk;
    }
    if (lse && (threadIdx.x & 31) == 0) lse[grow * kH + h] = wsum > 0.f ? mx + logf(wsum) : -INFINITY;
}

// CTAs per query row.  One CTA fills an SM's shared memory, so the grid
// runs in waves of num_sms() CTAs; pick the split count that minimises
// waves x (blocks per CTA + one block's worth of per-CTA overhead).
int choose_splits(int64_t rows, int k) {
    if (rows <= 0) return 1;
    const int nblk = std::max(1, (k + kBlk - 1) / kBlk);
    const int64_t nsm = num_sms();
    int best = 1;
    int64_t best_cost = -1;
    for (int sp = 1; sp <= std::min(16, nblk); ++sp) {
        const int64_t waves = (rows * sp + nsm - 1) / nsm;
        const int64_t cost = waves * ((nblk + sp - 1) / sp + 1);
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best = sp;
        }
    }
    return best;
}

// Splits merged inside a cluster: the count divides the heads and is small
// enough that a cluster of that many one-SM CTAs always fits in a GPC.
bool merge_in_cluster(int splits) { return splits > 1 && splits <= kMaxClusterMerge && kH % splits == 0; }

}  // namespace

// The split count depends only on the batch bounds, never on how many rows
// one launch covers, so a row's arithmetic is the same in every call.
size_t sparse_mla_scratch_bytes(const BatchDev& bd, int64_t rows_per_seq, int k) {
    const int64_t rows = rows_per_seq * bd.B;
    const int splits = choose_splits((int64_t)bd.B * bd.max_q, k);
    if (splits <= 1 || merge_in_cluster(splits)) return 0;
    return (size_t)rows * splits * kH * (kDV + 1) * sizeof(float);
}

cudaError_t launch_sparse_mla(const BatchDev& bd, RowRange rr, const uint16_t* q, const uint16_t* kv,
                              const int32_t* idx, bool idx_local, int k, float sm_scale, uint16_t* out,
                              float* lse, void* scratch, size_t scratch_bytes, int32_t* status,
                              cudaStream_t stream, bool after_previous) {
    const int32_t rows_per_seq = min(rr.i1, bd.max_q) - rr.i0;
    if (rows_per_seq <= 0) return cudaSuccess;
    const int64_t rows = (int64_t)rows_per_seq * bd.B;
    const int splits = choose_splits((int64_t)bd.B * bd.max_q, k);
    const int per_split = ((k + splits - 1) / splits + kBlk - 1) / kBlk * kBlk;
    const bool cluster_merge = merge_in_cluster(splits);
    float* part_o = nullptr;
    float* part_lse = nullptr;
    if (splits > 1 && !cluster_merge) {
        const size_t need = sparse_mla_scratch_bytes(bd, rows_per_seq, k);
        if (!scratch || scratch_bytes < need) return cudaErrorInvalidValue;
        part_o = static_cast<float*>(scratch);
        part_lse = part_o + (size_t)rows * splits * kH * kDV;
    }
    CUtensorMap tm_q;
    if (!make_tmap_bf16_2d(&tm_q, q, kDQK, (uint64_t)bd.total_q * kH, 64, kH)) return cudaErrorInvalidValue;
    cudaError_t e =
        cudaFuncSetAttribute(sparse_mla_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    // caches larger than a fraction of L2 are read from HBM: prefetch one
    // block ahead (a cache that stays L2-resident gains nothing from it, and
    // a CTA of a single block only duplicates its own gather: 8 x 202,752
    // decode, 16 splits of one block, 28.6 -> 26.9 us without)
    const int l2_prefetch =
        (int64_t)bd.B * bd.max_ctx * (kDQK * 2) > kL2PrefetchBytes && per_split > kBlk ? 1 : 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(rows_per_seq * splits), (unsigned)bd.B);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cluster_merge ? (unsigned)splits : 1u;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = after_previous ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    e = cudaLaunchKernelEx(&cfg, sparse_mla_tc_kernel, bd, rr, tm_q, kv, idx, idx_local ? 1 : 0, k, rows_per_seq,
                           splits, per_split, l2_prefetch, cluster_merge ? 1 : 0, sm_scale, out, lse, part_o,
                           part_lse, status);
    if (e != cudaSuccess) return e;
    count_launches(1);
    if (splits == 1 || cluster_merge) return e;
    merge_kernel<<<dim3(rows_per_seq * 8, bd.B), 256, 0, stream>>>(bd, rr, rows_per_seq, splits, part_o,
                                                                  part_lse, out, lse, status);
    e = cudaGetLastError();
    if (e == cudaSuccess) count_launches(1);
    return e;
}

}  // namespace dsa
