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
// Work items are (query row, segment of its selected list); a CTA walks
// items blockIdx.x, + gridDim.x, ... (one persistent CTA per SM), or holds
// one item when a row's segments merge in a cluster.  With only 64
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
//               into nine 64-column chunks laid out 128B-swizzled; they
//               scan an item's indices (one round trip) and publish its
//               block count.  When the caches do not stay in L2, the rows
//               of the next block are prefetched into L2 (the first two
//               blocks' during the scan), so that a gather waits on L2
//               rather than on HBM, and split items gather with an
//               evict-first policy (each row is read once)
//   warp 2      TMEM owner; loads each item's Q by TMA; MMA issuer
//   warps 3..10 softmax: thread = one gathered row and 32 of the heads (two
//               warps per TMEM lane quarter).  The running per-head max m
//               only moves when some score exceeds it by more than 2^8 (a
//               vote over the block); only then is the exact block max
//               taken (warp max by redux.sync, then across lane quarters)
//               and O^T rescaled in TMEM.  p = 2^(s*c - m) in fp32, written
//               as bf16 P^T over the RoPE chunk (free once S^T is done);
//               final normalisation straight from TMEM into the output (or
//               a split's fp32 partial), one column per thread.  A CTA's
//               first item starts with a side-effect-free pass over the
//               block code while the first tile is in flight (the code is
//               otherwise fetched cold)
// Behind a top-k launch (programmatic dependent launch), a CTA sets itself
// up before the dependency wait, which only the producers take.
// A single 144 KiB row tile fits next to Q (72 KiB); it is refilled chunk
// by chunk as soon as the MMAs that read each chunk have completed.
// Split-K partials (for few query rows): with 2, 4 or 8 splits the CTAs of
// a row form a cluster; each rank merges a share of the heads from its own
// TMEM and the other ranks' normalised outputs, which arrive by bulk copies
// into its shared memory (no scratch memory).  Other split counts write
// fp32 partials that merge_kernel combines.
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
[[maybe_unused]] __device__ __forceinline__ void tmem_ld_hpt(uint32_t taddr, uint32_t (&r)[16]) {
    tmem_ld_32x32b_x16(taddr, r);
}
constexpr int64_t kL2PrefetchBytes = int64_t(128) << 20;  // cache bytes above which rows are prefetched
constexpr int kPrefetchAhead = 1;                         // blocks prefetched ahead of the gather
constexpr int kMaxClusterMerge = 8;                       // most splits merged inside a cluster (portable size)
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
constexpr int kOffScan = kOffL + 7 * kH * 4;                  // int [producer warp]: an item's last valid index
constexpr int kOffMisc = kOffScan + 16;                       // u32: tmem base, abort, block counts of two items
constexpr int kOffBar = kOffMisc + 16;
constexpr int kBarQ = 0;
constexpr int kBarKV = 1;                                     // [9]: chunk c landed
constexpr int kBarPair = kBarKV + kChunks;                    // [4]: chunks 2i, 2i+1 consumed
constexpr int kBarS = kBarPair + 4;                           // S^T ready
constexpr int kBarP = kBarS + 1;                              // P^T written (one arrival per softmax warp)
constexpr int kBarO = kBarP + 1;                              // PV of a block done (chunk 8 free)
constexpr int kBarIdx = kBarO + 1;                            // [2]: indices of a block published
constexpr int kBarDrain = kBarIdx + 2;
constexpr int kBarRecv = kBarDrain + 1;                       // cluster merge: the peers' pieces landed
constexpr int kBarInfo = kBarRecv + 1;                        // [2]: an item's block count published
constexpr int kBarOFree = kBarInfo + 2;                       // an item's output read out of TMEM (one arrival per softmax warp)
constexpr int kBarSlotFree = kBarOFree + 1;                   // [2]: an info slot read (the MMA thread + one per softmax warp)
constexpr int kBarPeerFree = kBarSlotFree + 2;                 // cluster merge: every peer's Q region may be written
constexpr int kBarRecvLse = kBarPeerFree + 1;                  // cluster merge: the peers' lse landed
constexpr int kNumBars = kBarRecvLse + 1;
constexpr int kSmemBytes = kOffBar + kNumBars * 8 + 1024;
static_assert(kSmemBytes <= 232448, "shared memory budget");
// Cluster merge of a row's S = 2, 4 or 8 splits (cluster rank = split).  A
// piece is what one softmax warp sends one peer for one 128-column block dv
// of O: the peer's kHPT / S heads of the warp's head group at the warp's 32
// columns, bf16 pairs of heads [j / 2][lane][j % 2], (32 / S) x 64 bytes.
// Sent from row-tile chunk 2 dv, which the last PV of block dv has just
// freed: [receiving rank][softmax warp] pieces, 16 KiB for every S.  Received
// into the Q region, free once the rank's last S^T is done: [sending rank]
// [dv][softmax warp] pieces, 64 KiB, then the senders' lse [rank][64].  The
// merge's output staging tiles (one per softmax warp, 32 x 32 bf16) sit in
// chunks 1 and 3, free by then.
constexpr int kMergeSlotsBytes = 65536;                                  // receive slots of all ranks
constexpr int kMergeLseRecv = kMergeSlotsBytes;                          // Q region: [sending rank][64] lse
constexpr int kStageBytes = 32 * 32 * 2;
static_assert(kSoftmaxWarps * kHPT * 64 <= kKVChunkBytes, "a block's pieces (S x 8 x (32 / S) x 64 bytes) fit a chunk");
static_assert(4 * kSoftmaxWarps * kHPT * 64 == kMergeSlotsBytes, "merge slots");
static_assert(kSoftmaxWarps / 2 * kStageBytes <= kKVChunkBytes, "half the staging tiles fit a chunk");
static_assert(kMergeLseRecv + kMaxClusterMerge * kH * 4 <= kChunks * kQChunkBytes, "receive slots in the Q region");
static_assert(kOffL % 16 == 0 && (6 * kH * 4) % 16 == 0, "the lse of s_l is a bulk copy source");
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0;                                // O^T: 4 blocks x 64 columns
constexpr uint32_t kTmemS = 256;                              // S^T: 64 columns

// A warp's results for NX rows of a row-major destination, one column per
// lane (columns d0 .. d0 + 31 of row x at dst + x * row_stride): staged in
// the warp's own shared-memory tile, then written back with 16-byte stores
// (a 2-byte store per lane and row cost ~16 cycles per warp instruction).
// dst and row_stride keep every row 16-byte aligned.
// Sums over a warp's 32 lanes of 32 values each, scattered: lane l returns
// the sum of v[l] (a butterfly that halves the values at every step: 31
// shuffles instead of 5 per value).
__device__ __forceinline__ float warp_sum_scatter32(const float (&v)[32], uint32_t lane) {
    float a[16], b[8], c[4], d[2];
    const bool b4 = (lane & 16u) != 0, b3 = (lane & 8u) != 0, b2 = (lane & 4u) != 0, b1 = (lane & 2u) != 0,
               b0 = (lane & 1u) != 0;
#pragma unroll
    for (int i = 0; i < 16; ++i)
        a[i] = (b4 ? v[i + 16] : v[i]) + __shfl_xor_sync(0xffffffffu, b4 ? v[i] : v[i + 16], 16);
#pragma unroll
    for (int i = 0; i < 8; ++i)
        b[i] = (b3 ? a[i + 8] : a[i]) + __shfl_xor_sync(0xffffffffu, b3 ? a[i] : a[i + 8], 8);
#pragma unroll
    for (int i = 0; i < 4; ++i)
        c[i] = (b2 ? b[i + 4] : b[i]) + __shfl_xor_sync(0xffffffffu, b2 ? b[i] : b[i + 4], 4);
#pragma unroll
    for (int i = 0; i < 2; ++i)
        d[i] = (b1 ? c[i + 2] : c[i]) + __shfl_xor_sync(0xffffffffu, b1 ? c[i] : c[i + 2], 2);
    return (b0 ? d[1] : d[0]) + __shfl_xor_sync(0xffffffffu, b0 ? d[0] : d[1], 1);
}

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

// The merge of a row's S = 2, 4 or 8 splits inside their cluster (rank =
// split), run by the softmax warps of every rank once the split's l and lse
// (s_l) and its output O^T (TMEM) are final.  Rank sp writes the heads
// h = sp (mod S):
//   out[h] = sum_s f_s[h] o_s[h] / l_s[h],
//   f_s = exp(lse_s - m) / sum_s' exp(lse_s' - m),  m = max_s lse_s,
// o_s / l_s the split's normalised output.  Each warp sends every peer its
// heads of the warp's 32 columns, normalised, in bf16, one piece per
// 128-column block as soon as it is converted (distributed shared memory
// moves ~14 bytes per clock); a rank's own term is read again from TMEM, in
// fp32.  The weights need every split's lse, which travels ahead of the
// pieces.
//
// Its loops stay rolled: this code runs once per CTA, from a cold
// instruction cache.
template <int S>
__device__ __forceinline__ void cluster_merge_tail(uint8_t* smem, const uint32_t tmem, const int sp, const int nblk,
                                                   const uint32_t last_ph, const int64_t grow,
                                                   uint16_t* __restrict__ out, float* __restrict__ lse,
                                                   int32_t* status) {
    constexpr int hq = kHPT / S;                          // a warp's heads of one rank
    constexpr uint32_t kPiece = (uint32_t)hq * 32u * 2u;
    constexpr uint32_t kSlot = (uint32_t)kMergeSlotsBytes / S;
    const uint32_t warp = warp_id(), lane = lane_id();
    const uint32_t lq = warp & 3u;
    const uint32_t wl = warp - kSoftmaxWarp0;
    const int h0 = ((int)wl >> 2) * kHPT;
    const int st = (int)threadIdx.x - 32 * kSoftmaxWarp0;
    const uint32_t lane_base = (lq * 32u) << 16;
    const float* s_l = reinterpret_cast<const float*>(smem + kOffL);
    float* s_f = reinterpret_cast<float*>(smem + kOffWmax);      // f_s[h] at [s][h] (block-max scratch)
    const uint32_t bar0 = smem_u32(smem + kOffBar);
    auto bar = [&](int n) { return bar0 + 8u * (uint32_t)n; };
    const uint32_t sQr = smem_u32(smem + kOffQ);
    // a peer's Q region is free once its MMAs have drained
    const bool peers_free = __shfl_sync(0xffffffffu, lane == 0 ? mbar_wait(bar(kBarPeerFree), 0) : false, 0);
    if (st == 0 && peers_free) {
        for (int q = 0; q < S; ++q)
            if (q != sp)
                bulk_copy_to_peer(map_to_cluster_rank(sQr + kMergeLseRecv + (uint32_t)sp * kH * 4, (uint32_t)q),
                                  smem_u32(smem + kOffL + 6 * kH * 4), kH * 4,
                                  map_to_cluster_rank(bar(kBarRecvLse), (uint32_t)q));
    }
    float inv[kHPT];                                      // 1 / l of this thread's heads
#pragma unroll
    for (int x = 0; x < kHPT; x += 4) {
        const float4 v = *reinterpret_cast<const float4*>(s_l + 5 * kH + h0 + x);
        inv[x] = v.x;
        inv[x + 1] = v.y;
        inv[x + 2] = v.z;
        inv[x + 3] = v.w;
    }
#pragma unroll 1
    for (int dv = 0; dv < 4; ++dv) {
        uint32_t u[kHPT];
        if (nblk > 0) {
            // this 128-column block of O^T is final once the last block's PV
            // has written it (last_ph: that block's phase)
            if (!mbar_wait(bar(kBarPair + dv), last_ph)) latch_status(status, DSA_ERR_TIMEOUT);
            tc_fence_after();
            tmem_ld_hpt(tmem + lane_base + kTmemO + dv * kH + h0, u);
            tmem_ld_wait();
        } else {
#pragma unroll
            for (int x = 0; x < kHPT; ++x) u[x] = 0u;
        }
        const uint32_t poff = ((uint32_t)dv * kSoftmaxWarps + wl) * kPiece;     // in a receive slot
        const uint32_t soff = (uint32_t)(2 * dv * kKVChunkBytes) + wl * kPiece;  // + q 8 kPiece: in the row tile
#pragma unroll
        for (int q = 0; q < S; ++q) {
            uint32_t* piece = reinterpret_cast<uint32_t*>(smem + kOffKV + soff + q * kSoftmaxWarps * kPiece);
#pragma unroll
            for (int j = 0; j < hq; j += 2) {
                const float va = __uint_as_float(u[q + S * j]) * inv[q + S * j];
                const float vb = __uint_as_float(u[q + S * (j + 1)]) * inv[q + S * (j + 1)];
                if (q != sp) piece[(j / 2) * 32 + lane] = pack_bf16x2(va, vb);
            }
        }
        fence_proxy_async_smem();      // the generic-proxy stores, before the bulk copies read them
        __syncwarp();
        if (lane == 0 && peers_free) {
            for (int q = 0; q < S; ++q)
                if (q != sp)
                    bulk_copy_to_peer(map_to_cluster_rank(sQr + (uint32_t)sp * kSlot + poff, (uint32_t)q),
                                      smem_u32(smem + kOffKV) + soff + (uint32_t)q * kSoftmaxWarps * kPiece,
                                      kPiece, map_to_cluster_rank(bar(kBarRecv), (uint32_t)q));
        }
    }
    // the weights, from every split's lse, while the pieces are in flight
    // (every wait below is agreed by all softmax threads)
    const bool got_lse = !named_bar_or(3, kSoftmaxThreads, !peers_free || !mbar_wait(bar(kBarRecvLse), 0));
    if (got_lse && st < kH) {
        const int h = st;
        const float* rl = reinterpret_cast<const float*>(smem + kOffQ + kMergeLseRecv);
        float ls[S];
        float mx = -INFINITY;
#pragma unroll
        for (int s2 = 0; s2 < S; ++s2) {
            ls[s2] = s2 == sp ? s_l[6 * kH + h] : rl[s2 * kH + h];
            mx = fmaxf(mx, ls[s2]);
        }
        float wsum = 0.f;
#pragma unroll
        for (int s2 = 0; s2 < S; ++s2)
            if (mx > -INFINITY && ls[s2] != -INFINITY) wsum += expf(ls[s2] - mx);
#pragma unroll
        for (int s2 = 0; s2 < S; ++s2)
            s_f[s2 * kH + h] = wsum > 0.f && ls[s2] != -INFINITY ? expf(ls[s2] - mx) / wsum : 0.f;
        if (lse && h % S == sp) lse[grow * kH + h] = wsum > 0.f ? mx + logf(wsum) : -INFINITY;
    }
    // every peer's pieces have landed
    const bool got = got_lse && !named_bar_or(3, kSoftmaxThreads, !mbar_wait(bar(kBarRecv), 0));
    if (!got) {
        latch_status(status, DSA_ERR_TIMEOUT);
        return;
    }
    uint16_t* stage = reinterpret_cast<uint16_t*>(smem + kOffKV + (2 * (wl / 4) + 1) * kKVChunkBytes +
                                                  (wl % 4) * kStageBytes);
    // the weights of this thread's heads h0 + sp + S j, every split
    float fw[hq][S];
#pragma unroll
    for (int j = 0; j < hq; ++j)
#pragma unroll
        for (int s2 = 0; s2 < S; ++s2) fw[j][s2] = s_f[s2 * kH + h0 + sp + S * j];
    tc_fence_after();
#pragma unroll 1
    for (int dv = 0; dv < 4; ++dv) {
        const uint32_t poff = ((uint32_t)dv * kSoftmaxWarps + wl) * kPiece;
        uint32_t u[kHPT];
        if (nblk > 0) {
            tmem_ld_hpt(tmem + lane_base + kTmemO + dv * kH + h0, u);
            tmem_ld_wait();
        } else {
#pragma unroll
            for (int x = 0; x < kHPT; ++x) u[x] = 0u;
        }
        uint16_t o16[hq];
#pragma unroll
        for (int j = 0; j < hq; j += 2) {
            // in split order, this rank's term at its place
            float acc_a = 0.f, acc_b = 0.f;
#pragma unroll
            for (int s2 = 0; s2 < S; ++s2) {
                float va, vb;
                if (s2 == sp) {
                    // u[sp + S j] with sp < S chosen by selects (no local-memory indexing)
                    uint32_t ua = u[S * j], ub = u[S * (j + 1)];
                    float ia = inv[S * j], ib = inv[S * (j + 1)];
#pragma unroll
                    for (int q = 1; q < S; ++q)
                        if (sp == q) {
                            ua = u[S * j + q];
                            ub = u[S * (j + 1) + q];
                            ia = inv[S * j + q];
                            ib = inv[S * (j + 1) + q];
                        }
                    va = __uint_as_float(ua) * ia;
                    vb = __uint_as_float(ub) * ib;
                } else {
                    const uint32_t w2 =
                        reinterpret_cast<const uint32_t*>(smem + kOffQ + s2 * kSlot + poff)[(j / 2) * 32 + lane];
                    va = __uint_as_float(w2 << 16);
                    vb = __uint_as_float(w2 & 0xFFFF0000u);
                }
                acc_a = fmaf(fw[j][s2], va, acc_a);
                acc_b = fmaf(fw[j + 1][s2], vb, acc_b);
            }
            const __nv_bfloat16 ba = __float2bfloat16_rn(acc_a), bb = __float2bfloat16_rn(acc_b);
            o16[j] = *reinterpret_cast<const uint16_t*>(&ba);
            o16[j + 1] = *reinterpret_cast<const uint16_t*>(&bb);
        }
        store_warp_tile(stage, o16, out + (grow * kH + h0 + sp) * kDV + dv * 128 + (int)(lq * 32),
                        (int64_t)S * kDV, lane);
    }
}

// What a CTA writes for its items.  Each kernel instance holds the code of
// one mode only: a CTA runs its once-per-item paths (set-up, first block,
// epilogue) from a cold instruction cache, so code it never runs costs it.
enum OutMode : int {
    kOutRows = 0,        // one split per row: bf16 output rows (and lse)
    kOutPartials = 1,    // fp32 split partials, merged by merge_kernel
    kOutCluster2 = 2,    // the row's 2, 4 or 8 splits merge inside a cluster
    kOutCluster4 = 4,
    kOutCluster8 = 8,
};

template <int kMode>
__global__ void __launch_bounds__(kThreads, 1)
    sparse_mla_tc_kernel(const BatchDev bd, const RowRange rr, const __grid_constant__ CUtensorMap tm_q,
                         const uint16_t* __restrict__ kv, const int32_t* __restrict__ idx, const int idx_local,
                         const int k, const int rows_per_seq, const int splits_arg, const int per_split,
                         const int l2_prefetch, const float sm_scale,
                         uint16_t* __restrict__ out,
                         float* __restrict__ lse,
                         float* __restrict__ part_o, float* __restrict__ part_lse, int32_t* status) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    constexpr bool kCluster = kMode >= kOutCluster2;
    const int splits = kCluster ? kMode : kMode == kOutRows ? 1 : splits_arg;

    const uint32_t sKV = smem_u32(smem + kOffKV);
    const uint32_t sQ = smem_u32(smem + kOffQ);
    int32_t* s_idx = reinterpret_cast<int32_t*>(smem + kOffIdx);
    float* s_wmax = reinterpret_cast<float*>(smem + kOffWmax);
    float* s_m = reinterpret_cast<float*>(smem + kOffM);
    float* s_alpha = reinterpret_cast<float*>(smem + kOffAlpha);
    float* s_thr = reinterpret_cast<float*>(smem + kOffThr);
    float* s_l = reinterpret_cast<float*>(smem + kOffL);
    volatile int32_t* s_scan = reinterpret_cast<volatile int32_t*>(smem + kOffScan);   // [producer warp]
    volatile uint32_t* misc = reinterpret_cast<volatile uint32_t*>(smem + kOffMisc);
    const uint32_t bar0 = smem_u32(smem + kOffBar);
    auto bar = [&](int n) { return bar0 + 8u * (uint32_t)n; };
    const uint32_t warp = warp_id(), lane = lane_id();

    // Work items: (sequence, query row, split) in that order, so the splits
    // of a row are consecutive.  A CTA takes items blockIdx.x, blockIdx.x +
    // gridDim.x, ...: one item when the splits of a row merge in a cluster
    // (the cluster's CTAs are the row's splits), else as many as the grid
    // leaves it (a persistent CTA: the next item's gathers and Q overlap the
    // previous item's softmax and output).  Every role walks the same items
    // and skips the same ones, so their block counts and barrier phases
    // agree; the block count of an item is published by the producers.
    const int64_t per_seq_items = (int64_t)rows_per_seq * splits;
    const int64_t n_items = (int64_t)bd.B * per_seq_items;
    struct Item {
        int b, sp;
        int32_t i, t;
        int64_t grow, prow;
        const int32_t* sel;
        int j_begin, j_end;
        SeqInfo sq;
    };
    auto item_at = [&](int64_t it, Item& o) -> bool {
        o.b = (int)(it / per_seq_items);
        const int64_t rem = it % per_seq_items;
        o.i = rr.i0 + (int32_t)(rem / splits);
        o.sp = (int)(rem % splits);
        if (!load_seq(bd, o.b, status, o.sq)) return false;
        if (o.i >= min(rr.i1, o.sq.nq)) return false;
        o.t = o.sq.ctx - o.sq.nq + o.i;
        o.grow = (int64_t)o.sq.q0 + o.i;
        o.sel = idx + buf_row(idx_local, o.sq, o.b, o.i, rr) * (int64_t)k;
        o.j_begin = o.sp * per_split;
        o.j_end = min(k, o.j_begin + per_split);
        o.prow = ((int64_t)o.b * rows_per_seq + (o.i - rr.i0)) * splits + o.sp;   // split partial row
        return true;
    };

    // Launched after the top-k that writes the indices (programmatic
    // dependent launch), a CTA sets itself up while that kernel finishes:
    // only the producers, which read the indices, wait for it.  Everything
    // else this kernel reads (q, the cache, the batch layout) was written
    // before the top-k started.
    Item first;
    const bool first_ok = (int64_t)blockIdx.x < n_items && item_at(blockIdx.x, first);
    auto get_item = [&](int64_t it, Item& o) -> bool {
        if (it != (int64_t)blockIdx.x) return item_at(it, o);
        o = first;
        return first_ok;
    };
    if (threadIdx.x == 32 * kMmaWarp) prefetch_tmap(&tm_q);
    if (threadIdx.x == 0) {
        for (int n = 0; n < kNumBars; ++n) {
            uint32_t count = 1;
            if (n == kBarP || n == kBarOFree) count = kSoftmaxThreads / 32;               // one per softmax warp
            if (n == kBarSlotFree || n == kBarSlotFree + 1) count = 1 + kSoftmaxThreads / 32;   // + the MMA thread
            if (n >= kBarKV && n < kBarKV + kChunks) count = 32 * kProducerWarps;         // every producer lane
            if (kCluster && n == kBarPeerFree) count = kCluster ? kMode - 1 : 1;        // one per peer
            mbar_init(bar(n), count);
        }
        // a row merged in a cluster receives, from every other split, its
        // slot of pieces and its lse
        if constexpr (kCluster) {
            mbar_arrive_expect_tx(bar(kBarRecv), (uint32_t)((kMode - 1) * (kMergeSlotsBytes / kMode)));
            mbar_arrive_expect_tx(bar(kBarRecvLse), (uint32_t)((kMode - 1) * kH * 4));
        }
        misc[1] = 0;
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
    const float c2 = sm_scale * kLog2e;      // logits in log2 units
    int c_nblk = 0, c_sp = 0;                // the (single) item of a cluster-merged CTA:
    int64_t c_grow = 0;                      // its block count, split and packed row
    bool had_item = false;

    if (warp < kProducerWarps) {
        // ----------------------------------------------------------- producers
        // producer lane gl = (rq, piece): rows 16n + rq of the block, 16-byte
        // piece `piece` of each 128-byte row chunk; 8 lanes cover one row
        // chunk (coalesced) and row r % 8 == rq % 8 fixes the swizzle
        const int gl = (int)threadIdx.x;
        const int rq = gl >> 3, piece = gl & 7;
        const uint32_t dpat = (uint32_t)(rq * 128 + ((piece ^ (rq & 7)) << 4));
        // A cache larger than L2 is read once per launch: the split
        // instances (decode-sized batches) mark a gathered line, prefetched
        // at normal priority so that it stays until this read, to be evicted
        // first; the lines that are read again (the kernel's code, q, the
        // outputs) then stay (decode 64 x 32,768 attention launched back to
        // back: 50.3 -> 46.2 us).  The row instance keeps the plain copies
        // (the hinted loop cost its prefill 1.5 %).
        const uint64_t evict_first = l2_evict_first_policy();
        constexpr int kPT = 32 * kProducerWarps;
        pdl_wait();              // the indices of the previous launch are complete
        bool ok = true;
        uint32_t gb = 0;         // blocks of all items so far: the phase of every per-block barrier
        uint32_t nitem = 0;      // items so far: the info slot and the phases of per-item barriers
        for (int64_t it = blockIdx.x; it < n_items; it += gridDim.x) {
            Item I;
            if (!get_item(it, I)) continue;
            const uint8_t* kv_seq = reinterpret_cast<const uint8_t*>(kv) + (int64_t)I.b * bd.stride * (kDQK * 2);
            // blocks of this segment: up to its last valid entry (16-byte
            // loads when the rows are 16-byte aligned, one round trip); with
            // L2 prefetching on, the rows of the first 1 + kPrefetchAhead
            // blocks are prefetched as their indices are seen
            // (in the split instances the softmax warps prefetch the first
            // item's rows: they are idle then, and the scan reaches its first
            // gathers sooner)
            auto prefetch_row = [&](int j, int32_t sv) {
                if (l2_prefetch && (kMode == kOutRows || nitem > 0) && j < I.j_begin + (1 + kPrefetchAhead) * kBlk &&
                    sv >= 0 && sv <= I.t)
                    prefetch_l2_bulk(kv_seq + (int64_t)sv * (kDQK * 2), kDQK * 2);
            };
            int last = -1;
            // with 16-byte loads, lane l of warp 0 holds entries 4l .. 4l + 3
            // of the first block: they go to shared memory from registers
            int4 blk0 = make_int4(-1, -1, -1, -1);
            const bool blk0_in_regs = (k & 3) == 0;
            if ((k & 3) == 0) {
                // at most kMaxTopk / 4 groups of four indices: every group of
                // this thread is loaded before any is tested (one round trip)
                constexpr int kScanIt = kMaxTopk / 4 / kPT;
                const int4* sel4 = reinterpret_cast<const int4*>(I.sel + I.j_begin);   // j_begin: a multiple of 128
                const int nq4 = (I.j_end - I.j_begin) >> 2;
                int4 vs[kScanIt];
#pragma unroll
                for (int u = 0; u < kScanIt; ++u) {
                    const int q = gl + u * kPT;
                    vs[u] = q < nq4 ? __ldg(sel4 + q) : make_int4(-1, -1, -1, -1);
                }
                blk0 = vs[0];
                static_assert(kPT >= 32 && kBlk == 4 * 32, "warp 0's first loads cover the first block");
#pragma unroll
                for (int u = 0; u < kScanIt; ++u) {
                    const int q = gl + u * kPT;
                    if (q >= nq4) break;
                    const int4 v = vs[u];
                    const int j = I.j_begin + 4 * q;
                    if (v.x >= 0) last = j;
                    if (v.y >= 0) last = j + 1;
                    if (v.z >= 0) last = j + 2;
                    if (v.w >= 0) last = j + 3;
                    prefetch_row(j, v.x);
                    prefetch_row(j + 1, v.y);
                    prefetch_row(j + 2, v.z);
                    prefetch_row(j + 3, v.w);
                }
                static_assert(kMaxTopk % (4 * kPT) == 0, "the index scan covers a whole segment");
            } else {
                for (int j = I.j_begin + gl; j < I.j_end; j += kPT) {
                    const int32_t sv = __ldg(I.sel + j);
                    if (sv >= 0) last = j;
                    prefetch_row(j, sv);
                }
            }
            last = __reduce_max_sync(0xffffffffu, last);
            if (lane == 0) s_scan[warp] = last;
            // the info slot of this item was last used by the item two
            // before: its readers (the MMA thread, every softmax warp) must
            // be done with it (each slot's barrier completes once per use,
            // and no reader can be a use ahead, so the phases never alias)
            bool wok = nitem < 2 || mbar_wait(bar(kBarSlotFree + (nitem & 1u)), ((nitem >> 1) - 1u) & 1u);
            // both producer warps agree (scan results, aborts) before either goes on
            if (named_bar_or(5, kPT, !wok || misc[1] != 0)) {
                ok = false;
                break;
            }
            for (int w2 = 0; w2 < kProducerWarps; ++w2) last = max(last, (int)s_scan[w2]);
            const int nblk = last < I.j_begin ? 0 : (last - I.j_begin) / kBlk + 1;
            named_bar_sync(4, kPT);          // s_scan is read by both warps before the next item writes it
            if (gl == 0) {
                misc[2 + (nitem & 1u)] = (uint32_t)nblk;
                mbar_arrive(bar(kBarInfo + (nitem & 1u)));
            }
            for (int jb = 0; jb < nblk; ++jb, ++gb) {
                const uint32_t ph = gb & 1u;
                int32_t* ib = s_idx + (gb & 1u) * kBlk;
                // this block's indices (warp 0) are loaded before the prefetch
                // below, so that the two round trips overlap; the first
                // block's come from the scan (entry 4 lane + u in v[u], else
                // entry 32 u + lane)
                const bool from_scan = jb == 0 && blk0_in_regs;
                int32_t v[4] = {blk0.x, blk0.y, blk0.z, blk0.w};
                if (warp == 0 && !from_scan) {
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int j = I.j_begin + jb * kBlk + u * 32 + (int)lane;
                        v[u] = (j < I.j_end) ? __ldg(I.sel + j) : -1;
                    }
                }
                // (the scan prefetched the blocks up to kPrefetchAhead)
                if (l2_prefetch && jb > 0 && jb + kPrefetchAhead < nblk) {
                    // the rows of block jb + kPrefetchAhead (valid indices only),
                    // one 1152-byte bulk prefetch each
                    for (int u = gl; u < kBlk; u += kPT) {
                        const int j = I.j_begin + (jb + kPrefetchAhead) * kBlk + u;
                        const int32_t sv = j < I.j_end ? __ldg(I.sel + j) : -1;
                        if (sv >= 0 && sv <= I.t) prefetch_l2_bulk(kv_seq + (int64_t)sv * (kDQK * 2), kDQK * 2);
                    }
                }
                if (warp == 0) {
                    // indices of this block: validated, -1 where invalid or past the segment
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        if (v[u] < -1 || v[u] > I.t) {
                            latch_status(status, DSA_ERR_BAD_INDEX);
                            v[u] = -1;
                        }
                    }
                    // buffer gb & 1 was last read by the softmax of block gb - 2,
                    // which finished before PV(gb - 2) started; these warps have
                    // already waited for PV(gb - 2) to complete (before refilling
                    // chunk 8 in block gb - 1), so the buffer is free and the
                    // block's indices and row offsets are ready before PV(gb - 1)
                    const bool wok2 = __all_sync(0xffffffffu, !misc[1]);
                    if (wok2) {
                        if (from_scan) {
                            reinterpret_cast<int4*>(ib)[lane] = make_int4(v[0], v[1], v[2], v[3]);
                        } else {
#pragma unroll
                            for (int u = 0; u < 4; ++u) ib[u * 32 + lane] = v[u];
                        }
                        __syncwarp();
                        if (lane == 0) mbar_arrive(bar(kBarIdx + (gb & 1u)));
                    } else {
                        misc[1] = 1;
                    }
                }
                // the block's indices are in shared memory; an abort seen by
                // either warp stops both (one barrier reduction, so they agree)
                if (named_bar_or(4, kPT, misc[1] != 0)) {
                    ok = false;
                    break;
                }
                uint32_t soff[kProducerRows];   // byte offset of each of this lane's rows (+ piece)
#pragma unroll
                for (int n = 0; n < kProducerRows; ++n) {
                    const int32_t sv = ib[4 * kProducerWarps * n + rq];
                    soff[n] = (uint32_t)(sv >= 0 ? sv : 0) * (uint32_t)(kDQK * 2) + (uint32_t)(piece * 16);
                }
                // the nine chunks (one copy of the loop per eviction policy)
                auto fill = [&](auto hinted) {
                    for (int c = 0; c < kChunks; ++c) {
                        // chunk c of the previous block (of this or an earlier
                        // item) must have been consumed: chunks 2i and 2i + 1
                        // are freed together (one wait per pair)
                        if (gb > 0 && (c == kVChunks || (c & 1) == 0)) {
                            const uint32_t fb = c < kVChunks ? bar(kBarPair + c / 2) : bar(kBarO);
                            ok = mbar_wait(fb, ph ^ 1u);
                            ok = __all_sync(0xffffffffu, ok);
                            if (!ok) break;
                        }
                        const uint8_t* src = kv_seq + c * 128;
                        const uint32_t dst = sKV + c * kKVChunkBytes + dpat;
#pragma unroll
                        for (int n = 0; n < kProducerRows; ++n) {
                            if constexpr (decltype(hinted)::value)
                                cp_async_16_hint(dst + (uint32_t)(512 * kProducerWarps) * n, src + soff[n],
                                                 evict_first);
                            else
                                cp_async_16(dst + (uint32_t)(512 * kProducerWarps) * n, src + soff[n]);
                        }
                        cp_async_arrive(bar(kBarKV + c));
                    }
                };
                if constexpr (kMode == kOutRows) {
                    fill(std::false_type{});
                } else {
                    if (l2_prefetch) fill(std::true_type{});
                    else fill(std::false_type{});
                }
                // both producer warps agree before either starts the next block
                if (named_bar_or(5, kPT, !ok)) {
                    ok = false;
                    misc[1] = 1;
                    break;
                }
            }
            if (!ok) break;
            ++nitem;
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
            bool ok = true, q_pending = false;
            uint32_t gb = 0, nitem = 0, nq = 0;
            int my_sp = 0;
            bool peers_told = false;
            // the peers of a cluster may send into this CTA's Q region once
            // nothing reads it any more
            auto tell_peers = [&]() {
                if constexpr (kCluster) {
                    for (int q = 0; q < kMode; ++q)
                        if (q != my_sp) mbar_arrive_peer(map_to_cluster_rank(bar(kBarPeerFree), (uint32_t)q));
                    peers_told = true;
                }
            };
            for (int64_t it = blockIdx.x; ok && it < n_items; it += gridDim.x) {
                Item I;
                if (!get_item(it, I)) continue;
                had_item = true;
                my_sp = I.sp;
                // Q of this item by TMA, once the S^T of the previous item's
                // last block (the last reader of the old Q) is done; issued
                // before the item's block count is known, so that it lands
                // while the producers scan the indices
                if (misc[1] || (gb > 0 && !mbar_wait(bar(kBarS), (gb - 1u) & 1u))) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(bar(kBarQ), kChunks * kQChunkBytes);
                for (int c = 0; c < kChunks; ++c)
                    tma_load_2d(sQ + c * kQChunkBytes, &tm_q, bar(kBarQ), c * 64, (int32_t)(I.grow * kH));
                q_pending = true;
                if (!mbar_wait(bar(kBarInfo + (nitem & 1u)), (nitem >> 1) & 1u)) {
                    ok = false;
                    break;
                }
                const int nblk = (int)misc[2 + (nitem & 1u)];
                mbar_arrive(bar(kBarSlotFree + (nitem & 1u)));
                if (!mbar_wait(bar(kBarQ), nq & 1u)) {
                    ok = false;
                    break;
                }
                q_pending = false;
                ++nq;
                tc_fence_after();
                for (int jb = 0; ok && jb < nblk; ++jb, ++gb) {
                    const uint32_t ph = gb & 1u;
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
                    // O^T += V^T . P^T once the softmax has written P^T; an
                    // item's first PV overwrites O^T, so it also waits until
                    // the previous item's output has been read out of TMEM
                    if (misc[1] || !mbar_wait(bar(kBarP), ph) ||
                        (jb == 0 && nitem > 0 && !mbar_wait(bar(kBarOFree), (nitem - 1u) & 1u))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // P^T of the last block is written, so its S^T, the last
                    // reader of Q, has completed
                    if (kCluster && jb == nblk - 1) tell_peers();
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
                ++nitem;
            }
            if (!ok) {
                latch_status(status, DSA_ERR_TIMEOUT);
                misc[1] = 1;
            }
            // every MMA this thread issued has finished once drain completes
            mma_commit(bar(kBarDrain));
            mbar_wait(bar(kBarDrain), 0);
            if (q_pending) mbar_wait(bar(kBarQ), nq & 1u);    // Q's copy must land before the CTA exits
            if (had_item && !peers_told) tell_peers();      // (no blocks, or an abort)
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------- softmax
        // warp w: TMEM lane quarter w % 4 (rows), head group (w - 3) / 4 of
        // kHPT heads
        const uint32_t lq = warp & 3u;
        const int h0 = ((int)(warp - kSoftmaxWarp0) >> 2) * kHPT;
        const int r = (int)(lq * 32 + lane);           // row of the block
        const int st = (int)threadIdx.x - 32 * kSoftmaxWarp0;   // 0..255 among the softmax threads
        const uint32_t lane_base = (lq * 32u) << 16;
        bool ok = true;
        uint32_t gb = 0, nitem = 0;
        for (int64_t it = blockIdx.x; it < n_items; it += gridDim.x) {
            Item I;
            if (!get_item(it, I)) continue;
            had_item = true;
            float lsum[kHPT];
#pragma unroll
            for (int x = 0; x < kHPT; ++x) lsum[x] = 0.f;
            int nblk = 0;
            // A CTA's first item starts with a dry run of the block code
            // (jb = -1), before the item's block count is known.  The softmax
            // warps wait microseconds for the first S^T tile, and code an SM
            // runs for the first time is fetched from L2 or HBM a few lines at
            // a time, which costs the first block more than its own work.  The
            // dry run reads the O^T columns of TMEM (nothing writes them
            // before the first P^T), writes no P^T, waits for and arrives on
            // no barrier; the running max, its bounds and the partial sums are
            // reset after it.
            for (int jb = nitem == 0 ? -1 : 0;; ++jb) {
                if (jb == 0) {
                    // the item's block count, published by the producers
                    const bool gi = !misc[1] && mbar_wait(bar(kBarInfo + (nitem & 1u)), (nitem >> 1) & 1u);
                    // every abort is agreed by all softmax threads before any
                    // named barrier, so none of them can be left waiting at one
                    if (named_bar_or(3, kSoftmaxThreads, !gi)) {
                        ok = false;
                        break;
                    }
                    nblk = (int)misc[2 + (nitem & 1u)];
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(kBarSlotFree + (nitem & 1u)));
                    if (nitem > 0) {
                        // a fresh running max (the previous item's output, the
                        // last reader of m, is done; the first item starts from
                        // the set-up's values)
                        if (st < kH) {
                            s_m[st] = -INFINITY;
                            s_thr[st] = -INFINITY;
                        }
                        named_bar_sync(1, kSoftmaxThreads);
                    }
                }
                if (jb >= 0 && jb >= nblk) break;
                const bool dry = jb < 0;
                const uint32_t ph = gb & 1u;
                const bool got = dry || (!misc[1] && mbar_wait(bar(kBarIdx + (gb & 1u)), (gb >> 1) & 1u) &&
                                         mbar_wait(bar(kBarS), ph));
                tc_fence_after();
                const bool valid = s_idx[(gb & 1u) * kBlk + r] >= 0;
                // the running max moves only when a score exceeds it by 2^8; the
                // vote compares raw scores with (m + 8) / c2 per head (a trigger
                // only: the exact block max below decides whether m moves).  The
                // bounds are read while the TMEM load is in flight.
                float s[kHPT];
                bool exceed = false;
                {
                    uint32_t u[kHPT];
                    tmem_ld_hpt(tmem + lane_base + (dry ? kTmemO : kTmemS) + h0, u);
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
                if (named_bar_or(2, kSoftmaxThreads, exceed || !got || dry)) {
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
                        const bool w = jb <= 0 || mbar_wait(bar(kBarO), ph ^ 1u);
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
                    if (!dry) *reinterpret_cast<uint4*>(p_row + ((c8 ^ (r & 7)) << 4)) = pk;
                }
                // one arrival per warp once all its lanes' P^T writes are fenced
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (dry) {
#pragma unroll
                    for (int x = 0; x < kHPT; ++x) lsum[x] = 0.f;
                    named_bar_sync(1, kSoftmaxThreads);      // the dry run's reads of m are done
                    if (st < kH) {
                        s_m[st] = -INFINITY;
                        s_thr[st] = -INFINITY;
                    }
                    named_bar_sync(1, kSoftmaxThreads);
                    if (kMode != kOutRows && l2_prefetch) {
                        // the rows of the first item's first 1 + kPrefetchAhead
                        // blocks (one index per thread; these warps are idle
                        // until the first S^T tile; the row instance keeps
                        // them in the producers' scan, its code unchanged)
                        pdl_wait();      // the indices of the previous launch are complete
                        const uint8_t* kv_seq =
                            reinterpret_cast<const uint8_t*>(kv) + (int64_t)I.b * bd.stride * (kDQK * 2);
                        for (int j = I.j_begin + st; j < min(I.j_end, I.j_begin + (1 + kPrefetchAhead) * kBlk);
                             j += kSoftmaxThreads) {
                            const int32_t sv = __ldg(I.sel + j);
                            if (sv >= 0 && sv <= I.t) prefetch_l2_bulk(kv_seq + (int64_t)sv * (kDQK * 2), kDQK * 2);
                        }
                    }
                    continue;
                }
                if (lane == 0) mbar_arrive(bar(kBarP));
                ++gb;
            }
            if (!ok) break;
            c_nblk = nblk;
            c_sp = I.sp;
            c_grow = I.grow;
            // ------------------------------------------------- item epilogue
            // l: the per-thread partial sums reduced over the 128 rows (lane
            // x of a warp ends with head h0 + x of its lane quarter)
            static_assert(kHPT == 32, "one head per lane in the l reduction");
            s_l[lq * kH + h0 + lane] = warp_sum_scatter32(lsum, lane);
            if constexpr (kCluster) {
                // (the merge waits for each 128-column block of the last PV)
                named_bar_sync(1, kSoftmaxThreads);
            } else {
                const bool got_o = nblk == 0 || mbar_wait(bar(kBarO), (gb - 1u) & 1u);
                // agreed by every softmax thread: the stores below end with a barrier
                if (named_bar_or(3, kSoftmaxThreads, !got_o)) {
                    ok = false;
                    break;
                }
            }
            if (st < kH) {
                const float lt = s_l[st] + s_l[kH + st] + s_l[2 * kH + st] + s_l[3 * kH + st];
                s_l[4 * kH + st] = lt;
                s_l[5 * kH + st] = lt > 0.f ? 1.f / lt : 0.f;
                const float ls = lt > 0.f ? (s_m[st] + log2f(lt)) * kLn2 : -INFINITY;
                if constexpr (kMode == kOutRows) {
                    if (lse) lse[I.grow * kH + st] = ls;
                } else if constexpr (kCluster) {
                    s_l[6 * kH + st] = ls;
                    fence_proxy_async_smem();      // sent to the peers from s_l by bulk copy
                } else {
                    part_lse[I.prow * kH + st] = ls;
                }
            }
            named_bar_sync(1, kSoftmaxThreads);
            if constexpr (!kCluster) {
                // every MMA of the item has completed (PV of its last block):
                // each thread stores its output column d of its heads straight
                // from TMEM (the row tile may already hold the next item's rows)
                tc_fence_after();
                float inv[kHPT];                              // 1 / l of this thread's heads
#pragma unroll
                for (int x = 0; x < kHPT; x += 4) {
                    const float4 v = *reinterpret_cast<const float4*>(s_l + 5 * kH + h0 + x);
                    inv[x] = v.x;
                    inv[x + 1] = v.y;
                    inv[x + 2] = v.z;
                    inv[x + 3] = v.w;
                }
                uint16_t* ob = out + (I.grow * kH + h0) * kDV;
                float* po = kMode == kOutPartials ? part_o + (I.prow * kH + h0) * kDV : nullptr;
                for (int dv = 0; dv < 4; ++dv) {
                    const int d = dv * 128 + r;               // output column of this thread
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
                        const float o = __uint_as_float(u[x]) * inv[x];
                        if constexpr (kMode == kOutRows) {
                            const __nv_bfloat16 b16 = __float2bfloat16_rn(o);
                            ob[x * kDV + d] = *reinterpret_cast<const uint16_t*>(&b16);
                        } else {
                            po[x * kDV + d] = o;
                        }
                    }
                }
                // O^T has been read: the next item's first PV may overwrite it
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(kBarOFree));
                // s_l and s_m are read by every thread before the next item resets them
                named_bar_sync(1, kSoftmaxThreads);
            }
            ++nitem;
        }
        if (!ok) {
            latch_status(status, DSA_ERR_TIMEOUT);
            misc[1] = 1;
        }
        if constexpr (kCluster) {
            if (ok && had_item)
                cluster_merge_tail<kMode>(smem, tmem, c_sp, c_nblk, (gb - 1u) & 1u, c_grow, out, lse, status);
        }
    }

    if constexpr (kCluster) {
        // a CTA's row tile is the source of its bulk copies and its Q region
        // their destination: none exits before every copy has landed (a
        // cluster's CTAs are the splits of one row: all have an item or none)
        if (first_ok) cg::this_cluster().sync();
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

// Splits merged inside a cluster: the count divides the heads and is small
// enough that a cluster of that many one-SM CTAs always fits in a GPC.
bool merge_in_cluster(int splits) { return splits > 1 && splits <= kMaxClusterMerge && kH % splits == 0; }

// CTAs per query row.  One CTA fills an SM's shared memory, so the grid
// runs in waves of num_sms() CTAs; pick the split count that minimises
// waves x (blocks per CTA + one block's worth of per-CTA overhead), plus
// one block for splits that merge through fp32 partials and a second
// launch rather than inside a cluster (8 x 202,752 decode: 8 cluster
// splits 24.0 us, 27.3 us from a cold L2, against 24.6 / 31.4 us for 16
// splits and partials).
int choose_splits(int64_t rows, int k) {
    if (rows <= 0) return 1;
    const int nblk = std::max(1, (k + kBlk - 1) / kBlk);
    const int64_t nsm = num_sms();
    int best = 1;
    int64_t best_cost = -1;
    for (int sp = 1; sp <= std::min(16, nblk); ++sp) {
        const int64_t waves = (rows * sp + nsm - 1) / nsm;
        const int64_t cost = waves * ((nblk + sp - 1) / sp + 1) + (sp > 1 && !merge_in_cluster(sp) ? 1 : 0);
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best = sp;
        }
    }
    return best;
}

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
    const int mode = splits == 1 ? kOutRows : cluster_merge ? splits : kOutPartials;
    auto* kern = mode == kOutRows       ? sparse_mla_tc_kernel<kOutRows>
                 : mode == kOutPartials ? sparse_mla_tc_kernel<kOutPartials>
                 : mode == kOutCluster2 ? sparse_mla_tc_kernel<kOutCluster2>
                 : mode == kOutCluster4 ? sparse_mla_tc_kernel<kOutCluster4>
                                        : sparse_mla_tc_kernel<kOutCluster8>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    // caches larger than a fraction of L2 are read from HBM: prefetch one
    // block ahead (a cache that stays L2-resident gains nothing from it, and
    // a CTA of a single block only duplicates its own gather: 8 x 202,752
    // decode, 16 splits of one block, 28.6 -> 26.9 us without)
    const int l2_prefetch =
        (int64_t)bd.B * bd.max_ctx * (kDQK * 2) > kL2PrefetchBytes && per_split > kBlk ? 1 : 0;
    cudaLaunchConfig_t cfg = {};
    // work items (sequence, query row, split): one CTA per item when the
    // splits of a row merge in a cluster, else a persistent CTA per SM
    const int64_t items = (int64_t)bd.B * rows_per_seq * splits;
    const int64_t ctas = cluster_merge ? items : std::min<int64_t>(items, num_sms());
    if (ctas >= (int64_t(1) << 31)) return cudaErrorInvalidValue;
    cfg.gridDim = dim3((unsigned)ctas, 1u);
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
    e = cudaLaunchKernelEx(&cfg, kern, bd, rr, tm_q, kv, idx, idx_local ? 1 : 0, k, rows_per_seq, splits,
                           per_split, l2_prefetch, sm_scale, out, lse, part_o, part_lse, status);
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
