// topk.cu -- deterministic causal top-k of indexer score rows.
//
// ("GLM-5.1 架构深度拆解", section 3.6 Steps 6-7: positions s > t are masked
// and min(index_topk, length) positions are kept; section 3.4: the
// selection must be deterministic; the GLM-5 explainer page: a query that
// sees fewer than 2048 positions keeps all of them.)
//
// One thread-block cluster of C CTAs per query row (C = 1 unless rows are
// long and few); CTA r owns the r-th contiguous slice of the row.  Scores
// map to order-preserving 32-bit keys (-0.0 folded onto +0.0).
//   1. A lower bound L for the k-th largest key: the lower edge of the
//      11-bit digit bin (the digit just below the bits all sampled keys
//      share) holding the (r+1)-th largest of 1024 evenly spaced keys of the
//      whole row, r sized so that well over k keys lie at or above it.
//      Every CTA of the cluster derives the same L.
//   2. One pass over the slice (16-byte loads, several in flight): warp w of
//      a CTA owns a contiguous segment and appends its keys >= L, in
//      position order, to a shared-memory region of its own (keys are
//      tested as floats against L; one warp scan per step places them).
//   3. The exact k-th largest key tau among the candidates of the cluster:
//      a radix select over the bits below those that L and the largest
//      candidate share (digits of up to 11 bits); each CTA counts
//      its candidates and every CTA sums the cluster's histograms through
//      distributed shared memory, so all derive the same digits.
//   4. The output in position order: candidates above tau and the first
//      `need` candidates equal to tau (ties go to the lower position), each
//      written at its rank; ranks add the counts of lower warps and lower
//      CTAs.  Positions come out ascending.
// Every key that is not a candidate lies below L <= tau, so the result is
// exactly the top-k of the row.  If the sample misjudges (fewer than k
// candidates in the cluster, or a full region) steps 3-4 run over the whole
// slices instead.  Atomics only count; the result is the same bit for bit
// on every run.
#include <cooperative_groups.h>

#include <algorithm>

#include "internal.h"
#include "ptx.cuh"

namespace cg = cooperative_groups;

namespace dsa {
namespace {

// Threads per CTA: 1024 when a launch has fewer rows than SMs (one CTA per
// SM, more warps to hide latency), else 512 (two CTAs per SM).
constexpr int kBins = 2048;
constexpr int kSample = 512;
constexpr int kRegion = 512;                 // candidate slots per warp
constexpr int kPrefetch = 8;                 // 16-byte loads in flight per lane (32 keys)
static_assert(kPrefetch <= 8, "a lane's candidate flags fill one 32-bit word, its counts one 64-bit word");
constexpr int kMaxCluster = 8;
constexpr int kLongRow = 65536;              // rows above this may be split over a cluster
constexpr int kKeysPerCta = 32768;

__device__ __forceinline__ uint32_t order_key(float f) {
    uint32_t u = __float_as_uint(f);
    if (u == 0x80000000u) u = 0u;     // -0.0 compares equal to +0.0
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// The float whose key is `key` (inverse of order_key; +0.0 for the key of
// zero).  For non-NaN x: x >= key_float(key) exactly when order_key(x) >= key,
// provided key_float(key) is not a NaN.
__device__ __forceinline__ float key_float(uint32_t key) {
    return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}

__device__ __forceinline__ uint32_t warp_inclusive_scan(uint32_t v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t n = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += n;
    }
    return v;
}

template <int NT>
struct alignas(16) TopkSmem {
    static constexpr int kMaxCand = NT / 32 * kRegion;
    uint32_t hist[kBins];                 // zero between selects
    uint32_t sample[kSample];
    uint32_t cand_key[kMaxCand];          // warp w: [w * kRegion, w * kRegion + count)
    int32_t cand_pos[kMaxCand];
    uint32_t warp_sums[32];
    uint32_t wcnt[32], wgt[32], weq[32], wmax[32];
    uint32_t group[kBins / 32];           // this CTA's counts of 64 groups of 32 bins (cluster selects)
    uint32_t small[64];                   // this CTA's keys of a small boundary bin
    uint32_t small_all[64];               // the bin's keys of the whole cluster
    uint32_t total, sel_digit, sel_above, sel_count, chunk_total;
    uint32_t small_n, small_all_n, small_tau, small_need;
    uint32_t cta_cand, cta_overflow, cta_gt, cta_eq, cta_max;   // read by the rest of the cluster
    uint32_t all_cand, all_overflow, all_max, pre_gt, pre_eq;    // the cluster's, combined by warp 0
};

// The k-th largest of the keys that `visit` hands to this thread's callback,
// over this CTA (nranks == 1) or over the whole cluster (nranks == cluster
// size).  Every such key agrees with `prefix0` above its low `hi` bits;
// those bits are resolved from the top in digits of up to 11 bits, at most
// `passes` of them (enough passes = exact).  Returns tau (the bits found,
// zero below) and sets need = how many keys matching tau belong to the top
// k.  Starting below the bits the keys share keeps them spread over many
// bins (few atomic collisions).  Once at most 64 keys (over the cluster)
// remain in the boundary bin, they are gathered and ranked directly.  S.hist must
// be zero on entry; zero on return.
template <int NT, typename Visit>
__device__ uint32_t radix_select(cg::cluster_group& cluster, int nranks, TopkSmem<NT>& S, uint32_t k, int hi,
                                 uint32_t prefix0, int passes, Visit visit, uint32_t& need_out) {
    constexpr int kWarps = NT / 32, kBinsPerThread = kBins / NT;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint32_t pmask = hi >= 32 ? 0u : ~((1u << hi) - 1u);
    uint32_t prefix = prefix0 & pmask, need = k;
    int top = hi;
#pragma unroll 1
    for (int p = 0; p < passes && top > 0; ++p) {
        const int sh = max(0, top - 11);
        const uint32_t dmask = (1u << (top - sh)) - 1u;
        top = sh;
        visit([&](uint32_t key) {
            if ((key & pmask) == prefix) atomicAdd(&S.hist[(key >> sh) & dmask], 1u);
        });
        if (nranks > 1) {
            // Over a cluster: the group of 32 bins that holds the need-th
            // largest key, from every rank's 64 group counts, then its bin
            // from every rank's 32 counts of that group (the bin the flat
            // scan below would find, from 3 % of the remote reads).
            constexpr int kGroups = kBins / 32;
            __syncthreads();                           // this rank's histogram is complete
            if (tid < kGroups) {
                uint32_t g = 0u;
#pragma unroll 8
                for (int b2 = 0; b2 < 32; ++b2) g += S.hist[32 * tid + b2];
                S.group[tid] = g;
            }
            cluster.sync();                            // every rank's group counts are ready
            if (warp == 0) {
                // lane l: groups 2l and 2l + 1, summed over the ranks in rank order
                uint32_t g0 = 0u, g1 = 0u;
                {
                    uint32_t r0[kMaxCluster], r1[kMaxCluster];
#pragma unroll
                    for (int r = 0; r < kMaxCluster; ++r) {
                        const uint32_t* h = cluster.map_shared_rank(S.group, (unsigned)min(r, nranks - 1));
                        r0[r] = r < nranks ? h[2 * lane] : 0u;
                        r1[r] = r < nranks ? h[2 * lane + 1] : 0u;
                    }
#pragma unroll
                    for (int r = 0; r < kMaxCluster; ++r) {
                        g0 += r0[r];
                        g1 += r1[r];
                    }
                }
                const uint32_t incl = warp_inclusive_scan(g0 + g1);
                const uint32_t total = __shfl_sync(0xffffffffu, incl, 31);
                const uint32_t above1 = total - incl;  // keys in groups above 2l + 1
                const uint32_t above0 = above1 + g1;   // keys in groups above 2l
                int grp = -1;
                uint32_t gabove = 0u;
                if (above1 < need && need <= above1 + g1) {
                    grp = 2 * (int)lane + 1;
                    gabove = above1;
                } else if (above0 < need && need <= above0 + g0) {
                    grp = 2 * (int)lane;
                    gabove = above0;
                }
                const uint32_t has = __ballot_sync(0xffffffffu, grp >= 0);
                const int src = has ? __ffs(has) - 1 : 0;
                grp = __shfl_sync(0xffffffffu, grp, src);
                gabove = __shfl_sync(0xffffffffu, gabove, src);
                if (has) {
                    // lane l: bin 32 grp + l, summed over the ranks in rank order
                    uint32_t rb[kMaxCluster];
#pragma unroll
                    for (int r = 0; r < kMaxCluster; ++r) {
                        const uint32_t* h = cluster.map_shared_rank(S.hist, (unsigned)min(r, nranks - 1));
                        rb[r] = r < nranks ? h[32 * grp + lane] : 0u;
                    }
                    uint32_t cb = 0u;
#pragma unroll
                    for (int r = 0; r < kMaxCluster; ++r) cb += rb[r];
                    const uint32_t bincl = warp_inclusive_scan(cb);
                    const uint32_t gtot = __shfl_sync(0xffffffffu, bincl, 31);
                    const uint32_t above = gabove + (gtot - bincl);   // keys in higher bins
                    if (above < need && need <= above + cb) {
                        S.sel_digit = (uint32_t)(32 * grp + (int)lane);
                        S.sel_above = above;
                        S.sel_count = cb;
                    }
                }
                if (lane == 0) S.total = total;
            }
            cluster.sync();                            // every remote read done before any bin is cleared
#pragma unroll
            for (int x = 0; x < kBinsPerThread; ++x) S.hist[kBinsPerThread * tid + x] = 0u;
            __syncthreads();
        } else {
            // thread tid owns bins [kBinsPerThread tid, kBinsPerThread (tid + 1))
            uint32_t c[kBinsPerThread];
            uint32_t mine = 0u;
            __syncthreads();
#pragma unroll
            for (int x = 0; x < kBinsPerThread; ++x) c[x] = S.hist[kBinsPerThread * tid + x];
#pragma unroll
            for (int x = 0; x < kBinsPerThread; ++x) {
                S.hist[kBinsPerThread * tid + x] = 0u;
                mine += c[x];
            }
            // keys in higher bins = total - inclusive scan in bin order
            const uint32_t incl_w = warp_inclusive_scan(mine);
            if (lane == 31) S.warp_sums[warp] = incl_w;
            __syncthreads();
            if (warp == 0) {
                const uint32_t v = lane < kWarps ? S.warp_sums[lane] : 0u;
                const uint32_t sc = warp_inclusive_scan(v);
                if (lane < kWarps) S.warp_sums[lane] = sc;
                if (lane == kWarps - 1) S.total = sc;
            }
            __syncthreads();
            uint32_t above = S.total - (incl_w + (warp ? S.warp_sums[warp - 1] : 0u));
#pragma unroll
            for (int x = kBinsPerThread - 1; x >= 0; --x) {
                if (above < need && need <= above + c[x]) {
                    S.sel_digit = (uint32_t)(kBinsPerThread * tid + x);
                    S.sel_above = above;
                    S.sel_count = c[x];
                }
                above += c[x];
            }
            __syncthreads();
        }
        need -= S.sel_above;
        prefix |= S.sel_digit << sh;
        pmask |= dmask << sh;
        if (passes > 1 && top > 0 && S.sel_count <= 64u) {
            // at most 64 keys (in the cluster) share the digits found so far:
            // gather them and rank them exactly instead of more passes
            if (tid == 0) S.small_n = 0u;
            __syncthreads();
            visit([&](uint32_t key) {
                if ((key & pmask) == prefix) {
                    const uint32_t at = atomicAdd(&S.small_n, 1u);
                    if (at < 64u) S.small[at] = key;
                }
            });
            if (nranks == 1) __syncthreads();
            else cluster.sync();
            // every rank's list, concatenated in rank order
            auto rank_smem = [&](int r) -> const TopkSmem<NT>* {
                return nranks == 1 ? &S : cluster.map_shared_rank(&S, r);
            };
            if (tid < 64 * nranks) {
                const int r = tid >> 6, e = tid & 63;
                // every rank's list length, loaded at once (predicated)
                uint32_t len[kMaxCluster];
#pragma unroll
                for (int r2 = 0; r2 < kMaxCluster; ++r2)
                    len[r2] = r2 < nranks ? min(rank_smem(min(r2, nranks - 1))->small_n, 64u) : 0u;
                uint32_t off = 0u, mine = 0u, tot = 0u;
#pragma unroll
                for (int r2 = 0; r2 < kMaxCluster; ++r2) {
                    off += r2 < r ? len[r2] : 0u;
                    mine = r2 == r ? len[r2] : mine;
                    tot += len[r2];
                }
                if ((uint32_t)e < mine && off + (uint32_t)e < 64u) S.small_all[off + e] = rank_smem(r)->small[e];
                if (tid == 0) S.small_all_n = min(tot, 64u);
            }
            __syncthreads();
            // thread t ranks key t / 8 against keys 8 (t % 8) .. 8 (t % 8) + 7;
            // eight lanes sum their counts
            if (tid < 512) {
                const uint32_t nb = S.small_all_n;
                const uint32_t q = (uint32_t)tid >> 3, sub = (uint32_t)tid & 7u;
                const uint32_t x = q < nb ? S.small_all[q] : 0u;
                uint32_t gt = 0u, eq = 0u;
#pragma unroll
                for (uint32_t o = 0; o < 8u; ++o) {
                    const uint32_t qq = sub * 8u + o;
                    const uint32_t y = S.small_all[qq];
                    gt += (qq < nb && y > x) ? 1u : 0u;
                    eq += (qq < nb && y == x) ? 1u : 0u;
                }
#pragma unroll
                for (int o = 1; o < 8; o <<= 1) {
                    gt += __shfl_xor_sync(0xffffffffu, gt, o);
                    eq += __shfl_xor_sync(0xffffffffu, eq, o);
                }
                // tau: the key with fewer than `need` larger keys and at least
                // `need` keys at or above it (every such thread agrees)
                if (sub == 0 && q < nb && gt < need && need <= gt + eq) {
                    S.small_tau = x;
                    S.small_need = need - gt;
                }
            }
            __syncthreads();
            prefix = S.small_tau;
            need = S.small_need;
            break;
        }
    }
    need_out = need;
    return prefix;
}

// Number of low bits in which keys of [lo, hi] may differ.
__device__ __forceinline__ int varying_bits(uint32_t lo, uint32_t hi) {
    return lo == hi ? 0 : 32 - __clz((int)(lo ^ hi));
}

// Exclusive prefix over the cluster's lower ranks of the CTA counts (gt, eq)
// stored in S.cta_gt / S.cta_eq; call after a cluster barrier.
template <int NT>
__device__ __forceinline__ void cluster_prefix(cg::cluster_group& cluster, int crank, TopkSmem<NT>& S,
                                               uint32_t& gt0, uint32_t& eq0) {
    // lane r of warp 0 loads lower rank r's counts (one remote read per
    // rank, not one per thread), the warp sums them, the CTA shares them
    if ((threadIdx.x >> 5) == 0) {
        const int r = (int)(threadIdx.x & 31);
        const TopkSmem<NT>* o = cluster.map_shared_rank(&S, (unsigned)min(r, max(crank - 1, 0)));
        uint32_t g = r < crank ? o->cta_gt : 0u, e = r < crank ? o->cta_eq : 0u;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            g += __shfl_xor_sync(0xffffffffu, g, off);
            e += __shfl_xor_sync(0xffffffffu, e, off);
        }
        if (r == 0) {
            S.pre_gt = g;
            S.pre_eq = e;
        }
    }
    __syncthreads();
    gt0 = S.pre_gt;
    eq0 = S.pre_eq;
}

// out[pos] = v for a rank pos < k; a rank outside the row would be a bug:
// it is skipped and latched instead of written.
__device__ __forceinline__ void put(int32_t* out, uint32_t pos, int k, int32_t v, int32_t* status) {
    if (pos < (uint32_t)k) out[pos] = v;
    else latch_status(status, DSA_ERR_INTERNAL);
}

template <int NT>
__global__ void __launch_bounds__(NT, NT <= 512 ? 2 : 1)
    topk_kernel(const BatchDev bd, const RowRange rr, const float* __restrict__ scores, const int64_t ld,
                const int scores_local, const int k, int32_t* __restrict__ idx, const int idx_local,
                const int csize, int32_t* status) {
    constexpr int kThreads = NT, kWarps = NT / 32, kBinsPerThread = kBins / NT;
    extern __shared__ __align__(16) uint8_t smem_raw[];
    TopkSmem<NT>& S = *reinterpret_cast<TopkSmem<NT>*>(smem_raw);
    cg::cluster_group cluster = cg::this_cluster();

    // every test below depends only on the row, so all CTAs of a cluster
    // take the same branch and reach the same cluster barriers
    pdl_launch_dependents();     // a dependent attention may start launching
    pdl_wait();                  // the scores of the previous launch are complete
    const int b = blockIdx.y;
    SeqInfo sq;
    if (!load_seq(bd, b, status, sq)) return;
    const int crank = (int)(blockIdx.x % (unsigned)csize);
    const int32_t i = rr.i0 + (int32_t)(blockIdx.x / (unsigned)csize);
    if (i >= min(rr.i1, sq.nq)) return;
    const int32_t t = sq.ctx - sq.nq + i;
    const int32_t n = t + 1;
    const float* row = scores + buf_row(scores_local, sq, b, i, rr) * ld;
    int32_t* out = idx + buf_row(idx_local, sq, b, i, rr) * (int64_t)k;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // a barrier over every thread that shares this row
    auto sync_row = [&]() {
        if (csize == 1) __syncthreads();
        else cluster.sync();
    };

    if (n <= k) {  // every causal position is selected
        if (crank == 0)
            for (int j = tid; j < k; j += kThreads) out[j] = j < n ? j : -1;
        return;
    }
    auto row_key = [&](int32_t j) -> uint32_t { return order_key(__ldg(row + j)); };

    // this CTA's slice [s_lo, s_hi) of the row (slices start on multiples of 128)
    const int32_t span = ((n + csize - 1) / csize + 127) & ~127;
    const int32_t s_lo = min(n, crank * span), s_hi = min(n, s_lo + span);

    // 1. the lower bound L (the same in every CTA): digits start below the
    // bits that all sample keys share
    const int32_t ns = min(n, kSample);
#pragma unroll
    for (int x = 0; x < kBinsPerThread; ++x) S.hist[kBinsPerThread * tid + x] = 0u;
    uint32_t smin = 0xFFFFFFFFu, smax = 0u;
    for (int q = tid; q < ns; q += kThreads) {
        const uint32_t key = row_key((int32_t)(((int64_t)q * n) / ns));
        S.sample[q] = key;
        smin = min(smin, key);
        smax = max(smax, key);
    }
    smin = __reduce_min_sync(0xffffffffu, smin);
    smax = __reduce_max_sync(0xffffffffu, smax);
    if (lane == 0) {
        S.wgt[warp] = smin;
        S.weq[warp] = smax;
    }
    __syncthreads();
    smin = __reduce_min_sync(0xffffffffu, lane < kWarps ? S.wgt[lane] : 0xFFFFFFFFu);
    smax = __reduce_max_sync(0xffffffffu, lane < kWarps ? S.weq[lane] : 0u);
    const float expect = (float)k * (float)ns / (float)n;
    const int32_t r = min(ns - 1, (int32_t)(1.25f * expect + 3.f * sqrtf(expect)) + 8);
    uint32_t unused;
    const uint32_t L = radix_select(cluster, 1, S, (uint32_t)(r + 1), varying_bits(smin, smax), smin, 1,
                                    [&](auto&& f) {
                                        for (int q = tid; q < ns; q += kThreads) f(S.sample[q]);
                                    },
                                    unused);

    // 2. one pass: warp w appends its keys >= L to its region, in position
    // order.  A step covers 128 x kPrefetch consecutive keys: lane l loads
    // the 16-byte groups l, l + 32, ... (coalesced, all in flight at once).
    // Keys are tested as floats against the float of L (the same order as
    // the keys, -0.0 == +0.0).  The per-group candidate counts of a lane
    // travel through one 64-bit warp scan (8-bit fields), which places every
    // candidate of the step in position order; their keys are read again
    // after the pass.
    const int32_t seg = ((s_hi - s_lo + kWarps - 1) / kWarps + 127) & ~127;
    const int32_t w_lo = min(s_hi, s_lo + warp * seg), w_hi = min(s_hi, w_lo + seg);
    uint32_t* rk = S.cand_key + warp * kRegion;
    int32_t* rp = S.cand_pos + warp * kRegion;
    const float Lf = key_float(L);
    uint32_t cnt = 0u;
    float fmx = -INFINITY;
    for (int32_t jb = w_lo; jb < w_hi; jb += 128 * kPrefetch) {
        float4 v[kPrefetch];
#pragma unroll
        for (int u = 0; u < kPrefetch; ++u) {
            const int32_t j = jb + 128 * u + 4 * (int32_t)lane;   // a multiple of 4 inside the padded row
            v[u] = j < w_hi ? __ldg(reinterpret_cast<const float4*>(row + j)) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        const bool tail = jb + 128 * kPrefetch > w_hi;    // warp-uniform
        uint32_t bits = 0u;                               // bit 4u + e: key jb + 128u + 4 lane + e
        uint64_t packed = 0u;
#pragma unroll
        for (int u = 0; u < kPrefetch; ++u) {
            float x[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
            uint32_t bu = 0u;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                bool c = x[e] >= Lf;
                if (tail) {
                    const bool in = jb + 128 * u + 4 * (int32_t)lane + e < w_hi;
                    c = c && in;
                    x[e] = in ? x[e] : -INFINITY;        // for the max only
                }
                bu |= (c ? 1u : 0u) << e;
                fmx = fmaxf(fmx, x[e]);
            }
            bits |= bu << (4 * u);
            packed |= (uint64_t)__popc(bu) << (8 * u);
        }
        uint64_t incl = packed;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint64_t nb = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += nb;
        }
        const uint64_t tot = __shfl_sync(0xffffffffu, incl, 31);
        uint32_t base = cnt;
#pragma unroll
        for (int u = 0; u < kPrefetch; ++u) {
            uint32_t at = base + ((uint32_t)((incl - packed) >> (8 * u)) & 0xFFu);
            for (uint32_t bb = (bits >> (4 * u)) & 0xFu; bb; bb &= bb - 1u) {
                const int32_t j = jb + 128 * u + 4 * (int32_t)lane + (int32_t)(__ffs(bb) - 1);
                if (at < (uint32_t)kRegion) rp[at] = j;
                ++at;
            }
            base += (uint32_t)(tot >> (8 * u)) & 0xFFu;
        }
        cnt = base;
    }
    // the candidates' keys, re-read (L1 or L2 hits) once the pass is done:
    // independent loads, many in flight (reading each as it was appended put
    // one round trip per candidate on the pass: 7 K of its ~12 K cycles in a
    // decode row)
    __syncwarp();
    {
        const uint32_t n = min(cnt, (uint32_t)kRegion);
#pragma unroll 4
        for (uint32_t s = lane; s < n; s += 32) rk[s] = row_key(rp[s]);
    }
    // an upper bound of the candidates (keys of the slice, -inf when empty)
    uint32_t cmax = fmx >= Lf ? order_key(fmx) : 0u;
    cmax = __reduce_max_sync(0xffffffffu, cmax);
    if (lane == 0) {
        S.wcnt[warp] = cnt;
        S.wmax[warp] = cmax;
    }
    __syncthreads();
    if (warp == 0) {
        const uint32_t c = lane < kWarps ? S.wcnt[lane] : 0u;
        const uint32_t tot = warp_inclusive_scan(c);
        const bool overflow = __any_sync(0xffffffffu, c > (uint32_t)kRegion);
        const uint32_t mx = __reduce_max_sync(0xffffffffu, lane < kWarps ? S.wmax[lane] : 0u);
        if (lane == 31) {
            S.cta_cand = tot;
            S.cta_overflow = overflow ? 1u : 0u;
            S.cta_max = mx;
        }
    }
    sync_row();
    uint32_t all_cand = 0u, any_overflow = 0u, all_max = 0u;
    if (csize == 1) {
        all_cand = S.cta_cand;
        any_overflow = S.cta_overflow;
        all_max = S.cta_max;
    } else {
        // lane q of warp 0 loads rank q's counts (one remote read per rank,
        // not one per thread), the warp combines them, the CTA shares them
        if (warp == 0) {
            const int q = lane;
            const TopkSmem<NT>* o = cluster.map_shared_rank(&S, (unsigned)min(q, csize - 1));
            uint32_t cc = q < csize ? o->cta_cand : 0u, co = q < csize ? o->cta_overflow : 0u,
                     cm = q < csize ? o->cta_max : 0u;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                cc += __shfl_xor_sync(0xffffffffu, cc, off);
                co |= __shfl_xor_sync(0xffffffffu, co, off);
                cm = max(cm, __shfl_xor_sync(0xffffffffu, cm, off));
            }
            if (lane == 0) {
                S.all_cand = cc;
                S.all_overflow = co;
                S.all_max = cm;
            }
        }
        __syncthreads();
        all_cand = S.all_cand;
        any_overflow = S.all_overflow;
        all_max = S.all_max;
    }
    const bool use_candidates = !any_overflow && all_cand >= (uint32_t)k;

    uint32_t need;
    if (use_candidates) {
        // 3. tau among the cluster's candidates; every candidate lies in
        // [L, all_max], so the bits the two share are known
        const uint32_t tau = radix_select(cluster, csize, S, (uint32_t)k, varying_bits(L, all_max), L, 3,
                                          [&](auto&& f) {
                                              const uint32_t c = S.wcnt[warp];
                                              for (uint32_t s = lane; s < c; s += 32) f(rk[s]);
                                          },
                                          need);
        // 4. ordered output: counts per warp, prefix over warps and lower CTAs
        const uint32_t c = S.wcnt[warp];
        uint32_t g = 0u, e = 0u;
        for (uint32_t s0 = 0; s0 < c; s0 += 32) {
            const uint32_t s = s0 + lane;
            const uint32_t key = s < c ? rk[s] : 0u;
            g += __popc(__ballot_sync(0xffffffffu, s < c && key > tau));
            e += __popc(__ballot_sync(0xffffffffu, s < c && key == tau));
        }
        if (lane == 0) {
            S.wgt[warp] = g;
            S.weq[warp] = e;
        }
        __syncthreads();
        if (warp == 0) {
            const uint32_t gv = lane < kWarps ? S.wgt[lane] : 0u, ev = lane < kWarps ? S.weq[lane] : 0u;
            const uint32_t gi = warp_inclusive_scan(gv);
            const uint32_t ei = warp_inclusive_scan(ev);
            if (lane < kWarps) {
                S.wgt[lane] = gi - gv;
                S.weq[lane] = ei - ev;
            }
            if (lane == 31) {
                S.cta_gt = gi;
                S.cta_eq = ei;
            }
        }
        sync_row();
        uint32_t gt0, eq0;
        cluster_prefix(cluster, crank, S, gt0, eq0);
        uint32_t gt_run = gt0 + S.wgt[warp], eq_run = eq0 + S.weq[warp];
        const uint32_t lower = (1u << lane) - 1u;
        for (uint32_t s0 = 0; s0 < c; s0 += 32) {
            const uint32_t s = s0 + lane;
            const uint32_t key = s < c ? rk[s] : 0u;
            const bool isg = s < c && key > tau, ise = s < c && key == tau;
            const uint32_t bg = __ballot_sync(0xffffffffu, isg), be = __ballot_sync(0xffffffffu, ise);
            const uint32_t gtb = gt_run + __popc(bg & lower), eqb = eq_run + __popc(be & lower);
            if (isg) put(out, gtb + min(eqb, need), k, rp[s], status);
            else if (ise && eqb < need) put(out, gtb + eqb, k, rp[s], status);
            gt_run += __popc(bg);
            eq_run += __popc(be);
        }
    } else {
        // the sample misjudged: select and write over the whole slices
        const int32_t len = s_hi - s_lo;
        auto slice_key = [&](int32_t j) -> uint32_t { return row_key(s_lo + j); };
        const uint32_t tau = radix_select(cluster, csize, S, (uint32_t)k, 32, 0u, 3,
                                          [&](auto&& f) {
                                              for (int32_t j = tid; j < len; j += kThreads) f(slice_key(j));
                                          },
                                          need);
        uint32_t g = 0u, e = 0u;
        for (int32_t j = tid; j < len; j += kThreads) {
            const uint32_t key = slice_key(j);
            g += key > tau;
            e += key == tau;
        }
        const uint32_t gw = warp_inclusive_scan(g), ew = warp_inclusive_scan(e);
        if (lane == 31) {
            S.wgt[warp] = gw;
            S.weq[warp] = ew;
        }
        __syncthreads();
        if (warp == 0) {
            const uint32_t gs = warp_inclusive_scan(lane < kWarps ? S.wgt[lane] : 0u);
            const uint32_t es = warp_inclusive_scan(lane < kWarps ? S.weq[lane] : 0u);
            if (lane == 31) {
                S.cta_gt = gs;
                S.cta_eq = es;
            }
        }
        sync_row();
        uint32_t gt_run, eq_run;
        cluster_prefix(cluster, crank, S, gt_run, eq_run);
        constexpr int kE = 4;
#pragma unroll 1
        for (int32_t base = 0; base < len; base += kThreads * kE) {
            const int32_t j0 = base + tid * kE;
            uint32_t kk[kE];
            uint32_t gc = 0u, ec = 0u;
#pragma unroll
            for (int x = 0; x < kE; ++x) {
                kk[x] = j0 + x < len ? slice_key(j0 + x) : 0u;
                if (j0 + x < len) {
                    gc += kk[x] > tau;
                    ec += kk[x] == tau;
                }
            }
            const uint32_t wi = warp_inclusive_scan(gc | (ec << 16));
            if (lane == 31) S.warp_sums[warp] = wi;
            __syncthreads();
            if (warp == 0) {
                const uint32_t s = warp_inclusive_scan(lane < kWarps ? S.warp_sums[lane] : 0u);
                if (lane < kWarps) S.warp_sums[lane] = s;
                if (lane == kWarps - 1) S.chunk_total = s;
            }
            __syncthreads();
            const uint32_t packed = wi + (warp ? S.warp_sums[warp - 1] : 0u);
            uint32_t gtb = gt_run + (packed & 0xFFFFu) - gc;
            uint32_t eqb = eq_run + (packed >> 16) - ec;
#pragma unroll
            for (int x = 0; x < kE; ++x) {
                if (j0 + x < len) {
                    if (kk[x] > tau) {
                        put(out, gtb + min(eqb, need), k, s_lo + j0 + x, status);
                        ++gtb;
                    } else if (kk[x] == tau) {
                        if (eqb < need) put(out, gtb + eqb, k, s_lo + j0 + x, status);
                        ++eqb;
                    }
                }
            }
            gt_run += S.chunk_total & 0xFFFFu;
            eq_run += S.chunk_total >> 16;
            __syncthreads();
        }
    }
    if (csize > 1) cluster.sync();                 // the cluster may still read this CTA's counts
}

template <int NT>
cudaError_t launch_nt(const BatchDev& bd, RowRange rr, const float* scores, int64_t ld, bool scores_local, int k,
                      int32_t* idx, bool idx_local, int csize, int32_t rows_per_seq, int32_t* status,
                      cudaStream_t stream, bool after_previous) {
    const size_t smem = sizeof(TopkSmem<NT>);
    cudaError_t e = cudaFuncSetAttribute(topk_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(rows_per_seq * csize), (unsigned)bd.B);
    cfg.blockDim = dim3(NT);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)csize;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = after_previous ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    e = cudaLaunchKernelEx(&cfg, topk_kernel<NT>, bd, rr, scores, ld, scores_local ? 1 : 0, k, idx,
                           idx_local ? 1 : 0, csize, status);
    if (e == cudaSuccess) count_launches(1);
    return e;
}

}  // namespace

cudaError_t launch_topk(const BatchDev& bd, RowRange rr, const float* scores, int64_t ld, bool scores_local,
                        int k, int32_t* idx, bool idx_local, int32_t* status, cudaStream_t stream,
                        bool after_previous) {
    const int32_t rows_per_seq = min(rr.i1, bd.max_q) - rr.i0;
    if (rows_per_seq <= 0) return cudaSuccess;
    // long rows, few of them: split each row over a cluster
    const int64_t rows = (int64_t)rows_per_seq * bd.B;
    int csize = 1;
    if (bd.max_ctx > kLongRow && rows < 2 * num_sms())
        csize = (int)std::min<int64_t>(kMaxCluster, ((int64_t)bd.max_ctx + kKeysPerCta - 1) / kKeysPerCta);
    return rows < num_sms() ? launch_nt<1024>(bd, rr, scores, ld, scores_local, k, idx, idx_local, csize, rows_per_seq,
                                            status, stream, after_previous)
                          : launch_nt<512>(bd, rr, scores, ld, scores_local, k, idx, idx_local, csize, rows_per_seq,
                                           status, stream, after_previous);
}

}  // namespace dsa
