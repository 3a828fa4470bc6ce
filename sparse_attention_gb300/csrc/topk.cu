// topk.cu -- deterministic causal top-k of indexer score rows.
//
// ("GLM-5.1 架构深度拆解", section 3.6 Steps 6-7: positions s > t are masked
// and min(index_topk, length) positions are kept; section 3.4: the
// selection must be deterministic; the GLM-5 explainer page: a query that
// sees fewer than 2048 positions keeps all of them.)
//
// One CTA per query row.  Scores map to order-preserving 32-bit keys (-0.0
// folded onto +0.0).  The selection is:
//   1. a lower bound L for the k-th largest key: the lower edge of the
//      leading-digit bin (top 11 bits) holding the (r+1)-th largest of 1024
//      evenly spaced keys, r sized so that well over k keys of the row lie
//      at or above it;
//   2. one pass over the row (16-byte loads): warp w owns a contiguous
//      segment and appends its keys >= L, in position order, to a region of
//      shared memory of its own (warp scans give the slots);
//   3. the exact k-th largest key tau among these candidates by a radix
//      select over three digits (11 + 11 + 10 bits), shared-memory
//      histograms restricted to the keys matching the digits found so far;
//   4. the output, warp by warp in position order: candidates above tau,
//      and the first `need` candidates equal to tau (ties go to the lower
//      position), each written at its rank; positions come out ascending.
// Every key that is not a candidate lies below L <= tau, so the result is
// exactly the top-k of the row.  When the sample misjudges (fewer than k
// candidates, or a warp's region overflows) the same select and an ordered
// output run over the whole row.  Atomics only count, so the result is the
// same bit for bit on every run.
#include <algorithm>

#include "internal.h"

namespace dsa {
namespace {

constexpr int kThreads = 512;                // two CTAs per SM
constexpr int kWarps = kThreads / 32;
constexpr int kBins = 2048;
constexpr int kBinsPerThread = kBins / kThreads;
constexpr int kSample = 1024;
constexpr int kRegion = 512;                 // candidate slots per warp
constexpr int kMaxCand = kWarps * kRegion;   // 8192
constexpr int kPrefetch = 6;                 // 16-byte loads in flight per lane

__device__ __forceinline__ uint32_t order_key(float f) {
    uint32_t u = __float_as_uint(f);
    if (u == 0x80000000u) u = 0u;     // -0.0 compares equal to +0.0
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
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

struct alignas(16) TopkSmem {
    uint32_t hist[kBins];                 // zero between selects
    uint32_t sample[kSample];
    uint32_t cand_key[kMaxCand];          // warp w: [w * kRegion, w * kRegion + count)
    int32_t cand_pos[kMaxCand];
    uint32_t warp_sums[32];
    uint32_t wcnt[32], wgt[32], weq[32];
    uint32_t total, sel_digit, sel_above, ok, chunk_total;
};

// The k-th largest of the keys j in [0, m) with valid_of(j), resolved to the
// first `passes` digits (3 = exact): returns tau (the digits found, zero
// below them) and sets need = how many keys matching tau belong to the top
// k.  S.hist must be zero on entry and is zero on return.  Four barriers
// per digit.
template <typename KeyOf, typename ValidOf>
__device__ uint32_t radix_select(TopkSmem& S, int32_t m, uint32_t k, int passes, KeyOf key_of, ValidOf valid_of,
                                 uint32_t& need_out) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint32_t prefix = 0u, pmask = 0u, need = k;
#pragma unroll 1
    for (int p = 0; p < passes; ++p) {
        const int sh = p == 0 ? 21 : (p == 1 ? 10 : 0);
        const uint32_t dmask = p == 2 ? 0x3FFu : 0x7FFu;
        for (int32_t j = tid; j < m; j += kThreads) {
            if (!valid_of(j)) continue;
            const uint32_t key = key_of(j);
            if ((key & pmask) == prefix) atomicAdd(&S.hist[(key >> sh) & dmask], 1u);
        }
        __syncthreads();
        // thread tid owns bins [4 tid, 4 tid + 4) (read, then cleared for
        // the next digit); keys in higher bins = total - inclusive scan
        uint32_t c[kBinsPerThread];
        uint32_t mine = 0u;
#pragma unroll
        for (int x = 0; x < kBinsPerThread; ++x) {
            c[x] = S.hist[kBinsPerThread * tid + x];
            S.hist[kBinsPerThread * tid + x] = 0u;
            mine += c[x];
        }
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
        uint32_t above = S.total - (incl_w + (warp ? S.warp_sums[warp - 1] : 0u));   // bins above this thread's
#pragma unroll
        for (int x = kBinsPerThread - 1; x >= 0; --x) {
            if (above < need && need <= above + c[x]) {
                S.sel_digit = (uint32_t)(kBinsPerThread * tid + x);
                S.sel_above = above;
            }
            above += c[x];
        }
        __syncthreads();
        need -= S.sel_above;
        prefix |= S.sel_digit << sh;
        pmask |= dmask << sh;
    }
    need_out = need;
    return prefix;
}

__global__ void __launch_bounds__(kThreads, 2)
    topk_kernel(const BatchDev bd, const RowRange rr, const float* __restrict__ scores, const int64_t ld,
                const int scores_local, const int k, int32_t* __restrict__ idx, const int idx_local,
                int32_t* status) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    TopkSmem& S = *reinterpret_cast<TopkSmem*>(smem_raw);

    const int b = blockIdx.y;
    SeqInfo sq;
    if (!load_seq(bd, b, status, sq)) return;
    const int32_t i = rr.i0 + (int32_t)blockIdx.x;
    if (i >= min(rr.i1, sq.nq)) return;
    const int32_t t = sq.ctx - sq.nq + i;
    const int32_t n = t + 1;
    const float* row = scores + buf_row(scores_local, sq, b, i, rr) * ld;
    int32_t* out = idx + buf_row(idx_local, sq, b, i, rr) * (int64_t)k;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    if (n <= k) {  // every causal position is selected
        for (int j = tid; j < k; j += kThreads) out[j] = j < n ? j : -1;
        return;
    }
    auto row_key = [&](int32_t j) -> uint32_t { return order_key(__ldg(row + j)); };

    // 1. the lower bound L: the smallest key of the leading-digit bin that
    //    holds the (r+1)-th largest sampled key
    const int32_t ns = min(n, kSample);
#pragma unroll
    for (int x = 0; x < kBinsPerThread; ++x) S.hist[kBinsPerThread * tid + x] = 0u;
    for (int q = tid; q < ns; q += kThreads) S.sample[q] = row_key((int32_t)(((int64_t)q * n) / ns));
    __syncthreads();
    const float expect = (float)k * (float)ns / (float)n;
    const int32_t r = min(ns - 1, (int32_t)(1.25f * expect + 3.f * sqrtf(expect)) + 8);
    uint32_t unused;
    const uint32_t L = radix_select(
        S, ns, (uint32_t)(r + 1), 1, [&](int32_t j) { return S.sample[j]; }, [](int32_t) { return true; }, unused);

    // 2. one pass: warp w appends its keys >= L to its region, in order
    const int32_t seg = ((n + kWarps - 1) / kWarps + 127) & ~127;
    const int32_t w_lo = min(n, warp * seg), w_hi = min(n, w_lo + seg);
    uint32_t* rk = S.cand_key + warp * kRegion;
    int32_t* rp = S.cand_pos + warp * kRegion;
    uint32_t cnt = 0u;
    for (int32_t jb = w_lo; jb < w_hi; jb += 128 * kPrefetch) {
        float4 v[kPrefetch];
#pragma unroll
        for (int u = 0; u < kPrefetch; ++u) {       // all loads in flight before any use
            const int32_t j = jb + 128 * u + 4 * lane;
            v[u] = j < w_hi ? __ldg(reinterpret_cast<const float4*>(row + j)) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < kPrefetch; ++u) {
            const int32_t j = jb + 128 * u + 4 * lane;   // a multiple of 4 inside the padded row
            const uint32_t kk[4] = {order_key(v[u].x), order_key(v[u].y), order_key(v[u].z), order_key(v[u].w)};
            uint32_t mine = 0u;
#pragma unroll
            for (int x = 0; x < 4; ++x) mine += (j + x < w_hi && kk[x] >= L) ? 1u : 0u;
            const uint32_t incl = warp_inclusive_scan(mine);
            uint32_t at = cnt + incl - mine;
#pragma unroll
            for (int x = 0; x < 4; ++x) {
                if (j + x < w_hi && kk[x] >= L) {
                    if (at < (uint32_t)kRegion) {
                        rk[at] = kk[x];
                        rp[at] = j + x;
                    }
                    ++at;
                }
            }
            cnt += __shfl_sync(0xffffffffu, incl, 31);
        }
    }
    if (lane == 0) S.wcnt[warp] = cnt;
    __syncthreads();
    if (warp == 0) {
        const uint32_t c = lane < kWarps ? S.wcnt[lane] : 0u;
        const uint32_t tot = warp_inclusive_scan(c);
        const bool overflow = __any_sync(0xffffffffu, c > (uint32_t)kRegion);
        if (lane == 31) S.ok = (!overflow && tot >= (uint32_t)k) ? 1u : 0u;
    }
    __syncthreads();

    uint32_t need;
    if (S.ok) {
        // 3. tau among the candidates (slots past a region's count are empty)
        const uint32_t tau = radix_select(
            S, kMaxCand, (uint32_t)k, 3, [&](int32_t j) { return S.cand_key[j]; },
            [&](int32_t j) { return (uint32_t)(j % kRegion) < S.wcnt[j / kRegion]; }, need);
        // 4. ordered output: counts per warp region, prefix over warps, write
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
        }
        __syncthreads();
        uint32_t gt_run = S.wgt[warp], eq_run = S.weq[warp];
        const uint32_t lower = (1u << lane) - 1u;
        for (uint32_t s0 = 0; s0 < c; s0 += 32) {
            const uint32_t s = s0 + lane;
            const uint32_t key = s < c ? rk[s] : 0u;
            const bool isg = s < c && key > tau, ise = s < c && key == tau;
            const uint32_t bg = __ballot_sync(0xffffffffu, isg), be = __ballot_sync(0xffffffffu, ise);
            const uint32_t gtb = gt_run + __popc(bg & lower), eqb = eq_run + __popc(be & lower);
            if (isg) out[gtb + min(eqb, need)] = rp[s];
            else if (ise && eqb < need) out[gtb + eqb] = rp[s];
            gt_run += __popc(bg);
            eq_run += __popc(be);
        }
    } else {
        // the sample misjudged: select and write over the whole row
        const uint32_t tau = radix_select(S, n, (uint32_t)k, 3, row_key, [](int32_t) { return true; }, need);
        uint32_t gt_run = 0u, eq_run = 0u;
        constexpr int kE = 4;
#pragma unroll 1
        for (int32_t base = 0; base < n; base += kThreads * kE) {
            const int32_t j0 = base + tid * kE;
            uint32_t kk[kE];
            uint32_t g = 0u, e = 0u;
#pragma unroll
            for (int x = 0; x < kE; ++x) {
                kk[x] = j0 + x < n ? row_key(j0 + x) : 0u;
                if (j0 + x < n) {
                    g += kk[x] > tau;
                    e += kk[x] == tau;
                }
            }
            const uint32_t wi = warp_inclusive_scan(g | (e << 16));
            if (lane == 31) S.warp_sums[warp] = wi;
            __syncthreads();
            if (warp == 0) {
                const uint32_t s = warp_inclusive_scan(lane < kWarps ? S.warp_sums[lane] : 0u);
                if (lane < kWarps) S.warp_sums[lane] = s;
                if (lane == kWarps - 1) S.chunk_total = s;
            }
            __syncthreads();
            const uint32_t packed = wi + (warp ? S.warp_sums[warp - 1] : 0u);
            uint32_t gtb = gt_run + (packed & 0xFFFFu) - g;
            uint32_t eqb = eq_run + (packed >> 16) - e;
#pragma unroll
            for (int x = 0; x < kE; ++x) {
                if (j0 + x < n) {
                    if (kk[x] > tau) {
                        out[gtb + min(eqb, need)] = j0 + x;
                        ++gtb;
                    } else if (kk[x] == tau) {
                        if (eqb < need) out[gtb + eqb] = j0 + x;
                        ++eqb;
                    }
                }
            }
            gt_run += S.chunk_total & 0xFFFFu;
            eq_run += S.chunk_total >> 16;
            __syncthreads();
        }
    }
}

}  // namespace

cudaError_t launch_topk(const BatchDev& bd, RowRange rr, const float* scores, int64_t ld, bool scores_local,
                        int k, int32_t* idx, bool idx_local, int32_t* status, cudaStream_t stream) {
    const int32_t rows_per_seq = min(rr.i1, bd.max_q) - rr.i0;
    if (rows_per_seq <= 0) return cudaSuccess;
    const size_t smem = sizeof(TopkSmem);
    cudaError_t e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)rows_per_seq, (unsigned)bd.B);
    topk_kernel<<<grid, kThreads, smem, stream>>>(bd, rr, scores, ld, scores_local ? 1 : 0, k, idx,
                                                  idx_local ? 1 : 0, status);
    e = cudaGetLastError();
    if (e == cudaSuccess) count_launches(1);
    return e;
}

}  // namespace dsa
