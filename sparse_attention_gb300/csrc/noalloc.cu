// noalloc.cu -- dsa_sparse_mla_fwd_noalloc: sparse MLA attention for callers
// that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at the point where they run attention:
// serving loops that plan every byte of device memory in advance and treat
// any allocation as a failure, or embedders (a host runtime, a plugin) whose
// allocator is not reachable from the thread that calls attention.  dsa_sparse_mla_fwd needs a caller-provided workspace for its
// split-K partials; this entry point instead keeps them in one fixed-size
// array of static device memory that the library owns.  Every GPU that loads
// the library holds the array (kNoAllocScratchBytes) until the process exits.
#include <mutex>

#include "internal.h"

namespace dsa {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;   // 32 MiB
constexpr int kMaxDevices = 64;

// Split-K partials of dsa_sparse_mla_fwd_noalloc.  Shared by every call on a
// device; a call overwrites every partial it later reads, so nothing needs
// clearing between calls.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the array on the current device, looked up once per
// device (the name is only a host-side stand-in for the array).  The cached
// address belongs to the device's primary context: after cudaDeviceReset
// the array is loaded again elsewhere, so this call is not usable after a
// reset in the same process.
cudaError_t scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace dsa

using namespace dsa;

extern "C" {

dsa_status dsa_sparse_mla_fwd_noalloc(const dsa_batch* batch, const uint16_t* q, const uint16_t* kv,
                                      const int32_t* idx, int k, float sm_scale, uint16_t* out, float* lse,
                                      int32_t* device_status, void* stream) {
    if (!batch) return DSA_ERR_INVALID_ARG;
    if (batch->batch < 1 || batch->batch > 65535 || batch->total_q < 0 || batch->max_q < 0 || batch->max_ctx < 0)
        return DSA_ERR_INVALID_ARG;
    if (batch->max_q > (1 << 19) || batch->total_q >= (1 << 26)) return DSA_ERR_UNSUPPORTED;
    if (batch->cache_stride < batch->max_ctx) return DSA_ERR_INVALID_ARG;
    if ((int64_t)batch->batch * batch->cache_stride >= (int64_t(1) << 31)) return DSA_ERR_UNSUPPORTED;
    if (!batch->q_off || !batch->ctx_len) return DSA_ERR_INVALID_ARG;
    if (k < 1 || k > kMaxTopk) return DSA_ERR_INVALID_ARG;
    if (batch->total_q == 0 || batch->max_q == 0) return DSA_OK;
    if (!q || !kv || !idx || !out) return DSA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(kv) || !aligned16(idx) || !aligned16(out) || (lse && !aligned16(lse)))
        return DSA_ERR_INVALID_ARG;
    if (!(sm_scale > 0.f) || sm_scale == INFINITY) return DSA_ERR_INVALID_ARG;
    const BatchDev bd{batch->batch, batch->total_q, batch->max_q, batch->max_ctx, batch->cache_stride,
                      batch->q_off, batch->ctx_len};
    const size_t need = sparse_mla_scratch_bytes(bd, batch->max_q, k);
    if (need > kNoAllocScratchBytes) return DSA_ERR_WORKSPACE;     // more partials than the static array holds
    void* scratch = nullptr;
    cudaError_t e = scratch_address(&scratch);
    if (e == cudaSuccess)
        e = launch_sparse_mla(bd, RowRange{0, batch->max_q}, q, kv, idx, false, k, sm_scale, out, lse, scratch,
                              kNoAllocScratchBytes, device_status, static_cast<cudaStream_t>(stream));
    return cuda_status(e);
}

}  // extern "C"
