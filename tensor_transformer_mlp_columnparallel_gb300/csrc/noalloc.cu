// tpmlp_forward_noalloc: the PARTIALS forward with its scratch (the T fp32
// partial sums that the row GEMM writes and the block-end reduce reads) in a
// fixed array of device memory that belongs to this library, so the caller
// needs neither cudaMalloc nor a workspace.
//
// Who needs it: callers that own no allocator, or may not use one on this
// path, e.g. a plug-in running inside a host program that hands out all
// device memory itself, or a latency-critical loop that must not risk the
// implicit device synchronisation or the failure of a cudaMalloc.
//
// The array is file-scope static device memory of TPMLP_NOALLOC_SCRATCH_BYTES.
// Every GPU that loads the library holds it until the process exits. Host code
// may not use the array's name as a device address, so the first call on each
// device asks the runtime for the address (cudaGetSymbolAddress, with that
// device current) and caches it; that first call should come before any
// stream capture.
#include <cuda_runtime.h>

#include <mutex>

#include "tpmlp_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[TPMLP_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set up once per
// device); NULL if the runtime cannot provide it.
void* scratch_on_current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_scratch_ptr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
        g_scratch_ptr[dev] = p;
    }
    return g_scratch_ptr[dev];
}

}  // namespace

extern "C" tpmlp_status tpmlp_forward_noalloc(tpmlp_dtype dt, int64_t N, int64_t D, int64_t F,
                                              int T, tpmlp_act act, const void* X,
                                              const void* const* W1, const void* const* b1,
                                              const void* const* W2, const void* b2, void* Y,
                                              void* const* H, void* const* Z, void* stream) {
    const size_t need =
        tpmlp_workspace_bytes(TPMLP_OP_FORWARD, dt, N, D, F, T, TPMLP_REDUCE_PARTIALS);
    if (need == (size_t)-1) return TPMLP_ERR_SHAPE;
    if (need > (size_t)TPMLP_NOALLOC_SCRATCH_BYTES) return TPMLP_ERR_WORKSPACE;
    void* scratch = nullptr;
    if (N > 0) {
        scratch = scratch_on_current_device();
        if (scratch == nullptr) return TPMLP_ERR_CUDA;
    }
    // The row GEMM overwrites every element of each partial before the reduce
    // reads it, so nothing left in the array by an earlier call is used.
    return tpmlp_forward(dt, N, D, F, T, act, X, W1, b1, W2, b2, Y, H, Z, TPMLP_REDUCE_PARTIALS,
                         scratch, TPMLP_NOALLOC_SCRATCH_BYTES, stream);
}
