// noalloc.cu -- mnb_run_noalloc: the LoRA path without a caller-provided T
// scratch buffer, for callers that cannot allocate device memory.
//
// mnb_run needs scratch memory for T = X * A ([batch*M, 32] FP16) when an
// adapter is given, and asks the caller for it.  Some callers cannot provide
// it: code hosted inside a runtime that owns every device allocation and
// gives plugins no allocator, or latency-critical loops where cudaMalloc and
// cudaFree are forbidden because they can synchronize the whole device.  This
// entry point keeps T in a fixed array in the library's own device memory
// instead, so it allocates nothing.
//
// The array holds at most kNoallocMaxRows token rows (batch * M); every GPU
// that loads the library keeps it (kNoallocMaxRows * 32 * 2 bytes = 512 KiB)
// until the process exits.  All calls share it: two calls whose kernels
// overlap on the GPU (different streams, or different host threads without
// ordering) race on it.  T is written in full before it is read, so nothing
// needs clearing between calls.
//
// Validation and results are those of mnb_run (the shared run path in api.cu
// resolves the scratch address after its own argument checks and device
// setup); the only difference is the row limit.
#include <mutex>

#include "mnb_internal.h"

namespace {

constexpr int kMaxDevices = 64;

// The scratch itself.  In host code this name is only a stand-in for the
// device symbol; its device address is fetched with cudaGetSymbolAddress.
static __device__ __align__(256) __half g_noalloc_T[mnb::kNoallocMaxRows * 32];

std::mutex g_mu;
// Per device: the context the address below belongs to (0 = none yet).  A
// symbol's address is valid only in the context that loaded the module, so it
// is looked up again when the device's current context changes.
unsigned long long g_T_ctx[kMaxDevices] = {};
__half* g_T_addr[kMaxDevices] = {};

}  // namespace

namespace mnb {

int noalloc_scratch(__half** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return MNB_ERR_NO_DEVICE;
    }
    unsigned long long ctx = 0;
    if (current_context_id(&ctx) != cudaSuccess) return MNB_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_T_ctx[dev] != ctx || !g_T_addr[dev]) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_T);
        if (e != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return MNB_ERR_CUDA;
        }
        g_T_addr[dev] = static_cast<__half*>(p);
        g_T_ctx[dev] = ctx;
    }
    *out = g_T_addr[dev];
    return MNB_OK;
}

}  // namespace mnb

extern "C" int mnb_run_noalloc(mnb_handle h, const void* X, const void* Wq, const void* scales, const void* zp,
                               const void* A, const void* B, int32_t rank, void* Y, int64_t batch, int64_t M,
                               void* stream) {
    return mnb::run_noalloc(h, X, Wq, scales, zp, A, B, rank, Y, batch, M, stream);
}

extern "C" int64_t mnb_noalloc_max_rows(void) { return mnb::kNoallocMaxRows; }
