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
#include <mutex>

#include "mnb_internal.h"

namespace {

constexpr int64_t kNoallocMaxRows = 8192;
constexpr int kMaxDevices = 64;

// The scratch itself.  In host code this name is only a stand-in for the
// device symbol; its device address is fetched with cudaGetSymbolAddress.
static __device__ __align__(256) __half g_noalloc_T[kNoallocMaxRows * 32];

std::mutex g_mu;
__half* g_T_addr[kMaxDevices] = {};

// Device address of the scratch on the current device (looked up once per device).
int scratch_address(__half** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return MNB_ERR_NO_DEVICE;
    }
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_T_addr[dev]) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_T);
        if (e != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return MNB_ERR_CUDA;
        }
        g_T_addr[dev] = static_cast<__half*>(p);
    }
    *out = g_T_addr[dev];
    return MNB_OK;
}

}  // namespace

extern "C" int mnb_run_noalloc(mnb_handle h, const void* X, const void* Wq, const void* scales, const void* zp,
                               const void* A, const void* B, int32_t rank, void* Y, int64_t batch, int64_t M,
                               void* stream) {
    if (!h || batch < 0 || M < 0) return MNB_ERR_ARG;
    if (batch > 0 && M > INT64_MAX / batch) return MNB_ERR_UNSUPPORTED;
    const bool adapter = rank != 0 && (A != nullptr || B != nullptr);
    if (!adapter) return mnb_run(h, X, Wq, scales, zp, A, B, rank, Y, nullptr, batch, M, stream);
    if (batch * M > kNoallocMaxRows) return MNB_ERR_UNSUPPORTED;  // beyond the fixed scratch
    __half* T = nullptr;
    if (batch * M > 0) {
        const int rc = scratch_address(&T);
        if (rc != MNB_OK) return rc;
    }
    return mnb_run(h, X, Wq, scales, zp, A, B, rank, Y, T, batch, M, stream);
}

extern "C" int64_t mnb_noalloc_max_rows(void) { return kNoallocMaxRows; }
