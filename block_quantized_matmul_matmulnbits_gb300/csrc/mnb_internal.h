// mnb_internal.h -- declarations shared between the C-ABI layer and the kernel
// translation units of libmnb.  Not installed; not part of the ABI.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "mnb.h"

namespace mnb {

// Error bits a kernel ORs into the library's device status word (passed to the
// kernel as a pointer) when one of its bounded waits gives up.
constexpr unsigned int kStatusTimeout = 1u;

// Largest dynamic shared memory the decode kernel is allowed to request.
constexpr int kGemvMaxSmem = 160 * 1024;

struct GemvArgs {
    const __half* X;     // [Mt, K]
    const uint8_t* Wq;   // [N, K*bits/8]
    const __half* S;     // [N, K/32]
    const uint8_t* Z;    // [N, K/32] or nullptr (default zero point)
    const __half* T;     // [Mt, 32] or nullptr
    const __half* B;     // [N, 32] or nullptr
    __half* Y;           // [Mt, N]
    int Mt, N, K;
    int rows_per_cta;    // output rows owned by one CTA
    int maxseg;          // tile segments one warp can touch (sizes the reduction buffer)
    int rank;            // 0 or 32
};

size_t gemv_smem_bytes(int warps, int maxseg, int tok);
cudaError_t gemv_prepare();
cudaError_t gemv_launch(const GemvArgs& a, const mnb_plan_info& p, int bits, bool pdl, cudaStream_t st);

// T = fp16(X * A), X [Mt, K], A [K, 32].  Deterministic split-K over a cluster.
cudaError_t lora_down_prepare();
cudaError_t lora_down_launch(const __half* X, const __half* A, __half* T, int Mt, int K, cudaStream_t st);

struct GemmArgs {
    const __half* X;
    const uint8_t* Wq;
    const __half* S;
    const uint8_t* Z;
    const __half* T;
    const __half* B;
    __half* Y;
    int Mt, N, K, bits, rank;
    unsigned int* status;  // device status word (bounded waits report here)
};
int gemm_token_tile(int Mt);  // token rows per prefill tile (multiple of 16, <= 256)
int gemm_threads();
cudaError_t gemm_prepare();
cudaError_t gemm_launch(const GemmArgs& a, const mnb_plan_info& p, bool pdl, cudaStream_t st);

// Y = 0 over `count` halfs (K == 0 case).
cudaError_t fill_zero_launch(__half* Y, size_t count, cudaStream_t st);

// W16[n, k] = fp16((q - zp) * scale) with the kernels' own dequant arithmetic.
cudaError_t dequant_launch(const uint8_t* Wq, const __half* S, const uint8_t* Z, int N, int K, int bits,
                           __half* W16, int variant, cudaStream_t st);

}  // namespace mnb
