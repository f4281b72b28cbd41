// mnb_internal.h -- declarations shared between the C-ABI layer and the kernel
// translation units of libmnb.  Not installed; not part of the ABI.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "mnb.h"

namespace mnb {

// Error bits a kernel ORs into the library's device status word (passed to the
// kernel as a pointer) when one of its bounded waits gives up.
constexpr unsigned int kStatusTimeout = 1u;

// Host-side TMA descriptors (tensor_map.cu).
cudaError_t tensor_map_prepare();
// Process-unique identity of the calling thread's current context (the
// device's primary context is made current first if none is).  Cached device
// addresses and kernel attributes are valid only in the context they were
// obtained in.
cudaError_t current_context_id(unsigned long long* id);
// Byte matrix [rows, rowbytes] (rowbytes % 128 == 0, <= 32 KB) as boxes of `box_rows`
// rows x `box_segs` 128-byte segments, 128-byte swizzled: [box_segs][box_rows][128]
// in shared memory (coordinates: 0, first row, first segment).
cudaError_t encode_codes_sw128(CUtensorMap* map, const void* base, uint64_t rowbytes, uint64_t rows,
                               uint32_t box_rows, uint32_t box_segs);
// Byte matrix [rows, rowbytes] (rowbytes % 256 == 0) seen as [rows][rowbytes/256][256]:
// one box copies `box_rows` rows x `box_chunks` 256-byte pieces, rows `box_chunks*256`
// bytes apart in shared memory.
cudaError_t encode_rows_3d(CUtensorMap* map, const void* base, uint64_t rowbytes, uint64_t rows, uint32_t box_chunks,
                           uint32_t box_rows);
cudaError_t encode_2d(CUtensorMap* map, const void* base, int elem_bytes, uint64_t cols, uint64_t rows,
                      uint64_t pitch_bytes, uint32_t box_cols, uint32_t box_rows, bool swizzle128);

// One projection of a decode launch.  A launch computes up to kMaxSeg
// projections of the same X; projection s owns the 16-row groups
// [g0, g0 + ceil(N / 16)) of the kernel's row space.
constexpr int kMaxSeg = 4;
struct GemvSeg {
    int g0;              // first 16-row group of this projection
    int N;               // output rows of this projection
    const uint8_t* Wq;   // [N, K*bits/8]
    const __half* S;     // [N, K/32]
    const uint8_t* Z;    // [N, K/32] or nullptr (every projection of a launch alike)
    const __half* bias;  // [N] or nullptr
    __half* Y;           // [Mt, N]
};

struct GemvArgs {
    int nseg;                 // projections (>= 1); rank > 0 only with one
    int G;                    // 16-row groups of all projections
    GemvSeg seg[kMaxSeg];
    const __half* X;     // [Mt, K]
    const __half* T;     // [Mt, 32] or nullptr
    const __half* B;     // [N, 32] or nullptr
    const uint8_t* Bq;   // INT8 up weight [N, 32] (one block a row), used instead of B, or nullptr
    const __half* Bs;    // [N] scales of Bq
    const uint8_t* Bz;   // [N] zero points of Bq, or nullptr (128)
    int Mt, K;
    int R;               // output rows owned by one CTA
    int CH;              // K bytes per row and pipeline stage (multiple of 64)
    int ring;            // shared-memory ring stages (2 or 4), set by the launcher
    int xrows;           // X rows staged in shared memory per CTA (0: X read from global)
    int rank;            // 0 or 32
    int x_wait;          // X may be written by the work queued before this kernel (early weights)
    int sms;             // SMs of the device (the launcher picks the CTAs per SM from it)
    int w3d;             // weights of a multi-chunk stage come as one 3-D TMA box (set by the launcher)
    unsigned int* status;
};

// Decode-kernel geometry for (N, K, token rows) on `sms` SMs: `ctas` CTAs, each owning
// whole 16-row groups (at most R rows), K bytes per stage; returns the shared memory it needs.
size_t gemv_geometry(int N, int K, int bits, int Mt, int sms, int* ctas, int* R, int* CH, int* tok, int* threads);
cudaError_t gemv_prepare();
cudaError_t gemv_launch(const GemvArgs& a, const mnb_plan_info& p, int bits, bool pdl, cudaStream_t st);
// The int8-activation variant (X quantized per block of 32 while staged, integer block dots);
// plan with 8 token rows per CTA.  cudaErrorNotSupported when K is too large to stage.
cudaError_t gemv_q8x_launch(const GemvArgs& a, const mnb_plan_info& p, int bits, bool pdl, cudaStream_t st);

// Single-token decode kernel (decode.cu): one token row, INT4 or INT8 weights,
// up to kMaxSeg projections of the same x laid end to end in one row space
// (rows [row0, row0 + N) belong to projection i), the optional FP16 rank-32
// adapter (one projection only; T computed in the same, cooperative, launch)
// and biases.
struct DecSeg {
    int row0;            // first row of this projection in the row space
    int N;               // its rows
    const uint8_t* Wq;   // [N, K*bits/8]
    const __half* S;     // [N, K/32]
    const uint8_t* Z;    // [N, K/32] or nullptr (default 2^(bits-1)); all projections alike
    const __half* bias;  // [N] or nullptr
    __half* Y;           // [1, N]
};
struct DecodeArgs {
    int nseg;            // projections (>= 1)
    int NR;              // rows of the row space (sum of the projections' N)
    DecSeg seg[kMaxSeg];
    const __half* X;     // [Mt, K]
    int Mt;              // token rows (1 for the single-token kernel)
    const __half* A;     // [K, 32] (FP16 adapter)
    const __half* B;     // [N, 32] (FP16 adapter)
    // INT8 adapter (single-token kernel; A and B unused): Aq [32, K] with As / Az
    // [32, K/32], Bq [N, 32] with Bs / Bz [N] (Az / Bz nullptr: 128)
    const uint8_t* Aq;
    const __half* As;
    const uint8_t* Az;
    const uint8_t* Bq;
    const __half* Bs;
    const uint8_t* Bz;
    __half* T;           // [1, 32]: T on return (adapter only)
    int K, bits;
    int SR, ring;        // rows per stage and stage slots (set by the launcher)
    int kparts;          // few-token kernel: a stage's K range arrives in this many slots
    int x_wait;          // X may be written by the work queued before this kernel
    unsigned int* status;
    void* ex;            // the adapter's exchange area (set by the launcher)
};
// Whether a call runs on this kernel: bits 4 or 8, one token row, 32 <= K <= 65536;
// with an adapter at most 256 rows per CTA (N rows over min(SMs, N / 16) CTAs).
bool decode_supported(int bits, int64_t Mt, int K, int64_t N, bool lora, int sms);
// CTAs, rows per stage, stage slots and shared memory of a launch.
// lq8: an INT8 adapter (its B rows' codes staged before they are dequantized).
void decode_geometry(int N, int K, int bits, bool lora, int sms, int* ctas, int* SR, int* ring, size_t* smem,
                     bool lq8 = false);
cudaError_t decode_prepare();
// Clear the adapter exchange areas of the current device (after a device-side
// timeout left one of them part way).
cudaError_t decode_reset_exchange();
cudaError_t decode_launch(const DecodeArgs& a, int rank, int sms, bool pdl, cudaStream_t st);

// Decode kernel for 2 .. 16 token rows (decode_mt.cu): the same row space (up to
// kMaxSeg projections); with an FP16 rank-32 adapter (one projection) B [N, 32] and
// T [Mt, 32] from the LoRA down kernel launched just before (read after
// griddepcontrol.wait).  Whether a call runs on it: bits 4 or 8,
// 2 <= Mt <= 16, K % 512 == 0 and K <= 7680, and x of the token rows plus two
// stage slots (with zero points) fitting in one SM's shared memory.
bool decode_mt_supported(int bits, int64_t Mt, int K, bool lora);
// CTAs, slots per 16-row stage (K parts), ring slots and shared memory of a launch.
void decode_mt_geometry(int N, int K, int bits, int Mt, bool zp, int sms, int* ctas, int* parts, int* ring,
                        size_t* smem);
cudaError_t decode_mt_prepare();
cudaError_t decode_mt_launch(const DecodeArgs& a, int sms, bool pdl, cudaStream_t st);

// T = fp16(X * A), X [Mt, K], A [K, 32].  Deterministic split-K over a cluster.
cudaError_t lora_down_prepare();
// max_ctas > 0 (Mt > 16, K % 256 == 0, a status word for its bounded waits): at most
// that many CTAs and no cluster, each taking all of K for its token rows, so that they
// fit on the SMs a following prefill kernel leaves idle (both down-weight formats).
cudaError_t lora_down_launch(const __half* X, const __half* A, __half* T, int Mt, int K, bool pdl, cudaStream_t st,
                             int max_ctas = 0, unsigned int* status = nullptr);
// The same with an INT8 down weight: Aq [32, K] (block-32 rows along K), As / Az [32, K/32]
// (Az nullptr: 128); A[k, r] = fp16((Aq[r, k] - zp) * scale).
cudaError_t lora_down_q8_launch(const __half* X, const uint8_t* Aq, const __half* As, const uint8_t* Az, __half* T,
                                int Mt, int K, bool pdl, cudaStream_t st, int max_ctas = 0,
                                unsigned int* status = nullptr);

struct GemmArgs {
    const __half* X;
    const uint8_t* Wq;
    const __half* S;
    const uint8_t* Z;
    const __half* T;
    const __half* B;
    const uint8_t* Bq;   // INT8 up weight [N, 32] instead of B, or nullptr
    const __half* Bs;    // [N]
    const uint8_t* Bz;   // [N] or nullptr (128)
    const __half* bias;  // [N] or nullptr
    __half* Y;
    int Mt, N, K, bits, rank;
    unsigned int* status;  // device status word (bounded waits report here)
};
int gemm_token_tile(int Mt);  // token rows per prefill tile (multiple of 16, <= 256)
int gemm_threads();
int gemm_split(int N, int Mt, int K, int sms);  // CTAs sharing one tile along K
cudaError_t gemm_prepare();
// x_wait: X may be written by the work queued before this grid (early weights)
cudaError_t gemm_launch(const GemmArgs& a, const mnb_plan_info& p, bool pdl, bool x_wait, cudaStream_t st);

// Y = 0 over `count` halfs (K == 0 case).
cudaError_t fill_zero_launch(__half* Y, size_t count, cudaStream_t st);
// Y[m, n] = fp16(sum_r T[m, r] B[n, r] (+ bias[n])), the adapter term alone (empty packed
// weight); B is FP16 [N, 32], or INT8 Bq [N, 32] with Bs / Bz [N] when Bq is not null.
cudaError_t lora_up_launch(const __half* T, const __half* B, const uint8_t* Bq, const __half* Bs, const uint8_t* Bz,
                           const __half* bias, __half* Y, int Mt, int N, cudaStream_t st);
// Y[m, n] = bias[n] for m < rows (K == 0 or an empty weight, with a bias)
cudaError_t fill_bias_launch(__half* Y, const __half* bias, size_t rows, size_t N, cudaStream_t st);

// One kernel whose bounded wait nothing satisfies: it records a timeout in `status`.
cudaError_t wait_check_launch(unsigned int* status, long long limit_cycles, cudaStream_t st);

// Xq[m, k] / Xs[m, k/32]: the int8 activation codes and binary32 block scales the
// int8-activation path computes (same device function), codes in K order.
cudaError_t quantize_x_launch(const __half* X, int Mt, int K, int8_t* Xq, float* Xs, cudaStream_t st);

// The fixed T scratch of mnb_run_noalloc (noalloc.cu): the most token rows it
// holds, and its device address in the current context (looked up with
// cudaGetSymbolAddress once per device and context).
constexpr int64_t kNoallocMaxRows = 8192;
int noalloc_scratch(__half** out);
// mnb_run with T in that scratch instead of a caller buffer (api.cu): the
// arguments, validation order and results of mnb_run; adapter calls with more
// than kNoallocMaxRows token rows return MNB_ERR_UNSUPPORTED.
int run_noalloc(mnb_handle h, const void* X, const void* Wq, const void* scales, const void* zp, const void* A,
                const void* B, int32_t rank, void* Y, int64_t batch, int64_t M, void* stream);

// W16[n, k] = fp16((q - zp) * scale) with the kernels' own dequant arithmetic.
cudaError_t dequant_launch(const uint8_t* Wq, const __half* S, const uint8_t* Z, int N, int K, int bits,
                           __half* W16, int variant, cudaStream_t st);

}  // namespace mnb
