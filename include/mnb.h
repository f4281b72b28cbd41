/*
 * mnb.h -- C ABI of libmnb.so: block-quantized MatMulNBits with a fused
 * rank-32 FP16 LoRA term, for NVIDIA GB300 (sm_103a).
 *
 *     Y[m, n] = sum_k X[m, k] * w[n, k]  +  sum_r T[m, r] * B[n, r],   T = X * A
 *     w[n, k] = (q[n, k] - zp[n, k / 32]) * scale[n, k / 32]
 *
 * The operation is the one defined by "[WebGPU] Fuse rank-32 quantized LoRA
 * with MatMulNBits" (onnxruntime pull request 33370), commit message adding
 * the MatMulNBitsLoRA operator: INT4 / block-32 base weights, replaceable FP16
 * rank-32 adapters, B read in its transposed [N, r] layout, an empty adapter
 * runs only the base projection, and the GEMV-style (decode) or GEMM-style
 * (prefill) implementation is chosen per call from the per-matrix row count
 * of X, independent of the batch size.  The dequantization map is the one of
 * DequantizeLinear followed by MatMul in "Fuse DQ->MatMulNBits for shared
 * initializers and skip outer-scope weights" (onnxruntime pull request 33800),
 * Description and repro.
 *
 * Conventions for every entry point
 *  - All tensor pointers are DEVICE pointers owned by the caller, row-major
 *    and contiguous, 16-byte aligned.  The library keeps no pointer after a
 *    call returns, copies nothing and never allocates device memory.
 *  - "fp16" is IEEE binary16.  Codes are unsigned.  INT4 codes are packed two
 *    per byte along K, code k = 2j in the low nibble of byte j; INT2 codes
 *    four per byte, code k = 4j + i in bits 2i..2i+1 of byte j (the 2-bit
 *    weights of the commit "Support empty packed weights in CPU and WebGPU
 *    MatMulNBits", referenced by "[WebGPU] Fuse rank-32 quantized LoRA with
 *    MatMulNBits", Description).
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls
 *    only enqueue work; they never synchronize the host, except
 *    mnb_sync_status.
 *  - Return value: MNB_OK (0) or a negative MNB_ERR_* code; on error nothing
 *    has been enqueued unless the code is MNB_ERR_CUDA.
 */
#ifndef MNB_H
#define MNB_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------ */
#define MNB_OK                   0
#define MNB_ERR_ARG             -1  /* NULL required pointer, negative size, bad handle */
#define MNB_ERR_UNSUPPORTED     -2  /* bits not 2/4/8, block_size not 32, K % 32 != 0 (K % 64 for 2 bits),
                                       rank not 0/32 */
#define MNB_ERR_ALIGN           -3  /* a tensor pointer is not 16-byte aligned */
#define MNB_ERR_CUDA            -4  /* a CUDA runtime call or kernel launch failed */
#define MNB_ERR_DEVICE_TIMEOUT  -5  /* a bounded device-side wait gave up (see mnb_sync_status) */
#define MNB_ERR_NO_DEVICE       -6  /* no usable sm_100-family GPU is current */

/* ---- routes (which kernel family ran the last call) -------------------- */
#define MNB_ROUTE_NONE  0   /* nothing launched: M, N or batch is 0 */
#define MNB_ROUTE_GEMV  1   /* decode kernel: weight-streaming, mma.sync fragments */
#define MNB_ROUTE_GEMM  2   /* prefill kernel: TMA + tcgen05 MMA with TMEM accumulators */
#define MNB_ROUTE_FILL  3   /* K == 0: the output is filled with zeros */

/* ---- flags (mnb_desc.flags) -------------------------------------------- */
/* The weight-side inputs (Wq, scales, zp, A, B) stay constant while calls are
 * in flight, so mnb_run may start streaming them before the work queued ahead
 * of it on the stream has finished (programmatic dependent launch): X and T
 * are still read only after that work completes.  Without this flag every
 * call starts after the preceding work on the stream, as usual. */
#define MNB_FLAG_EARLY_WEIGHTS  1

/* ---- mode (mnb_desc.mode) ---------------------------------------------- */
#define MNB_MODE_AUTO        0  /* GEMV when the per-matrix M <= gemv_max_m, else GEMM */
#define MNB_MODE_FORCE_GEMV  1  /* always the decode kernel (any M) */
#define MNB_MODE_FORCE_GEMM  2  /* always the prefill kernel (any M) */

typedef struct mnb_handle_s* mnb_handle;

/* Fixed properties of one quantized projection.
 *   N, K        output features and input features (K % 32 == 0, both >= 0;
 *               K % 64 == 0 for 2-bit weights: rows of whole 16-byte units)
 *   bits        2, 4 or 8
 *   block_size  32 (the only supported block)
 *   max_rank    0 or 32: the largest adapter rank mnb_run will be given
 *   mode        MNB_MODE_*
 *   gemv_max_m  largest per-matrix M routed to the decode kernel in AUTO
 *               mode; <= 0 selects the default 16
 *   flags       0 or MNB_FLAG_EARLY_WEIGHTS */
typedef struct {
    int64_t N;
    int64_t K;
    int32_t bits;
    int32_t block_size;
    int32_t max_rank;
    int32_t mode;
    int32_t gemv_max_m;
    int32_t flags;
} mnb_desc;

/* Launch plan of one call, as computed by the dispatcher (host only). */
typedef struct {
    int32_t route;          /* MNB_ROUTE_* */
    int32_t lora_kernel;    /* 1 if the LoRA down projection kernel runs first */
    int32_t grid_x, grid_y; /* grid of the main kernel */
    int32_t block_threads;  /* threads per CTA of the main kernel */
    int32_t rows_per_cta;   /* GEMV: most output rows a CTA owns (whole 16-row groups, dealt out
                               evenly); GEMM: output rows per tile */
    int32_t k_splits;       /* GEMV: rows per pipeline stage (single- and few-token decode
                               kernels, a whole row each) or K bytes per row and stage (general
                               multi-token kernel); GEMM: CTAs (one cluster) sharing a tile
                               along K, 1 = persistent CTAs over tiles */
    int32_t tokens_per_cta; /* GEMV: token columns per CTA (1, 8 or 16); GEMM: token tile */
} mnb_plan_info;

/* Validate `desc` and create a handle.  Host memory only: no device call is
 * made, so this works without a GPU.  Errors: MNB_ERR_ARG (NULL pointers,
 * negative N/K), MNB_ERR_UNSUPPORTED (bits, block_size, K % 32, max_rank). */
int mnb_create(const mnb_desc* desc, mnb_handle* out);

/* Release a handle (NULL is ignored).  Enqueued work is not waited for. */
void mnb_destroy(mnb_handle h);

/* Y = X * dequant(Wq)^T (+ (X * A) * B^T), enqueued on `stream`.
 *   X       fp16 [batch, M, K]
 *   Wq      uint8 [N, K/32, 32*bits/8]: 8 (INT2), 16 (INT4) or 32 (INT8) bytes a block
 *   scales  fp16 [N, K/32]
 *   zp      uint8 [N, K/32], or NULL for the default 2^(bits-1) (2, 8, 128)
 *   A, B    fp16 [K, rank] and [N, rank] (B is the transposed up weight);
 *           both NULL or rank == 0 selects the empty adapter (base only)
 *   rank    0 or 32, at most desc.max_rank
 *   Y       fp16 [batch, M, N], written entirely
 *   T_ws    fp16 [batch*M, rank] scratch for T = X * A (rounded to fp16, the
 *           FP16 intermediate of the fused operator); may be NULL when the
 *           adapter is empty.  Its contents on return are T.
 * The kernel family is chosen from the per-matrix row count M (not batch*M).
 * M, N or batch == 0 launches nothing; K == 0 writes zeros.
 * Wq == NULL with K > 0 is an empty packed weight (the rule of "Support empty
 * packed weights in CPU and WebGPU MatMulNBits", referenced by "[WebGPU] Fuse
 * rank-32 quantized LoRA with MatMulNBits", Description): the base term is
 * zero, scales and zp are not read (may be NULL), Y keeps its logical shape
 * and holds zeros -- or, with an adapter, T * B^T alone (route FILL, one LoRA
 * down and one small up-projection kernel).  mnb_plan describes the call with
 * a nonempty weight.
 * Every row of X is independent: [batch, M] gives the same bits as one matrix
 * of batch*M rows routed the same way.  Results are deterministic run to run.
 * A single-token call with an adapter is one cooperative launch whose CTAs add
 * up T through one of 32 exchange areas of the library, handed out in turn per
 * launch: at most 32 such launches may run at the same time (on different
 * streams).
 * Errors: MNB_ERR_ARG, MNB_ERR_UNSUPPORTED, MNB_ERR_ALIGN, MNB_ERR_NO_DEVICE,
 * MNB_ERR_CUDA.  No allocation and no host synchronization happen here. */
int mnb_run(mnb_handle h,
            const void* X, const void* Wq, const void* scales, const void* zp,
            const void* A, const void* B, int32_t rank,
            void* Y, void* T_ws,
            int64_t batch, int64_t M, void* stream);

/* mnb_run with an optional bias: Y[m, n] = fp16_rne(sum + bias[n]), the bias
 * added to every row before the one rounding.  With K == 0 every row of Y is
 * the bias.  Follows the operator's optional bias input: "[WebGPU] Fuse rank-32
 * quantized LoRA with MatMulNBits", referenced commit "Support empty packed
 * weights in CPU and WebGPU MatMulNBits", Description (the output holds zeros
 * or the broadcast bias).
 *   bias    fp16 [N], 16-byte aligned, or NULL (then exactly mnb_run)
 * All other arguments, results and errors are those of mnb_run. */
int mnb_run_bias(mnb_handle h,
                 const void* X, const void* Wq, const void* scales, const void* zp,
                 const void* A, const void* B, int32_t rank, const void* bias,
                 void* Y, void* T_ws,
                 int64_t batch, int64_t M, void* stream);

/* mnb_run_bias with INT8 block-32 rank-32 adapters instead of FP16 ones: the
 * INT4 base with "block-32 INT8 adapters" and their "original INT8
 * arithmetic" of "[WebGPU] Fuse rank-32 quantized LoRA with MatMulNBits"
 * (commit message adding the INT8-adapter graph fusion and kernels, and the
 * later MatMulNBitsQLoRA commit).  Each adapter projection is an 8-bit
 * MatMulNBits weight:
 *   Aq        uint8 [32, K/32, 32]  down projection: rank rows along K
 *   A_scales  fp16 [32, K/32];  A_zp uint8 [32, K/32] or NULL (128)
 *   Bq        uint8 [N, 1, 32]     up projection: N rows along the rank
 *   B_scales  fp16 [N];  B_zp uint8 [N] or NULL (128)
 * a[k, r] = fp16((Aq[r, k] - zp) * scale), b[n, r] likewise (exact q - zp,
 * one rounding, as the base weights), T = fp16(X * a), Y = fp16(base + T * b^T
 * (+ bias)).  Aq and Bq both NULL, or rank == 0, is the empty adapter.  All
 * pointers 16-byte aligned.  Other arguments, results and errors as mnb_run_bias. */
int mnb_run_qlora(mnb_handle h,
                  const void* X, const void* Wq, const void* scales, const void* zp,
                  const void* Aq, const void* A_scales, const void* A_zp,
                  const void* Bq, const void* B_scales, const void* B_zp, int32_t rank,
                  const void* bias, void* Y, void* T_ws,
                  int64_t batch, int64_t M, void* stream);

/* mnb_run_bias with the int8-activation base ("accuracy level 4" of "[WebGPU]
 * Fuse rank-32 quantized LoRA with MatMulNBits", Performance; its
 * MatMulNBitsLoRA commit keeps "DP4A activation quantization for the base,
 * with original FP16 X for T"):
 *   per row of X and block of 32 along K, in binary32: amax = max |x|;
 *   codes xq = clamp(rint(x * (127 / amax)), -127, 127), scale xs = amax / 127
 *   (amax == 0: codes 0, scale 0);
 *   Y = fp16(sum_b xs * scale_w * sum_{k in b} xq * (q - zp)  + T * B^T (+ bias))
 * with the integer sums exact (u8 x s8 tensor-core dots) and T from the FP16
 * X.  Runs on the decode kernel for every M (8 token rows per CTA); X is
 * quantized while it is staged, no workspace.  Arguments, results and errors
 * as mnb_run_bias; MNB_ERR_UNSUPPORTED also when K is too large to stage
 * in shared memory (K above about 12,000). */
int mnb_run_q8x(mnb_handle h,
                const void* X, const void* Wq, const void* scales, const void* zp,
                const void* A, const void* B, int32_t rank, const void* bias,
                void* Y, void* T_ws,
                int64_t batch, int64_t M, void* stream);

/* Failure-detection check: one kernel runs the library's bounded device wait
 * (the one every pipeline barrier uses) on a barrier that nothing completes;
 * after `limit_cycles` SM cycles (1e3 .. 4e9; the kernels use 4e9, about 2 s)
 * it gives up, sets the timeout bit of the device status word and returns.
 * A following mnb_sync_status reports MNB_ERR_DEVICE_TIMEOUT once (and clears
 * the bit); the CUDA context stays usable.  No fault, trap or hang.
 * Errors: MNB_ERR_ARG (limit out of range), MNB_ERR_NO_DEVICE, MNB_ERR_CUDA. */
int mnb_check_wait_timeout(int64_t limit_cycles, void* stream);

/* The activation quantization of mnb_run_q8x on its own (same device
 * function): X fp16 [Mt, K] -> Xq int8 [Mt, K] (K order), Xs float [Mt, K/32].
 * Errors: MNB_ERR_ARG, MNB_ERR_UNSUPPORTED (K % 32), MNB_ERR_ALIGN, MNB_ERR_CUDA. */
int mnb_quantize_x(const void* X, int64_t Mt, int64_t K, void* Xq, void* Xs, void* stream);

/* One projection of mnb_run_multi (all pointers device, 16-byte aligned). */
typedef struct {
    int64_t N;            /* output features of this projection (>= 0) */
    const void* Wq;       /* uint8 [N, K/32, 32*bits/8], or NULL: an empty packed weight */
    const void* scales;   /* fp16 [N, K/32] (unused when Wq is NULL) */
    const void* zp;       /* uint8 [N, K/32] or NULL (default); all nonempty members alike */
    const void* bias;     /* fp16 [N] or NULL */
    void* Y;              /* fp16 [batch, M, N] */
} mnb_projection;

/* Several projections of the same X in one call -- the fused QKV / MLP
 * projections that "Support empty packed weights in CPU and WebGPU
 * MatMulNBits" (referenced by "[WebGPU] Fuse rank-32 quantized LoRA with
 * MatMulNBits", Description) keeps: the nonempty members are computed, an
 * empty member (Wq NULL) gets the shared zero / bias fallback.
 *   h        handle of the fused weight: K, bits, mode and flags as for
 *            mnb_run; desc.N must equal the sum of the members' N
 *   proj     1 to 4 members; each Y_i[m, n] = fp16(sum_k X[m, k] w_i[n, k] (+ bias_i[n]))
 * Decode route: ONE decode-kernel launch over all nonempty members (their
 * 16-row groups laid end to end), plus one fill launch per empty member.
 * Prefill route: one tensor-core launch per nonempty member.  Each member's
 * result is bitwise the result of mnb_run_bias on that member alone.  No
 * adapter.  Errors: MNB_ERR_ARG (N mismatch, NULL required pointer),
 * MNB_ERR_UNSUPPORTED (more than 4 members, mixed zero-point presence),
 * MNB_ERR_ALIGN, MNB_ERR_NO_DEVICE, MNB_ERR_CUDA. */
int mnb_run_multi(mnb_handle h, const void* X, const mnb_projection* proj, int32_t nproj,
                  int64_t batch, int64_t M, void* stream);

/* Rewrite a DequantizeLinear weight into this layout (HOST pointers, host
 * code, no device call): the transposed initializers that "Fuse
 * DQ->MatMulNBits for shared initializers and skip outer-scope weights"
 * (Description) writes when it turns DequantizeLinear -> MatMul into
 * MatMulNBits.
 *   w_q      uint8 [K, N], one code per byte, each < 2^bits (else MNB_ERR_ARG)
 *   w_scale  fp16 [K/32, N] when `blocked`, else one per-tensor value
 *   w_zp     uint8, shaped like w_scale, or NULL (DequantizeLinear's default 0)
 *   Wq       out uint8 [N, K/32, 32*bits/8];  scales out fp16 [N, K/32];
 *   zp       out uint8 [N, K/32], always written (explicit, since 0 is not
 *            this library's default)
 * Then mnb_run on (X, Wq, scales, zp) equals X * DequantizeLinear(w_q)
 * within the usual tolerance.  Errors: MNB_ERR_ARG, MNB_ERR_UNSUPPORTED
 * (bits, block size, K % 32). */
int mnb_transpose_dq_weight(const uint8_t* w_q, const uint16_t* w_scale, const uint8_t* w_zp,
                            int64_t K, int64_t N, int32_t bits, int32_t block_size, int32_t blocked,
                            uint8_t* Wq, uint16_t* scales, uint8_t* zp);

/* The plan mnb_run would use for (batch, M, rank) on a GPU with `sm_count`
 * SMs (sm_count <= 0: query the current device).  Host only.  Follows the
 * auto mode selection of the MatMulNBitsLoRA commit message (per-matrix row
 * count, independent of batch). */
int mnb_plan(mnb_handle h, int64_t batch, int64_t M, int32_t rank, int32_t sm_count,
             mnb_plan_info* out);

/* MNB_ROUTE_* of the last successful mnb_run on this handle. */
int mnb_last_route(mnb_handle h);

/* Synchronize `stream`, then read and clear the library's device status word.
 * Returns MNB_OK, MNB_ERR_DEVICE_TIMEOUT when a bounded device-side wait of a
 * kernel gave up since the last call (that kernel's output is then
 * incomplete; the adapter exchange areas are then cleared, so no call may be
 * in flight on another stream), or MNB_ERR_CUDA. */
int mnb_sync_status(mnb_handle h, void* stream);

/* Human-readable name of a status code (static string). */
const char* mnb_status_str(int code);

/* The dequantization step on its own: W16[n, k] = fp16_rne((q - zp) * scale),
 * the weight map of DequantizeLinear in "Fuse DQ->MatMulNBits for shared
 * initializers and skip outer-scope weights" (Description), computed with the
 * same device arithmetic as the matmul kernels.  Exact: one rounding.
 *   W16      fp16 [N, K] output
 *   variant  0 = the natural-order unpacking the prefill kernel uses,
 *            1 = the pair-interleaved unpacking the decode kernel uses
 *            (both must give identical bits; INT8 has only the natural one)
 * Errors as for mnb_run. */
int mnb_dequant(const void* Wq, const void* scales, const void* zp,
                int64_t N, int64_t K, int32_t bits, int32_t block_size,
                void* W16, int32_t variant, void* stream);

/* The LoRA down projection on its own: T[m, r] = fp16_rne(sum_k X[m, k] A[k, r]),
 * "T" of the fuse_up / fuse_down steps in the MatMulNBitsLoRA commit message.
 *   X fp16 [Mt, K], A fp16 [K, rank], T fp16 [Mt, rank]; rank == 32. */
int mnb_lora_down(const void* X, const void* A, void* T, int64_t Mt, int64_t K, int32_t rank,
                  void* stream);

/* mnb_run without the T_ws argument, for callers that cannot allocate device
 * memory: code running inside a host runtime that owns every device
 * allocation and gives plugins no allocator, or latency-critical loops where
 * cudaMalloc / cudaFree are not allowed because they can synchronize the
 * device.  The pages have no counterpart to this entry point; it exists only
 * for such callers.
 *   Arguments, argument checks (in the same order) and results are those of
 *   mnb_run, minus T_ws.  T lives in a fixed array inside the library's
 *   device memory (512 KiB on every GPU that loads the library, held until
 *   the process exits), so at most mnb_noalloc_max_rows() = 8192 token rows
 *   (batch * M) are accepted when an adapter is given; larger calls return
 *   MNB_ERR_UNSUPPORTED and launch nothing.  Without an adapter there is no
 *   limit.
 *   No cudaMalloc, cudaFree or other allocating call is made.  The first call
 *   with an adapter in a context (per device; again after the device's
 *   current context changed) looks up the array's device address
 *   (cudaGetSymbolAddress); make that first call before any stream capture.
 *   Every call shares the one array: calls whose kernels may overlap on the
 *   GPU (other streams, or other host threads without ordering) race on it. */
int mnb_run_noalloc(mnb_handle h,
                    const void* X, const void* Wq, const void* scales, const void* zp,
                    const void* A, const void* B, int32_t rank,
                    void* Y, int64_t batch, int64_t M, void* stream);

/* Largest batch * M mnb_run_noalloc accepts with an adapter. */
int64_t mnb_noalloc_max_rows(void);

#ifdef __cplusplus
}
#endif
#endif /* MNB_H */
