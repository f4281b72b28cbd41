// lora_down.cu -- the LoRA down projection T = fp16(X * A), X [Mt, K], A [K, 32].
//
// This is "T" of both fused paths in "[WebGPU] Fuse rank-32 quantized LoRA with
// MatMulNBits" (onnxruntime PR 33370, commit message adding MatMulNBitsLoRA):
// fuse_up computes T first and the base GEMM adds T * Bt^T in its epilogue;
// fuse_down pairs T with the decode GEMV.  T is kept as an FP16 intermediate
// ("preserving FP16 rounding").
//
// The down weight is FP16 A [K, 32], or an INT8 block-32 weight Aq [32, K]
// (the INT8 adapters of the same page's later commits), dequantized while it is
// staged with the base kernels' arithmetic (exact q - zp, one rounding).
//
// Design (sm_103a): K is split across the CTAs of one thread-block cluster
// (up to 8).  Each CTA stages its slices of A and X in padded shared memory
// with every 16-byte copy in flight at once (A, a weight, before the
// griddepcontrol.wait on the producer of X; X after it), runs ldmatrix-fed
// mma.sync m16n8k16 over 64 token rows x 32 ranks with FP32 accumulators, and
// leaves its partial in shared memory.  After a
// cluster barrier every CTA finishes an interleaved share of the outputs,
// adding the partials of all CTAs in rank order through distributed shared
// memory, rounds once to FP16 and stores T.  No atomics, so T is bitwise
// reproducible.  The kernel signals programmatic launch completion right
// after its own griddepcontrol.wait: the matmul kernel queued after it then
// starts only once the work before this kernel has completed, so it may read
// X at once and waits (griddepcontrol.wait) only for T.
//
// Ahead of a prefill grid that leaves SMs idle, a second kernel takes the same
// projection onto those SMs only (lora_down_rows_kernel, below): a cluster's
// CTAs could not be placed together on scattered idle SMs, so each CTA sums all
// of K for its groups of 64 token rows, with X fed by TMA.  It then runs beside
// the prefill kernel, which needs T only at its last stage.
#include "common.cuh"
#include "mnb_internal.h"

namespace mnb {

namespace {

constexpr int kTok = 64;        // token rows per CTA (4 warps x 16)
constexpr int kPiece = 512;     // K columns staged per pass (one pass when K <= 8 * 512)
constexpr int kPitchA = 40;     // halfs per staged A row (32 + 8 pad: conflict-free ldmatrix)
constexpr int kPitchX = kPiece + 8;  // halfs per staged X row (pad: conflict-free ldmatrix)
constexpr int kMaxCluster = 8;
constexpr int kLoraSmem = kPiece * kPitchA * 2 + kTok * kPitchX * 2 + kTok * 32 * 4;

__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// 16-byte global -> shared copy; src_bytes == 0 writes zeros and reads nothing.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}

constexpr int kPitchR = kPiece + 8;  // halfs per staged rank row of a dequantized INT8 A slice
static_assert(32 * kPitchR <= kPiece * kPitchA, "the INT8 A slice reuses the FP16 A slice's space");
static_assert(16 * kPitchX * 2 + 32 * kPiece <= kTok * kPitchX * 2, "raw INT8 A fits the X tile's unused rows");
static_assert(32 * (kPiece / 16) <= 8 * 128, "a pass's INT8 A items fit eight per thread");

// The down weight in one of two formats: FP16 A [K, 32], or INT8 Aq [32, K]
// (block-32 rows along K) with FP16 scales As and zero points Az [32, K/32].
struct DownWeight {
    const __half* A;
    const uint8_t* Aq;
    const __half* As;
    const uint8_t* Az;
};

template <bool Q8>
__global__ void __launch_bounds__(128) lora_down_kernel(const __half* __restrict__ X, const DownWeight W,
                                                         __half* __restrict__ T, int Mt, int K, int nsplit) {
    extern __shared__ __align__(16) unsigned char lds_raw[];
    // FP16 A: [kPiece][kPitchA] (k-major, read transposed); INT8 A: dequantized
    // into [32][kPitchR] (rank-major, read as is)
    __half* As = reinterpret_cast<__half*>(lds_raw);
    __half* Xs = As + kPiece * kPitchA;                                       // [kTok][kPitchX]
    float* part = reinterpret_cast<float*>(Xs + kTok * kPitchX);              // [kTok][32]

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t rank = cluster_rank();
    // Few token rows (decode): one 16-row tile per CTA and the four warps split
    // the K slice; otherwise 64 token rows per CTA, one 16-row tile per warp.
    const bool few = Mt <= 16;
    const int tokc = few ? 16 : kTok;
    const int tokb = blockIdx.y * tokc;  // first token row of this CTA
    const int ntok = min(tokc, Mt - tokb);
    const int wrow = few ? 0 : warp * 16;
    const int nch = K / 16;
    const int c0 = (int)((long long)rank * nch / nsplit), c1 = (int)((long long)(rank + 1) * nch / nsplit);

    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[i][e] = 0.f;

    bool waited = false;
    for (int kb = 16 * c0; kb < 16 * c1; kb += kPiece) {
        const int klen = min(kPiece, 16 * c1 - kb);
        // A (a weight) first, then X once the producer of X has finished.
        // INT8 A, few token rows: raw codes go through cp.async into the unused rows of
        // the X tile (in flight together with X), their block scales and zero points into
        // registers; the dequant runs shared-to-shared once both have landed.
        constexpr int kBatch = 8;  // 16-code items per thread and pass: 32 ranks x 512 / 16 / 128
        uint32_t qsc[kBatch], qzz[kBatch];
        unsigned char* raw = reinterpret_cast<unsigned char*>(Xs + 16 * kPitchX);  // [32][klen] bytes
        const bool q8_async = Q8 && few;
        if constexpr (Q8) {
            const int pc = klen / 16, nblk = K / 32, items = 32 * pc;
            if (few) {
                for (int idx = tid; idx < items; idx += blockDim.x) {
                    const int r = idx / pc, c = idx - r * pc;
                    cp_async16(smem_u32(raw + r * klen + c * 16), W.Aq + (size_t)r * K + kb + c * 16, 16);
                }
#pragma unroll
                for (int j = 0; j < kBatch; ++j) {
                    const int idx = min(j * 128 + tid, items - 1);  // clamped: loads stay in bounds
                    const int r = idx / pc, b = r * nblk + (kb + (idx - r * pc) * 16) / 32;
                    qsc[j] = reinterpret_cast<const uint16_t*>(W.As)[b];
                    qzz[j] = W.Az ? (uint32_t)W.Az[b] : 128u;
                }
            } else {
            // many token rows: 16 codes of one rank row per item, kBatch per thread in
            // flight (all loads first, then the dequant)
            for (int base = 0; base < items; base += kBatch * 128) {
                uint4 v[kBatch];
                uint32_t sc[kBatch], zz[kBatch];
#pragma unroll
                for (int j = 0; j < kBatch; ++j) {
                    const int idx = min(base + j * 128 + tid, items - 1);  // clamped: loads stay in bounds
                    const int r = idx / pc, c = idx - r * pc;
                    const int k = kb + c * 16, b = r * nblk + k / 32;
                    v[j] = __ldg(reinterpret_cast<const uint4*>(W.Aq + (size_t)r * K + k));
                    sc[j] = reinterpret_cast<const uint16_t*>(W.As)[b];
                    zz[j] = W.Az ? (uint32_t)W.Az[b] : 128u;
                }
#pragma unroll
                for (int j = 0; j < kBatch; ++j) {
                    const int idx = base + j * 128 + tid;
                    if (idx >= items) break;
                    const int r = idx / pc, c = idx - r * pc;
                    const DqConst dc = dq_const(zz[j], (uint16_t)sc[j]);
                    uint32_t d[8];
                    dq_int8_natural(v[j].x, dc, &d[0]);
                    dq_int8_natural(v[j].y, dc, &d[2]);
                    dq_int8_natural(v[j].z, dc, &d[4]);
                    dq_int8_natural(v[j].w, dc, &d[6]);
                    uint4* dst = reinterpret_cast<uint4*>(&As[r * kPitchR + c * 16]);
                    dst[0] = make_uint4(d[0], d[1], d[2], d[3]);
                    dst[1] = make_uint4(d[4], d[5], d[6], d[7]);
                }
            }
            }
        } else {
            for (int idx = tid; idx < klen * 4; idx += blockDim.x) {
                const int row = idx >> 2, c = idx & 3;
                cp_async16(smem_u32(&As[row * kPitchA + c * 8]), W.A + (size_t)(kb + row) * 32 + c * 8, 16);
            }
        }
        if (!waited) {
            pdl_wait();
            pdl_launch_dependents();  // the work before this kernel is complete: X is readable
            waited = true;
        }
        const int xc = klen / 8;  // 16-byte chunks per token row
        for (int idx = tid; idx < tokc * xc; idx += blockDim.x) {
            const int row = idx / xc, c = idx - row * xc;
            const bool ok = row < ntok;
            cp_async16(smem_u32(&Xs[row * kPitchX + c * 8]), ok ? X + (size_t)(tokb + row) * K + kb + c * 8 : X,
                       ok ? 16u : 0u);
        }
        cp_async_wait_all();
        __syncthreads();
        if (q8_async) {  // raw INT8 codes -> the rank-major FP16 tile (exact q - zp, one rounding)
            const int pc = klen / 16, items = 32 * pc;
#pragma unroll
            for (int j = 0; j < kBatch; ++j) {
                const int idx = j * 128 + tid;
                if (idx >= items) break;
                const int r = idx / pc, c = idx - r * pc;
                const uint4 v = *reinterpret_cast<const uint4*>(raw + r * klen + c * 16);
                const DqConst dc = dq_const(qzz[j], (uint16_t)qsc[j]);
                uint32_t d[8];
                dq_int8_natural(v.x, dc, &d[0]);
                dq_int8_natural(v.y, dc, &d[2]);
                dq_int8_natural(v.z, dc, &d[4]);
                dq_int8_natural(v.w, dc, &d[6]);
                uint4* dst = reinterpret_cast<uint4*>(&As[r * kPitchR + c * 16]);
                dst[0] = make_uint4(d[0], d[1], d[2], d[3]);
                dst[1] = make_uint4(d[4], d[5], d[6], d[7]);
            }
            __syncthreads();
        }
        const int mat = lane >> 3, row8 = lane & 7;
        for (int kk = few ? 16 * warp : 0; kk < klen; kk += few ? 64 : 16) {
            // A operand: X rows wrow .. +15, K columns kk .. kk+15 (row-major 16x16)
            uint32_t a0, a1, a2, a3;
            ldsm_x4(smem_u32(&Xs[(wrow + (mat & 1) * 8 + row8) * kPitchX + kk + (mat >> 1) * 8]), a0, a1, a2, a3);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t b0, b1, b2, b3;
                if constexpr (Q8)  // rank rows h*16 .. +15, K columns kk .. kk+15
                    ldsm_x4(smem_u32(&As[(h * 16 + (mat >> 1) * 8 + row8) * kPitchR + kk + (mat & 1) * 8]), b0, b1,
                            b2, b3);
                else
                    ldsm_x4_t(smem_u32(&As[(kk + (mat & 1) * 8 + row8) * kPitchA + h * 16 + (mat >> 1) * 8]), b0, b1,
                              b2, b3);
                mma_16816(acc[2 * h], a0, a1, a2, a3, b0, b1);
                mma_16816(acc[2 * h + 1], a0, a1, a2, a3, b2, b3);
            }
        }
        __syncthreads();
    }
    if (!waited) {
        pdl_wait();
        pdl_launch_dependents();
    }

    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
        const int r = nt * 8 + 2 * t;
        part[(warp * 16 + g) * 32 + r] = acc[nt][0];
        part[(warp * 16 + g) * 32 + r + 1] = acc[nt][1];
        part[(warp * 16 + g + 8) * 32 + r] = acc[nt][2];
        part[(warp * 16 + g + 8) * 32 + r + 1] = acc[nt][3];
    }
    if (few) {  // add the four warps' K quarters in warp order into rows 0..15
        __syncthreads();
        for (int idx = tid; idx < 16 * 32; idx += blockDim.x)
            part[idx] = ((part[idx] + part[512 + idx]) + part[1024 + idx]) + part[1536 + idx];
    }
    cluster_sync_all();
    // Every CTA of the cluster finishes an interleaved share of the valid
    // outputs; each output adds the partials in rank order 0..nsplit-1.
    const int valid = ntok * 32;
    for (int idx = (int)rank * blockDim.x + tid; idx < valid; idx += nsplit * blockDim.x) {
        const uint32_t la = smem_u32(&part[idx]);
        float v[kMaxCluster];
#pragma unroll
        for (int q = 0; q < kMaxCluster; ++q) v[q] = q < nsplit ? ld_peer_f32(la, (uint32_t)q) : 0.f;
        float s = 0.f;
#pragma unroll
        for (int q = 0; q < kMaxCluster; ++q)
            if (q < nsplit) s += v[q];
        T[(size_t)(tokb + idx / 32) * 32 + (idx & 31)] = __float2half_rn(s);
    }
    cluster_sync_all();  // keep every CTA's shared memory alive until all peers have read it
}

// The same projection for the SMs a prefill grid leaves idle (FP16 A, more than
// 16 token rows): no cluster -- its CTAs could not be placed together there -- so a
// CTA takes all of K for groups of 64 token rows, gridDim.x groups apart.  K runs
// in pieces of 256 through a ring of four buffers: X by four TMA boxes of 64 rows x
// 64 K (128-byte swizzle) on an mbarrier, A by cp.async into padded rows, the
// copies of pieces p + 1 .. p + 3 in flight while piece p is multiplied (a CTA
// streams its rows from HBM alone, so it needs many bytes in flight).  One CTA sums a row's whole K
// in a fixed order, so T is the same bits every run.
constexpr int kRPiece = 256;                          // K per piece
constexpr int kRXBytes = kTok * kRPiece * 2;          // X of a piece: 4 boxes of 8 KB
constexpr int kRABytes = kRPiece * kPitchA * 2;       // A of a piece, padded rows
constexpr int kRPitchR = kRPiece + 8;                 // INT8 A: halfs per dequantized rank row of a piece
static_assert(32 * kRPitchR * 2 <= kRABytes, "a dequantized INT8 A piece fits the FP16 one's space");
constexpr int kRThreads = 256;                        // 8 warps: 4 row tiles x 2 halves of a piece's K
constexpr int kRQItems = 32 * kRPiece / 16 / kRThreads;  // INT8 A: 16-code items per thread and piece
constexpr int kRBuf = kRXBytes + kRABytes;
static_assert(kRABytes % 1024 == 0, "the next buffer's X boxes stay 1024-aligned");
constexpr int kRBufs = 4;                             // ring of K pieces
constexpr int kRRed = 4 * 32 * 16 * 4;                // the second K half's accumulators, [row tile][lane][16]
constexpr int kRowsSmem = kRBufs * kRBuf + 64 + kRRed + 1024;  // buffers, barriers, reduction, alignment

template <bool Q8>
__global__ void __launch_bounds__(kRThreads) lora_down_rows_kernel(const __grid_constant__ CUtensorMap tmX, const DownWeight W,
                                                              __half* __restrict__ T, int Mt, int K,
                                                              unsigned int* status) {
    extern __shared__ unsigned char lds_raw[];
    const uint32_t base_raw = smem_u32(lds_raw);
    const uint32_t sbase = (base_raw + 1023u) & ~1023u;  // 1024-aligned: swizzle atoms
    unsigned char* sptr = lds_raw + (sbase - base_raw);
    const uint32_t bars = sbase + (uint32_t)(kRBufs * kRBuf);
    auto xbuf = [&](int b) { return sbase + (uint32_t)(b * kRBuf); };
    auto abuf = [&](int b) { return reinterpret_cast<__half*>(sptr + b * kRBuf + kRXBytes); };
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int wrow = (warp & 3) * 16;  // this warp's 16 token rows of the group
    const int kh = warp >> 2;          // and its half of every piece's K
    float* red = reinterpret_cast<float*>(sptr + kRBufs * kRBuf + 64);
    const int npiece = K / kRPiece;
    if (tid == 0) {
        for (int b = 0; b < kRBufs; ++b) mbar_init(bars + 8u * (uint32_t)b, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmX)) : "memory");
    }
    __syncthreads();
    bool waited = false, ok = true;
    int pc = 0;  // pieces consumed so far: piece pc is in buffer pc % kRBufs, its barrier's phase (pc / kRBufs) & 1
    for (int grp = blockIdx.x; ok && grp * kTok < Mt; grp += gridDim.x) {
        const int tokb = grp * kTok;
        // INT8 A of piece p: this thread's kRQItems items of 16 codes (rank idx / 16, codes
        // 16 (idx % 16) .. of the piece), loaded into registers, then dequantized (exact
        // q - zp, one rounding) into the rank-major tile [32][kRPitchR] of buffer b
        uint4 qv[kRQItems];
        uint32_t qs[kRQItems], qz[kRQItems];
        auto q8_load = [&](int p) {
            const int kb = p * kRPiece, nblk = K / 32;
#pragma unroll
            for (int j = 0; j < kRQItems; ++j) {
                const int idx = j * kRThreads + tid, r = idx >> 4, c = idx & 15;
                const int b = r * nblk + (kb + 16 * c) / 32;
                qv[j] = __ldg(reinterpret_cast<const uint4*>(W.Aq + (size_t)r * K + kb + 16 * c));
                qs[j] = reinterpret_cast<const uint16_t*>(W.As)[b];
                qz[j] = W.Az ? (uint32_t)W.Az[b] : 128u;
            }
        };
        auto q8_store = [&](int b) {
            __half* a_s = abuf(b);
#pragma unroll
            for (int j = 0; j < kRQItems; ++j) {
                const int idx = j * kRThreads + tid, r = idx >> 4, c = idx & 15;
                const DqConst dc = dq_const(qz[j], (uint16_t)qs[j]);
                uint32_t d[8];
                dq_int8_natural(qv[j].x, dc, &d[0]);
                dq_int8_natural(qv[j].y, dc, &d[2]);
                dq_int8_natural(qv[j].z, dc, &d[4]);
                dq_int8_natural(qv[j].w, dc, &d[6]);
                uint4* dst = reinterpret_cast<uint4*>(a_s + r * kRPitchR + 16 * c);
                dst[0] = make_uint4(d[0], d[1], d[2], d[3]);
                dst[1] = make_uint4(d[4], d[5], d[6], d[7]);
            }
        };
        // issue the copies of K piece p into buffer b (A first: a weight, not behind the
        // wait; INT8 A only loaded here, dequantized by q8_store)
        auto stage = [&](int p, int b) {
            const int kb = p * kRPiece;
            if constexpr (Q8) {
                q8_load(p);
            } else {
                __half* a_s = abuf(b);
                for (int idx = tid; idx < kRPiece * 4; idx += blockDim.x) {
                    const int row = idx >> 2, c = idx & 3;
                    cp_async16(smem_u32(a_s + row * kPitchA + c * 8), W.A + (size_t)(kb + row) * 32 + c * 8, 16);
                }
            }
            asm volatile("cp.async.commit_group;" ::: "memory");
            if (!waited) {
                pdl_wait();
                pdl_launch_dependents();  // the work before this kernel is complete: X is readable
                waited = true;
            }
            if (tid == 0) {  // rows past Mt read as zero
                const uint32_t bar = bars + 8u * (uint32_t)b;
                mbar_arrive_tx(bar, (uint32_t)kRXBytes);
#pragma unroll
                for (int q = 0; q < kRPiece / 64; ++q)
                    tma_load_2d(xbuf(b) + (uint32_t)(q * kTok * 128), &tmX, kb + 64 * q, tokb, bar);
            }
        };
        float acc[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[i][e] = 0.f;
        for (int p = 0; p < kRBufs - 1 && p < npiece; ++p) {
            stage(p, (pc + p) % kRBufs);
            if constexpr (Q8) q8_store((pc + p) % kRBufs);
        }
        if constexpr (Q8) __syncthreads();  // the prologue's dequantized A
        for (int p = 0; p < npiece; ++p, ++pc) {
            const int b = pc % kRBufs;
            // the buffer of piece p + 3 was last read by piece p - 1 (the block passed the
            // barrier at the end of that piece)
            const bool ahead3 = p + kRBufs - 1 < npiece;
            if (ahead3) stage(p + kRBufs - 1, (pc + kRBufs - 1) % kRBufs);
            // A of piece p has landed once at most the groups committed after it are pending
            const int ahead = min(kRBufs - 1, npiece - 1 - p);
            if (ahead >= 3)
                asm volatile("cp.async.wait_group 3;" ::: "memory");
            else if (ahead == 2)
                asm volatile("cp.async.wait_group 2;" ::: "memory");
            else if (ahead == 1)
                asm volatile("cp.async.wait_group 1;" ::: "memory");
            else
                asm volatile("cp.async.wait_group 0;" ::: "memory");
            ok = mbar_wait(bars + 8u * (uint32_t)b, (uint32_t)(pc / kRBufs) & 1u, status, false);  // X of piece p
            ok = __syncthreads_and(ok) != 0;  // the block decides together
            if (!ok) break;
            const __half* a_s = abuf(b);
            const int mat = lane >> 3, row8 = lane & 7;
            const int xr = wrow + (mat & 1) * 8 + row8;  // this lane's X row for ldmatrix
#pragma unroll 4
            for (int kk = kh * (kRPiece / 2); kk < (kh + 1) * (kRPiece / 2); kk += 16) {
                uint32_t a0, a1, a2, a3;  // X rows wrow .. +15, K columns kk .. kk+15 (box kk / 64, swizzled)
                const int chunk = ((kk & 63) >> 3) + (mat >> 1);
                ldsm_x4(xbuf(b) + (uint32_t)((kk >> 6) * kTok * 128 + xr * 128 + ((chunk ^ (xr & 7)) << 4)), a0, a1,
                        a2, a3);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint32_t b0, b1, b2, b3;
                    if constexpr (Q8)  // rank rows h*16 .. +15, K columns kk .. kk+15
                        ldsm_x4(smem_u32(a_s + (h * 16 + (mat >> 1) * 8 + row8) * kRPitchR + kk + (mat & 1) * 8), b0,
                                b1, b2, b3);
                    else
                        ldsm_x4_t(smem_u32(a_s + (kk + (mat & 1) * 8 + row8) * kPitchA + h * 16 + (mat >> 1) * 8), b0,
                                  b1, b2, b3);
                    mma_16816(acc[2 * h], a0, a1, a2, a3, b0, b1);
                    mma_16816(acc[2 * h + 1], a0, a1, a2, a3, b2, b3);
                }
            }
            // INT8 A of piece p + 3, loaded before this piece's MMAs, into the buffer piece
            // p - 1 left (read by every thread before the block passed the last barrier)
            if constexpr (Q8)
                if (ahead3) q8_store((pc + kRBufs - 1) % kRBufs);
            __syncthreads();  // this buffer is refilled kRBufs - 1 pieces on
        }
        if (!ok) break;
        // the second K halves' sums to the first halves' warps, added in that order
        if (kh == 1) {
#pragma unroll
            for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) red[((warp & 3) * 32 + lane) * 16 + nt * 4 + e] = acc[nt][e];
        }
        __syncthreads();
        if (kh == 1) continue;  // (the next group's first barrier waits for the readers below)
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[nt][e] += red[((warp & 3) * 32 + lane) * 16 + nt * 4 + e];
        const int g = lane >> 2, t = lane & 3;
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
            const int r = nt * 8 + 2 * t;
            const int m0 = tokb + wrow + g, m1 = m0 + 8;
            if (m0 < Mt)
                *reinterpret_cast<__half2*>(&T[(size_t)m0 * 32 + r]) = __floats2half2_rn(acc[nt][0], acc[nt][1]);
            if (m1 < Mt)
                *reinterpret_cast<__half2*>(&T[(size_t)m1 * 32 + r]) = __floats2half2_rn(acc[nt][2], acc[nt][3]);
        }
    }
    if (!waited) {
        pdl_wait();
        pdl_launch_dependents();
    }
}

}  // namespace

cudaError_t lora_down_prepare() {
    cudaError_t e = cudaFuncSetAttribute(lora_down_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kLoraSmem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(lora_down_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kLoraSmem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(lora_down_rows_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kRowsSmem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(lora_down_rows_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kRowsSmem);
    return e;
}

namespace {

cudaError_t launch_down(const __half* X, const DownWeight& W, bool q8, __half* T, int Mt, int K, bool pdl,
                        cudaStream_t st) {
    const int nch = K / 16;
    int nsplit = nch < kMaxCluster ? nch : kMaxCluster;
    if (nsplit < 1) nsplit = 1;
    cudaLaunchConfig_t cfg = {};
    const int tokc = Mt <= 16 ? 16 : kTok;
    cfg.gridDim = dim3(nsplit, (Mt + tokc - 1) / tokc);
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = kLoraSmem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = nsplit;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 2 : 1;
    return q8 ? cudaLaunchKernelEx(&cfg, lora_down_kernel<true>, X, W, T, Mt, K, nsplit)
              : cudaLaunchKernelEx(&cfg, lora_down_kernel<false>, X, W, T, Mt, K, nsplit);
}

}  // namespace

namespace {

// The rows kernel on at most max_ctas SMs (the caller checked Mt > 16, K % kRPiece == 0).
cudaError_t launch_rows(const __half* X, const DownWeight& W, bool q8, __half* T, int Mt, int K, bool pdl,
                        int max_ctas, unsigned int* status, cudaStream_t st) {
    CUtensorMap tx;  // X [Mt x K] FP16, boxes of 64 rows x 64 K, 128-byte swizzle
    cudaError_t e = encode_2d(&tx, X, 2, (uint64_t)K, (uint64_t)Mt, (uint64_t)K * 2, 64u, (uint32_t)kTok, true);
    if (e != cudaSuccess) return e;
    const int groups = (Mt + kTok - 1) / kTok;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(groups < max_ctas ? groups : max_ctas);
    cfg.blockDim = dim3(kRThreads);
    cfg.dynamicSmemBytes = kRowsSmem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return q8 ? cudaLaunchKernelEx(&cfg, lora_down_rows_kernel<true>, tx, W, T, Mt, K, status)
              : cudaLaunchKernelEx(&cfg, lora_down_rows_kernel<false>, tx, W, T, Mt, K, status);
}

bool use_rows(int max_ctas, const unsigned int* status, int Mt, int K) {
    return max_ctas > 0 && status && Mt > 16 && K % kRPiece == 0;
}

}  // namespace

cudaError_t lora_down_launch(const __half* X, const __half* A, __half* T, int Mt, int K, bool pdl, cudaStream_t st,
                             int max_ctas, unsigned int* status) {
    const DownWeight W{A, nullptr, nullptr, nullptr};
    if (use_rows(max_ctas, status, Mt, K)) return launch_rows(X, W, false, T, Mt, K, pdl, max_ctas, status, st);
    return launch_down(X, W, false, T, Mt, K, pdl, st);
}

cudaError_t lora_down_q8_launch(const __half* X, const uint8_t* Aq, const __half* As, const uint8_t* Az, __half* T,
                                int Mt, int K, bool pdl, cudaStream_t st, int max_ctas, unsigned int* status) {
    const DownWeight W{nullptr, Aq, As, Az};
    if (use_rows(max_ctas, status, Mt, K)) return launch_rows(X, W, true, T, Mt, K, pdl, max_ctas, status, st);
    return launch_down(X, W, true, T, Mt, K, pdl, st);
}

}  // namespace mnb
