// gemv.cu -- decode kernel (few token rows): a weight-streaming GEMV.
//
// Computes Y[m, n] = sum_k X[m, k] w[n, k] (+ sum_r T[m, r] B[n, r]) for up to
// 16 token rows per CTA, the "fuse_down" decode path of "[WebGPU] Fuse rank-32
// quantized LoRA with MatMulNBits" (onnxruntime PR 33370, commit message
// adding MatMulNBitsLoRA: base GEMV and LoRA down projection first, then the
// base plus T * Bt^T), restated for sm_103a:
//
//  * Every packed weight byte is read from HBM exactly once per token group:
//    CTA c owns output rows [c R, (c+1) R) with R = ceil(N / #SMs), so every SM
//    streams the same number of bytes.
//  * Inside a CTA the work is a list of items (16-row tile, 64-byte K step);
//    warp w takes the contiguous item range [w I / W, (w+1) I / W), so all
//    warps carry the same load whatever the shape.  A thread loads 16 bytes
//    of two rows (g and g+8 of the tile) per step with 128-bit loads that
//    bypass L1; 4 steps are in flight per thread before any is consumed.
//  * Codes are unpacked and dequantized in registers (exact (q - zp), one
//    rounding by the scale, see common.cuh) straight into the A fragments of
//    mma.sync m16n8k16 (FP16 in, FP32 accumulate), the 8 or 16 token rows
//    being the N side.  INT4 uses the pair-interleaved unpacking: the K order
//    inside each 8-code word is permuted identically for the weight and the X
//    fragment, which leaves the sum unchanged.
//  * Partial sums of the warps that share a tile are added in shared memory in
//    a fixed order (deterministic, no atomics), then the LoRA term is added:
//    T (written by the LoRA down kernel, which this grid waits for with
//    griddepcontrol.wait only now, after the weight stream) times the
//    adapter row B[n, :].  Output is rounded once to FP16.
#include "common.cuh"
#include "mnb_internal.h"

namespace mnb {

namespace {

// K steps in flight per thread: 4 with one n8 token tile, 2 with two (registers).
template <int NT>
struct Unroll {
    static constexpr int value = NT == 1 ? 4 : 2;
};

__device__ __forceinline__ uint4 ldg_stream16(const uint8_t* p) {
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(p));
    return r;
}

__device__ __forceinline__ uint32_t word_of(const uint4& v, int i) {
    return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

template <int BITS, bool HAS_ZP, int NT>
__global__ void __launch_bounds__(512, 1) gemv_kernel(const GemvArgs a) {
    extern __shared__ __align__(16) float red[];  // [W][maxseg][16][TOK] then T rows
    constexpr int TOK = 8 * NT;
    constexpr uint32_t kDefaultZp = 1u << (BITS - 1);
    constexpr int kBytesPerBlock = 32 * BITS / 8;  // 16 (INT4) or 32 (INT8)
    constexpr int kUnroll = Unroll<NT>::value;

    const int lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int warp = threadIdx.x >> 5, W = blockDim.x >> 5;
    const int rowbytes = a.K * BITS / 8;
    const int nblk = a.K >> 5;
    const int steps = (rowbytes + 63) >> 6;
    const int row_begin = blockIdx.x * a.rows_per_cta;
    const int row_end = min(a.N, row_begin + a.rows_per_cta);
    const int nrows = row_end - row_begin;
    const int RT = (nrows + 15) >> 4;
    const int token0 = blockIdx.y * TOK;
    const int total = RT * steps;  // items; bounded by the host plan (< 2^31 / 16)
    const int i0 = (int)((long long)total * warp / W), i1 = (int)((long long)total * (warp + 1) / W);
    const int tile_first = i0 / steps;

    __shared__ int wrange[2 * 32];  // item range [i0, i1) of every warp, read by the epilogue
    if (lane == 0) {
        wrange[2 * warp] = i0;
        wrange[2 * warp + 1] = i1;
    }

    for (int i = i0; i < i1;) {
        const int tile = i / steps;
        const int js = i - tile * steps;
        const int je = min(steps, js + (i1 - i));
        i += je - js;

        const int rA = row_begin + tile * 16 + g, rB = rA + 8;
        const bool vA = rA < row_end, vB = rB < row_end;
        const uint8_t* wA = a.Wq + (size_t)rA * rowbytes;
        const uint8_t* wB = a.Wq + (size_t)rB * rowbytes;
        const uint16_t* sA = reinterpret_cast<const uint16_t*>(a.S) + (size_t)rA * nblk;
        const uint16_t* sB = reinterpret_cast<const uint16_t*>(a.S) + (size_t)rB * nblk;
        const uint8_t* zA = a.Z + (size_t)rA * nblk;
        const uint8_t* zB = a.Z + (size_t)rB * nblk;

        float acc[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[nt][e] = 0.f;

        for (int j = js; j < je; j += kUnroll) {
            uint4 wa[kUnroll], wb[kUnroll];
            uint32_t sa[kUnroll], sb[kUnroll], za[kUnroll], zb[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int off = (j + u) * 64 + t * 16;
                const bool kv = (j + u < je) && off < rowbytes;
                const int blk = off / kBytesPerBlock;
                const bool la = kv && vA, lb = kv && vB;
                wa[u] = la ? ldg_stream16(wA + off) : make_uint4(0, 0, 0, 0);
                wb[u] = lb ? ldg_stream16(wB + off) : make_uint4(0, 0, 0, 0);
                sa[u] = la ? __ldg(sA + blk) : 0u;
                sb[u] = lb ? __ldg(sB + blk) : 0u;
                if (HAS_ZP) {
                    za[u] = la ? __ldg(zA + blk) : 0u;
                    zb[u] = lb ? __ldg(zB + blk) : 0u;
                } else {
                    za[u] = kDefaultZp;
                    zb[u] = kDefaultZp;
                }
            }
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                if (j + u >= je) break;  // warp-uniform
                const int off = (j + u) * 64 + t * 16;
                const bool kv = off < rowbytes;
                const int k0 = off * 8 / BITS;  // first K index of this thread's 16 bytes
                const DqConst cA = dq_const(za[u], (uint16_t)sa[u]);
                const DqConst cB = dq_const(zb[u], (uint16_t)sb[u]);
                if constexpr (BITS == 4) {
                    // 32 codes = 4 words of 8 codes; X in the same interleaved pair order.
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        uint32_t dA[4], dB[4];
                        dq_int4_interleaved(word_of(wa[u], w), cA, dA);
                        dq_int4_interleaved(word_of(wb[u], w), cB, dB);
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            const int tok = token0 + nt * 8 + g;
                            uint4 xv = make_uint4(0, 0, 0, 0);
                            if (kv && tok < a.Mt)
                                xv = __ldg(reinterpret_cast<const uint4*>(a.X + (size_t)tok * a.K + k0 + 8 * w));
                            const uint32_t x04 = prmt(xv.x, xv.z, 0x5410u), x15 = prmt(xv.x, xv.z, 0x7632u);
                            const uint32_t x26 = prmt(xv.y, xv.w, 0x5410u), x37 = prmt(xv.y, xv.w, 0x7632u);
                            mma_16816(acc[nt], dA[0], dB[0], dA[1], dB[1], x04, x15);
                            mma_16816(acc[nt], dA[2], dB[2], dA[3], dB[3], x26, x37);
                        }
                    }
                } else {
                    // 16 codes = 4 words of 4 codes, natural pair order.
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        uint4 xv[NT];
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            const int tok = token0 + nt * 8 + g;
                            xv[nt] = make_uint4(0, 0, 0, 0);
                            if (kv && tok < a.Mt)
                                xv[nt] = __ldg(reinterpret_cast<const uint4*>(a.X + (size_t)tok * a.K + k0 + 8 * h));
                        }
#pragma unroll
                        for (int ww = 0; ww < 2; ++ww) {
                            const int w = 2 * h + ww;
                            uint32_t dA[2], dB[2];
                            dq_int8_natural(word_of(wa[u], w), cA, dA);
                            dq_int8_natural(word_of(wb[u], w), cB, dB);
#pragma unroll
                            for (int nt = 0; nt < NT; ++nt) {
                                const uint32_t b0 = ww == 0 ? xv[nt].x : xv[nt].z;
                                const uint32_t b1 = ww == 0 ? xv[nt].y : xv[nt].w;
                                mma_16816(acc[nt], dA[0], dB[0], dA[1], dB[1], b0, b1);
                            }
                        }
                    }
                }
            }
        }

        // C fragment: (row g, tokens 2t, 2t+1) and (row g+8, same tokens), per n8 tile.
        float* r = red + ((size_t)(warp * a.maxseg + (tile - tile_first)) * 16) * TOK;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            r[g * TOK + nt * 8 + 2 * t] = acc[nt][0];
            r[g * TOK + nt * 8 + 2 * t + 1] = acc[nt][1];
            r[(g + 8) * TOK + nt * 8 + 2 * t] = acc[nt][2];
            r[(g + 8) * TOK + nt * 8 + 2 * t + 1] = acc[nt][3];
        }
    }

    __half* tsm = reinterpret_cast<__half*>(red + (size_t)W * a.maxseg * 16 * TOK);
    if (a.rank > 0) {
        pdl_wait();  // T is written by the LoRA down kernel that precedes this grid
        for (int idx = threadIdx.x; idx < TOK * 32; idx += blockDim.x) {
            const int tok = token0 + idx / 32;
            tsm[idx] = tok < a.Mt ? a.T[(size_t)tok * 32 + (idx & 31)] : __float2half_rn(0.f);
        }
    }
    __syncthreads();

    for (int idx = threadIdx.x; idx < nrows * TOK; idx += blockDim.x) {
        const int tok = idx / nrows, rr = idx - tok * nrows;
        const int token = token0 + tok;
        if (token >= a.Mt) continue;
        const int tile = rr >> 4, rit = rr & 15;
        float sum = 0.f;
        const int t_lo = tile * steps, t_hi = t_lo + steps;
        for (int w = 0; w < W; ++w) {  // fixed order over the warps that covered this tile
            const int w0 = wrange[2 * w], w1 = wrange[2 * w + 1];
            if (w0 >= w1 || w1 <= t_lo || w0 >= t_hi) continue;
            const int tf = w0 / steps;
            sum += red[((size_t)(w * a.maxseg + (tile - tf)) * 16 + rit) * TOK + tok];
        }
        const int n = row_begin + rr;
        if (a.rank > 0) {
            const uint4* brow = reinterpret_cast<const uint4*>(a.B + (size_t)n * 32);
            float l = 0.f;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint4 bv = __ldg(brow + q);
                const __half* bh = reinterpret_cast<const __half*>(&bv);
#pragma unroll
                for (int e = 0; e < 8; ++e) l = fmaf(__half2float(tsm[tok * 32 + q * 8 + e]), __half2float(bh[e]), l);
            }
            sum += l;
        }
        a.Y[(size_t)token * a.N + n] = __float2half_rn(sum);
    }
}

template <int BITS, bool HAS_ZP, int NT>
cudaError_t launch_one(const GemvArgs& a, dim3 grid, int threads, size_t smem, bool pdl, cudaStream_t st) {
    static_assert(NT == 1 || NT == 2, "token tiles");
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, gemv_kernel<BITS, HAS_ZP, NT>, a);
}

}  // namespace

size_t gemv_smem_bytes(int warps, int maxseg, int tok) {
    return (size_t)warps * maxseg * 16 * tok * sizeof(float) + (size_t)tok * 32 * sizeof(__half);
}

cudaError_t gemv_prepare() {
    const int bytes = kGemvMaxSmem;
    cudaError_t e = cudaSuccess;
#define MNB_SET(B, Z, T)                                                                                       \
    if (e == cudaSuccess)                                                                                      \
        e = cudaFuncSetAttribute(gemv_kernel<B, Z, T>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    MNB_SET(4, false, 1) MNB_SET(4, false, 2) MNB_SET(4, true, 1) MNB_SET(4, true, 2)
    MNB_SET(8, false, 1) MNB_SET(8, false, 2) MNB_SET(8, true, 1) MNB_SET(8, true, 2)
#undef MNB_SET
    return e;
}

cudaError_t gemv_launch(const GemvArgs& a, const mnb_plan_info& p, int bits, bool pdl, cudaStream_t st) {
    const dim3 grid(p.grid_x, p.grid_y);
    const int nt = p.tokens_per_cta / 8;
    const size_t smem = gemv_smem_bytes(p.block_threads / 32, a.maxseg, p.tokens_per_cta);
    const bool zp = a.Z != nullptr;
    if (bits == 4) {
        if (zp) return nt == 1 ? launch_one<4, true, 1>(a, grid, p.block_threads, smem, pdl, st)
                               : launch_one<4, true, 2>(a, grid, p.block_threads, smem, pdl, st);
        return nt == 1 ? launch_one<4, false, 1>(a, grid, p.block_threads, smem, pdl, st)
                       : launch_one<4, false, 2>(a, grid, p.block_threads, smem, pdl, st);
    }
    if (zp) return nt == 1 ? launch_one<8, true, 1>(a, grid, p.block_threads, smem, pdl, st)
                           : launch_one<8, true, 2>(a, grid, p.block_threads, smem, pdl, st);
    return nt == 1 ? launch_one<8, false, 1>(a, grid, p.block_threads, smem, pdl, st)
                   : launch_one<8, false, 2>(a, grid, p.block_threads, smem, pdl, st);
}

}  // namespace mnb
