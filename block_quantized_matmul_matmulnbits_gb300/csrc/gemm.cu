// gemm.cu -- prefill kernel (many token rows): a tcgen05 tensor-core contraction.
//
// Computes Y[m, n] = sum_k X[m, k] w[n, k] + sum_r T[m, r] B[n, r], the
// "fuse_up" prefill path of "[WebGPU] Fuse rank-32 quantized LoRA with
// MatMulNBits" (onnxruntime PR 33370, commit message adding MatMulNBitsLoRA:
// T first, then the base GEMM "with an integrated T * Bt^T epilogue"),
// restated for sm_103a:
//
//  * One CTA per SM, persistent over output tiles of 128 weight rows x BN
//    token rows (BN <= 256, token tiles fastest so that CTAs running together
//    share a weight tile in L2).
//  * Warp 0 (one lane) is the TMA producer: per 64-wide K step it loads the X
//    tile [BN x 64] FP16 with the 128-byte swizzle and the packed weight tile
//    [128 rows x 64 codes] into a 4-deep shared-memory ring (mbarrier
//    complete_tx).
//  * Warps 6..13 dequantize the packed tile -- exact (q - zp), one rounding by
//    the FP16 scale, the DequantizeLinear map of "Fuse DQ->MatMulNBits for
//    shared initializers and skip outer-scope weights" (PR 33800) -- into the
//    canonical K-major 128B-swizzled FP16 operand layout, then fence the
//    generic->async proxy and arrive on the stage's barrier.
//  * Warp 1 allocates tensor memory (two 128 x BN FP32 accumulators, so the
//    epilogue of one tile overlaps the main loop of the next) and one lane
//    issues tcgen05.mma.kind::f16 (A = dequantized weights, B = X, both from
//    shared memory descriptors), committing each stage back to the producer.
//  * The LoRA term is one more K step with A = B_lora[n, 0:32] and B =
//    T[m, 0:32] (written into the same ring by the dequant warps after
//    griddepcontrol.wait on the LoRA down kernel), so it accumulates into the
//    same tensor-memory tile: the integrated T * Bt^T epilogue.
//  * Warps 2..5 read the accumulator with tcgen05.ld (warp w owns TMEM lanes
//    32 (w % 4) .. +31 = weight rows), round once to FP16 and store Y.
//  * Every mbarrier wait is bounded: after ~2 s the kernel records a timeout
//    in the status word, stops, lets its copies land and frees its TMEM.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "mnb_internal.h"

namespace mnb {

namespace {

constexpr int BM = 128;          // weight rows per tile (MMA M)
constexpr int BK = 64;           // K per pipeline step: one 128-byte swizzle atom of FP16
constexpr int kStages = 4;
constexpr int kMaxBN = 256;
constexpr int kThreads = 448;    // 14 warps
constexpr int kDqWarp0 = 6;      // first dequant warp
constexpr int kDqThreads = 256;
constexpr int kEpiThreads = 128;
constexpr int kXSlot = kMaxBN * 128;    // bytes
constexpr int kWSlot = BM * 128;        // dequantized FP16 A tile
constexpr int kPSlot = BM * 64;         // packed codes (INT8 needs 64 B per row)
constexpr int kStageBytes = kXSlot + kWSlot + kPSlot;
constexpr int kBarOffset = kStages * kStageBytes;
constexpr int kNumBars = 3 * kStages + 4 + 1;
constexpr int kSmemBytes = kBarOffset + kNumBars * 8 + 16 + 1024;  // + alignment slack
static_assert(kSmemBytes <= 232448, "shared memory budget");

// ------------------------------------------------------------------ tcgen05 wrappers

__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// K-major operand in the canonical 128-byte swizzled layout: 8-row atoms of
// 128-byte rows, atoms 1024 bytes apart (stride byte offset), version 1.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)1 << 16;            // leading byte offset (unused for swizzled K-major)
    d |= (uint64_t)(1024 >> 4) << 32;  // stride byte offset
    d |= (uint64_t)1 << 46;            // descriptor version
    d |= (uint64_t)2 << 61;            // 128-byte swizzle
    return d;
}

// kind::f16 instruction descriptor: FP32 accumulate, FP16 A and B, both K-major.
__host__ __device__ constexpr uint32_t f16_idesc(int m, int n) {
    return (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t v[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15}, [%16];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]),
          "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t swz128(int row, int chunk) {  // byte offset in a K-major SW128 tile
    return (uint32_t)((row >> 3) * 1024 + (row & 7) * 128 + ((chunk ^ (row & 7)) << 4));
}

struct GemmParams {
    GemmArgs a;
    int BN;          // token rows per tile (multiple of 16, <= 256)
    int tiles_m;     // token tiles
    int tiles;       // total tiles
    int ksteps;      // 64-wide K steps
    int tmem_cols;   // allocated tensor-memory columns (power of two >= 2 BN)
};

template <int BITS, bool HAS_ZP>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW, const GemmParams P) {
    extern __shared__ unsigned char smem_raw[];
    const uint32_t base_raw = smem_u32(smem_raw);
    const uint32_t sbase = (base_raw + 1023u) & ~1023u;  // 1024-aligned: swizzle atoms
    unsigned char* sptr = smem_raw + (sbase - base_raw);

    const uint32_t bars = sbase + kBarOffset;
    auto full_tma = [&](int s) { return bars + 8u * s; };
    auto full_w = [&](int s) { return bars + 8u * (kStages + s); };
    auto empty = [&](int s) { return bars + 8u * (2 * kStages + s); };
    auto acc_full = [&](int a) { return bars + 8u * (3 * kStages + a); };
    auto acc_empty = [&](int a) { return bars + 8u * (3 * kStages + 2 + a); };
    const uint32_t drain = bars + 8u * (3 * kStages + 4);  // teardown: all MMAs of this CTA done
    const uint32_t tmem_slot = bars + 8u * kNumBars;
    auto xslot = [&](int s) { return sbase + (uint32_t)(s * kStageBytes); };
    auto wslot = [&](int s) { return sbase + (uint32_t)(s * kStageBytes + kXSlot); };
    auto pslot = [&](int s) { return (uint32_t)(s * kStageBytes + kXSlot + kWSlot); };  // offset from sptr

    const GemmArgs& a = P.a;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool lora = a.rank > 0;
    const int steps_per_tile = P.ksteps + (lora ? 1 : 0);
    const int BN = P.BN;
    unsigned int* status = a.status;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full_tma(s), 1);
            mbar_init(full_w(s), kDqThreads);
            mbar_init(empty(s), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(acc_full(i), 1);
            mbar_init(acc_empty(i), kEpiThreads);
        }
        mbar_init(drain, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(tmem_slot),
                     "r"(P.tmem_cols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(sptr + kBarOffset + 8 * kNumBars);
    pdl_launch_dependents();

    const int nblk = a.K / 32;
    const uint32_t x_bytes = (uint32_t)BN * 128u;
    const uint32_t w_bytes = (uint32_t)BM * (uint32_t)(BK * BITS / 8);

    if (warp == 0) {
        // ---------------------------------------------------------------- TMA producer
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmX)) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmW)) : "memory");
            int step = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < P.tiles; tile += gridDim.x) {
                const int m0 = (tile % P.tiles_m) * BN, n0 = (tile / P.tiles_m) * BM;
                for (int i = 0; ok && i < steps_per_tile; ++i, ++step) {
                    const int s = step % kStages;
                    const uint32_t ph = (uint32_t)(step / kStages) & 1u;
                    if (!(ok = mbar_wait(empty(s), ph ^ 1u, status))) break;
                    if (i < P.ksteps) {
                        mbar_arrive_tx(full_tma(s), x_bytes + w_bytes);
                        tma_load_2d(xslot(s), &tmX, i * BK, m0, full_tma(s));
                        tma_load_2d(sbase + pslot(s), &tmW, i * (BK * BITS / 8), n0, full_tma(s));
                    } else {
                        mbar_arrive(full_tma(s));  // LoRA step: the slot is free, nothing to load
                    }
                }
            }
            // let every copy issued into the ring land before the CTA can exit
            for (int j = 1; j <= kStages && step - j >= 0; ++j) {
                const int st = step - j;
                if (!mbar_wait(full_tma(st % kStages), (uint32_t)(st / kStages) & 1u, status, false)) break;
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t idesc = f16_idesc(BM, BN);
            int step = 0, tl = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < P.tiles; tile += gridDim.x, ++tl) {
                const int acc = tl & 1;
                if (!(ok = mbar_wait(acc_empty(acc), ((uint32_t)(tl >> 1) & 1u) ^ 1u, status))) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
                for (int i = 0; i < steps_per_tile; ++i, ++step) {
                    const int s = step % kStages;
                    const uint32_t ph = (uint32_t)(step / kStages) & 1u;
                    if (!(ok = mbar_wait(full_tma(s), ph, status))) break;
                    if (!(ok = mbar_wait(full_w(s), ph, status))) break;
                    tc_fence_after();
                    const int kk = i < P.ksteps ? BK / 16 : 2;  // the LoRA step covers K = 32
                    for (int j = 0; j < kk; ++j)
                        tc_mma(d_tmem, sw128_desc(wslot(s) + 32u * j), sw128_desc(xslot(s) + 32u * j), idesc,
                               (i > 0 || j > 0) ? 1u : 0u);
                    tc_commit(empty(s));
                }
                if (ok) tc_commit(acc_full(acc));
            }
            tc_commit(drain);  // tensor memory is freed only after every issued MMA has finished
            mbar_wait(drain, 0, status, false);
        }
        __syncwarp();
    } else if (warp < kDqWarp0) {
        // ---------------------------------------------------------------- epilogue
        const int q = warp & 3;  // TMEM lane quarter of this warp
        const int row = q * 32 + lane;
        int tl = 0;
        for (int tile = blockIdx.x; tile < P.tiles; tile += gridDim.x, ++tl) {
            const int m0 = (tile % P.tiles_m) * BN, n0 = (tile / P.tiles_m) * BM;
            const int acc = tl & 1;
            if (!mbar_wait(acc_full(acc), (uint32_t)(tl >> 1) & 1u, status)) break;
            tc_fence_after();
            const int n = n0 + row;
            for (int c = 0; c < BN; c += 16) {
                uint32_t v[16];
                tmem_ld16(tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN + c), v);
                if (n < a.N) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int m = m0 + c + j;
                        if (m < a.Mt) a.Y[(size_t)m * a.N + n] = __float2half_rn(__uint_as_float(v[j]));
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(acc_empty(acc));
        }
    } else {
        // ---------------------------------------------------------------- dequant
        const int d = threadIdx.x - kDqWarp0 * 32;  // 0..255
        const int r = d & (BM - 1), h = d >> 7;     // row of the tile, which block of the step
        constexpr int kPrefetch = 4;                // scale / zero-point loads in flight
        constexpr uint32_t kDefaultZp = 1u << (BITS - 1);
        int step = 0;
        bool ok = true, waited = false;
        for (int tile = blockIdx.x; ok && tile < P.tiles; tile += gridDim.x) {
            const int m0 = (tile % P.tiles_m) * BN, n0 = (tile / P.tiles_m) * BM;
            const int n = n0 + r;
            const bool row_ok = n < a.N;
            const uint16_t* srow = reinterpret_cast<const uint16_t*>(a.S) + (size_t)n * nblk;
            const uint8_t* zrow = a.Z + (size_t)n * nblk;
            uint32_t sc[kPrefetch], zz[kPrefetch];
#pragma unroll
            for (int u = 0; u < kPrefetch; ++u) {
                const int blk = 2 * u + h;
                const bool v = row_ok && blk < nblk && u < P.ksteps;
                sc[u] = v ? (uint32_t)__ldg(srow + blk) : 0u;
                zz[u] = HAS_ZP ? (v ? (uint32_t)__ldg(zrow + blk) : 0u) : kDefaultZp;
            }
            for (int i0 = 0; ok && i0 < P.ksteps; i0 += kPrefetch) {
#pragma unroll
                for (int u = 0; u < kPrefetch; ++u) {
                    const int i = i0 + u;
                    if (i >= P.ksteps) break;
                    const int s = step % kStages;
                    const uint32_t ph = (uint32_t)(step / kStages) & 1u;
                    if (!(ok = mbar_wait(full_tma(s), ph, status))) break;
                    const DqConst dc = dq_const(zz[u], (uint16_t)sc[u]);
                    {  // refill this prefetch slot with step i + kPrefetch
                        const int blk = 2 * (i + kPrefetch) + h;
                        const bool v = row_ok && blk < nblk;
                        sc[u] = v ? (uint32_t)__ldg(srow + blk) : 0u;
                        if (HAS_ZP) zz[u] = v ? (uint32_t)__ldg(zrow + blk) : 0u;
                    }
                    const uint32_t wrow = wslot(s);
                    uint32_t out[16];
                    if constexpr (BITS == 4) {
                        const uint4 pk = *reinterpret_cast<const uint4*>(sptr + pslot(s) + r * 32 + h * 16);
                        const uint32_t wv[4] = {pk.x, pk.y, pk.z, pk.w};
#pragma unroll
                        for (int w = 0; w < 4; ++w) dq_int4_natural(wv[w], dc, &out[4 * w]);
                    } else {
                        const uint4 p0 = *reinterpret_cast<const uint4*>(sptr + pslot(s) + r * 64 + h * 32);
                        const uint4 p1 = *reinterpret_cast<const uint4*>(sptr + pslot(s) + r * 64 + h * 32 + 16);
                        const uint32_t wv[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
#pragma unroll
                        for (int w = 0; w < 8; ++w) dq_int8_natural(wv[w], dc, &out[2 * w]);
                    }
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const uint32_t dst = wrow + swz128(r, 4 * h + c);
                        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(out[4 * c]),
                                     "r"(out[4 * c + 1]), "r"(out[4 * c + 2]), "r"(out[4 * c + 3])
                                     : "memory");
                    }
                    fence_proxy_async();
                    mbar_arrive(full_w(s));
                    ++step;
                }
            }
            if (ok && lora) {
                const int s = step % kStages;
                const uint32_t ph = (uint32_t)(step / kStages) & 1u;
                if (!(ok = mbar_wait(full_tma(s), ph, status))) break;
                if (!waited) {
                    pdl_wait();  // T is written by the LoRA down kernel queued before this grid
                    waited = true;
                }
                if (h == 0) {  // A operand: B_lora[n, 0:32] in chunks 0..3 of row r
                    const uint4* brow = reinterpret_cast<const uint4*>(a.B + (size_t)n * 32);
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const uint4 v = row_ok ? __ldg(brow + c) : make_uint4(0, 0, 0, 0);
                        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(wslot(s) + swz128(r, c)),
                                     "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                                     : "memory");
                    }
                }
                for (int idx = d; idx < BN * 4; idx += kDqThreads) {  // B operand: T[m, 0:32]
                    const int tr = idx >> 2, c = idx & 3;
                    const int m = m0 + tr;
                    const uint4 v = m < a.Mt ? *reinterpret_cast<const uint4*>(a.T + (size_t)m * 32 + c * 8)
                                             : make_uint4(0, 0, 0, 0);
                    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(xslot(s) + swz128(tr, c)), "r"(v.x),
                                 "r"(v.y), "r"(v.z), "r"(v.w)
                                 : "memory");
                }
                fence_proxy_async();
                mbar_arrive(full_w(s));
                ++step;
            }
        }
    }

    // ---------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(P.tmem_cols)
                     : "memory");
    }
}

// ------------------------------------------------------------------ host side

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

cudaError_t load_encoder() {
    if (g_encode) return cudaSuccess;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    const cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) return e != cudaSuccess ? e : cudaErrorNotSupported;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    return cudaSuccess;
}

template <int BITS, bool HAS_ZP>
cudaError_t set_attr() {
    return cudaFuncSetAttribute(gemm_kernel<BITS, HAS_ZP>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
}

template <int BITS, bool HAS_ZP>
cudaError_t launch(const CUtensorMap& tx, const CUtensorMap& tw, const GemmParams& P, int grid, bool pdl,
                   cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, gemm_kernel<BITS, HAS_ZP>, tx, tw, P);
}

}  // namespace

int gemm_token_tile(int Mt) {
    if (Mt >= kMaxBN) return kMaxBN;
    int bn = (Mt + 15) / 16 * 16;
    return bn < 16 ? 16 : bn;
}

int gemm_threads() { return kThreads; }

cudaError_t gemm_prepare() {
    cudaError_t e = load_encoder();
    if (e == cudaSuccess) e = set_attr<4, false>();
    if (e == cudaSuccess) e = set_attr<4, true>();
    if (e == cudaSuccess) e = set_attr<8, false>();
    if (e == cudaSuccess) e = set_attr<8, true>();
    return e;
}

cudaError_t gemm_launch(const GemmArgs& a, const mnb_plan_info& p, bool pdl, cudaStream_t st) {
    if (!g_encode) return cudaErrorNotSupported;
    GemmParams P;
    P.a = a;
    P.BN = p.tokens_per_cta;
    P.tiles_m = (a.Mt + P.BN - 1) / P.BN;
    P.tiles = P.tiles_m * ((a.N + BM - 1) / BM);
    P.ksteps = (a.K + BK - 1) / BK;
    int cols = 32;
    while (cols < 2 * P.BN) cols *= 2;
    P.tmem_cols = cols;

    CUtensorMap tx, tw;
    {
        const cuuint64_t dims[2] = {(cuuint64_t)a.K, (cuuint64_t)a.Mt};
        const cuuint64_t strides[1] = {(cuuint64_t)a.K * 2};
        const cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)P.BN};
        const cuuint32_t es[2] = {1, 1};
        if (g_encode(&tx, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<__half*>(a.X), dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    {
        const int rowbytes = a.K * a.bits / 8;
        const cuuint64_t dims[2] = {(cuuint64_t)rowbytes, (cuuint64_t)a.N};
        const cuuint64_t strides[1] = {(cuuint64_t)rowbytes};
        const cuuint32_t box[2] = {(cuuint32_t)(BK * a.bits / 8), (cuuint32_t)BM};
        const cuuint32_t es[2] = {1, 1};
        if (g_encode(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(a.Wq), dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    const int grid = p.grid_x;
    const bool zp = a.Z != nullptr;
    if (a.bits == 4) return zp ? launch<4, true>(tx, tw, P, grid, pdl, st) : launch<4, false>(tx, tw, P, grid, pdl, st);
    return zp ? launch<8, true>(tx, tw, P, grid, pdl, st) : launch<8, false>(tx, tw, P, grid, pdl, st);
}

}  // namespace mnb
