// gemm.cu -- tensor-core kernel: the prefill contraction, and decode shapes
// split along K.
//
// Computes Y[m, n] = sum_k X[m, k] w[n, k] + sum_r T[m, r] B[n, r], the
// "fuse_up" prefill path of "[WebGPU] Fuse rank-32 quantized LoRA with
// MatMulNBits" (onnxruntime PR 33370, commit message adding MatMulNBitsLoRA:
// T first, then the base GEMM "with an integrated T * Bt^T epilogue"),
// restated for sm_103a:
//
//  * Output tiles of 128 weight rows x BN token rows (BN <= 256).  With enough
//    tiles one CTA per SM runs persistently over them (token tiles fastest, so
//    CTAs running together share a weight tile in L2).  With few tiles (decode
//    shapes) the K range of a tile is split over the S CTAs of a thread-block
//    cluster; their partial tiles are added in rank order through distributed
//    shared memory (deterministic, no atomics).
//  * The K loop runs in stages of xk 64-wide K steps (xk = 2 when a CTA takes
//    whole rows of an even number of K steps, else 1).  A stage is one X slot
//    in shared memory plus xk dequantized A steps in tensor memory, with one
//    "full" barrier (the X copy's bytes and every dequant warp's arrival) and
//    one "empty" barrier (the MMAs are done): the single MMA thread spends a
//    few hundred cycles on every wait and every commit, as much as on issuing
//    several MMAs, so it waits once and commits once per stage instead of
//    twice each per K step.
//  * Each dequant thread takes its block of both K steps of a stage together:
//    two independent chains of loads and arithmetic, one tensor-memory store
//    wait.  The dequant warps are few (two a scheduler) and latency-bound, so
//    that overlap, not the arithmetic, sets their rate.
//  * Two producer warps, so that the weight stream runs ahead of X: warp 0
//    copies the packed weights of 128 rows in super-stages of 128 or 256
//    bytes per row (TMA boxes of 128 rows x 128 bytes, 128-byte swizzle),
//    warp 14 the X tile of a stage: [BN x 64] FP16 per K step, xk of them in
//    one 3-D box (TMA, 128-byte swizzle).  Few large boxes: one TMA copy
//    costs about as much as a small one, so per-row copies of a few hundred
//    bytes cannot feed an SM.
//  * Warps 6..13 dequantize: exact (q - zp), one rounding by the FP16 scale --
//    the DequantizeLinear map of "Fuse DQ->MatMulNBits for shared initializers
//    and skip outer-scope weights" (PR 33800) -- straight into tensor memory
//    (tcgen05.st: a warp writes its own quarter of the 128 rows, one row per
//    lane, half of the step's K each), then arrive on the stage's barrier
//    once its xk steps are written.
//    The A operand never passes through shared memory: per K step that saves
//    writing and reading 16 KB there, next to the 32 KB of X the MMA reads.
//  * Warp 1 allocates tensor memory (one or two 128 x BN FP32 accumulators and
//    the A steps of the stage ring) and one lane issues tcgen05.mma.kind::f16
//    (A from tensor memory, B = X from a shared memory descriptor), committing
//    each stage back to both producers with one commit.
//  * The LoRA term is one more K step (in the last K split of a tile) with A =
//    B_lora[n, 0:32] (FP16, or dequantized from an INT8 block-32 up weight)
//    and B = T[m, 0:32], written into the ring by the dequant
//    warps after griddepcontrol.wait on the LoRA down kernel: the integrated
//    T * Bt^T epilogue, accumulated into the same tensor-memory tile.
//  * Warps 2..5 read the accumulator with tcgen05.ld (warp w owns TMEM lanes
//    32 (w % 4) .. +31 = weight rows), round once to FP16 and store Y.
//  * Every mbarrier wait is bounded: after ~2 s the kernel records a timeout
//    in the status word, stops, lets its copies and MMAs land and frees its
//    tensor memory.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "mnb_internal.h"

namespace mnb {

namespace {

constexpr int BM = 128;          // weight rows per tile (MMA M)
constexpr int BK = 64;           // K per pipeline step: one 128-byte swizzle atom of FP16
constexpr int kMaxBN = 256;
constexpr int kThreads = 480;    // 15 warps
constexpr int kDqWarp0 = 6;      // first dequant warp
constexpr int kXWarp = 14;       // X producer
constexpr int kDqThreads = 256;
constexpr int kDqWarps = kDqThreads / 32;  // arrivals on the dequant barriers: one per warp
constexpr int kEpiThreads = 128;
constexpr int kACols = BK / 2;    // tensor-memory columns of one dequantized A stage (128 rows x 64 FP16)
constexpr int kPBox = BM * 128;  // one packed-weight TMA box: 128 rows x 128 bytes
constexpr int kMaxSplit = 8;
constexpr uint32_t kSmemBudget = 232448;

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

// tcgen05.mma.kind::f16 with A in tensor memory ([a_tmem]: rows in lanes, K along
// the columns, two FP16 values a 32-bit column) and B from a shared-memory descriptor.
__device__ __forceinline__ void tc_mma_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

// 16 consecutive 32-bit columns of this warp's 32 tensor-memory lanes (one per
// thread); the registers are read at issue, the write completes asynchronously
// (tmem_wait_st).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t v[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
        "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
        : "memory");
}

__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// A 2-D TMA store of a shared-memory tile (async proxy; bulk group of this thread).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int c0, int c1) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c0), "r"(c1), "r"(src)
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

__host__ __device__ inline uint32_t g_align(uint32_t x, uint32_t a) { return (x + a - 1) / a * a; }

// Shared-memory plan, identical on host and device.
// The split-K partial tile (128 x BN FP32) reuses the ring from offset 0: a
// CTA of a split runs one unit, and once its accumulator is complete every
// copy into the ring has landed and every read of it has finished.
// Two rings in shared memory: stages (nx slots of xk K steps of X) and
// packed-weight super-stages (np slots), then (ystage) the output staging.  The
// stages' dequantized A steps (nw = nx xk) live in tensor memory beside the
// accumulators: columns [0, nacc BN) hold one or two 128 x BN FP32
// accumulators, A step t of the ring starts at column a_col + 32 t.
struct GemmLayout {
    uint32_t xslot;    // bytes of one X slot (BN rows x 128 B, 1024-aligned)
    int nx, nw, np;    // stages (X slots), their A steps in tensor memory, packed super-stages
    int pboxes;        // TMA boxes per packed super-stage (128 packed bytes of each row per box)
    uint32_t pstage;   // bytes of one packed super-stage
    int nacc;          // accumulators (two: a tile's epilogue runs under the next tile's MMAs)
    uint32_t a_col, tmem_cols;
    uint32_t p_off, y_off, red_bytes, bar_off, total;
};

// ystage: the epilogue stages the FP16 output tile in shared memory, a
// [BN tokens][32 rows] part per epilogue warp, each written with one TMA store.
__host__ __device__ inline GemmLayout gemm_layout(int BN, int xk, int ystage) {
    GemmLayout L;
    L.xslot = g_align((uint32_t)(xk * BN) * 128u, 1024u);
    // Small token tiles (decode shapes) are bound by the weight stream: deep
    // packed ring, large super-stages.  Large tiles give the space to the stages.
    L.pboxes = BN <= 64 ? 2 : 1;
    L.pstage = (uint32_t)(L.pboxes * kPBox);
    L.np = BN <= 64 ? 4 : 2;
    // 512 columns of tensor memory: two accumulators where four A stages still fit
    L.nacc = 2 * BN + 4 * kACols <= 512 ? 2 : 1;
    L.a_col = g_align((uint32_t)(L.nacc * BN), 32u);
    L.tmem_cols = 512u;
    L.red_bytes = (uint32_t)BM * BN * 4u;
    // One ring of stages: stage s holds xk K steps of X (an X slot) and their xk
    // dequantized A steps (tensor memory), filled and released together.
    const uint32_t ybytes = ystage ? (uint32_t)(BM * BN * 2) : 0u;
    const uint32_t fixed = L.np * L.pstage + ybytes + 512u + 1024u;
    int nx = fixed < kSmemBudget ? (int)((kSmemBudget - fixed) / L.xslot) : 0;
    const int nx_tmem = (int)((512u - L.a_col) / kACols) / xk;
    if (nx > nx_tmem) nx = nx_tmem;
    if (nx > 12) nx = 12;
    L.nx = nx;
    L.nw = nx * xk;
    L.p_off = (uint32_t)nx * L.xslot;
    L.y_off = L.p_off + (uint32_t)L.np * L.pstage;
    L.bar_off = L.y_off + ybytes;
    L.total = L.bar_off + 512u + 1024u;
    return L;
}

struct GemmParams {
    GemmArgs a;
    int BN;         // token rows per tile (multiple of 16, <= 256)
    int tiles_m;    // token tiles
    int tiles;      // total tiles
    int ksteps;     // 64-wide K steps of a full row
    int split;      // CTAs (one cluster) sharing a tile along K; 1 = persistent over tiles
    int xk;         // K steps per X copy: 2 = one 3-D box of two 64-wide K slices (split 1, even K steps)
    int ystage;     // output tile through shared memory and a TMA store (split 1, N % 8 == 0)
    int tpre;       // T of a CTA's first tile staged early by the epilogue warps (ystage, rank > 0)
    int x_wait;     // X may be written by the work queued before this grid: wait for it
};

// One unit of work of a CTA: a tile and a K-step range.
struct Unit {
    int n0, m0, i0, i1;
    bool lora;  // this unit adds the LoRA K step
};

__device__ __forceinline__ bool next_unit(const GemmParams& P, int& cursor, Unit& u) {
    const int split = P.split;
    int tile;
    int cr = 0;
    if (split == 1) {
        tile = cursor;
        cursor += gridDim.x;
    } else {
        if (cursor != (int)blockIdx.x) return false;  // one unit per CTA
        tile = (int)blockIdx.x / split;
        cr = (int)blockIdx.x % split;
        cursor = -1;
    }
    if (tile < 0 || tile >= P.tiles) return false;
    u.m0 = (tile % P.tiles_m) * P.BN;
    u.n0 = (tile / P.tiles_m) * BM;
    u.i0 = (int)((long long)cr * P.ksteps / split);
    u.i1 = (int)((long long)(cr + 1) * P.ksteps / split);
    u.lora = P.a.rank > 0 && cr == split - 1;
    return true;
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_barrier() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ float4 ld_peer_f32x4(uint32_t local_addr, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local_addr), "r"(rank));
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(remote));
    return v;
}

template <int BITS, bool HAS_ZP>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                const __grid_constant__ CUtensorMap tmY, const GemmParams P) {
    extern __shared__ unsigned char smem_raw[];
    const uint32_t base_raw = smem_u32(smem_raw);
    const uint32_t sbase = (base_raw + 1023u) & ~1023u;  // 1024-aligned: swizzle atoms
    unsigned char* sptr = smem_raw + (sbase - base_raw);
    const GemmLayout L = gemm_layout(P.BN, P.xk, P.ystage);
    const int nx = L.nx, np = L.np;

    const uint32_t bars = sbase + L.bar_off;
    // Stage s: full_x (X landed and its A steps written: the X producer's
    // arrival with the copy's bytes, one arrival per dequant warp), empty_x (the
    // MMAs are done with both).  The single MMA thread then waits once and
    // commits once per stage: each of those costs it a few hundred cycles, as
    // much as issuing several MMAs.
    auto full_x = [&](int s) { return bars + 8u * s; };
    auto empty_x = [&](int s) { return bars + 8u * (nx + s); };
    const int b0 = 2 * nx;
    auto full_p = [&](int j) { return bars + 8u * (b0 + j); };
    auto empty_p = [&](int j) { return bars + 8u * (b0 + np + j); };
    auto acc_full = [&](int a) { return bars + 8u * (b0 + 2 * np + a); };
    auto acc_empty = [&](int a) { return bars + 8u * (b0 + 2 * np + 2 + a); };
    const uint32_t drain = bars + 8u * (b0 + 2 * np + 4);
    const uint32_t tmem_slot = drain + 8u;
    const uint32_t t_ready = drain + 16u;  // T of the first unit staged (tpre)
    auto xslot = [&](int s) { return sbase + (uint32_t)s * L.xslot; };

    const GemmArgs& a = P.a;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int BN = P.BN;
    constexpr int kStepBytes = BK * BITS / 8;  // packed bytes of one K step per row
    const int kps = L.pboxes * 128 / kStepBytes;  // K steps per packed super-stage (a power of two)
    unsigned int* status = a.status;

    if (threadIdx.x == 0) {
        for (int s = 0; s < nx; ++s) {
            mbar_init(full_x(s), 1 + kDqWarps);
            mbar_init(empty_x(s), 1);
        }
        for (int j = 0; j < np; ++j) {
            mbar_init(full_p(j), 1);
            mbar_init(empty_p(j), kDqWarps);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(acc_full(i), 1);
            mbar_init(acc_empty(i), kEpiThreads);
        }
        mbar_init(drain, 1);
        mbar_init(t_ready, kEpiThreads / 32);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(tmem_slot),
                     "r"(L.tmem_cols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(sptr + (tmem_slot - sbase));
    pdl_launch_dependents();

    const int nblk = a.K / 32;
    const int xk = P.xk;
    const uint32_t x_tile = (uint32_t)BN * 128u;  // one K step of X in a slot
    const uint32_t x_bytes = (uint32_t)xk * x_tile;

    if (warp == 0) {
        // ---------------------------------------------------------------- packed-weight producer
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmW)) : "memory");
            int pstep = 0, cursor = blockIdx.x;
            bool ok = true;
            Unit u;
            while (ok && next_unit(P, cursor, u)) {
                for (int i = u.i0; i < u.i1; i += kps, ++pstep) {
                    const int j = pstep % np;
                    const uint32_t ph = (uint32_t)(pstep / np) & 1u;
                    if (!(ok = mbar_wait_sleep(empty_p(j), ph ^ 1u, status, 64))) break;
                    // boxes holding this unit's K steps; rows past N and bytes past K read as zero
                    const int bytes = min(kps, u.i1 - i) * kStepBytes;
                    const int nbox = (bytes + 127) / 128;
                    mbar_arrive_tx(full_p(j), (uint32_t)(nbox * kPBox));
                    const uint32_t dst = sbase + L.p_off + (uint32_t)j * L.pstage;
                    for (int b = 0; b < nbox; ++b)
                        tma_load_2d(dst + (uint32_t)b * kPBox, &tmW, i * kStepBytes + 128 * b, u.n0, full_p(j));
                }
            }
            // let every copy issued into the ring land before the CTA can exit
            for (int j = 1; j <= np && pstep - j >= 0; ++j) {
                const int st = pstep - j;
                if (!mbar_wait(full_p(st % np), (uint32_t)(st / np) & 1u, status, false)) break;
            }
        }
        __syncwarp();
    } else if (warp == kXWarp) {
        // ---------------------------------------------------------------- X producer
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmX)) : "memory");
            int step = 0, cursor = blockIdx.x;  // step: X stages (xk K steps each, or the LoRA step)
            bool ok = true, x_ready = P.x_wait == 0;
            Unit u;
            while (ok && next_unit(P, cursor, u)) {
                const int nkx = (u.i1 - u.i0) / xk;  // K stages (xk divides the range)
                const int nst = nkx + (u.lora ? 1 : 0);
                for (int i = 0; i < nst; ++i, ++step) {
                    const int s = step % nx;
                    const uint32_t ph = (uint32_t)(step / nx) & 1u;
                    if (!(ok = mbar_wait_sleep(empty_x(s), ph ^ 1u, status, 64))) break;
                    if (i >= nkx) {  // LoRA step: the dequant warps fill the slot
                        mbar_arrive(full_x(s));
                        continue;
                    }
                    if (!x_ready) {
                        pdl_wait();  // weights went ahead; X only after the preceding work
                        x_ready = true;
                    }
                    mbar_arrive_tx(full_x(s), x_bytes);
                    if (xk == 1)
                        tma_load_2d(xslot(s), &tmX, (u.i0 + i) * BK, u.m0, full_x(s));
                    else  // [K slice][token row][128 B]: one 128B-swizzled tile per K step
                        tma_load_3d(xslot(s), &tmX, 0, u.m0, u.i0 + i * xk, full_x(s));
                }
            }
            for (int j = 1; j <= nx && step - j >= 0; ++j) {
                const int st = step - j;
                if (!mbar_wait(full_x(st % nx), (uint32_t)(st / nx) & 1u, status, false)) break;
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t idesc = f16_idesc(BM, BN);
            int sx = 0, tl = 0, cursor = blockIdx.x;  // sx: ring slot of the stage, ph: its phase
            uint32_t ph = 0;
            bool ok = true;
            Unit u;
            while (ok && next_unit(P, cursor, u)) {
                const int acc = tl % L.nacc, use = tl / L.nacc;
                if (!(ok = mbar_wait(acc_empty(acc), ((uint32_t)use & 1u) ^ 1u, status))) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
                const int nkx = (u.i1 - u.i0) / xk;
                const int nst = nkx + (u.lora ? 1 : 0);
                for (int i = 0; i < nst; ++i) {
                    if (!(ok = mbar_wait(full_x(sx), ph, status))) break;
                    tc_fence_after();
                    // K = 16 a MMA: 8 columns of A, 32 bytes of an X row (2 in the descriptor's address field)
                    uint32_t a_tmem = tmem_base + L.a_col + (uint32_t)(sx * xk * kACols);
                    uint64_t bd = sw128_desc(xslot(sx));
                    if (i >= nkx) {  // the LoRA step: K = 32
                        if (P.tpre && tl == 0) bd = sw128_desc(sbase + L.y_off);  // T staged by the epilogue warps
                        tc_mma_ta(d_tmem, a_tmem, bd, idesc, 1u);
                        tc_mma_ta(d_tmem, a_tmem + 8u, bd + 2u, idesc, 1u);
                    } else {
                        for (int sub = 0; sub < xk; ++sub) {
#pragma unroll
                            for (int j = 0; j < BK / 16; ++j)
                                tc_mma_ta(d_tmem, a_tmem + 8u * j, bd + 2u * j, idesc, (i | sub | j) ? 1u : 0u);
                            a_tmem += kACols;
                            bd += x_tile >> 4;
                        }
                    }
                    tc_commit(empty_x(sx));  // the X slot and the stage's A steps
                    if (++sx == nx) {
                        sx = 0;
                        ph ^= 1u;
                    }
                }
                if (ok) tc_commit(acc_full(acc));
                ++tl;
            }
            tc_commit(drain);  // tensor memory is freed only after every issued MMA has finished
            mbar_wait(drain, 0, status, false);
        }
        __syncwarp();
    } else if (warp < kDqWarp0) {
        // ---------------------------------------------------------------- epilogue
        const int q = warp & 3;  // TMEM lane quarter of this warp
        const int row = q * 32 + lane;
        int tl = 0, cursor = blockIdx.x;
        Unit u;
        while (next_unit(P, cursor, u)) {
            const int acc = tl % L.nacc, use = tl / L.nacc;
            if (P.tpre && tl == 0 && u.lora) {
                // T of the CTA's first tile into the output staging, unused until this tile's
                // epilogue, while the K loop runs: the LoRA stage then copies nothing
                pdl_wait();  // T is written by the LoRA down kernel queued before this grid
                const uint32_t tst = sbase + L.y_off;
                for (int idx = threadIdx.x - 64; idx < BN * 4; idx += kEpiThreads) {  // warps 2..5
                    const int tr = idx >> 2, c = idx & 3;
                    const int m = u.m0 + tr;
                    const uint4 v = m < a.Mt ? *reinterpret_cast<const uint4*>(a.T + (size_t)m * 32 + c * 8)
                                             : make_uint4(0, 0, 0, 0);
                    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(tst + swz128(tr, c)), "r"(v.x),
                                 "r"(v.y), "r"(v.z), "r"(v.w)
                                 : "memory");
                }
                fence_proxy_async();  // before the MMA reads it
                __syncwarp();
                if (lane == 0) mbar_arrive(t_ready);
            }
            // the epilogue waits a whole tile: it sleeps, so as not to take issue slots from the
            // dequant; the warp decides together (it synchronises below)
            if (!__all_sync(0xffffffffu, mbar_wait_sleep(acc_full(acc), (uint32_t)use & 1u, status, 1000))) break;
            tc_fence_after();
            const int n = u.n0 + row;
            if (P.ystage) {
                // This warp's 32 rows of the output tile, [BN tokens][32 rows] FP16 in shared
                // memory (64 contiguous bytes a token), then one TMA store by lane 0; rows
                // past N and tokens past Mt are clipped by the store.  Only the warp
                // synchronises, so a wait given up by one warp blocks no other.
                const uint32_t ystg = sbase + L.y_off + (uint32_t)(q * BN * 64);
                const float bn = a.bias && n < a.N ? __half2float(a.bias[n]) : 0.f;
                for (int c = 0; c < BN; c += 16) {
                    uint32_t v[16];
                    tmem_ld16(tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN + c), v);
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const __half h = __float2half_rn(__uint_as_float(v[j]) + bn);
                        asm volatile("st.shared.u16 [%0], %1;" ::"r"(ystg + (uint32_t)(((c + j) * 32 + lane) * 2)),
                                     "h"(__half_as_ushort(h))
                                     : "memory");
                    }
                }
                tc_fence_before();
                mbar_arrive(acc_empty(acc));  // tensor memory read: the next tile's MMAs may start
                fence_proxy_async();          // the staged rows, before the TMA reads them
                __syncwarp();
                if (lane == 0) {
                    tma_store_2d(&tmY, ystg, u.n0 + q * 32, u.m0);
                    asm volatile("cp.async.bulk.commit_group;\n\tcp.async.bulk.wait_group.read 0;" ::: "memory");
                }
                __syncwarp();  // the staging rows are free again
                ++tl;
                continue;
            }
            for (int c = 0; c < BN; c += 16) {
                uint32_t v[16];
                tmem_ld16(tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN + c), v);
                if (P.split > 1) {  // partial tile for the cluster reduction
                    float4* dst = reinterpret_cast<float4*>(sptr + ((uint32_t)row * BN + c) * 4u);
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        dst[j] = make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                                             __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3]));
                } else if (n < a.N) {
                    const float bn = a.bias ? __half2float(a.bias[n]) : 0.f;
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int m = u.m0 + c + j;
                        if (m < a.Mt) a.Y[(size_t)m * a.N + n] = __float2half_rn(__uint_as_float(v[j]) + bn);
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(acc_empty(acc));
            ++tl;
        }
        if (P.ystage && lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");  // the output writes, complete
    } else {
        // ---------------------------------------------------------------- dequant
        // thread -> (row r, block h of the step): a warp owns the 32 rows of its
        // tensor-memory lane quarter (warp % 4) and one block of every step (warps
        // 6..9 the first, 10..13 the second); a quarter warp's swizzled 16-byte
        // reads of the packed box hit 8 distinct bank groups
        const int d = threadIdx.x - kDqWarp0 * 32;  // 0..255
        const int dl = lane;
        const int r = (warp & 3) * 32 + lane;
        const int h = (warp - kDqWarp0) >> 2;
        const uint32_t a_lane = tmem_base + ((uint32_t)((warp & 3) * 32) << 16) + L.a_col + (uint32_t)h * 16u;
        constexpr int kPrefetch = 6;                // scale / zero-point loads in flight (steps; even)
        static_assert(kPrefetch % 2 == 0, "steps are dequantized in pairs");
        constexpr uint32_t kDefaultZp = 1u << (BITS - 1);
        int pstep = 0, xs = 0, du = 0, cursor = blockIdx.x;  // xs: stages, du: units
        bool ok = true, waited = false;
        Unit u;
        while (ok && next_unit(P, cursor, u)) {
            const int n = u.n0 + r;
            const bool row_ok = n < a.N;
            const uint16_t* srow = reinterpret_cast<const uint16_t*>(a.S) + (size_t)(row_ok ? n : 0) * nblk;
            const uint8_t* zrow = a.Z + (size_t)(row_ok ? n : 0) * nblk;
            // The loads are unconditional (clamped to a valid address) and the
            // validity is kept as a bit: a select on a load's result right
            // after it would wait for the load and defeat the prefetch.
            uint32_t sc[kPrefetch], zz[kPrefetch];
            uint32_t vmask = 0;
#pragma unroll
            for (int v = 0; v < kPrefetch; ++v) {
                const int blk = 2 * (u.i0 + v) + h;
                const bool ld = row_ok && blk < nblk && u.i0 + v < u.i1;
                const int bc = ld ? blk : 0;
                sc[v] = (uint32_t)__ldg(srow + bc);
                zz[v] = HAS_ZP ? (uint32_t)__ldg(zrow + bc) : kDefaultZp;
                vmask |= ld ? (1u << v) : 0u;
            }
            int cur_p = 0;
            // One row's block h of step v of the prefetch window (packed super-stage cur_p).
            auto dq_step = [&](int v, int local, uint32_t(&out)[16]) {
                // invalid block (row past N, K tail): scale 0 makes its products 0
                const uint16_t sv = ((vmask >> v) & 1u) ? (uint16_t)sc[v] : (uint16_t)0;
                // this step's bytes of row r: box li*kStepBytes/128, 16-byte chunk c0 (+1)
                const int li = (local & (kps - 1));
                const int pb = li * kStepBytes;
                const int c0 = ((pb & 127) >> 4) + (BITS == 2 ? 0 : h * (kStepBytes / 32));
                const unsigned char* prow =
                    sptr + L.p_off + (uint32_t)cur_p * L.pstage + (uint32_t)(pb >> 7) * kPBox + (uint32_t)r * 128u;
                if constexpr (BITS == 2) {  // the step's 16 bytes are one chunk; block h is its half h
                    const Dq2Const d2 = dq2_const(zz[v], sv);
                    const uint4 pk = *reinterpret_cast<const uint4*>(prow + ((c0 ^ (r & 7)) << 4));
                    dq_int2_natural(h ? pk.z : pk.x, d2, &out[0]);
                    dq_int2_natural(h ? pk.w : pk.y, d2, &out[8]);
                } else if constexpr (BITS == 4) {
                    const DqConst dc = dq_const(zz[v], sv);
                    const uint4 pk = *reinterpret_cast<const uint4*>(prow + ((c0 ^ (r & 7)) << 4));
                    const uint32_t wv[4] = {pk.x, pk.y, pk.z, pk.w};
#pragma unroll
                    for (int w = 0; w < 4; ++w) dq_int4_natural(wv[w], dc, &out[4 * w]);
                } else {
                    const DqConst dc = dq_const(zz[v], sv);
                    const uint4 p0 = *reinterpret_cast<const uint4*>(prow + ((c0 ^ (r & 7)) << 4));
                    const uint4 p1 = *reinterpret_cast<const uint4*>(prow + (((c0 + 1) ^ (r & 7)) << 4));
                    const uint32_t wv[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
#pragma unroll
                    for (int w = 0; w < 8; ++w) dq_int8_natural(wv[w], dc, &out[2 * w]);
                }
            };
            // Steps in pairs: one stage (xk = 2) or two (xk = 1).  A pair's two blocks are
            // independent, so their loads and arithmetic overlap, and their stores are
            // waited for once.  Pairs start at even unit-local steps, so a packed
            // super-stage (an even number of steps) never changes inside one.
            for (int i0 = u.i0; ok && i0 < u.i1; i0 += kPrefetch) {
#pragma unroll
                for (int v = 0; v < kPrefetch; v += 2) {
                    const int i = i0 + v;
                    if (i >= u.i1) break;
                    const bool two = i + 1 < u.i1;  // always with xk = 2 (an even number of steps)
                    const int local = i - u.i0;
                    // the warp decides together (it arrives once per warp below)
                    if ((local & (kps - 1)) == 0) {
                        cur_p = pstep % np;
                        ok = __all_sync(0xffffffffu, mbar_wait_sleep(full_p(cur_p), (uint32_t)(pstep / np) & 1u, status, 32));
                        if (!ok) break;
                        ++pstep;
                    }
                    const bool split2 = xk == 1 && two;  // the second step is a stage of its own
                    const int sx0 = xs % nx, sx1 = split2 ? (xs + 1) % nx : sx0;
                    const int s0 = sx0 * xk, s1 = split2 ? sx1 : s0 + 1;  // A steps of the ring
                    // the MMA is done with the stage(s)
                    ok = __all_sync(0xffffffffu, mbar_wait_sleep(empty_x(sx0), ((uint32_t)(xs / nx) & 1u) ^ 1u, status, 32));
                    if (ok && split2)
                        ok = __all_sync(0xffffffffu,
                                        mbar_wait_sleep(empty_x(sx1), ((uint32_t)((xs + 1) / nx) & 1u) ^ 1u, status, 32));
                    if (!ok) break;
                    uint32_t out0[16], out1[16];
                    dq_step(v, local, out0);
                    if (two) dq_step(v + 1, local + 1, out1);
                    // each block's 32 FP16 values: 16 columns of row r in its A step
                    tmem_st16(a_lane + (uint32_t)(s0 * kACols), out0);
                    if (two) tmem_st16(a_lane + (uint32_t)(s1 * kACols), out1);
                    tmem_wait_st();  // the stores complete, before the MMA thread is told
                    tc_fence_before();
                    __syncwarp();
                    if (dl == 0) {  // one arrival per warp: its lanes are ordered before lane 0 here
                        mbar_arrive(full_x(sx0));
                        if (split2) mbar_arrive(full_x(sx1));
                        if (!two || ((local + 1) & (kps - 1)) == kps - 1 || i + 1 == u.i1 - 1)
                            mbar_arrive(empty_p(cur_p));  // the packed super-stage is consumed
                    }
                    xs += split2 ? 2 : 1;
#pragma unroll
                    for (int t = 0; t < 2; ++t) {  // refill the prefetch slots with steps i + t + kPrefetch
                        const int it = i + t + kPrefetch;
                        const int blk = 2 * it + h;
                        const bool ld = row_ok && blk < nblk && it < u.i1;
                        const int bc = ld ? blk : 0;
                        sc[v + t] = (uint32_t)__ldg(srow + bc);
                        if (HAS_ZP) zz[v + t] = (uint32_t)__ldg(zrow + bc);
                        vmask = ld ? (vmask | (1u << (v + t))) : (vmask & ~(1u << (v + t)));
                    }
                }
            }
            if (ok && u.lora) {
                const int sx = xs % nx, s = sx * xk;
                ok = __all_sync(0xffffffffu, mbar_wait(empty_x(sx), ((uint32_t)(xs / nx) & 1u) ^ 1u, status));
                if (!ok) break;
                const bool t_staged = P.tpre && du == 0;  // T already in the output staging
                if (!waited && !t_staged) {
                    pdl_wait();  // T is written by the LoRA down kernel queued before this grid
                    waited = true;
                }
                if (h == 0) {  // A operand: row r's 32 adapter values in columns 0..15 of stage s
                    uint32_t o[16];
                    if (a.Bq) {  // from the INT8 up weight: one block per row
                        const size_t nn = (size_t)(row_ok ? n : 0);
                        const uint4* brow = reinterpret_cast<const uint4*>(a.Bq + nn * 32);
                        const uint4 p0 = __ldg(brow), p1 = __ldg(brow + 1);
                        const uint16_t sbits = row_ok ? reinterpret_cast<const uint16_t*>(a.Bs)[nn] : (uint16_t)0;
                        const DqConst bc = dq_const(a.Bz ? (uint32_t)a.Bz[nn] : 128u, sbits);  // scale 0: row past N
                        const uint32_t wv[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
#pragma unroll
                        for (int w = 0; w < 8; ++w) dq_int8_natural(wv[w], bc, &o[2 * w]);
                    } else {  // B_lora[n, 0:32]
                        const uint4* brow = reinterpret_cast<const uint4*>(a.B + (size_t)(row_ok ? n : 0) * 32);
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            const uint4 v = row_ok ? __ldg(brow + c) : make_uint4(0, 0, 0, 0);
                            o[4 * c] = v.x;
                            o[4 * c + 1] = v.y;
                            o[4 * c + 2] = v.z;
                            o[4 * c + 3] = v.w;
                        }
                    }
                    tmem_st16(a_lane + (uint32_t)(s * kACols), o);  // h == 0: columns 0..15
                }
                for (int idx = t_staged ? BN * 4 : d; idx < BN * 4; idx += kDqThreads) {  // B operand: T[m, 0:32]
                    const int tr = idx >> 2, c = idx & 3;
                    const int m = u.m0 + tr;
                    const uint4 v = m < a.Mt ? *reinterpret_cast<const uint4*>(a.T + (size_t)m * 32 + c * 8)
                                             : make_uint4(0, 0, 0, 0);
                    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(xslot(sx) + swz128(tr, c)), "r"(v.x),
                                 "r"(v.y), "r"(v.z), "r"(v.w)
                                 : "memory");
                }
                fence_proxy_async();  // T in the X slot, before the MMA reads it
                tmem_wait_st();       // the adapter rows in tensor memory, likewise
                tc_fence_before();
                if (t_staged) {  // T staged by the epilogue warps (their arrival orders it before ours)
                    ok = __all_sync(0xffffffffu, mbar_wait(t_ready, 0, status));
                    if (!ok) break;
                }
                __syncwarp();
                if (dl == 0) mbar_arrive(full_x(sx));
                ++xs;
            }
            ++du;
        }
    }

    // ---------------------------------------------------------------- teardown
    tmem_wait_st();  // a role that stopped early may have stores in flight
    tc_fence_before();
    __syncthreads();
    if (P.split > 1) {
        // Split-K: every CTA of the cluster holds a partial 128 x BN tile; rank q
        // finishes a contiguous slice of the token columns, adding the partials
        // of ranks 0..S-1 in order.
        cluster_barrier();
        if (warp >= 2 && warp < kDqWarp0 && (*reinterpret_cast<volatile unsigned int*>(status) & kStatusTimeout) == 0) {
            const int q = warp & 3, row = q * 32 + lane;
            const uint32_t rank = cluster_ctarank();
            const int S = P.split;
            const int tile = (int)blockIdx.x / S;
            const int m0 = (tile % P.tiles_m) * BN, n0 = (tile / P.tiles_m) * BM;
            const int ncol4 = (min(BN, a.Mt - m0) + 3) / 4;  // token columns holding valid rows
            const int c0 = (int)((long long)rank * ncol4 / S), c1 = (int)((long long)(rank + 1) * ncol4 / S);
            const int n = n0 + row;
            for (int c4 = c0; c4 < c1; ++c4) {
                const uint32_t la = sbase + ((uint32_t)row * BN + (uint32_t)c4 * 4u) * 4u;
                float4 sum = ld_peer_f32x4(la, 0);
                for (int qq = 1; qq < S; ++qq) {
                    const float4 v = ld_peer_f32x4(la, (uint32_t)qq);
                    sum.x += v.x;
                    sum.y += v.y;
                    sum.z += v.z;
                    sum.w += v.w;
                }
                if (n < a.N) {
                    const float bn = a.bias ? __half2float(a.bias[n]) : 0.f;
                    const float vals[4] = {sum.x + bn, sum.y + bn, sum.z + bn, sum.w + bn};
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int m = m0 + c4 * 4 + j;
                        if (m < a.Mt) a.Y[(size_t)m * a.N + n] = __float2half_rn(vals[j]);
                    }
                }
            }
        }
        cluster_barrier();  // keep every CTA's partial alive until all peers have read it
    }
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(L.tmem_cols)
                     : "memory");
    }
}

// ------------------------------------------------------------------ host side

template <int BITS, bool HAS_ZP>
cudaError_t set_attr() {
    return cudaFuncSetAttribute(gemm_kernel<BITS, HAS_ZP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)kSmemBudget);
}

template <int BITS, bool HAS_ZP>
cudaError_t launch(const CUtensorMap& tx, const CUtensorMap& tw, const CUtensorMap& ty, const GemmParams& P, int grid,
                   size_t smem, bool pdl,
                   cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (P.split > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = P.split;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    if (pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, gemm_kernel<BITS, HAS_ZP>, tx, tw, ty, P);
}

}  // namespace

int gemm_token_tile(int Mt) {
    if (Mt >= kMaxBN) return kMaxBN;
    int bn = (Mt + 15) / 16 * 16;
    return bn < 16 ? 16 : bn;
}

int gemm_threads() { return kThreads; }

// K splits per tile: enough CTAs for the SMs when the tiles alone are too few.
int gemm_split(int N, int Mt, int K, int sms) {
    const int BN = gemm_token_tile(Mt);
    const int tiles = ((N + BM - 1) / BM) * ((Mt + BN - 1) / BN);
    const int ksteps = (K + BK - 1) / BK;
    if (sms <= 0 || tiles * 2 > sms) return 1;
    int s = sms / tiles;
    if (s > kMaxSplit) s = kMaxSplit;
    if (s > ksteps) s = ksteps;
    return s < 2 ? 1 : s;
}

cudaError_t gemm_prepare() {
    cudaError_t e = tensor_map_prepare();
    if (e == cudaSuccess) e = set_attr<2, false>();
    if (e == cudaSuccess) e = set_attr<2, true>();
    if (e == cudaSuccess) e = set_attr<4, false>();
    if (e == cudaSuccess) e = set_attr<4, true>();
    if (e == cudaSuccess) e = set_attr<8, false>();
    if (e == cudaSuccess) e = set_attr<8, true>();
    return e;
}

cudaError_t gemm_launch(const GemmArgs& a, const mnb_plan_info& p, bool pdl, bool x_wait, cudaStream_t st) {
    GemmParams P;
    P.a = a;
    P.BN = p.tokens_per_cta;
    P.tiles_m = (a.Mt + P.BN - 1) / P.BN;
    P.tiles = P.tiles_m * ((a.N + BM - 1) / BM);
    P.ksteps = (a.K + BK - 1) / BK;
    P.split = p.k_splits > 1 ? p.k_splits : 1;
    P.x_wait = x_wait ? 1 : 0;
    P.ystage = P.split == 1 && a.N % 8 == 0 ? 1 : 0;  // TMA store: 16-byte row pitch
    P.tpre = P.ystage && a.rank > 0 ? 1 : 0;
    // Two K steps of X a copy where a whole row is one unit and its K steps pair
    // up: a copy costs the SM's TMA about the same time whatever its size, and one
    // 64-wide step of a 256-token tile is too little to keep the MMA fed.
    P.xk = (P.split == 1 && a.K % (2 * BK) == 0 && a.K * 2 / 128 <= 256 && gemm_layout(P.BN, 2, P.ystage).nx >= 2) ? 2 : 1;
    const GemmLayout L = gemm_layout(P.BN, P.xk, P.ystage);
    if (L.nx < 2 || L.total > kSmemBudget || (P.split > 1 && L.red_bytes > L.bar_off))
        return cudaErrorInvalidConfiguration;

    CUtensorMap tx;  // X [Mt x K] FP16: 2-D boxes of BN rows x 64, or 3-D boxes of two such K slices
    cudaError_t e = P.xk == 1 ? encode_2d(&tx, a.X, 2, (uint64_t)a.K, (uint64_t)a.Mt, (uint64_t)a.K * 2, (uint32_t)BK,
                                          (uint32_t)P.BN, true)
                              : encode_codes_sw128(&tx, a.X, (uint64_t)a.K * 2, (uint64_t)a.Mt, (uint32_t)P.BN, 2u);
    if (e != cudaSuccess) return e;
    CUtensorMap tw;  // packed weights [N rows x K*bits/8 bytes], boxes of 128 rows x 128 bytes
    e = encode_2d(&tw, a.Wq, 1, (uint64_t)a.K * a.bits / 8, (uint64_t)a.N, (uint64_t)a.K * a.bits / 8, 128u, (uint32_t)BM,
                  true);
    if (e != cudaSuccess) return e;
    CUtensorMap ty = tw;  // Y [Mt x N] FP16, boxes of BN tokens x 32 rows (unused without ystage)
    if (P.ystage) {
        e = encode_2d(&ty, a.Y, 2, (uint64_t)a.N, (uint64_t)a.Mt, (uint64_t)a.N * 2, 32u, (uint32_t)P.BN, false);
        if (e != cudaSuccess) return e;
    }
    const int grid = p.grid_x;
    const bool zp = a.Z != nullptr;
    if (a.bits == 2)
        return zp ? launch<2, true>(tx, tw, ty, P, grid, L.total, pdl, st)
                  : launch<2, false>(tx, tw, ty, P, grid, L.total, pdl, st);
    if (a.bits == 4)
        return zp ? launch<4, true>(tx, tw, ty, P, grid, L.total, pdl, st)
                  : launch<4, false>(tx, tw, ty, P, grid, L.total, pdl, st);
    return zp ? launch<8, true>(tx, tw, ty, P, grid, L.total, pdl, st)
              : launch<8, false>(tx, tw, ty, P, grid, L.total, pdl, st);
}

}  // namespace mnb
