// gemv.cu -- decode kernel (few token rows): a weight-streaming GEMV.
//
// Computes Y[m, n] = sum_k X[m, k] w[n, k] (+ sum_r T[m, r] B[n, r]) for up to
// 16 token rows per CTA, the "fuse_down" decode path of "[WebGPU] Fuse rank-32
// quantized LoRA with MatMulNBits" (onnxruntime PR 33370, commit message
// adding MatMulNBitsLoRA: base GEMV and LoRA down projection first, then the
// base plus T * Bt^T), restated for sm_103a:
//
//  * One launch may compute up to four projections of the same X (the fused
//    QKV / MLP projections of the empty-packed-weights commit referenced by
//    the same page): their 16-row groups are laid end to end and a small table
//    in parameter space gives each group its projection's pointers.
//  * Every packed weight byte is read from HBM once per token group.  Rows are
//    dealt out in whole 16-row groups: CTA c of C owns groups
//    [c G / C, (c+1) G / C) of the G = ceil(N / 16), and C is chosen so that
//    the most groups any SM has to run (CTAs per SM x groups per CTA) is least.
//  * A producer warp streams the CTA's rows through a ring of shared-memory
//    stages.  A stage is one 16-row group x one K chunk of at most 1 KB per
//    row: one 1-D bulk copy when a chunk is a full row (the rows are
//    contiguous), else one 3-D TMA box of 16 rows x 4 pieces of 256 bytes,
//    together with the group's scales, zero points and adapter rows B[n, :].
//    A copy costs about the same to issue whatever its size, so the copies
//    are few and large: per-row copies of 1 KB cannot feed an SM.
//    The producer never waits on the work queued before this kernel: weights
//    are prefetched while that work (or the LoRA down kernel) still runs.
//  * Eight consumer warps wait (griddepcontrol.wait) for X only when the
//    kernel may start before the work queued ahead of it has completed (early
//    weights, no adapter); after the LoRA down kernel of the same call -- which
//    lets this kernel start only once that work is complete -- they read X at
//    once and wait for T at the first group's epilogue, so the two kernels
//    overlap.  They split
//    each stage along K in 64-byte pieces: 16-byte loads of rows g and g+8
//    from shared memory, exact (q - zp) and one rounding by the scale in
//    registers (common.cuh), straight into mma.sync m16n8k16 A fragments with
//    the 8 or 16 token rows as the N side (FP32 accumulate, independent
//    accumulator chains, X fragments prefetched one stage ahead).  INT4 uses
//    the pair-interleaved unpacking (codes j and j + 4 of a word in one
//    half2), INT2 pairs codes j and j + 8; the same K permutation is applied
//    to the X fragment, which leaves the sum unchanged.
//  * After a group's last chunk warp 0 adds the LoRA term sum_r B[n, r] T[m, r]
//    to its accumulators (two m16n8k16 per token tile from the stage's B rows
//    and T in shared memory), the warps' partial sums are added in shared
//    memory in warp order (deterministic, no atomics), and each output is
//    rounded once to FP16.
//  * Waits on the ring are bounded and report through the status word.
#include <cstring>

#include "common.cuh"
#include "mnb_internal.h"

namespace mnb {

namespace {

constexpr int kConsumerWarps = 8;
constexpr int kThreadsGemv = (kConsumerWarps + 1) * 32;  // + one producer warp
constexpr int kMaxRing = 4;                                // most ring stages
constexpr uint32_t kXStageMax = 64 * 1024;                 // largest X tile staged in shared memory
constexpr uint32_t kXStageSmall = 24 * 1024;               // X tiles this small leave room for 3 CTAs per SM
constexpr uint32_t kTwoPerSm = 113 * 1024;                 // shared memory of a CTA when two share an SM
constexpr uint32_t kThreePerSm = 75 * 1024;                // ... and when three do
constexpr int kGroup = 16;                                 // rows per stage / MMA tile
constexpr int kMaxChunk = 1024;                            // K bytes per row and stage
// Inside a stage's adapter region (1 KB: 16 FP16 rows of B, or 16 INT8 rows of
// 32 bytes followed by their scales and zero points)
constexpr uint32_t kBqScale = 512;                         // 16 x 2 bytes (+ 16 bytes slack)
constexpr uint32_t kBqZero = 576;                          // 16 bytes (+ 16 bytes slack)

struct GemvLayout {
    uint32_t stage;            // bytes of one ring stage
    uint32_t w, sc, zp, b;     // offsets inside a stage: codes, scales, zero points, B rows
    uint32_t x, t, red, bars, total;
};

__host__ __device__ inline uint32_t align_up(uint32_t x, uint32_t a) { return (x + a - 1) / a * a; }

// Bytes per staged FP16 X row: 16 bytes of padding put the eight token rows a
// thread quad column reads in distinct banks.
__host__ __device__ inline uint32_t xs_pitch(int K) { return (uint32_t)K * 2u + 16u; }

// Shared-memory layout, identical on host and device.  `ch` = K bytes per chunk,
// `ring` = stages (2 to 4), `xbytes` = staged X (0 when X is read from global).
__host__ __device__ inline GemvLayout gemv_layout(int ch, int nblk, int tok, int ring, uint32_t xbytes) {
    GemvLayout L;
    L.w = 0;
    L.sc = align_up((uint32_t)kGroup * ch + 128u, 128u);  // + slack: the last 128-byte piece may pass CH
    L.zp = L.sc + align_up((uint32_t)kGroup * nblk * 2u + 32u, 128u);
    L.b = L.zp + align_up((uint32_t)kGroup * nblk + 32u, 128u);
    L.stage = L.b + kGroup * 64u;
    uint32_t off = (uint32_t)ring * L.stage;
    L.x = off;
    off += align_up(xbytes, 128u);
    L.t = off;
    off += align_up((uint32_t)tok * 64u, 128u);
    L.red = off;  // two buffers (alternate groups)
    off += 2u * kConsumerWarps * kGroup * tok * 4u;
    L.bars = align_up(off, 16u);
    L.total = L.bars + 2 * (uint32_t)ring * 8;
    return L;
}

// CTAs per SM: three when there are rows enough for them and the kernel is a
// single-token-tile one with X staged (it then fits 72 registers without
// spilling and a two-stage ring in a third of the shared memory), two
// otherwise (96 registers: more independent work per thread).
inline int gemv_ctas_per_sm(int N, int nt, uint32_t xbytes, int sms) {
    return nt == 1 && xbytes > 0 && xbytes <= kXStageSmall && (N + kGroup - 1) / kGroup > 2 * sms ? 3 : 2;
}

// Ring stages with two CTAs per SM: two when a CTA has at most two stages, else four.
inline int gemv_ring(int nstages) { return nstages <= 2 ? 2 : kMaxRing; }

// The ring for a CTA.  Two CTAs per SM: four stages, or two when four would not
// leave room for both next to a large staged X tile.  Three CTAs per SM (small
// stages): the deepest ring of up to four stages that fits a third of the SM.
inline int gemv_pick_ring(int ch, int nblk, int tok, int nstages, int occ, uint32_t xbytes) {
    if (occ == 3) {
        for (int ring = kMaxRing; ring > 2; --ring)
            if (ring <= nstages && gemv_layout(ch, nblk, tok, ring, xbytes).total <= kThreePerSm) return ring;
        return 2;
    }
    const int ring = gemv_ring(nstages);
    return ring > 2 && gemv_layout(ch, nblk, tok, ring, xbytes).total > kTwoPerSm ? 2 : ring;
}

__device__ __forceinline__ uint32_t word_of(const uint4& v, int i) {
    return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// Plain C++ shared-memory loads (byte offsets into the dynamic shared array):
// ordered after the mbarrier waits by their memory clobber, otherwise free to
// be scheduled early by the compiler.
__device__ __forceinline__ uint4 lds128(const unsigned char* sm, uint32_t off) {
    return *reinterpret_cast<const uint4*>(sm + off);
}
__device__ __forceinline__ uint32_t lds_u16(const unsigned char* sm, uint32_t off) {
    return *reinterpret_cast<const uint16_t*>(sm + off);
}
__device__ __forceinline__ uint32_t lds_u8(const unsigned char* sm, uint32_t off) { return sm[off]; }

// Int8-activation path: staged position p of a 32-code block holds the code
// of K index q8x_perm<BITS>(p) within the block -- the order in which a thread
// quad's share of the block comes out of the weight unpacking (thread t of a
// quad owns codes 8t .. 8t+7; k-slots 4t..4t+3 and 16+4t..16+4t+3 of the
// m16n8k32 fragment).
template <int BITS>
__host__ __device__ constexpr int q8x_perm(int p) {
    return BITS == 8 ? p
         : BITS == 4 ? 8 * ((p & 15) >> 2) + 2 * (p & 3) + (p >> 4)
                     : 8 * ((p & 15) >> 2) + 2 * (p >> 4) + 4 * (p & 1) + ((p & 3) >> 1);
}

// 4 x 4 transpose of 32-bit words across the lanes of a thread quad (t = lane & 3):
// on return w[j] holds word t of quad lane j's input.  Four shuffles.
__device__ __forceinline__ void quad_transpose(uint32_t w[4], int t) {
    const bool o = (t & 1) != 0, hi = (t & 2) != 0;
    const uint32_t a = __shfl_xor_sync(0xffffffffu, o ? w[0] : w[1], 1);
    const uint32_t b = __shfl_xor_sync(0xffffffffu, o ? w[2] : w[3], 1);
    if (o) {
        w[0] = a;
        w[2] = b;
    } else {
        w[1] = a;
        w[3] = b;
    }
    const uint32_t c = __shfl_xor_sync(0xffffffffu, hi ? w[0] : w[2], 2);
    const uint32_t d = __shfl_xor_sync(0xffffffffu, hi ? w[1] : w[3], 2);
    if (hi) {
        w[0] = c;
        w[1] = d;
    } else {
        w[2] = c;
        w[3] = d;
    }
}

// Staged int8 X of one token tile: codes [tok][K + 16] (padded rows: the
// B-operand loads of 8 token rows hit distinct banks), then per (token, block)
// the binary32 scale and the code sum.
__host__ __device__ inline uint32_t q8x_stage_bytes(int tok, int K) {
    return (uint32_t)tok * ((uint32_t)K + 16u) + (uint32_t)tok * (uint32_t)(K / 32) * 8u;
}

// 3-D TMA descriptors of the projections' packed weights (multi-chunk stages).
struct GemvMaps {
    CUtensorMap m[kMaxSeg];
};

// Ring slot and pass parity of stage st.  Three-CTA kernels may run rings of
// three stages and step a counter; the others have rings of two or four
// stages and take them from st (both forms give the same slot and parity).
template <int OCC>
struct RingPosT {
    int s = 0;
    uint32_t ph = 0;
    __device__ __forceinline__ void step(int ring) {
        if constexpr (OCC == 3) {
            if (++s == ring) {
                s = 0;
                ph ^= 1u;
            }
        }
    }
    __device__ __forceinline__ int slot(int st, int rmask) const { return OCC == 3 ? s : st & rmask; }
    __device__ __forceinline__ uint32_t parity(int st, int ring) const {
        return OCC == 3 ? ph : (uint32_t)(st / ring) & 1u;
    }
};

template <int BITS, bool HAS_ZP, int NT, bool XS, int OCC, bool Q8X>
__global__ void __launch_bounds__(kThreadsGemv, OCC)
    gemv_kernel(const __grid_constant__ GemvMaps maps, const __grid_constant__ GemvArgs a) {
    static_assert(!Q8X || (NT == 1 && XS), "the int8-activation path stages one 8-token tile");
    extern __shared__ __align__(1024) unsigned char sm[];
    constexpr int TOK = 8 * NT;
    constexpr uint32_t kDefaultZp = 1u << (BITS - 1);
    constexpr int kBpb = 32 * BITS / 8;  // packed bytes per quantization block

    const int nblk = a.K >> 5;
    const int rowbytes = a.K * BITS / 8;
    const int CH = a.CH;                                  // K bytes per chunk
    const int nchunk = (rowbytes + CH - 1) / CH;
    const int ring = a.ring, rmask = a.ring - 1;
    const GemvLayout L =
        gemv_layout(CH, nblk, TOK, ring, Q8X ? q8x_stage_bytes(TOK, a.K) : XS ? (uint32_t)a.xrows * xs_pitch(a.K) : 0u);
    const uint32_t sb = smem_u32(sm);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // groups [g_begin, g_end) of the row space of all projections
    const int G = a.G;
    const int g_begin = (int)((long long)blockIdx.x * G / gridDim.x);
    const int ngroups = (int)((long long)(blockIdx.x + 1) * G / gridDim.x) - g_begin;
    // projection owning group gq (the table lives in parameter space: no local copy)
    auto seg_of = [&](int gq) {
        int sg = 0;
#pragma unroll
        for (int i = 1; i < kMaxSeg; ++i) sg += (i < a.nseg && gq >= a.seg[i].g0) ? 1 : 0;
        return sg;
    };
    const int nstages = ngroups * nchunk;
    const int token0 = blockIdx.y * TOK;
    unsigned int* status = a.status;

    auto full = [&](int s) { return sb + L.bars + 8u * s; };
    auto empty = [&](int s) { return sb + L.bars + 8u * (ring + s); };

    if (threadIdx.x == 0) {
        for (int s = 0; s < ring; ++s) {
            mbar_init(full(s), 2);  // lane 0: bulk copies (+ bytes); lane 1: tail bytes
            mbar_init(empty(s), kConsumerWarps);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    pdl_launch_dependents();

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------------ producer
        if (lane < 2) {
            bool ok = true;
            RingPosT<OCC> rp;
            for (int st = 0; ok && st < nstages; ++st, rp.step(ring)) {
                const int s = rp.slot(st, rmask);
                const int q = st / nchunk, c = st - q * nchunk;
                const int sg = seg_of(g_begin + q);
                const GemvSeg& pj = a.seg[sg];
                const int ra = (g_begin + q - pj.g0) * kGroup, rows = min(kGroup, pj.N - ra);  // rows of projection sg
                const uint64_t total_s = (uint64_t)pj.N * nblk * 2, total_z = (uint64_t)pj.N * nblk;
                const uint32_t slot = sb + (uint32_t)s * L.stage;
                if (!(ok = mbar_wait(empty(s), rp.parity(st, ring) ^ 1u, status))) break;
                // scales / zero points of the group's full rows as 16-byte aligned supersets;
                // bytes past the last 16-byte boundary of an array come from lane 1
                const uint64_t s0 = (uint64_t)ra * nblk * 2, s1 = (uint64_t)(ra + rows) * nblk * 2;
                const uint64_t s_lo = s0 & ~15ull, s_hi = min((s1 + 15) & ~15ull, total_s & ~15ull);
                const uint64_t z0 = (uint64_t)ra * nblk, z1 = (uint64_t)(ra + rows) * nblk;
                const uint64_t z_lo = z0 & ~15ull, z_hi = min((z1 + 15) & ~15ull, total_z & ~15ull);
                // INT8 adapter rows: their scales (2 bytes) and zero points (1 byte) the same way;
                // ra is a multiple of 16, so both start on a 16-byte boundary
                const uint64_t qs0 = (uint64_t)ra * 2, qs1 = (uint64_t)(ra + rows) * 2;
                const uint64_t qs_lo = qs0, qs_hi = min((qs1 + 15) & ~15ull, ((uint64_t)pj.N * 2) & ~15ull);
                const uint64_t qz_lo = (uint64_t)ra, qz1 = (uint64_t)(ra + rows);
                const uint64_t qz_hi = min((qz1 + 15) & ~15ull, (uint64_t)pj.N & ~15ull);
                if (lane == 0) {
                    const int cb = min(CH, rowbytes - c * CH);  // bytes of this chunk per row
                    // a 3-D box always lands whole (rows past N, pieces past K read as zero)
                    uint32_t bytes = nchunk > 1 && a.w3d ? (uint32_t)kGroup * (uint32_t)CH : (uint32_t)rows * (uint32_t)cb;
                    if (s_hi > s_lo) bytes += (uint32_t)(s_hi - s_lo);
                    if (HAS_ZP && z_hi > z_lo) bytes += (uint32_t)(z_hi - z_lo);
                    if (a.rank > 0) bytes += (uint32_t)rows * (a.Bq ? 32u : 64u);
                    if (a.rank > 0 && a.Bq) {
                        if (qs_hi > qs_lo) bytes += (uint32_t)(qs_hi - qs_lo);
                        if (a.Bz && qz_hi > qz_lo) bytes += (uint32_t)(qz_hi - qz_lo);
                    }
                    mbar_arrive_tx(full(s), bytes);
                    const uint8_t* src = pj.Wq + (size_t)ra * rowbytes + (size_t)c * CH;
                    if (nchunk == 1) {
                        bulk_load(slot + L.w, src, (uint32_t)(rows * rowbytes), full(s));  // rows are contiguous
                    } else if (a.w3d) {
                        tma_load_3d(slot + L.w, &maps.m[sg], 0, c * CH / 256, ra, full(s));
                    } else {
                        for (int i = 0; i < rows; ++i)
                            bulk_load(slot + L.w + (uint32_t)(i * CH), src + (size_t)i * rowbytes, (uint32_t)cb, full(s));
                    }
                    if (s_hi > s_lo)
                        bulk_load(slot + L.sc, reinterpret_cast<const uint8_t*>(pj.S) + s_lo, (uint32_t)(s_hi - s_lo),
                                  full(s));
                    if (HAS_ZP && z_hi > z_lo) bulk_load(slot + L.zp, pj.Z + z_lo, (uint32_t)(z_hi - z_lo), full(s));
                    if (a.rank > 0 && !a.Bq) bulk_load(slot + L.b, a.B + (size_t)ra * 32, (uint32_t)rows * 64u, full(s));
                    if (a.rank > 0 && a.Bq) {
                        bulk_load(slot + L.b, a.Bq + (size_t)ra * 32, (uint32_t)rows * 32u, full(s));
                        if (qs_hi > qs_lo)
                            bulk_load(slot + L.b + kBqScale, reinterpret_cast<const uint8_t*>(a.Bs) + qs_lo,
                                      (uint32_t)(qs_hi - qs_lo), full(s));
                        if (a.Bz && qz_hi > qz_lo)
                            bulk_load(slot + L.b + kBqZero, a.Bz + qz_lo, (uint32_t)(qz_hi - qz_lo), full(s));
                    }
                } else {
                    unsigned char* st8 = sm + (uint32_t)s * L.stage;
                    for (uint64_t i = max(s_hi, s_lo); i < s1; ++i)
                        st8[L.sc + (uint32_t)(i - s_lo)] = reinterpret_cast<const uint8_t*>(pj.S)[i];
                    if (HAS_ZP)
                        for (uint64_t i = max(z_hi, z_lo); i < z1; ++i) st8[L.zp + (uint32_t)(i - z_lo)] = pj.Z[i];
                    if (a.rank > 0 && a.Bq) {
                        for (uint64_t i = max(qs_hi, qs_lo); i < qs1; ++i)
                            st8[L.b + kBqScale + (uint32_t)(i - qs_lo)] = reinterpret_cast<const uint8_t*>(a.Bs)[i];
                        if (a.Bz)
                            for (uint64_t i = max(qz_hi, qz_lo); i < qz1; ++i)
                                st8[L.b + kBqZero + (uint32_t)(i - qz_lo)] = a.Bz[i];
                    }
                    mbar_arrive(full(s));
                }
            }
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int g = lane >> 2, t = lane & 3;
    const int ctid = threadIdx.x;  // 0..255
    if (a.x_wait) pdl_wait();  // X is produced by work queued before this kernel
    bool t_ready = a.rank == 0;
    if constexpr (Q8X) {
        // X rows of this token group quantized to int8 per block of 32 (quantize_block32),
        // codes stored in q8x_perm order; rows past Mt get scale 0 and sum 0
        const uint32_t xp = (uint32_t)a.K + 16u;
        float* xsc = reinterpret_cast<float*>(sm + L.x + TOK * xp);
        int* xsum = reinterpret_cast<int*>(xsc + TOK * nblk);
        const int mv = min(TOK, a.Mt - token0);
        for (int i = ctid; i < TOK * nblk; i += kConsumerWarps * 32) {
            const int row = i / nblk, b = i - row * nblk;
            if (row >= mv) {
                xsc[i] = 0.f;
                xsum[i] = 0;
                continue;
            }
            int qv[32], sum;
            const float scale = quantize_block32(a.X + (size_t)(token0 + row) * a.K + b * 32, qv, sum);
            uint32_t wd[8];
#pragma unroll
            for (int p4 = 0; p4 < 8; ++p4) {
                uint32_t w = 0;
#pragma unroll
                for (int j = 0; j < 4; ++j) w |= ((uint32_t)qv[q8x_perm<BITS>(4 * p4 + j)] & 0xFFu) << (8 * j);
                wd[p4] = w;
            }
            uint4* dst = reinterpret_cast<uint4*>(sm + L.x + (uint32_t)row * xp + (uint32_t)b * 32u);
            dst[0] = make_uint4(wd[0], wd[1], wd[2], wd[3]);
            dst[1] = make_uint4(wd[4], wd[5], wd[6], wd[7]);
            xsc[i] = scale;
            xsum[i] = sum;
        }
        named_barrier_sync(1, kConsumerWarps * 32);
    } else if (XS) {
        // X rows of this token group into shared memory, once; for INT4 each group
        // of 8 codes is stored in the pair-interleaved order (0,4,1,5,2,6,3,7) the
        // unpacking produces, so the inner loop needs no permutes.
        const int mv = min(TOK, a.Mt - token0);
        if constexpr (BITS == 2) {
            // INT2: each group of 16 codes as the pairs (x_j, x_{j+8}), j = 0..7
            const int kc = a.K / 16;
            for (int i = ctid; i < mv * kc; i += kConsumerWarps * 32) {
                const int row = i / kc, c16 = i - row * kc;
                const uint4* src = reinterpret_cast<const uint4*>(a.X + (size_t)(token0 + row) * a.K) + 2 * c16;
                const uint4 v0 = __ldg(src), v1 = __ldg(src + 1);
                uint32_t xw[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) xw[j] = prmt(word_of(v0, j >> 1), word_of(v1, j >> 1), (j & 1) ? 0x7632u : 0x5410u);
                uint4* dst = reinterpret_cast<uint4*>(sm + L.x + (uint32_t)row * xs_pitch(a.K) + (uint32_t)c16 * 32u);
                dst[0] = make_uint4(xw[0], xw[1], xw[2], xw[3]);
                dst[1] = make_uint4(xw[4], xw[5], xw[6], xw[7]);
            }
        } else {
            const int kc = a.K / 8;
            for (int i = ctid; i < mv * kc; i += kConsumerWarps * 32) {
                const int row = i / kc, c8 = i - row * kc;
                uint4 v = __ldg(reinterpret_cast<const uint4*>(a.X + (size_t)(token0 + row) * a.K) + c8);
                if (BITS == 4)
                    v = make_uint4(prmt(v.x, v.z, 0x5410u), prmt(v.x, v.z, 0x7632u), prmt(v.y, v.w, 0x5410u),
                                   prmt(v.y, v.w, 0x7632u));
                *reinterpret_cast<uint4*>(sm + L.x + (uint32_t)row * xs_pitch(a.K) + (uint32_t)c8 * 16u) = v;
            }
        }
        named_barrier_sync(1, kConsumerWarps * 32);
    }
    float* red = reinterpret_cast<float*>(sm + L.red);
    const int npieces = (CH + 127) / 128;  // 128-byte pieces per chunk row: 32 bytes per thread and row
    // shared-memory row pitch: a single-chunk group is one contiguous copy of full rows
    const uint32_t pitch = nchunk == 1 ? (uint32_t)rowbytes : (uint32_t)CH;

    // Independent accumulator chains per n8 tile, summed at the end of a group,
    // so consecutive MMAs of a warp do not wait on each other.
    constexpr int kChains = NT == 1 ? 4 : 2;
    float acc[NT][kChains][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int qq = 0; qq < kChains; ++qq)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[nt][qq][e] = 0.f;

    // Loop-invariant per-thread pieces of every address.  Loads are issued
    // unconditionally at clamped, in-bounds addresses; invalid values are then
    // replaced by zeros with selects, so the inner loop has no branches.
    const __half* xrow[NT];
    bool xok[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int tok = token0 + nt * 8 + g;
        xok[nt] = tok < a.Mt;
        xrow[nt] = a.X + (size_t)(xok[nt] ? tok : 0) * a.K;
    }
    const int Mt = a.Mt, rank = a.rank;
    // last X element offset at which one half's X loads (8 halfs per 16-byte load) stay inside the row
    const int xmax = a.K - 8 * (BITS == 4 ? 4 : 2);
    const uint32_t w_thr = L.w + (uint32_t)g * pitch + (uint32_t)t * 32u;      // row g, this thread's 32 bytes
    const uint32_t w_rowB = 8u * pitch;                                         // row g+8 relative to row g
    const uint32_t s_thr = L.sc + (uint32_t)g * (uint32_t)nblk * 2u;           // scales of row g
    const uint32_t z_thr = L.zp + (uint32_t)g * (uint32_t)nblk;                // zero points of row g
    const uint32_t s_rowB = 8u * (uint32_t)nblk * 2u, z_rowB = 8u * (uint32_t)nblk;
    const int blk_thr = t * 32 / kBpb;  // block of the thread's first byte within a 128-byte piece

    bool ok = true;
    int q = 0, c = 0;  // group and chunk of stage st (counters: no divisions in the loop)
    RingPosT<OCC> rp;
    for (int st = 0; st < nstages; ++st, rp.step(ring)) {
        const int s = rp.slot(st, rmask);
        const GemvSeg& pj = a.seg[seg_of(g_begin + q)];
        const int ra = (g_begin + q - pj.g0) * kGroup, rows = min(kGroup, pj.N - ra);  // rows of this projection
        if (ok) ok = mbar_wait(full(s), rp.parity(st, ring), status);
        const uint32_t soff = (uint32_t)s * L.stage;  // byte offset of the stage in `sm`
        const uint32_t s_al = ((uint32_t)ra * (uint32_t)nblk * 2u) & 15u;  // scale copy alignment offset
        const uint32_t z_al = ((uint32_t)ra * (uint32_t)nblk) & 15u;
        const bool vA = g < rows, vB = g + 8 < rows;
        const int kchunk = c * CH;
        if constexpr (Q8X) {
            // One 32-code block per warp step: quad thread t unpacks codes 8t..8t+7 of
            // rows g and g+8 into u8 fragments, one m16n8k32 gives the exact int32 dot
            // with the token rows' int8 codes, then y += sw * sx * (dot - zp * sum(xq)).
            const uint32_t xp = (uint32_t)a.K + 16u;
            const float* xsc = reinterpret_cast<const float*>(sm + L.x + TOK * xp);
            const int* xsum = reinterpret_cast<const int*>(xsc + TOK * nblk);
            // per block: the int32 dot and its scaling into the accumulators
            auto block_dot = [&](int blk, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3) {
                const uint32_t so = soff + s_thr + s_al + (uint32_t)blk * 2u;
                const uint32_t s0bits = lds_u16(sm, so), s8bits = lds_u16(sm, so + s_rowB);
                const float swA = vA ? __half2float(__ushort_as_half((unsigned short)s0bits)) : 0.f;
                const float swB = vB ? __half2float(__ushort_as_half((unsigned short)s8bits)) : 0.f;
                int zA = (int)kDefaultZp, zB = (int)kDefaultZp;
                if (HAS_ZP) {
                    const uint32_t zo = soff + z_thr + z_al + (uint32_t)blk;
                    zA = (int)lds_u8(sm, zo);
                    zB = (int)lds_u8(sm, zo + z_rowB);
                }
                const uint32_t xo = L.x + (uint32_t)g * xp + (uint32_t)blk * 32u;
                const uint32_t b0 = *reinterpret_cast<const uint32_t*>(sm + xo + 4 * t);
                const uint32_t b1 = *reinterpret_cast<const uint32_t*>(sm + xo + 16 + 4 * t);
                int d[4];
                mma_16832_u8s8(d, a0, a1, a2, a3, b0, b1);
                const int t0 = 2 * t;  // token rows of (d0, d2) and (d1, d3): t0, t0 + 1
                const float sx0 = xsc[t0 * nblk + blk], sx1 = xsc[(t0 + 1) * nblk + blk];
                const int q0 = xsum[t0 * nblk + blk], q1 = xsum[(t0 + 1) * nblk + blk];
                float* ac = acc[0][0];
                ac[0] = fmaf((float)(d[0] - zA * q0), swA * sx0, ac[0]);
                ac[1] = fmaf((float)(d[1] - zA * q1), swA * sx1, ac[1]);
                ac[2] = fmaf((float)(d[2] - zB * q0), swB * sx0, ac[2]);
                ac[3] = fmaf((float)(d[3] - zB * q1), swB * sx1, ac[3]);
            };
            if constexpr (BITS != 2) {
                // 128 bytes of rows g and g+8 per warp step: each lane loads 16 bytes from
                // either 64-byte half (even rows the first half first, odd rows the second:
                // every load instruction covers all 32 banks), then a quad transpose gives
                // lane t word t of each 16-byte chunk -- its share of the fragment.
                for (int sp = warp; ok && sp < npieces; sp += kConsumerWarps) {
                    const int kseg = kchunk + sp * 128;
                    if (kseg >= rowbytes) break;
                    const uint32_t odd = (uint32_t)(g & 1);
                    const uint32_t rA = soff + L.w + (uint32_t)g * pitch + (uint32_t)sp * 128u + 16u * (uint32_t)t;
                    const uint4 l0 = lds128(sm, rA + 64u * odd), l1 = lds128(sm, rA + 64u * (1u - odd));
                    const uint4 l2 = lds128(sm, rA + w_rowB + 64u * odd), l3 = lds128(sm, rA + w_rowB + 64u * (1u - odd));
                    const uint4 pA = odd ? l1 : l0, qA = odd ? l0 : l1, pB = odd ? l3 : l2, qB = odd ? l2 : l3;
                    uint32_t PA[4] = {pA.x, pA.y, pA.z, pA.w}, QA[4] = {qA.x, qA.y, qA.z, qA.w};
                    uint32_t PB[4] = {pB.x, pB.y, pB.z, pB.w}, QB[4] = {qB.x, qB.y, qB.z, qB.w};
                    quad_transpose(PA, t);
                    quad_transpose(QA, t);
                    quad_transpose(PB, t);
                    quad_transpose(QB, t);
                    if constexpr (BITS == 4) {  // 16-byte blocks: chunk j is block j
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const int kbyte = kseg + 16 * j;
                            if (kbyte >= rowbytes) break;
                            const uint32_t u = j < 4 ? PA[j & 3] : QA[j & 3], v = j < 4 ? PB[j & 3] : QB[j & 3];
                            block_dot(kbyte / kBpb, u & 0x0F0F0F0Fu, v & 0x0F0F0F0Fu, (u >> 4) & 0x0F0F0F0Fu,
                                      (v >> 4) & 0x0F0F0F0Fu);
                        }
                    } else {  // 32-byte blocks: chunks 2j, 2j+1 are block j
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const int kbyte = kseg + 32 * j;
                            if (kbyte >= rowbytes) break;
                            const uint32_t a0 = j < 2 ? PA[(2 * j) & 3] : QA[(2 * j) & 3];
                            const uint32_t a2 = j < 2 ? PA[(2 * j + 1) & 3] : QA[(2 * j + 1) & 3];
                            const uint32_t a1 = j < 2 ? PB[(2 * j) & 3] : QB[(2 * j) & 3];
                            const uint32_t a3 = j < 2 ? PB[(2 * j + 1) & 3] : QB[(2 * j + 1) & 3];
                            block_dot(kbyte / kBpb, a0, a1, a2, a3);
                        }
                    }
                }
            } else {
            // INT2 (8-byte blocks): one block per warp step, each thread's 2 bytes of
            // rows g and g+8 loaded directly
            const int bpc = CH / kBpb;
            for (int bl = warp; ok && bl < bpc; bl += kConsumerWarps) {
                const int kbyte = kchunk + bl * kBpb;
                if (kbyte >= rowbytes) break;
                const uint32_t wa = soff + L.w + (uint32_t)g * pitch + (uint32_t)(bl * kBpb);
                const uint32_t u = lds_u16(sm, wa + 2 * t), v = lds_u16(sm, wa + w_rowB + 2 * t);
                block_dot(kbyte / kBpb, (u & 0x0303u) | (((u >> 2) & 0x0303u) << 16),
                          (v & 0x0303u) | (((v >> 2) & 0x0303u) << 16),
                          ((u >> 4) & 0x0303u) | (((u >> 6) & 0x0303u) << 16),
                          ((v >> 4) & 0x0303u) | (((v >> 6) & 0x0303u) << 16));
            }
            }
        } else
        for (int p = warp; ok && p < npieces; p += kConsumerWarps) {
            const int kb = kchunk + p * 128 + t * 32;  // first byte of this thread's 32 in the row
            const uint32_t wpc = soff + w_thr + (uint32_t)p * 128u;
            const int blk0 = (kchunk + p * 128) / kBpb + blk_thr;
#pragma unroll
            for (int h = 0; h < 2; ++h) {  // two 16-byte halves
                const int kbh = kb + 16 * h;
                const bool kv = kbh < rowbytes;
                if constexpr (BITS == 2) {
                    // 16 bytes = 64 codes = two blocks: words 2 bb and 2 bb + 1 are block
                    // blk0 + 2 h + bb.  K % 64 == 0, so a half is whole or wholly past K.
                    const int kx = kbh * 4;  // first code of the half
                    const uint4 wa = lds128(sm, wpc + 16u * h);
                    const uint4 wb = lds128(sm, wpc + 16u * h + w_rowB);
#pragma unroll
                    for (int bb = 0; bb < 2; ++bb) {
                        const int blk = blk0 + 2 * h + bb;
                        const uint32_t so = soff + s_thr + s_al + (uint32_t)blk * 2u;
                        const uint32_t sa0 = lds_u16(sm, so), sb0 = lds_u16(sm, so + s_rowB);
                        const uint32_t sa = (kv && vA) ? sa0 : 0u;
                        const uint32_t sbv = (kv && vB) ? sb0 : 0u;
                        uint32_t za = kDefaultZp, zb = kDefaultZp;
                        if (HAS_ZP) {
                            const uint32_t zo = soff + z_thr + z_al + (uint32_t)blk;
                            za = lds_u8(sm, zo);
                            zb = lds_u8(sm, zo + z_rowB);
                        }
                        const Dq2Const cA = dq2_const(za, (uint16_t)sa);
                        const Dq2Const cB = dq2_const(zb, (uint16_t)sbv);
#pragma unroll
                        for (int ww = 0; ww < 2; ++ww) {
                            const int w = 2 * bb + ww;
                            uint32_t dA[8], dB[8];
                            dq_int2_interleaved(word_of(wa, w), cA, dA);
                            dq_int2_interleaved(word_of(wb, w), cB, dB);
#pragma unroll
                            for (int nt = 0; nt < NT; ++nt) {
                                // X pairs (x_j, x_{j+8}) of the word's 16 codes
                                const bool use = kv && xok[nt];
                                uint4 v0 = make_uint4(0, 0, 0, 0), v1 = v0;
                                uint32_t xw[8];
                                if (XS) {
                                    if (use) {
                                        const uint32_t xo = L.x + (uint32_t)(nt * 8 + g) * xs_pitch(a.K) + (uint32_t)(kx + 16 * w) * 2u;
                                        v0 = lds128(sm, xo);
                                        v1 = lds128(sm, xo + 16u);
                                    }
#pragma unroll
                                    for (int j = 0; j < 4; ++j) {
                                        xw[j] = word_of(v0, j);
                                        xw[4 + j] = word_of(v1, j);
                                    }
                                } else {
                                    if (use) {
                                        const uint4* xp = reinterpret_cast<const uint4*>(xrow[nt] + kx + 16 * w);
                                        v0 = __ldg(xp);
                                        v1 = __ldg(xp + 1);
                                    }
#pragma unroll
                                    for (int j = 0; j < 8; ++j)
                                        xw[j] = prmt(word_of(v0, j >> 1), word_of(v1, j >> 1), (j & 1) ? 0x7632u : 0x5410u);
                                }
#pragma unroll
                                for (int i = 0; i < 4; ++i)
                                    mma_16816(acc[nt][(4 * w + i) % kChains], dA[2 * i], dB[2 * i], dA[2 * i + 1],
                                              dB[2 * i + 1], xw[2 * i], xw[2 * i + 1]);
                            }
                        }
                    }
                    continue;
                }
                const int blk = blk0 + (BITS == 4 ? h : 0);
                // X of these 16 bytes' codes, for this thread's token rows
                constexpr int kXv = BITS == 4 ? 4 : 2;
                const int kx = min(kbh * 8 / BITS, xmax);
                uint4 xv[NT][kXv];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const bool use = kv && xok[nt];
#pragma unroll
                    for (int w = 0; w < kXv; ++w) {
                        uint4 v = make_uint4(0, 0, 0, 0);
                        if (XS) {
                            if (use) v = lds128(sm, L.x + (uint32_t)(nt * 8 + g) * xs_pitch(a.K) + (uint32_t)kx * 2u + 16u * w);
                        } else {
                            if (use) v = __ldg(reinterpret_cast<const uint4*>(xrow[nt] + kx) + w);  // predicated
                        }
                        xv[nt][w] = v;
                    }
                }
                const uint4 wa = lds128(sm, wpc + 16u * h);
                const uint4 wb = lds128(sm, wpc + 16u * h + w_rowB);
                const uint32_t so = soff + s_thr + s_al + (uint32_t)blk * 2u;
                const uint32_t sa0 = lds_u16(sm, so), sb0 = lds_u16(sm, so + s_rowB);
                const uint32_t sa = (kv && vA) ? sa0 : 0u;  // a zero scale removes the row / K tail
                const uint32_t sbv = (kv && vB) ? sb0 : 0u;
                uint32_t za = kDefaultZp, zb = kDefaultZp;
                if (HAS_ZP) {
                    const uint32_t zo = soff + z_thr + z_al + (uint32_t)blk;
                    za = lds_u8(sm, zo);
                    zb = lds_u8(sm, zo + z_rowB);
                }
                const DqConst cA = dq_const(za, (uint16_t)sa);
                const DqConst cB = dq_const(zb, (uint16_t)sbv);
                if constexpr (BITS == 4) {
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        uint32_t dA[4], dB[4];
                        dq_int4_interleaved(word_of(wa, w), cA, dA);
                        dq_int4_interleaved(word_of(wb, w), cB, dB);
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            const uint4 x = xv[nt][w];
                            // staged X is already in pair-interleaved order
                            const uint32_t x04 = XS ? x.x : prmt(x.x, x.z, 0x5410u);
                            const uint32_t x15 = XS ? x.y : prmt(x.x, x.z, 0x7632u);
                            const uint32_t x26 = XS ? x.z : prmt(x.y, x.w, 0x5410u);
                            const uint32_t x37 = XS ? x.w : prmt(x.y, x.w, 0x7632u);
                            mma_16816(acc[nt][(2 * w) % kChains], dA[0], dB[0], dA[1], dB[1], x04, x15);
                            mma_16816(acc[nt][(2 * w + 1) % kChains], dA[2], dB[2], dA[3], dB[3], x26, x37);
                        }
                    }
                } else {
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        uint32_t dA[2], dB[2];
                        dq_int8_natural(word_of(wa, w), cA, dA);
                        dq_int8_natural(word_of(wb, w), cB, dB);
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            const uint4 x = xv[nt][w >> 1];
                            const uint32_t b0 = (w & 1) == 0 ? x.x : x.z;
                            const uint32_t b1 = (w & 1) == 0 ? x.y : x.w;
                            mma_16816(acc[nt][w % kChains], dA[0], dB[0], dA[1], dB[1], b0, b1);
                        }
                    }
                }
            }
        }
        const bool last_chunk = c == nchunk - 1;
        if (++c == nchunk) {
            c = 0;
            ++q;
        }
        if (!last_chunk) {
            __syncwarp();
            if (ok && lane == 0) mbar_arrive(empty(s));
            continue;
        }

        // Last chunk of the group: partial sums (row g, tokens 2t, 2t+1), (row g+8,
        // same), per n8 tile.  The buffer alternates between groups, so one barrier
        // per group suffices: a warp writes the partials of group q+2 only after
        // every warp passed group q+1's barrier, i.e. after all reads of group q.
        if (!t_ready) {  // first epilogue: T of the LoRA down kernel queued just before
            pdl_wait();
            for (int i = ctid; i < TOK * 32; i += kConsumerWarps * 32) {
                const int tok = token0 + i / 32;
                reinterpret_cast<__half*>(sm + L.t)[i] =
                    tok < a.Mt ? a.T[(size_t)tok * 32 + (i & 31)] : __float2half_rn(0.f);
            }
            named_barrier_sync(1, kConsumerWarps * 32);
            t_ready = true;
        }
        if (rank > 0 && warp == 0) {
            // LoRA term of the group's 16 rows, sum_r B[n, r] T[m, r], on the tensor
            // cores: two m16n8k16 per token tile (A = the stage's B rows, B = T),
            // into this warp's accumulators, so the warp-order sum below adds it.
            const unsigned char* bs = sm + soff + L.b;  // 16 rows x 32 halves (INT8: 16 rows x 32 bytes)
            const unsigned char* ts = sm + L.t;         // TOK rows x 32 halves
            DqConst q0 = {}, q8 = {};
            if (a.Bq) {  // INT8 adapter rows g and g + 8: one block per row
                const uint16_t* sc = reinterpret_cast<const uint16_t*>(bs + kBqScale);
                q0 = dq_const(a.Bz ? (uint32_t)bs[kBqZero + g] : 128u, sc[g]);
                q8 = dq_const(a.Bz ? (uint32_t)bs[kBqZero + g + 8] : 128u, sc[g + 8]);
            }
#pragma unroll
            for (int kc = 0; kc < 2; ++kc) {
                uint32_t b0r0, b0r8, b8r0, b8r8;
                if (a.Bq) {  // the two codes of a pair as 1024 + q in each half, then exact q - zp, one rounding
                    const uint32_t o = (uint32_t)(16 * kc + 2 * t);
                    auto pair = [&](int row, uint32_t off, const DqConst& c) {
                        const uint32_t v = *reinterpret_cast<const uint16_t*>(bs + row * 32 + off);
                        return hmul2_rn(hsub2_rn(prmt(v, 0x64646464u, 0x4140u), c.c0), c.s2);
                    };
                    b0r0 = pair(g, o, q0);
                    b0r8 = pair(g + 8, o, q8);
                    b8r0 = pair(g, o + 8, q0);
                    b8r8 = pair(g + 8, o + 8, q8);
                } else {
                    const uint32_t o = (uint32_t)(16 * kc + 2 * t) * 2u;
                    b0r0 = *reinterpret_cast<const uint32_t*>(bs + g * 64 + o);
                    b0r8 = *reinterpret_cast<const uint32_t*>(bs + (g + 8) * 64 + o);
                    b8r0 = *reinterpret_cast<const uint32_t*>(bs + g * 64 + o + 16);
                    b8r8 = *reinterpret_cast<const uint32_t*>(bs + (g + 8) * 64 + o + 16);
                }
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const unsigned char* trow = ts + (nt * 8 + g) * 64 + (16 * kc + 2 * t) * 2;  // T[m, 16kc + 2t]
                    mma_16816(acc[nt][0], b0r0, b0r8, b8r0, b8r8, *reinterpret_cast<const uint32_t*>(trow),
                              *reinterpret_cast<const uint32_t*>(trow + 16));
                }
            }
        }
        float* redq = red + (size_t)((q - 1) & 1) * kConsumerWarps * kGroup * TOK;
        float* r = redq + (size_t)warp * kGroup * TOK;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            float v[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                v[e] = acc[nt][0][e];
#pragma unroll
                for (int qq = 1; qq < kChains; ++qq) v[e] += acc[nt][qq][e];
#pragma unroll
                for (int qq = 0; qq < kChains; ++qq) acc[nt][qq][e] = 0.f;
            }
            r[g * TOK + nt * 8 + 2 * t] = v[0];
            r[g * TOK + nt * 8 + 2 * t + 1] = v[1];
            r[(g + 8) * TOK + nt * 8 + 2 * t] = v[2];
            r[(g + 8) * TOK + nt * 8 + 2 * t + 1] = v[3];
        }
        named_barrier_sync(1, kConsumerWarps * 32);
        // one output per thread: row rr = ctid % 16, token tok = ctid / 16
        const int rr = ctid & (kGroup - 1), tok = ctid >> 4;
        const int token = token0 + tok;
        if (ok && tok < TOK && rr < rows && token < Mt) {
            // warps that held work: 128-byte pieces, or (int8 activations) whole blocks
            const int nw = min(kConsumerWarps, Q8X && BITS == 2 ? CH / kBpb : npieces);
            float sum = 0.f;
            for (int w = 0; w < nw; ++w) sum += redq[((size_t)w * kGroup + rr) * TOK + tok];  // fixed warp order
            if (pj.bias) sum += __half2float(pj.bias[ra + rr]);
            pj.Y[(size_t)token * pj.N + ra + rr] = __float2half_rn(sum);
        }
        __syncwarp();
        if (ok && lane == 0) mbar_arrive(empty(s));
    }
}

template <int BITS, bool HAS_ZP, int NT, bool XS, int OCC, bool Q8X = false>
cudaError_t launch_one(const GemvArgs& a, dim3 grid, size_t smem, bool pdl, cudaStream_t st) {
    static_assert(NT == 1 || NT == 2, "token tiles");
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreadsGemv);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    // weights of multi-chunk stages as 3-D boxes when the row length allows it
    GemvMaps maps;
    memset(&maps, 0, sizeof(maps));
    GemvArgs b = a;
    b.w3d = 0;
    const uint64_t rowbytes = (uint64_t)a.K * BITS / 8;
    if (rowbytes > (uint64_t)a.CH && rowbytes % 256 == 0 && a.CH % 256 == 0) {
        for (int i = 0; i < a.nseg; ++i) {
            const cudaError_t e = encode_rows_3d(&maps.m[i], a.seg[i].Wq, rowbytes, (uint64_t)a.seg[i].N,
                                                 (uint32_t)(a.CH / 256), kGroup);
            if (e != cudaSuccess) return e;
        }
        b.w3d = 1;
    }
    return cudaLaunchKernelEx(&cfg, gemv_kernel<BITS, HAS_ZP, NT, XS, OCC, Q8X>, maps, b);
}

template <int BITS, bool HAS_ZP, int NT>
cudaError_t launch_xs(const GemvArgs& a, dim3 grid, size_t smem, bool xs, int occ, bool pdl, cudaStream_t st) {
    if constexpr (NT == 1) {
        if (xs && occ == 3) return launch_one<BITS, HAS_ZP, 1, true, 3>(a, grid, smem, pdl, st);
    }
    return xs ? launch_one<BITS, HAS_ZP, NT, true, 2>(a, grid, smem, pdl, st)
              : launch_one<BITS, HAS_ZP, NT, false, 2>(a, grid, smem, pdl, st);
}

}  // namespace

size_t gemv_geometry(int N, int K, int bits, int Mt, int sms, int* ctas_out, int* R_out, int* CH_out, int* tok_out,
                     int* threads) {
    const int tok = Mt <= 8 ? 8 : 16;
    const uint32_t xrows = (uint32_t)(Mt < tok ? Mt : tok);  // X rows one CTA stages
    const bool xs = xrows * xs_pitch(K) <= kXStageMax;
    const uint32_t xbytes = xs ? xrows * xs_pitch(K) : 0u;
    // two or three CTAs per SM, but at least one 16-row group per CTA
    const int occ = gemv_ctas_per_sm(N, tok / 8, xbytes, sms > 0 ? sms : 1);
    int ctas = occ * (sms > 0 ? sms : 1);
    if (ctas > (N + kGroup - 1) / kGroup) ctas = (N + kGroup - 1) / kGroup;
    if (ctas < 1) ctas = 1;
    // fewest groups on the busiest SM; among equals, more CTAs (more warps)
    const int G = (N + kGroup - 1) / kGroup, s = sms > 0 ? sms : 1;
    int best = ctas, best_cost = 1 << 30;
    for (int cc = ctas; cc >= 1; --cc) {
        const int cost = ((cc + s - 1) / s) * ((G + cc - 1) / cc);
        if (cost < best_cost) {
            best_cost = cost;
            best = cc;
        }
    }
    ctas = best;
    const int R = kGroup * ((G + ctas - 1) / ctas);  // rows of the largest share
    const int nblk = K / 32;
    const int rowbytes = K * bits / 8;
    // K chunk: a full row when it fits (one contiguous copy per group), else 1 KB
    int CH = rowbytes <= kMaxChunk ? rowbytes : kMaxChunk;
    CH = (CH + 63) / 64 * 64;
    if (CH < 64) CH = 64;
    *ctas_out = ctas;
    *R_out = R;
    *CH_out = CH;
    *tok_out = tok;
    *threads = kThreadsGemv;
    const int nstages = (R + kGroup - 1) / kGroup * ((rowbytes + CH - 1) / CH);
    return gemv_layout(CH, nblk, tok, gemv_pick_ring(CH, nblk, tok, nstages, occ, xbytes), xbytes).total;
}

cudaError_t gemv_prepare() {
    cudaError_t e = tensor_map_prepare();
#define MNB_SET(B, Z, T)                                                                                       \
    if (e == cudaSuccess)                                                                                      \
        e = cudaFuncSetAttribute(gemv_kernel<B, Z, T, false, 2, false>,                                        \
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);                     \
    if (e == cudaSuccess)                                                                                      \
        e = cudaFuncSetAttribute(gemv_kernel<B, Z, T, true, 2, false>,                                         \
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);                     \
    if (e == cudaSuccess && T == 1)                                                                            \
        e = cudaFuncSetAttribute(gemv_kernel<B, Z, 1, true, 3, false>,                                         \
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);                     \
    if (e == cudaSuccess && T == 1)                                                                            \
        e = cudaFuncSetAttribute(gemv_kernel<B, Z, 1, true, 2, true>,                                          \
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    MNB_SET(2, false, 1) MNB_SET(2, false, 2) MNB_SET(2, true, 1) MNB_SET(2, true, 2)
    MNB_SET(4, false, 1) MNB_SET(4, false, 2) MNB_SET(4, true, 1) MNB_SET(4, true, 2)
    MNB_SET(8, false, 1) MNB_SET(8, false, 2) MNB_SET(8, true, 1) MNB_SET(8, true, 2)
#undef MNB_SET
    return e;
}

cudaError_t gemv_launch(const GemvArgs& a_in, const mnb_plan_info& p, int bits, bool pdl, cudaStream_t st) {
    GemvArgs a = a_in;
    const int tok = p.tokens_per_cta;
    const int rowbytes = a.K * bits / 8;
    const int nstages = (a.R + kGroup - 1) / kGroup * ((rowbytes + a.CH - 1) / a.CH);
    const uint32_t xrows = (uint32_t)(a.Mt < tok ? a.Mt : tok);
    const bool xs = xrows * xs_pitch(a.K) <= kXStageMax;
    const uint32_t xbytes = xs ? xrows * xs_pitch(a.K) : 0u;
    const int occ = gemv_ctas_per_sm(a.G * kGroup, tok / 8, xbytes, a.sms > 0 ? a.sms : 1);
    a.ring = gemv_pick_ring(a.CH, a.K / 32, tok, nstages, occ, xbytes);
    a.xrows = xs ? (int)xrows : 0;
    const size_t smem = gemv_layout(a.CH, a.K / 32, tok, a.ring, xbytes).total;
    if (smem > 227 * 1024) return cudaErrorInvalidConfiguration;
    const dim3 grid(p.grid_x, p.grid_y);
    const bool zp = a.seg[0].Z != nullptr;
    const int nt = tok / 8;
    if (bits == 2) {
        if (zp) return nt == 1 ? launch_xs<2, true, 1>(a, grid, smem, xs, occ, pdl, st)
                               : launch_xs<2, true, 2>(a, grid, smem, xs, occ, pdl, st);
        return nt == 1 ? launch_xs<2, false, 1>(a, grid, smem, xs, occ, pdl, st)
                       : launch_xs<2, false, 2>(a, grid, smem, xs, occ, pdl, st);
    }
    if (bits == 4) {
        if (zp) return nt == 1 ? launch_xs<4, true, 1>(a, grid, smem, xs, occ, pdl, st)
                               : launch_xs<4, true, 2>(a, grid, smem, xs, occ, pdl, st);
        return nt == 1 ? launch_xs<4, false, 1>(a, grid, smem, xs, occ, pdl, st)
                       : launch_xs<4, false, 2>(a, grid, smem, xs, occ, pdl, st);
    }
    if (zp) return nt == 1 ? launch_xs<8, true, 1>(a, grid, smem, xs, occ, pdl, st)
                           : launch_xs<8, true, 2>(a, grid, smem, xs, occ, pdl, st);
    return nt == 1 ? launch_xs<8, false, 1>(a, grid, smem, xs, occ, pdl, st)
                   : launch_xs<8, false, 2>(a, grid, smem, xs, occ, pdl, st);
}

// The int8-activation decode path: one 8-token tile per CTA row of the grid,
// X always staged (quantized) in shared memory.
cudaError_t gemv_q8x_launch(const GemvArgs& a_in, const mnb_plan_info& p, int bits, bool pdl, cudaStream_t st) {
    GemvArgs a = a_in;
    const int rowbytes = a.K * bits / 8;
    const int nstages = (a.R + kGroup - 1) / kGroup * ((rowbytes + a.CH - 1) / a.CH);
    a.ring = gemv_ring(nstages);
    a.xrows = a.Mt < 8 ? a.Mt : 8;
    size_t smem = gemv_layout(a.CH, a.K / 32, 8, a.ring, q8x_stage_bytes(8, a.K)).total;
    if (smem > 227 * 1024 && a.ring > 2) {  // large K: the staged codes leave room for two stages
        a.ring = 2;
        smem = gemv_layout(a.CH, a.K / 32, 8, a.ring, q8x_stage_bytes(8, a.K)).total;
    }
    if (smem > 227 * 1024) return cudaErrorNotSupported;
    const dim3 grid(p.grid_x, p.grid_y);
    const bool zp = a.seg[0].Z != nullptr;
    if (bits == 2)
        return zp ? launch_one<2, true, 1, true, 2, true>(a, grid, smem, pdl, st)
                  : launch_one<2, false, 1, true, 2, true>(a, grid, smem, pdl, st);
    if (bits == 4)
        return zp ? launch_one<4, true, 1, true, 2, true>(a, grid, smem, pdl, st)
                  : launch_one<4, false, 1, true, 2, true>(a, grid, smem, pdl, st);
    return zp ? launch_one<8, true, 1, true, 2, true>(a, grid, smem, pdl, st)
              : launch_one<8, false, 1, true, 2, true>(a, grid, smem, pdl, st);
}

}  // namespace mnb
