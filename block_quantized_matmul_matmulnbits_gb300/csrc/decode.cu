// decode.cu -- single-token decode kernel: one launch computes
//
//     Y[n] = sum_k x[k] w[n, k]  (+ sum_r T[r] B[n, r],  T = fp16(x A))  (+ bias[n])
//
// for one token row x, the "fuse_down" decode path of "[WebGPU] Fuse rank-32
// quantized LoRA with MatMulNBits" (onnxruntime PR 33370, commit message adding
// MatMulNBitsLoRA: the base GEMV and the LoRA down projection T first, then the
// base plus T * Bt^T), restated for sm_103a.  Both adapter projections are
// fused into this one kernel, so the base weights are read exactly once and a
// call is one launch.
//
// Design:
//  * Rows are split evenly over the CTAs (one per SM): CTA c owns rows
//    [c N / C, (c + 1) N / C), so every SM moves the same number of weight
//    bytes.  Its rows are contiguous in memory: one producer lane streams them
//    into shared memory in stages of up to SR rows (codes and adapter rows
//    B[n, :] as 1-D bulk copies, scales and zero points as 2-D TMA boxes whose
//    rows are 16 bytes wider than the data, so that reading one value from
//    each of eight rows is free of bank conflicts), and when the CTA's whole
//    share fits it is copied before anything else happens.  Weights are
//    constant, so the copies start before the work queued ahead of this
//    kernel has finished (programmatic dependent launch); only x waits for it.
//  * The multiply runs on mma.sync m16n8k16 (FP16 in, FP32 accumulate) with 16
//    weight rows as M.  A code is fed to the tensor core as the FP16 value
//    q * 2^-24 (the code's bits placed in the mantissa of a subnormal half:
//    exact), so unpacking is a mask (INT4) or a byte permute (INT8) and no
//    dequant arithmetic runs per weight.  The eight MMA columns, which one
//    token row would leave idle, each collect one (block, class) of codes:
//    thread t of a quad owns block t of a group of four blocks, its A pairs
//    go to columns 2t and 2t + 1, and only the threads supplying those
//    columns carry x in their B fragment (x is staged per thread role, so a B
//    fragment is one 16-byte load, zeros included).  After a group of four
//    blocks each thread holds, for its two rows, the block sums sum_k x q of
//    its block, and applies the block's scale and zero point once, in FP32:
//        y += s * (sum_k x q - zp * sum_k x).
//  * The adapter runs on a warp of its own, beside the weight stream and the
//    base dot products.  Every CTA takes an equal slice of K, copies its slice
//    of A into shared memory with the weights (one bulk copy), forms the
//    partial sums of T on the tensor cores (movmatrix turns A's rows into the
//    MMA's K-major operand) and adds them to per-rank words in global memory
//    as fixed-point integers with a count; once the counts show every CTA of
//    the launch (the launch is cooperative, so all of its CTAs are resident
//    together) each CTA reads T (integer sums: the same bits whatever the
//    order of the additions), rounds T once to FP16 and forms
//    sum_r T[r] B[n, r] for its rows (two MMAs per 16 rows) from a copy of
//    its B rows.  An INT8 adapter (block-32 Aq [32, K], Bq [N, 32]) is
//    dequantized by the same warp (exact q - zp, one rounding by the FP16
//    scale): its A slice into a k-major FP16 tile before x arrives, its B rows
//    while the other CTAs' partials of T arrive.  The consumers keep each row's base sum in FP32 and add the
//    adapter term before the one rounding of the output, at the end.  No
//    thread-block clusters: cluster placement put two CTAs of one launch on
//    the same SM while others stayed idle.
//  * Eight consumer warps split every 16-row tile's rounds (warp w takes
//    rounds w, w + 8, ...), so a row's summation order depends on K alone;
//    partial sums are added in warp order (no atomics): results are
//    deterministic and independent of how rows were split into CTAs.
//  * Every mbarrier wait is bounded and reports through the status word.
#include <cuda.h>

#include <atomic>
#include <cstring>
#include <type_traits>

#include "common.cuh"
#include "decode_common.cuh"
#include "mnb_internal.h"

namespace mnb {

namespace {

using namespace dec;

constexpr int kCW = 8;                     // consumer warps
constexpr int kRk = 32;                    // adapter rank
constexpr int kMaxLoraRows = 256;          // adapter: most rows per CTA (B rows and sums stay in shared memory)
constexpr int kExSlots = 32;               // adapter exchange areas (calls in flight on different streams)
constexpr int kExMaxC = 240;               // most CTAs of a launch (the count field of an exchange word)
constexpr int kBlkPerRound = 4;            // quantization blocks a warp covers per round
constexpr int kMaxSR = 128;                // most rows per stage

// Threads of a CTA: the consumer warps, the producer warp, and with an adapter the adapter warp.
__host__ __device__ constexpr int dec_threads(bool lora) { return (kCW + (lora ? 2 : 1)) * 32; }

// The adapter's exchange of partial T between the CTAs of one launch.  A launch
// reads `gen` and works in generation gen & 1.  Each rank has kExSub 64-bit
// words (each on its own 128-byte line, so few CTAs meet on one): CTA c adds
// to word c % kExSub, atomically, its partial as a fixed-point number (units
// of 2^-32) plus one count in the top byte.  Integer sums do not depend on the
// order of the additions, so T is the same bits on every run; a CTA knows a
// rank is complete when the counts of its words add up to the CTAs of the
// launch.  CTA 0 then clears the other generation (used by the launch before,
// to be used by the next) and advances `gen`.  Two words a rank: one makes the
// adds to a word queue up (4.85 us per call at 4096 x 4096), more make every
// poll read more (4.76 with four, 5.58 with eight, 4.72 to 4.74 with two).
constexpr int kExSub = 2;
struct LoraEx {
    unsigned int gen;
    unsigned int pad_[31];
    unsigned long long acc[2][kRk][kExSub][16];  // [generation][rank][word], word 0 of each line
};
constexpr unsigned long long kExCount = 1ull << 56;  // one CTA's count in an exchange word
// A partial (|v| < 2^22) as a signed multiple of 2^-32 plus one count.
__device__ __forceinline__ unsigned long long ex_word(float v) {
    long long q = __float2ll_rn(v * 4294967296.f);
    const long long lim = 1ll << 54;
    q = q > lim ? lim : (q < -lim ? -lim : q);
    return (unsigned long long)q + kExCount;
}
__device__ __forceinline__ unsigned int ex_count(unsigned long long w) {
    return (unsigned int)((w + (kExCount >> 1)) >> 56);
}
// The partials a word holds, in units of 2^-32.
__device__ __forceinline__ long long ex_value(unsigned long long w) {
    return (long long)(w - (unsigned long long)ex_count(w) * kExCount);
}
__device__ LoraEx g_lora_ex[kExSlots];

__host__ __device__ inline int round16(int x) { return (x + 15) & ~15; }
// Rows of the adapter's per-CTA buffers: the most rows a CTA owns, in whole 16-row tiles.
__host__ __device__ inline int lora_rows(int NR, int C) { return round16((NR + C - 1) / C); }

// A stage's rows [0, h) and [h, rs), h = ceil(rs / 2), land in two regions of
// the slot; the MMA rows of a 16-row tile alternate between them (even MMA rows
// from the first, odd from the second).  The two rows a quarter-warp reads with
// one 16-byte load per thread (MMA rows 2p and 2p + 1) then never share banks,
// which rows of one region would when packed rows are a multiple of 128 bytes:
// the second region starts 64 bytes past a 128-byte boundary for INT4 (thread t
// reads bytes [16 t, 16 t + 16) of a 64-byte round) and 16 bytes past it for
// INT8 (bytes [32 t, 32 t + 16) or [32 t + 16, 32 t + 32) of a 128-byte round).
__host__ __device__ inline int dec_half(int rs) { return (rs + 1) / 2; }

// Shared memory plan, identical on host and device.  A stage slot holds SR
// rows: codes (two regions of SR / 2 rows, [SR/2][rowbytes] each), scales
// [SR][spitch] and zero points [SR][zpitch]
// (each + 32 bytes for the aligned superset of a bulk copy).  With an adapter
// (lrows > 0): the CTA's adapter rows B[n, :] [lrows][32] FP16, the adapter
// term and the base sum of each row [lrows] FP32, T [32] FP16, and the first
// 64 K rows of the CTA's slice of A, astg [64][32] FP16 (k-major).
struct DecLayout {
    uint32_t r1, sc, zp, slot;  // offsets inside a slot (second code region, scales, zero points), slot bytes
    uint32_t xs, sxs, red, bown, lorb, ybuf, t16, braw, astg, bars, total;
};

// lq8: an INT8 adapter, whose B rows' codes [lrows][32] (then each row's scale and zero
// point as one word [lrows]) land in braw before they are dequantized into bown, and
// whose A slice is dequantized into astg (an FP16 A slice is copied there as is).
__host__ __device__ inline DecLayout dec_layout(int SR, int ring, int bits, int rowbytes, int nblk, int nblkR,
                                                int lrows, bool lq8 = false) {
    const DecPitch P = dec_pitch(nblk);
    DecLayout L;
    const uint32_t half = (uint32_t)(SR / 2) * (uint32_t)rowbytes;
    L.r1 = al128(half) + (bits == 4 ? 64u : 16u);
    L.sc = al128(L.r1 + half);
    L.zp = al128(L.sc + (uint32_t)SR * P.spitch + 32u);
    L.slot = al128(L.zp + (uint32_t)SR * P.zpitch + 32u);
    uint32_t off = (uint32_t)ring * L.slot;
    // x in the MMA's operand order: 128 bytes a block (two thread roles), then 64 zero
    // bytes starting 32 bytes into a line (their banks differ from both roles' reads)
    L.xs = off;
    off = al128(off + (uint32_t)nblkR * 128u + 96u);
    L.sxs = off;  // per block: sum of x, times 2^-24
    off = al128(off + (uint32_t)nblkR * 4u);
    L.red = off;  // two buffers [SR / 16][kCW][16] FP32
    off += 2u * (uint32_t)(SR / 16) * kCW * 16u * 4u;
    L.bown = al128(off);
    off = L.bown + (uint32_t)lrows * 64u;
    L.lorb = off;
    off += (uint32_t)lrows * 4u;
    L.ybuf = off;
    off += (uint32_t)lrows * 4u;
    L.t16 = off;
    off += lrows > 0 ? kRk * 2u : 0u;
    L.braw = al128(off);
    off = L.braw + (lq8 ? (uint32_t)lrows * 36u : 0u);
    L.astg = al128(off);  // the adapter's first 64 K rows of A, k-major FP16
    off = L.astg + (lrows > 0 ? 64u * kRk * 2u : 0u);
    L.bars = al128(off);
    // full and empty per slot, then B rows, adapter done and the A slice
    L.total = L.bars + (2u * (uint32_t)ring + 3u) * 8u;
    return L;
}

// Staged x, per block (128 bytes): role 0 (threads carrying class 0) then role 1,
// 64 bytes each, every B fragment (b0, b1) one 8-byte pair with the other role's
// half zero.  INT4, word i (codes 8i .. 8i+7 of the block): role 0 at 16 i holds
// {(x0, x4), 0, (x2, x6), 0}, role 1 at 64 + 16 i holds {0, (x1, x5), 0, (x3, x7)}.
// INT8, word i (codes 4i .. 4i+3): role 0 at 8 i holds {(x0, x1), 0}, role 1 at
// 64 + 8 i holds {0, (x2, x3)}.

__device__ __forceinline__ void movmatrix_t(uint32_t& x) {
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %0;" : "+r"(x));
}

// Global-memory accesses of the adapter exchange, at GPU scope.
__device__ __forceinline__ uint32_t ld_relaxed_u32(const unsigned int* p) {
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

// The adapter's FP16 A pair (A[k][c], A[k][c + 1]) from the INT8 down weight Aq [32, K]
// (rank rows, block-32 along K): each value fp16((q - zp) * scale), rounded once.
__device__ __forceinline__ uint32_t q8_apair(const DecodeArgs& a, int k, int c) {
    const int nblk = a.K >> 5;
    uint32_t w = 0;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const int r = c + e, b = r * nblk + (k >> 5);
        const int q = (int)a.Aq[(size_t)r * a.K + k], zp = a.Az ? (int)a.Az[b] : 128;
        const __half v = __hmul(__int2half_rn(q - zp), __ushort_as_half(reinterpret_cast<const uint16_t*>(a.As)[b]));
        w |= (uint32_t)__half_as_ushort(v) << (16 * e);
    }
    return w;
}

template <int BITS, bool HAS_ZP, bool LORA, bool Q8L>
__global__ void __launch_bounds__(dec_threads(LORA), 2)
    decode_kernel(const __grid_constant__ DecMaps maps, const __grid_constant__ DecodeArgs a) {
    using U = Unpack<BITS>;
    constexpr int kWB = U::kWordsPerBlock;
    constexpr uint32_t kDefaultZp = 1u << (BITS - 1);
    extern __shared__ __align__(1024) unsigned char sm[];

    const int K = a.K, NR = a.NR;
    const int nblk = K >> 5;
    const int nround = (nblk + kBlkPerRound - 1) / kBlkPerRound;
    const int nblkR = nround * kBlkPerRound;
    const int rowbytes = K * BITS / 8;
    const int SR = a.SR, ring = a.ring;
    const int C = gridDim.x;
    const DecLayout L = dec_layout(SR, ring, BITS, rowbytes, nblk, nblkR, LORA ? lora_rows(NR, C) : 0, Q8L);
    const DecPitch P = dec_pitch(nblk);
    const uint32_t sb = smem_u32(sm);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r0 = (int)((long long)blockIdx.x * NR / C), r1 = (int)((long long)(blockIdx.x + 1) * NR / C);
    unsigned int* status = a.status;

    auto full = [&](int s) { return sb + L.bars + 8u * (uint32_t)s; };
    auto empty = [&](int s) { return sb + L.bars + 8u * (uint32_t)(ring + s); };
    const uint32_t bbar = sb + L.bars + 16u * (uint32_t)ring;  // adapter: the CTA's B rows landed
    const uint32_t lready = bbar + 8u;                          // adapter: T B^T of the CTA's rows is in place
    const uint32_t abar = bbar + 16u;                           // adapter (FP16 A): its slice of A landed

    if (threadIdx.x == 0) {
        for (int s = 0; s < ring; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), kCW);
        }
        if (LORA) {
            mbar_init(bbar, 1);
            mbar_init(lready, 1);
            mbar_init(abar, 1);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    pdl_launch_dependents();

    if (warp == kCW) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            bool ok = true;
            int issued = 0;
            StageIt it = {r0, 0, 0, 0};
            if (r0 < r1) it.settle(a, r1, SR);
            for (int st = 0; ok && it.pos < r1; ++st, ++issued, it.next(a, r1, SR)) {
                const int s = st % ring;
                const uint32_t par = (uint32_t)(st / ring) & 1u;
                if (st >= ring && !(ok = mbar_wait(empty(s), par ^ 1u, status))) break;
                const DecSeg& pj = a.seg[it.seg];
                const int ra = it.ra, rs = it.rs;
                unsigned char* slot = sm + (size_t)s * L.slot;
                const uint32_t sslot = sb + (uint32_t)s * L.slot;
                // dense copies: the 16-byte aligned superset of the stage's scales / zero
                // points; bytes past the last 16-byte boundary of an array are stored here
                const uint64_t total_s = (uint64_t)pj.N * nblk * 2, total_z = (uint64_t)pj.N * nblk;
                const uint64_t s0 = (uint64_t)ra * nblk * 2, s1 = (uint64_t)(ra + rs) * nblk * 2;
                const uint64_t s_lo = s0 & ~15ull, s_hi = min((s1 + 15) & ~15ull, total_s & ~15ull);
                const uint64_t z0 = (uint64_t)ra * nblk, z1 = (uint64_t)(ra + rs) * nblk;
                const uint64_t z_lo = z0 & ~15ull, z_hi = min((z1 + 15) & ~15ull, total_z & ~15ull);
                uint32_t bytes = (uint32_t)rs * (uint32_t)rowbytes;
                if (P.tma_s) {
                    bytes += (uint32_t)SR * P.spitch;  // a whole box always lands (rows past N read as zero)
                } else {
                    for (uint64_t i = max(s_hi, s_lo); i < s1; ++i)
                        slot[L.sc + (uint32_t)(i - s_lo)] = reinterpret_cast<const uint8_t*>(pj.S)[i];
                    if (s_hi > s_lo) bytes += (uint32_t)(s_hi - s_lo);
                }
                if (HAS_ZP) {
                    if (P.tma_z) {
                        bytes += (uint32_t)SR * P.zpitch;
                    } else {
                        for (uint64_t i = max(z_hi, z_lo); i < z1; ++i) slot[L.zp + (uint32_t)(i - z_lo)] = pj.Z[i];
                        if (z_hi > z_lo) bytes += (uint32_t)(z_hi - z_lo);
                    }
                }
                mbar_arrive_tx(full(s), bytes);
                // codes: rows [0, h) and [h, rs) into the two regions
                const uint8_t* src = pj.Wq + (size_t)ra * rowbytes;
                const uint32_t c0 = (uint32_t)dec_half(rs) * (uint32_t)rowbytes, cb = (uint32_t)rs * (uint32_t)rowbytes;
                for (uint32_t off = 0; off < c0; off += 32768u)
                    bulk_load(sslot + off, src + off, min(32768u, c0 - off), full(s));
                for (uint32_t off = c0; off < cb; off += 32768u)
                    bulk_load(sslot + L.r1 + (off - c0), src + off, min(32768u, cb - off), full(s));
                if (P.tma_s)
                    tma_load_2d(sslot + L.sc, &maps.s[it.seg], 0, ra, full(s));
                else if (s_hi > s_lo)
                    bulk_load(sslot + L.sc, reinterpret_cast<const uint8_t*>(pj.S) + s_lo, (uint32_t)(s_hi - s_lo),
                              full(s));
                if (HAS_ZP) {
                    if (P.tma_z)
                        tma_load_2d(sslot + L.zp, &maps.z[it.seg], 0, ra, full(s));
                    else if (z_hi > z_lo)
                        bulk_load(sslot + L.zp, pj.Z + z_lo, (uint32_t)(z_hi - z_lo), full(s));
                }
            }
            // no copy may still be in flight when the CTA exits (a consumer may have given up)
            for (int st = issued > ring ? issued - ring : 0; st < issued; ++st)
                mbar_wait(full(st % ring), (uint32_t)(st / ring) & 1u, status, false);
        }
        return;
    }

    if constexpr (LORA) {
        if (warp == kCW + 1) {
            // -------------------------------------------------------- adapter
            // T = fp16(x A) from every CTA's partial over an equal slice of K, then
            // T B^T for this CTA's rows.  Its B rows and its slice of A are weights:
            // copied before waiting for x.
            const int g = lane >> 2, t = lane & 3;
            const int nrows = r1 - r0;
            if (lane == 0 && nrows > 0) {
                if constexpr (Q8L) {  // the rows' INT8 codes, dequantized into B rows once T is under way
                    mbar_arrive_tx(bbar, (uint32_t)nrows * 32u);
                    bulk_load(sb + L.braw, a.Bq + (size_t)r0 * kRk, (uint32_t)nrows * 32u, bbar);
                } else {
                    mbar_arrive_tx(bbar, (uint32_t)nrows * 64u);
                    bulk_load(sb + L.bown, a.B + (size_t)r0 * kRk, (uint32_t)nrows * 64u, bbar);
                }
            }
            if constexpr (Q8L) {  // each B row's scale and zero point, read while nothing waits on them
                uint32_t* bsz = reinterpret_cast<uint32_t*>(sm + L.braw + (uint32_t)lora_rows(NR, C) * 32u);
                for (int rr = lane; rr < nrows; rr += 32) {
                    const int n = r0 + rr;
                    bsz[rr] = (uint32_t)reinterpret_cast<const uint16_t*>(a.Bs)[n] |
                              ((a.Bz ? (uint32_t)a.Bz[n] : 128u) << 16);
                }
            }
            // K steps (16 wide) [c S / C, (c + 1) S / C) of CTA c.  A step is 2 K
            // sub-blocks x 4 rank sub-blocks of 8 x 8, each loaded in its natural
            // fragment (thread (g, t) holds ranks 2t, 2t+1 of K row g) and transposed
            // by movmatrix into the MMA's B fragment.
            constexpr int kMaxSteps = 4;
            const int S = K / 16;
            const int step0 = (int)((long long)blockIdx.x * S / C);
            const int nsteps = (int)((long long)(blockIdx.x + 1) * S / C) - step0;
            uint32_t areg[kMaxSteps][8];
            const int ns = nsteps < kMaxSteps ? nsteps : kMaxSteps;  // steps staged in astg
            bool a_ok = true;
            if constexpr (!Q8L) {
                // FP16 A: the slice's first ns steps (16 K rows of 32 ranks each, contiguous
                // in A) in one bulk copy.  Per-lane 4-byte loads here were measured to slow
                // the consumer warps of the previous call on the SM, whose rounds run
                // while this CTA starts.
                if (lane == 0 && ns > 0) {
                    mbar_arrive_tx(abar, (uint32_t)ns * 16u * kRk * 2u);
                    bulk_load(sb + L.astg, a.A + (size_t)step0 * 16 * kRk, (uint32_t)ns * 16u * kRk * 2u, abar);
                }
                a_ok = ns == 0 || mbar_wait(abar, 0u, status);
            }
            if constexpr (Q8L) {
                // lane r: rank r's codes of the first kMaxSteps steps (16-byte loads, all in
                // flight together), dequantized into the k-major FP16 tile astg
                __half* ast = reinterpret_cast<__half*>(sm + L.astg);
                const int k_lo = step0 * 16;
                uint4 qv[kMaxSteps];
                uint32_t qs[kMaxSteps], qz[kMaxSteps];
#pragma unroll
                for (int i = 0; i < kMaxSteps; ++i) {
                    const int k = k_lo + 16 * (i < ns ? i : 0), b = lane * (K >> 5) + (k >> 5);
                    qv[i] = __ldg(reinterpret_cast<const uint4*>(a.Aq + (size_t)lane * K + k));
                    qs[i] = reinterpret_cast<const uint16_t*>(a.As)[b];
                    qz[i] = a.Az ? (uint32_t)a.Az[b] : 128u;
                }
#pragma unroll
                for (int i = 0; i < kMaxSteps; ++i) {
                    if (i >= ns) break;
                    const DqConst dc = dq_const(qz[i], (uint16_t)qs[i]);
                    const uint32_t wv[4] = {qv[i].x, qv[i].y, qv[i].z, qv[i].w};
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        uint32_t d[2];
                        dq_int8_natural(wv[w], dc, d);  // codes 4w .. 4w+3 of the step
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            ast[(i * 16 + 4 * w + e) * kRk + lane] =
                                __ushort_as_half((uint16_t)(d[e >> 1] >> (16 * (e & 1))));
                    }
                }
                __syncwarp();
            }
#pragma unroll
            for (int i = 0; i < kMaxSteps; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j)  // K row (j / 4) 8 + g of step i, ranks (j % 4) 8 + 2t, + 1
                    areg[i][j] = i < ns && a_ok ? *reinterpret_cast<const uint32_t*>(
                                                      reinterpret_cast<const __half*>(sm + L.astg) +
                                                      (i * 16 + (j >> 2) * 8 + g) * kRk + (j & 3) * 8 + 2 * t)
                                                : 0u;
            // The area's generation: its last writer is the launch before this one on the
            // area (kExSlots launches back), finished before this one starts.
            LoraEx* ex = static_cast<LoraEx*>(a.ex);
            const uint32_t gen = ld_relaxed_u32(&ex->gen);
            const int gs = (int)(gen & 1u);
            if (a.x_wait) pdl_wait();
            float tacc[4][4];
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
                for (int e = 0; e < 4; ++e) tacc[j][e] = 0.f;
            const uint32_t* xw = reinterpret_cast<const uint32_t*>(a.X);
            for (int i0 = 0; i0 < nsteps; i0 += kMaxSteps) {
                // x of the chunk's steps for token row 0 (rows 1..15 of the MMA are empty)
                uint32_t xr[kMaxSteps][2];
#pragma unroll
                for (int i = 0; i < kMaxSteps; ++i) {
                    const int k0 = (step0 + i0 + i) * 16;
                    const bool on = g == 0 && i0 + i < nsteps;
                    xr[i][0] = on ? xw[(k0 >> 1) + t] : 0u;
                    xr[i][1] = on ? xw[(k0 >> 1) + 4 + t] : 0u;
                }
#pragma unroll
                for (int i = 0; i < kMaxSteps; ++i) {
                    if (i0 + i >= nsteps) break;
                    uint32_t bfr[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        if (i0 == 0) {
                            bfr[j] = areg[i][j];
                        } else {
                            const int kk = (step0 + i0 + i) * 16 + (j >> 2) * 8 + g;
                            if constexpr (Q8L)
                                bfr[j] = q8_apair(a, kk, (j & 3) * 8 + 2 * t);
                            else
                                bfr[j] = __ldg(reinterpret_cast<const uint32_t*>(a.A + (size_t)kk * kRk + (j & 3) * 8 + 2 * t));
                        }
                        movmatrix_t(bfr[j]);
                    }
#pragma unroll
                    for (int j = 0; j < 4; ++j) mma_16816(tacc[j], xr[i][0], 0u, xr[i][1], 0u, bfr[j], bfr[4 + j]);
                }
            }
            // token row 0: thread (0, t) holds ranks 8j + 2t, 8j + 2t + 1: add them to the words
            const int sub = (int)(blockIdx.x % kExSub);
            if (g == 0) {
#pragma unroll
                for (int j = 0; j < 4; ++j)
#pragma unroll
                    for (int e = 0; e < 2; ++e)
                        atomicAdd(&ex->acc[gs][8 * j + 2 * t + e][sub][0], ex_word(tacc[j][e]));
            }
            if constexpr (Q8L) {
                // the B rows from their INT8 codes while the other CTAs' partials arrive:
                // row n's 32 values fp16((q - zp) * scale) (one block a row), into bown
                if (nrows > 0 && mbar_wait(bbar, 0u, status)) {
                    const uint32_t* bsz = reinterpret_cast<const uint32_t*>(sm + L.braw + (uint32_t)lora_rows(NR, C) * 32u);
                    for (int rr = lane; rr < nrows; rr += 32) {
                        const uint4* src = reinterpret_cast<const uint4*>(sm + L.braw + (uint32_t)rr * 32u);
                        const uint4 p0 = src[0], p1 = src[1];
                        const DqConst dc = dq_const(bsz[rr] >> 16, (uint16_t)(bsz[rr] & 0xFFFFu));
                        const uint32_t wv[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
                        uint32_t o[16];
#pragma unroll
                        for (int w = 0; w < 8; ++w) dq_int8_natural(wv[w], dc, &o[2 * w]);
                        uint4* dst = reinterpret_cast<uint4*>(sm + L.bown + (uint32_t)rr * 64u);
#pragma unroll
                        for (int c = 0; c < 4; ++c) dst[c] = make_uint4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]);
                    }
                }
                __syncwarp();
            }
            // T[lane] once every CTA has added its partial (bounded wait: the launch is
            // cooperative, so all of its CTAs are resident)
            const long long t0 = clock64();
            long long tq = 0;
            auto poll = [&](int r) {  // the partials of rank r, once all are in (false: gave up)
                for (;;) {
                    unsigned long long w[kExSub];
#pragma unroll
                    for (int u = 0; u < kExSub; ++u) w[u] = ld_relaxed_u64(&ex->acc[gs][r][u][0]);
                    unsigned int cnt = 0;
                    long long q = 0;
#pragma unroll
                    for (int u = 0; u < kExSub; ++u) {
                        cnt += ex_count(w[u]);
                        q += ex_value(w[u]);
                    }
                    if (cnt >= (unsigned int)C) {
                        tq = q;
                        return true;
                    }
                    if (clock64() - t0 > kWaitCycles) return false;
                    __nanosleep(200);
                }
            };
            bool ok = poll(lane);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok && lane == 0) atomicOr(status, kStatusTimeout);
            const __half th = __double2half((double)tq * 0x1p-32);  // T, rounded once
            reinterpret_cast<__half*>(sm + L.t16)[lane] = th;
            if (blockIdx.x == 0) a.T[lane] = th;
            __syncwarp();
            // sum_r B[n, r] T[r] for each 16-row tile: A = B rows (16 x 16 per MMA), B = T in column 0
            if (nrows > 0 && !mbar_wait(bbar, 0u, status)) ok = false;
            float* lorb = reinterpret_cast<float*>(sm + L.lorb);
            const __half* th16 = reinterpret_cast<const __half*>(sm + L.t16);
            for (int tl = 0; ok && tl * 16 < nrows; ++tl) {
                const unsigned char* bs = sm + L.bown + (uint32_t)(tl * 16) * 64u;
                float dl[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int kc = 0; kc < 2; ++kc) {
                    const uint32_t o = (uint32_t)(16 * kc + 2 * t) * 2u;
                    const uint32_t b0r0 = *reinterpret_cast<const uint32_t*>(bs + g * 64 + o);
                    const uint32_t b0r8 = *reinterpret_cast<const uint32_t*>(bs + (g + 8) * 64 + o);
                    const uint32_t b8r0 = *reinterpret_cast<const uint32_t*>(bs + g * 64 + o + 16);
                    const uint32_t b8r8 = *reinterpret_cast<const uint32_t*>(bs + (g + 8) * 64 + o + 16);
                    const uint32_t t0r = g == 0 ? *reinterpret_cast<const uint32_t*>(th16 + 16 * kc + 2 * t) : 0u;
                    const uint32_t t1r = g == 0 ? *reinterpret_cast<const uint32_t*>(th16 + 16 * kc + 2 * t + 8) : 0u;
                    mma_16816(dl, b0r0, b0r8, b8r0, b8r8, t0r, t1r);
                }
                if (t == 0) {  // column 0: rows g, g + 8
                    lorb[tl * 16 + g] = dl[0];
                    lorb[tl * 16 + g + 8] = dl[2];
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(lready);  // releases this warp's shared-memory writes
            if (blockIdx.x == 0) {
                // the other generation (the launch before this one on the area) for the next
#pragma unroll
                for (int u = 0; u < kExSub; ++u) ex->acc[gs ^ 1][lane][u][0] = 0ull;
                __syncwarp();
                if (lane == 0 && ok) {
                    __threadfence();
                    *reinterpret_cast<volatile unsigned int*>(&ex->gen) = gen + 1u;
                }
            }
            return;
        }
    }

    // ---------------------------------------------------------------- consumers
    const int g = lane >> 2, t = lane & 3;
    const int ctid = threadIdx.x;  // 0 .. 255
    constexpr uint32_t kNamed = 1;  // named barrier of the consumer warps

    // The first stage's weights need no wait for earlier work: take them first.  So do the
    // biases of the rows this thread writes first (the first stage's, or with an adapter the
    // first row of the final pass).
    bool ok = true;
    StageIt it = {r0, 0, 0, 0};
    float bias0 = 0.f;
    if (r0 < r1) {
        it.settle(a, r1, SR);
        const DecSeg& pj = a.seg[it.seg];
        if (pj.bias) {
            if (LORA) {
                if (ctid < r1 - r0) bias0 = __half2float(pj.bias[r0 + ctid]);
            } else if (warp < (it.rs + 15) / 16 && lane < 16) {
                const int m = lane & 7, rr = warp * 8 + (m >> 1) + (lane >> 3) * 4, hh = dec_half(it.rs);
                const int row = (m & 1) ? hh + rr : rr;
                if ((m & 1) ? row < it.rs : rr < hh) bias0 = __half2float(pj.bias[it.ra + row]);
            }
        }
        ok = mbar_wait(full(0), 0u, status);
    }

    // ---- x: wait for the work that produces it, then stage it in the MMA's operand order
    if (a.x_wait) pdl_wait();
    {
        const uint4* xg = reinterpret_cast<const uint4*>(a.X);
        float* sxs = reinterpret_cast<float*>(sm + L.sxs);
        constexpr int kXU = 4;  // 8-code groups in flight per thread
        for (int i0 = 0; i0 < nblkR * 4; i0 += kXU * kCW * 32) {  // 4 groups a block
            uint4 v[kXU];
#pragma unroll
            for (int u = 0; u < kXU; ++u) {
                const int i = i0 + u * kCW * 32 + ctid;
                v[u] = (i >> 2) < nblk ? __ldg(xg + i) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int u = 0; u < kXU; ++u) {
                if (i0 + u * kCW * 32 >= nblkR * 4) break;  // the same for every thread
                const int i = i0 + u * kCW * 32 + ctid;  // every lane runs every step: the shuffles below
                const int b = i >> 2, q = i & 3;
                const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&v[u].x));
                const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&v[u].y));
                const float2 f2 = __half22float2(*reinterpret_cast<const __half2*>(&v[u].z));
                const float2 f3 = __half22float2(*reinterpret_cast<const __half2*>(&v[u].w));
                float part = ((f0.x + f0.y) + (f1.x + f1.y)) + ((f2.x + f2.y) + (f3.x + f3.y));
                part += __shfl_xor_sync(0xffffffffu, part, 1);
                part += __shfl_xor_sync(0xffffffffu, part, 2);
                if (b >= nblkR) continue;
                if (q == 0) sxs[b] = part * kUnit;
                unsigned char* xb = sm + L.xs + (uint32_t)b * 128u;
                if constexpr (BITS == 4) {  // group q = word q: (x0,x4) (x2,x6) | (x1,x5) (x3,x7)
                    *reinterpret_cast<uint4*>(xb + q * 16) =
                        make_uint4(prmt(v[u].x, v[u].z, 0x5410u), 0u, prmt(v[u].y, v[u].w, 0x5410u), 0u);
                    *reinterpret_cast<uint4*>(xb + 64 + q * 16) =
                        make_uint4(0u, prmt(v[u].x, v[u].z, 0x7632u), 0u, prmt(v[u].y, v[u].w, 0x7632u));
                } else {  // group q = words 2q, 2q+1: (x0,x1) (x4,x5) | (x2,x3) (x6,x7)
                    *reinterpret_cast<uint4*>(xb + q * 16) = make_uint4(v[u].x, 0u, v[u].z, 0u);
                    *reinterpret_cast<uint4*>(xb + 64 + q * 16) = make_uint4(0u, v[u].y, 0u, v[u].w);
                }
            }
        }
        if (ctid < 16) reinterpret_cast<uint32_t*>(sm + L.xs + (uint32_t)nblkR * 128u + 32u)[ctid] = 0u;  // zero region
    }
    named_barrier_sync(kNamed, kCW * 32);

    // ---- the stages
    float* red = reinterpret_cast<float*>(sm + L.red);
    // This thread's x role: class 0 of block t when g == 2t, class 1 when g == 2t + 1,
    // else the zero region.
    const bool act0 = g == 2 * t, act1 = g == 2 * t + 1;
    const uint32_t xs_base = act0 ? L.xs + (uint32_t)t * 128u
                           : act1 ? L.xs + (uint32_t)t * 128u + 64u
                                  : L.xs + (uint32_t)nblkR * 128u + 32u;
    const uint32_t xs_step = act0 || act1 ? (uint32_t)(kCW * kBlkPerRound * 128) : 0u;  // per round of this warp
    const int tiles_max = SR / 16;

    for (int st = 0; it.pos < r1; ++st, it.next(a, r1, SR)) {
        const int s = st % ring;
        const uint32_t par = (uint32_t)(st / ring) & 1u;
        const DecSeg& pj = a.seg[it.seg];
        const int ra = it.ra, rs = it.rs;
        const int ntile = (rs + 15) / 16;
        const int hh = dec_half(rs);
        if (ok) ok = mbar_wait(full(s), par, status);
        const uint32_t soff = (uint32_t)s * L.slot;
        // where row 0's scales / zero points start in the slot (dense copies: the aligned superset)
        const uint32_t s_base = soff + L.sc + (P.tma_s ? 0u : (((uint32_t)ra * (uint32_t)nblk * 2u) & 15u));
        const uint32_t z_base = soff + L.zp + (P.tma_z ? 0u : (((uint32_t)ra * (uint32_t)nblk) & 15u));
        float* redb = red + (st & 1) * tiles_max * kCW * 16;
        // This warp's rounds of NTL tiles at once (the x fragments serve both; their MMA
        // chains are independent).  Per round: the block sums of the thread's block for
        // rows g and g + 8 of each tile, then scale and zero point in FP32.
        auto tiles = [&](auto ntl_c, int tl0) {
            constexpr int NTL = decltype(ntl_c)::value;
            float v[NTL][2];
            // 32-bit shared addresses of this thread's words, scales and zero points in its
            // first round, for rows g (A) and g + 8 (B) of each tile; all step by 32 blocks
            uint32_t wA[NTL], wB[NTL], sA_[NTL], sB_[NTL], zA_[NTL], zB_[NTL];
            const int blk0 = warp * kBlkPerRound + t;  // this thread's block in its first round
#pragma unroll
            for (int i = 0; i < NTL; ++i) {
                v[i][0] = v[i][1] = 0.f;  // rows g and g + 8, units of 2^-24
                // MMA rows g, g + 8: row (tl 8 + g / 2) resp. (tl 8 + g / 2 + 4) of region g & 1
                const uint32_t rr = (uint32_t)((tl0 + i) * 8 + (g >> 1));
                const uint32_t row = (g & 1 ? (uint32_t)hh : 0u) + rr;  // the stage row of MMA row g
                wA[i] = sb + soff + (g & 1 ? L.r1 : 0u) + rr * (uint32_t)rowbytes + (uint32_t)blk0 * (uint32_t)(kWB * 4);
                wB[i] = wA[i] + 4u * (uint32_t)rowbytes;
                sA_[i] = sb + s_base + row * P.spitch + (uint32_t)blk0 * 2u;
                sB_[i] = sA_[i] + 4u * P.spitch;
                zA_[i] = sb + z_base + row * P.zpitch + (uint32_t)blk0;
                zB_[i] = zA_[i] + 4u * P.zpitch;
            }
            uint32_t xo = sb + xs_base + (uint32_t)warp * (uint32_t)(kBlkPerRound * 128) * ((act0 || act1) ? 1u : 0u);
            uint32_t sxa = sb + L.sxs + (uint32_t)blk0 * 4u;
            constexpr uint32_t kWStep = kCW * kBlkPerRound * kWB * 4, kSStep = kCW * kBlkPerRound * 2,
                               kZStep = kCW * kBlkPerRound, kXStep = kCW * kBlkPerRound * 4;
            // One round: columns 2t, 2t+1 of this thread = classes 0, 1 of block 4 rd + t for
            // rows g, g+8.  Two MMA chains per tile, whatever the tiles processed together (a
            // row's arithmetic must not depend on it); a chain's first MMA starts from zero.
            // The round's scales, zero points and sum of x are loaded first, so that their
            // latency passes under the MMAs.
            auto epilogue = [&](float (&d)[NTL][2][4], const uint32_t (&sAr)[NTL], const uint32_t (&sBr)[NTL],
                                const uint32_t (&zAr)[NTL], const uint32_t (&zBr)[NTL], float sx, bool inK) {
#pragma unroll
                for (int i = 0; i < NTL; ++i) {
                    const float sA = inK ? h2f(sAr[i]) : 0.f;  // past K: no scale (a dense copy holds other bytes)
                    const float sB = inK ? h2f(sBr[i]) : 0.f;
                    const float zA = HAS_ZP ? u8f(zAr[i]) : (float)kDefaultZp;
                    const float zB = HAS_ZP ? u8f(zBr[i]) : (float)kDefaultZp;
                    const float dd0 = d[i][0][0] + d[i][1][0], dd1 = d[i][0][1] + d[i][1][1];
                    const float dd2 = d[i][0][2] + d[i][1][2], dd3 = d[i][0][3] + d[i][1][3];
                    // sum_k x q of the block in units of 2^-24 (INT4: class 1, the high nibble, reads as 16 q)
                    const float u0 = fmaf(-zA, sx, fmaf(U::kHiWeight, dd1, dd0));
                    const float u1 = fmaf(-zB, sx, fmaf(U::kHiWeight, dd3, dd2));
                    v[i][0] = fmaf(sA, u0, v[i][0]);
                    v[i][1] = fmaf(sB, u1, v[i][1]);
                }
            };
            auto meta = [&](uint32_t (&sAr)[NTL], uint32_t (&sBr)[NTL], uint32_t (&zAr)[NTL], uint32_t (&zBr)[NTL]) {
#pragma unroll
                for (int i = 0; i < NTL; ++i) {
                    sAr[i] = lds_u16_s(sA_[i]);
                    sBr[i] = lds_u16_s(sB_[i]);
                    zAr[i] = HAS_ZP ? lds_u8_s(zA_[i]) : 0u;
                    zBr[i] = HAS_ZP ? lds_u8_s(zB_[i]) : 0u;
                    sA_[i] += kSStep;
                    sB_[i] += kSStep;
                    zA_[i] += kZStep;
                    zB_[i] += kZStep;
                }
            };
            if constexpr (BITS == 4) {
                // 16 bytes of rows g and g + 8 per tile and round.  The next round's codes go
                // into the same registers as soon as this round's last word is unpacked, so
                // their loads pass under this round's last MMAs and epilogue.
                uint4 ca[NTL], cb[NTL];
                auto codes = [&]() {
#pragma unroll
                    for (int i = 0; i < NTL; ++i) {
                        ca[i] = lds128_s<0>(wA[i]);
                        cb[i] = lds128_s<0>(wB[i]);
                        wA[i] += kWStep;
                        wB[i] += kWStep;
                    }
                };
                if (warp < nround) codes();
#pragma unroll 1
                for (int rd = warp; rd < nround; rd += kCW) {
                    uint32_t sAr[NTL], sBr[NTL], zAr[NTL], zBr[NTL];
                    const float sx = lds_f32_s(sxa);
                    meta(sAr, sBr, zAr, zBr);
                    float d[NTL][2][4];
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        // word w: one 16-byte x load = the B pairs of its two MMAs
                        const uint4 xw = w == 0 ? lds128_s<0>(xo)
                                       : w == 1 ? lds128_s<16>(xo)
                                       : w == 2 ? lds128_s<32>(xo)
                                                : lds128_s<48>(xo);
                        uint32_t pa[NTL][4], pb[NTL][4];
#pragma unroll
                        for (int i = 0; i < NTL; ++i) {
                            const uint32_t wa4[4] = {ca[i].x, ca[i].y, ca[i].z, ca[i].w};
                            const uint32_t wb4[4] = {cb[i].x, cb[i].y, cb[i].z, cb[i].w};
                            U::pairs(wa4[w], pa[i]);
                            U::pairs(wb4[w], pb[i]);
                        }
                        if (w == 3 && rd + kCW < nround) codes();
#pragma unroll
                        for (int i = 0; i < NTL; ++i) {
                            if (w == 0) {
                                mma_16816_z(d[i][0], pa[i][0], pb[i][0], pa[i][1], pb[i][1], xw.x, xw.y);
                                mma_16816_z(d[i][1], pa[i][2], pb[i][2], pa[i][3], pb[i][3], xw.z, xw.w);
                            } else {
                                mma_16816(d[i][0], pa[i][0], pb[i][0], pa[i][1], pb[i][1], xw.x, xw.y);
                                mma_16816(d[i][1], pa[i][2], pb[i][2], pa[i][3], pb[i][3], xw.z, xw.w);
                            }
                        }
                    }
                    xo += xs_step;
                    sxa += kXStep;
                    epilogue(d, sAr, sBr, zAr, zBr, sx, rd * kBlkPerRound + t < nblk);
                }
            } else {
#pragma unroll 1
                for (int rd = warp; rd < nround; rd += kCW) {
                    float d[NTL][2][4];
#pragma unroll
                    for (int q = 0; q < kWB / 4; ++q) {  // 16 bytes of each row at a time
                        uint4 wa[NTL], wb[NTL];
#pragma unroll
                        for (int i = 0; i < NTL; ++i) {
                            wa[i] = q == 0 ? lds128_s<0>(wA[i]) : lds128_s<16>(wA[i]);
                            wb[i] = q == 0 ? lds128_s<0>(wB[i]) : lds128_s<16>(wB[i]);
                        }
                        // words 4q .. 4q+3: an 8-byte B pair each
                        const uint4 xa = q == 0 ? lds128_s<0>(xo) : lds128_s<32>(xo);
                        const uint4 xb = q == 0 ? lds128_s<16>(xo) : lds128_s<48>(xo);
                        const uint32_t X[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
#pragma unroll
                        for (int w = 0; w < 4; ++w)
#pragma unroll
                            for (int i = 0; i < NTL; ++i) {
                                const uint32_t wa4[4] = {wa[i].x, wa[i].y, wa[i].z, wa[i].w};
                                const uint32_t wb4[4] = {wb[i].x, wb[i].y, wb[i].z, wb[i].w};
                                uint32_t pa[2], pb[2];
                                U::pairs(wa4[w], pa);
                                U::pairs(wb4[w], pb);
                                if (q == 0 && w < 2)
                                    mma_16816_z(d[i][w & 1], pa[0], pb[0], pa[1], pb[1], X[2 * w], X[2 * w + 1]);
                                else
                                    mma_16816(d[i][w & 1], pa[0], pb[0], pa[1], pb[1], X[2 * w], X[2 * w + 1]);
                            }
                    }
#pragma unroll
                    for (int i = 0; i < NTL; ++i) {
                        wA[i] += kWStep;
                        wB[i] += kWStep;
                    }
                    uint32_t sAr[NTL], sBr[NTL], zAr[NTL], zBr[NTL];
                    const float sx = lds_f32_s(sxa);
                    meta(sAr, sBr, zAr, zBr);
                    xo += xs_step;
                    sxa += kXStep;
                    epilogue(d, sAr, sBr, zAr, zBr, sx, rd * kBlkPerRound + t < nblk);
                }
            }
            // the quad's four blocks, then this warp's rows into the reduction buffer
#pragma unroll
            for (int i = 0; i < NTL; ++i) {
                float v0 = v[i][0], v1 = v[i][1];
                v0 += __shfl_xor_sync(0xffffffffu, v0, 1);
                v1 += __shfl_xor_sync(0xffffffffu, v1, 1);
                v0 += __shfl_xor_sync(0xffffffffu, v0, 2);
                v1 += __shfl_xor_sync(0xffffffffu, v1, 2);
                if (t == 0) {
                    redb[((tl0 + i) * kCW + warp) * 16 + g] = v0;
                    redb[((tl0 + i) * kCW + warp) * 16 + g + 8] = v1;
                }
            }
        };
        if (ok) {
            for (int tl0 = 0; tl0 < ntile; tl0 += 2) {
                if (tl0 + 1 < ntile)
                    tiles(std::integral_constant<int, 2>{}, tl0);
                else
                    tiles(std::integral_constant<int, 1>{}, tl0);
            }
        }
        named_barrier_sync(kNamed, kCW * 32);
        __syncwarp();
        if (lane == 0) mbar_arrive(empty(s));  // every read of the slot is done
        if (warp < ntile && lane < 16) {
            // MMA row `lane` of tile `warp`: row warp 8 + lane / 2 (+ 4 for lane >= 8) of region lane & 1
            const int m = lane & 7, rr = warp * 8 + (m >> 1) + (lane >> 3) * 4;
            const int row = (m & 1) ? hh + rr : rr;
            if (ok && ((m & 1) ? row < rs : rr < hh)) {
                float v = 0.f;
#pragma unroll
                for (int w = 0; w < kCW; ++w) v += redb[(warp * kCW + w) * 16 + lane];  // warp order
                const float y = v * (1.0f / kUnit);
                if (LORA) {  // the adapter term comes at the end
                    reinterpret_cast<float*>(sm + L.ybuf)[it.pos - r0 + row] = y;
                } else {
                    const float bn = st == 0 ? bias0 : (pj.bias ? __half2float(pj.bias[ra + row]) : 0.f);
                    pj.Y[ra + row] = __float2half_rn(pj.bias ? y + bn : y);
                }
            }
        }
    }
    if constexpr (LORA) {
        // each row: base + T B^T (one adapter projection: one segment), + bias, rounded once
        named_barrier_sync(kNamed, kCW * 32);
        if (r0 < r1 && ok && mbar_wait(lready, 0u, status)) {
            const DecSeg& pj = a.seg[0];
            const float* ybuf = reinterpret_cast<const float*>(sm + L.ybuf);
            const float* lorb = reinterpret_cast<const float*>(sm + L.lorb);
            for (int row = ctid; row < r1 - r0; row += kCW * 32) {
                float y = ybuf[row] + lorb[row];
                if (pj.bias) y += row == ctid ? bias0 : __half2float(pj.bias[r0 + row]);
                pj.Y[r0 + row] = __float2half_rn(y);
            }
        }
    }
}

template <int BITS, bool HAS_ZP, bool LORA, bool Q8L = false>
cudaError_t dec_launch_one(const DecMaps& maps, const DecodeArgs& a, int ctas, size_t smem, bool pdl,
                           cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ctas);
    cfg.blockDim = dim3(dec_threads(LORA));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    if (LORA) {  // the adapter's CTAs wait for one another: all resident at once
        attr[na].id = cudaLaunchAttributeCooperative;
        attr[na].val.cooperative = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, decode_kernel<BITS, HAS_ZP, LORA, Q8L>, maps, a);
}

constexpr int kMaxDev = 64;
// Per device (set up in its current context): the exchange areas' device address
// and the next area to hand out.
LoraEx* g_ex_base[kMaxDev] = {};
std::atomic<unsigned int> g_ex_next[kMaxDev];

int dec_ctas(int N, int sms) {
    int C = (N + 15) / 16;
    const int s = sms > 0 ? sms : 1;
    if (C > s) C = s;
    if (C > kExMaxC) C = kExMaxC;
    return C < 1 ? 1 : C;
}

}  // namespace

bool decode_supported(int bits, int64_t Mt, int K, int64_t N, bool lora, int sms) {
    if (!((bits == 4 || bits == 8) && Mt == 1 && K >= 32 && K <= 65536)) return false;
    if (lora && (N > (int64_t)INT32_MAX || lora_rows((int)N, dec_ctas((int)N, sms)) > kMaxLoraRows)) return false;
    return true;
}

void decode_geometry(int N, int K, int bits, bool lora, int sms, int* ctas, int* SR, int* ring, size_t* smem,
                     bool lq8) {
    const int C = dec_ctas(N, sms);
    const int nblk = K / 32, nround = (nblk + kBlkPerRound - 1) / kBlkPerRound, nblkR = nround * kBlkPerRound;
    const int rowbytes = K * bits / 8;
    const int rmax = (N + C - 1) / C;
    const int lrows = lora ? lora_rows(N, C) : 0;
    // The whole share in one stage when it fits in half an SM's shared memory: two CTAs
    // per SM, so the next call's CTA prefetches its share while this one finishes.
    // Larger shares stream through a ring of ~200 KB (one CTA per SM), in stages of at
    // least ~24 KB (fewer per-stage barriers for short rows).
    constexpr uint32_t kHalfSm = 112u * 1024u, kRing = 200u * 1024u;
    int sr = 16;
    while (sr < rmax) sr *= 2;
    if (sr <= kMaxSR && dec_layout(sr, 1, bits, rowbytes, nblk, nblkR, lrows, lq8).total <= kHalfSm) {
        *SR = sr;
        *ring = 1;
    } else {
        int sr2 = 16;
        while (sr2 < 64 && dec_layout(sr2, 1, bits, rowbytes, nblk, nblkR, lrows, lq8).slot < 24u * 1024u) sr2 *= 2;
        int r = 1;
        while (r < 16 && dec_layout(sr2, r + 1, bits, rowbytes, nblk, nblkR, lrows, lq8).total <= kRing) ++r;
        *SR = sr2;
        *ring = r;
    }
    *ctas = C;
    *smem = dec_layout(*SR, *ring, bits, rowbytes, nblk, nblkR, lrows, lq8).total;
}

cudaError_t decode_prepare() {
    cudaError_t e = tensor_map_prepare();
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
#define MNB_DEC_SET(B, Z, L, Q)                                                                                    \
    if (e == cudaSuccess)                                                                                            \
        e = cudaFuncSetAttribute(decode_kernel<B, Z, L, Q>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024); \
    if (e == cudaSuccess) /* the largest carveout: two CTAs of up to ~112 KB per SM */                                \
        e = cudaFuncSetAttribute(decode_kernel<B, Z, L, Q>, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    MNB_DEC_SET(4, false, false, false) MNB_DEC_SET(4, true, false, false)
    MNB_DEC_SET(4, false, true, false) MNB_DEC_SET(4, true, true, false)
    MNB_DEC_SET(4, false, true, true) MNB_DEC_SET(4, true, true, true)
    MNB_DEC_SET(8, false, false, false) MNB_DEC_SET(8, true, false, false)
    MNB_DEC_SET(8, false, true, false) MNB_DEC_SET(8, true, true, false)
    MNB_DEC_SET(8, false, true, true) MNB_DEC_SET(8, true, true, true)
#undef MNB_DEC_SET
    void* ex = nullptr;
    if (e == cudaSuccess) e = cudaGetSymbolAddress(&ex, g_lora_ex);
    if (e == cudaSuccess) g_ex_base[dev] = static_cast<LoraEx*>(ex);
    return e;
}

cudaError_t decode_reset_exchange() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev || !g_ex_base[dev]) return cudaSuccess;
    return cudaMemset(g_ex_base[dev], 0, sizeof(g_lora_ex));
}

cudaError_t decode_launch(const DecodeArgs& a_in, int rank, int sms, bool pdl, cudaStream_t st) {
    DecodeArgs a = a_in;
    int C, SR, ring;
    size_t smem;
    const int bits = a.bits;
    const bool q8l = rank > 0 && a.Aq != nullptr;  // INT8 adapter
    decode_geometry(a.NR, a.K, bits, rank > 0, sms, &C, &SR, &ring, &smem, q8l);
    if (smem > 227 * 1024) return cudaErrorNotSupported;
    a.SR = SR;
    a.ring = ring;
    if (rank > 0) {
        if (a.nseg != 1 || lora_rows(a.NR, C) > kMaxLoraRows) return cudaErrorNotSupported;
        int dev = -1;
        if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev || !g_ex_base[dev])
            return cudaErrorInvalidDevice;
        // one exchange area per call, round robin: calls in flight at once on
        // different streams use different areas
        a.ex = g_ex_base[dev] + (g_ex_next[dev].fetch_add(1u, std::memory_order_relaxed) % kExSlots);
    }
    // scale / zero-point boxes of SR rows, each row padded to the shared-memory pitch
    DecMaps maps;
    memset(&maps, 0, sizeof(maps));
    const int nblk = a.K / 32;
    const DecPitch P = dec_pitch(nblk);
    const bool zp = a.seg[0].Z != nullptr, lora = rank > 0;
    for (int i = 0; i < a.nseg; ++i) {
        cudaError_t e = cudaSuccess;
        if (P.tma_s)
            e = encode_2d(&maps.s[i], a.seg[i].S, 2, (uint64_t)nblk, (uint64_t)a.seg[i].N, (uint64_t)nblk * 2,
                          P.spitch / 2u, (uint32_t)SR, false);
        if (e == cudaSuccess && zp && P.tma_z)
            e = encode_2d(&maps.z[i], a.seg[i].Z, 1, (uint64_t)nblk, (uint64_t)a.seg[i].N, (uint64_t)nblk,
                          P.zpitch, (uint32_t)SR, false);
        if (e != cudaSuccess) return e;
    }
    if (bits == 4) {
        if (q8l)
            return zp ? dec_launch_one<4, true, true, true>(maps, a, C, smem, pdl, st)
                      : dec_launch_one<4, false, true, true>(maps, a, C, smem, pdl, st);
        if (lora)
            return zp ? dec_launch_one<4, true, true>(maps, a, C, smem, pdl, st)
                      : dec_launch_one<4, false, true>(maps, a, C, smem, pdl, st);
        return zp ? dec_launch_one<4, true, false>(maps, a, C, smem, pdl, st)
                  : dec_launch_one<4, false, false>(maps, a, C, smem, pdl, st);
    }
    if (q8l)
        return zp ? dec_launch_one<8, true, true, true>(maps, a, C, smem, pdl, st)
                  : dec_launch_one<8, false, true, true>(maps, a, C, smem, pdl, st);
    if (lora)
        return zp ? dec_launch_one<8, true, true>(maps, a, C, smem, pdl, st)
                  : dec_launch_one<8, false, true>(maps, a, C, smem, pdl, st);
    return zp ? dec_launch_one<8, true, false>(maps, a, C, smem, pdl, st)
              : dec_launch_one<8, false, false>(maps, a, C, smem, pdl, st);
}

}  // namespace mnb
