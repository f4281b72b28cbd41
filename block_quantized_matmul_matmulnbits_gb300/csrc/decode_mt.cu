// decode_mt.cu -- decode kernel for a few token rows (2 .. 16): one launch computes
//
//     Y[m, n] = sum_k X[m, k] w[n, k]  (+ sum_r T[m, r] B[n, r])  (+ bias[n])
//
// for every token row m, the decode ("fuse_down") path of "[WebGPU] Fuse rank-32
// quantized LoRA with MatMulNBits" (onnxruntime PR 33370, commit message adding
// MatMulNBitsLoRA: the decode mode is chosen from the per-matrix row count; the base
// GEMV and T = X A first, then base plus T B^T), restated for sm_103a with the token
// rows as the MMA's N.  T comes from the LoRA down kernel launched just before.
//
// Design:
//  * Rows are split evenly over the CTAs (one per SM), as in the single-token
//    kernel.  A producer warp streams the CTA's rows through a ring of slots: a
//    16-row stage arrives as `kparts` slots, each a K range of the 16 rows (codes
//    as one 3-D TMA box of 16 rows x the range's 128-byte segments, 128-byte
//    swizzle: 16-byte chunk c of row r lands at c ^ (r & 7), so one 4-byte load
//    per thread reads 8 rows x 4 words in 32 different banks; scales and zero
//    points as 2-D TMA boxes with padded rows).  The whole share is prefetched
//    into L2 once x is staged (before that it would only queue behind the x loads).
//  * mma.sync m16n8k16 with 16 weight rows as M and 8 token rows as N.  A code
//    reaches the tensor core as the FP16 value q * 2^-24 (exact), so unpacking is
//    a mask (INT4) or a byte permute (INT8).  An INT4 word's low and high nibbles
//    go to two MMAs (the high nibble reads as 16 q, its x is staged as x / 16),
//    each covering one half of a block's codes for the quad's four words.  The
//    MMAs of a block start from -zp * sum_k x, so they end at sum_k x (q - zp),
//    and the thread applies y += s * that in FP32.
//  * Warp w takes blocks w, w + 16, ... of every stage, for every token tile:
//    a block's codes are unpacked once for all the token rows.  x is staged once
//    per CTA by the thread that reads it: each thread keeps the B fragments of its
//    blocks (16 bytes a block and token tile) and their sums of x (one MMA with
//    all codes 1).
//  * The consumer warps never wait for one another: each frees a slot when it has
//    read it, and hands its partial sums of a stage to a reducer warp through a
//    pair of barriers; the reducer adds the 16 warps' partials in a fixed order
//    (no atomics) while the consumers work on the next stage.  Results are
//    deterministic and independent of how the rows were split into CTAs.
//  * Every mbarrier wait is bounded and reports through the status word.
#include <cuda.h>

#include <cstring>
#include <type_traits>

#include "common.cuh"
#include "decode_common.cuh"
#include "mnb_internal.h"

namespace mnb {

namespace {

using namespace dec;

constexpr int kMtCW = 16;                         // consumer warps
constexpr int kMtThreads = (kMtCW + 2) * 32;      // + the producer and the reducer warps
constexpr int kMtSR = 16;                         // rows per stage: one box
constexpr int kMtMaxRing = 12;
constexpr uint32_t kMtSmem = 227u * 1024u;        // shared memory of one CTA per SM
constexpr uint32_t kXF = kMtCW * 512u;            // x fragments of one block and token tile, all warps
constexpr uint32_t kQF = kMtCW * 64u;             // MMA starting values of one block and token tile, all warps
constexpr int kPS = 20;                           // partials: floats between two outputs (16 warps + 4)

// Shared-memory loads at a 32-bit address plus a constant offset (the assembler folds
// the addition into the load); volatile: they stay after the barrier waits before them.
__device__ __forceinline__ uint32_t lds32_dyn(uint32_t a, uint32_t off) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a + off));
    return v;
}
__device__ __forceinline__ uint32_t lds16_dyn(uint32_t a, uint32_t off) {
    uint16_t v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a + off));
    return v;
}
__device__ __forceinline__ uint32_t lds8_dyn(uint32_t a, uint32_t off) {
    uint32_t v;
    asm volatile("ld.shared.u8 %0, [%1];" : "=r"(v) : "r"(a + off));
    return v;
}
__device__ __forceinline__ uint4 lds128_dyn(uint32_t a, uint32_t off) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a + off));
    return v;
}
__device__ __forceinline__ void sts128(uint32_t a, uint4 v) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}
// Predicated shared-memory store and mbarrier arrival (no branch around them).
__device__ __forceinline__ void sts128_if(bool p, uint32_t a, uint4 v) {
    asm volatile(
        "{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %0, 0;\n\t"
        "@q st.shared.v4.u32 [%1], {%2, %3, %4, %5};\n\t}" ::"r"((uint32_t)p),
        "r"(a), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
        : "memory");
}
__device__ __forceinline__ void mbar_arrive_if(bool p, uint32_t bar) {
    asm volatile(
        "{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %0, 0;\n\t"
        "@q mbarrier.arrive.shared::cta.b64 _, [%1];\n\t}" ::"r"((uint32_t)p),
        "r"(bar)
        : "memory");
}
// A register copy the compiler keeps where it stands.
__device__ __forceinline__ float fmov_here(float x) {
    float y;
    asm volatile("mov.b32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ uint4 ldg128_nc(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}
__device__ __forceinline__ uint2 ldg64_nc(const void* p) {
    uint2 v;
    asm volatile("ld.global.nc.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}

// Shared memory plan, identical on host and device.  Slot s holds a K range of one
// 16-row stage: codes at s * codes (one box [segment][16 rows][128 B]), scales at
// sc + s * 16 spitch, zero points at zp + s * 16 zpitch.  After the ring (unless the
// threads keep them in registers): the threads' x fragments [block][token tile]
// [warp][lane][16 B] and the MMAs' starting values [block][token tile][warp][t][4]
// FP32; then the warps' partials of a stage, in one buffer or (with x in registers,
// where shared memory is plentiful) two, stage st in buffer st % buffers: [output
// (token row x 16 + row)][warp] FP32 (kPS floats an output), the barriers
// full[ring], empty[ring], "x staged", "partials written"[2] and "partials added"[2],
// and a flag: every consumer's waits ended in time.
struct MtLayout {
    uint32_t codes, sc, zp;
    uint32_t spitch, zpitch;
    uint32_t xs, cq, red, bars, total;
};

__host__ __device__ inline MtLayout mt_layout(int ring, int bits, int K, int nt8, int parts, bool zp, bool xreg) {
    const int nblk = K / 32, nbp = nblk / parts;
    const uint32_t rowbytes = (uint32_t)K * (uint32_t)bits / 8u / (uint32_t)parts;  // of a slot's K range
    const DecPitch P = dec_pitch(nbp);
    MtLayout L;
    L.codes = 16u * rowbytes;  // a multiple of 2048: the boxes stay 1024-aligned
    L.spitch = P.spitch;
    L.zpitch = P.zpitch;
    L.sc = (uint32_t)ring * L.codes;
    L.zp = L.sc + (uint32_t)ring * (uint32_t)kMtSR * P.spitch;
    L.xs = al128(L.zp + (zp ? (uint32_t)ring * (uint32_t)kMtSR * P.zpitch : 0u));
    L.cq = L.xs + (xreg ? 0u : (uint32_t)nblk * (uint32_t)nt8 * 512u);
    L.red = al128(L.cq + (xreg ? 0u : (uint32_t)nblk * (uint32_t)nt8 * 64u));
    L.bars = al128(L.red + (xreg ? 2u : 1u) * 16u * 8u * (uint32_t)nt8 * (uint32_t)kPS * 4u);
    L.total = L.bars + (2u * (uint32_t)ring + 6u) * 8u;  // + the "waits ended in time" flag
    return L;
}

// The CTA's rows as 16-row stages that never straddle two projections.  The
// current projection's bounds stay in registers: the kernel parameters (indexed by
// a register) are read again only when the stages move to the next projection.
struct MtRows {
    int pos, r1;         // first row of the stage (row space), end of the CTA's rows
    int seg, row0, end;  // current projection, its first row and end (row space)
    int ra, rs;          // the stage's first row inside the projection, its rows
    __device__ __forceinline__ void load(const DecodeArgs& a) {
        while (seg + 1 < a.nseg && pos >= a.seg[seg + 1].row0) ++seg;  // empty projections start where the next does
        row0 = a.seg[seg].row0;
        end = row0 + a.seg[seg].N;
    }
    __device__ __forceinline__ void set() {
        rs = min(min(kMtSR, r1 - pos), end - pos);
        ra = pos - row0;
    }
    __device__ __forceinline__ void init(const DecodeArgs& a, int r0, int r1_) {
        pos = r0;
        r1 = r1_;
        seg = 0;
        if (pos < r1) {
            load(a);
            set();
        }
    }
    // Next stage; true when it starts a new projection.
    __device__ __forceinline__ bool next(const DecodeArgs& a) {
        pos += rs;
        if (pos >= r1) return false;
        const bool moved = pos >= end;
        if (moved) load(a);
        set();
        return moved;
    }
};

// TMA descriptors per projection: codes (3-D, swizzled), scales and zero points.
struct MtMaps {
    CUtensorMap c[kMaxSeg];
    CUtensorMap s[kMaxSeg];
    CUtensorMap z[kMaxSeg];
};

// A CTA's shared-memory plan and barriers, as every role sees them.
struct MtCtx {
    MtLayout L;
    uint32_t sb;  // shared base, 1024-aligned
    unsigned char* sm;
    int ring, H, nblk, r0, r1, nt8, nbuf;  // nbuf: buffers of partials
    unsigned int* status;
    __device__ __forceinline__ uint32_t full(int s) const { return sb + L.bars + 8u * (uint32_t)s; }
    __device__ __forceinline__ uint32_t empty(int s) const { return sb + L.bars + 8u * (uint32_t)(ring + s); }
    __device__ __forceinline__ uint32_t xready() const { return sb + L.bars + 16u * (uint32_t)ring; }
    // buffer b of the partials: written by all consumer warps, then added
    __device__ __forceinline__ uint32_t pfull(int b) const { return xready() + 8u + 8u * (uint32_t)b; }
    __device__ __forceinline__ uint32_t pfree(int b) const { return xready() + 24u + 8u * (uint32_t)b; }
    __device__ __forceinline__ float* red(int b) const {
        return reinterpret_cast<float*>(sm + L.red) + b * (128 * nt8 * kPS);
    }
    __device__ __forceinline__ volatile int* in_time() const {
        return reinterpret_cast<volatile int*>(sm + L.bars + 16u * (uint32_t)ring + 40u);
    }
};

// The plan and the barriers (set up by thread 0); then the whole CTA meets and the
// dependent launch is released.
template <int BITS, bool HAS_ZP>
__device__ __forceinline__ MtCtx mt_setup(const DecodeArgs& a, int nt8, bool xreg, unsigned char* sm_raw) {
    MtCtx c;
    c.ring = a.ring;
    c.H = a.kparts;
    c.nblk = a.K >> 5;
    c.nt8 = nt8;
    c.nbuf = xreg ? 2 : 1;
    c.L = mt_layout(c.ring, BITS, a.K, nt8, c.H, HAS_ZP, xreg);
    c.sb = (smem_u32(sm_raw) + 1023u) & ~1023u;  // swizzled boxes want 1024-byte alignment
    c.sm = sm_raw + (c.sb - smem_u32(sm_raw));
    const int C = gridDim.x;
    c.r0 = (int)((long long)blockIdx.x * a.NR / C);
    c.r1 = (int)((long long)(blockIdx.x + 1) * a.NR / C);
    c.status = a.status;
    if (threadIdx.x == 0) {
        for (int s = 0; s < c.ring; ++s) {
            mbar_init(c.full(s), 1);
            mbar_init(c.empty(s), kMtCW);
        }
        mbar_init(c.xready(), kMtCW);
        for (int b = 0; b < 2; ++b) {
            mbar_init(c.pfull(b), kMtCW);
            mbar_init(c.pfree(b), 1);
        }
        *c.in_time() = 1;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    pdl_launch_dependents();
    return c;
}

// The producer (one thread): the CTA's stages as slots of K ranges through the ring.
// Whole 16-row boxes land, rows past N reading as zero; the MMA rows of a shorter
// stage past its end read the next rows, and are not stored.
template <int BITS, bool HAS_ZP>
__device__ __forceinline__ void mt_produce(const MtMaps& maps, const DecodeArgs& a, const MtCtx& c) {
    const int K = a.K, H = c.H, ring = c.ring, nblk = c.nblk, r0 = c.r0, r1 = c.r1;
    const MtLayout& L = c.L;
    const uint32_t rowbytes = (uint32_t)K * BITS / 8u;
    const int segp = (int)(rowbytes / 128u) / H, nbp = nblk / H;  // per slot
    const uint32_t bytes = L.codes + (uint32_t)kMtSR * L.spitch + (HAS_ZP ? (uint32_t)kMtSR * L.zpitch : 0u);
    bool ok = true;
    int q = 0;  // slots issued
    MtRows it;
    it.init(a, r0, r1);
    for (; ok && it.pos < r1; it.next(a)) {
        for (int h = 0; h < H; ++h, ++q) {
            const int s = q % ring;
            const uint32_t par = (uint32_t)(q / ring) & 1u;
            if (q == ring) {
                // The ring is full: once x is staged, the rest of the share into L2 at
                // once, so that the refills come from L2 while HBM streams the
                // remainder at full rate.
                mbar_wait(c.xready(), 0u, c.status);
                for (int sg = 0; sg < a.nseg; ++sg) {
                    const DecSeg& pg = a.seg[sg];
                    const int lo = max(r0, pg.row0), hi = min(r1, pg.row0 + pg.N);
                    if (lo >= hi) continue;
                    const size_t ra = (size_t)(lo - pg.row0), n = (size_t)(hi - lo);
                    for (size_t off = 0; off < n * rowbytes; off += (1u << 20))
                        prefetch_l2_bulk(pg.Wq + ra * rowbytes + off,
                                         (uint32_t)min((size_t)(1u << 20), n * rowbytes - off));
                    prefetch_l2_bulk(reinterpret_cast<const uint8_t*>(pg.S) + ra * nblk * 2, (uint32_t)(n * nblk * 2));
                    if (HAS_ZP) prefetch_l2_bulk(pg.Z + ra * nblk, (uint32_t)(n * nblk));
                }
            }
            if (q >= ring && !(ok = mbar_wait(c.empty(s), par ^ 1u, c.status))) break;
            mbar_arrive_tx(c.full(s), bytes);
            tma_load_3d(c.sb + (uint32_t)s * L.codes, &maps.c[it.seg], 0, it.ra, h * segp, c.full(s));
            tma_load_2d(c.sb + L.sc + (uint32_t)s * kMtSR * L.spitch, &maps.s[it.seg], h * nbp, it.ra, c.full(s));
            if (HAS_ZP)
                tma_load_2d(c.sb + L.zp + (uint32_t)s * kMtSR * L.zpitch, &maps.z[it.seg], h * nbp, it.ra, c.full(s));
        }
    }
    // no copy may still be in flight when the CTA exits (a consumer may have given up)
    for (int i = q > ring ? q - ring : 0; i < q; ++i) mbar_wait(c.full(i % ring), (uint32_t)(i / ring) & 1u, c.status, false);
}

// The reducer (one warp): output o = lane + 32 i of a stage is token row o >> 4, row
// o & 15, the sum of the 16 warps' partials in warp order (plus, with an adapter,
// sum_r T[tok, r] B[n, r]), one rounding.  The adapter term comes from two MMAs per
// token tile (16 rows of B x T of 8 token rows, FP32 accumulation), which the warp
// stores in the partials' unit (times 2^-24, exact) as a 17th partial of each output.
// T is the previous launch's output (the LoRA down kernel): read after the wait for it.
template <int NT8>
__device__ __forceinline__ void mt_reduce(const DecodeArgs& a, const MtCtx& c, int lane) {
    if (c.r0 >= c.r1) return;
    const bool lora = a.B != nullptr;
    const int g = lane >> 2, t = lane & 3;
    bool ok = true;
    // T fragments (the MMA's B operand): token row 8 jt + g, ranks 16 ks + 2t, + 1 and + 8, + 9
    uint32_t tf[NT8][2][2];
#pragma unroll
    for (int jt = 0; jt < NT8; ++jt)
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) tf[jt][ks][0] = tf[jt][ks][1] = 0u;
    if (lora) {
        pdl_wait();
#pragma unroll
        for (int jt = 0; jt < NT8; ++jt) {
            const int tok = 8 * jt + g;
            if (tok < a.Mt) {
                const __half* tr = a.T + (size_t)tok * 32 + 2 * t;
#pragma unroll
                for (int ks = 0; ks < 2; ++ks) {
                    tf[jt][ks][0] = ldg_nc_u32(tr + 16 * ks);
                    tf[jt][ks][1] = ldg_nc_u32(tr + 16 * ks + 8);
                }
            }
        }
    }
    MtRows it;
    it.init(a, c.r0, c.r1);
    __half* Yp = a.seg[it.seg].Y;
    const __half* bp = a.seg[it.seg].bias;
    int Np = a.seg[it.seg].N;
    bool moved = false;
    for (int st = 0; it.pos < c.r1; moved = it.next(a), ++st) {
        if (moved) {
            Yp = a.seg[it.seg].Y;
            bp = a.seg[it.seg].bias;
            Np = a.seg[it.seg].N;
        }
        // the stage's adapter rows (the MMA's A operand: rows g, g + 8, ranks as T's),
        // loaded before the wait for the partials so that their latency passes under it
        uint32_t bf[2][4];
#pragma unroll
        for (int ks = 0; ks < 2; ++ks)
#pragma unroll
            for (int e = 0; e < 4; ++e) bf[ks][e] = 0u;
        if (lora) {
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                const int r = g + 8 * hr;
                if (r < it.rs) {
                    const __half* br = a.B + (size_t)(it.ra + r) * 32 + 2 * t;
#pragma unroll
                    for (int ks = 0; ks < 2; ++ks) {
                        bf[ks][hr] = ldg_nc_u32(br + 16 * ks);
                        bf[ks][2 + hr] = ldg_nc_u32(br + 16 * ks + 8);
                    }
                }
            }
        }
        const int b = st % c.nbuf, use = st / c.nbuf;  // stage st's buffer, in its use-th use
        if (ok) ok = mbar_wait(c.pfull(b), (uint32_t)use & 1u, c.status) && *c.in_time();
        float* red = c.red(b);
        if (lora) {
#pragma unroll
            for (int jt = 0; jt < NT8; ++jt) {
                float d[4];
                mma_16816_z(d, bf[0][0], bf[0][1], bf[0][2], bf[0][3], tf[jt][0][0], tf[jt][0][1]);
                mma_16816(d, bf[1][0], bf[1][1], bf[1][2], bf[1][3], tf[jt][1][0], tf[jt][1][1]);
                // d: rows g, g + 8 x token rows 8 jt + 2t, + 1; output o = token row x 16 + row
                float* pl = red + ((8 * jt + 2 * t) * 16 + g) * kPS + kMtCW;
                pl[0] = d[0] * kUnit;
                pl[16 * kPS] = d[1] * kUnit;
                pl[8 * kPS] = d[2] * kUnit;
                pl[24 * kPS] = d[3] * kUnit;
            }
            __syncwarp();
        }
        float y[NT8 * 4];
#pragma unroll
        for (int i = 0; i < NT8 * 4; ++i) {
            const float* po = red + (lane + 32 * i) * kPS;
            const float4* pr = reinterpret_cast<const float4*>(po);
            const float4 p0 = pr[0], p1 = pr[1], p2 = pr[2], p3 = pr[3];
            y[i] = ((((((((((((((p0.x + p0.y) + p0.z) + p0.w) + p1.x) + p1.y) + p1.z) + p1.w) + p2.x) + p2.y) +
                          p2.z) + p2.w) + p3.x) + p3.y) + p3.z) + p3.w;
            if (lora) y[i] += po[kMtCW];
        }
        __syncwarp();
        mbar_arrive_if(lane == 0, c.pfree(b));  // every lane's reads are done
#pragma unroll
        for (int i = 0; i < NT8 * 4; ++i) {
            const int o = lane + 32 * i, tok = o >> 4, m = o & 15;
            if (ok && m < it.rs && tok < a.Mt) {
                float v = y[i] * (1.0f / kUnit);
                if (bp) v += __half2float(bp[it.ra + m]);
                Yp[(size_t)tok * Np + it.ra + m] = __float2half_rn(v);
            }
        }
    }
}

// A consumer warp hands its partials of stage st (thread (g, t): rows g, g + 8 x
// tokens 8 jt + 2t, + 1; offset pw in a buffer) to the reducer, once the reducer has
// added the stage that used the same buffer before.
template <int NT8>
__device__ __forceinline__ void mt_hand_over(const MtCtx& c, int pw, const float (&v)[NT8][4], int st, bool& ok,
                                             int lane) {
    const int b = st % c.nbuf, use = st / c.nbuf;
    if (use > 0 && ok) ok = mbar_wait(c.pfree(b), (uint32_t)(use - 1) & 1u, c.status);
    if (!ok) *c.in_time() = 0;
    float* pt0 = c.red(b) + pw;
#pragma unroll
    for (int jt = 0; jt < NT8; ++jt) {
        float* pt = pt0 + 128 * jt * kPS;
        pt[0] = v[jt][0];
        pt[16 * kPS] = v[jt][1];
        pt[8 * kPS] = v[jt][2];
        pt[24 * kPS] = v[jt][3];
    }
    __threadfence_block();
    __syncwarp();
    mbar_arrive_if(lane == 0, c.pfull(b));
}

template <int BITS, bool HAS_ZP, int NT8, int UB>
__global__ void __launch_bounds__(kMtThreads, 1)
    decode_mt_kernel(const __grid_constant__ MtMaps maps, const __grid_constant__ DecodeArgs a) {
    using U = Unpack<BITS>;
    constexpr uint32_t kDefaultZp = 1u << (BITS - 1);
    constexpr int kProducer = kMtCW, kReducer = kMtCW + 1;
    extern __shared__ unsigned char sm_raw[];
    const MtCtx c = mt_setup<BITS, HAS_ZP>(a, NT8, false, sm_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp == kProducer) {
        if (lane == 0) mt_produce<BITS, HAS_ZP>(maps, a, c);
        return;
    }
    if (warp == kReducer) {
        mt_reduce<NT8>(a, c, lane);
        return;
    }
    const int K = a.K, Mt = a.Mt, H = c.H, ring = c.ring, r0 = c.r0, r1 = c.r1;
    const int nj = c.nblk / kMtCW, njp = nj / H;  // blocks of a warp: per stage, per slot
    const MtLayout& L = c.L;
    const uint32_t sb = c.sb;
    unsigned int* status = c.status;

    // ---------------------------------------------------------------- consumers
    const int g = lane >> 2, t = lane & 3;
    if (r0 >= r1) {
        mbar_arrive_if(lane == 0, c.xready());
        return;
    }
    bool ok = true;

    // This thread's x fragment of its j-th block (block warp + kMtCW j) and token tile
    // jt at xf + (j NT8 + jt) kXF; at qf + (j NT8 + jt) kQF the MMA's starting
    // accumulator for rows g, g + 8 and tokens 2t, 2t + 1 of the tile: (c0, c1, c0, c1),
    // c = -8 sum_k x (INT4) or -128 sum_k x (INT8) without zero points, c = sum_k x
    // with them (times the rows' -zp then), all times 2^-24.
    const uint32_t xf = sb + L.xs + (uint32_t)warp * 512u + (uint32_t)lane * 16u;
    const uint32_t qf = sb + L.cq + (uint32_t)warp * 64u + (uint32_t)t * 16u;

    // ---- x of every token row: wait for the work that produces it, then stage it
    if (a.x_wait) pdl_wait();
    {
        // A constant code of 1 (2^-24) and, for INT4 high nibbles, 16 (their x is x / 16):
        // the MMA then gives sum_k x 2^-24 of the block for the tile's tokens.
        constexpr uint32_t kOne = 0x00010001u, kHi = BITS == 4 ? 0x00100010u : kOne;
        constexpr float kZs = HAS_ZP ? 1.f : -(float)kDefaultZp;
        constexpr int kXU = 8;  // fragments in flight per thread
        const __half2 k16 = __float2half2_rn(0.0625f);
        const int npc = nj * NT8;
        for (int i0 = 0; i0 < npc; i0 += kXU) {
            uint4 v[kXU];
#pragma unroll
            for (int u = 0; u < kXU; ++u) {
                const int i = i0 + u, j = i / NT8, tok = 8 * (i % NT8) + g;
                v[u] = make_uint4(0u, 0u, 0u, 0u);
                if (i < npc && tok < Mt) {
                    const __half* p = a.X + (size_t)tok * K + (size_t)(warp + kMtCW * j) * 32;
                    if constexpr (BITS == 4) {
                        v[u] = ldg128_nc(p + 8 * t);  // word t: x[8t .. 8t + 7]
                    } else {
                        const uint2 lo = ldg64_nc(p + 4 * t), hi = ldg64_nc(p + 16 + 4 * t);  // words t, t + 4
                        v[u] = make_uint4(lo.x, lo.y, hi.x, hi.y);
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < kXU; ++u) {
                const int i = i0 + u;
                if (i >= npc) break;  // the same for every thread
                uint4 o = v[u];
                if constexpr (BITS == 4) {  // (x0, x4) (x2, x6) (x1, x5)/16 (x3, x7)/16
                    const uint32_t h15 = prmt(o.x, o.z, 0x7632u), h37 = prmt(o.y, o.w, 0x7632u);
                    const __half2 s15 = __hmul2(*reinterpret_cast<const __half2*>(&h15), k16);
                    const __half2 s37 = __hmul2(*reinterpret_cast<const __half2*>(&h37), k16);
                    o = make_uint4(prmt(o.x, o.z, 0x5410u), prmt(o.y, o.w, 0x5410u),
                                   *reinterpret_cast<const uint32_t*>(&s15), *reinterpret_cast<const uint32_t*>(&s37));
                }
                sts128(xf + (uint32_t)i * kXF, o);
                float d[4];
                mma_16816_z(d, kOne, kOne, kOne, kOne, o.x, o.y);
                mma_16816(d, kHi, kHi, kHi, kHi, o.z, o.w);
                const uint32_t c0 = __float_as_uint(kZs * d[0]), c1 = __float_as_uint(kZs * d[1]);
                sts128_if(g == 0, qf + (uint32_t)i * kQF, make_uint4(c0, c1, c0, c1));
            }
        }
        __syncwarp();
        mbar_arrive_if(lane == 0, c.xready());
    }

    // ---- the stages
    // Codes of block b in the slot's box, row r: INT4 16 bytes at segment b >> 3, chunk
    // b & 7; INT8 32 bytes at segment b >> 2, chunks 2 (b & 3) and 2 (b & 3) + 1; a
    // segment is [16 rows][128 B], row r + 8 1024 bytes after row r.  Along this warp's
    // blocks (b = warp + 16 j) the chunk is fixed and the segment steps by a constant;
    // a slot starts at a multiple of 16 blocks.
    const uint32_t ch0 = BITS == 4 ? (uint32_t)(warp & 7) : 2u * (uint32_t)(warp & 3);
    const uint32_t c_off = (uint32_t)(BITS == 4 ? warp >> 3 : warp >> 2) * 2048u + (uint32_t)g * 128u +
                           ((ch0 ^ (uint32_t)g) << 4) + 4u * (uint32_t)t;
    const uint32_t c_hi = BITS == 4 ? 0u : (((ch0 + 1u) ^ (uint32_t)g) << 4) - ((ch0 ^ (uint32_t)g) << 4);  // word t + 4
    constexpr uint32_t kCStep = (BITS == 4 ? kMtCW / 8 : kMtCW / 4) * 2048u;
    constexpr uint32_t kSStep = 2u * kMtCW, kZStep = kMtCW;
    // the slot cursor: index, phase, and this thread's codes, scales and zero points in it
    int s = 0;
    uint32_t par = 0u;
    const uint32_t c_first = sb + c_off, s_first = sb + L.sc + (uint32_t)g * L.spitch + (uint32_t)warp * 2u;
    const uint32_t z_first = sb + L.zp + (uint32_t)g * L.zpitch + (uint32_t)warp;
    const uint32_t s8 = 8u * L.spitch, z8 = 8u * L.zpitch;
    uint32_t cS = c_first, sS = s_first, zS = z_first;
    // this thread's partials: rows g, g + 8 x tokens 8 jt + 2t, + 1
    const int pw = (32 * t + g) * kPS + warp;  // this thread's partials in a buffer
    MtRows it;
    it.init(a, r0, r1);
    for (int st = 0; it.pos < r1; it.next(a), ++st) {
        float v[NT8][4];
#pragma unroll
        for (int jt = 0; jt < NT8; ++jt) v[jt][0] = v[jt][1] = v[jt][2] = v[jt][3] = 0.f;
        uint32_t xo = xf, qo = qf;  // the slots follow each other in K, and so do the fragments
        for (int h = 0; h < H; ++h) {
            // after a timeout the slot's stale bytes are read all the same (in bounds)
            // and the reducer stores nothing
            if (ok) ok = mbar_wait(c.full(s), par, status);
            uint32_t cA = cS, sA = sS, zA = zS;
#pragma unroll 1
            for (int j = 0; j < njp; j += UB) {
                // UB blocks: every load first, then the MMAs, then the FP32 block
                // epilogues, so that the blocks' latencies overlap
                uint32_t wa[UB][2], wb[UB][2], sc[UB][2];
                [[maybe_unused]] uint32_t zq[UB][2];
                uint4 xw[UB][NT8], cq[UB][NT8];
#pragma unroll
                for (int u = 0; u < UB; ++u) {
                    wa[u][0] = lds32_dyn(cA, u * kCStep);
                    wb[u][0] = lds32_dyn(cA, u * kCStep + 1024u);
                    if constexpr (BITS == 8) {
                        wa[u][1] = lds32_dyn(cA + c_hi, u * kCStep);
                        wb[u][1] = lds32_dyn(cA + c_hi, u * kCStep + 1024u);
                    }
                    sc[u][0] = lds16_dyn(sA, u * kSStep);
                    sc[u][1] = lds16_dyn(sA + s8, u * kSStep);
                    if constexpr (HAS_ZP) {
                        zq[u][0] = lds8_dyn(zA, u * kZStep);
                        zq[u][1] = lds8_dyn(zA + z8, u * kZStep);
                    }
#pragma unroll
                    for (int jt = 0; jt < NT8; ++jt) {
                        xw[u][jt] = lds128_dyn(xo, (u * NT8 + jt) * kXF);
                        cq[u][jt] = lds128_dyn(qo, (u * NT8 + jt) * kQF);
                    }
                }
                float d[UB][NT8][4];
#pragma unroll
                for (int u = 0; u < UB; ++u) {
#pragma unroll
                    for (int jt = 0; jt < NT8; ++jt) {
                        if constexpr (HAS_ZP) {  // start at -zp sum_k x
                            const float zpA = u8f(zq[u][0]), zpB = u8f(zq[u][1]);
                            d[u][jt][0] = -zpA * __uint_as_float(cq[u][jt].x);
                            d[u][jt][1] = -zpA * __uint_as_float(cq[u][jt].y);
                            d[u][jt][2] = -zpB * __uint_as_float(cq[u][jt].z);
                            d[u][jt][3] = -zpB * __uint_as_float(cq[u][jt].w);
                        } else {
                            d[u][jt][0] = __uint_as_float(cq[u][jt].x);
                            d[u][jt][1] = __uint_as_float(cq[u][jt].y);
                            d[u][jt][2] = __uint_as_float(cq[u][jt].z);
                            d[u][jt][3] = __uint_as_float(cq[u][jt].w);
                        }
                    }
                    if constexpr (BITS == 4) {
                        uint32_t pa[4], pb[4];
                        U::pairs(wa[u][0], pa);
                        U::pairs(wb[u][0], pb);
#pragma unroll
                        for (int jt = 0; jt < NT8; ++jt) {
                            mma_16816(d[u][jt], pa[0], pb[0], pa[2], pb[2], xw[u][jt].x, xw[u][jt].y);  // low nibbles
                            mma_16816(d[u][jt], pa[1], pb[1], pa[3], pb[3], xw[u][jt].z, xw[u][jt].w);  // high: 16 q, x / 16
                        }
                    } else {
                        uint32_t pa0[2], pa1[2], pb0[2], pb1[2];
                        U::pairs(wa[u][0], pa0);
                        U::pairs(wa[u][1], pa1);
                        U::pairs(wb[u][0], pb0);
                        U::pairs(wb[u][1], pb1);
#pragma unroll
                        for (int jt = 0; jt < NT8; ++jt) {
                            mma_16816(d[u][jt], pa0[0], pb0[0], pa0[1], pb0[1], xw[u][jt].x, xw[u][jt].y);  // words t
                            mma_16816(d[u][jt], pa1[0], pb1[0], pa1[1], pb1[1], xw[u][jt].z, xw[u][jt].w);  // words t + 4
                        }
                    }
                }
                // y += s (sum_k x q - zp sum_k x), in units of 2^-24
#pragma unroll
                for (int u = 0; u < UB; ++u) {
                    const float scA = h2f(sc[u][0]), scB = h2f(sc[u][1]);
#pragma unroll
                    for (int jt = 0; jt < NT8; ++jt)
#pragma unroll
                        for (int e = 0; e < 4; ++e) v[jt][e] = fmaf(e < 2 ? scA : scB, d[u][jt][e], v[jt][e]);
                }
                cA += UB * kCStep;
                sA += UB * kSStep;
                zA += UB * kZStep;
                xo += UB * NT8 * kXF;
                qo += UB * NT8 * kQF;
            }
            __syncwarp();
            mbar_arrive_if(lane == 0, c.empty(s));  // this warp's reads of the slot are done
            if (++s == ring) {
                s = 0;
                par ^= 1u;
                cS = c_first;
                sS = s_first;
                zS = z_first;
            } else {
                cS += L.codes;
                sS += (uint32_t)kMtSR * L.spitch;
                zS += (uint32_t)kMtSR * L.zpitch;
            }
        }
        mt_hand_over<NT8>(c, pw, v, st, ok, lane);
    }
}

// The same consumers for one token tile at K = 4096 with x kept in registers: each
// thread holds the B fragments of its 8 blocks and their MMA starting values for
// the whole launch, so a block costs two code loads and half a scale load from
// shared memory.  Warp w takes the block pairs (2w, 2w + 1) + 32 k, k = 0 .. 3: one
// 4-byte load reads the scales of a pair, one 2-byte load its zero points.  H slots
// a stage (K halves or the whole K).
template <int BITS, bool HAS_ZP, int H>
__global__ void __launch_bounds__(kMtThreads, 1)
    decode_mt_xr_kernel(const __grid_constant__ MtMaps maps, const __grid_constant__ DecodeArgs a) {
    using U = Unpack<BITS>;
    constexpr uint32_t kDefaultZp = 1u << (BITS - 1);
    constexpr int kProducer = kMtCW, kReducer = kMtCW + 1;
    constexpr int NJ = 8, PPS = NJ / 2 / H, GP = BITS == 4 ? 2 : 1;  // blocks of a warp per stage, pairs per slot, pairs per step
    constexpr uint32_t kPair = (BITS == 4 ? 4u : 8u) * 2048u;  // codes: 32 blocks further, in a slot's box
    extern __shared__ unsigned char sm_raw[];
    const MtCtx c = mt_setup<BITS, HAS_ZP>(a, 1, true, sm_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp == kProducer) {
        if (lane == 0) mt_produce<BITS, HAS_ZP>(maps, a, c);
        return;
    }
    if (warp == kReducer) {
        mt_reduce<1>(a, c, lane);
        return;
    }
    const int K = a.K, Mt = a.Mt, ring = c.ring, r0 = c.r0, r1 = c.r1;
    const MtLayout& L = c.L;
    const uint32_t sb = c.sb;
    unsigned int* status = c.status;
    const int g = lane >> 2, t = lane & 3;
    if (r0 >= r1) {
        mbar_arrive_if(lane == 0, c.xready());
        return;
    }
    bool ok = true;

    // ---- x of the token rows: fragment j is block 2 warp + (j & 1) + 32 (j >> 1), token row g
    uint32_t xw[NJ][4];
    float sx0[NJ], sx1[NJ];  // the MMA's starting values for tokens 2t, 2t + 1 (see the other kernel)
    if (a.x_wait) pdl_wait();
    {
        constexpr uint32_t kOne = 0x00010001u, kHi = BITS == 4 ? 0x00100010u : kOne;
        constexpr float kZs = HAS_ZP ? 1.f : -(float)kDefaultZp;
        const __half2 k16 = __float2half2_rn(0.0625f);
        const __half* xr = a.X + (size_t)g * K + (size_t)(2 * warp) * 32 + (BITS == 4 ? 8 * t : 4 * t);
        uint4 v[NJ];
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
            const __half* p = xr + ((j & 1) + 32 * (j >> 1)) * 32;
            v[j] = make_uint4(0u, 0u, 0u, 0u);
            if (g < Mt) {
                if constexpr (BITS == 4) {
                    v[j] = ldg128_nc(p);  // word t: x[8t .. 8t + 7]
                } else {
                    const uint2 lo = ldg64_nc(p), hi = ldg64_nc(p + 16);  // words t, t + 4
                    v[j] = make_uint4(lo.x, lo.y, hi.x, hi.y);
                }
            }
        }
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
            uint4 o = v[j];
            if constexpr (BITS == 4) {  // (x0, x4) (x2, x6) (x1, x5)/16 (x3, x7)/16
                const uint32_t h15 = prmt(o.x, o.z, 0x7632u), h37 = prmt(o.y, o.w, 0x7632u);
                const __half2 s15 = __hmul2(*reinterpret_cast<const __half2*>(&h15), k16);
                const __half2 s37 = __hmul2(*reinterpret_cast<const __half2*>(&h37), k16);
                o = make_uint4(prmt(o.x, o.z, 0x5410u), prmt(o.y, o.w, 0x5410u),
                               *reinterpret_cast<const uint32_t*>(&s15), *reinterpret_cast<const uint32_t*>(&s37));
            }
            xw[j][0] = o.x;
            xw[j][1] = o.y;
            xw[j][2] = o.z;
            xw[j][3] = o.w;
            float d[4];
            mma_16816_z(d, kOne, kOne, kOne, kOne, o.x, o.y);
            mma_16816(d, kHi, kHi, kHi, kHi, o.z, o.w);
            sx0[j] = kZs * d[0];
            sx1[j] = kZs * d[1];
        }
    }
    mbar_arrive_if(lane == 0, c.xready());

    // ---- the stages
    // Codes of block b in the slot's box (segment [16 rows][128 B], row r + 8 1024 bytes
    // after row r): INT4 16 bytes at segment b >> 3, chunk b & 7; INT8 32 bytes at
    // segment b >> 2, chunks 2 (b & 3) and 2 (b & 3) + 1.  Block e of this warp's pair
    // (b = 2 warp + e + 32 k): this thread's word at off[e][0] (and word t + 4 at
    // off[e][1]) plus k kPair.
    const uint32_t w2 = 2u * (uint32_t)warp, gg = (uint32_t)g;
    uint32_t off[2][2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        if constexpr (BITS == 4) {
            const uint32_t ch = (w2 & 7u) + (uint32_t)e;
            off[e][0] = (w2 >> 3) * 2048u + gg * 128u + ((ch ^ gg) << 4) + 4u * (uint32_t)t;
            off[e][1] = off[e][0];
        } else {
            const uint32_t ch = 2u * (w2 & 3u) + 2u * (uint32_t)e;
            off[e][0] = (w2 >> 2) * 2048u + gg * 128u + ((ch ^ gg) << 4) + 4u * (uint32_t)t;
            off[e][1] = (w2 >> 2) * 2048u + gg * 128u + (((ch + 1u) ^ gg) << 4) + 4u * (uint32_t)t;
        }
    }
    const uint32_t s_off = gg * L.spitch + 2u * w2, z_off = gg * L.zpitch + w2;
    const uint32_t s8 = 8u * L.spitch, z8 = 8u * L.zpitch;
    // the slot cursor: index, phase, and the slot's codes, scales and zero points
    int s = 0;
    uint32_t par = 0u;
    uint32_t cS = sb, sS = sb + L.sc + s_off, zS = sb + L.zp + z_off;
    const int pw = (32 * t + g) * kPS + warp;  // this thread's partials in a buffer
    MtRows it;
    it.init(a, r0, r1);
    for (int st = 0; it.pos < r1; it.next(a), ++st) {
        float v[1][4] = {{0.f, 0.f, 0.f, 0.f}};  // rows g, g + 8 x tokens 2t, 2t + 1
#pragma unroll
        for (int h = 0; h < H; ++h) {
            // after a timeout the slot's stale bytes are read all the same (in bounds)
            // and the reducer stores nothing
            if (ok) ok = mbar_wait(c.full(s), par, status);
            const uint32_t c0 = cS + off[0][0], c1 = cS + off[1][0];
            [[maybe_unused]] const uint32_t c0h = cS + off[0][1], c1h = cS + off[1][1];
#pragma unroll
            for (int k0 = 0; k0 < PPS; k0 += GP) {
                uint32_t wa[GP][2][2], wb[GP][2][2], scA[GP], scB[GP];
                [[maybe_unused]] uint32_t zqA[GP], zqB[GP];
#pragma unroll
                for (int kk = 0; kk < GP; ++kk) {
                    const uint32_t kp = (uint32_t)(k0 + kk);
                    wa[kk][0][0] = lds32_dyn(c0, kp * kPair);
                    wb[kk][0][0] = lds32_dyn(c0, kp * kPair + 1024u);
                    wa[kk][1][0] = lds32_dyn(c1, kp * kPair);
                    wb[kk][1][0] = lds32_dyn(c1, kp * kPair + 1024u);
                    if constexpr (BITS == 8) {
                        wa[kk][0][1] = lds32_dyn(c0h, kp * kPair);
                        wb[kk][0][1] = lds32_dyn(c0h, kp * kPair + 1024u);
                        wa[kk][1][1] = lds32_dyn(c1h, kp * kPair);
                        wb[kk][1][1] = lds32_dyn(c1h, kp * kPair + 1024u);
                    }
                    scA[kk] = lds32_dyn(sS, kp * 64u);
                    scB[kk] = lds32_dyn(sS + s8, kp * 64u);
                    if constexpr (HAS_ZP) {
                        zqA[kk] = lds16_dyn(zS, kp * 32u);
                        zqB[kk] = lds16_dyn(zS + z8, kp * 32u);
                    }
                }
                float d[GP][2][4];
#pragma unroll
                for (int kk = 0; kk < GP; ++kk)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int j = 2 * (h * PPS + k0 + kk) + e;
                        if constexpr (HAS_ZP) {  // start at -zp sum_k x
                            const float zA = u8f((zqA[kk] >> (8 * e)) & 0xFFu), zB = u8f((zqB[kk] >> (8 * e)) & 0xFFu);
                            d[kk][e][0] = -zA * sx0[j];
                            d[kk][e][1] = -zA * sx1[j];
                            d[kk][e][2] = -zB * sx0[j];
                            d[kk][e][3] = -zB * sx1[j];
                        } else {  // copied here, not once outside the loop (that would hold 32 more registers)
                            d[kk][e][0] = fmov_here(sx0[j]);
                            d[kk][e][1] = fmov_here(sx1[j]);
                            d[kk][e][2] = fmov_here(sx0[j]);
                            d[kk][e][3] = fmov_here(sx1[j]);
                        }
                        if constexpr (BITS == 4) {
                            uint32_t pa[4], pb[4];
                            U::pairs(wa[kk][e][0], pa);
                            U::pairs(wb[kk][e][0], pb);
                            mma_16816(d[kk][e], pa[0], pb[0], pa[2], pb[2], xw[j][0], xw[j][1]);  // low nibbles
                            mma_16816(d[kk][e], pa[1], pb[1], pa[3], pb[3], xw[j][2], xw[j][3]);  // high: 16 q, x / 16
                        } else {
                            uint32_t pa0[2], pa1[2], pb0[2], pb1[2];
                            U::pairs(wa[kk][e][0], pa0);
                            U::pairs(wa[kk][e][1], pa1);
                            U::pairs(wb[kk][e][0], pb0);
                            U::pairs(wb[kk][e][1], pb1);
                            mma_16816(d[kk][e], pa0[0], pb0[0], pa0[1], pb0[1], xw[j][0], xw[j][1]);  // words t
                            mma_16816(d[kk][e], pa1[0], pb1[0], pa1[1], pb1[1], xw[j][2], xw[j][3]);  // words t + 4
                        }
                    }
                // y += s (sum_k x q - zp sum_k x), in units of 2^-24
#pragma unroll
                for (int kk = 0; kk < GP; ++kk) {
                    const float2 sa = __half22float2(*reinterpret_cast<const __half2*>(&scA[kk]));
                    const float2 sbb = __half22float2(*reinterpret_cast<const __half2*>(&scB[kk]));
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const float ssA = e ? sa.y : sa.x, ssB = e ? sbb.y : sbb.x;
                        v[0][0] = fmaf(ssA, d[kk][e][0], v[0][0]);
                        v[0][1] = fmaf(ssA, d[kk][e][1], v[0][1]);
                        v[0][2] = fmaf(ssB, d[kk][e][2], v[0][2]);
                        v[0][3] = fmaf(ssB, d[kk][e][3], v[0][3]);
                    }
                }
            }
            __syncwarp();
            mbar_arrive_if(lane == 0, c.empty(s));  // this warp's reads of the slot are done
            if (++s == ring) {
                s = 0;
                par ^= 1u;
                cS = sb;
                sS = sb + L.sc + s_off;
                zS = sb + L.zp + z_off;
            } else {
                cS += L.codes;
                sS += (uint32_t)kMtSR * L.spitch;
                zS += (uint32_t)kMtSR * L.zpitch;
            }
        }
        mt_hand_over<1>(c, pw, v, st, ok, lane);
    }
}

template <int BITS, bool HAS_ZP, int NT8, int UB>
cudaError_t mt_launch_one(const MtMaps& maps, const DecodeArgs& a, int ctas, size_t smem, bool pdl, cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ctas);
    cfg.blockDim = dim3(kMtThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    int na = 0;
    if (pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, decode_mt_kernel<BITS, HAS_ZP, NT8, UB>, maps, a);
}

// The kernels: bits x zero points x token tiles x blocks per loop step of a warp
// (4, 2, 1 for one token tile; 2, 1 for two).
template <int BITS, bool HAS_ZP>
cudaError_t mt_launch_bz(int nt8, int ub, const MtMaps& maps, const DecodeArgs& a, int ctas, size_t smem, bool pdl,
                         cudaStream_t st) {
    if (nt8 == 1) {
        if (ub == 4) return mt_launch_one<BITS, HAS_ZP, 1, 4>(maps, a, ctas, smem, pdl, st);
        if (ub == 2) return mt_launch_one<BITS, HAS_ZP, 1, 2>(maps, a, ctas, smem, pdl, st);
        return mt_launch_one<BITS, HAS_ZP, 1, 1>(maps, a, ctas, smem, pdl, st);
    }
    if (ub == 2) return mt_launch_one<BITS, HAS_ZP, 2, 2>(maps, a, ctas, smem, pdl, st);
    return mt_launch_one<BITS, HAS_ZP, 2, 1>(maps, a, ctas, smem, pdl, st);
}

template <int BITS, bool HAS_ZP, int H>
cudaError_t mt_launch_xr(const MtMaps& maps, const DecodeArgs& a, int ctas, size_t smem, bool pdl, cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ctas);
    cfg.blockDim = dim3(kMtThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    int na = 0;
    if (pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, decode_mt_xr_kernel<BITS, HAS_ZP, H>, maps, a);
}

template <int BITS, bool HAS_ZP, int NT8, int UB>
cudaError_t mt_set_one() {
    return cudaFuncSetAttribute(decode_mt_kernel<BITS, HAS_ZP, NT8, UB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)kMtSmem);
}

template <int BITS, bool HAS_ZP>
cudaError_t mt_set_smem() {
    cudaError_t e = mt_set_one<BITS, HAS_ZP, 1, 4>();
    if (e == cudaSuccess) e = mt_set_one<BITS, HAS_ZP, 1, 2>();
    if (e == cudaSuccess) e = mt_set_one<BITS, HAS_ZP, 1, 1>();
    if (e == cudaSuccess) e = mt_set_one<BITS, HAS_ZP, 2, 2>();
    if (e == cudaSuccess) e = mt_set_one<BITS, HAS_ZP, 2, 1>();
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(decode_mt_xr_kernel<BITS, HAS_ZP, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kMtSmem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(decode_mt_xr_kernel<BITS, HAS_ZP, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kMtSmem);
    return e;
}

int mt_ctas(int N, int sms) {
    int C = (N + 15) / 16;
    const int s = sms > 0 ? sms : 1;
    if (C > s) C = s;
    return C < 1 ? 1 : C;
}

int mt_nt8(int Mt) { return Mt <= 8 ? 1 : 2; }

// Blocks per loop step of a warp: the most (up to 4 for one token tile, 2 for two)
// that divide the warp's blocks in a slot.
int mt_ub(int nt8, int njp) {
    const int top = nt8 == 1 ? 4 : 2;
    for (int u = top; u > 1; u /= 2)
        if (njp % u == 0) return u;
    return 1;
}

// Slots per stage (K parts) and ring depth: among the plans whose slots give the
// warps the most blocks per loop step, the one that keeps the most code bytes in
// flight while the slowest warp works on one slot, (ring - 1) x slot; fewer parts on
// a tie.
struct MtGeo {
    int parts, ring, ub;
    uint32_t smem;
};

// x in registers: one token tile at K = 4096, one or two slots a stage.
bool mt_xreg(int K, int Mt) { return K == 4096 && mt_nt8(Mt) == 1; }

MtGeo mt_geo(int bits, int K, int Mt, bool zp) {
    const int nt8 = mt_nt8(Mt), nj = K / 32 / kMtCW;
    const bool xreg = mt_xreg(K, Mt);
    MtGeo best = {0, 0, 0, 0u};
    uint64_t best_bytes = 0;
    for (int parts = 1; parts <= (xreg ? 2 : 4); parts *= 2) {
        if (nj % parts != 0) continue;
        const int ub = mt_ub(nt8, nj / parts);
        if (best.parts && ub < best.ub) continue;
        for (int r = 2; r <= kMtMaxRing; ++r) {
            const MtLayout L = mt_layout(r, bits, K, nt8, parts, zp, xreg);
            if (L.total + 1024u > kMtSmem) break;
            const uint64_t bytes = (uint64_t)(r - 1) * L.codes;
            if (ub > best.ub || bytes > best_bytes) {
                best_bytes = bytes;
                best = {parts, r, ub, L.total + 1024u};
            }
        }
    }
    return best;
}

}  // namespace

bool decode_mt_supported(int bits, int64_t Mt, int K, bool lora) {
    (void)lora;  // an FP16 rank-32 adapter: T from the LoRA down kernel, T B^T by the reducer warp
    if ((bits != 4 && bits != 8) || Mt < 2 || Mt > 16) return false;
    if (K <= 0 || K % 512 != 0 || K > 7680) return false;  // TMA boxes of scales / zero points, swizzled code rows
    return mt_geo(bits, K, (int)Mt, true).parts > 0;        // with zero points: the larger plan
}

void decode_mt_geometry(int N, int K, int bits, int Mt, bool zp, int sms, int* ctas, int* parts, int* ring,
                        size_t* smem) {
    const MtGeo G = mt_geo(bits, K, Mt, zp);
    *ctas = mt_ctas(N, sms);
    *parts = G.parts;
    *ring = G.ring;
    *smem = G.smem;
}

cudaError_t decode_mt_prepare() {
    cudaError_t e = tensor_map_prepare();
    if (e == cudaSuccess) e = mt_set_smem<4, false>();
    if (e == cudaSuccess) e = mt_set_smem<4, true>();
    if (e == cudaSuccess) e = mt_set_smem<8, false>();
    if (e == cudaSuccess) e = mt_set_smem<8, true>();
    return e;
}

cudaError_t decode_mt_launch(const DecodeArgs& a_in, int sms, bool pdl, cudaStream_t st) {
    DecodeArgs a = a_in;
    const int bits = a.bits, K = a.K, nblk = K / 32;
    const bool zp = a.seg[0].Z != nullptr;
    if (!decode_mt_supported(bits, a.Mt, K, a.B != nullptr)) return cudaErrorNotSupported;
    const MtGeo G = mt_geo(bits, K, a.Mt, zp);
    const int C = mt_ctas(a.NR, sms);
    a.SR = kMtSR;
    a.ring = G.ring;
    a.kparts = G.parts;
    const int nbp = nblk / G.parts;
    const DecPitch P = dec_pitch(nbp);
    const uint64_t rowbytes = (uint64_t)K * bits / 8;
    MtMaps maps;
    memset(&maps, 0, sizeof(maps));
    for (int i = 0; i < a.nseg; ++i) {
        cudaError_t e = encode_codes_sw128(&maps.c[i], a.seg[i].Wq, rowbytes, (uint64_t)a.seg[i].N, (uint32_t)kMtSR,
                                           (uint32_t)(rowbytes / 128 / G.parts));
        if (e == cudaSuccess)
            e = encode_2d(&maps.s[i], a.seg[i].S, 2, (uint64_t)nblk, (uint64_t)a.seg[i].N, (uint64_t)nblk * 2,
                          P.spitch / 2u, (uint32_t)kMtSR, false);
        if (e == cudaSuccess && zp)
            e = encode_2d(&maps.z[i], a.seg[i].Z, 1, (uint64_t)nblk, (uint64_t)a.seg[i].N, (uint64_t)nblk, P.zpitch,
                          (uint32_t)kMtSR, false);
        if (e != cudaSuccess) return e;
    }
    const int nt8 = mt_nt8(a.Mt);
    const size_t smem = G.smem;
    if (mt_xreg(K, a.Mt)) {
        if (bits == 4) {
            if (zp) return G.parts == 2 ? mt_launch_xr<4, true, 2>(maps, a, C, smem, pdl, st) : mt_launch_xr<4, true, 1>(maps, a, C, smem, pdl, st);
            return G.parts == 2 ? mt_launch_xr<4, false, 2>(maps, a, C, smem, pdl, st) : mt_launch_xr<4, false, 1>(maps, a, C, smem, pdl, st);
        }
        if (zp) return G.parts == 2 ? mt_launch_xr<8, true, 2>(maps, a, C, smem, pdl, st) : mt_launch_xr<8, true, 1>(maps, a, C, smem, pdl, st);
        return G.parts == 2 ? mt_launch_xr<8, false, 2>(maps, a, C, smem, pdl, st) : mt_launch_xr<8, false, 1>(maps, a, C, smem, pdl, st);
    }
    if (bits == 4)
        return zp ? mt_launch_bz<4, true>(nt8, G.ub, maps, a, C, smem, pdl, st)
                  : mt_launch_bz<4, false>(nt8, G.ub, maps, a, C, smem, pdl, st);
    return zp ? mt_launch_bz<8, true>(nt8, G.ub, maps, a, C, smem, pdl, st)
              : mt_launch_bz<8, false>(nt8, G.ub, maps, a, C, smem, pdl, st);
}

}  // namespace mnb
