// common.cuh -- device helpers shared by the libmnb kernels (sm_103a).
//
// The dequantization helpers implement w = (q - zp) * scale with exactly one
// rounding to FP16, the weight map of DequantizeLinear in "Fuse
// DQ->MatMulNBits for shared initializers and skip outer-scope weights"
// (onnxruntime PR 33800, Description).  How:
//   * a code q (< 2^bits) is placed in the low fraction bits of the FP16
//     value 1024 (bits 0x6400), giving exactly 1024 + q (or 1024 + 16 q when
//     the code sits in the upper nibble of a byte);
//   * subtracting 1024 + zp (or, for the x16 form, multiplying by 1/16 and
//     adding -(64 + zp) in one fused step) yields q - zp exactly: every
//     operand and result is an integer below 2048 in magnitude;
//   * one multiply by the FP16 scale rounds once, to nearest even.
// All half2 arithmetic is issued with explicit .rn PTX so that no contraction
// can merge the exact subtraction into the rounded multiply.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "mnb_internal.h"

namespace mnb {


// ---------------------------------------------------------------- bit tricks

__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t mask, uint32_t magic) {
    uint32_t d;  // (a & mask) | magic
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(mask), "r"(magic));
    return d;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

__device__ __forceinline__ uint32_t hsub2_rn(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ uint32_t hmul2_rn(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ uint32_t hfma2_rn(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

constexpr uint32_t kMagic1024x2 = 0x64006400u;  // half2(1024, 1024)
constexpr uint32_t kHalf960x2 = 0x63806380u;    // half2(960, 960)
constexpr uint32_t kSixteenthX2 = 0x2C002C00u;  // half2(1/16, 1/16)
constexpr uint32_t kOneSixteenth = 0x2C003C00u; // half2(lo = 1, hi = 1/16)

// Per-block constants of the dequant: c0 = half2(1024 + zp), c1 = half2(-(64 + zp)),
// s2 = half2(scale).  zp < 1024, so 1024 + zp is the bit pattern 0x6400 | zp.
struct DqConst {
    uint32_t c0, c1, s2;
};

__device__ __forceinline__ DqConst dq_const(uint32_t zp, uint16_t scale_bits) {
    DqConst c;
    c.c0 = kMagic1024x2 | (zp * 0x00010001u);
    c.c1 = hsub2_rn(kHalf960x2, c.c0);  // 960 - (1024 + zp), exact
    c.s2 = (uint32_t)scale_bits * 0x00010001u;
    return c;
}

// INT4, pair-interleaved order (decode kernel).  Word w holds codes k0..k7
// (k0 in bits 0..3).  Output half2s: d0 = (w_k0, w_k4), d1 = (w_k1, w_k5),
// d2 = (w_k2, w_k6), d3 = (w_k3, w_k7).
__device__ __forceinline__ void dq_int4_interleaved(uint32_t w, const DqConst& c, uint32_t d[4]) {
    const uint32_t w8 = w >> 8;
    const uint32_t h0 = lop3_and_or(w, 0x000F000Fu, kMagic1024x2);   // 1024 + (k0, k4)
    const uint32_t h1 = lop3_and_or(w, 0x00F000F0u, kMagic1024x2);   // 1024 + 16 (k1, k5)
    const uint32_t h2 = lop3_and_or(w8, 0x000F000Fu, kMagic1024x2);  // 1024 + (k2, k6)
    const uint32_t h3 = lop3_and_or(w8, 0x00F000F0u, kMagic1024x2);  // 1024 + 16 (k3, k7)
    d[0] = hmul2_rn(hsub2_rn(h0, c.c0), c.s2);
    d[1] = hmul2_rn(hfma2_rn(h1, kSixteenthX2, c.c1), c.s2);
    d[2] = hmul2_rn(hsub2_rn(h2, c.c0), c.s2);
    d[3] = hmul2_rn(hfma2_rn(h3, kSixteenthX2, c.c1), c.s2);
}

// INT4, natural order (prefill kernel, K-major FP16 operand).  Output half2s:
// d[j] = (w_k{2j}, w_k{2j+1}).  Byte j is copied to both halves, its low
// nibble read as 1024 + q in the low half and its high nibble as 1024 + 16 q
// in the high half; one fused step with per-half constants removes both.
__device__ __forceinline__ void dq_int4_natural(uint32_t w, const DqConst& c, uint32_t d[4]) {
    // per-half offset (lo: -(1024 + zp), hi: -(64 + zp))
    const uint32_t off = prmt(c.c0 ^ 0x80008000u, c.c1, 0x7610u);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t t = prmt(w, 0u, 0x4040u | (uint32_t)j | ((uint32_t)j << 8));
        const uint32_t h = lop3_and_or(t, 0x00F0000Fu, kMagic1024x2);
        d[j] = hmul2_rn(hfma2_rn(h, kOneSixteenth, off), c.s2);
    }
}

// INT8, natural order.  Word w holds codes k0..k3.  d0 = (w_k0, w_k1), d1 = (w_k2, w_k3).
__device__ __forceinline__ void dq_int8_natural(uint32_t w, const DqConst& c, uint32_t d[2]) {
    const uint32_t h01 = prmt(w, 0x64646464u, 0x4140u);  // bytes [q0, 0x64, q1, 0x64]
    const uint32_t h23 = prmt(w, 0x64646464u, 0x4342u);  // bytes [q2, 0x64, q3, 0x64]
    d[0] = hmul2_rn(hsub2_rn(h01, c.c0), c.s2);
    d[1] = hmul2_rn(hsub2_rn(h23, c.c0), c.s2);
}

// INT2: four codes per byte, code 4b + i in bits 2i..2i+1 of byte b.  A code
// masked in place at bit 2i of a half's fraction reads as 1024 + 4^i q; one
// fused multiply by 4^-i (exact: a power of two) and add of -(1024 4^-i + zp)
// leaves q - zp exactly (every value an integer below 2048 in magnitude), and
// the multiply by the scale rounds once.
__host__ __device__ constexpr uint32_t int2_mul(int i) {  // half2(4^-i): 1, 1/4, 1/16, 1/64
    return i == 0 ? 0x3C003C00u : i == 1 ? 0x34003400u : i == 2 ? 0x2C002C00u : 0x24002400u;
}
__host__ __device__ constexpr uint32_t int2_base(int i) {  // half2(1024 - 1024 4^-i): 0, 768, 960, 1008
    return i == 0 ? 0x00000000u : i == 1 ? 0x62006200u : i == 2 ? 0x63806380u : 0x63E063E0u;
}

struct Dq2Const {
    uint32_t off[4];  // half2(-(1024 4^-i + zp)), i = 0..3
    uint32_t s2;
};

__device__ __forceinline__ Dq2Const dq2_const(uint32_t zp, uint16_t scale_bits) {
    Dq2Const c;
    const uint32_t z = kMagic1024x2 | (zp * 0x00010001u);  // half2(1024 + zp)
#pragma unroll
    for (int i = 0; i < 4; ++i) c.off[i] = hsub2_rn(int2_base(i), z);
    c.s2 = (uint32_t)scale_bits * 0x00010001u;
    return c;
}

// Pair-interleaved order (decode kernel).  Word w holds codes k0..k15.  Output
// half2s d[j] = (w_kj, w_k{j+8}), j = 0..7: code j sits at bit 2j and code
// j + 8 at bit 16 + 2j, so one mask serves both halves.
__device__ __forceinline__ void dq_int2_interleaved(uint32_t w, const Dq2Const& c, uint32_t d[8]) {
    const uint32_t w8 = w >> 8;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int i = j & 3;
        const uint32_t h = lop3_and_or(j < 4 ? w : w8, 0x00030003u << (2 * i), kMagic1024x2);
        d[j] = hmul2_rn(hfma2_rn(h, int2_mul(i), c.off[i]), c.s2);
    }
}

// Natural order (prefill kernel, K-major FP16 operand).  d[j] = (w_k{2j},
// w_k{2j+1}), j = 0..7.  Byte b is copied to both halves; the low half keeps
// code 4b (bit 0) or 4b + 2 (bit 4), the high half code 4b + 1 (bit 2) or
// 4b + 3 (bit 6), each removed with its own power of two.
__device__ __forceinline__ void dq_int2_natural(uint32_t w, const Dq2Const& c, uint32_t d[8]) {
    const uint32_t m01 = prmt(int2_mul(0), int2_mul(1), 0x7610u);  // (lo 1, hi 1/4)
    const uint32_t m23 = prmt(int2_mul(2), int2_mul(3), 0x7610u);  // (lo 1/16, hi 1/64)
    const uint32_t o01 = prmt(c.off[0], c.off[1], 0x7610u);
    const uint32_t o23 = prmt(c.off[2], c.off[3], 0x7610u);
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        const uint32_t t = prmt(w, 0u, 0x4040u | (uint32_t)b | ((uint32_t)b << 8));
        const uint32_t h01 = lop3_and_or(t, 0x000C0003u, kMagic1024x2);
        const uint32_t h23 = lop3_and_or(t, 0x00C00030u, kMagic1024x2);
        d[2 * b] = hmul2_rn(hfma2_rn(h01, m01, o01), c.s2);
        d[2 * b + 1] = hmul2_rn(hfma2_rn(h23, m23, o23), c.s2);
    }
}

// ---------------------------------------------------------------- tensor ops

// D = A(16x16, row) * B(16x8, col) + C, FP16 inputs, FP32 accumulate.  Not
// volatile: only its data dependences order it, so the compiler may overlap
// independent MMAs with the loads and unpacking around them.
__device__ __forceinline__ void mma_16816(float d[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// The same with C = 0: D = A * B (no accumulator input to clear first).
__device__ __forceinline__ void mma_16816_z(float d[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                            uint32_t b0, uint32_t b1) {
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%10, %10, %10, %10};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.f));
}

// D = A(16x32 u8, row) * B(32x8 s8, col), exact int32, C = 0: the integer dot
// of the int8-activation path (weight codes unsigned, activation codes signed).
__device__ __forceinline__ void mma_16832_u8s8(int d[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k32.row.col.s32.u8.s8.s32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%10, %10, %10, %10};"
        : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "r"(0));
}

// ---------------------------------------------------------------- int8 activations

// One block of 32 activations to int8, every step in binary32 with one
// rounding to nearest: amax = max |x|; amax == 0 gives codes 0 and scale 0;
// else inv = 127 / amax, code = clamp(rint(x * inv), -127, 127) (ties to
// even), scale = amax / 127.  `x` is 16-byte aligned; `q` receives the codes
// in K order, the return value is the scale, `sum` the sum of the codes.
__device__ __forceinline__ float quantize_block32(const __half* x, int q[32], int& sum) {
    float v[32];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint4 u = __ldg(reinterpret_cast<const uint4*>(x) + j);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
            v[8 * j + 2 * i] = f.x;
            v[8 * j + 2 * i + 1] = f.y;
        }
    }
    float amax = 0.f;
#pragma unroll
    for (int j = 0; j < 32; ++j) amax = fmaxf(amax, fabsf(v[j]));
    sum = 0;
    if (amax == 0.f) {
#pragma unroll
        for (int j = 0; j < 32; ++j) q[j] = 0;
        return 0.f;
    }
    const float inv = __fdiv_rn(127.f, amax);
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        const int c = __float2int_rn(__fmul_rn(v[j], inv));
        q[j] = c > 127 ? 127 : (c < -127 ? -127 : c);
        sum += q[j];
    }
    return __fdiv_rn(amax, 127.f);
}

// ---------------------------------------------------------------- launch ordering

// Programmatic dependent launch: allow the next kernel on the stream to start.
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Wait until the preceding kernel on the stream has completed and its writes
// are visible (returns at once when this grid was not launched dependently).
__device__ __forceinline__ void pdl_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier / TMA

// Bounded waits give up after this many SM cycles (~2 s at 2 GHz).
constexpr long long kWaitCycles = 4000000000LL;

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

// One bounded probe of a phase: the thread may be suspended in hardware for up
// to ~50 us waiting for it (suspend-time hint), so waiting warps do not spin.
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, 50000;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase of `parity` to complete.  Returns false (and
// records a timeout) when the limit passes, or -- when `abortable` -- as soon
// as another role of the kernel has already given up.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, unsigned int* status,
                                          bool abortable = true, long long limit = kWaitCycles) {
    if (mbar_try(bar, parity)) return true;
    const long long t0 = clock64();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try(bar, parity)) return true;
        if ((it & 7u) == 0) {
            if (abortable && (*reinterpret_cast<volatile unsigned int*>(status) & kStatusTimeout)) return false;
            if (clock64() - t0 > limit) {
                atomicOr(status, kStatusTimeout);
                return false;
            }
        }
    }
}

// mbar_wait for a role whose wait is long and not on the critical path: between
// probes the warp sleeps about `ns` nanoseconds, leaving its issue slots to the
// warps that are working.
__device__ __forceinline__ bool mbar_wait_sleep(uint32_t bar, uint32_t parity, unsigned int* status, uint32_t ns) {
    if (mbar_try(bar, parity)) return true;
    const long long t0 = clock64();
    for (;;) {
        __nanosleep(ns);
        if (mbar_try(bar, parity)) return true;
        if (*reinterpret_cast<volatile unsigned int*>(status) & kStatusTimeout) return false;
        if (clock64() - t0 > kWaitCycles) {
            atomicOr(status, kStatusTimeout);
            return false;
        }
    }
}

// Bring `bytes` (a multiple of 16, from a 16-byte aligned address) into L2 without
// waiting: later copies of the range then find it there.
__device__ __forceinline__ void prefetch_l2_bulk(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(
            dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
        : "memory");
}

// 1-D bulk copy global -> shared (16-byte aligned addresses, size a multiple of 16).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

// ---------------------------------------------------------------- thread-block clusters

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// A float in the shared memory of CTA `rank` of the cluster, at the address
// `local_addr` has in this CTA.  Volatile keeps it after the cluster barrier
// (also volatile); having no memory clobber lets several such loads be issued
// back to back.
__device__ __forceinline__ float ld_peer_f32(uint32_t local_addr, uint32_t rank) {
    uint32_t remote;
    float v;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local_addr), "r"(rank));
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote));
    return v;
}

__device__ __forceinline__ void named_barrier_sync(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

}  // namespace mnb
