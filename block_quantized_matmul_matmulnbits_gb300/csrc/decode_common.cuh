// decode_common.cuh -- pieces shared by the two decode kernels that stream a
// CTA's share of weight rows through shared memory (decode.cu: one token row;
// decode_mt.cu: several token rows).
#pragma once

#include <cuda.h>

#include "common.cuh"
#include "mnb_internal.h"

namespace mnb {
namespace dec {

constexpr float kUnit = 1.0f / 16777216.f;  // a code q reaches the MMA as q * 2^-24

// Shared-memory loads at a 32-bit shared address plus an immediate offset.
// Volatile: they stay after the barrier waits before them in program order.
template <int OFF = 0>
__device__ __forceinline__ uint4 lds128_s(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4+%5];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(a), "n"(OFF));
    return v;
}
__device__ __forceinline__ uint32_t lds_u16_s(uint32_t a) {
    uint16_t v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ uint32_t lds_u8_s(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.u8 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ float lds_f32_s(uint32_t a) {
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(a));
    return v;
}

__host__ __device__ inline uint32_t al128(uint32_t x) { return (x + 127u) & ~127u; }

// How a stage's scales and zero points land in shared memory: rows `spitch` /
// `zpitch` bytes apart.  With TMA boxes the rows carry 16 bytes of padding (the
// box is wider than the tensor, the extra columns read as zero); with bulk
// copies they are dense, starting at a 16-byte aligned superset.
struct DecPitch {
    int tma_s, tma_z;      // copied as 2-D TMA boxes (else 1-D bulk copies)
    uint32_t spitch, zpitch;
};

__host__ __device__ inline DecPitch dec_pitch(int nblk) {
    DecPitch p;
    p.tma_s = nblk % 8 == 0 && nblk + 8 <= 256;    // 16-byte global rows, box within 256 elements
    p.tma_z = nblk % 16 == 0 && nblk + 16 <= 256;
    p.spitch = p.tma_s ? (uint32_t)(nblk + 8) * 2u : (uint32_t)nblk * 2u;
    p.zpitch = p.tma_z ? (uint32_t)(nblk + 16) : (uint32_t)nblk;
    return p;
}

// Codes of a weight word as the subnormal FP16 pairs the MMA takes.
// INT4 word = codes c0..c7 (c0 in bits 0..3): lo0 = (c0, c4), hi0 = 16 (c1, c5),
// lo1 = (c2, c6), hi1 = 16 (c3, c7), each times 2^-24.
// INT8 word = codes c0..c3: p0 = (c0, c1), p1 = (c2, c3), times 2^-24.
template <int BITS>
struct Unpack;

template <>
struct Unpack<4> {
    static constexpr int kWordsPerBlock = 4;  // 16 bytes a block and row
    static constexpr float kHiWeight = 1.f / 16.f;  // class 1 codes sit 4 bits higher: they read as 16 q
    __device__ __forceinline__ static void pairs(uint32_t w, uint32_t a[4]) {
        const uint32_t w8 = w >> 8;
        a[0] = w & 0x000F000Fu;
        a[1] = w & 0x00F000F0u;
        a[2] = w8 & 0x000F000Fu;
        a[3] = w8 & 0x00F000F0u;
    }
};

template <>
struct Unpack<8> {
    static constexpr int kWordsPerBlock = 8;
    static constexpr float kHiWeight = 1.f;
    __device__ __forceinline__ static void pairs(uint32_t w, uint32_t a[2]) {
        a[0] = prmt(w, 0u, 0x4140u);
        a[1] = prmt(w, 0u, 0x4342u);
    }
};

// A load kept in program order with the other volatile asm (the prefetch before
// griddepcontrol.wait stays before it).
__device__ __forceinline__ uint32_t ldg_nc_u32(const void* p) {
    uint32_t v;
    asm volatile("ld.global.nc.b32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ float h2f(uint32_t bits16) { return __half2float(__ushort_as_half((unsigned short)bits16)); }
// A byte as an exact float, without the conversion unit: 2^23 + z read as binary32, minus 2^23.
__device__ __forceinline__ float u8f(uint32_t z) { return __uint_as_float(0x4B000000u | z) - 8388608.f; }

// TMA descriptors of the projections' scales and zero points (rows padded in shared memory).
struct DecMaps {
    CUtensorMap s[kMaxSeg];
    CUtensorMap z[kMaxSeg];
};

// The CTA's rows as a sequence of stages: at most SR rows, never across two
// projections (each stage is contiguous in one projection's arrays).  Producer
// and consumers step through the same sequence.
struct StageIt {
    int pos, seg;  // first row-space row of the stage, its projection
    int ra, rs;    // its first row inside the projection, rows
    __device__ __forceinline__ void settle(const DecodeArgs& a, int r1, int SR) {
        while (seg + 1 < a.nseg && pos >= a.seg[seg + 1].row0) ++seg;
        const int send = a.seg[seg].row0 + a.seg[seg].N;
        rs = min(min(SR, r1 - pos), send - pos);
        ra = pos - a.seg[seg].row0;
    }
    __device__ __forceinline__ void next(const DecodeArgs& a, int r1, int SR) {
        pos += rs;
        if (pos < r1) settle(a, r1, SR);
    }
};

}  // namespace dec
}  // namespace mnb
