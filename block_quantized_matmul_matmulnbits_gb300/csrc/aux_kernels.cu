// aux_kernels.cu -- the two small kernels around the matmuls.
//
//  * fill_zero: K == 0 leaves every sum empty, so the output keeps its logical
//    shape and holds zeros -- the empty packed weight rule of "[WebGPU] Fuse
//    rank-32 quantized LoRA with MatMulNBits" (onnxruntime PR 33370, commit
//    message on empty packed weights: the WebGPU side records a fill dispatch
//    so that graph replay rewrites the output).
//  * lora_up: an empty packed weight with an adapter leaves only the adapter
//    term, Y = T * Bt^T (+ bias), on the CUDA cores.
//  * wait_check: the kernels' bounded wait, run out on purpose on a barrier
//    nothing arrives on, so the timeout path can be checked without a fault.
//  * quantize_x: the int8-activation quantization of X on its own (the device
//    function the int8-activation decode path stages X with), for checks.
//  * dequant: the dequantization step on its own, W16 = fp16((q - zp) * scale),
//    the DequantizeLinear weight map of "Fuse DQ->MatMulNBits for shared
//    initializers and skip outer-scope weights" (onnxruntime PR 33800,
//    Description).  It runs the exact device helpers of the matmul kernels
//    (variant 0: natural order, variant 1: the decode kernel's pair-interleaved
//    INT4 / INT2 order, un-permuted on store) so their bits can be checked one
//    by one.
#include "common.cuh"
#include "mnb_internal.h"

namespace mnb {

namespace {

__global__ void fill_zero_kernel(uint4* __restrict__ y16, size_t n16, __half* __restrict__ tail, size_t ntail) {
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += stride) y16[i] = make_uint4(0, 0, 0, 0);
    if (blockIdx.x == 0)
        for (size_t i = threadIdx.x; i < ntail; i += blockDim.x) tail[i] = __float2half_rn(0.f);
}

// The kernels' bounded wait on a phase that nothing completes: no thread ever
// arrives on the barrier, so the wait gives up after `limit` cycles, records
// the timeout in the status word and the kernel returns normally.
__global__ void wait_check_kernel(unsigned int* status, long long limit) {
    __shared__ __align__(8) unsigned long long bar;
    const uint32_t b = smem_u32(&bar);
    if (threadIdx.x == 0) {
        mbar_init(b, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (threadIdx.x == 0) mbar_wait(b, 0u, status, false, limit);
}

// One thread per (row, block of 32): codes in K order and the block scale.
__global__ void quantize_x_kernel(const __half* __restrict__ X, int Mt, int K, int8_t* __restrict__ Xq,
                                  float* __restrict__ Xs) {
    const int nblk = K / 32;
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (long long)Mt * nblk) return;
    const int m = (int)(i / nblk), b = (int)(i % nblk);
    int q[32], sum;
    Xs[i] = quantize_block32(X + (size_t)m * K + b * 32, q, sum);
    uint32_t w[8];
#pragma unroll
    for (int j = 0; j < 8; ++j)
        w[j] = ((uint32_t)q[4 * j] & 0xFFu) | (((uint32_t)q[4 * j + 1] & 0xFFu) << 8) |
               (((uint32_t)q[4 * j + 2] & 0xFFu) << 16) | (((uint32_t)q[4 * j + 3] & 0xFFu) << 24);
    uint4* dst = reinterpret_cast<uint4*>(Xq + (size_t)m * K + b * 32);
    dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
    dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
}

template <int BITS>
__global__ void dequant_kernel(const uint8_t* __restrict__ Wq, const __half* __restrict__ S,
                               const uint8_t* __restrict__ Z, int N, int K, __half* __restrict__ W16,
                               int variant) {
    const int rowbytes = K * BITS / 8;
    const int chunks = rowbytes / 16;  // 16 packed bytes per thread
    const long long total = (long long)N * chunks;
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= total) return;
    const int n = (int)(i / chunks), c = (int)(i % chunks);
    const int nblk = K / 32;
    const int blk = c * 16 / (32 * BITS / 8);
    const uint4 v = *reinterpret_cast<const uint4*>(Wq + (size_t)n * rowbytes + (size_t)c * 16);
    const uint16_t sbits = reinterpret_cast<const uint16_t*>(S)[(size_t)n * nblk + blk];
    const uint32_t zp = Z ? Z[(size_t)n * nblk + blk] : (1u << (BITS - 1));
    const DqConst dc = dq_const(zp, sbits);
    const uint32_t words[4] = {v.x, v.y, v.z, v.w};
    const int k0 = c * 16 * 8 / BITS;
    uint32_t out[16];  // up to 32 halfs as half2 words
    if constexpr (BITS == 2) {  // 64 codes: words 0, 1 are block blk, words 2, 3 block blk + 1
        uint32_t o2[32];
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            const int b = blk + (w >> 1);
            const uint16_t sb2 = reinterpret_cast<const uint16_t*>(S)[(size_t)n * nblk + b];
            const uint32_t z2 = Z ? Z[(size_t)n * nblk + b] : 2u;
            const Dq2Const c2 = dq2_const(z2, sb2);
            uint32_t d[8];
            if (variant == 0) {
                dq_int2_natural(words[w], c2, d);
#pragma unroll
                for (int j = 0; j < 8; ++j) o2[8 * w + j] = d[j];
            } else {
                dq_int2_interleaved(words[w], c2, d);  // d[j] = (k_j, k_{j+8})
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    o2[8 * w + i] = prmt(d[2 * i], d[2 * i + 1], 0x5410u);      // (k_{2i}, k_{2i+1})
                    o2[8 * w + 4 + i] = prmt(d[2 * i], d[2 * i + 1], 0x7632u);  // (k_{2i+8}, k_{2i+9})
                }
            }
        }
        uint4* dst = reinterpret_cast<uint4*>(W16 + (size_t)n * K + k0);
#pragma unroll
        for (int q = 0; q < 8; ++q) dst[q] = make_uint4(o2[4 * q], o2[4 * q + 1], o2[4 * q + 2], o2[4 * q + 3]);
    } else if constexpr (BITS == 4) {
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            uint32_t d[4];
            if (variant == 0) {
                dq_int4_natural(words[w], dc, d);
                out[4 * w + 0] = d[0];
                out[4 * w + 1] = d[1];
                out[4 * w + 2] = d[2];
                out[4 * w + 3] = d[3];
            } else {
                dq_int4_interleaved(words[w], dc, d);  // (k0,k4) (k1,k5) (k2,k6) (k3,k7)
                out[4 * w + 0] = prmt(d[0], d[1], 0x5410u);  // (k0, k1)
                out[4 * w + 1] = prmt(d[2], d[3], 0x5410u);  // (k2, k3)
                out[4 * w + 2] = prmt(d[0], d[1], 0x7632u);  // (k4, k5)
                out[4 * w + 3] = prmt(d[2], d[3], 0x7632u);  // (k6, k7)
            }
        }
        uint4* dst = reinterpret_cast<uint4*>(W16 + (size_t)n * K + k0);
#pragma unroll
        for (int q = 0; q < 4; ++q) dst[q] = make_uint4(out[4 * q], out[4 * q + 1], out[4 * q + 2], out[4 * q + 3]);
    } else {
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            uint32_t d[2];
            dq_int8_natural(words[w], dc, d);
            out[2 * w] = d[0];
            out[2 * w + 1] = d[1];
        }
        uint4* dst = reinterpret_cast<uint4*>(W16 + (size_t)n * K + k0);
        dst[0] = make_uint4(out[0], out[1], out[2], out[3]);
        dst[1] = make_uint4(out[4], out[5], out[6], out[7]);
    }
}

}  // namespace

namespace {
// K == 0 with a bias: every output row is the bias (the output keeps its
// logical shape and holds zeros or the broadcast bias).
__global__ void fill_bias_kernel(__half* __restrict__ Y, const __half* __restrict__ bias, size_t rows, size_t N) {
    const size_t total = rows * N, stride = (size_t)gridDim.x * blockDim.x;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) Y[i] = bias[i % N];
}

// An empty packed weight with an adapter: Y[m, n] = fp16(sum_r T[m, r] B[n, r]
// (+ bias[n])), the adapter term alone, summed in FP32 in r order (each
// FP16 x FP16 product is exact in FP32).
__global__ void lora_up_kernel(const __half* __restrict__ T, const __half* __restrict__ B,
                               const uint8_t* __restrict__ Bq, const __half* __restrict__ Bs,
                               const uint8_t* __restrict__ Bz, const __half* __restrict__ bias,
                               __half* __restrict__ Y, int Mt, int N) {
    const size_t total = (size_t)Mt * (size_t)N;
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
        const size_t m = i / (size_t)N, n = i % (size_t)N;
        const __half2* t = reinterpret_cast<const __half2*>(T + m * 32);
        float s = 0.f;
        if (Bq) {  // INT8 row: b = fp16((q - zp) * scale), the product exact in FP32 and rounded once
            const float sc = __half2float(Bs[n]);
            const int z = Bz ? Bz[n] : 128;
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                const float2 tv = __half22float2(t[r]);
                const float b0 = __half2float(__float2half_rn((float)((int)Bq[n * 32 + 2 * r] - z) * sc));
                const float b1 = __half2float(__float2half_rn((float)((int)Bq[n * 32 + 2 * r + 1] - z) * sc));
                s += tv.x * b0;
                s += tv.y * b1;
            }
        } else {
            const __half2* b = reinterpret_cast<const __half2*>(B + n * 32);
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                const float2 tv = __half22float2(t[r]), bv = __half22float2(b[r]);
                s += tv.x * bv.x;
                s += tv.y * bv.y;
            }
        }
        if (bias) s += __half2float(bias[n]);
        Y[i] = __float2half_rn(s);
    }
}
}  // namespace

cudaError_t fill_bias_launch(__half* Y, const __half* bias, size_t rows, size_t N, cudaStream_t st) {
    const size_t total = rows * N;
    if (total == 0) return cudaSuccess;
    size_t blocks = (total + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    fill_bias_kernel<<<(unsigned)blocks, 256, 0, st>>>(Y, bias, rows, N);
    return cudaGetLastError();
}

cudaError_t wait_check_launch(unsigned int* status, long long limit_cycles, cudaStream_t st) {
    wait_check_kernel<<<1, 32, 0, st>>>(status, limit_cycles);
    return cudaGetLastError();
}

cudaError_t quantize_x_launch(const __half* X, int Mt, int K, int8_t* Xq, float* Xs, cudaStream_t st) {
    const long long total = (long long)Mt * (K / 32);
    if (total == 0) return cudaSuccess;
    quantize_x_kernel<<<(unsigned)((total + 127) / 128), 128, 0, st>>>(X, Mt, K, Xq, Xs);
    return cudaGetLastError();
}

cudaError_t lora_up_launch(const __half* T, const __half* B, const uint8_t* Bq, const __half* Bs, const uint8_t* Bz,
                           const __half* bias, __half* Y, int Mt, int N, cudaStream_t st) {
    const size_t total = (size_t)Mt * (size_t)N;
    if (total == 0) return cudaSuccess;
    size_t blocks = (total + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    lora_up_kernel<<<(unsigned)blocks, 256, 0, st>>>(T, B, Bq, Bs, Bz, bias, Y, Mt, N);
    return cudaGetLastError();
}

cudaError_t fill_zero_launch(__half* Y, size_t count, cudaStream_t st) {
    const size_t n16 = count / 8, ntail = count % 8;
    size_t blocks = (n16 + 255) / 256;
    if (blocks < 1) blocks = 1;
    if (blocks > 4096) blocks = 4096;
    fill_zero_kernel<<<(unsigned)blocks, 256, 0, st>>>(reinterpret_cast<uint4*>(Y), n16, Y + n16 * 8, ntail);
    return cudaGetLastError();
}

cudaError_t dequant_launch(const uint8_t* Wq, const __half* S, const uint8_t* Z, int N, int K, int bits,
                           __half* W16, int variant, cudaStream_t st) {
    const long long total = (long long)N * (K * bits / 8 / 16);
    if (total == 0) return cudaSuccess;
    const unsigned blocks = (unsigned)((total + 255) / 256);
    if (bits == 2)
        dequant_kernel<2><<<blocks, 256, 0, st>>>(Wq, S, Z, N, K, W16, variant);
    else if (bits == 4)
        dequant_kernel<4><<<blocks, 256, 0, st>>>(Wq, S, Z, N, K, W16, variant);
    else
        dequant_kernel<8><<<blocks, 256, 0, st>>>(Wq, S, Z, N, K, W16, variant);
    return cudaGetLastError();
}

}  // namespace mnb
