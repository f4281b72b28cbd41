// tensor_map.cu -- host-side TMA descriptor encoding shared by the kernels,
// and the identity of the current context.  The driver functions
// (cuTensorMapEncodeTiled, cuCtxGetCurrent, cuCtxGetId) are fetched from the
// driver through the runtime, so the library links only the (static) CUDA
// runtime.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "mnb_internal.h"

namespace mnb {

namespace {
std::mutex g_mu;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
PFN_cuCtxGetId_v12000 g_ctx_id = nullptr;

cudaError_t driver_fn(const char* name, int version, void** fn) {
    cudaDriverEntryPointQueryResult q;
    const cudaError_t e = cudaGetDriverEntryPointByVersion(name, fn, version, cudaEnableDefault, &q);
    if (e != cudaSuccess) return e;
    return q == cudaDriverEntryPointSuccess && *fn ? cudaSuccess : cudaErrorNotSupported;
}
}  // namespace

cudaError_t current_context_id(unsigned long long* id) {
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (!g_ctx_current || !g_ctx_id) {
            void *a = nullptr, *b = nullptr;
            cudaError_t e = driver_fn("cuCtxGetCurrent", 4000, &a);
            if (e == cudaSuccess) e = driver_fn("cuCtxGetId", 12000, &b);
            if (e != cudaSuccess) return e;
            g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(a);
            g_ctx_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(b);
        }
    }
    CUcontext ctx = nullptr;
    if (g_ctx_current(&ctx) != CUDA_SUCCESS) return cudaErrorUnknown;
    if (!ctx) {
        // the runtime creates the device's primary context lazily: make it current
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e == cudaSuccess) e = cudaSetDevice(dev);
        if (e != cudaSuccess) return e;
        if (g_ctx_current(&ctx) != CUDA_SUCCESS || !ctx) return cudaErrorUnknown;
    }
    return g_ctx_id(ctx, id) == CUDA_SUCCESS ? cudaSuccess : cudaErrorUnknown;
}

cudaError_t tensor_map_prepare() {
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_encode) return cudaSuccess;
    void* fn = nullptr;
    const cudaError_t e = driver_fn("cuTensorMapEncodeTiled", 12000, &fn);
    if (e != cudaSuccess) return e;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    return cudaSuccess;
}

// Row-major 2-D tensor [rows, cols] of `elem_bytes` elements, row pitch
// `pitch_bytes`, copied in boxes of [box_rows, box_cols]; out-of-range
// elements of a box read as zero.
cudaError_t encode_2d(CUtensorMap* map, const void* base, int elem_bytes, uint64_t cols, uint64_t rows,
                      uint64_t pitch_bytes, uint32_t box_cols, uint32_t box_rows, bool swizzle128) {
    if (!g_encode) return cudaErrorNotSupported;
    const CUtensorMapDataType dt = elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)pitch_bytes};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t es[2] = {1, 1};
    const CUresult r = g_encode(map, dt, 2, const_cast<void*>(base), dims, strides, box, es,
                                CU_TENSOR_MAP_INTERLEAVE_NONE,
                                swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t encode_rows_3d(CUtensorMap* map, const void* base, uint64_t rowbytes, uint64_t rows, uint32_t box_chunks,
                           uint32_t box_rows) {
    if (!g_encode) return cudaErrorNotSupported;
    if (rowbytes % 256 != 0) return cudaErrorInvalidValue;
    const cuuint64_t dims[3] = {256, (cuuint64_t)(rowbytes / 256), (cuuint64_t)rows};
    const cuuint64_t strides[2] = {256, (cuuint64_t)rowbytes};
    const cuuint32_t box[3] = {256, box_chunks, box_rows};
    const cuuint32_t es[3] = {1, 1, 1};
    const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, es,
                                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Rows of packed codes as 3-D boxes for a 128-byte swizzle: dims (128 bytes of a row,
// row, 128-byte segment), box (128, box_rows, box_segs).  In shared memory a box is
// [segment][box_rows][128 B] with chunk c of row r at c ^ (r & 7).
cudaError_t encode_codes_sw128(CUtensorMap* map, const void* base, uint64_t rowbytes, uint64_t rows,
                               uint32_t box_rows, uint32_t box_segs) {
    if (!g_encode) return cudaErrorNotSupported;
    if (rowbytes % 128 != 0 || rowbytes / 128 > 256 || box_segs == 0 || box_segs > rowbytes / 128)
        return cudaErrorInvalidValue;
    const cuuint64_t dims[3] = {128, (cuuint64_t)rows, (cuuint64_t)(rowbytes / 128)};
    const cuuint64_t strides[2] = {(cuuint64_t)rowbytes, 128};
    const cuuint32_t box[3] = {128, box_rows, box_segs};
    const cuuint32_t es[3] = {1, 1, 1};
    const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, es,
                                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace mnb
