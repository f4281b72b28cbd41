// dq_layout.cu -- host utility: a DequantizeLinear weight rewritten into the
// MatMulNBits layout.
//
// "Fuse DQ->MatMulNBits for shared initializers and skip outer-scope weights"
// (onnxruntime PR 33800, Description) fuses DequantizeLinear(w_q, w_scale,
// w_zp) -> MatMul into MatMulNBits by writing new, transposed initializers
// from the originals: the DQ weight is [K, N] (MatMul's right operand, codes
// along N in memory) with its scale and zero point per tensor or per block of
// `block_size` rows along K; MatMulNBits wants each output row n's codes
// contiguous along K, packed, with one scale and zero point per (n, block).
// This is that rewrite, done once on the host.  DequantizeLinear's zero point
// defaults to 0 (not MatMulNBits' 2^(bits-1)), so explicit zero points are
// always written.
#include <stdint.h>
#include <string.h>

#include "mnb.h"

extern "C" int mnb_transpose_dq_weight(const uint8_t* w_q, const uint16_t* w_scale, const uint8_t* w_zp, int64_t K,
                                       int64_t N, int32_t bits, int32_t block_size, int32_t blocked, uint8_t* Wq,
                                       uint16_t* scales, uint8_t* zp) {
    if (K < 0 || N < 0) return MNB_ERR_ARG;
    if (bits != 2 && bits != 4 && bits != 8) return MNB_ERR_UNSUPPORTED;
    if (block_size != 32 || K % block_size != 0) return MNB_ERR_UNSUPPORTED;
    if (K == 0 || N == 0) return MNB_OK;
    if (!w_q || !w_scale || !Wq || !scales || !zp) return MNB_ERR_ARG;
    const int64_t nblk = K / block_size;
    const int per_byte = 8 / bits;
    const int64_t rowbytes = K / per_byte;
    const uint32_t limit = 1u << bits;
    for (int64_t k = 0; k < K; ++k)  // every code must fit the target width
        for (int64_t n = 0; n < N; ++n)
            if (w_q[k * N + n] >= limit) return MNB_ERR_ARG;
    for (int64_t n = 0; n < N; ++n) {
        uint8_t* row = Wq + n * rowbytes;
        memset(row, 0, (size_t)rowbytes);
        for (int64_t k = 0; k < K; ++k)
            row[k / per_byte] |= (uint8_t)(w_q[k * N + n] << (bits * (int)(k % per_byte)));
        for (int64_t b = 0; b < nblk; ++b) {
            const int64_t src = blocked ? b * N + n : 0;  // [K/bs, N] or one value
            scales[n * nblk + b] = w_scale[src];
            zp[n * nblk + b] = w_zp ? w_zp[src] : 0;
        }
    }
    return MNB_OK;
}
