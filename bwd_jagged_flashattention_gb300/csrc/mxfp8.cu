// mxfp8.cu -- MXFP8 quantization of V for the MXFP8 forward (fwd.cu, kMx).
//
// The MXFP8 variant quantizes the operands of its P V product to FP8 with
// scale factors (TLX porta l'attenzione jagged su Blackwell oltre FA4 con un
// terzo del codice, section "The turning point").  V's contraction dimension
// is the key, so its blocks of 32 run along the keys of one sequence, per
// head and column: within 128-key block n of sequence b, chunk c holds keys
// 128 n + 32 c .. + 31 (fewer at the sequence end).  Per chunk and column,
// X = floor(log2(max |v|)) - 8 (clamped to E8M0's range [-127, 127]; -127 for
// an all-zero chunk), each v is stored as E4M3(v / 2^X) (nearest, ties to
// even, saturating at 448), and the scale byte X + 127 goes to
// v_scale[((block_start[b] + n) * H + h) * D + d][c]; a chunk past the
// sequence end gets 0.  All of it is exact fp32 arithmetic on the bf16
// inputs, so the codes are bit-for-bit reproducible.
#include <cuda_runtime.h>

#include "kernels.h"
#include "ptx.cuh"

namespace jfa {
namespace {

// floor(log2(a)) - 8 for a finite a >= 0, clamped to [-127, 127]; -127 for 0.
// Read from a's bits (subnormals from the leading mantissa bit).
__device__ __forceinline__ int mx_exponent(float a) {
    if (a == 0.0f) return -127;
    const uint32_t u = __float_as_uint(a);
    const int eb = static_cast<int>((u >> 23) & 0xFFu);
    const int fl = eb != 0 ? eb - 127 : (31 - __clz(static_cast<int>(u & 0x7FFFFFu))) - 149;
    return max(-127, min(127, fl - 8));
}

// 2^-X for X in [-127, 127] (2^-127 is the subnormal with mantissa bit 22).
__device__ __forceinline__ float exp2_neg(int X) {
    return X <= 126 ? __int_as_float((127 - X) << 23) : __int_as_float(1 << 22);
}

// One CTA per 128-key block nb.  Work unit = (32-key chunk c, 8 adjacent
// columns of one head): its thread reads the chunk's rows as 16-byte vectors
// (a warp covers 512 contiguous bytes of a row), takes the 8 column maxima,
// then reads the rows again (now from L1) to write 8 codes per row as one
// 8-byte store.  The scale bytes meet in shared memory ([column][chunk], the
// output layout) and leave as 16-byte words.
constexpr int kQuantThreads = 256;

__global__ void __launch_bounds__(kQuantThreads) jfa_quant_v_mxfp8_kernel(const uint16_t* __restrict__ v,
                                                                          const int32_t* __restrict__ offsets,
                                                                          const int32_t* __restrict__ block_start,
                                                                          int B, int H, int D,
                                                                          uint8_t* __restrict__ v8,
                                                                          uint32_t* __restrict__ v_scale) {
    extern __shared__ uint32_t sc_words[];  // [H * D] scale words of this block
    const int64_t nb = blockIdx.x;
    // The sequence holding block nb: the largest b with block_start[b] <= nb
    // (block_start[0] = 0 <= nb < block_start[B]; empty sequences repeat a
    // value, and the largest such b is the non-empty one).
    int lo = 0, hi = B;
    while (hi - lo > 1) {
        const int mid = (lo + hi) / 2;
        if (block_start[mid] <= nb) lo = mid;
        else hi = mid;
    }
    const int b = lo;
    const int n = static_cast<int>(nb - block_start[b]);
    const int64_t row0 = static_cast<int64_t>(offsets[b]) + 128 * n;
    const int nk = min(128, offsets[b + 1] - offsets[b] - 128 * n);
    const int64_t stride = static_cast<int64_t>(H) * D;  // elements per key row
    const int groups = H * D / 8;                         // 8-column groups per row
    uint8_t* sc = reinterpret_cast<uint8_t*>(sc_words);
    for (int u = threadIdx.x; u < 4 * groups; u += blockDim.x) {
        const int c = u / groups, g = u % groups;
        const int col = 8 * g;  // h * D + d, d a multiple of 8 (never crosses a head)
        const int k0 = 32 * c, cnt = min(32, nk - k0);
        uint32_t code[8];
        if (cnt <= 0) {  // no key in this chunk: scale code 0
#pragma unroll
            for (int e = 0; e < 8; ++e) code[e] = 0;
        } else {
            const uint4* src = reinterpret_cast<const uint4*>(v + (row0 + k0) * stride + col);
            const int64_t rstep = stride / 8;  // uint4 per row
            float amax[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) amax[e] = 0.0f;
#pragma unroll 8
            for (int k = 0; k < cnt; ++k) {
                const uint4 w = __ldg(src + k * rstep);
                const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    amax[2 * q] = fmaxf(amax[2 * q], fabsf(bf16lo_to_f32(ww[q])));
                    amax[2 * q + 1] = fmaxf(amax[2 * q + 1], fabsf(__uint_as_float(ww[q] & 0xFFFF0000u)));
                }
            }
            float s[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int X = mx_exponent(amax[e]);
                code[e] = static_cast<uint32_t>(X + 127);
                s[e] = exp2_neg(X);
            }
            uint2* dst = reinterpret_cast<uint2*>(v8 + (row0 + k0) * stride + col);
            const int64_t dstep = stride / 8;  // uint2 per row
#pragma unroll 8
            for (int k = 0; k < cnt; ++k) {
                const uint4 w = __ldg(src + k * rstep);
                const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
                uint32_t pk[2];
#pragma unroll
                for (int q = 0; q < 2; ++q)
                    pk[q] = cvt_e4m3x2(bf16lo_to_f32(ww[2 * q]) * s[4 * q],
                                       __uint_as_float(ww[2 * q] & 0xFFFF0000u) * s[4 * q + 1]) |
                            (cvt_e4m3x2(bf16lo_to_f32(ww[2 * q + 1]) * s[4 * q + 2],
                                        __uint_as_float(ww[2 * q + 1] & 0xFFFF0000u) * s[4 * q + 3])
                             << 16);
                dst[k * dstep] = make_uint2(pk[0], pk[1]);
            }
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) sc[(col + e) * 4 + c] = static_cast<uint8_t>(code[e]);
    }
    __syncthreads();
    uint4* out = reinterpret_cast<uint4*>(v_scale + nb * stride);
    for (int i = threadIdx.x; i < H * D / 4; i += blockDim.x) out[i] = reinterpret_cast<const uint4*>(sc_words)[i];
}

}  // namespace

cudaError_t launch_quant_v_mxfp8(const uint16_t* v, const int32_t* offsets, const int32_t* block_start, int B,
                                 int64_t n_blocks, int H, int D, uint8_t* v8, uint32_t* v_scale, cudaStream_t s) {
    if (n_blocks <= 0) return cudaSuccess;
    if (n_blocks > 0x7FFFFFFF) return cudaErrorInvalidValue;
    const size_t smem = static_cast<size_t>(H) * D * 4;  // at most 255 x 128 x 4 = 130,560 bytes
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(jfa_quant_v_mxfp8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
        return cudaErrorInvalidValue;
    jfa_quant_v_mxfp8_kernel<<<static_cast<unsigned>(n_blocks), kQuantThreads, smem, s>>>(v, offsets, block_start, B,
                                                                                        H, D, v8, v_scale);
    return cudaGetLastError();
}

}  // namespace jfa
