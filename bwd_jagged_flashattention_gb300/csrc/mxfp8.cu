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

// One CTA per 128-key block nb.  Thread i takes column pairs (h, d, d + 1),
// d even, i, i + 256, ...; for each chunk it reads the chunk's keys (a warp
// reads 32 consecutive pairs = 128 bytes of one row), finds both columns'
// maxima, then writes the codes (2 bytes per key) and, at the end, both
// columns' four scale bytes as one 8-byte store.
__global__ void __launch_bounds__(256) jfa_quant_v_mxfp8_kernel(const uint16_t* __restrict__ v,
                                                                const int32_t* __restrict__ offsets,
                                                                const int32_t* __restrict__ block_start, int B,
                                                                int H, int D, uint8_t* __restrict__ v8,
                                                                uint32_t* __restrict__ v_scale) {
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
    const int pairs = H * D / 2;
    for (int cp = threadIdx.x; cp < pairs; cp += blockDim.x) {
        const int h = cp / (D / 2), d = 2 * (cp % (D / 2));
        const int64_t col = static_cast<int64_t>(h) * D + d;
        const int64_t stride = static_cast<int64_t>(H) * D;
        uint32_t sc0 = 0, sc1 = 0;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
            const int k0 = 32 * c, cnt = min(32, nk - k0);
            if (cnt <= 0) break;  // no key left: the remaining scale bytes stay 0
            uint32_t w[32];
            float a0 = 0.0f, a1 = 0.0f;
#pragma unroll
            for (int k = 0; k < 32; ++k) {
                w[k] = 0;
                if (k < cnt) {
                    w[k] = __ldg(reinterpret_cast<const uint32_t*>(v + (row0 + k0 + k) * stride + col));
                    a0 = fmaxf(a0, fabsf(bf16lo_to_f32(w[k])));
                    a1 = fmaxf(a1, fabsf(__uint_as_float(w[k] & 0xFFFF0000u)));
                }
            }
            const int X0 = mx_exponent(a0), X1 = mx_exponent(a1);
            const float s0 = exp2_neg(X0), s1 = exp2_neg(X1);
#pragma unroll
            for (int k = 0; k < 32; ++k)
                if (k < cnt)
                    *reinterpret_cast<uint16_t*>(v8 + (row0 + k0 + k) * stride + col) = static_cast<uint16_t>(
                        cvt_e4m3x2(bf16lo_to_f32(w[k]) * s0, __uint_as_float(w[k] & 0xFFFF0000u) * s1));
            sc0 |= static_cast<uint32_t>(X0 + 127) << (8 * c);
            sc1 |= static_cast<uint32_t>(X1 + 127) << (8 * c);
        }
        *reinterpret_cast<uint2*>(v_scale + (nb * H + h) * D + d) = make_uint2(sc0, sc1);
    }
}

}  // namespace

cudaError_t launch_quant_v_mxfp8(const uint16_t* v, const int32_t* offsets, const int32_t* block_start, int B,
                                 int64_t n_blocks, int H, int D, uint8_t* v8, uint32_t* v_scale, cudaStream_t s) {
    if (n_blocks <= 0) return cudaSuccess;
    if (n_blocks > 0x7FFFFFFF) return cudaErrorInvalidValue;
    jfa_quant_v_mxfp8_kernel<<<static_cast<unsigned>(n_blocks), 256, 0, s>>>(v, offsets, block_start, B, H, D, v8,
                                                                            v_scale);
    return cudaGetLastError();
}

}  // namespace jfa
