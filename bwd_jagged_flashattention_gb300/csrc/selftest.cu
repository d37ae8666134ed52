// selftest.cu -- single-tile checks of the tcgen05/TMA building blocks.
//
// One CTA computes a 128x128x128 bf16 product into an fp32 TMEM accumulator
// with the same descriptor conventions the attention kernels use, and writes
// the fp32 result to global memory, so that a test can compare it with a
// library matmul.  Modes:
//   0  A K-major [M][K],  B K-major [N][K]          C = A B^T   (S = Q K^T)
//   1  A K-major [M][K],  B MN-major [K][N]          C = A B     (O = P V, P in smem)
//   2  A from TMEM,       B MN-major [K][N]          C = A B     (O = P V, P in TMEM)
//   3  A MN-major [K][M], B MN-major [K][N]          C = A^T B   (dQ = dS K)
//   4  like 1, issued as two N=64 halves
#include <cuda_runtime.h>

#include "../../include/jfa_selftest.h"
#include "host_util.h"
#include "ptx.cuh"

namespace jfa {
namespace {

constexpr int kTile = 128;
constexpr int kSlabBytes = 128 * 128;  // 128 rows x 64 bf16 (one 128-byte swizzle span)

__global__ void __launch_bounds__(128, 1)
    selftest_mma_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                        const uint16_t* __restrict__ a_global, float* __restrict__ c, int mode,
                        uint32_t* status) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem;                     // 2 slabs, 32 KB
    uint8_t* sB = smem + 2 * kSlabBytes;    // 2 slabs, 32 KB
    __shared__ uint64_t bars[2];
    __shared__ uint32_t tmem_base_s;
    __shared__ uint32_t abort_flag;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    AbortState ab{&abort_flag, status, kDefaultWaitLimitNs};

    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(&tmem_base_s, 256);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_s;

    if (threadIdx.x == 0) {
        mbar_arrive_expect_tx(&bars[0], 4 * kSlabBytes);
        for (int s = 0; s < 2; ++s) {
            tma_load_2d(sA + s * kSlabBytes, &map_a, &bars[0], 64 * s, 0);
            tma_load_2d(sB + s * kSlabBytes, &map_b, &bars[0], 64 * s, 0);
        }
    }
    bool ok = mbar_wait(&bars[0], 0, ab);

    if (mode == 2) {
        // Each thread packs its own row of A (bf16 pairs) into TMEM columns [128, 192).
        const int row = threadIdx.x;
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>(warp * 32) << 16);
        for (int chunk = 0; chunk < 4; ++chunk) {
            uint32_t r[16];
            for (int i = 0; i < 16; ++i) {
                const uint16_t lo = a_global[row * kTile + chunk * 32 + 2 * i];
                const uint16_t hi = a_global[row * kTile + chunk * 32 + 2 * i + 1];
                r[i] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
            }
            tmem_st16(lane_addr + 128 + chunk * 16, r);
        }
        tmem_st_wait();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    if (threadIdx.x == 0 && ok) {
        const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sB);
        for (int kk = 0; kk < kTile / 16; ++kk) {
            const uint32_t acc = kk > 0;
            const uint32_t kmaj_off = (kk / 4) * kSlabBytes + (kk % 4) * 32;  // K-major: 16 elems = 32 B
            const uint32_t mn_off = kk * 16 * 128;                            // MN-major: 16 rows of 128 B
            switch (mode) {
                case 0:
                    mma_ss(tmem, smem_desc(a0 + kmaj_off, 16, 1024), smem_desc(b0 + kmaj_off, 16, 1024),
                           idesc_bf16_f32(128, 128, 0, 0), acc);
                    break;
                case 1:
                    mma_ss(tmem, smem_desc(a0 + kmaj_off, 16, 1024), smem_desc(b0 + mn_off, kSlabBytes, 1024),
                           idesc_bf16_f32(128, 128, 0, 1), acc);
                    break;
                case 2:
                    mma_ts(tmem, tmem + 128 + kk * 8, smem_desc(b0 + mn_off, kSlabBytes, 1024),
                           idesc_bf16_f32(128, 128, 0, 1), acc);
                    break;
                case 3:
                    mma_ss(tmem, smem_desc(a0 + mn_off, kSlabBytes, 1024), smem_desc(b0 + mn_off, kSlabBytes, 1024),
                           idesc_bf16_f32(128, 128, 1, 1), acc);
                    break;
                case 4:
                    for (int h = 0; h < 2; ++h)
                        mma_ss(tmem + 64 * h, smem_desc(a0 + kmaj_off, 16, 1024),
                               smem_desc(b0 + h * kSlabBytes + mn_off, kSlabBytes, 1024),
                               idesc_bf16_f32(128, 64, 0, 1), acc);
                    break;
                default:
                    break;
            }
        }
        mma_commit(&bars[1]);
    }
    __syncwarp();
    ok = mbar_wait(&bars[1], 0, ab) && ok;
    tc_fence_after();

    const int row = warp * 32 + lane;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    for (int chunk = 0; chunk < 4; ++chunk) {
        uint32_t r[32];
        tmem_ld32(lane_addr + chunk * 32, r);
        tmem_ld_wait();
        if (ok)
            for (int i = 0; i < 32; ++i) c[row * kTile + chunk * 32 + i] = __uint_as_float(r[i]);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 256);
}

// Abort-path check (no fault, no trap): warp 1 waits on a barrier nothing
// arrives at, under the given limit; warp 2 waits on another such barrier
// with a limit 2000 times longer, so it can only return early through the
// CTA abort flag warp 1 raises; warp 0 holds 32 TMEM columns for the
// kernel's lifetime and frees them at the end, as the attention kernels do.
// Every wait is bounded, so the kernel returns; out[w - 1] = 1 if warp w's
// wait completed, 0 if it gave up.
__global__ void __launch_bounds__(96, 1) selftest_timeout_kernel(uint32_t* status, uint64_t limit_ns, uint32_t* out) {
    __shared__ uint64_t bars[2];
    __shared__ uint32_t tmem_base_s;
    __shared__ uint32_t abort_flag;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(&tmem_base_s, 32);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp > 0) {
        const AbortState ab{&abort_flag, status, warp == 1 ? limit_ns : 2000 * limit_ns};
        const bool ok = mbar_wait_warp(&bars[warp - 1], 0, ab);
        if (lane == 0) out[warp - 1] = ok ? 1u : 0u;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem_base_s, 32);
}

bool map_128x128_bf16(CUtensorMap* m, const void* p) {
    const uint64_t dims[2] = {128, 128};
    const uint64_t strides[1] = {128 * 2};
    const uint32_t box[2] = {64, 128};
    return encode_tensor_map(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p, dims, strides, box,
                             CU_TENSOR_MAP_SWIZZLE_128B);
}

}  // namespace
}  // namespace jfa

extern "C" int jfa_selftest_mma(int mode, const void* a, const void* b, float* c, unsigned int* status,
                                void* stream) {
    using namespace jfa;
    if (mode < 0 || mode > 4 || !a || !b || !c || !status) return 1;
    if ((reinterpret_cast<uintptr_t>(a) | reinterpret_cast<uintptr_t>(b)) & 15) return 1;
    CUtensorMap ma, mb;
    if (!map_128x128_bf16(&ma, a) || !map_128x128_bf16(&mb, b)) return 4;
    const int smem = 4 * 128 * 128 + 1024;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaFuncSetAttribute(selftest_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return 4;
    selftest_mma_kernel<<<1, 128, smem, s>>>(ma, mb, static_cast<const uint16_t*>(a), c, mode,
                                             reinterpret_cast<uint32_t*>(status));
    return cudaGetLastError() == cudaSuccess ? 0 : 4;
}

extern "C" int jfa_selftest_timeout(unsigned long long limit_ns, unsigned int* status, unsigned int* out,
                                    void* stream) {
    using namespace jfa;
    if (!status || !out || limit_ns == 0 || limit_ns > 1000000000ull) return 1;
    selftest_timeout_kernel<<<1, 96, 0, static_cast<cudaStream_t>(stream)>>>(
        reinterpret_cast<uint32_t*>(status), static_cast<uint64_t>(limit_ns), reinterpret_cast<uint32_t*>(out));
    return cudaGetLastError() == cudaSuccess ? 0 : 4;
}
