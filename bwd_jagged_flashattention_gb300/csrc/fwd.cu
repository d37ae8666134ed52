// fwd.cu -- Jagged Flash Attention forward for sm_103a.
//
// Persistent, warp-specialised kernel: one CTA per SM walks its slice of the
// host schedule (items of up to two 128-row query tiles of one sequence and
// head that share every K/V tile).  Roles, as the pages describe them
// (Meta's TLX Jagged Flash Attention Beats FA4 on Blackwell With 3x Less
// Code, section "What TLX changes"):
//   warps 0-3  softmax + correction + epilogue for query tile 0
//   warps 4-7  the same for query tile 1
//   warp  8    TMA loads: Q tiles once per item, K/V tiles through a ring
//   warp  9    tcgen05 MMA issue (one thread) and TMEM allocation
// Tensor memory (512 columns): S0 | S1 | O0 | O1.  P (bf16) is written back
// over the first half of its S columns and fed to the PV product straight
// from TMEM (S and P have non-overlapping lifetimes, as the pages' TMEM
// aliasing describes).
//
// Online softmax: running row max m and sum l in the log2 domain.  O is
// rescaled in TMEM only when a block raises the max by more than 2^8
// (otherwise the stale max is kept; P stays <= 256, exact after the final
// division by l).  The KV loop is peeled into an unmasked bulk pass and a
// masked tail (section "Optimizations layered on top", "Loop peeling").
#include <cuda_runtime.h>

#include "kernels.h"
#include "ptx.cuh"

namespace jfa {
namespace {

constexpr int kFwdThreads = 320;
constexpr int kWarpTma = 8;
constexpr int kWarpMma = 9;
constexpr float kRescaleLog2 = 8.0f;
constexpr float kLn2 = 0.6931471805599453f;

template <int D>
struct FwdLayout {
    static constexpr int kSlabBytes = 128 * 128;  // 128 rows x 64 bf16 (one swizzle span)
    static constexpr int kSlabs = D / 64;
    static constexpr int kTileBytes = kSlabs * kSlabBytes;
    static constexpr int kSlots = D == 128 ? 4 : 8;  // K/V ring tiles
    static constexpr int kQOff = 0;
    static constexpr int kRingOff = 2 * kTileBytes;
    static constexpr int kBytes = (2 + kSlots) * kTileBytes;
    static constexpr int kDynSmem = kBytes + 1024;
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kOCol = 256;
};

struct FwdBars {
    uint64_t q_full, q_empty;
    uint64_t kv_full[8], kv_empty[8];
    uint64_t s_full[2], p_full[2], o_full[2], o_empty[2];
    uint64_t mma_done;
    uint32_t tmem_base;
    uint32_t abort_flag;
};

struct FwdItem {
    int b, h, kv_start, Lk, m0, nq, q_row0, q_rows;
    int nblk[2], nfull[2], nb;
};

// Every role derives the same per-item loop bounds from the work item.
__device__ __forceinline__ FwdItem decode_fwd(const WorkItem& w, const FwdParams& p) {
    FwdItem it;
    it.b = w.b;
    it.kv_start = w.kv_start;
    it.Lk = w.kv_len;
    it.h = static_cast<int>(w.packed & 0xFFu);
    it.m0 = static_cast<int>((w.packed >> 8) & 0x7FFFFFu);
    it.nq = 1 + static_cast<int>(w.packed >> 31);
    it.q_row0 = p.broadcast_q ? 0 : w.kv_start;
    it.q_rows = p.broadcast_q ? p.Lq : w.kv_len;
    const int nkv = (it.Lk + 127) / 128;
    it.nb = 0;
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        if (t < it.nq) {
            const int m = it.m0 + t;
            it.nblk[t] = p.causal ? min(m + 1, nkv) : nkv;
            it.nfull[t] = p.causal ? min(m, it.Lk / 128) : it.Lk / 128;
        } else {
            it.nblk[t] = 0;
            it.nfull[t] = 0;
        }
        it.nb = max(it.nb, it.nblk[t]);
    }
    return it;
}

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
    return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// S(tmem) = Q K^T: both operands K-major in 128-byte-swizzled slabs of 64
// columns; one K=16 step advances 32 bytes inside a slab.
template <int D>
__device__ __forceinline__ void issue_qk(uint32_t d_tmem, uint32_t q_addr, uint32_t k_addr) {
    constexpr uint32_t idesc = idesc_bf16_f32(128, 128, 0, 0);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = (kk / 4) * 16384 + (kk % 4) * 32;
        mma_ss(d_tmem, smem_desc(q_addr + off, 16, 1024), smem_desc(k_addr + off, 16, 1024), idesc, kk > 0);
    }
}

// O(tmem) (+)= P(tmem, bf16) V: V is MN-major (D contiguous); one K=16 step
// covers 16 key rows = 2048 bytes; the 64-column slabs are 16 KB apart.
template <int D>
__device__ __forceinline__ void issue_pv(uint32_t d_tmem, uint32_t p_tmem, uint32_t v_addr, uint32_t acc) {
    constexpr uint32_t idesc = idesc_bf16_f32(128, D, 0, 1);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
        mma_ts(d_tmem, p_tmem + kk * 8, smem_desc(v_addr + kk * 2048, 16384, 1024), idesc, (acc | kk) != 0);
}

// ---------------------------------------------------------------------------
// TMA producer (one thread).
// ---------------------------------------------------------------------------
template <int D>
__device__ void fwd_tma_role(const FwdParams& p, const CUtensorMap* mq, const CUtensorMap* mk,
                             const CUtensorMap* mv, uint8_t* smem, FwdBars& bars, int ib, int ie,
                             const AbortState& ab) {
    using L = FwdLayout<D>;
    prefetch_tensormap(mq);
    prefetch_tensormap(mk);
    prefetch_tensormap(mv);
    uint32_t ring = 0, q_loads = 0;
    for (int i = ib; i < ie; ++i) {
        const FwdItem it = decode_fwd(p.items[i], p);
        if (it.nb == 0) continue;
        if (!mbar_wait(&bars.q_empty, (q_loads & 1) ^ 1, ab)) goto done;
        mbar_arrive_expect_tx(&bars.q_full, it.nq * L::kTileBytes);
        for (int t = 0; t < it.nq; ++t)
#pragma unroll
            for (int s = 0; s < L::kSlabs; ++s)
                tma_load_2d(smem + L::kQOff + t * L::kTileBytes + s * L::kSlabBytes, mq, &bars.q_full,
                            it.h * D + 64 * s, it.q_row0 + 128 * (it.m0 + t));
        ++q_loads;
        for (int j = 0; j < it.nb; ++j) {
            for (int kv = 0; kv < 2; ++kv) {
                const uint32_t slot = ring % L::kSlots;
                if (!mbar_wait(&bars.kv_empty[slot], ((ring / L::kSlots) & 1) ^ 1, ab)) goto done;
                mbar_arrive_expect_tx(&bars.kv_full[slot], L::kTileBytes);
#pragma unroll
                for (int s = 0; s < L::kSlabs; ++s)
                    tma_load_2d(smem + L::kRingOff + slot * L::kTileBytes + s * L::kSlabBytes, kv ? mv : mk,
                                &bars.kv_full[slot], it.h * D + 64 * s, it.kv_start + 128 * j);
                ++ring;
            }
        }
    }
done:
    // Let every issued copy land before the CTA can exit.
    for (uint32_t r = ring > L::kSlots ? ring - L::kSlots : 0; r < ring; ++r)
        mbar_wait_drain(&bars.kv_full[r % L::kSlots], (r / L::kSlots) & 1);
    if (q_loads) mbar_wait_drain(&bars.q_full, (q_loads - 1) & 1);
}

// ---------------------------------------------------------------------------
// MMA issuer (one thread).  Order per item (FA-style ping-pong of the two
// query tiles so one tile's softmax overlaps the other tile's products):
//   S0=Q0K0, S1=Q1K0, then for each block j: O0+=P0Vj, S0=Q0K(j+1),
//   O1+=P1Vj, S1=Q1K(j+1).
// ---------------------------------------------------------------------------
template <int D>
__device__ void fwd_mma_role(const FwdParams& p, uint8_t* smem, FwdBars& bars, uint32_t tmem, int ib, int ie,
                             const AbortState& ab) {
    using L = FwdLayout<D>;
    const uint32_t q_base = smem_u32(smem + L::kQOff);
    const uint32_t ring_base = smem_u32(smem + L::kRingOff);
    uint32_t ring = 0, q_ph = 0;
    uint32_t p_ph[2] = {0, 0}, oe_ph[2] = {1, 1};
    for (int i = ib; i < ie; ++i) {
        const FwdItem it = decode_fwd(p.items[i], p);
        if (it.nb == 0) continue;
        if (!mbar_wait(&bars.q_full, q_ph, ab)) goto done;
        q_ph ^= 1;
        uint32_t kslot = ring % L::kSlots;
        if (!mbar_wait(&bars.kv_full[kslot], (ring / L::kSlots) & 1, ab)) goto done;
        ++ring;
        tc_fence_after();
#pragma unroll
        for (int t = 0; t < 2; ++t)
            if (it.nblk[t] > 0) {
                issue_qk<D>(tmem + t * 128, q_base + t * L::kTileBytes, ring_base + kslot * L::kTileBytes);
                mma_commit(&bars.s_full[t]);
            }
        mma_commit(&bars.kv_empty[kslot]);
        if (it.nb == 1) mma_commit(&bars.q_empty);
        for (int j = 0; j < it.nb; ++j) {
            const uint32_t vslot = ring % L::kSlots;
            if (!mbar_wait(&bars.kv_full[vslot], (ring / L::kSlots) & 1, ab)) goto done;
            ++ring;
            const bool has_next = j + 1 < it.nb;
            if (has_next) {
                kslot = ring % L::kSlots;
                if (!mbar_wait(&bars.kv_full[kslot], (ring / L::kSlots) & 1, ab)) goto done;
                ++ring;
            }
            tc_fence_after();
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                if (j >= it.nblk[t]) continue;
                if (j == 0) {
                    if (!mbar_wait(&bars.o_empty[t], oe_ph[t], ab)) goto done;
                    oe_ph[t] ^= 1;
                }
                if (!mbar_wait(&bars.p_full[t], p_ph[t], ab)) goto done;
                p_ph[t] ^= 1;
                tc_fence_after();
                issue_pv<D>(tmem + L::kOCol + t * D, tmem + t * 128, ring_base + vslot * L::kTileBytes, j > 0);
                if (j == it.nblk[t] - 1) mma_commit(&bars.o_full[t]);
                if (j + 1 < it.nblk[t]) {
                    issue_qk<D>(tmem + t * 128, q_base + t * L::kTileBytes, ring_base + kslot * L::kTileBytes);
                    mma_commit(&bars.s_full[t]);
                }
            }
            mma_commit(&bars.kv_empty[vslot]);
            if (has_next) {
                mma_commit(&bars.kv_empty[kslot]);
                if (j + 2 == it.nb) mma_commit(&bars.q_empty);
            }
        }
    }
done:
    // All issued MMAs must finish before TMEM is released.
    mma_commit(&bars.mma_done);
    mbar_wait_drain(&bars.mma_done, 0);
}

// ---------------------------------------------------------------------------
// Softmax / correction / epilogue (one warpgroup per query tile; thread r
// owns query row r of the tile = TMEM lane r).
// ---------------------------------------------------------------------------
template <int D, bool kMask>
__device__ __forceinline__ void softmax_block(const FwdParams& p, const FwdItem& it, int j, int qpos,
                                              uint32_t s_addr, uint32_t o_addr, float& m_use, float& l) {
    uint32_t sr[4][32];
#pragma unroll
    for (int c = 0; c < 4; ++c) tmem_ld32(s_addr + c * 32, sr[c]);
    tmem_ld_wait();
    if (kMask) {
        const int kbase = 128 * j;
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const int key = kbase + c * 32 + i;
                const bool vis = key < it.Lk && (!p.causal || key <= qpos);
                if (!vis) sr[c][i] = __float_as_uint(-INFINITY);
            }
    }
    float mx = -INFINITY;
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int i = 0; i < 32; ++i) mx = fmaxf(mx, __uint_as_float(sr[c][i]));
    const float m_new = fmaxf(m_use, mx * p.scale_log2);
    float corr = 1.0f;
    bool resc = false;
    if (j == 0) {
        m_use = m_new;
    } else if (m_new > m_use + kRescaleLog2) {
        corr = ex2_approx(m_use - m_new);
        m_use = m_new;
        resc = true;
    }
    const float base = m_use == -INFINITY ? 0.0f : m_use;
    float rs = 0.0f;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const float p0 = ex2_approx(fmaf(__uint_as_float(sr[c][2 * i]), p.scale_log2, -base));
            const float p1 = ex2_approx(fmaf(__uint_as_float(sr[c][2 * i + 1]), p.scale_log2, -base));
            rs += p0 + p1;
            pk[i] = pack_bf16x2(p0, p1);
        }
        tmem_st16(s_addr + c * 16, pk);
    }
    l = l * corr + rs;
    if (__any_sync(0xffffffffu, resc)) {
#pragma unroll
        for (int oc = 0; oc < D / 32; ++oc) {
            uint32_t orr[32];
            tmem_ld32(o_addr + oc * 32, orr);
            tmem_ld_wait();
            uint32_t lo[16], hi[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                lo[i] = __float_as_uint(__uint_as_float(orr[i]) * corr);
                hi[i] = __float_as_uint(__uint_as_float(orr[16 + i]) * corr);
            }
            tmem_st16(o_addr + oc * 32, lo);
            tmem_st16(o_addr + oc * 32 + 16, hi);
        }
    }
    tmem_st_wait();
}

template <int D>
__device__ void fwd_softmax_role(const FwdParams& p, FwdBars& bars, uint32_t tmem, int ib, int ie,
                                 const AbortState& ab) {
    using L = FwdLayout<D>;
    const int t = threadIdx.x / 128;
    const int row = threadIdx.x % 128;
    const int wq = (threadIdx.x / 32) % 4;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t s_addr = tmem + lane_off + t * 128;
    const uint32_t o_addr = tmem + lane_off + L::kOCol + t * D;
    uint32_t s_ph = 0, o_ph = 0;
    for (int i = ib; i < ie; ++i) {
        const FwdItem it = decode_fwd(p.items[i], p);
        if (t >= it.nq) continue;
        const int nblk = t == 0 ? it.nblk[0] : it.nblk[1];   // scalar copies: no
        const int nfull = t == 0 ? it.nfull[0] : it.nfull[1];  // dynamic array indexing
        const int qpos = 128 * (it.m0 + t) + row;
        const bool valid = qpos < it.q_rows;
        const int64_t orow = p.broadcast_q ? static_cast<int64_t>(it.b) * p.Lq + qpos
                                           : static_cast<int64_t>(it.q_row0) + qpos;
        uint16_t* optr = p.o + (orow * p.H + it.h) * D;
        const int64_t lse_idx = p.broadcast_q ? (static_cast<int64_t>(it.b) * p.H + it.h) * p.Lq + qpos
                                              : static_cast<int64_t>(it.h) * p.N + it.q_row0 + qpos;
        if (nblk == 0) {  // empty sequence: O = 0, LSE = -inf
            if (valid) {
#pragma unroll
                for (int v = 0; v < D / 8; ++v) reinterpret_cast<uint4*>(optr)[v] = make_uint4(0, 0, 0, 0);
                p.lse[lse_idx] = -INFINITY;
            }
            continue;
        }
        float m_use = -INFINITY, l = 0.0f;
        int j = 0;
        for (; j < nfull; ++j) {  // bulk: every key visible, no mask
            if (!mbar_wait_warp(&bars.s_full[t], s_ph, ab)) goto done;
            s_ph ^= 1;
            tc_fence_after();
            softmax_block<D, false>(p, it, j, qpos, s_addr, o_addr, m_use, l);
            tc_fence_before();
            mbar_arrive(&bars.p_full[t]);
        }
        for (; j < nblk; ++j) {  // tail: ragged end and/or causal diagonal
            if (!mbar_wait_warp(&bars.s_full[t], s_ph, ab)) goto done;
            s_ph ^= 1;
            tc_fence_after();
            softmax_block<D, true>(p, it, j, qpos, s_addr, o_addr, m_use, l);
            tc_fence_before();
            mbar_arrive(&bars.p_full[t]);
        }
        // Epilogue: O / l to bf16, LSE = ln(sum exp) of the scaled scores.
        if (!mbar_wait_warp(&bars.o_full[t], o_ph, ab)) goto done;
        o_ph ^= 1;
        tc_fence_after();
        {
            uint32_t orr[D / 32][32];
#pragma unroll
            for (int oc = 0; oc < D / 32; ++oc) tmem_ld32(o_addr + oc * 32, orr[oc]);
            tmem_ld_wait();
            tc_fence_before();
            mbar_arrive(&bars.o_empty[t]);  // TMEM O is free: the next item's PV may start
            if (valid) {
                const float inv = l > 0.0f ? 1.0f / l : 0.0f;
#pragma unroll
                for (int oc = 0; oc < D / 32; ++oc)
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        uint4 u;
                        u.x = pack_bf16x2(__uint_as_float(orr[oc][8 * v + 0]) * inv,
                                          __uint_as_float(orr[oc][8 * v + 1]) * inv);
                        u.y = pack_bf16x2(__uint_as_float(orr[oc][8 * v + 2]) * inv,
                                          __uint_as_float(orr[oc][8 * v + 3]) * inv);
                        u.z = pack_bf16x2(__uint_as_float(orr[oc][8 * v + 4]) * inv,
                                          __uint_as_float(orr[oc][8 * v + 5]) * inv);
                        u.w = pack_bf16x2(__uint_as_float(orr[oc][8 * v + 6]) * inv,
                                          __uint_as_float(orr[oc][8 * v + 7]) * inv);
                        reinterpret_cast<uint4*>(optr + oc * 32)[v] = u;
                    }
                p.lse[lse_idx] = l > 0.0f ? (m_use + lg2_approx(l)) * kLn2 : -INFINITY;
            }
        }
    }
done:;
}

template <int D>
__global__ void __launch_bounds__(kFwdThreads, 1)
    jfa_fwd_kernel(const FwdParams p, const __grid_constant__ CUtensorMap map_q,
                   const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v) {
    using L = FwdLayout<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024(smem_raw);
    __shared__ FwdBars bars;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int ib = p.cta_start[blockIdx.x], ie = p.cta_start[blockIdx.x + 1];
    const AbortState ab{&bars.abort_flag, p.status};

    if (threadIdx.x == 0) {
        bars.abort_flag = 0;
        mbar_init(&bars.q_full, 1);
        mbar_init(&bars.q_empty, 1);
        for (int s = 0; s < L::kSlots; ++s) {
            mbar_init(&bars.kv_full[s], 1);
            mbar_init(&bars.kv_empty[s], 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(&bars.s_full[t], 1);
            mbar_init(&bars.p_full[t], 128);
            mbar_init(&bars.o_full[t], 1);
            mbar_init(&bars.o_empty[t], 128);
        }
        mbar_init(&bars.mma_done, 1);
        fence_mbar_init();
    }
    if (warp == kWarpMma) {
        tmem_alloc(&bars.tmem_base, L::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars.tmem_base;

    if (warp < 8) {
        fwd_softmax_role<D>(p, bars, tmem, ib, ie, ab);
    } else if (warp == kWarpTma) {
        if (lane == 0) fwd_tma_role<D>(p, &map_q, &map_k, &map_v, smem, bars, ib, ie, ab);
        __syncwarp();
    } else {
        if (lane == 0) fwd_mma_role<D>(p, smem, bars, tmem, ib, ie, ab);
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kWarpMma) tmem_dealloc(tmem, L::kTmemCols);
}

template <int D>
cudaError_t launch_fwd_d(const FwdParams& p, const FwdMaps& m, int grid, cudaStream_t s) {
    using L = FwdLayout<D>;
    static bool configured = false;
    if (!configured) {
        cudaError_t e =
            cudaFuncSetAttribute(jfa_fwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kDynSmem);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    jfa_fwd_kernel<D><<<grid, kFwdThreads, L::kDynSmem, s>>>(p, m.q, m.k, m.v);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd(int D, const FwdParams& p, const FwdMaps& m, int grid, cudaStream_t s) {
    if (grid <= 0) return cudaSuccess;
    return D == 128 ? launch_fwd_d<128>(p, m, grid, s) : launch_fwd_d<64>(p, m, grid, s);
}

}  // namespace jfa
