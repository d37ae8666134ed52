// bwd.cu -- Jagged Flash Attention backward for sm_103a.
//
// Two kernels:
//   jfa_bwd_pre    Delta = rowsum(dO * O) in fp32 (LSE layout).  The pages do
//                  not name it; FlashAttention's backward needs it.
//   jfa_bwd_kernel persistent, warp-specialised main pass.
//
// The main pass walks items (sequence b, head h, key/value tile n of 128
// rows) and loops over the query tiles that see that key tile.  For query
// tile i (128 rows), with K, V the item's tiles:
//   S^T  = K Q_i^T                       (TMEM, fp32)
//   dP^T = V dO_i^T                      (TMEM, fp32)
//   P^T  = exp(scale S^T - LSE_i)        (bf16, written over S^T in TMEM)
//   dV  += P^T dO_i                      (A operand straight from TMEM)
//   dS^T = P^T * (dP^T - Delta_i)        (bf16, shared memory)
//   dK  += dS^T Q_i                      (TMEM accumulator for the item)
//   dQ_i = dS_i K                        (TMEM, over the dP^T columns)
// dQ_i is read out by a dedicated warpgroup, which frees its TMEM columns at
// once and then streams it through two 16-column fp32 shared-memory stages (64-byte swizzle)
// into TMA bulk reduce-adds on the global fp32 dQ.  In broadcast-Q mode every
// sequence adds into the same dQ [Lq,H,D]: the pages call this contended
// reduction the first backward bottleneck and hide it with a double-buffered
// shared-memory pipeline and an early release of the dQ tensor memory
// (Meta's TLX Jagged Flash Attention Beats FA4 on Blackwell With 3x Less
// Code, section "Optimizations layered on top"; Meta's 3.2K-line Triton
// kernel outruns FlashAttention-4 on jagged Blackwell attention, second
// paragraph).  dK/dV stay in TMEM for the whole item and are written once.
//
// Roles (128 x (JFA_BWD_COMPUTE_WGS + 2) threads; listed for one compute warpgroup):
//   warps 0-3  compute: P^T and dS^T (thread r = key row r = TMEM lane r)
//   warps 4-7  dQ readout + reduce-add; dK/dV epilogue (staged, coalesced)
//   warp  8    loads: K, V per item; Q_i (+ LSE_i, Delta_i) and dO_i per tile
//   warp  9    tcgen05 MMA issue and TMEM allocation
//   warps 10-11 idle (they give their registers to the compute warps)
#include <cuda_runtime.h>

#include "kernels.h"
#include "ptx.cuh"
#include "trace.cuh"

namespace jfa {
namespace {

// Tuning knob (compile-time): L2 prefetch of the next item's tiles (measured
// slower on the ads workload, so off by default).
// Compute / dQ warpgroups -> MMA hand-offs (p_full, ds_full, dq_empty):
// 1 = one arrival per warp (lane 0, after the warp's fences and a
// __syncwarp), 0 = one per thread.  Measured on the ads step: no gain
// (385.3 vs 382.9 us).
#ifndef JFA_BWD_WARP_ARRIVE
#define JFA_BWD_WARP_ARRIVE 0
#endif
#ifndef JFA_BWD_PREFETCH
#define JFA_BWD_PREFETCH 0
#endif
// dK/dV epilogue: 1 = staged through the dS buffer (free at the end of an
// item) with coalesced copies, 0 = each thread stores its own row (ads step
// with the last dQ first: 478 vs 483 us).
// Exponent pairs (of every 16) computed on the FMA pipe in unmasked tiles.
// Measured: any share > 0 is slower on GB300 (the passes are latency-bound,
// not special-function-bound), so the default keeps every exponential on the SFU.
#ifndef JFA_BWD_POLY_PAIRS
#define JFA_BWD_POLY_PAIRS 0
#endif
// dQ before dK: 1 = on the last query tile of an item (releases K one
// product earlier; ads step 483 vs 492 us), 2 = on every tile (the dQ
// readout, and so the next dP^T, also comes sooner; 467.6 vs 470.4 us).
#ifndef JFA_BWD_DQ_FIRST
#define JFA_BWD_DQ_FIRST 2
#endif
// The compute warps keep P (packed bf16) in registers from the P pass to the
// dS pass, so the next query tile's S^T may overwrite the S^T/P^T columns as
// soon as dV has read P^T: it is issued right after dV instead of after dS.
#ifndef JFA_BWD_EARLY_S
#define JFA_BWD_EARLY_S 1
#endif
#ifndef JFA_BWD_EPI_STAGED
#define JFA_BWD_EPI_STAGED 1
#endif
// Who stores an item's dK / dV: 1 = the compute warpgroup (staged through its
// own dS tile, while the next item's K loads), 0 = the dQ warpgroup after the
// item's last dQ reduce (staged per JFA_BWD_EPI_STAGED).  Ads step: 453.9 vs
// 467.4 us.
// With the compute warpgroup's epilogue: whole 128-row tiles of dK/dV leave
// through TMA stores issued by one thread (the warpgroup only stages them;
// ads step 443.1 vs 453.5 us).
#ifndef JFA_BWD_EPI_TMA
#define JFA_BWD_EPI_TMA 1
#endif
#ifndef JFA_BWD_EPI_ON_COMPUTE
#define JFA_BWD_EPI_ON_COMPUTE 1
#endif

// Compute warpgroups: 1 = one warpgroup computes every query column of its
// key rows; 2 = two warpgroups, 64 columns each (and one dK/dV store each).
#ifndef JFA_BWD_COMPUTE_WGS
#define JFA_BWD_COMPUTE_WGS 2
#endif
constexpr int kCW = JFA_BWD_COMPUTE_WGS;
static_assert(kCW == 1 || kCW == 2, "one or two compute warpgroups");
// (kCW + 2) warpgroups: compute, dQ, and load + MMA + two idle warps.
// Registers move from the load/MMA warpgroup to the others, never beyond the
// launch budget: one compute warpgroup 384 x 168 = 64,512 =
// 128 x (192 + 168 + 144); two, 512 x 128 = 65,536 = 128 x (2 x 120 + 160 + 112).
constexpr int kBwdThreads = 128 * (kCW + 2);
constexpr uint32_t kLaunchRegs = kCW == 1 ? 168 : 128;
// Registers per thread of each warpgroup with two compute warpgroups.
#ifndef JFA_BWD_CW2_CREGS
#define JFA_BWD_CW2_CREGS 120
#endif
#ifndef JFA_BWD_CW2_DQREGS
#define JFA_BWD_CW2_DQREGS 160
#endif
#ifndef JFA_BWD_CW2_AREGS
#define JFA_BWD_CW2_AREGS 112
#endif
constexpr uint32_t kComputeRegs = kCW == 1 ? 192 : JFA_BWD_CW2_CREGS;
constexpr uint32_t kDqRegs = kCW == 1 ? 168 : JFA_BWD_CW2_DQREGS;
constexpr uint32_t kAuxRegs = kCW == 1 ? 144 : JFA_BWD_CW2_AREGS;
static_assert(128 * (kCW * kComputeRegs + kDqRegs + kAuxRegs) <= kBwdThreads * kLaunchRegs,
              "register split exceeds launch");
constexpr int kWarpDq = 4 * kCW;        // first warp of the dQ warpgroup
constexpr int kWarpLoad = 4 * kCW + 4;
constexpr int kWarpMma = 4 * kCW + 5;
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct BwdLayout {
    static constexpr int kSlabBytes = 16384;
    static constexpr int kSlabs = D / 64;
    static constexpr int kTileBytes = kSlabs * kSlabBytes;
    static constexpr int kK = 0;
    static constexpr int kV = kTileBytes;
    static constexpr int kQ = 2 * kTileBytes;   // two stages
    static constexpr int kDO = 4 * kTileBytes;  // one stage
    static constexpr int kDS = 5 * kTileBytes;  // 128 x 128 bf16 = 32 KB
    static constexpr int kDQ = kDS + 32768;     // two stages of 128 x 16 fp32
    static constexpr int kDQStage = 128 * 16 * 4;
    static constexpr int kStats = kDQ + 2 * kDQStage;  // two stages of {lse2[128], delta[128]}
    static constexpr int kBytes = kStats + 2 * 1024;
    static constexpr int kDynSmem = kBytes + 1024;
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kColS = 0, kColDP = 128, kColDK = 256, kColDV = 256 + D;
};

struct BwdBars {
    uint64_t k_full, k_empty, v_full, v_empty;
    uint64_t q_full[2], q_empty[2];
    uint64_t do_full, do_empty;
    uint64_t s_full, dp_full, p_full, ds_full, ds_empty;
    uint64_t dq_full, dq_empty;
    uint64_t dkv_full, dv_empty, dk_empty, ds_free;
    uint64_t mma_done;
    uint32_t tmem_base;
    uint32_t abort_flag;
};

struct BwdItem {
    int b, h, kv_start, Lk, n, q_row0, o_row0, q_rows, i0, i1;
};

__device__ __forceinline__ BwdItem decode_bwd(const WorkItem& w, const BwdParams& p) {
    BwdItem it;
    it.b = w.b;
    it.kv_start = w.kv_start;
    it.Lk = w.kv_len;
    it.h = static_cast<int>(w.packed & 0xFFu);
    it.n = static_cast<int>((w.packed >> 8) & 0x7FFFFFu);
    it.q_row0 = p.broadcast_q ? 0 : w.kv_start;
    it.o_row0 = p.broadcast_q ? w.b * p.Lq : w.kv_start;
    it.q_rows = p.broadcast_q ? p.Lq : w.kv_len;
    it.i0 = p.causal ? it.n : 0;
    it.i1 = (it.q_rows + 127) / 128;
    return it;
}

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
    return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Uniform decision across the 128 threads of named barrier `id`.
__device__ __forceinline__ bool group_all(int id, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, %2, 128, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}\n"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(pred)), "r"(id)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ void group_sync(int id) { asm volatile("bar.sync %0, 128;" ::"r"(id) : "memory"); }

// Barrier over compute warpgroup wg (ids 2 and 3; the dQ warpgroup uses id 1).
__device__ __forceinline__ void compute_sync(int wg) { asm volatile("bar.sync %0, 128;" ::"r"(2 + wg) : "memory"); }

// Operand descriptors are built once per buffer; each MMA adds a
// compile-time offset (16-byte units) so the issuing thread stays lean.
__device__ __forceinline__ uint64_t kmajor_desc(uint32_t saddr) { return smem_desc(saddr, 16, 1024); }
__device__ __forceinline__ uint64_t mnmajor_desc(uint32_t saddr) { return smem_desc(saddr, 16384, 1024); }

// C(tmem) = A B^T with both operands K-major [rows][D] (S^T = K Q^T, dP^T = V dO^T).
template <int D>
__device__ __forceinline__ void issue_kmajor(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc) {
    constexpr uint32_t idesc = idesc_bf16_f32(128, 128, 0, 0);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
        const uint64_t off = ((kk / 4) * 16384 + (kk % 4) * 32) / 16;
        mma_ss(d_tmem, a_desc + off, b_desc + off, idesc, kk > 0);
    }
}

// dV (+)= P^T dO: A = P^T from TMEM (bf16 pairs), B = dO_i [q][D] MN-major.
// TMEM column of P^T for K step kk (16 queries = 8 columns of bf16 pairs):
// packed from column 0 with one compute warpgroup, each 32-query chunk over
// its own S^T columns with two.
__device__ __forceinline__ constexpr uint32_t p_col(int kk) {
    return kCW == 1 ? static_cast<uint32_t>(kk * 8) : static_cast<uint32_t>((kk / 2) * 32 + (kk % 2) * 8);
}

template <int D>
__device__ __forceinline__ void issue_dv(uint32_t d_tmem, uint32_t p_tmem, uint64_t do_desc, uint32_t acc) {
    constexpr uint32_t idesc = idesc_bf16_f32(128, D, 0, 1);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) mma_ts(d_tmem, p_tmem + p_col(kk), do_desc + kk * (2048 / 16), idesc, (acc | kk) != 0);
}

// dK (+)= dS^T Q: A = dS^T [key][q] K-major (smem), B = Q_i [q][D] MN-major.
template <int D>
__device__ __forceinline__ void issue_dk(uint32_t d_tmem, uint64_t ds_desc_k, uint64_t q_desc_mn, uint32_t acc) {
    constexpr uint32_t idesc = idesc_bf16_f32(128, D, 0, 1);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        const uint64_t aoff = ((kk / 4) * 16384 + (kk % 4) * 32) / 16;
        mma_ss(d_tmem, ds_desc_k + aoff, q_desc_mn + kk * (2048 / 16), idesc, (acc | kk) != 0);
    }
}

// dQ = dS K: A = dS [q][key] read MN-major from the dS^T buffer, B = K [key][D] MN-major.
template <int D>
__device__ __forceinline__ void issue_dq(uint32_t d_tmem, uint64_t ds_desc_mn, uint64_t k_desc_mn) {
    constexpr uint32_t idesc = idesc_bf16_f32(128, D, 1, 1);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) mma_ss(d_tmem, ds_desc_mn + kk * (2048 / 16), k_desc_mn + kk * (2048 / 16), idesc, kk > 0);
}

// LSE (as log2; -inf rows become +inf so P = 0) and Delta of queries
// 128*i + 4*lane .. +3 of item `it` (out-of-range queries: +inf and 0).
__device__ __forceinline__ void load_stats(const BwdParams& p, const BwdItem& it, int i, int lane, float (&l2)[4],
                                           float (&dl)[4]) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const int qi = 128 * i + lane * 4 + e;
        l2[e] = INFINITY;
        dl[e] = 0.0f;
        if (qi < it.q_rows) {
            const int64_t si = p.broadcast_q ? (static_cast<int64_t>(it.b) * p.H + it.h) * p.Lq + qi
                                             : static_cast<int64_t>(it.h) * p.N + it.q_row0 + qi;
            const float lv = p.lse[si];
            l2[e] = lv == -INFINITY ? INFINITY : lv * kLog2e;
            dl[e] = p.delta[si];
        }
    }
}

// ---------------------------------------------------------------------------
// Load warp (all 32 lanes: lane 0 issues TMA, every lane stages statistics).
// ---------------------------------------------------------------------------
template <int D>
__device__ void bwd_load_role(const BwdParams& p, const BwdMaps* m, uint8_t* smem, BwdBars& bars, int ib, int ie,
                              const AbortState& ab) {
    using L = BwdLayout<D>;
    const int lane = threadIdx.x % 32;
    if (lane == 0) {
        prefetch_tensormap(&m->q);
        prefetch_tensormap(&m->k);
        prefetch_tensormap(&m->v);
        prefetch_tensormap(&m->dout);
    }
    uint32_t k_cnt = 0, v_cnt = 0, q_cnt = 0, do_cnt = 0;
    // Broadcast Q: the (head, query tile) each Q stage holds, so a tile that
    // is already resident is not loaded again (the statistics still are).
    // Key = head << 16 | tile (tiles < 2^16 since Lq <= 2^23); -1 = empty.
    int stage_key0 = -1, stage_key1 = -1;
    for (int idx = ib; idx < ie; ++idx) {
        const BwdItem it = decode_bwd(p.items[idx], p);
        const int kv_row = it.kv_start + 128 * it.n;
        if (lane == 0) JFA_TRACE_EVENT(1, 8, idx, 0);
        if (!mbar_wait_warp(&bars.k_empty, (k_cnt & 1) ^ 1, ab)) goto done;
        if (lane == 0) JFA_TRACE_EVENT(2, 8, idx, 0);
        if (lane == 0) {
            mbar_arrive_expect_tx(&bars.k_full, L::kTileBytes);
#pragma unroll
            for (int s = 0; s < L::kSlabs; ++s)
                tma_load_2d(smem + L::kK + s * L::kSlabBytes, &m->k, &bars.k_full, it.h * D + 64 * s, kv_row);
        }
        ++k_cnt;
        if (!mbar_wait_warp(&bars.v_empty, (v_cnt & 1) ^ 1, ab)) goto done;
        if (lane == 0) {
            mbar_arrive_expect_tx(&bars.v_full, L::kTileBytes);
#pragma unroll
            for (int s = 0; s < L::kSlabs; ++s)
                tma_load_2d(smem + L::kV + s * L::kSlabBytes, &m->v, &bars.v_full, it.h * D + 64 * s, kv_row);
        }
        ++v_cnt;
        if (lane == 0) JFA_TRACE_EVENT(3, 8, idx, 0);
        if (JFA_BWD_PREFETCH && lane == 0 && idx + 1 < ie) {  // next item's K, V, Q, dO tiles into L2 (after this item's loads)
            const BwdItem nx = decode_bwd(p.items[idx + 1], p);
#pragma unroll
            for (int s = 0; s < L::kSlabs; ++s) {
                tma_prefetch_2d(&m->k, nx.h * D + 64 * s, nx.kv_start + 128 * nx.n);
                tma_prefetch_2d(&m->v, nx.h * D + 64 * s, nx.kv_start + 128 * nx.n);
                for (int i = nx.i0; i < nx.i1; ++i) {
                    tma_prefetch_2d(&m->dout, nx.h * D + 64 * s, nx.o_row0 + 128 * i);
                    if (!p.broadcast_q) tma_prefetch_2d(&m->q, nx.h * D + 64 * s, nx.q_row0 + 128 * i);
                }
            }
        }

        for (int i = it.i0; i < it.i1; ++i) {
            const int st = q_cnt % 2;
            if (!mbar_wait_warp(&bars.q_empty[st], ((q_cnt / 2) & 1) ^ 1, ab)) goto done;
            // LSE_i (as log2) and Delta_i for the 128 queries of the tile.
            // (Loading them a tile ahead measured slower: they stay in L2.)
            float* lse2 = reinterpret_cast<float*>(smem + L::kStats + st * 1024);
            float* delta = lse2 + 128;
            float l2[4], dl[4];
            load_stats(p, it, i, lane, l2, dl);
            *reinterpret_cast<float4*>(lse2 + lane * 4) = make_float4(l2[0], l2[1], l2[2], l2[3]);
            *reinterpret_cast<float4*>(delta + lane * 4) = make_float4(dl[0], dl[1], dl[2], dl[3]);
            __syncwarp();
            const int key = (it.h << 16) | i;
            if (p.broadcast_q && (st == 0 ? stage_key0 : stage_key1) == key) {
                if (lane == 0) mbar_arrive(&bars.q_full[st]);  // Q_i already resident: statistics only
            } else {
                if (lane == 0) {
                    mbar_arrive_expect_tx(&bars.q_full[st], L::kTileBytes);
#pragma unroll
                    for (int s = 0; s < L::kSlabs; ++s)
                        tma_load_2d(smem + L::kQ + st * L::kTileBytes + s * L::kSlabBytes, &m->q, &bars.q_full[st],
                                    it.h * D + 64 * s, it.q_row0 + 128 * i);
                }
                if (st == 0)
                    stage_key0 = key;
                else
                    stage_key1 = key;
            }
            ++q_cnt;
            if (lane == 0) JFA_TRACE_EVENT(4, 8, i, 0);
            if (!mbar_wait_warp(&bars.do_empty, (do_cnt & 1) ^ 1, ab)) goto done;
            if (lane == 0) {
                mbar_arrive_expect_tx(&bars.do_full, L::kTileBytes);
#pragma unroll
                for (int s = 0; s < L::kSlabs; ++s)
                    tma_load_2d(smem + L::kDO + s * L::kSlabBytes, &m->dout, &bars.do_full, it.h * D + 64 * s,
                                it.o_row0 + 128 * i);
            }
            ++do_cnt;
            if (lane == 0) JFA_TRACE_EVENT(5, 8, i, 0);
        }
    }
done:
    // Let every issued copy land before the CTA can exit.
    if (lane == 0) {
        if (k_cnt) mbar_wait_drain(&bars.k_full, (k_cnt - 1) & 1);
        if (v_cnt) mbar_wait_drain(&bars.v_full, (v_cnt - 1) & 1);
        for (uint32_t c = q_cnt > 2 ? q_cnt - 2 : 0; c < q_cnt; ++c) mbar_wait_drain(&bars.q_full[c % 2], (c / 2) & 1);
        if (do_cnt) mbar_wait_drain(&bars.do_full, (do_cnt - 1) & 1);
    }
    __syncwarp();
}

// ---------------------------------------------------------------------------
// MMA issuer (one thread).
// ---------------------------------------------------------------------------
template <int D>
__device__ void bwd_mma_role(const BwdParams& p, uint8_t* smem, BwdBars& bars, uint32_t tmem, int ib, int ie,
                             const AbortState& ab) {
    using L = BwdLayout<D>;
    const uint64_t dK_k = kmajor_desc(smem_u32(smem + L::kK)), dK_mn = mnmajor_desc(smem_u32(smem + L::kK));
    const uint64_t dV_k = kmajor_desc(smem_u32(smem + L::kV));
    const uint64_t dQ_k = kmajor_desc(smem_u32(smem + L::kQ)), dQ_mn = mnmajor_desc(smem_u32(smem + L::kQ));
    const uint64_t dDO_k = kmajor_desc(smem_u32(smem + L::kDO)), dDO_mn = mnmajor_desc(smem_u32(smem + L::kDO));
    const uint64_t dDS_k = kmajor_desc(smem_u32(smem + L::kDS)), dDS_mn = mnmajor_desc(smem_u32(smem + L::kDS));
    constexpr uint64_t kTileUnits = L::kTileBytes / 16;
    uint32_t it_cnt = 0, q_cnt = 0, tile_cnt = 0;
    for (int idx = ib; idx < ie; ++idx) {
        const BwdItem it = decode_bwd(p.items[idx], p);
        JFA_TRACE_EVENT(10, 9, idx, 0);
        if (!mbar_wait(&bars.k_full, it_cnt & 1, ab)) goto done;
        JFA_TRACE_EVENT(11, 9, idx, 0);
        if (!mbar_wait(&bars.v_full, it_cnt & 1, ab)) goto done;
        JFA_TRACE_EVENT(12, 9, idx, 0);
        // S^T of the first query tile; later tiles' S^T are issued as soon as
        // the previous tile's dS^T is written (before its dK and dQ), so the
        // compute warps can start the next P while the tensor core finishes
        // dK and dQ of this tile.
        {
            const int st = q_cnt % 2;
            if (!mbar_wait(&bars.q_full[st], (q_cnt / 2) & 1, ab)) goto done;
            JFA_TRACE_EVENT(13, 9, it.i0, 0);
            tc_fence_after();
            issue_kmajor<D>(tmem + L::kColS, dK_k, dQ_k + st * kTileUnits);  // S^T = K Q^T
            mma_commit(&bars.s_full);
        }
        for (int i = it.i0; i < it.i1; ++i) {
            const int st = q_cnt % 2;
            if (!mbar_wait(&bars.do_full, tile_cnt & 1, ab)) goto done;
            JFA_TRACE_EVENT(15, 9, i, 0);
            if (!mbar_wait(&bars.dq_empty, (tile_cnt & 1) ^ 1, ab)) goto done;  // previous dQ read out
            JFA_TRACE_EVENT(16, 9, i, 0);
            tc_fence_after();
            issue_kmajor<D>(tmem + L::kColDP, dV_k, dDO_k);  // dP^T = V dO^T
            mma_commit(&bars.dp_full);
            if (i == it.i1 - 1) mma_commit(&bars.v_empty);
            if (i == it.i0) {  // the previous item's dV has been read out of TMEM
                if (!mbar_wait(&bars.dv_empty, (it_cnt & 1) ^ 1, ab)) goto done;
                JFA_TRACE_EVENT(18, 9, i, 0);
            }
            if (!mbar_wait(&bars.p_full, tile_cnt & 1, ab)) goto done;
            JFA_TRACE_EVENT(19, 9, i, 0);
            tc_fence_after();
            issue_dv<D>(tmem + L::kColDV, tmem + L::kColS, dDO_mn, i > it.i0);
            mma_commit(&bars.do_empty);
            if (JFA_BWD_EARLY_S && i + 1 < it.i1) {  // next tile's S^T right behind dV (which reads P^T first)
                const int st2 = (q_cnt + 1) % 2;
                if (!mbar_wait(&bars.q_full[st2], ((q_cnt + 1) / 2) & 1, ab)) goto done;
                tc_fence_after();
                issue_kmajor<D>(tmem + L::kColS, dK_k, dQ_k + st2 * kTileUnits);
                mma_commit(&bars.s_full);
            }
            if (!mbar_wait(&bars.ds_full, tile_cnt & 1, ab)) goto done;
            JFA_TRACE_EVENT(20, 9, i, 0);
            if (!JFA_BWD_EARLY_S && i + 1 < it.i1) {  // next tile's S^T: T_S is free (P^T read by dV and by the dS pass)
                const int st2 = (q_cnt + 1) % 2;
                if (!mbar_wait(&bars.q_full[st2], ((q_cnt + 1) / 2) & 1, ab)) goto done;
                tc_fence_after();
                issue_kmajor<D>(tmem + L::kColS, dK_k, dQ_k + st2 * kTileUnits);
                mma_commit(&bars.s_full);
            }
            if (i == it.i0) {  // ... and its dK
                if (!mbar_wait(&bars.dk_empty, (it_cnt & 1) ^ 1, ab)) goto done;
            }
            tc_fence_after();
            if ((JFA_BWD_DQ_FIRST && i == it.i1 - 1) || JFA_BWD_DQ_FIRST == 2) {
                // dQ first: on the last tile K can then be released (and the next
                // item's K loaded) while dK runs; on every tile (mode 2) the dQ
                // readout, and with it the next dP^T, comes one product sooner.
                issue_dq<D>(tmem + L::kColDP, dDS_mn, dK_mn);
                mma_commit(&bars.dq_full);
                if (i == it.i1 - 1) mma_commit(&bars.k_empty);
                issue_dk<D>(tmem + L::kColDK, dDS_k, dQ_mn + st * kTileUnits, i > it.i0);
                mma_commit(&bars.q_empty[st]);
                mma_commit(&bars.ds_empty);
            } else {
                issue_dk<D>(tmem + L::kColDK, dDS_k, dQ_mn + st * kTileUnits, i > it.i0);
                mma_commit(&bars.q_empty[st]);
                issue_dq<D>(tmem + L::kColDP, dDS_mn, dK_mn);
                mma_commit(&bars.dq_full);
                mma_commit(&bars.ds_empty);
            }
            ++q_cnt;
            ++tile_cnt;
        }
        mma_commit(&bars.dkv_full);
        if (!JFA_BWD_DQ_FIRST) mma_commit(&bars.k_empty);
        ++it_cnt;
    }
done:
    mma_commit(&bars.mma_done);
    mbar_wait_drain(&bars.mma_done, 0);
}

// ---------------------------------------------------------------------------
// Compute warpgroup: P^T into TMEM, dS^T into shared memory.
// ---------------------------------------------------------------------------
template <int D, bool kMask>
__device__ __forceinline__ void bwd_compute_p(const BwdParams& p, const float* lse2, uint32_t s_addr, int key,
                                              int qbase, int q_rows, bool row_valid, uint32_t (&pkeep)[64]) {
    // All 128 scores of this key row in one batch of TMEM loads, one wait.
    uint32_t sr[4][32];
#pragma unroll
    for (int c = 0; c < 4; ++c) tmem_ld32(s_addr + c * 32, sr[c]);
    tmem_ld_wait();
    // Queries qbase .. qbase + nvis - 1 see this key (sequence end, causal bound).
    int nvis = 128;
    if (kMask) {
        nvis = row_valid ? min(128, q_rows - qbase) : 0;
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        uint32_t pk[16];
        float l2[32];  // the 32 queries' log2-LSE, read 4 at a time (same address for every thread)
#pragma unroll
        for (int v = 0; v < 8; ++v) {
            const float4 f = reinterpret_cast<const float4*>(lse2)[c * 8 + v];
            l2[4 * v] = f.x;
            l2[4 * v + 1] = f.y;
            l2[4 * v + 2] = f.z;
            l2[4 * v + 3] = f.w;
        }
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            const int q0 = c * 32 + 2 * e;
            float x0, x1;
            ffma2(x0, x1, __uint_as_float(sr[c][2 * e]), __uint_as_float(sr[c][2 * e + 1]), p.scale_log2,
                  p.scale_log2, -l2[2 * e], -l2[2 * e + 1]);
            float p0, p1;
            if (!kMask && poly_pair<JFA_BWD_POLY_PAIRS>(e)) {  // part of the exponentials on the FMA pipe (no -inf here)
                exp2_fma2(x0, x1, p0, p1);
            } else {
                p0 = ex2_approx(x0);
                p1 = ex2_approx(x1);
            }
            if (kMask) {
                if (q0 >= nvis || (p.causal && key > qbase + q0)) p0 = 0.0f;
                if (q0 + 1 >= nvis || (p.causal && key > qbase + q0 + 1)) p1 = 0.0f;
            }
            pk[e] = pack_bf16x2(p0, p1);
            pkeep[c * 16 + e] = pk[e];
        }
        tmem_st16(s_addr + c * 16, pk);
    }
    tmem_st_wait();
}

// Two compute warpgroups: warpgroup g owns query columns 64g .. 64g+63 of
// every key row (32-column chunks c0 = 2g and c0 + 1).  One chunk of S^T is
// in registers at a time and the log2-LSE values are read 4 at a time, so a
// thread needs about half the registers of the one-warpgroup pass.  The two
// warpgroups run concurrently, so chunk c's P^T (16 columns of bf16 pairs)
// goes over the first half of chunk c's own S^T columns (c * 32), never over
// S^T columns the other warpgroup may not have read yet; the dV product
// reads it from there (p_col()).
template <int D, bool kMask>
__device__ __forceinline__ void bwd_compute_p_cols(const BwdParams& p, const float* lse2, uint32_t s_addr, int key,
                                                   int qbase, int q_rows, bool row_valid, int c0,
                                                   uint32_t (&pkeep)[32]) {
    int nvis = 128;
    if (kMask) nvis = row_valid ? min(128, q_rows - qbase) : 0;
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
        const int c = c0 + cc;
        uint32_t sr[32];
        tmem_ld32(s_addr + c * 32, sr);
        tmem_ld_wait();
        uint32_t pk[16];
#pragma unroll
        for (int e2 = 0; e2 < 8; ++e2) {
            const float4 f = reinterpret_cast<const float4*>(lse2)[c * 8 + e2];  // queries c*32 + 4*e2 .. +3
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int e = 2 * e2 + h;
                const int q0 = c * 32 + 2 * e;
                float x0, x1;
                ffma2(x0, x1, __uint_as_float(sr[2 * e]), __uint_as_float(sr[2 * e + 1]), p.scale_log2, p.scale_log2,
                      -(h ? f.z : f.x), -(h ? f.w : f.y));
                float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
                if (kMask) {
                    if (q0 >= nvis || (p.causal && key > qbase + q0)) p0 = 0.0f;
                    if (q0 + 1 >= nvis || (p.causal && key > qbase + q0 + 1)) p1 = 0.0f;
                }
                pk[e] = pack_bf16x2(p0, p1);
                pkeep[cc * 16 + e] = pk[e];
            }
        }
        tmem_st16(s_addr + c * 32, pk);  // over the first half of its own S^T chunk
    }
    tmem_st_wait();
}

// dS^T for warpgroup g's 64 query columns (slab g of the dS^T tile).
template <int D>
__device__ __forceinline__ void bwd_compute_ds_cols(const float* delta, uint32_t dp_addr, uint8_t* ds_tile, int row,
                                                    int c0, const uint32_t (&pkeep)[32]) {
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
        const int c = c0 + cc;
        uint32_t dp[32];
        tmem_ld32(dp_addr + c * 32, dp);
        tmem_ld_wait();
        uint32_t pk[16];
#pragma unroll
        for (int e2 = 0; e2 < 8; ++e2) {
            const float4 f = reinterpret_cast<const float4*>(delta)[c * 8 + e2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int e = 2 * e2 + h;
                const float d0 = bf16lo_to_f32(pkeep[cc * 16 + e]) * (__uint_as_float(dp[2 * e]) - (h ? f.z : f.x));
                const float d1 = bf16hi_to_f32(pkeep[cc * 16 + e]) * (__uint_as_float(dp[2 * e + 1]) - (h ? f.w : f.y));
                pk[e] = pack_bf16x2(d0, d1);
            }
        }
        uint8_t* slab = ds_tile + (c / 2) * 16384 + row * 128;
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            const int chunk = ((c % 2) * 4 + v) ^ (row % 8);
            *reinterpret_cast<uint4*>(slab + chunk * 16) = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
        }
    }
}

// dS^T from dP^T (TMEM, 32 columns at a time) and P kept in registers.
template <int D>
__device__ __forceinline__ void bwd_compute_ds_regs(const float* delta, uint32_t dp_addr, uint8_t* ds_tile, int row,
                                                    const uint32_t (&pkeep)[64]) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        uint32_t dp[32];
        tmem_ld32(dp_addr + c * 32, dp);
        float dl[32];  // Delta of the 32 queries, read 4 at a time
#pragma unroll
        for (int v = 0; v < 8; ++v) {
            const float4 f = reinterpret_cast<const float4*>(delta)[c * 8 + v];
            dl[4 * v] = f.x;
            dl[4 * v + 1] = f.y;
            dl[4 * v + 2] = f.z;
            dl[4 * v + 3] = f.w;
        }
        tmem_ld_wait();
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            const float d0 = bf16lo_to_f32(pkeep[c * 16 + e]) * (__uint_as_float(dp[2 * e]) - dl[2 * e]);
            const float d1 = bf16hi_to_f32(pkeep[c * 16 + e]) * (__uint_as_float(dp[2 * e + 1]) - dl[2 * e + 1]);
            pk[e] = pack_bf16x2(d0, d1);
        }
        uint8_t* slab = ds_tile + (c / 2) * 16384 + row * 128;
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            const int chunk = ((c % 2) * 4 + v) ^ (row % 8);
            *reinterpret_cast<uint4*>(slab + chunk * 16) = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
        }
    }
}

template <int D>
__device__ __forceinline__ void bwd_compute_ds(const float* delta, uint32_t s_addr, uint32_t dp_addr, uint8_t* ds_tile,
                                               int row) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {  // two halves of 64 queries: one TMEM wait each
        uint32_t dp[2][32], pp[2][16];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            tmem_ld32(dp_addr + (2 * h + u) * 32, dp[u]);
            tmem_ld16(s_addr + (2 * h + u) * 16, pp[u]);
        }
        tmem_ld_wait();
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int c = 2 * h + u;
            uint32_t pk[16];
            float dl[32];  // Delta of the 32 queries, read 4 at a time
#pragma unroll
            for (int v = 0; v < 8; ++v) {
                const float4 f = reinterpret_cast<const float4*>(delta)[c * 8 + v];
                dl[4 * v] = f.x;
                dl[4 * v + 1] = f.y;
                dl[4 * v + 2] = f.z;
                dl[4 * v + 3] = f.w;
            }
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const float d0 = bf16lo_to_f32(pp[u][e]) * (__uint_as_float(dp[u][2 * e]) - dl[2 * e]);
                const float d1 = bf16hi_to_f32(pp[u][e]) * (__uint_as_float(dp[u][2 * e + 1]) - dl[2 * e + 1]);
                pk[e] = pack_bf16x2(d0, d1);
            }
            // Row `row`, queries c*32 .. c*32+31: slab c/2, 16-byte chunks (c%2)*4 .. +3,
            // stored at chunk ^ (row % 8) (128-byte swizzle, as TMA would place them).
            uint8_t* slab = ds_tile + (c / 2) * 16384 + row * 128;
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                const int chunk = ((c % 2) * 4 + v) ^ (row % 8);
                *reinterpret_cast<uint4*>(slab + chunk * 16) =
                    make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
            }
        }
    }
}

// Hand-off to the MMA thread after a warpgroup's tcgen05 / shared-memory
// writes (already fenced for the async proxy where needed): every thread
// fences, then every thread arrives or, with JFA_BWD_WARP_ARRIVE, lane 0 of
// each warp once the warp has synchronised.
constexpr uint32_t kArrivePerWarp = JFA_BWD_WARP_ARRIVE ? 1 : 32;  // arrivals per warp
__device__ __forceinline__ void handoff_arrive(uint64_t* bar) {
    tc_fence_before();
    if (JFA_BWD_WARP_ARRIVE) {
        __syncwarp();
        if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
    } else {
        mbar_arrive(bar);
    }
}

template <int D>
__device__ void bwd_compute_role(const BwdParams& p, const BwdMaps* maps, uint8_t* smem, BwdBars& bars,
                                 uint32_t tmem, int ib, int ie, const AbortState& ab) {
    using L = BwdLayout<D>;
    const int row = threadIdx.x % 128;  // key row = TMEM lane
    const int wg = threadIdx.x / 128;   // compute warpgroup (its query columns with two)
    const uint32_t lane_off = static_cast<uint32_t>(((threadIdx.x / 32) % 4) * 32) << 16;
    const uint32_t s_addr = tmem + lane_off + L::kColS;
    const uint32_t dp_addr = tmem + lane_off + L::kColDP;
    uint8_t* ds_tile = smem + L::kDS;
    uint32_t q_cnt = 0, tile_cnt = 0, item_cnt = 0;
    for (int idx = ib; idx < ie; ++idx, ++item_cnt) {
        const BwdItem it = decode_bwd(p.items[idx], p);
        const int key = 128 * it.n + row;
        const bool row_valid = key < it.Lk;
        const bool kv_full_tile = 128 * (it.n + 1) <= it.Lk;
        if (threadIdx.x == 0) JFA_TRACE_EVENT(30, 0, idx, 0);
        for (int i = it.i0; i < it.i1; ++i) {
            const int st = q_cnt % 2;
            const float* lse2 = reinterpret_cast<const float*>(smem + L::kStats + st * 1024);
            const float* delta = lse2 + 128;
            if (!mbar_wait_warp(&bars.q_full[st], (q_cnt / 2) & 1, ab)) goto done;
            if (!mbar_wait_warp(&bars.s_full, tile_cnt & 1, ab)) goto done;
            if (threadIdx.x == 0) JFA_TRACE_EVENT(31, 0, i, 0);
            tc_fence_after();
            const bool unmasked = kv_full_tile && 128 * (i + 1) <= it.q_rows && !(p.causal && i == it.n);
            uint32_t pkeep[kCW == 1 ? 64 : 32];
            if constexpr (kCW == 1) {
                if (unmasked)
                    bwd_compute_p<D, false>(p, lse2, s_addr, key, 128 * i, it.q_rows, row_valid, pkeep);
                else
                    bwd_compute_p<D, true>(p, lse2, s_addr, key, 128 * i, it.q_rows, row_valid, pkeep);
            } else {
                if (unmasked)
                    bwd_compute_p_cols<D, false>(p, lse2, s_addr, key, 128 * i, it.q_rows, row_valid, 2 * wg, pkeep);
                else
                    bwd_compute_p_cols<D, true>(p, lse2, s_addr, key, 128 * i, it.q_rows, row_valid, 2 * wg, pkeep);
            }
            if (threadIdx.x == 0) JFA_TRACE_EVENT(32, 0, i, 0);
            handoff_arrive(&bars.p_full);
            if (!mbar_wait_warp(&bars.dp_full, tile_cnt & 1, ab)) goto done;
            if (threadIdx.x == 0) JFA_TRACE_EVENT(33, 0, i, 0);
            if (!mbar_wait_warp(&bars.ds_empty, (tile_cnt & 1) ^ 1, ab)) goto done;
            if (!JFA_BWD_EPI_ON_COMPUTE && JFA_BWD_EPI_STAGED && i == it.i0) {  // the previous item's dK/dV staging has left the buffer
                if (!mbar_wait_warp(&bars.ds_free, (item_cnt & 1) ^ 1, ab)) goto done;
            }
            if (threadIdx.x == 0) JFA_TRACE_EVENT(34, 0, i, 0);
            tc_fence_after();
            if (JFA_BWD_EPI_ON_COMPUTE && JFA_BWD_EPI_TMA && i == it.i0) {  // the last item's dK/dV stores have read the tile
                if (row == 0) bulk_wait_group_read<0>();
                compute_sync(wg);
            }
            if constexpr (kCW == 2) {
                bwd_compute_ds_cols<D>(delta, dp_addr, ds_tile, row, 2 * wg, pkeep);
            } else {
                if (JFA_BWD_EARLY_S)
                    bwd_compute_ds_regs<D>(delta, dp_addr, ds_tile, row, pkeep);
                else
                    bwd_compute_ds<D>(delta, s_addr, dp_addr, ds_tile, row);
            }
            fence_proxy_async_smem();
            if (threadIdx.x == 0) JFA_TRACE_EVENT(35, 0, i, 0);
            handoff_arrive(&bars.ds_full);
            ++q_cnt;
            ++tile_cnt;
        }
        if (JFA_BWD_EPI_ON_COMPUTE) {
            // This item's dK / dV, while the next item's K tile loads: once
            // every product of the item is done (dkv_full, which also means
            // the last dK / dQ have read dS), 64-column halves go TMEM ->
            // registers -> 128-byte-swizzled stage in the dS tile -> coalesced
            // row copies (a warp store covers 4 whole lines; rows past the
            // sequence end are skipped).  Each accumulator's columns are
            // released after its last half is read.
            if (!mbar_wait_warp(&bars.dkv_full, item_cnt & 1, ab)) goto done;
            if (threadIdx.x == 0) JFA_TRACE_EVENT(36, 0, idx, 0);
            tc_fence_after();
            const int rows_valid = min(128, it.Lk - 128 * it.n);
            const int64_t row0 = static_cast<int64_t>(it.kv_start) + 128 * it.n;
            // Whole tiles leave by TMA stores; a ragged tail tile (which must not
            // touch the next sequence's rows) by coalesced row copies.
            const bool tma_ok = JFA_BWD_EPI_TMA && rows_valid == 128;
            if (!tma_ok && JFA_BWD_EPI_TMA) {  // the last item's stores have read the stages
                if (row == 0) bulk_wait_group_read<0>();
                compute_sync(wg);
            }
#pragma unroll
            for (int which = 0; which < 2; ++which) {  // 0: dV, 1: dK (scaled); with two warpgroups, warpgroup `which`
                if (kCW == 2 && which != wg) continue;
                const uint32_t col = which ? L::kColDK : L::kColDV;
                const float sc = which ? p.scale : 1.0f;
                uint16_t* out = which ? p.dk : p.dv;
#pragma unroll
                for (int half = 0; half < D / 64; ++half) {
                    uint32_t v[2][32];
                    tmem_ld32(tmem + lane_off + col + half * 64, v[0]);
                    tmem_ld32(tmem + lane_off + col + half * 64 + 32, v[1]);
                    tmem_ld_wait();
                    if (half == D / 64 - 1) {
                        tc_fence_before();
                        mbar_arrive(which ? &bars.dk_empty : &bars.dv_empty);
                    }
                    // Stage (which * halves + half) % 2: dV's halves, then dK's, alternate
                    // the two 16 KB halves of the dS tile.
                    // (two warpgroups: each its own slab, both halves in turn)
                    uint8_t* stage = ds_tile + (kCW == 2 ? wg : ((which * (D / 64) + half) % 2)) * 16384;
                    if (tma_ok && (kCW == 2 ? half > 0 : which == 1)) {  // the store that used this stage has read it
                        if (row == 0) bulk_wait_group_read<kCW == 2 ? 0 : 1>();
                        compute_sync(wg);
                    }
#pragma unroll
                    for (int ch = 0; ch < 8; ++ch) {
                        const uint32_t* f = &v[ch / 4][(ch % 4) * 8];
                        *reinterpret_cast<uint4*>(stage + row * 128 + ((ch ^ (row & 7)) * 16)) =
                            make_uint4(pack_bf16x2(__uint_as_float(f[0]) * sc, __uint_as_float(f[1]) * sc),
                                       pack_bf16x2(__uint_as_float(f[2]) * sc, __uint_as_float(f[3]) * sc),
                                       pack_bf16x2(__uint_as_float(f[4]) * sc, __uint_as_float(f[5]) * sc),
                                       pack_bf16x2(__uint_as_float(f[6]) * sc, __uint_as_float(f[7]) * sc));
                    }
                    if (tma_ok) {  // whole tile: one TMA store of the 128 x 64 stage
                        fence_proxy_async_smem();
                        compute_sync(wg);
                        if (row == 0) {
                            tma_store_2d(which ? &maps->dk : &maps->dv, stage, it.h * D + half * 64,
                                         static_cast<int>(row0));
                            bulk_commit_group();
                        }
                        continue;
                    }
                    compute_sync(wg);
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const int q = row + 128 * k;
                        const int rr = q >> 3, ch = q & 7;
                        if (rr < rows_valid)
                            *reinterpret_cast<uint4*>(out + ((row0 + rr) * p.H + it.h) * D + half * 64 + ch * 8) =
                                *reinterpret_cast<const uint4*>(stage + rr * 128 + ((ch ^ (rr & 7)) * 16));
                    }
                    compute_sync(wg);
                }
            }
            if (threadIdx.x == 0) JFA_TRACE_EVENT(37, 0, idx, 0);
        }
    }
done:
    if (JFA_BWD_EPI_TMA && row == 0) bulk_wait_group<0>();  // every dK/dV store has completed
}

// ---------------------------------------------------------------------------
// dQ warpgroup: TMEM dQ -> registers (release TMEM) -> two 128x16 fp32 smem
// stages -> TMA bulk reduce-add into global dQ.  Then the item's dK/dV.
// ---------------------------------------------------------------------------
template <int D>
__device__ void bwd_dq_role(const BwdParams& p, const CUtensorMap* map_dq, uint8_t* smem, BwdBars& bars,
                            uint32_t tmem, int ib, int ie, const AbortState& ab) {
    using L = BwdLayout<D>;
    const int r = threadIdx.x - 32 * kWarpDq;  // query row of the tile (TMEM lane)
    const bool issuer = r == 0;
    const uint32_t lane_off = static_cast<uint32_t>(((threadIdx.x / 32) % 4) * 32) << 16;
    const uint32_t dq_addr = tmem + lane_off + L::kColDP;
    uint8_t* stage_base = smem + L::kDQ;
    uint32_t tile_cnt = 0, it_cnt = 0, stage_uses = 0;
    if (issuer) prefetch_tensormap(map_dq);
    for (int idx = ib; idx < ie; ++idx) {
        const BwdItem it = decode_bwd(p.items[idx], p);
        // Broadcast dQ goes to this CTA's partial buffer (group blockIdx % G);
        // a final pass sums the G partials.
        const int dq_row0 = p.broadcast_q ? static_cast<int>(blockIdx.x % p.dq_groups) * p.Lq : it.q_row0;
        for (int i = it.i0; i < it.i1; ++i) {
            bool ok = mbar_wait_warp(&bars.dq_full, tile_cnt & 1, ab);
            if (!group_all(1, ok)) goto done;
            if (issuer) JFA_TRACE_EVENT(41, 4, i, 0);
            tc_fence_after();
            uint32_t v[D / 32][32];
#pragma unroll
            for (int c = 0; c < D / 32; ++c) tmem_ld32(dq_addr + c * 32, v[c]);
            tmem_ld_wait();
            handoff_arrive(&bars.dq_empty);  // early release: the next dP^T/dQ may overwrite these columns
            if (issuer) JFA_TRACE_EVENT(42, 4, i, 0);
#pragma unroll
            for (int sl = 0; sl < D / 16; ++sl) {
                const int st = stage_uses % 2;
                uint8_t* stage = stage_base + st * L::kDQStage;
                if (issuer) bulk_wait_group_read<1>();  // the reduce that last used this stage has read it
                group_sync(1);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    // 64-byte swizzle (what the tensor map declares): chunk k of row r
                    // sits at chunk k ^ ((r >> 1) & 3), which also spreads the banks.
                    const uint32_t* src = &v[sl / 2][(sl % 2) * 16 + k * 4];
                    *reinterpret_cast<float4*>(stage + r * 64 + ((k ^ ((r >> 1) & 3)) * 16)) =
                        make_float4(__uint_as_float(src[0]) * p.scale, __uint_as_float(src[1]) * p.scale,
                                    __uint_as_float(src[2]) * p.scale, __uint_as_float(src[3]) * p.scale);
                }
                fence_proxy_async_smem();
                group_sync(1);
                if (issuer) {
                    tma_reduce_add_2d(map_dq, stage, it.h * D + sl * 16, dq_row0 + 128 * i);
                    bulk_commit_group();
                }
                ++stage_uses;
            }
            if (issuer) JFA_TRACE_EVENT(43, 4, i, 0);
            ++tile_cnt;
        }
        if (JFA_BWD_EPI_ON_COMPUTE) continue;  // the compute warpgroup stores this item's dK / dV
        // dK / dV epilogue in 64-column halves: TMEM -> registers -> the dS
        // tile's smem (free once the item's last dK/dQ products are done;
        // 128-byte swizzle) -> coalesced row copies (each warp store covers
        // four whole 128-byte segments; rows past the sequence end are
        // skipped).  dV's TMEM is released after its last half is read, then
        // dK's, so the next item's products can start; ds_free tells the
        // compute warps when they may write dS again.
        {
            bool ok = mbar_wait_warp(&bars.dkv_full, it_cnt & 1, ab);
            if (!group_all(1, ok)) goto done;
            if (issuer) JFA_TRACE_EVENT(44, 4, idx, 0);
            tc_fence_after();
            uint8_t* ep_stage = smem + L::kDS;  // dK/dV staging: the dS tile is free until ds_free
            const int rows_valid = min(128, it.Lk - 128 * it.n);
            const int64_t row0 = static_cast<int64_t>(it.kv_start) + 128 * it.n;
#pragma unroll
            for (int which = 0; which < 2; ++which) {  // 0: dV, 1: dK (scaled)
                const uint32_t col = which ? L::kColDK : L::kColDV;
                const float sc = which ? p.scale : 1.0f;
                uint16_t* out = which ? p.dk : p.dv;
#pragma unroll
                for (int half = 0; half < D / 64; ++half) {
                    uint32_t v[2][32];
                    tmem_ld32(tmem + lane_off + col + half * 64, v[0]);
                    tmem_ld32(tmem + lane_off + col + half * 64 + 32, v[1]);
                    tmem_ld_wait();
                    if (half == D / 64 - 1) {
                        tc_fence_before();
                        mbar_arrive(which ? &bars.dk_empty : &bars.dv_empty);
                    }
                    if (!JFA_BWD_EPI_STAGED) {
                        if (r < rows_valid) {
                            uint4* dst = reinterpret_cast<uint4*>(out + ((row0 + r) * p.H + it.h) * D + half * 64);
#pragma unroll
                            for (int ch = 0; ch < 8; ++ch) {
                                const uint32_t* f = &v[ch / 4][(ch % 4) * 8];
                                dst[ch] = make_uint4(pack_bf16x2(__uint_as_float(f[0]) * sc, __uint_as_float(f[1]) * sc),
                                                     pack_bf16x2(__uint_as_float(f[2]) * sc, __uint_as_float(f[3]) * sc),
                                                     pack_bf16x2(__uint_as_float(f[4]) * sc, __uint_as_float(f[5]) * sc),
                                                     pack_bf16x2(__uint_as_float(f[6]) * sc, __uint_as_float(f[7]) * sc));
                            }
                        }
                        continue;
                    }
#pragma unroll
                    for (int ch = 0; ch < 8; ++ch) {
                        const uint32_t* f = &v[ch / 4][(ch % 4) * 8];
                        *reinterpret_cast<uint4*>(ep_stage + half * 16384 + r * 128 + ((ch ^ (r & 7)) * 16)) =
                            make_uint4(pack_bf16x2(__uint_as_float(f[0]) * sc, __uint_as_float(f[1]) * sc),
                                       pack_bf16x2(__uint_as_float(f[2]) * sc, __uint_as_float(f[3]) * sc),
                                       pack_bf16x2(__uint_as_float(f[4]) * sc, __uint_as_float(f[5]) * sc),
                                       pack_bf16x2(__uint_as_float(f[6]) * sc, __uint_as_float(f[7]) * sc));
                    }
                    group_sync(1);
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const int q = r + 128 * k;
                        const int rr = q >> 3, ch = q & 7;
                        if (rr < rows_valid)
                            *reinterpret_cast<uint4*>(out + ((row0 + rr) * p.H + it.h) * D + half * 64 + ch * 8) =
                                *reinterpret_cast<const uint4*>(ep_stage + half * 16384 + rr * 128 +
                                                                ((ch ^ (rr & 7)) * 16));
                    }
                    group_sync(1);
                }
            }
            if (JFA_BWD_EPI_STAGED) mbar_arrive(&bars.ds_free);  // the compute warps may write dS again
            if (issuer) JFA_TRACE_EVENT(45, 4, idx, 0);
            ++it_cnt;
        }
    }
done:
    if (issuer) bulk_wait_group<0>();
}

template <int D>
__global__ void __launch_bounds__(kBwdThreads, 1)
    jfa_bwd_kernel(const BwdParams p, const __grid_constant__ BwdMaps maps) {
    using L = BwdLayout<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024(smem_raw);
    __shared__ BwdBars bars;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int ib = p.cta_start[blockIdx.x], ie = p.cta_start[blockIdx.x + 1];
    const AbortState ab{&bars.abort_flag, p.status};

    JFA_TRACE_INIT();
    if (threadIdx.x == 0) {
        bars.abort_flag = 0;
        mbar_init(&bars.k_full, 1);
        mbar_init(&bars.k_empty, 1);
        mbar_init(&bars.v_full, 1);
        mbar_init(&bars.v_empty, 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bars.q_full[s], 1);
            mbar_init(&bars.q_empty[s], 1);
        }
        mbar_init(&bars.do_full, 1);
        mbar_init(&bars.do_empty, 1);
        mbar_init(&bars.s_full, 1);
        mbar_init(&bars.dp_full, 1);
        mbar_init(&bars.p_full, 4 * kCW * kArrivePerWarp);
        mbar_init(&bars.ds_full, 4 * kCW * kArrivePerWarp);
        mbar_init(&bars.ds_empty, 1);
        mbar_init(&bars.dq_full, 1);
        mbar_init(&bars.dq_empty, 4 * kArrivePerWarp);
        mbar_init(&bars.dkv_full, 1);
        mbar_init(&bars.dv_empty, 128);
        mbar_init(&bars.dk_empty, 128);
        mbar_init(&bars.ds_free, 128);
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

    if (warp < kWarpDq) {
        if constexpr (kComputeRegs > kLaunchRegs) regs_inc<kComputeRegs>();
        if constexpr (kComputeRegs < kLaunchRegs) regs_dec<kComputeRegs>();
        bwd_compute_role<D>(p, &maps, smem, bars, tmem, ib, ie, ab);
    } else if (warp < kWarpDq + 4) {
        if constexpr (kDqRegs > kLaunchRegs) regs_inc<kDqRegs>();
        bwd_dq_role<D>(p, &maps.dq, smem, bars, tmem, ib, ie, ab);
    } else {
        regs_dec<kAuxRegs>();
        if (warp == kWarpLoad) {
            bwd_load_role<D>(p, &maps, smem, bars, ib, ie, ab);
        } else if (warp == kWarpMma) {
            if (lane == 0) bwd_mma_role<D>(p, smem, bars, tmem, ib, ie, ab);
            __syncwarp();
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kWarpMma) tmem_dealloc(tmem, L::kTmemCols);
}

// Delta pre-pass shape: 16-byte chunks each lane reads from O and from dO per
// (row, head) pair (ads step: 1 -> 59.3 us, 2 -> 49.4 us, 4 -> 51.3 us), and
// the grid cap in blocks per SM (8 -> 70 us, 16 and 32 alike).
#ifndef JFA_PRE_VEC
#define JFA_PRE_VEC 2
#endif
#ifndef JFA_PRE_BLOCKS_PER_SM
#define JFA_PRE_BLOCKS_PER_SM 16
#endif

// Delta[row] = sum_d dO[row, d] * O[row, d] (fp32), JFA_PRE_VEC 16-byte
// chunks per lane; D / (8 * JFA_PRE_VEC) consecutive lanes own one (row, head)
// pair.
template <int D>
__global__ void __launch_bounds__(256) jfa_bwd_pre_kernel(const PreParams p) {
    constexpr int kVec = JFA_PRE_VEC;
    constexpr int kLanes = D / (8 * kVec);
    const int64_t total = p.rows;
    const int sub = threadIdx.x % kLanes;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * (blockDim.x / kLanes);
    int64_t pair = static_cast<int64_t>(blockIdx.x) * (blockDim.x / kLanes) + threadIdx.x / kLanes;
    // All lanes of a group iterate together so the shuffles below stay converged.
    const int64_t iters = (total + stride - 1) / stride;
    for (int64_t k = 0; k < iters; ++k, pair += stride) {
        float acc = 0.0f;
        const bool in = pair < total;
        if (in) {
            uint4 a[kVec], b[kVec];
#pragma unroll
            for (int u = 0; u < kVec; ++u) {
                a[u] = reinterpret_cast<const uint4*>(p.o + pair * D)[sub * kVec + u];
                b[u] = reinterpret_cast<const uint4*>(p.dout + pair * D)[sub * kVec + u];
            }
#pragma unroll
            for (int u = 0; u < kVec; ++u) {
                const uint32_t aw[4] = {a[u].x, a[u].y, a[u].z, a[u].w}, bw[4] = {b[u].x, b[u].y, b[u].z, b[u].w};
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    acc = fmaf(bf16lo_to_f32(aw[w]), bf16lo_to_f32(bw[w]), acc);
                    acc = fmaf(bf16hi_to_f32(aw[w]), bf16hi_to_f32(bw[w]), acc);
                }
            }
        }
#pragma unroll
        for (int off = kLanes / 2; off > 0; off /= 2) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (in && sub == 0) {
            const int64_t orow = pair / p.H;
            const int h = static_cast<int>(pair % p.H);
            int64_t di;
            if (p.broadcast_q) {
                const int64_t b = orow / p.Lq, i = orow % p.Lq;
                di = (b * p.H + h) * p.Lq + i;
            } else {
                di = static_cast<int64_t>(h) * p.N + orow;
            }
            p.delta[di] = acc;
        }
    }
}

// dq[e] = sum over g of partial[g * n + e] (float4 lanes; n is a multiple of 4).
__global__ void __launch_bounds__(256) jfa_dq_sum_kernel(const float4* __restrict__ partial, float4* __restrict__ dq,
                                                         int64_t n4, int groups) {
    for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < n4;
         e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        float4 acc = partial[e];
        for (int g = 1; g < groups; ++g) {
            const float4 v = partial[g * n4 + e];
            acc.x += v.x;
            acc.y += v.y;
            acc.z += v.z;
            acc.w += v.w;
        }
        dq[e] = acc;
    }
}

template <int D>
cudaError_t launch_bwd_d(const BwdParams& p, const BwdMaps& m, int grid, cudaStream_t s) {
    using L = BwdLayout<D>;
    static bool configured = false;
    if (!configured) {
        // The register split is only safe at exactly kLaunchRegs per thread.
        cudaFuncAttributes fa;
        cudaError_t e = cudaFuncGetAttributes(&fa, jfa_bwd_kernel<D>);
        if (e != cudaSuccess) return e;
        if (fa.numRegs != static_cast<int>(kLaunchRegs)) return cudaErrorInvalidKernelImage;
        e = cudaFuncSetAttribute(jfa_bwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kDynSmem);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    jfa_bwd_kernel<D><<<grid, kBwdThreads, L::kDynSmem, s>>>(p, m);
    return cudaGetLastError();
}

// Block-sparse backward: the keys of an unselected tile have no weight in
// any query's softmax, so their dK and dV rows are zero.  One tile per CTA
// (grid-stride over the list), 16-byte stores of one head's D columns.
__global__ void __launch_bounds__(256) jfa_zero_tiles_kernel(const ZeroTile* tiles, int64_t n, uint16_t* dk,
                                                             uint16_t* dv, int H, int D) {
    const int vecs = D / 8;  // 16-byte vectors per row
    for (int64_t t = blockIdx.x; t < n; t += gridDim.x) {
        const int4 z = __ldg(reinterpret_cast<const int4*>(tiles) + t);  // row0, rows, h
        for (int e = threadIdx.x; e < z.y * vecs; e += blockDim.x) {
            const int64_t off = ((static_cast<int64_t>(z.x) + e / vecs) * H + z.z) * D + (e % vecs) * 8;
            *reinterpret_cast<uint4*>(dk + off) = make_uint4(0u, 0u, 0u, 0u);
            *reinterpret_cast<uint4*>(dv + off) = make_uint4(0u, 0u, 0u, 0u);
        }
    }
}

}  // namespace

cudaError_t launch_zero_tiles(const ZeroTile* tiles, int64_t n, uint16_t* dk, uint16_t* dv, int H, int D,
                              cudaStream_t s) {
    if (n <= 0) return cudaSuccess;
    const int grid = static_cast<int>(n < 152 * 16 ? n : 152 * 16);
    jfa_zero_tiles_kernel<<<grid, 256, 0, s>>>(tiles, n, dk, dv, H, D);
    return cudaGetLastError();
}

cudaError_t launch_bwd_pre(const PreParams& p, cudaStream_t s) {
    if (p.rows <= 0) return cudaSuccess;
    const int lanes = p.D / (8 * JFA_PRE_VEC);
    const int pairs_per_block = 256 / lanes;
    int64_t blocks = (p.rows + pairs_per_block - 1) / pairs_per_block;
    if (blocks > 152 * JFA_PRE_BLOCKS_PER_SM) blocks = 152 * JFA_PRE_BLOCKS_PER_SM;
    if (p.D == 128)
        jfa_bwd_pre_kernel<128><<<static_cast<int>(blocks), 256, 0, s>>>(p);
    else
        jfa_bwd_pre_kernel<64><<<static_cast<int>(blocks), 256, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_dq_sum(const float* partial, float* dq, int64_t n, int groups, cudaStream_t s) {
    if (n <= 0) return cudaSuccess;
    const int64_t n4 = n / 4;
    int64_t blocks = (n4 + 255) / 256;
    if (blocks > 152 * 8) blocks = 152 * 8;
    jfa_dq_sum_kernel<<<static_cast<int>(blocks), 256, 0, s>>>(reinterpret_cast<const float4*>(partial),
                                                               reinterpret_cast<float4*>(dq), n4, groups);
    return cudaGetLastError();
}

cudaError_t launch_bwd(int D, const BwdParams& p, const BwdMaps& m, int grid, cudaStream_t s) {
    if (grid <= 0) return cudaSuccess;
    return D == 128 ? launch_bwd_d<128>(p, m, grid, s) : launch_bwd_d<64>(p, m, grid, s);
}

}  // namespace jfa

JFA_TRACE_DEFINE_READER(jfa_trace_read_bwd)
