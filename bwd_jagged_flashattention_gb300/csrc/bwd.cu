// bwd.cu -- Jagged Flash Attention backward for sm_103a.
//
// One persistent, warp-specialised kernel walks items (sequence b, head h,
// key/value tile n of 128 rows) and loops over the query tiles that see that
// key tile.  For query tile i (128 rows), with K, V the item's tiles:
//   S^T  = K Q_i^T                       (TMEM, fp32)
//   dP^T = V dO_i^T                      (TMEM, fp32)
//   P^T  = exp(scale S^T - LSE_i)        (bf16, written over S^T in TMEM)
//   dV  += P^T dO_i                      (A operand straight from TMEM)
//   dS^T = P^T * (dP^T - Delta_i)        (bf16, shared memory)
//   dK  += dS^T Q_i                      (TMEM accumulator for the item)
//   dQ_i = dS_i K                        (TMEM, over the dP^T columns)
// dQ_i is read out by a dedicated warpgroup, which frees its TMEM columns at
// once and then streams it through two 16-column fp32 shared-memory stages
// (64-byte swizzle) into TMA bulk reduce-adds on the global fp32 dQ.  In
// broadcast-Q mode every sequence adds into the same dQ [Lq,H,D]: the pages
// call this contended reduction the first backward bottleneck and hide it
// with a double-buffered shared-memory pipeline and an early release of the
// dQ tensor memory (Meta's TLX Jagged Flash Attention Beats FA4 on Blackwell
// With 3x Less Code, section "Optimizations layered on top"; Meta's 3.2K-line
// Triton kernel outruns FlashAttention-4 on jagged Blackwell attention,
// second paragraph).  dK/dV stay in TMEM for the whole item and are written
// once.
//
// Delta = rowsum(dO * O), which the dS step needs (FlashAttention's backward;
// the pages do not name the step), comes from a separate pass over O and dO
// (jfa_bwd_pre_kernel) launched just before the main kernel.
//
// Roles (512 threads):
//   warps 0-3, 4-7  compute: P^T and dS^T for query columns 0-63 / 64-127
//                   (thread r = key row r = TMEM lane r); dV / dK epilogue
//   warps 8-11      dQ readout + reduce-add
//   warp  12        loads: K, V per item; Q_i (+ LSE_i), dO_i, Delta_i per tile
//                   (with Cluster Launch Control also the run-time deal)
//   warp  13        tcgen05 MMA issue and TMEM allocation
//   warps 14-15     idle (they complete the fourth warpgroup, whose register
//                   share the load and MMA warps take)
#include <cuda_runtime.h>
#include <climits>

#include "host_util.h"
#include "kernels.h"
#include "ptx.cuh"

namespace jfa {
namespace {

// Register split (setmaxnreg): the launch gives 512 x 128 = 65,536; then
// 120 per compute thread, 160 per dQ thread and 112 per load / MMA / idle
// thread, which sums to the same 65,536.
constexpr int kCW = 2;  // compute warpgroups
constexpr int kBwdThreads = 128 * (kCW + 2);
constexpr uint32_t kLaunchRegs = 128;
constexpr uint32_t kComputeRegs = 120;
constexpr uint32_t kDqRegs = 160;
constexpr uint32_t kAuxRegs = 112;
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

// Items of a CTA in the Cluster Launch Control mode: the load warp publishes
// each item index through a small ring, the other roles read it from there.
constexpr int kItemQ = 4;
// Readers of a ring slot: the MMA warp, the compute warps and the dQ warps
// (lane 0 of each arrives once it has the index).
constexpr uint32_t kItemReaders = 1 + 4 * kCW + 4;

struct BwdBars {
    alignas(16) uint32_t clc_resp[4];  // Cluster Launch Control response (16 bytes)
    uint64_t clc_bar;
    uint64_t iq_full[kItemQ], iq_empty[kItemQ];
    int32_t item_q[kItemQ];
    // k_full: the item's K and V tiles and its first Q tile landed (one
    // barrier for the three loads; q_full of that tile covers the statistics).
    // k_empty: every product of the item that reads K or V has completed.
    uint64_t k_full, k_empty;
    uint64_t q_full[2], q_empty[2];
    uint64_t dl_full[2];  // Delta of the query tile in stats stage [st] is staged
    // do_full: the tile's dO landed and the dQ warps have read the previous
    // tile's dQ out of TMEM (the dP^T of this tile overwrites those columns).
    uint64_t do_full, do_empty;
    uint64_t s_full, dp_full, p_full, ds_full, ds_empty;
    uint64_t dq_full;
    // There is no barrier for the dK/dV read-out: each compute thread reads
    // its accumulator rows before it arrives on the next item's first p_full,
    // and the MMA warp waits on that p_full before the item's first dV and dK.
    uint64_t dkv_full;
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

// Cluster Launch Control: the item index each role takes next from the
// ring the load warp fills (-1 at the end, or when the CTA aborts).  The
// roles keep the static schedule's loop over [ib, ie) -- with ie = INT_MAX in
// this mode -- and replace its counter by the index read here.
struct ItemRing {
    uint32_t n = 0;  // ring slots read so far
    __device__ __forceinline__ int read(BwdBars& bars, const AbortState& ab) {
        const int slot = static_cast<int>(n % kItemQ);
        if (!mbar_wait_warp(&bars.iq_full[slot], (n / kItemQ) & 1, ab)) return -1;
        ++n;
        const int v = *reinterpret_cast<volatile int32_t*>(&bars.item_q[slot]);
        __syncwarp();
        if ((threadIdx.x & 31) == 0) mbar_arrive(&bars.iq_empty[slot]);
        return v;
    }
};

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
__device__ __forceinline__ void issue_kmajor(uint32_t lead, uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc) {
    constexpr uint32_t idesc = idesc_bf16_f32(128, 128, 0, 0);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
        const uint64_t off = ((kk / 4) * 16384 + (kk % 4) * 32) / 16;
        mma_ss_p(lead, d_tmem, a_desc + off, b_desc + off, idesc, kk > 0);
    }
}

// dV (+)= P^T dO: A = P^T from TMEM (bf16 pairs), B = dO_i [q][D] MN-major.
// Each compute warpgroup packs its 32-query chunk c of P^T over the first
// half of chunk c's own S^T columns, so K step kk (16 queries = 8 columns of
// bf16 pairs) reads TMEM column (kk / 2) * 32 + (kk % 2) * 8.
__device__ __forceinline__ constexpr uint32_t p_col(int kk) {
    return static_cast<uint32_t>((kk / 2) * 32 + (kk % 2) * 8);
}

template <int D>
__device__ __forceinline__ void issue_dv(uint32_t lead, uint32_t d_tmem, uint32_t p_tmem, uint64_t do_desc,
                                         uint32_t acc) {
    constexpr uint32_t idesc = idesc_bf16_f32(128, D, 0, 1);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
        mma_ts_p(lead, d_tmem, p_tmem + p_col(kk), do_desc + kk * (2048 / 16), idesc, (acc | kk) != 0);
}

// dK (+)= dS^T Q: A = dS^T [key][q] K-major (smem), B = Q_i [q][D] MN-major.
template <int D>
__device__ __forceinline__ void issue_dk(uint32_t lead, uint32_t d_tmem, uint64_t ds_desc_k, uint64_t q_desc_mn,
                                         uint32_t acc) {
    constexpr uint32_t idesc = idesc_bf16_f32(128, D, 0, 1);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        const uint64_t aoff = ((kk / 4) * 16384 + (kk % 4) * 32) / 16;
        mma_ss_p(lead, d_tmem, ds_desc_k + aoff, q_desc_mn + kk * (2048 / 16), idesc, (acc | kk) != 0);
    }
}

// dQ = dS K: A = dS [q][key] read MN-major from the dS^T buffer, B = K [key][D] MN-major.
template <int D>
__device__ __forceinline__ void issue_dq(uint32_t lead, uint32_t d_tmem, uint64_t ds_desc_mn, uint64_t k_desc_mn) {
    constexpr uint32_t idesc = idesc_bf16_f32(128, D, 1, 1);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
        mma_ss_p(lead, d_tmem, ds_desc_mn + kk * (2048 / 16), k_desc_mn + kk * (2048 / 16), idesc, kk > 0);
}

// Index of query qi of item `it` in the LSE / Delta layout ([B,H,Lq] or [H,N]).
__device__ __forceinline__ int64_t stat_index(const BwdParams& p, const BwdItem& it, int qi) {
    return p.broadcast_q ? (static_cast<int64_t>(it.b) * p.H + it.h) * p.Lq + qi
                         : static_cast<int64_t>(it.h) * p.N + it.q_row0 + qi;
}

// ---------------------------------------------------------------------------
// Load warp (all 32 lanes: lane 0 issues TMA, every lane stages statistics).
// ---------------------------------------------------------------------------
template <int D, bool kDyn>
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
    uint32_t k_cnt = 0, q_cnt = 0, do_cnt = 0;
    bool k_open = false;  // k_full's phase still waits for its closing arrival
    // Broadcast Q: the (head, query tile) each Q stage holds, so a tile that
    // is already resident is not loaded again (the statistics still are).
    // Key = head << 16 | tile (tiles < 2^16 since Lq <= 2^23); -1 = empty.
    int stage_key0 = -1, stage_key1 = -1;
    // Cluster Launch Control: this CTA's own item first, then every CTA it
    // cancels before that one starts; each index goes to the other roles
    // through the ring (-1 last).
    // Queues instead: the next item of this CTA's queue, taken (atomically)
    // one item ahead; lane 0 holds the position until it is needed.
    const bool from_queue = kDyn && p.queue != nullptr;
    const int qg = from_queue ? static_cast<int>(blockIdx.x) % p.n_queues : 0;
    auto queue_item = [&](int taken) {
        const int v = __shfl_sync(0xffffffffu, taken, 0);
        const int q0 = p.cta_start[qg], q1 = p.cta_start[qg + 1];
        return v < q1 - q0 ? q0 + v : -1;
    };
    int taken = 0;
    int cur = static_cast<int>(blockIdx.x);
    if (from_queue) {
        if (lane == 0) taken = atomicAdd(p.queue + qg, 1);
        cur = queue_item(taken);
    }
    uint32_t published = 0, clc_phase = 0;
    bool clc_inflight = false;
    for (int k = ib; k < ie; ++k) {
        int idx = k;
        if constexpr (kDyn) {
            idx = cur;
            const int slot = static_cast<int>(published % kItemQ);
            if (!mbar_wait_warp(&bars.iq_empty[slot], ((published / kItemQ) & 1) ^ 1, ab)) goto done;
            if (lane == 0) {
                bars.item_q[slot] = idx;
                mbar_arrive(&bars.iq_full[slot]);
            }
            ++published;
            if (idx < 0) break;
            if (from_queue) {  // take the next item while this one's tiles load
                if (lane == 0) taken = atomicAdd(p.queue + qg, 1);
            } else {
                if (lane == 0) {  // ask for the next item while this one's tiles load
                    mbar_arrive_expect_tx(&bars.clc_bar, 16);
                    clc_try_cancel(bars.clc_resp, &bars.clc_bar);
                }
                clc_inflight = true;
            }
        }
        const BwdItem it = decode_bwd(p.items[idx], p);
        const int kv_row = it.kv_start + 128 * it.n;
        if (!mbar_wait_warp(&bars.k_empty, (k_cnt & 1) ^ 1, ab)) goto done;
        if (lane == 0) {
            // K and V; the item's first Q tile lands on the same barrier, and
            // its arrival closes the phase.
            mbar_expect_tx(&bars.k_full, 2 * L::kTileBytes);
#pragma unroll
            for (int s = 0; s < L::kSlabs; ++s)
                tma_load_2d(smem + L::kK + s * L::kSlabBytes, &m->k, &bars.k_full, it.h * D + 64 * s, kv_row);
        }
        ++k_cnt;
        // V's buffer is free too: k_empty is committed after every product that reads V.
        if (lane == 0) {
#pragma unroll
            for (int s = 0; s < L::kSlabs; ++s)
                tma_load_2d(smem + L::kV + s * L::kSlabBytes, &m->v, &bars.k_full, it.h * D + 64 * s, kv_row);
        }
        k_open = true;

        for (int i = it.i0; i < it.i1; ++i) {
            const int st = q_cnt % 2;
            if (!mbar_wait_warp(&bars.q_empty[st], ((q_cnt / 2) & 1) ^ 1, ab)) goto done;
            // LSE_i (as log2; -inf rows become +inf so P = 0; out-of-range
            // queries +inf) for the 128 queries of the tile, 4 per lane.
            float* lse2 = reinterpret_cast<float*>(smem + L::kStats + st * 1024);
            float* delta = lse2 + 128;
            {
                float l2[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int qi = 128 * i + lane * 4 + e;
                    l2[e] = INFINITY;
                    if (qi < it.q_rows) {
                        const float lv = p.lse[stat_index(p, it, qi)];
                        l2[e] = lv == -INFINITY ? INFINITY : lv * kLog2e;
                    }
                }
                *reinterpret_cast<float4*>(lse2 + lane * 4) = make_float4(l2[0], l2[1], l2[2], l2[3]);
            }
            __syncwarp();
            const int key = (it.h << 16) | i;
            // The item's first Q tile completes on k_full (q_full then only
            // says that the statistics are staged).
            const bool first = i == it.i0;
            if (p.broadcast_q && (st == 0 ? stage_key0 : stage_key1) == key) {
                if (lane == 0) {
                    mbar_arrive(&bars.q_full[st]);  // Q_i already resident: statistics only
                    if (first) mbar_arrive(&bars.k_full);
                }
            } else {
                if (lane == 0) {
                    uint64_t* qbar = first ? &bars.k_full : &bars.q_full[st];
                    mbar_arrive_expect_tx(qbar, L::kTileBytes);
#pragma unroll
                    for (int s = 0; s < L::kSlabs; ++s)
                        tma_load_2d(smem + L::kQ + st * L::kTileBytes + s * L::kSlabBytes, &m->q, qbar,
                                    it.h * D + 64 * s, it.q_row0 + 128 * i);
                    if (first) mbar_arrive(&bars.q_full[st]);
                }
                if (st == 0)
                    stage_key0 = key;
                else
                    stage_key1 = key;
            }
            if (first) k_open = false;
            ++q_cnt;
            if (!mbar_wait_warp(&bars.do_empty, (do_cnt & 1) ^ 1, ab)) goto done;
            if (lane == 0) {
                mbar_arrive_expect_tx(&bars.do_full, L::kTileBytes);
#pragma unroll
                for (int s = 0; s < L::kSlabs; ++s)
                    tma_load_2d(smem + L::kDO + s * L::kSlabBytes, &m->dout, &bars.do_full, it.h * D + 64 * s,
                                it.o_row0 + 128 * i);
            }
            ++do_cnt;
            // Delta_i, from the pre-pass.
            {
                float dl[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int qi = 128 * i + lane * 4 + e;
                    dl[e] = qi < it.q_rows ? p.delta[stat_index(p, it, qi)] : 0.0f;
                }
                *reinterpret_cast<float4*>(delta + lane * 4) = make_float4(dl[0], dl[1], dl[2], dl[3]);
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars.dl_full[st]);
            }
        }
        if constexpr (kDyn) {  // the next item: a canceled CTA's index, or -1 when none is left
            if (from_queue) {
                cur = queue_item(taken);
                continue;
            }
            if (!mbar_wait_warp(&bars.clc_bar, clc_phase & 1, ab)) goto done;
            ++clc_phase;
            clc_inflight = false;
            cur = clc_response_ctaid_x(bars.clc_resp);
            if (cur >= p.n_items) {  // not an index of this grid: stop (and report it) rather than read past the list
                if (lane == 0 && p.status) atomicOr(p.status, 1u << kDevTimeout);
                cur = -1;
            }
        }
    }
done:
    // Let every issued copy (and a pending launch-control response) land before the CTA can exit.
    if (lane == 0 && clc_inflight) mbar_wait_drain(&bars.clc_bar, clc_phase & 1);
    if (lane == 0) {
        if (k_open) mbar_arrive(&bars.k_full);  // left before the item's first Q tile
        if (k_cnt) mbar_wait_drain(&bars.k_full, (k_cnt - 1) & 1);
        for (uint32_t c = q_cnt > 2 ? q_cnt - 2 : 0; c < q_cnt; ++c) mbar_wait_drain(&bars.q_full[c % 2], (c / 2) & 1);
        if (do_cnt) mbar_wait_drain(&bars.do_full, (do_cnt - 1) & 1);
    }
    __syncwarp();
}

// ---------------------------------------------------------------------------
// MMA issuer (one warp, lane 0 issuing).  Per query tile: dP^T, then dV (once P^T is in
// TMEM), then the next tile's S^T right behind dV (which reads P^T first),
// then dQ before dK, so the dQ readout -- and with it the next dP^T, which
// reuses dQ's columns -- and on the last tile the release of K come one
// product sooner.
// ---------------------------------------------------------------------------
template <int D, bool kDyn>
__device__ void bwd_mma_role(const BwdParams& p, uint8_t* smem, BwdBars& bars, uint32_t tmem, int ib, int ie,
                             const AbortState& ab) {
    using L = BwdLayout<D>;
    // The whole warp runs this role (uniform control flow and operands); only
    // lane 0 issues the products and commits.
    const uint32_t lead = (threadIdx.x & 31) == 0 ? 1u : 0u;
    const uint64_t dK_k = kmajor_desc(smem_u32(smem + L::kK)), dK_mn = mnmajor_desc(smem_u32(smem + L::kK));
    const uint64_t dV_k = kmajor_desc(smem_u32(smem + L::kV));
    const uint64_t dQ_k = kmajor_desc(smem_u32(smem + L::kQ)), dQ_mn = mnmajor_desc(smem_u32(smem + L::kQ));
    const uint64_t dDO_k = kmajor_desc(smem_u32(smem + L::kDO)), dDO_mn = mnmajor_desc(smem_u32(smem + L::kDO));
    const uint64_t dDS_k = kmajor_desc(smem_u32(smem + L::kDS)), dDS_mn = mnmajor_desc(smem_u32(smem + L::kDS));
    constexpr uint64_t kTileUnits = L::kTileBytes / 16;
    uint32_t it_cnt = 0, q_cnt = 0, tile_cnt = 0;
    ItemRing ring;
    for (int k = ib; k < ie; ++k) {
        int idx = k;
        if constexpr (kDyn) {
            if ((idx = ring.read(bars, ab)) < 0) break;
        }
        const BwdItem it = decode_bwd(p.items[idx], p);
        if (!mbar_wait(&bars.k_full, it_cnt & 1, ab)) goto done;  // K, V (and the first Q tile)
        {  // S^T of the item's first query tile
            const int st = q_cnt % 2;
            tc_fence_after();
            issue_kmajor<D>(lead, tmem + L::kColS, dK_k, dQ_k + st * kTileUnits);  // S^T = K Q^T
            mma_commit_p(lead, &bars.s_full);
        }
        for (int i = it.i0; i < it.i1; ++i) {
            const int st = q_cnt % 2;
            if (!mbar_wait(&bars.do_full, tile_cnt & 1, ab)) goto done;
            tc_fence_after();
            issue_kmajor<D>(lead, tmem + L::kColDP, dV_k, dDO_k);  // dP^T = V dO^T
            mma_commit_p(lead, &bars.dp_full);
            if (!mbar_wait(&bars.p_full, tile_cnt & 1, ab)) goto done;
            tc_fence_after();
            issue_dv<D>(lead, tmem + L::kColDV, tmem + L::kColS, dDO_mn, i > it.i0);
            mma_commit_p(lead, &bars.do_empty);
            if (i + 1 < it.i1) {  // next tile's S^T (the compute warps keep P in registers)
                const int st2 = (q_cnt + 1) % 2;
                if (!mbar_wait(&bars.q_full[st2], ((q_cnt + 1) / 2) & 1, ab)) goto done;
                tc_fence_after();
                issue_kmajor<D>(lead, tmem + L::kColS, dK_k, dQ_k + st2 * kTileUnits);
                mma_commit_p(lead, &bars.s_full);
            }
            if (!mbar_wait(&bars.ds_full, tile_cnt & 1, ab)) goto done;
            tc_fence_after();
            issue_dq<D>(lead, tmem + L::kColDP, dDS_mn, dK_mn);
            mma_commit_p(lead, &bars.dq_full);
            if (i == it.i1 - 1) mma_commit_p(lead, &bars.k_empty);
            issue_dk<D>(lead, tmem + L::kColDK, dDS_k, dQ_mn + st * kTileUnits, i > it.i0);
            mma_commit_p(lead, &bars.q_empty[st]);
            mma_commit_p(lead, &bars.ds_empty);
            ++q_cnt;
            ++tile_cnt;
        }
        mma_commit_p(lead, &bars.dkv_full);
        ++it_cnt;
    }
done:
    mma_commit_p(lead, &bars.mma_done);
    mbar_wait_drain(&bars.mma_done, 0);
}

// ---------------------------------------------------------------------------
// Compute warpgroups: warpgroup g owns query columns 64g .. 64g+63 of every
// key row (32-column chunks c0 = 2g and c0 + 1).  One chunk of S^T is in
// registers at a time and the log2-LSE values are read 4 at a time.  The two
// warpgroups run concurrently, so chunk c's P^T (16 columns of bf16 pairs)
// goes over the first half of chunk c's own S^T columns (c * 32), never over
// S^T columns the other warpgroup may not have read yet; the dV product reads
// it from there (p_col()).  P stays in registers (pkeep) for the dS pass.
// ---------------------------------------------------------------------------
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
                const float p0 = bf16lo_to_f32(pkeep[cc * 16 + e]), p1 = bf16hi_to_f32(pkeep[cc * 16 + e]);
                // dS = P (dP - Delta) as P dP - P Delta: one paired multiply
                // and one paired FMA per two columns (ads step: 8 us less
                // than two scalar subtract-multiply pairs).
                float d0, d1, n0, n1;
                fmul2(n0, n1, p0, p1, -(h ? f.z : f.x), -(h ? f.w : f.y));
                ffma2(d0, d1, p0, p1, __uint_as_float(dp[2 * e]), __uint_as_float(dp[2 * e + 1]), n0, n1);
                pk[e] = pack_bf16x2(d0, d1);
            }
        }
        // Row `row`, queries c*32 .. c*32+31: slab c/2, 16-byte chunks (c%2)*4 .. +3,
        // stored at chunk ^ (row % 8) (128-byte swizzle, as TMA would place them).
        uint8_t* slab = ds_tile + (c / 2) * 16384 + row * 128;
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            const int chunk = ((c % 2) * 4 + v) ^ (row % 8);
            *reinterpret_cast<uint4*>(slab + chunk * 16) = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
        }
    }
}

// Hand-off to the MMA thread after a warpgroup's tcgen05 / shared-memory
// writes (already fenced for the async proxy where needed): every thread
// fences, then arrives.
__device__ __forceinline__ void handoff_arrive(uint64_t* bar) {
    tc_fence_before();
    mbar_arrive(bar);
}

template <int D, bool kDyn>
__device__ void bwd_compute_role(const BwdParams& p, const BwdMaps* maps, uint8_t* smem, BwdBars& bars,
                                 uint32_t tmem, int ib, int ie, const AbortState& ab) {
    using L = BwdLayout<D>;
    const int row = threadIdx.x % 128;  // key row = TMEM lane
    const int wg = threadIdx.x / 128;   // compute warpgroup: its query columns
    const uint32_t lane_off = static_cast<uint32_t>(((threadIdx.x / 32) % 4) * 32) << 16;
    const uint32_t s_addr = tmem + lane_off + L::kColS;
    const uint32_t dp_addr = tmem + lane_off + L::kColDP;
    uint8_t* ds_tile = smem + L::kDS;
    uint32_t q_cnt = 0, tile_cnt = 0, item_cnt = 0;
    ItemRing ring;
    for (int k = ib; k < ie; ++k, ++item_cnt) {
        int idx = k;
        if constexpr (kDyn) {
            if ((idx = ring.read(bars, ab)) < 0) break;
        }
        const BwdItem it = decode_bwd(p.items[idx], p);
        const int key = 128 * it.n + row;
        const bool row_valid = key < it.Lk;
        const bool kv_full_tile = 128 * (it.n + 1) <= it.Lk;
        for (int i = it.i0; i < it.i1; ++i) {
            const int st = q_cnt % 2;
            const float* lse2 = reinterpret_cast<const float*>(smem + L::kStats + st * 1024);
            const float* delta = lse2 + 128;
            if (!mbar_wait_warp(&bars.q_full[st], (q_cnt / 2) & 1, ab)) goto done;
            if (!mbar_wait_warp(&bars.s_full, tile_cnt & 1, ab)) goto done;
            tc_fence_after();
            const bool unmasked = kv_full_tile && 128 * (i + 1) <= it.q_rows && !(p.causal && i == it.n);
            uint32_t pkeep[32];
            if (unmasked)
                bwd_compute_p_cols<D, false>(p, lse2, s_addr, key, 128 * i, it.q_rows, row_valid, 2 * wg, pkeep);
            else
                bwd_compute_p_cols<D, true>(p, lse2, s_addr, key, 128 * i, it.q_rows, row_valid, 2 * wg, pkeep);
            handoff_arrive(&bars.p_full);
            if (!mbar_wait_warp(&bars.dp_full, tile_cnt & 1, ab)) goto done;
            if (!mbar_wait_warp(&bars.ds_empty, (tile_cnt & 1) ^ 1, ab)) goto done;
            if (!mbar_wait_warp(&bars.dl_full[st], (q_cnt / 2) & 1, ab)) goto done;
            tc_fence_after();
            if (i == it.i0) {  // the last item's dK/dV stores have read the tile
                if (row == 0) bulk_wait_group_read<0>();
                compute_sync(wg);
            }
            bwd_compute_ds_cols<D>(delta, dp_addr, ds_tile, row, 2 * wg, pkeep);
            fence_proxy_async_smem();
            handoff_arrive(&bars.ds_full);
            ++q_cnt;
            ++tile_cnt;
        }
        // This item's dK (warpgroup 1, scaled) or dV (warpgroup 0), while the
        // next item's K tile loads: once every product of the item is done
        // (dkv_full, which also means the last dK / dQ have read dS), 64-column
        // halves go TMEM -> registers -> 128-byte-swizzled stage in the
        // warpgroup's slab of the dS tile -> a TMA store of the whole tile, or
        // for a ragged tail tile (which must not touch the next sequence's
        // rows) coalesced row copies.  The accumulator's columns are free for
        // the next item once this thread arrives on that item's first p_full
        // (the MMA warp waits on it before the item's first dV and dK).
        {
            if (!mbar_wait_warp(&bars.dkv_full, item_cnt & 1, ab)) goto done;
            tc_fence_after();
            const int rows_valid = min(128, it.Lk - 128 * it.n);
            const int64_t row0 = static_cast<int64_t>(it.kv_start) + 128 * it.n;
            const bool tma_ok = rows_valid == 128;
            if (!tma_ok) {  // the last item's stores have read the stage
                if (row == 0) bulk_wait_group_read<0>();
                compute_sync(wg);
            }
            const uint32_t col = wg ? L::kColDK : L::kColDV;
            const float sc = wg ? p.scale : 1.0f;
            uint16_t* out = wg ? p.dk : p.dv;
            uint8_t* stage = ds_tile + wg * 16384;
#pragma unroll
            for (int half = 0; half < D / 64; ++half) {
                uint32_t v[2][32];
                tmem_ld32(tmem + lane_off + col + half * 64, v[0]);
                tmem_ld32(tmem + lane_off + col + half * 64 + 32, v[1]);
                tmem_ld_wait();
                if (tma_ok && half > 0) {  // the store that used this stage has read it
                    if (row == 0) bulk_wait_group_read<0>();
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
                        tma_store_2d(wg ? &maps->dk : &maps->dv, stage, it.h * D + half * 64, static_cast<int>(row0));
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
    }
done:
    if (row == 0) bulk_wait_group<0>();  // every dK/dV store has completed
}

// ---------------------------------------------------------------------------
// dQ warpgroup: TMEM dQ -> registers (release TMEM) -> two 128x16 fp32 smem
// stages -> TMA bulk reduce-add into global dQ.
// ---------------------------------------------------------------------------
template <int D, bool kDyn>
__device__ void bwd_dq_role(const BwdParams& p, const CUtensorMap* map_dq, uint8_t* smem, BwdBars& bars,
                            uint32_t tmem, int ib, int ie, const AbortState& ab) {
    using L = BwdLayout<D>;
    const int r = threadIdx.x - 32 * kWarpDq;  // query row of the tile (TMEM lane)
    const bool issuer = r == 0;
    const uint32_t lane_off = static_cast<uint32_t>(((threadIdx.x / 32) % 4) * 32) << 16;
    const uint32_t dq_addr = tmem + lane_off + L::kColDP;
    uint8_t* stage_base = smem + L::kDQ;
    uint32_t tile_cnt = 0, stage_uses = 0;
    if (issuer) prefetch_tensormap(map_dq);
    // do_full's phase t also counts the read-out of dQ t-1; for the first
    // tile there is none, so arrive for it now.
    mbar_arrive(&bars.do_full);
    ItemRing ring;
    for (int k = ib; k < ie; ++k) {
        int idx = k;
        if constexpr (kDyn) {
            if ((idx = ring.read(bars, ab)) < 0) break;
        }
        const BwdItem it = decode_bwd(p.items[idx], p);
        for (int i = it.i0; i < it.i1; ++i) {
            bool ok = mbar_wait_warp(&bars.dq_full, tile_cnt & 1, ab);
            if (!group_all(1, ok)) goto done;
            tc_fence_after();
            uint32_t v[D / 32][32];
#pragma unroll
            for (int c = 0; c < D / 32; ++c) tmem_ld32(dq_addr + c * 32, v[c]);
            tmem_ld_wait();
            // early release: the next dP^T/dQ may overwrite these columns
            handoff_arrive(&bars.do_full);
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
                    tma_reduce_add_2d(map_dq, stage, it.h * D + sl * 16, it.q_row0 + 128 * i);
                    bulk_commit_group();
                }
                ++stage_uses;
            }
            ++tile_cnt;
        }
    }
done:
    if (issuer) bulk_wait_group<0>();
}

template <int D, bool kDyn>
__global__ void __launch_bounds__(kBwdThreads, 1)
    jfa_bwd_kernel(const BwdParams p, const __grid_constant__ BwdMaps maps) {
    using L = BwdLayout<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024(smem_raw);
    __shared__ BwdBars bars;
    const int warp = threadIdx.x / 32;
    const int ib = kDyn ? 0 : p.cta_start[blockIdx.x];
    const int ie = kDyn ? INT_MAX : p.cta_start[blockIdx.x + 1];  // dynamic: the roles stop at a -1 index
    const AbortState ab{&bars.abort_flag, p.status, p.wait_ns};

    if (threadIdx.x == 0) {
        bars.abort_flag = 0;
        mbar_init(&bars.clc_bar, 1);
        for (int s = 0; s < kItemQ; ++s) {
            mbar_init(&bars.iq_full[s], 1);
            mbar_init(&bars.iq_empty[s], kItemReaders);
        }
        mbar_init(&bars.k_full, 1);
        mbar_init(&bars.k_empty, 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bars.q_full[s], 1);
            mbar_init(&bars.q_empty[s], 1);
            mbar_init(&bars.dl_full[s], 1);
        }
        // dO landed (one arrival and the bytes) and, merged in, the dQ warps'
        // read-out of the previous tile's dQ (128 arrivals).
        mbar_init(&bars.do_full, 1 + 4 * 32);
        mbar_init(&bars.do_empty, 1);
        mbar_init(&bars.s_full, 1);
        mbar_init(&bars.dp_full, 1);
        mbar_init(&bars.p_full, 4 * kCW * 32);
        mbar_init(&bars.ds_full, 4 * kCW * 32);
        mbar_init(&bars.ds_empty, 1);
        mbar_init(&bars.dq_full, 1);
        mbar_init(&bars.dkv_full, 1);
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
        regs_dec<kComputeRegs>();
        bwd_compute_role<D, kDyn>(p, &maps, smem, bars, tmem, ib, ie, ab);
    } else if (warp < kWarpDq + 4) {
        regs_inc<kDqRegs>();
        bwd_dq_role<D, kDyn>(p, &maps.dq, smem, bars, tmem, ib, ie, ab);
    } else {
        regs_dec<kAuxRegs>();
        if (warp == kWarpLoad) {
            bwd_load_role<D, kDyn>(p, &maps, smem, bars, ib, ie, ab);
        } else if (warp == kWarpMma) {
            bwd_mma_role<D, kDyn>(p, smem, bars, tmem, ib, ie, ab);
            __syncwarp();
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kWarpMma) tmem_dealloc(tmem, L::kTmemCols);
}

template <int D, bool kDyn>
cudaError_t launch_bwd_dk(const BwdParams& p, const BwdMaps& m, int grid, cudaStream_t s) {
    using L = BwdLayout<D>;
    static bool configured = false;
    if (!configured) {
        // The register split is only safe at exactly kLaunchRegs per thread.
        cudaFuncAttributes fa;
        cudaError_t e = cudaFuncGetAttributes(&fa, jfa_bwd_kernel<D, kDyn>);
        if (e != cudaSuccess) return e;
        if (fa.numRegs != static_cast<int>(kLaunchRegs)) return cudaErrorInvalidKernelImage;
        e = cudaFuncSetAttribute(jfa_bwd_kernel<D, kDyn>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kDynSmem);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    jfa_bwd_kernel<D, kDyn><<<grid, kBwdThreads, L::kDynSmem, s>>>(p, m);
    return cudaGetLastError();
}

// The static schedule and the Cluster Launch Control mode are separate
// instantiations, so the static kernel carries none of the run-time deal.
template <int D>
cudaError_t launch_bwd_d(const BwdParams& p, const BwdMaps& m, int grid, cudaStream_t s) {
    return p.clc ? launch_bwd_dk<D, true>(p, m, grid, s) : launch_bwd_dk<D, false>(p, m, grid, s);
}

// Delta[row] = sum_d dO[row, d] * O[row, d] (fp32) for every (O row, head)
// pair: D / 16 consecutive lanes own one pair, each reading two 16-byte
// chunks of O and of dO (ads step: one chunk 59.3 us, two 49.4 us, four
// 51.3 us).
template <int D>
__global__ void __launch_bounds__(256) jfa_bwd_pre_kernel(const PreParams p) {
    // The main kernel's tile schedule, from the pinned host buffer the host
    // built it in (instead of a host-to-device copy in the stream before this
    // kernel).
    for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < p.sched_vec16;
         e += static_cast<int64_t>(gridDim.x) * blockDim.x)
        p.sched_dst[e] = p.sched_src[e];
    // dQ starts at zero (the main kernel adds every tile's dQ into it).
    for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < p.dq_vec4;
         e += static_cast<int64_t>(gridDim.x) * blockDim.x)
        reinterpret_cast<float4*>(p.dq)[e] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    constexpr int kVec = 2;
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
                // Streaming (evict-first) loads: O and dO are read once here;
                // cached loads measured 53 vs 45 us on the ads step.
                a[u] = __ldcs(reinterpret_cast<const uint4*>(p.o + pair * D) + sub * kVec + u);
                b[u] = __ldcs(reinterpret_cast<const uint4*>(p.dout + pair * D) + sub * kVec + u);
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
    // Grid-stride, at most 16 blocks per SM (8 per SM: 70 us on the ads step;
    // 16 and 32 alike, 49 us).
    const int lanes = p.D / 16;
    const int pairs_per_block = 256 / lanes;
    int64_t blocks = (p.rows + pairs_per_block - 1) / pairs_per_block;
    const int cap = 16 * (device_sm_count() > 0 ? device_sm_count() : 152);
    if (blocks > cap) blocks = cap;
    if (p.D == 128)
        jfa_bwd_pre_kernel<128><<<static_cast<int>(blocks), 256, 0, s>>>(p);
    else
        jfa_bwd_pre_kernel<64><<<static_cast<int>(blocks), 256, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_bwd(int D, const BwdParams& p, const BwdMaps& m, int grid, cudaStream_t s) {
    if (grid <= 0) return cudaSuccess;
    return D == 128 ? launch_bwd_d<128>(p, m, grid, s) : launch_bwd_d<64>(p, m, grid, s);
}

}  // namespace jfa

