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
//   warps 10-11 idle (they only give their registers to the softmax warps)
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
//
// MXFP8 variant (kMx; TLX porta l'attenzione jagged su Blackwell oltre FA4
// con un terzo del codice, section "The turning point": P quantized to FP8
// on the fly, scale factors in tensor memory): V arrives as E4M3 with one
// E8M0 scale per 32 keys and column, and the PV product is block-scaled
// E4M3 (tcgen05 kind::mxf8f6f4).  The softmax keeps the running max at an
// integer (log2 domain), gives every 32-key chunk of its row the exponent
// X = floor(chunk max) - 8, writes P / 2^X as E4M3 over the first 32
// columns of S and the four chunk exponents next to it (column 32 + warp),
// plus its lane quarter's copy of the block's V scales (columns 64..).
// Q K^T stays bf16: with S0 | S1 | O0 | O1 filling TMEM at D = 128 there is
// no column left for its scale factors while both S tiles are live.
#include <cuda_runtime.h>

#include "kernels.h"
#include "ptx.cuh"

namespace jfa {
namespace {

// K/V ring depth in 128-row tiles at D = 128 (twice as many at D = 64):
// three slots cost 23 us on the ads step, a fifth gained nothing.
constexpr int kRingSlots = 4;

// 384 threads = three warpgroups: two softmax warpgroups and one holding the
// TMA warp, the MMA warp and two idle warps.  Registers are moved from the
// third warpgroup to the softmax ones: launch 384 x 168 = 64,512; after the
// split 256 x kSoftmaxRegs + 128 x kAuxRegs = 64,512 (never more than launch;
// below 88 the TMA/MMA roles spill, from 200 up the softmax does not).
constexpr int kFwdThreads = 384;
constexpr uint32_t kLaunchRegs = 168;
constexpr uint32_t kSoftmaxRegs = 208;
constexpr uint32_t kAuxRegs = 88;
static_assert(256 * kSoftmaxRegs + 128 * kAuxRegs <= kFwdThreads * kLaunchRegs, "register split exceeds launch");
constexpr int kWarpTma = 8;
constexpr int kWarpMma = 9;
constexpr float kRescaleLog2 = 8.0f;
constexpr float kLn2 = 0.6931471805599453f;

template <int D>
struct FwdLayout {
    static constexpr int kSlabBytes = 128 * 128;  // 128 rows x 64 bf16 (one swizzle span)
    static constexpr int kSlabs = D / 64;
    static constexpr int kTileBytes = kSlabs * kSlabBytes;
    static constexpr int kSlots = D == 128 ? kRingSlots : 2 * kRingSlots;  // K/V ring tiles
    static constexpr int kQOff = 0;
    static constexpr int kRingOff = 2 * kTileBytes;
    // Epilogue staging: 128 rows x 64 columns of bf16 (16 KB) per softmax warpgroup.
    static constexpr int kStageOff = (2 + kSlots) * kTileBytes;
    static constexpr int kStageBytes = 16384;
    static constexpr int kBytes = kStageOff + 2 * kStageBytes;
    static constexpr int kDynSmem = kBytes + 1024;
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kOCol = 256;
};

struct FwdBars {
    uint64_t q_full, q_empty;
    uint64_t kv_full[2 * kRingSlots], kv_empty[2 * kRingSlots];
    // No barrier for the O read-out: a softmax thread reads its O row out of
    // TMEM before it arrives on the next item's first p_full of that tile,
    // and the MMA warp waits on that p_full before the item's first P V.
    uint64_t s_full[2], p_full[2], o_full[2];
    uint64_t mma_done;
    uint32_t tmem_base;
    uint32_t abort_flag;
};

struct FwdItem {
    int b, h, kv_start, Lk, m0, nq, q_row0, q_rows;
    int slot;     // split-KV chunk: its partial (O, LSE) slot; -1 for a whole item
    int sel_off;  // block-sparse: the item's first entry in the selected-block list
    int nblk[2], nfull[2], nb;
};

// Every role derives the same per-item loop bounds from the work item.
// kSparse: the call has a block-sparse selection (p.sel set); the dense
// kernel is a separate instantiation without the selection look-up.
template <bool kSparse>
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
    int nkv = (it.Lk + 127) / 128, full = it.Lk / 128;
    it.sel_off = 0;
    it.slot = w.b < 0 ? -w.b - 1 : -1;  // a split-KV chunk (its keys are kv_start .. + kv_len)
    if (kSparse) {  // block-sparse (never causal): visit only the selected blocks, in ascending order
        const int4 s = __ldg(reinterpret_cast<const int4*>(p.sel) + static_cast<int64_t>(it.b) * p.H + it.h);
        it.sel_off = s.x;
        nkv = s.y;
        full = s.z;  // a ragged last block, when selected, is the last one visited
    }
    it.nb = 0;
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        if (t < it.nq) {
            const int m = it.m0 + t;
            it.nblk[t] = p.causal ? min(m + 1, nkv) : nkv;
            it.nfull[t] = p.causal ? min(m, full) : full;
        } else {
            it.nblk[t] = 0;
            it.nfull[t] = 0;
        }
        it.nb = max(it.nb, it.nblk[t]);
    }
    return it;
}

// Key block (counted from the sequence start) of the item's j-th visited block.
template <bool kSparse>
__device__ __forceinline__ int kv_block(const FwdParams& p, const FwdItem& it, int j) {
    return kSparse ? __ldg(p.sel_blocks + it.sel_off + j) : j;
}

// Broadcast Q: an item reuses the Q tiles already in shared memory when it
// reads the same ones (same head, first tile and tile count) as the last item
// that loaded them.  The TMA and MMA threads take the same decision from the
// same item sequence; Q is released (q_empty) only after the last item of a
// run, so loads and releases stay one-to-one.
struct QKey {
    int h = -1, m0 = -1, nq = -1;
    __device__ __forceinline__ bool same(const FwdItem& it) const { return it.h == h && it.m0 == m0 && it.nq == nq; }
    __device__ __forceinline__ void set(const FwdItem& it) {
        h = it.h;
        m0 = it.m0;
        nq = it.nq;
    }
};

// Whether the next item that uses Q after item i reads the same Q tiles
// (`next` = item i + 1, already loaded; empty sequences in between are rare
// and read on the spot).
template <bool kSparse>
__device__ __forceinline__ bool next_item_reuses_q(const FwdParams& p, const FwdItem& it, const WorkItem& next, int i,
                                                   int ie) {
    if (!p.broadcast_q || i + 1 >= ie) return false;
    FwdItem nx = decode_fwd<kSparse>(next, p);
    for (int k = i + 1; nx.nb == 0;) {
        if (++k >= ie) return false;
        nx = decode_fwd<kSparse>(p.items[k], p);
    }
    return nx.h == it.h && nx.m0 == it.m0 && nx.nq == it.nq;
}

// Hand-off from a softmax warpgroup to the MMA thread after its tcgen05
// stores or loads: every thread fences, then arrives (count 128).
constexpr uint32_t kHandoffCount = 128;
__device__ __forceinline__ void handoff_arrive(uint64_t* bar) {
    tc_fence_before();
    mbar_arrive(bar);
}

// Barrier over the 128 threads of one softmax warpgroup (ids 1 and 2).
__device__ __forceinline__ void group_sync(int id) { asm volatile("bar.sync %0, 128;" ::"r"(id) : "memory"); }

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
    return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Operand descriptors are built once per buffer; one MMA then only adds a
// compile-time offset (in 16-byte units) to the start-address field, which
// keeps the single issuing thread's instruction count per MMA minimal.
__device__ __forceinline__ uint64_t kmajor_desc(uint32_t saddr) { return smem_desc(saddr, 16, 1024); }
__device__ __forceinline__ uint64_t mnmajor_desc(uint32_t saddr) { return smem_desc(saddr, 16384, 1024); }

// S(tmem) = Q K^T: both operands K-major in 128-byte-swizzled slabs of 64
// columns; one K=16 step advances 32 bytes inside a slab.
template <int D>
__device__ __forceinline__ void issue_qk(uint32_t lead, uint32_t d_tmem, uint64_t q_desc, uint64_t k_desc) {
    constexpr uint32_t idesc = idesc_bf16_f32(128, 128, 0, 0);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
        constexpr uint64_t unit = 16;
        const uint64_t off = ((kk / 4) * 16384 + (kk % 4) * 32) / unit;
        mma_ss_p(lead, d_tmem, q_desc + off, k_desc + off, idesc, kk > 0);
    }
}

// O(tmem) (+)= P(tmem, bf16) V: V is MN-major (D contiguous); one K=16 step
// covers 16 key rows = 2048 bytes; the 64-column slabs are 16 KB apart.
template <int D>
__device__ __forceinline__ void issue_pv(uint32_t lead, uint32_t d_tmem, uint32_t p_tmem, uint64_t v_desc,
                                         uint32_t acc) {
    constexpr uint32_t idesc = idesc_bf16_f32(128, D, 0, 1);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
        mma_ts_p(lead, d_tmem, p_tmem + kk * 8, v_desc + kk * (2048 / 16), idesc, (acc | kk) != 0);
}

// TMEM columns (from a tile's S base) of the MXFP8 product's scale factors:
// P's chunk exponents, then this block's V scales (D / 32 columns).
constexpr uint32_t kSfaCol = 32, kSfbCol = 64;

// O(tmem) (+)= P(tmem, E4M3) V(smem, E4M3), block-scaled: four K=32 steps,
// step c using byte c of the scale words (keys 32c .. 32c+31).  V is
// MN-major with D-byte rows (128-byte swizzle at D=128, 64-byte at D=64);
// one step covers 32 rows.
template <int D>
__device__ __forceinline__ void issue_pv_mx(uint32_t lead, uint32_t d_tmem, uint32_t p_tmem, uint64_t v_desc,
                                            uint32_t acc) {
#pragma unroll
    for (int c = 0; c < 4; ++c)
        mma_ts_mx_p(lead, d_tmem, p_tmem + c * 8, v_desc + c * (32 * D / 16), idesc_mxf8_e4m3(128, D, 1, c, c),
                    p_tmem + kSfaCol, p_tmem + kSfbCol, (acc | c) != 0);
}

// ---------------------------------------------------------------------------
// TMA producer (one thread).
// ---------------------------------------------------------------------------
template <int D, bool kSparse, bool kMx>
__device__ void fwd_tma_role(const FwdParams& p, const CUtensorMap* mq, const CUtensorMap* mk,
                             const CUtensorMap* mv, uint8_t* smem, FwdBars& bars, int ib, int ie,
                             const AbortState& ab) {
    using L = FwdLayout<D>;
    prefetch_tensormap(mq);
    prefetch_tensormap(mk);
    prefetch_tensormap(mv);
    uint32_t ring = 0, q_loads = 0;
    // K and V blocks are read once per forward: evict them from L2 first, so
    // more of the O rows the kernel writes (which the backward's Delta pass
    // reads next) stay there (ads step: forward 137 vs 141 us, Delta pass 43
    // vs 45 us).
    const uint64_t kv_policy = l2_policy_evict_first();
    QKey qk;
    WorkItem wn = load_item(p.items, ib, ie);
    for (int i = ib; i < ie; ++i) {
        const WorkItem wc = wn;
        wn = load_item(p.items, i + 1, ie);
        const FwdItem it = decode_fwd<kSparse>(wc, p);
        if (it.nb == 0) continue;
        if (!(p.broadcast_q && qk.same(it))) {  // else: the resident Q tiles serve this item too
            if (!mbar_wait(&bars.q_empty, (q_loads & 1) ^ 1, ab)) goto done;
            mbar_arrive_expect_tx(&bars.q_full, it.nq * L::kTileBytes);
            for (int t = 0; t < it.nq; ++t)
#pragma unroll
                for (int s = 0; s < L::kSlabs; ++s)
                    tma_load_2d(smem + L::kQOff + t * L::kTileBytes + s * L::kSlabBytes, mq, &bars.q_full,
                                it.h * D + 64 * s, it.q_row0 + 128 * (it.m0 + t));
            ++q_loads;
            qk.set(it);
        }
        for (int j = 0; j < it.nb; ++j) {
            for (int kv = 0; kv < 2; ++kv) {
                const uint32_t slot = ring % L::kSlots;
                // Releases come in the same pairs (one commit frees V(j) and K(j+1)),
                // so a K tile's slot is free once the V slot before it was; only
                // the stream's first K, alone, has a release of its own.
                if ((kv || ring == L::kSlots) &&
                    !mbar_wait(&bars.kv_empty[slot], ((ring / L::kSlots) & 1) ^ 1, ab))
                    goto done;
                // V tiles sit at odd ring positions, K tiles at even ones.  A K
                // tile after the first completes on the barrier of the V tile
                // before it (V(j) with K(j+1), or an item's last V with the next
                // item's first K): V's bytes are announced without an arrival,
                // and K's arrival closes the pair, so the MMA warp waits once per
                // block.  Both tiles of a pair are released together anyway.
                uint64_t* full = &bars.kv_full[!kv && ring > 0 ? (ring - 1) % L::kSlots : slot];
                mbar_expect_tx(full, kMx && kv ? 128 * D : L::kTileBytes);  // E4M3 V: 128 rows x D bytes
                if (kMx && kv) {
                    tma_load_2d_hint(smem + L::kRingOff + slot * L::kTileBytes, mv, full, it.h * D,
                                     it.kv_start + 128 * j, kv_policy);
                } else {
#pragma unroll
                    for (int s = 0; s < L::kSlabs; ++s)
                        tma_load_2d_hint(smem + L::kRingOff + slot * L::kTileBytes + s * L::kSlabBytes, kv ? mv : mk,
                                         full, it.h * D + 64 * s, it.kv_start + 128 * kv_block<kSparse>(p, it, j),
                                         kv_policy);
                }
                if (!kv) mbar_arrive(full);
                ++ring;
            }
        }
    }
done:
    // The last V tile has no K after it to close its barrier's phase; with no
    // tile at all, close the first K's phase, which the MMA warp waits on.
    if (ring % 2 == 0) mbar_arrive(&bars.kv_full[ring > 0 ? (ring - 1) % L::kSlots : 0]);
    // Let every issued copy land before the CTA can exit (a K tile completes
    // with the V tile before it; any older pair has completed, since a later
    // tile reused its slot).
    for (uint32_t r = ring > L::kSlots ? ring - L::kSlots : 0; r < ring; ++r)
        if (r == 0 || r % 2 == 1) mbar_wait_drain(&bars.kv_full[r % L::kSlots], (r / L::kSlots) & 1);
    if (q_loads) mbar_wait_drain(&bars.q_full, (q_loads - 1) & 1);
}

// ---------------------------------------------------------------------------
// MMA issuer (one thread).  Order per item (FA-style ping-pong of the two
// query tiles so one tile's softmax overlaps the other tile's products):
//   S0=Q0K0, S1=Q1K0, then for each block j: O0+=P0Vj, S0=Q0K(j+1),
//   O1+=P1Vj, S1=Q1K(j+1).
// ---------------------------------------------------------------------------
template <int D, bool kSparse, bool kMx>
__device__ void fwd_mma_role(const FwdParams& p, uint8_t* smem, FwdBars& bars, uint32_t tmem, int ib, int ie,
                             const AbortState& ab) {
    using L = FwdLayout<D>;
    // The whole warp runs this role (uniform control flow and operands); only
    // lane 0 issues the products and commits.
    const uint32_t lead = (threadIdx.x & 31) == 0 ? 1u : 0u;
    const uint64_t q_desc = kmajor_desc(smem_u32(smem + L::kQOff));
    const uint64_t k_desc = kmajor_desc(smem_u32(smem + L::kRingOff));
    const uint64_t v_desc = kMx ? smem_desc_swz(smem_u32(smem + L::kRingOff), 16384, 8 * D, D == 128 ? 2u : 4u)
                                : mnmajor_desc(smem_u32(smem + L::kRingOff));
    constexpr uint64_t kTileUnits = L::kTileBytes / 16;  // descriptor step between tiles
    uint32_t ring = 0, q_ph = 0;
    uint32_t p_ph[2] = {0, 0};
    QKey qk;
    WorkItem wn = load_item(p.items, ib, ie), wn2 = load_item(p.items, ib + 1, ie);
    // Paired ring: only the stream's first K tile has a barrier phase of its
    // own (the load warp closes it even when it loads nothing); every later K
    // lands with the V tile before it.
    if (!mbar_wait(&bars.kv_full[0], 0, ab)) goto done;
    for (int i = ib; i < ie; ++i) {
        const WorkItem wc = wn;
        wn = wn2;  // item i + 1, loaded an iteration ago
        wn2 = load_item(p.items, i + 2, ie);
        const FwdItem it = decode_fwd<kSparse>(wc, p);
        if (it.nb == 0) continue;
        if (!(p.broadcast_q && qk.same(it))) {
            if (!mbar_wait(&bars.q_full, q_ph, ab)) goto done;
            q_ph ^= 1;
            qk.set(it);
        }
        const bool release_q = !next_item_reuses_q<kSparse>(p, it, wn, i, ie);  // this item is the run's last Q user
        const uint32_t kpos = ring;
        uint32_t kslot = kpos % L::kSlots;  // landed with the V tile before it (or the stream's first K)
        ++ring;
        tc_fence_after();
#pragma unroll
        for (int t = 0; t < 2; ++t)
            if (it.nblk[t] > 0) {
                issue_qk<D>(lead, tmem + t * 128, q_desc + t * kTileUnits, k_desc + kslot * kTileUnits);
                mma_commit_p(lead, &bars.s_full[t]);
            }
        // (paired: this K frees its slot together with the previous item's last V)
        mma_commit_p(lead, &bars.kv_empty[kpos > 0 ? (kpos - 1) % L::kSlots : kslot]);
        if (it.nb == 1 && release_q) mma_commit_p(lead, &bars.q_empty);
        for (int j = 0; j < it.nb; ++j) {
            const uint32_t vslot = ring % L::kSlots;
            if (!mbar_wait(&bars.kv_full[vslot], (ring / L::kSlots) & 1, ab)) goto done;  // V(j) and K(j+1)
            ++ring;
            const bool has_next = j + 1 < it.nb;
            if (has_next) {
                kslot = ring % L::kSlots;
                ++ring;
            }
            tc_fence_after();
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                if (j >= it.nblk[t]) continue;
                if (!mbar_wait(&bars.p_full[t], p_ph[t], ab)) goto done;
                p_ph[t] ^= 1;
                tc_fence_after();
                if (kMx)
                    issue_pv_mx<D>(lead, tmem + L::kOCol + t * D, tmem + t * 128, v_desc + vslot * kTileUnits, j > 0);
                else
                    issue_pv<D>(lead, tmem + L::kOCol + t * D, tmem + t * 128, v_desc + vslot * kTileUnits, j > 0);
                if (j == it.nblk[t] - 1) mma_commit_p(lead, &bars.o_full[t]);
                if (j + 1 < it.nblk[t]) {
                    issue_qk<D>(lead, tmem + t * 128, q_desc + t * kTileUnits, k_desc + kslot * kTileUnits);
                    mma_commit_p(lead, &bars.s_full[t]);
                }
            }
            // V(j) and K(j+1) are free: one commit for the pair (an item's last V
            // goes with the next item's first K)
            if (has_next) {
                mma_commit_p(lead, &bars.kv_empty[vslot]);
                if (j + 2 == it.nb && release_q) mma_commit_p(lead, &bars.q_empty);
            }
        }
    }
done:
    // All issued MMAs must finish before TMEM is released.  A CTA that never
    // took a K/V tile (no items, or only empty ones) issued none.
    if (ring > 0) {
        mma_commit_p(lead, &bars.mma_done);
        mbar_wait_drain(&bars.mma_done, 0);
    }
}

// ---------------------------------------------------------------------------
// Softmax / correction / epilogue (one warpgroup per query tile; thread r
// owns query row r of the tile = TMEM lane r).
// ---------------------------------------------------------------------------
template <int D, bool kSparse, bool kMask>
__device__ __forceinline__ void softmax_block(const FwdParams& p, const FwdItem& it, int j, int qpos,
                                              uint32_t s_addr, uint32_t o_addr, float& m_use, float& l) {
    uint32_t sr[4][32];
#pragma unroll
    for (int c = 0; c < 4; ++c) tmem_ld32(s_addr + c * 32, sr[c]);
    tmem_ld_wait();
    if (kMask) {
        // Keys kbase .. kbase + nvis - 1 are visible to this row: the
        // sequence end and (causal) the diagonal bound one count.
        const int kbase = 128 * kv_block<kSparse>(p, it, j);
        int nvis = it.Lk - kbase;
        if (p.causal) nvis = min(nvis, qpos - kbase + 1);
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int i = 0; i < 32; ++i)
                if (c * 32 + i >= nvis) sr[c][i] = __float_as_uint(-INFINITY);
    }
    // Row max: 8 independent running maxima (short dependency chains), then
    // a 3-level tree; three-input max halves the instruction count.
    float mxs[8];
#pragma unroll
    for (int a = 0; a < 8; ++a) mxs[a] = fmaxf(__uint_as_float(sr[a / 2][(a % 2) * 16]),
                                               __uint_as_float(sr[a / 2][(a % 2) * 16 + 1]));
#pragma unroll
    for (int a = 0; a < 8; ++a) {
        const uint32_t* src = &sr[a / 2][(a % 2) * 16];
#pragma unroll
        for (int i = 2; i < 16; i += 2) mxs[a] = fmax3(mxs[a], __uint_as_float(src[i]), __uint_as_float(src[i + 1]));
    }
    const float mx = fmaxf(fmax3(mxs[0], mxs[1], mxs[2]), fmax3(fmax3(mxs[3], mxs[4], mxs[5]), mxs[6], mxs[7]));
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
    // P = 2^(s * scale_log2 - base): paired FMAs, then the hardware exp2;
    // the row sum uses four paired (add.f32x2) partial sums (ads step:
    // 158.7 vs 164.4 us with eight scalar ones).
    float rss[8];
#pragma unroll
    for (int a = 0; a < 8; ++a) rss[a] = 0.0f;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            float x0, x1;
            ffma2(x0, x1, __uint_as_float(sr[c][2 * e]), __uint_as_float(sr[c][2 * e + 1]), p.scale_log2, p.scale_log2,
                  -base, -base);
            const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
            const int a = (c * 2 + e / 8) & 6;
            float s0 = a == 0 ? rss[0] : a == 2 ? rss[2] : a == 4 ? rss[4] : rss[6];
            float s1 = a == 0 ? rss[1] : a == 2 ? rss[3] : a == 4 ? rss[5] : rss[7];
            fadd2(s0, s1, s0, s1, p0, p1);
            if (a == 0) { rss[0] = s0; rss[1] = s1; }
            else if (a == 2) { rss[2] = s0; rss[3] = s1; }
            else if (a == 4) { rss[4] = s0; rss[5] = s1; }
            else { rss[6] = s0; rss[7] = s1; }
            pk[e] = pack_bf16x2(p0, p1);
        }
        tmem_st16(s_addr + c * 16, pk);
    }
    const float rs = ((rss[0] + rss[1]) + (rss[2] + rss[3])) + ((rss[4] + rss[5]) + (rss[6] + rss[7]));
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

// MXFP8 block: the same online softmax with an integer running max, then
// per 32-key chunk c the exponent X_c = floor(max_c(x) - m) - 8 (x the
// log2-domain logit, m the running max; clamped to E8M0's normal range) and
// the weights 2^(x - m - X_c) rounded to E4M3 (in [0, 512), saturating at
// 448).  Relative to the integer m, X_c + m = floor(max_c(x)) - 8 whatever m
// is, so the quantized weights do not depend on the online schedule.  The row
// sum takes the unquantized weights, sum_c 2^X_c sum_{j in c} 2^(x_j - m - X_c).
// vsc: this lane's words of the block's V scales (column 32 w + lane of
// word w), copied into its lane quarter of the scale columns.
template <int D, bool kMask>
__device__ __forceinline__ void softmax_block_mx(const FwdParams& p, const FwdItem& it, int j, int qpos, int wq,
                                                 uint32_t s_addr, uint32_t o_addr, const uint32_t (&vsc)[D / 32],
                                                 float& m_use, float& l) {
    uint32_t sr[4][32];
#pragma unroll
    for (int c = 0; c < 4; ++c) tmem_ld32(s_addr + c * 32, sr[c]);
    tmem_ld_wait();
    if (kMask) {
        const int kbase = 128 * j;
        int nvis = it.Lk - kbase;
        if (p.causal) nvis = min(nvis, qpos - kbase + 1);
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int i = 0; i < 32; ++i)
                if (c * 32 + i >= nvis) sr[c][i] = __float_as_uint(-INFINITY);
    }
    float mxc[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        float a = fmaxf(__uint_as_float(sr[c][0]), __uint_as_float(sr[c][1]));
        float b = fmaxf(__uint_as_float(sr[c][16]), __uint_as_float(sr[c][17]));
#pragma unroll
        for (int i = 2; i < 16; i += 2) {
            a = fmax3(a, __uint_as_float(sr[c][i]), __uint_as_float(sr[c][i + 1]));
            b = fmax3(b, __uint_as_float(sr[c][16 + i]), __uint_as_float(sr[c][17 + i]));
        }
        mxc[c] = fmaxf(a, b);
    }
    const float mx = fmaxf(fmaxf(mxc[0], mxc[1]), fmaxf(mxc[2], mxc[3]));
    const float m_new = fmaxf(m_use, mx * p.scale_log2);
    float corr = 1.0f;
    bool resc = false;
    if (j == 0) {
        m_use = ceilf(m_new);
    } else if (m_new > m_use + kRescaleLog2) {
        const float m_int = ceilf(m_new);
        corr = ex2_approx(m_use - m_int);
        m_use = m_int;
        resc = true;
    }
    const float base = m_use == -INFINITY ? 0.0f : m_use;
    uint32_t sfa = 0;
    float rs = 0.0f;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const float xm = fmaf(mxc[c], p.scale_log2, -base);
        const int e = xm == -INFINITY ? -126 : max(-126, min(127, static_cast<int>(floorf(xm)) - 8));
        const float cb = base + static_cast<float>(e);
        float r0 = 0.0f, r1 = 0.0f;
        uint32_t pk[8];
#pragma unroll
        for (int w = 0; w < 8; ++w) {
            float x0, x1, x2, x3;
            ffma2(x0, x1, __uint_as_float(sr[c][4 * w]), __uint_as_float(sr[c][4 * w + 1]), p.scale_log2,
                  p.scale_log2, -cb, -cb);
            ffma2(x2, x3, __uint_as_float(sr[c][4 * w + 2]), __uint_as_float(sr[c][4 * w + 3]), p.scale_log2,
                  p.scale_log2, -cb, -cb);
            const float p0 = ex2_approx(x0), p1 = ex2_approx(x1), p2 = ex2_approx(x2), p3 = ex2_approx(x3);
            fadd2(r0, r1, r0, r1, p0, p1);
            fadd2(r0, r1, r0, r1, p2, p3);
            pk[w] = cvt_e4m3x2(p0, p1) | (cvt_e4m3x2(p2, p3) << 16);
        }
        tmem_st8(s_addr + c * 8, pk);
        rs += (r0 + r1) * exp2i(e);
        sfa |= static_cast<uint32_t>(e + 127) << (8 * c);
    }
    tmem_st1(s_addr + kSfaCol + wq, sfa);
    if constexpr (D == 128) tmem_st4(s_addr + kSfbCol, vsc);
    else tmem_st2(s_addr + kSfbCol, vsc);
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

// This lane's words of the V scales of key block blk (column 32 w + lane).
template <int D>
__device__ __forceinline__ void load_vscale(const FwdParams& p, int64_t blk, int h, uint32_t (&v)[D / 32]) {
    const uint32_t* src = p.v_scale + (blk * p.H + h) * D + (threadIdx.x & 31);
#pragma unroll
    for (int w = 0; w < D / 32; ++w) v[w] = __ldg(src + 32 * w);
}

template <int D, bool kSparse, bool kMx>
__device__ void fwd_softmax_role(const FwdParams& p, const CUtensorMap* map_o, uint8_t* smem, FwdBars& bars,
                                 uint32_t tmem, int ib, int ie, const AbortState& ab) {
    using L = FwdLayout<D>;
    const int t = threadIdx.x / 128;
    const int row = threadIdx.x % 128;
    const int wq = (threadIdx.x / 32) % 4;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t s_addr = tmem + lane_off + t * 128;
    const uint32_t o_addr = tmem + lane_off + L::kOCol + t * D;
    uint32_t s_ph = 0, o_ph = 0;
    WorkItem wn = load_item(p.items, ib, ie);
    for (int i = ib; i < ie; ++i) {
        const WorkItem wc = wn;
        wn = load_item(p.items, i + 1, ie);
        const FwdItem it = decode_fwd<kSparse>(wc, p);
        if (t >= it.nq) continue;
        const int nblk = t == 0 ? it.nblk[0] : it.nblk[1];   // scalar copies: no
        const int nfull = t == 0 ? it.nfull[0] : it.nfull[1];  // dynamic array indexing
        const int qpos = 128 * (it.m0 + t) + row;
        const bool valid = qpos < it.q_rows;
        const int64_t orow = p.broadcast_q ? static_cast<int64_t>(it.b) * p.Lq + qpos
                                           : static_cast<int64_t>(it.q_row0) + qpos;
        uint16_t* optr = p.o + (orow * p.H + it.h) * D;  // this row of O (empty-sequence path)
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
        // MXFP8: this lane's V-scale words, fetched one block ahead
        uint32_t vsc[D / 32], vsn[D / 32];
        const int64_t blk0 = !kMx ? 0
                             : it.slot >= 0 ? static_cast<int64_t>(__ldg(p.split_block0 + it.slot))
                                            : static_cast<int64_t>(__ldg(p.block_start + it.b));
        if (kMx) load_vscale<D>(p, blk0, it.h, vsn);
        for (; j < nfull; ++j) {  // bulk: every key visible, no mask
            if (kMx) {
#pragma unroll
                for (int w = 0; w < D / 32; ++w) vsc[w] = vsn[w];
                if (j + 1 < nblk) load_vscale<D>(p, blk0 + j + 1, it.h, vsn);
            }
            if (!mbar_wait_warp(&bars.s_full[t], s_ph, ab)) goto done;
            s_ph ^= 1;
            tc_fence_after();
            if constexpr (kMx)
                softmax_block_mx<D, false>(p, it, j, qpos, wq, s_addr, o_addr, vsc, m_use, l);
            else
                softmax_block<D, kSparse, false>(p, it, j, qpos, s_addr, o_addr, m_use, l);
            handoff_arrive(&bars.p_full[t]);
        }
        for (; j < nblk; ++j) {  // tail: ragged end and/or causal diagonal
            if (kMx) {
#pragma unroll
                for (int w = 0; w < D / 32; ++w) vsc[w] = vsn[w];
                if (j + 1 < nblk) load_vscale<D>(p, blk0 + j + 1, it.h, vsn);
            }
            if (!mbar_wait_warp(&bars.s_full[t], s_ph, ab)) goto done;
            s_ph ^= 1;
            tc_fence_after();
            if constexpr (kMx)
                softmax_block_mx<D, true>(p, it, j, qpos, wq, s_addr, o_addr, vsc, m_use, l);
            else
                softmax_block<D, kSparse, true>(p, it, j, qpos, s_addr, o_addr, m_use, l);
            handoff_arrive(&bars.p_full[t]);
        }
        // Epilogue: O / l to bf16, LSE = ln(sum exp) of the scaled scores.
        // O leaves TMEM first (freeing it for the next item's PV), then goes
        // out through a 128-byte-swizzled smem stage in 64-column halves, so
        // each warp store covers four whole 128-byte segments.
        if (!mbar_wait_warp(&bars.o_full[t], o_ph, ab)) goto done;
        o_ph ^= 1;
        tc_fence_after();
        {
            uint32_t orr[D / 32][32];
#pragma unroll
            for (int oc = 0; oc < D / 32; ++oc) tmem_ld32(o_addr + oc * 32, orr[oc]);
            tmem_ld_wait();
            const float inv = l > 0.0f ? 1.0f / l : 0.0f;
            if (!kSparse && it.slot >= 0) {  // split-KV chunk: fp32 O and LSE of its keys for the merge pass
                if (valid) {
                    const int64_t prow = static_cast<int64_t>(it.slot) * 128 + row;
                    p.lse_part[prow] = l > 0.0f ? (m_use + lg2_approx(l)) * kLn2 : -INFINITY;
                    float4* dst = reinterpret_cast<float4*>(p.o_part + prow * D);
#pragma unroll
                    for (int c = 0; c < D / 4; ++c) {
                        const uint32_t* f = &orr[c / 8][(c % 8) * 4];
                        dst[c] = make_float4(__uint_as_float(f[0]) * inv, __uint_as_float(f[1]) * inv,
                                             __uint_as_float(f[2]) * inv, __uint_as_float(f[3]) * inv);
                    }
                }
                continue;
            }
            if (valid) p.lse[lse_idx] = l > 0.0f ? (m_use + lg2_approx(l)) * kLn2 : -INFINITY;
            uint8_t* stage = smem + L::kStageOff + t * L::kStageBytes;
            const int64_t row0 = p.broadcast_q ? static_cast<int64_t>(it.b) * p.Lq + 128 * (it.m0 + t)
                                               : static_cast<int64_t>(it.q_row0) + 128 * (it.m0 + t);
            const int rows_valid = min(128, it.q_rows - 128 * (it.m0 + t));
#pragma unroll
            for (int half = 0; half < D / 64; ++half) {
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {  // 8 bf16 per 16-byte chunk
                    const uint32_t* f = &orr[half * 2 + ch / 4][(ch % 4) * 8];
                    const uint4 u = make_uint4(pack_bf16x2(__uint_as_float(f[0]) * inv, __uint_as_float(f[1]) * inv),
                                               pack_bf16x2(__uint_as_float(f[2]) * inv, __uint_as_float(f[3]) * inv),
                                               pack_bf16x2(__uint_as_float(f[4]) * inv, __uint_as_float(f[5]) * inv),
                                               pack_bf16x2(__uint_as_float(f[6]) * inv, __uint_as_float(f[7]) * inv));
                    *reinterpret_cast<uint4*>(stage + row * 128 + ((ch ^ (row & 7)) * 16)) = u;
                }
                group_sync(1 + t);
                // 128 rows x 8 chunks: thread k of the warpgroup copies chunks k, k+128, ...
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int q = row + 128 * k;
                    const int r = q >> 3, ch = q & 7;
                    if (r < rows_valid) {
                        const uint4 u = *reinterpret_cast<const uint4*>(stage + r * 128 + ((ch ^ (r & 7)) * 16));
                        *reinterpret_cast<uint4*>(p.o + ((row0 + r) * p.H + it.h) * D + half * 64 + ch * 8) = u;
                    }
                }
                group_sync(1 + t);
            }
        }
    }
done:
    return;
}

template <int D, bool kSparse, bool kMx>
__global__ void __launch_bounds__(kFwdThreads, 1)
    jfa_fwd_kernel(const FwdParams p, const __grid_constant__ CUtensorMap map_q,
                   const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v,
                   const __grid_constant__ CUtensorMap map_o) {
    using L = FwdLayout<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024(smem_raw);
    __shared__ FwdBars bars;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int ib = p.cta_start[blockIdx.x], ie = p.cta_start[blockIdx.x + 1];
    const AbortState ab{&bars.abort_flag, p.status, p.wait_ns};

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
            mbar_init(&bars.p_full[t], kHandoffCount);
            mbar_init(&bars.o_full[t], 1);
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
        regs_inc<kSoftmaxRegs>();
        fwd_softmax_role<D, kSparse, kMx>(p, &map_o, smem, bars, tmem, ib, ie, ab);
    } else {
        regs_dec<kAuxRegs>();
        if (warp == kWarpTma) {
            if (lane == 0) fwd_tma_role<D, kSparse, kMx>(p, &map_q, &map_k, &map_v, smem, bars, ib, ie, ab);
            __syncwarp();
        } else if (warp == kWarpMma) {
            fwd_mma_role<D, kSparse, kMx>(p, smem, bars, tmem, ib, ie, ab);
            __syncwarp();
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kWarpMma) tmem_dealloc(tmem, L::kTmemCols);
}

// Split-KV merge (see scheduler.h): LSE = ln sum_c exp(LSE_c) and
// O = sum_c exp(LSE_c - LSE) O_c for every split query tile, written as bf16
// to the broadcast O [B, Lq, H, D] with LSE [B, H, Lq].  One CTA per (split
// tile, 32-row block, 32-column slice); lane = row, and the 8 warps share the
// chunks (warp w takes c = w, w + 8, ...), their partial maxima, sums and
// weighted rows combined through shared memory.
template <int D>
__global__ void __launch_bounds__(256) jfa_fwd_merge_kernel(const SplitGroup* groups, const float* o_part,
                                                            const float* lse_part, uint16_t* o, float* lse, int Lq,
                                                            int H) {
    constexpr int kSlices = D / 32;
    __shared__ float red_m[8][32], red_s[8][32];
    __shared__ float red_o[8][32][33];
    const int gi = blockIdx.x / (4 * kSlices), rb = (blockIdx.x / kSlices) % 4, cs = blockIdx.x % kSlices;
    const int lane = threadIdx.x % 32, warp = threadIdx.x / 32;
    const int4 g = __ldg(reinterpret_cast<const int4*>(groups) + gi);  // b, slot0, chunks, h | tile << 8
    const int h = g.w & 0xFF, tile = static_cast<int>(static_cast<uint32_t>(g.w) >> 8);
    const int row = rb * 32 + lane;
    const float* lp = lse_part + static_cast<int64_t>(g.y) * 128 + row;
    float mx = -INFINITY;
    for (int c = warp; c < g.z; c += 8) mx = fmaxf(mx, lp[c * 128]);
    red_m[warp][lane] = mx;
    __syncthreads();
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < 8; ++w) M = fmaxf(M, red_m[w][lane]);
    float sum = 0.0f;
    if (M != -INFINITY)
        for (int c = warp; c < g.z; c += 8) sum += expf(lp[c * 128] - M);
    red_s[warp][lane] = sum;
    __syncthreads();
    float S = 0.0f;
#pragma unroll
    for (int w = 0; w < 8; ++w) S += red_s[w][lane];
    const float L = M == -INFINITY ? -INFINITY : M + logf(S);
    float acc[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) acc[e] = 0.0f;
    if (L != -INFINITY) {
#pragma unroll 2
        for (int c = warp; c < g.z; c += 8) {
            const float wt = expf(lp[c * 128] - L);
            const float4* src = reinterpret_cast<const float4*>(
                o_part + (static_cast<int64_t>(g.y + c) * 128 + row) * D + cs * 32);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float4 v = src[e];
                acc[4 * e] += wt * v.x;
                acc[4 * e + 1] += wt * v.y;
                acc[4 * e + 2] += wt * v.z;
                acc[4 * e + 3] += wt * v.w;
            }
        }
    }
#pragma unroll
    for (int e = 0; e < 32; ++e) red_o[warp][lane][e] = acc[e];
    __syncthreads();
    // Thread t: row t % 32 of the block, columns 4 * (t / 32) .. + 3 of the slice.
    const int r = threadIdx.x % 32, e0 = 4 * (threadIdx.x / 32);
    const int q = tile * 128 + rb * 32 + r;
    if (q < Lq) {
        float out[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            float v = 0.0f;
#pragma unroll
            for (int w = 0; w < 8; ++w) v += red_o[w][r][e0 + k];
            out[k] = v;
        }
        const int64_t orow = (static_cast<int64_t>(g.x) * Lq + q) * H + h;
        *reinterpret_cast<uint2*>(o + orow * D + cs * 32 + e0) =
            make_uint2(pack_bf16x2(out[0], out[1]), pack_bf16x2(out[2], out[3]));
    }
    if (cs == 0 && warp == 0 && tile * 128 + row < Lq) lse[(static_cast<int64_t>(g.x) * H + h) * Lq + tile * 128 + row] = L;
}

template <int D, bool kSparse, bool kMx>
cudaError_t launch_fwd_d(const FwdParams& p, const FwdMaps& m, int grid, cudaStream_t s) {
    using L = FwdLayout<D>;
    static bool configured = false;
    if (!configured) {
        // The register split above is only safe if the kernel launches with
        // exactly kLaunchRegs registers per thread; refuse to launch otherwise.
        cudaFuncAttributes fa;
        cudaError_t e = cudaFuncGetAttributes(&fa, jfa_fwd_kernel<D, kSparse, kMx>);
        if (e != cudaSuccess) return e;
        if (fa.numRegs != static_cast<int>(kLaunchRegs)) return cudaErrorInvalidKernelImage;
        e = cudaFuncSetAttribute(jfa_fwd_kernel<D, kSparse, kMx>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 L::kDynSmem);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    jfa_fwd_kernel<D, kSparse, kMx><<<grid, kFwdThreads, L::kDynSmem, s>>>(p, m.q, m.k, m.v, m.o);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_merge(int D, const SplitGroup* groups, int64_t n_groups, const float* o_part,
                             const float* lse_part, uint16_t* o, float* lse, int Lq, int H, cudaStream_t s) {
    if (n_groups <= 0) return cudaSuccess;
    const int grid = static_cast<int>(n_groups) * 4 * (D / 32);
    if (D == 128)
        jfa_fwd_merge_kernel<128><<<grid, 256, 0, s>>>(groups, o_part, lse_part, o, lse, Lq, H);
    else
        jfa_fwd_merge_kernel<64><<<grid, 256, 0, s>>>(groups, o_part, lse_part, o, lse, Lq, H);
    return cudaGetLastError();
}

cudaError_t launch_fwd(int D, const FwdParams& p, const FwdMaps& m, int grid, cudaStream_t s) {
    if (grid <= 0) return cudaSuccess;
    if (p.sel)
        return D == 128 ? launch_fwd_d<128, true, false>(p, m, grid, s) : launch_fwd_d<64, true, false>(p, m, grid, s);
    if (p.v_scale)
        return D == 128 ? launch_fwd_d<128, false, true>(p, m, grid, s) : launch_fwd_d<64, false, true>(p, m, grid, s);
    return D == 128 ? launch_fwd_d<128, false, false>(p, m, grid, s) : launch_fwd_d<64, false, false>(p, m, grid, s);
}

}  // namespace jfa
