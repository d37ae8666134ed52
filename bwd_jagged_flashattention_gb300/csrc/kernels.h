// kernels.h -- launch parameters of the attention kernels and the host-side
// launch functions (implemented in fwd.cu / bwd.cu, called by jfa_api.cu).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "scheduler.h"

namespace jfa {

struct FwdParams {
    const WorkItem* items;     // device, CSR-ordered by CTA
    const int32_t* cta_start;  // device, [grid + 1]
    uint16_t* o;               // bf16 output
    float* lse;                // fp32 output
    uint32_t* status;          // device status word
    int Lq, H, N;
    int broadcast_q, causal;
    float scale_log2;          // softmax scale * log2(e)
    uint64_t wait_ns = 4000000000ull;    // limit of one barrier wait (jfa_set_wait_limit)
    const SparseSel* sel = nullptr;      // block-sparse: selection per (b, h) at b * H + h; null = dense
    const int32_t* sel_blocks = nullptr; // block-sparse: the selected block indices the records point into
    float* o_part = nullptr;             // split-KV chunks: fp32 O [slot][128][D] (null: no split items)
    float* lse_part = nullptr;           // split-KV chunks: fp32 LSE [slot][128]
    // MXFP8 P V (null: bf16 V): E8M0 scales of V, one 32-bit word (the four
    // 32-key chunks of a 128-key block) per (block, head, column) at
    // (block_start[b] + n) * H * D + h * D + d; block_start[b] = first block of sequence b.
    const uint32_t* v_scale = nullptr;
    const int32_t* block_start = nullptr;
    // MXFP8 split-KV chunks: per slot, the first key block of the chunk (in the
    // numbering of block_start); a chunk's work item carries its slot, not b.
    const int32_t* split_block0 = nullptr;
};

struct BwdParams {
    const WorkItem* items;
    const int32_t* cta_start;
    const float* lse;          // [B,H,Lq] or [H,N]
    uint16_t* dk;              // bf16 [N,H,D]
    uint16_t* dv;              // bf16 [N,H,D]
    uint32_t* status;
    int Lq, H, N;
    int broadcast_q, causal;
    // 1: items dealt at run time -- by Cluster Launch Control (queue null: one
    // CTA per item of the cost-sorted list, each resident CTA taking over CTAs
    // that have not started) or from queues (queue set: CTA c takes the next
    // item of queue c % n_queues, items [cta_start[g], cta_start[g + 1]), by
    // atomically incrementing queue[g]); 0: the static schedule, CTA p owning
    // items [cta_start[p], cta_start[p + 1]).
    int clc;
    int n_items;               // items in the list (the grid size with Cluster Launch Control)
    int n_queues;
    int32_t* queue;            // take counters (zero at launch), or null
    float scale, scale_log2;
    uint64_t wait_ns;          // limit of one barrier wait (jfa_set_wait_limit)
    const float* delta;        // same layout as lse (the pre-pass writes it)
};

struct PreParams {
    const uint16_t* o;         // bf16, O layout
    const uint16_t* dout;      // bf16, O layout
    float* delta;              // fp32, LSE layout
    float* dq;                 // fp32 dQ, zeroed by the same kernel (dq_vec4 float4 vectors)
    int64_t dq_vec4;
    int64_t rows;              // number of (row, head) pairs = O rows * H
    int B, Lq, H, N, D;
    int broadcast_q;
    // Optional: the backward's tile schedule, copied by this kernel from the
    // host's pinned staging buffer (its device mapping) into the workspace.
    const uint4* sched_src = nullptr;
    uint4* sched_dst = nullptr;
    int64_t sched_vec16 = 0;
};

#ifdef __CUDACC__
// Work item i of a CTA's list as one 16-byte load (an all-zero item past the
// end).  The kernels read each item one iteration ahead, so the load's latency
// hides behind the previous item's work instead of delaying the item's start.
__device__ __forceinline__ WorkItem load_item(const WorkItem* items, int i, int ie) {
    if (i >= ie) return WorkItem{0, 0, 0, 0u};
    const int4 v = __ldg(reinterpret_cast<const int4*>(items) + i);
    return WorkItem{v.x, v.y, v.z, static_cast<uint32_t>(v.w)};
}
#endif

// Tensor maps for one call.  Q/K/V/dO are viewed as 2D [rows, H*D] bf16
// with 64x128 boxes (128-byte swizzle); dQ as 2D [rows, H*D] fp32.
struct FwdMaps {
    CUtensorMap q, k, v;
    CUtensorMap o;  // bf16 [O rows, H*D] output, same boxes (O TMA stores)
};
struct BwdMaps {
    CUtensorMap q, k, v, dout, dq;
    CUtensorMap dk, dv;  // bf16 [N, H*D] outputs, same boxes as K/V (dK/dV TMA stores)
};

cudaError_t launch_fwd(int D, const FwdParams& p, const FwdMaps& m, int grid, cudaStream_t s);
// Split-KV merge of n_groups split query tiles into the broadcast O / LSE.
cudaError_t launch_fwd_merge(int D, const SplitGroup* groups, int64_t n_groups, const float* o_part,
                             const float* lse_part, uint16_t* o, float* lse, int Lq, int H, cudaStream_t s);
// Delta = rowsum(dO * O) in fp32 (LSE layout), and dQ zeroed, before launch_bwd on the same stream.
cudaError_t launch_bwd_pre(const PreParams& p, cudaStream_t s);
cudaError_t launch_bwd(int D, const BwdParams& p, const BwdMaps& m, int grid, cudaStream_t s);
// MXFP8 quantization of bf16 V [N,H,D] into E4M3 codes (same layout) and
// E8M0 scales [NB,H,D,4]: one CTA per 128-key block (NB blocks in total;
// block_start has B + 1 entries).
cudaError_t launch_quant_v_mxfp8(const uint16_t* v, const int32_t* offsets, const int32_t* block_start, int B,
                                 int64_t n_blocks, int H, int D, uint8_t* v8, uint32_t* v_scale, cudaStream_t s);
// Block-sparse backward: zero the dK and dV rows of the n unselected key tiles.
cudaError_t launch_zero_tiles(const ZeroTile* tiles, int64_t n, uint16_t* dk, uint16_t* dv, int H, int D,
                              cudaStream_t s);

}  // namespace jfa
