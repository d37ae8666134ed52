// scheduler.h -- host tile scheduler: work items, cost model, LPT sort and
// zigzag deal to persistent CTAs.
//
// The pages describe this step for the forward pass: tiles are sorted on the
// host by their KV workload in descending order and handed to the SMs in a
// zigzag pattern, which recovered about 20% of forward time at negligible CPU
// cost (Meta's TLX Jagged Flash Attention Beats FA4 on Blackwell With 3x Less
// Code, section "Optimizations layered on top", the paragraph after the
// list; "Scheduling jagged tiles across SMs" in the same list).  The backward
// uses the same sort over its own items.  For the forward the library deals
// each sorted item to the CTA with the least work so far (greedy longest-
// processing-time, kSchedLptGreedy), the rule the zigzag approximates: on the
// ads forward (about 13 items per CTA, item costs up to 65 block products)
// zigzag leaves the busiest CTA 1.32x the mean load, greedy 1.02x (forward
// 158 -> 136 us).  The backward keeps the zigzag: its items are nearly
// uniform (every CTA within 1.3% of the mean either way), and with equal costs
// the greedy rule degenerates to round-robin, measured 2% slower.
//
// Broadcast Q (one dense Q shared by every sequence): when the head count H
// divides the CTA count P, each head gets its own group of P/H CTAs (CTAs
// h, h+H, h+2H, ...) and the sort and deal run within each group.  Every head has the same item
// costs, so the groups' loads match and CTA g of every group works on the
// same sequences at the same time (their K/V/dO rows, which interleave the
// heads in memory, are read together), while each CTA only ever reads one
// head's Q tiles.  Each CTA's items are then grouped (stably) by the Q tiles
// they read -- head, and for the forward the first query tile -- so that runs
// of consecutive items share the resident Q tiles.  The order of a CTA's own
// items does not change its total work, only how often it reloads Q.
#pragma once
#include <cstdint>

namespace jfa {

// One unit of persistent-kernel work (16 bytes, read once per item).
//   forward : query tiles [tile, tile + 1 + two) of sequence b, head h
//   backward: key/value tile `tile` of sequence b, head h
struct WorkItem {
    int32_t b;         // sequence index
    int32_t kv_start;  // first packed row of the sequence (offsets[b])
    int32_t kv_len;    // sequence length (offsets[b+1] - offsets[b])
    uint32_t packed;   // h | tile << 8 | two << 31
};
static_assert(sizeof(WorkItem) == 16, "WorkItem must stay 16 bytes");

constexpr int kTileRows = 128;          // rows per Q or K/V tile
constexpr int kMaxCtas = 1023;          // schedule bound on persistent CTAs
constexpr int kMaxSeqLen = 1 << 23;     // tile index must fit 23 bits

inline uint32_t pack_item(int h, int tile, int two) {
    return static_cast<uint32_t>(h) | (static_cast<uint32_t>(tile) << 8) | (static_cast<uint32_t>(two) << 31);
}

enum SchedPolicy {
    kSchedLptZigzag = 0,  // cost-descending stable sort, then zigzag deal (the pages' deal)
    kSchedNaive = 1,      // generation order, round-robin deal (ablation)
    kSchedLptGreedy = 2,  // cost-descending stable sort, each item to the least-loaded CTA (the library's)
    kSchedClc = 3,        // backward only: the cost-sorted list, one CTA per item, dealt at run time by
                          // Cluster Launch Control (each resident CTA takes over CTAs not yet started)
    kSchedQueue = 4,      // backward only: one cost-sorted queue per head group (broadcast Q, H | P; else one
                          // queue), taken from at run time by the persistent CTAs of that group
};

// kSchedQueue layout of cta_start: entries 0..G are the queues' bounds (queue
// g = items [cta_start[g], cta_start[g + 1])), entries G+1 .. 2G are the
// queues' take counters, zero in the uploaded schedule.

// Whether broadcast-Q items are dealt per head group (H divides P).
bool head_partition(int broadcast_q, int H, int P);
// Number of queues of a kSchedQueue schedule.
inline int queue_groups(int broadcast_q, int H, int P) { return head_partition(broadcast_q, H, P) ? H : 1; }

// Upper bound on the number of items either pass produces.
int64_t max_work_items(int B, int64_t total_len, int Lq, int H, int broadcast_q);

// Block-sparse selection (the pages' block-sparse variant only adds
// iteration over selected key blocks: TLX porta l'attenzione jagged su
// Blackwell oltre FA4 con un terzo del codice, section "The turning point").
// Keys come in blocks of 128 counted from each sequence's start; block n of
// sequence b is selected for head h iff mask[(block_start[b] + n) * H + h]
// != 0, block_start[b] = sum over b' < b of ceil(len_b' / 128).
struct SparseSel {     // forward, one per (b, h) at index b * H + h
    int32_t off;       // first entry of the pair's selected blocks in the block list
    int32_t n_sel;     // selected blocks (ascending block indices)
    int32_t n_full;    // of those, blocks with 128 keys (all but a ragged last block)
    int32_t pad;
};
struct ZeroTile {      // backward: an unselected key tile, whose dK and dV rows are zero
    int32_t row0;      // first packed row
    int32_t rows;      // rows in the tile (<= 128)
    int32_t h;         // head
    int32_t pad;
};
static_assert(sizeof(SparseSel) == 16 && sizeof(ZeroTile) == 16, "16-byte records");
struct SparseSpec {
    const uint8_t* mask;  // host uint8 [NB, H]
    SparseSel* sel;       // out (forward): B * H records
    int32_t* blocks;      // out (forward): selected block indices, capacity cap
    ZeroTile* zero;       // out (backward): capacity cap
    int64_t cap;          // >= NB * H
    int64_t n_blocks = 0, n_zero = 0;  // out: entries written
};

// NB = sum_b ceil(len_b / 128).
int64_t num_kv_blocks(const int32_t* offsets, int B);

// Split-KV for the broadcast-Q forward (load balance under length skew): a
// query tile of one (sequence, head) whose key loop alone costs more than
// 1.5x an average CTA's share of the work is cut into key chunks, each a work item of
// its own that writes its O (normalised by its own row sums) and its LSE in
// fp32 to a slot; a merge pass combines each split tile's chunks:
//     LSE = ln sum_c exp(LSE_c),   O = sum_c exp(LSE_c - LSE) O_c.
// A chunk item is encoded like a shorter sequence: kv_start / kv_len cover
// the chunk's keys, the packed field holds (h, query tile, one tile), and
// b = -(slot + 1) marks it.
constexpr int kMaxSplitSlots = 512;   // partial (O, LSE) slots in a workspace
constexpr int kMinSplitBlocks = 4;    // key blocks per chunk, at least
struct SplitGroup {                   // one split query tile; its chunks own slots [slot0, slot0 + n)
    int32_t b;
    int32_t slot0;
    int32_t n;
    uint32_t packed;                  // h | query tile << 8
};
static_assert(sizeof(SplitGroup) == 16, "16-byte record");
struct SplitSpec {
    SplitGroup* groups;               // out: capacity kMaxSplitSlots
    int64_t n_groups = 0, n_slots = 0;
    // out (if set; capacity kMaxSplitSlots): per slot, the index of its
    // chunk's first 128-key block over all sequences' blocks in order -- what
    // the MXFP8 forward needs to find the chunk's V scales.
    int32_t* slot_block0 = nullptr;
};

// Build a schedule.  Writes `n` items into `items` (capacity max_items) and
// the CSR bounds cta_start[0..P] (CTA p owns items [cta_start[p],
// cta_start[p+1])).  Returns n, or -1 if a capacity is too small.
// is_bwd selects the backward item decomposition and cost.  With `sparse`
// (not causal): forward items keep their query tiles and cost the selected
// blocks only, and sparse->sel / blocks list each pair's selected blocks;
// backward items exist only for selected key tiles, the others go to
// sparse->zero.
// With `split` (broadcast-Q forward without a block-sparse selection):
// split-KV as above.
int64_t build_schedule(const int32_t* offsets, int B, int Lq, int H, int broadcast_q, int causal, int is_bwd,
                       int P, int policy, WorkItem* items, int32_t* cta_start, int64_t max_items,
                       SparseSpec* sparse = nullptr, SplitSpec* split = nullptr);

// Allocation-free twin of build_schedule with kSchedLptGreedy (same items,
// order and deal) for callers that cannot allocate: every array comes from
// the caller.
//   gen, order, owner: capacity max_items each; fill: P entries;
//   buckets: kCostBuckets + 2 entries.  Costs of kCostBuckets - 1 or more
//   share the last bucket (their relative order stays the generation order).
constexpr int64_t kCostBuckets = 65536;
int64_t build_schedule_noalloc(const int32_t* offsets, int B, int Lq, int H, int broadcast_q, int causal, int is_bwd,
                               int P, WorkItem* items, int32_t* cta_start, int64_t max_items, WorkItem* gen,
                               int64_t* order, int32_t* owner, int32_t* fill, int64_t* buckets);

// Cost of one item in 128x128 block-products (+1 fixed per-item overhead).
int64_t item_cost(const WorkItem& w, int Lq, int broadcast_q, int causal, int is_bwd);

}  // namespace jfa
