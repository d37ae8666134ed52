// scheduler.cpp -- see scheduler.h.
#include "scheduler.h"

#include <algorithm>
#include <vector>

namespace jfa {

namespace {
inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Host scratch of the builders, kept per thread across calls: the schedule
// is rebuilt on every call, and fresh allocations of this size cost more in
// page faults than the whole build.
struct Scratch {
    std::vector<WorkItem> gen;
    std::vector<int64_t> cost, order, heap, buckets;
    std::vector<int32_t> owner, fill;
};
Scratch& scratch() {
    static thread_local Scratch s;
    return s;
}
}  // namespace

bool head_partition(int broadcast_q, int H, int P) { return broadcast_q && H > 1 && H <= 255 && P % H == 0; }

int64_t max_work_items(int B, int64_t total_len, int Lq, int H, int broadcast_q) {
    if (B <= 0 || H <= 0) return 0;
    // backward: sum_b ceil(L_b/128) <= N/128 + B; forward pairs of q tiles
    // are never more.  Broadcast forward: B * ceil(ceil(Lq/128)/2).
    int64_t bwd = static_cast<int64_t>(H) * (total_len / kTileRows + B);
    int64_t fwd = broadcast_q ? static_cast<int64_t>(B) * H * ceil_div(ceil_div(std::max(Lq, 0), kTileRows), 2)
                              : static_cast<int64_t>(H) * (total_len / (2 * kTileRows) + B);
    return std::max<int64_t>(std::max(bwd, fwd), 1);
}

int64_t num_kv_blocks(const int32_t* offsets, int B) {
    int64_t nb = 0;
    for (int b = 0; b < B; ++b) nb += ceil_div(offsets[b + 1] - offsets[b], kTileRows);
    return nb;
}

int64_t item_cost(const WorkItem& w, int Lq, int broadcast_q, int causal, int is_bwd) {
    const int64_t Lk = w.kv_len;
    const int tile = static_cast<int>((w.packed >> 8) & 0x7FFFFFu);
    const int two = static_cast<int>(w.packed >> 31);
    const int64_t nkv = ceil_div(Lk, kTileRows);
    if (!is_bwd) {
        int64_t blocks = 0;
        for (int t = 0; t <= two; ++t) {
            const int64_t m = tile + t;
            blocks += causal ? std::min<int64_t>(m + 1, nkv) : nkv;
        }
        return blocks + 1;
    }
    const int64_t nq = broadcast_q ? ceil_div(Lq, kTileRows) : nkv;
    const int64_t visited = causal ? (nq - tile) : nq;
    return visited + 1;
}

namespace {

// CTA of the item at position pos of head h's cost-sorted items, dealt
// zigzag over that head's G CTAs {h, h + H, h + 2H, ...}: the H CTAs that
// work on the same sequences at the same time have neighbouring indices.
inline int32_t zigzag_head_cta(int64_t pos, int h, int G, int H) {
    const int64_t r = pos / G, lane = pos % G;
    return static_cast<int32_t>(((r & 1) ? (G - 1 - lane) : lane) * H + h);
}

// Restore the min-heap property below slot k of heap[0..size).
inline void sift_down(int64_t* heap, int size, int k) {
    for (;;) {
        int c = 2 * k + 1;
        if (c >= size) return;
        if (c + 1 < size && heap[c + 1] < heap[c]) ++c;
        if (heap[k] <= heap[c]) return;
        std::swap(heap[k], heap[c]);
        k = c;
    }
}

// Deal the n cost-sorted items gen[order[i]] to CTAs (owner[i]).
//   zigzag: sorted position i, round r = i / P, lane p = i % P; CTA p on even
//           rounds, CTA P-1-p on odd rounds (the pages' deal);
//   greedy: each item to the CTA with the least cost so far (ties: lowest
//           lane) -- the longest-processing-time rule zigzag approximates;
//   naive:  round-robin.
// Broadcast Q with H | P (head_partition()): the deal runs within each head's
// group of G = P/H CTAs {h, h+H, ...}.  heap: scratch of P int64 (greedy).
void deal(const WorkItem* gen, const int64_t* order, const int64_t* cost, int64_t n, int Lq, int H, int broadcast_q,
          int causal, int is_bwd, int P, int policy, int32_t* owner, int64_t* heap) {
    const bool by_head = policy != kSchedNaive && head_partition(broadcast_q, H, P);
    const int groups = by_head ? H : 1, G = P / groups;
    if (policy == kSchedLptGreedy) {
        // One min-heap per group of keys load * 1024 + lane (lane < 1024).
        for (int g = 0; g < groups; ++g)
            for (int lane = 0; lane < G; ++lane) heap[g * G + lane] = lane;  // sorted: a valid heap
        for (int64_t i = 0; i < n; ++i) {
            const WorkItem& w = gen[order[i]];
            const int g = by_head ? static_cast<int>(w.packed & 0xFFu) : 0;
            int64_t* hs = heap + static_cast<int64_t>(g) * G;
            const int lane = static_cast<int>(hs[0] & 1023);
            hs[0] += (cost ? cost[order[i]] : item_cost(w, Lq, broadcast_q, causal, is_bwd)) * 1024;
            sift_down(hs, G, 0);
            owner[i] = by_head ? lane * H + g : lane;
        }
        return;
    }
    // Running (lane, round parity) per group instead of a division per item.
    int lane_of[256] = {0};
    bool odd_of[256] = {false};
    for (int64_t i = 0; i < n; ++i) {
        const int g = by_head ? static_cast<int>(gen[order[i]].packed & 0xFFu) : 0;
        const int lane = lane_of[g];
        const bool zig = policy == kSchedLptZigzag || by_head;
        const int slot = (zig && odd_of[g]) ? G - 1 - lane : lane;
        owner[i] = by_head ? slot * H + g : slot;
        if (++lane_of[g] == G) {
            lane_of[g] = 0;
            odd_of[g] = !odd_of[g];
        }
    }
}

// Key of the Q tiles an item reads in broadcast mode: the head and (forward)
// the first query tile.  Consecutive items of one CTA with equal keys share
// the resident Q tiles, so the kernels load them once per run of equal keys.
inline uint32_t q_key(const WorkItem& w, int is_bwd) {
    const uint32_t h = w.packed & 0xFFu;
    const uint32_t tile = (w.packed >> 8) & 0x7FFFFFu;
    return is_bwd ? h : (h << 23) | tile;
}

// Stable in-place grouping of each CTA's items by q_key (insertion sort: the
// CTA's item count is small, and no allocation is needed).  The deal -- which
// CTA owns which item, and so every CTA's total cost -- is unchanged.
void group_by_q(WorkItem* items, const int32_t* cta_start, int P, int is_bwd) {
    for (int p = 0; p < P; ++p) {
        for (int64_t i = cta_start[p] + 1; i < cta_start[p + 1]; ++i) {
            const WorkItem w = items[i];
            const uint32_t k = q_key(w, is_bwd);
            int64_t j = i;
            while (j > cta_start[p] && q_key(items[j - 1], is_bwd) > k) {
                items[j] = items[j - 1];
                --j;
            }
            items[j] = w;
        }
    }
}

// Split-KV (see scheduler.h): replace every broadcast-Q forward item whose
// cost exceeds 1.5x the average per-CTA load by single-tile key chunks of
// about half that load (at least kMinSplitBlocks blocks), within the slot and
// item capacities; items are taken in generation order, so the result
// depends only on the offsets.  (Items up to 1.5x the average are left to
// the longest-first deal: splitting them cost more in chunk overhead and the
// merge than it gained, e.g. 75.6 vs 67.4 us on the first 256 ads sequences.)
void split_long_items(std::vector<WorkItem>& gen, std::vector<int64_t>& cost, int P, int64_t max_items,
                      const int32_t* offsets, int B, SplitSpec* split) {
    // First 128-key block of every sequence (only for slot_block0).
    std::vector<int64_t> bs;
    if (split->slot_block0) {
        bs.resize(static_cast<size_t>(B) + 1);
        bs[0] = 0;
        for (int b = 0; b < B; ++b) bs[b + 1] = bs[b] + ceil_div(offsets[b + 1] - offsets[b], kTileRows);
    }
    int64_t total = 0;
    for (int64_t c : cost) total += c;
    const int64_t avg = total / P;
    const int64_t chunk = std::max<int64_t>(kMinSplitBlocks, avg / 2);
    std::vector<WorkItem> out_items;
    std::vector<int64_t> out_cost;
    int64_t budget = max_items - static_cast<int64_t>(gen.size());  // extra items the capacity allows
    for (size_t i = 0; i < gen.size(); ++i) {
        const WorkItem& w = gen[i];
        const int64_t nkv = ceil_div(w.kv_len, kTileRows);
        const int tile = static_cast<int>((w.packed >> 8) & 0x7FFFFFu);
        const int tiles = 1 + static_cast<int>(w.packed >> 31);
        const int64_t chunks = ceil_div(nkv, chunk);
        if (2 * cost[i] <= 3 * avg || chunks < 2 || split->n_slots + tiles * chunks > kMaxSplitSlots ||
            tiles * chunks - 1 > budget) {
            out_items.push_back(w);
            out_cost.push_back(cost[i]);
            continue;
        }
        budget -= tiles * chunks - 1;
        const int h = static_cast<int>(w.packed & 0xFFu);
        for (int t = 0; t < tiles; ++t) {
            SplitGroup& g = split->groups[split->n_groups++];
            g.b = w.b;
            g.slot0 = static_cast<int32_t>(split->n_slots);
            g.n = static_cast<int32_t>(chunks);
            g.packed = static_cast<uint32_t>(h) | (static_cast<uint32_t>(tile + t) << 8);
            for (int64_t c = 0; c < chunks; ++c) {
                const int64_t j0 = c * chunk, j1 = std::min(nkv, j0 + chunk);
                const int64_t k0 = j0 * kTileRows, k1 = std::min<int64_t>(w.kv_len, j1 * kTileRows);
                const int32_t slot = static_cast<int32_t>(split->n_slots++);
                if (split->slot_block0) split->slot_block0[slot] = static_cast<int32_t>(bs[w.b] + j0);
                out_items.push_back({-(slot + 1), static_cast<int32_t>(w.kv_start + k0), static_cast<int32_t>(k1 - k0),
                                     pack_item(h, tile + t, 0)});
                out_cost.push_back((j1 - j0) + 1);
            }
        }
    }
    gen.swap(out_items);
    cost.swap(out_cost);
}

}  // namespace

int64_t build_schedule(const int32_t* offsets, int B, int Lq, int H, int broadcast_q, int causal, int is_bwd,
                       int P, int policy, WorkItem* items, int32_t* cta_start, int64_t max_items,
                       SparseSpec* sparse, SplitSpec* split) {
    if (P <= 0 || P > kMaxCtas) return -1;
    if (sparse && causal) return -1;
    // Cluster Launch Control: the backward's cost-sorted list as one CTA's
    // slice (the kernel launches one CTA per entry).
    if (policy == kSchedClc && (!is_bwd || P != 1)) return -1;
    if (policy == kSchedQueue && !is_bwd) return -1;
    Scratch& sc = scratch();
    // Broadcast-Q backward without a selection or causal mask, per-head CTA
    // groups, the pages' zigzag: every item costs the same (its ceil(Lq/128)
    // query tiles + 1), so the cost-sorted order is the generation order and
    // the deal is a running zigzag per head.  One pass then places every item
    // straight into its CTA's slice of the list -- the schedule the general
    // path below builds with its separate sort, deal and placement passes.
    if (is_bwd && broadcast_q && !causal && !sparse && policy == kSchedLptZigzag &&
        head_partition(broadcast_q, H, P)) {
        const int G = P / H;
        int64_t per_head = 0;
        for (int b = 0; b < B; ++b) per_head += ceil_div(offsets[b + 1] - offsets[b], kTileRows);
        if (per_head * H > max_items) return -1;
        // Rounds of G items per head: every lane gets one item per full round;
        // the last, partial round covers lanes 0 .. rem-1 (even round) or
        // G-rem .. G-1 (odd round).
        const int64_t full = per_head / G, rem = per_head % G;
        cta_start[0] = 0;
        for (int c = 0; c < P; ++c) {
            const int lane = c / H;
            const bool extra = rem > 0 && ((full & 1) ? lane >= G - rem : lane < rem);
            cta_start[c + 1] = cta_start[c] + static_cast<int32_t>(full + (extra ? 1 : 0));
        }
        std::vector<int32_t>& fill = sc.fill;
        fill.assign(cta_start, cta_start + P);
        int lane_of[256] = {0};
        bool odd_of[256] = {false};
        for (int b = 0; b < B; ++b) {
            const int32_t Lk = offsets[b + 1] - offsets[b];
            const int64_t nkv = ceil_div(Lk, kTileRows);
            for (int h = 0; h < H; ++h)
                for (int64_t n = 0; n < nkv; ++n) {
                    const int lane = lane_of[h];
                    const int cta = (odd_of[h] ? G - 1 - lane : lane) * H + h;
                    items[fill[cta]++] = WorkItem{b, offsets[b], Lk, pack_item(h, static_cast<int>(n), 0)};
                    if (++lane_of[h] == G) {
                        lane_of[h] = 0;
                        odd_of[h] = !odd_of[h];
                    }
                }
        }
        if (split) split->n_groups = split->n_slots = 0;
        return per_head * H;
    }
    // 1. Generate items in (b, h, tile) order, with their costs.
    std::vector<WorkItem>& gen = sc.gen;
    std::vector<int64_t>& cost = sc.cost;
    gen.clear();
    cost.clear();
    int64_t bstart = 0;  // global index of the sequence's first key block
    if (sparse) sparse->n_blocks = sparse->n_zero = 0;
    for (int b = 0; b < B; ++b) {
        const int32_t Lk = offsets[b + 1] - offsets[b];
        const int64_t nkv = ceil_div(Lk, kTileRows);
        if (sparse && (bstart + nkv) * H > sparse->cap) return -1;
        if (!is_bwd) {
            const int64_t nq = broadcast_q ? ceil_div(Lq, kTileRows) : nkv;
            // broadcast rows exist even for an empty sequence (their O is 0, LSE -inf)
            for (int h = 0; h < H; ++h) {
                int64_t blocks = nkv;  // key blocks each query tile of the item visits (non-causal)
                if (sparse) {
                    SparseSel& sel = sparse->sel[static_cast<int64_t>(b) * H + h];
                    sel.off = static_cast<int32_t>(sparse->n_blocks);
                    sel.n_full = 0;
                    for (int64_t n = 0; n < nkv; ++n) {
                        if (!sparse->mask[(bstart + n) * H + h]) continue;
                        sparse->blocks[sparse->n_blocks++] = static_cast<int32_t>(n);
                        if (Lk - n * kTileRows >= kTileRows) ++sel.n_full;
                    }
                    sel.n_sel = static_cast<int32_t>(sparse->n_blocks - sel.off);
                    sel.pad = 0;
                    blocks = sel.n_sel;
                }
                for (int64_t m = 0; m < nq; m += 2) {
                    const WorkItem w{b, offsets[b], Lk, pack_item(h, static_cast<int>(m), m + 1 < nq ? 1 : 0)};
                    gen.push_back(w);
                    cost.push_back(sparse ? (m + 1 < nq ? 2 : 1) * blocks + 1
                                          : item_cost(w, Lq, broadcast_q, causal, is_bwd));
                }
            }
        } else {
            for (int h = 0; h < H; ++h)
                for (int64_t n = 0; n < nkv; ++n) {
                    if (sparse && !sparse->mask[(bstart + n) * H + h]) {
                        const int64_t row0 = offsets[b] + n * kTileRows;
                        sparse->zero[sparse->n_zero++] = {static_cast<int32_t>(row0),
                                                          static_cast<int32_t>(std::min<int64_t>(kTileRows, offsets[b + 1] - row0)),
                                                          h, 0};
                        continue;
                    }
                    const WorkItem w{b, offsets[b], Lk, pack_item(h, static_cast<int>(n), 0)};
                    gen.push_back(w);
                    cost.push_back(item_cost(w, Lq, broadcast_q, causal, is_bwd));
                }
        }
        bstart += nkv;
        if (static_cast<int64_t>(gen.size()) > max_items) return -1;
    }
    if (split) split->n_groups = split->n_slots = 0;
    if (split && !is_bwd && broadcast_q && !sparse && policy != kSchedNaive && !gen.empty())
        split_long_items(gen, cost, P, max_items, offsets, B, split);
    const int64_t n = static_cast<int64_t>(gen.size());

    // 2. Order: cost-descending, stable (counting sort on the integer cost).
    std::vector<int64_t>& order = sc.order;
    order.resize(static_cast<size_t>(n));
    if (policy != kSchedNaive && n > 0) {
        int64_t cmax = 0;
        for (int64_t i = 0; i < n; ++i) cmax = std::max(cmax, cost[i]);
        std::vector<int64_t>& start = sc.buckets;
        start.assign(static_cast<size_t>(cmax + 2), 0);
        for (int64_t i = 0; i < n; ++i) ++start[cmax - cost[i] + 1];  // bucket 0 = largest cost
        for (int64_t c = 1; c <= cmax + 1; ++c) start[c] += start[c - 1];
        for (int64_t i = 0; i < n; ++i) order[start[cmax - cost[i]]++] = i;
    } else {
        for (int64_t i = 0; i < n; ++i) order[i] = i;
    }

    // 3q. Queues: each item to its head group's queue, in the sorted order
    // (longest first); the CTAs of the group take them at run time.
    if (policy == kSchedQueue) {
        const int G = queue_groups(broadcast_q, H, P);
        std::fill(cta_start, cta_start + 2 * G + 1, 0);
        for (int64_t i = 0; i < n; ++i) ++cta_start[(G > 1 ? static_cast<int>(gen[order[i]].packed & 0xFFu) : 0) + 1];
        for (int g = 0; g < G; ++g) cta_start[g + 1] += cta_start[g];
        std::vector<int32_t>& fill = sc.fill;
        fill.assign(cta_start, cta_start + G);
        for (int64_t i = 0; i < n; ++i) {
            const WorkItem& w = gen[order[i]];
            items[fill[G > 1 ? static_cast<int>(w.packed & 0xFFu) : 0]++] = w;
        }
        return n;
    }

    // 3. Deal (see deal()).
    std::vector<int32_t>& owner = sc.owner;
    owner.resize(static_cast<size_t>(n));
    std::vector<int64_t>& heap = sc.heap;
    heap.resize(static_cast<size_t>(P));
    deal(gen.data(), order.data(), cost.data(), n, Lq, H, broadcast_q, causal, is_bwd, P, policy, owner.data(),
         heap.data());
    std::fill(cta_start, cta_start + P + 1, 0);
    for (int64_t i = 0; i < n; ++i) ++cta_start[owner[i] + 1];
    for (int p = 0; p < P; ++p) cta_start[p + 1] += cta_start[p];
    std::vector<int32_t>& fill = sc.fill;
    fill.assign(cta_start, cta_start + P);
    for (int64_t i = 0; i < n; ++i) items[fill[owner[i]]++] = gen[order[i]];
    // 4. Broadcast Q: group each CTA's items by the Q tiles they read.  Not
    // for Cluster Launch Control: a resident CTA's successive items lie about
    // one SM count apart in the list, so grouping shares no Q tile; it would
    // only make the CTAs that run together all add into one head's dQ.
    if (broadcast_q && policy != kSchedNaive && policy != kSchedClc) group_by_q(items, cta_start, P, is_bwd);
    return n;
}

int64_t build_schedule_noalloc(const int32_t* offsets, int B, int Lq, int H, int broadcast_q, int causal, int is_bwd,
                               int P, WorkItem* items, int32_t* cta_start, int64_t max_items, WorkItem* gen,
                               int64_t* order, int32_t* owner, int32_t* fill, int64_t* buckets) {
    if (P <= 0 || P > kMaxCtas) return -1;
    int64_t n = 0;
    for (int b = 0; b < B; ++b) {
        const int32_t Lk = offsets[b + 1] - offsets[b];
        const int64_t nkv = ceil_div(Lk, kTileRows);
        const int64_t ntiles = is_bwd ? nkv : (broadcast_q ? ceil_div(Lq, kTileRows) : nkv);
        const int64_t step = is_bwd ? 1 : 2;
        for (int h = 0; h < H; ++h)
            for (int64_t m = 0; m < ntiles; m += step) {
                if (n >= max_items) return -1;
                const int two = (!is_bwd && m + 1 < ntiles) ? 1 : 0;
                gen[n++] = {b, offsets[b], Lk, pack_item(h, static_cast<int>(m), two)};
            }
    }
    // Stable counting sort, largest cost first (bucket 0).
    for (int64_t c = 0; c < kCostBuckets + 2; ++c) buckets[c] = 0;
    for (int64_t i = 0; i < n; ++i) {
        const int64_t cost = std::min<int64_t>(item_cost(gen[i], Lq, broadcast_q, causal, is_bwd), kCostBuckets - 1);
        ++buckets[(kCostBuckets - 1 - cost) + 1];
    }
    for (int64_t c = 1; c < kCostBuckets + 2; ++c) buckets[c] += buckets[c - 1];
    for (int64_t i = 0; i < n; ++i) {
        const int64_t cost = std::min<int64_t>(item_cost(gen[i], Lq, broadcast_q, causal, is_bwd), kCostBuckets - 1);
        order[buckets[kCostBuckets - 1 - cost]++] = i;
    }
    // Greedy deal (the sort's buckets now serve as the heaps), then CSR
    // placement in deal order.
    deal(gen, order, nullptr, n, Lq, H, broadcast_q, causal, is_bwd, P, kSchedLptGreedy, owner, buckets);
    for (int p = 0; p <= P; ++p) cta_start[p] = 0;
    for (int64_t i = 0; i < n; ++i) ++cta_start[owner[i] + 1];
    for (int p = 0; p < P; ++p) cta_start[p + 1] += cta_start[p];
    for (int p = 0; p < P; ++p) fill[p] = cta_start[p];
    for (int64_t i = 0; i < n; ++i) items[fill[owner[i]]++] = gen[order[i]];
    if (broadcast_q) group_by_q(items, cta_start, P, is_bwd);
    return n;
}

}  // namespace jfa

// Host-only C entries used by the scheduler's unit tests (no GPU needed).
extern "C" long long jfa_host_build_schedule_noalloc(const int32_t* offsets, int B, int Lq, int H, int broadcast_q,
                                                     int causal, int is_bwd, int P, void* items, int32_t* cta_start,
                                                     long long max_items) {
    const size_t cap = static_cast<size_t>(max_items > 0 ? max_items : 1);
    std::vector<jfa::WorkItem> gen(cap);
    std::vector<int64_t> order(cap), buckets(static_cast<size_t>(jfa::kCostBuckets + 2));
    std::vector<int32_t> owner(cap), fill(static_cast<size_t>(P > 0 ? P : 1));
    return jfa::build_schedule_noalloc(offsets, B, Lq, H, broadcast_q, causal, is_bwd, P,
                                       static_cast<jfa::WorkItem*>(items), cta_start, max_items, gen.data(),
                                       order.data(), owner.data(), fill.data(), buckets.data());
}

extern "C" long long jfa_host_build_schedule(const int32_t* offsets, int B, int Lq, int H, int broadcast_q,
                                             int causal, int is_bwd, int P, int policy, void* items,
                                             int32_t* cta_start, long long max_items) {
    return jfa::build_schedule(offsets, B, Lq, H, broadcast_q, causal, is_bwd, P, policy,
                               static_cast<jfa::WorkItem*>(items), cta_start, max_items);
}

// Block-sparse schedule (library policy: greedy forward, zigzag backward) with
// its selection tables; counts[0] = selected-block entries, counts[1] =
// unselected backward tiles.  Returns the item count or -1.
extern "C" long long jfa_host_build_schedule_sparse(const int32_t* offsets, int B, int Lq, int H, int broadcast_q,
                                                    int is_bwd, int P, const uint8_t* mask, void* items,
                                                    int32_t* cta_start, long long max_items, void* sel,
                                                    int32_t* blocks, void* zero, long long cap, long long* counts) {
    jfa::SparseSpec sp;
    sp.mask = mask;
    sp.sel = static_cast<jfa::SparseSel*>(sel);
    sp.blocks = blocks;
    sp.zero = static_cast<jfa::ZeroTile*>(zero);
    sp.cap = cap;
    const long long n = jfa::build_schedule(offsets, B, Lq, H, broadcast_q, 0, is_bwd, P,
                                            is_bwd ? jfa::kSchedLptZigzag : jfa::kSchedLptGreedy,
                                            static_cast<jfa::WorkItem*>(items), cta_start, max_items, &sp);
    counts[0] = sp.n_blocks;
    counts[1] = sp.n_zero;
    return n;
}

// Broadcast-Q forward schedule with split-KV (the library's greedy deal);
// counts[0] = split groups, counts[1] = partial slots.  Returns the item
// count or -1.
extern "C" long long jfa_host_build_schedule_split(const int32_t* offsets, int B, int Lq, int H, int P, void* items,
                                                   int32_t* cta_start, long long max_items, void* groups,
                                                   long long* counts, int32_t* slot_block0) {
    jfa::SplitSpec sp;
    sp.groups = static_cast<jfa::SplitGroup*>(groups);
    sp.slot_block0 = slot_block0;  // may be null
    const long long n = jfa::build_schedule(offsets, B, Lq, H, 1, 0, 0, P, jfa::kSchedLptGreedy,
                                            static_cast<jfa::WorkItem*>(items), cta_start, max_items, nullptr, &sp);
    counts[0] = sp.n_groups;
    counts[1] = sp.n_slots;
    return n;
}
