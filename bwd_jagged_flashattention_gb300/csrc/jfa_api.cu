// jfa_api.cu -- the C ABI declared in include/jfa.h: argument checks, the
// host schedule (staged through a small pinned ring), TMA tensor maps and
// the kernel launches.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstring>
#include <functional>
#include <mutex>
#include <vector>

#include "../../include/jfa.h"
#include "host_util.h"
#include "kernels.h"
#include "scheduler.h"

namespace jfa {
namespace {

constexpr size_t kStatusBytes = 256;

constexpr size_t kCtaStartBytes = 4096;  // (kMaxCtas + 1) int32, rounded up

// Split-KV of long broadcast-Q forward items (scheduler.h); 0 turns it off
// (for measuring what it gains).
#ifndef JFA_FWD_SPLIT_KV
#define JFA_FWD_SPLIT_KV 1
#endif

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Deal policies of the two passes' schedules (jfa_set_schedule_policy).
std::atomic<int> g_fwd_policy{kSchedLptGreedy}, g_bwd_policy{kSchedLptZigzag};

// A schedule region holds the CTA bounds and the items, then (block-sparse
// calls only) the selection tables: forward, one SparseSel per (b, h) and the
// selected block indices; backward, the unselected tiles (ZeroTile).
struct WsLayout {
    size_t fwd_off, bwd_off, fwd_region, bwd_region, delta_off, delta_bytes, total;
    size_t sel_off, blocks_off, zero_off;  // offsets inside a region
    size_t split_off;                      // forward region: split-KV groups (broadcast Q)
    size_t split_blk_off;                  // forward region: each split slot's first key block (MXFP8 V scales)
    size_t opart_off, lpart_off;           // split-KV partial O / LSE (broadcast Q; 0 bytes otherwise)
    int64_t max_items, sel_cap;            // sel_cap >= NB * H (NB = key blocks over all sequences)
};

bool ws_layout(int B, int64_t N, int Lq, int H, int D, int broadcast_q, WsLayout* w) {
    if (B < 0 || N < 0 || H <= 0) return false;
    w->max_items = max_work_items(B, N, Lq, H, broadcast_q);
    w->sel_cap = (N / kTileRows + B) * H + 1;  // (+1: also holds block_start[0..B] of the MXFP8 calls)
    w->sel_off = align_up(kCtaStartBytes + static_cast<size_t>(w->max_items) * sizeof(WorkItem), 256);
    w->blocks_off = w->sel_off + align_up(static_cast<size_t>(B) * H * sizeof(SparseSel), 256);
    w->zero_off = w->sel_off;
    w->split_off = w->blocks_off + align_up(static_cast<size_t>(w->sel_cap) * sizeof(int32_t), 256);
    w->split_blk_off = w->split_off + (broadcast_q ? align_up(kMaxSplitSlots * sizeof(SplitGroup), 256) : 0);
    w->fwd_region = w->split_blk_off + (broadcast_q ? align_up(kMaxSplitSlots * sizeof(int32_t), 256) : 0);
    w->bwd_region = w->zero_off + align_up(static_cast<size_t>(w->sel_cap) * sizeof(ZeroTile), 256);
    w->fwd_off = kStatusBytes;
    w->bwd_off = w->fwd_off + w->fwd_region;
    w->delta_off = w->bwd_off + w->bwd_region;
    const int64_t stat_elems = broadcast_q ? static_cast<int64_t>(B) * H * Lq : static_cast<int64_t>(H) * N;
    w->delta_bytes = align_up(static_cast<size_t>(stat_elems) * sizeof(float), 256);
    w->opart_off = w->delta_off + w->delta_bytes;
    w->lpart_off = w->opart_off + (broadcast_q ? align_up(static_cast<size_t>(kMaxSplitSlots) * 128 * D * 4, 256) : 0);
    w->total = w->lpart_off + (broadcast_q ? align_up(static_cast<size_t>(kMaxSplitSlots) * 128 * 4, 256) : 0);
    return true;
}

// ---------------------------------------------------------------------------
// Pinned staging ring for schedules: a slot is reused only after the copy
// that last read it has executed (its event has completed).
// ---------------------------------------------------------------------------
struct StageSlot {
    void* buf = nullptr;
    size_t cap = 0;
    cudaEvent_t ev = nullptr;
    bool used = false;
};

struct DeviceStage {
    std::mutex mu;
    StageSlot slots[4];
    unsigned next = 0;
};

DeviceStage& device_stage(int dev) {
    static DeviceStage stages[64];
    return stages[dev & 63];
}

// Runs fill(buf) on a pinned slot of at least `need` bytes; fill writes the
// slot and enqueues the copies that read it on `stream`.  The slot's event is
// recorded after them, so the slot is reused only once they have executed.
template <typename F>
jfa_status with_stage(size_t need, cudaStream_t stream, F&& fill) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return JFA_ERR_CUDA;
    DeviceStage& ds = device_stage(dev);
    std::lock_guard<std::mutex> lock(ds.mu);
    StageSlot& slot = ds.slots[ds.next++ % 4];
    if (slot.used && cudaEventSynchronize(slot.ev) != cudaSuccess) return JFA_ERR_CUDA;
    if (slot.cap < need) {
        if (slot.buf) cudaFreeHost(slot.buf);
        slot.buf = nullptr;
        slot.cap = 0;
        if (cudaHostAlloc(&slot.buf, need, cudaHostAllocDefault) != cudaSuccess) return JFA_ERR_CUDA;
        slot.cap = need;
    }
    if (!slot.ev && cudaEventCreateWithFlags(&slot.ev, cudaEventDisableTiming) != cudaSuccess) return JFA_ERR_CUDA;
    const jfa_status st = fill(static_cast<char*>(slot.buf));
    if (st != JFA_OK) return st;
    if (cudaEventRecord(slot.ev, stream) != cudaSuccess) return JFA_ERR_CUDA;
    slot.used = true;
    return JFA_OK;
}

// Hands a staged schedule (its device-mapped pinned source and byte count) to
// a kernel launched from inside the staging call, which either moves it into
// the workspace region (the backward's Delta pass) or reads it where it is
// (the forward kernel).
using ScheduleUpload = std::function<cudaError_t(const void* src_dev, size_t bytes)>;

// Builds the schedule into a pinned slot laid out like the workspace region
// (WsLayout) and enqueues its copy into ws_region -- or, given `upload` and a
// non-empty schedule of CTA bounds and items alone, calls upload instead (the
// slot is then read by upload's kernel, which its reuse event follows).  With a block
// mask (block-sparse) the selection tables follow; *n_zero receives the number
// of unselected backward tiles.  Returns the item count (>= 0) or -1 on error.
int64_t stage_schedule(const int32_t* offsets, int B, int Lq, int H, int broadcast_q, int causal, int is_bwd, int P,
                       int policy, const WsLayout& w, const uint8_t* mask, void* ws_region, cudaStream_t stream,
                       int64_t* n_zero, int64_t* n_split_groups, jfa_status* st,
                       const ScheduleUpload* upload = nullptr) {
    const int64_t max_items = w.max_items;
    const bool may_split = JFA_FWD_SPLIT_KV && !is_bwd && !mask && broadcast_q && n_split_groups;
    const size_t need = (mask || may_split) ? (is_bwd ? w.bwd_region : w.fwd_region)
                                            : kCtaStartBytes + static_cast<size_t>(max_items) * sizeof(WorkItem);
    int64_t n = -1;
    SparseSpec sp;
    SplitSpec split;
    *st = with_stage(need, stream, [&](char* buf) -> jfa_status {
        int32_t* cta_start = reinterpret_cast<int32_t*>(buf);
        WorkItem* items = reinterpret_cast<WorkItem*>(buf + kCtaStartBytes);
        if (mask) {
            sp.mask = mask;
            sp.sel = reinterpret_cast<SparseSel*>(buf + w.sel_off);
            sp.blocks = reinterpret_cast<int32_t*>(buf + w.blocks_off);
            sp.zero = reinterpret_cast<ZeroTile*>(buf + w.zero_off);
            sp.cap = w.sel_cap;
        }
        split.groups = reinterpret_cast<SplitGroup*>(buf + w.split_off);
        split.slot_block0 = reinterpret_cast<int32_t*>(buf + w.split_blk_off);
        n = build_schedule(offsets, B, Lq, H, broadcast_q, causal, is_bwd, P, policy,
                           items, cta_start, max_items, mask ? &sp : nullptr, may_split ? &split : nullptr);
        if (n < 0) return JFA_ERR_WORKSPACE;
        char* dst = static_cast<char*>(ws_region);
        const size_t bytes = kCtaStartBytes + static_cast<size_t>(n) * sizeof(WorkItem);
        void* src_dev = nullptr;
        // (only for the CTA bounds and items alone: with selection or split
        // tables after them, everything is copied)
        const bool extras = mask || (may_split && split.n_groups > 0);
        if (upload && n > 0 && !extras && cudaHostGetDevicePointer(&src_dev, buf, 0) != cudaSuccess) {
            cudaGetLastError();  // not mapped: clear the error and copy instead
            src_dev = nullptr;
        }
        bool ok = src_dev ? (*upload)(src_dev, bytes) == cudaSuccess
                          : cudaMemcpyAsync(dst, buf, bytes, cudaMemcpyHostToDevice, stream) == cudaSuccess;
        if (mask && !is_bwd) {
            ok = ok && cudaMemcpyAsync(dst + w.sel_off, buf + w.sel_off, static_cast<size_t>(B) * H * sizeof(SparseSel),
                                       cudaMemcpyHostToDevice, stream) == cudaSuccess;
            ok = ok && (sp.n_blocks == 0 ||
                        cudaMemcpyAsync(dst + w.blocks_off, buf + w.blocks_off, sp.n_blocks * sizeof(int32_t),
                                        cudaMemcpyHostToDevice, stream) == cudaSuccess);
        }
        if (mask && is_bwd)
            ok = ok && (sp.n_zero == 0 ||
                        cudaMemcpyAsync(dst + w.zero_off, buf + w.zero_off, sp.n_zero * sizeof(ZeroTile),
                                        cudaMemcpyHostToDevice, stream) == cudaSuccess);
        if (may_split) {
            ok = ok && (split.n_groups == 0 ||
                        cudaMemcpyAsync(dst + w.split_off, buf + w.split_off, split.n_groups * sizeof(SplitGroup),
                                        cudaMemcpyHostToDevice, stream) == cudaSuccess);
            ok = ok && (split.n_slots == 0 ||
                        cudaMemcpyAsync(dst + w.split_blk_off, buf + w.split_blk_off, split.n_slots * sizeof(int32_t),
                                        cudaMemcpyHostToDevice, stream) == cudaSuccess);
        }
        return ok ? JFA_OK : JFA_ERR_CUDA;
    });
    if (*st != JFA_OK) return -1;
    if (n_zero) *n_zero = mask ? sp.n_zero : 0;
    if (n_split_groups) *n_split_groups = may_split ? split.n_groups : 0;
    return n;
}

// First 128-key block of every sequence (block_start[b], b = 0..B; the last
// entry is the total NB) into dst (device, B + 1 int32).  Returns NB in *nb.
jfa_status stage_block_starts(const int32_t* offsets, int B, void* dst, cudaStream_t stream, int64_t* nb) {
    return with_stage(sizeof(int32_t) * (static_cast<size_t>(B) + 1), stream, [&](char* buf) -> jfa_status {
        int32_t* bs = reinterpret_cast<int32_t*>(buf);
        int64_t acc = 0;
        for (int b = 0; b < B; ++b) {
            bs[b] = static_cast<int32_t>(acc);
            acc += (static_cast<int64_t>(offsets[b + 1]) - offsets[b] + 127) / 128;
        }
        bs[B] = static_cast<int32_t>(acc);
        *nb = acc;
        return cudaMemcpyAsync(dst, buf, sizeof(int32_t) * (static_cast<size_t>(B) + 1), cudaMemcpyHostToDevice,
                               stream) == cudaSuccess
                   ? JFA_OK
                   : JFA_ERR_CUDA;
    });
}

// ---------------------------------------------------------------------------
// Argument checks shared by both passes.
// ---------------------------------------------------------------------------
inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

struct Problem {
    int B, Lq, H, D, broadcast_q, causal;
    int64_t N;
    float scale;
    std::vector<int32_t> off_copy;
    const int32_t* off;
};

jfa_status check_common(int B, int Lq, int H, int D, int broadcast_q, int causal, float scale,
                        const int32_t* offsets_dev, const int32_t* offsets_host, cudaStream_t stream, Problem* pr) {
    if (B < 0 || H <= 0 || Lq < 0) return JFA_ERR_INVALID_ARG;
    if (!std::isfinite(scale)) return JFA_ERR_INVALID_ARG;
    if (D != 64 && D != 128) return JFA_ERR_UNSUPPORTED;
    if (H > 255) return JFA_ERR_UNSUPPORTED;
    if (broadcast_q && causal) return JFA_ERR_UNSUPPORTED;
    if (broadcast_q && Lq > kMaxSeqLen) return JFA_ERR_UNSUPPORTED;
    if (!offsets_host && !offsets_dev) return JFA_ERR_INVALID_ARG;
    pr->B = B;
    pr->Lq = broadcast_q ? Lq : 0;
    pr->H = H;
    pr->D = D;
    pr->broadcast_q = broadcast_q ? 1 : 0;
    pr->causal = causal ? 1 : 0;
    pr->scale = scale > 0.0f ? scale : 1.0f / std::sqrt(static_cast<float>(D));
    if (offsets_host) {
        pr->off = offsets_host;
    } else {
        pr->off_copy.resize(static_cast<size_t>(B) + 1);
        if (cudaMemcpyAsync(pr->off_copy.data(), offsets_dev, sizeof(int32_t) * (static_cast<size_t>(B) + 1),
                            cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
            cudaStreamSynchronize(stream) != cudaSuccess)
            return JFA_ERR_CUDA;
        pr->off = pr->off_copy.data();
    }
    if (pr->off[0] != 0) return JFA_ERR_INVALID_ARG;
    for (int b = 0; b < B; ++b) {
        const int64_t len = static_cast<int64_t>(pr->off[b + 1]) - pr->off[b];
        if (len < 0) return JFA_ERR_INVALID_ARG;
        if (len > kMaxSeqLen) return JFA_ERR_UNSUPPORTED;
    }
    pr->N = pr->off[B];
    return JFA_OK;
}

jfa_status check_workspace(const Problem& pr, void* workspace, size_t ws_bytes, WsLayout* w) {
    if (!ws_layout(pr.B, pr.N, pr.Lq, pr.H, pr.D, pr.broadcast_q, w)) return JFA_ERR_INVALID_ARG;
    if (!workspace || !aligned(workspace, 256) || ws_bytes < w->total) return JFA_ERR_WORKSPACE;
    return JFA_OK;
}

// A 2D [rows, H*D] view with 64x128 bf16 boxes and 128-byte swizzle.
bool map_rows_bf16(CUtensorMap* m, const void* base, int64_t rows, int H, int D, const void* fallback) {
    const uint64_t dims[2] = {static_cast<uint64_t>(H) * D, static_cast<uint64_t>(rows > 0 ? rows : 1)};
    const uint64_t strides[1] = {static_cast<uint64_t>(H) * D * 2};
    const uint32_t box[2] = {64, 128};
    return encode_tensor_map(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, rows > 0 ? base : fallback, dims, strides, box,
                             CU_TENSOR_MAP_SWIZZLE_128B);
}

// A 2D [rows, H*D] E4M3 (byte) view with D x 128 boxes: one box is a whole
// 128-row tile of one head (128-byte swizzle at D=128, 64-byte at D=64).
bool map_rows_e4m3(CUtensorMap* m, const void* base, int64_t rows, int H, int D, const void* fallback) {
    const uint64_t dims[2] = {static_cast<uint64_t>(H) * D, static_cast<uint64_t>(rows > 0 ? rows : 1)};
    const uint64_t strides[1] = {static_cast<uint64_t>(H) * D};
    const uint32_t box[2] = {static_cast<uint32_t>(D), 128};
    return encode_tensor_map(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, rows > 0 ? base : fallback, dims, strides, box,
                             D == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B);
}

// A 2D [rows, H*D] fp32 view with 16x128 boxes and 64-byte swizzle (dQ reduce-add).
bool map_rows_f32(CUtensorMap* m, const void* base, int64_t rows, int H, int D, const void* fallback) {
    const uint64_t dims[2] = {static_cast<uint64_t>(H) * D, static_cast<uint64_t>(rows > 0 ? rows : 1)};
    const uint64_t strides[1] = {static_cast<uint64_t>(H) * D * 4};
    const uint32_t box[2] = {16, 128};
    return encode_tensor_map(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, rows > 0 ? base : fallback, dims, strides, box,
                             CU_TENSOR_MAP_SWIZZLE_64B);
}

int ctas_for(int64_t items) {
    const int sms = device_sm_count();
    int p = sms > 0 ? sms : 1;
    if (p > kMaxCtas) p = kMaxCtas;
    if (items < p) p = static_cast<int>(items > 0 ? items : 1);
    return p;
}

int64_t count_items(const Problem& pr, int is_bwd) {
    int64_t n = 0;
    for (int b = 0; b < pr.B; ++b) {
        const int64_t Lk = static_cast<int64_t>(pr.off[b + 1]) - pr.off[b];
        const int64_t nkv = (Lk + 127) / 128;
        if (is_bwd)
            n += nkv;
        else
            n += ((pr.broadcast_q ? (pr.Lq + 127) / 128 : nkv) + 1) / 2;
    }
    return n * pr.H;
}

// ---------------------------------------------------------------------------
// Optional per-kernel event timing (jfa_profile_enable / jfa_profile_read).
// ---------------------------------------------------------------------------
enum ProfKind { kProfFwd = 0, kProfPre = 1, kProfBwd = 2, kProfZero = 3, kProfMerge = 4, kProfQuant = 5,
                kProfKinds = 6 };

struct Profiler {
    std::mutex mu;
    bool on = false;
    std::vector<cudaEvent_t> pool;
    std::vector<std::pair<int, std::pair<cudaEvent_t, cudaEvent_t>>> pending;
};

Profiler& profiler() {
    static Profiler p;
    return p;
}

cudaEvent_t prof_event(Profiler& p) {
    if (!p.pool.empty()) {
        cudaEvent_t e = p.pool.back();
        p.pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    cudaEventCreate(&e);
    return e;
}

// Runs `launch` between two recorded events when profiling is on.
template <typename F>
cudaError_t timed_launch(int kind, cudaStream_t s, F&& launch) {
    Profiler& p = profiler();
    cudaEvent_t a = nullptr, b = nullptr;
    {
        std::lock_guard<std::mutex> lock(p.mu);
        if (p.on) {
            a = prof_event(p);
            b = prof_event(p);
        }
    }
    if (a) cudaEventRecord(a, s);
    cudaError_t e = launch();
    if (b) {
        cudaEventRecord(b, s);
        std::lock_guard<std::mutex> lock(p.mu);
        p.pending.push_back({kind, {a, b}});
    }
    return e;
}

}  // namespace
}  // namespace jfa

using namespace jfa;

extern "C" size_t jfa_workspace_bytes(int B, int total_len, int Lq, int H, int D, int broadcast_q, int causal) {
    (void)causal;
    if (D != 64 && D != 128) return 0;
    WsLayout w;
    if (!ws_layout(B, total_len, broadcast_q ? Lq : 0, H, D, broadcast_q, &w)) return 0;
    return w.total;
}

extern "C" int jfa_num_ctas(void) { return ctas_for(1 << 30); }

extern "C" jfa_status jfa_set_wait_limit(unsigned long long ns) {
    set_wait_limit_ns(ns ? static_cast<uint64_t>(ns) : 4000000000ull);
    return JFA_OK;
}

extern "C" jfa_status jfa_set_schedule_policy(int fwd_policy, int bwd_policy) {
    auto ok = [](int v) { return v == kSchedLptZigzag || v == kSchedNaive || v == kSchedLptGreedy; };
    if (!ok(fwd_policy) || !(ok(bwd_policy) || bwd_policy == kSchedClc || bwd_policy == kSchedQueue))
        return JFA_ERR_INVALID_ARG;
    g_fwd_policy.store(fwd_policy);
    g_bwd_policy.store(bwd_policy);
    return JFA_OK;
}

// Forward for jfa_fwd (mask == NULL, v_scale == NULL), jfa_fwd_block_sparse
// (mask) and jfa_fwd_mxfp8 (v_scale: v holds E4M3 codes).
static jfa_status fwd_impl(const void* q, const void* k, const void* v, const int32_t* offsets_dev,
                           const int32_t* offsets_host, const uint8_t* mask, bool mx, const void* v_scale, int B,
                           int Lq, int H, int D, int broadcast_q, int causal, float scale, void* o, float* lse,
                           void* workspace, size_t workspace_bytes, void* stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    Problem pr;
    jfa_status st = check_common(B, Lq, H, D, broadcast_q, causal, scale, offsets_dev, offsets_host, s, &pr);
    if (st != JFA_OK) return st;
    WsLayout w;
    if ((st = check_workspace(pr, workspace, workspace_bytes, &w)) != JFA_OK) return st;
    const int64_t q_rows = pr.broadcast_q ? pr.Lq : pr.N;
    const int64_t o_rows = pr.broadcast_q ? static_cast<int64_t>(pr.B) * pr.Lq : pr.N;
    if ((q_rows > 0 && !q) || (pr.N > 0 && (!k || !v || (mx && !v_scale))) || (o_rows > 0 && (!o || !lse)))
        return JFA_ERR_INVALID_ARG;
    if (pr.N == 0) v_scale = nullptr;  // no key: nothing is quantized (the bf16 kernel writes the empty rows)
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(lse, 4) ||
        !aligned(v_scale, 16))
        return JFA_ERR_UNSUPPORTED;
    if (o_rows == 0) return JFA_OK;  // nothing to compute

    char* ws = static_cast<char*>(workspace);
    // Broadcast Q (split-KV possible): every SM, since splitting can make
    // more items than the batch has; CTAs left without items exit at once.
    // (An MXFP8 chunk finds its V scales through its slot's first block.)
    const bool may_split = pr.broadcast_q && !mask;
    const int64_t n_items = may_split ? (int64_t{1} << 30) : count_items(pr, 0);
    const int P = ctas_for(n_items);
    FwdMaps maps;
    FwdParams p;
    auto build = [&]() -> bool {
        const bool v_ok = v_scale ? map_rows_e4m3(&maps.v, v, pr.N, H, D, workspace)
                                  : map_rows_bf16(&maps.v, v, pr.N, H, D, workspace);
        if (!map_rows_bf16(&maps.q, q, q_rows, H, D, workspace) || !map_rows_bf16(&maps.k, k, pr.N, H, D, workspace) ||
            !v_ok || !map_rows_bf16(&maps.o, o, o_rows, H, D, workspace))
            return false;
        p.cta_start = reinterpret_cast<const int32_t*>(ws + w.fwd_off);
        p.items = reinterpret_cast<const WorkItem*>(ws + w.fwd_off + kCtaStartBytes);
        p.o = static_cast<uint16_t*>(o);
        p.lse = lse;
        p.status = reinterpret_cast<uint32_t*>(ws);
        p.Lq = pr.Lq;
        p.H = H;
        p.N = static_cast<int>(pr.N);
        p.broadcast_q = pr.broadcast_q;
        p.causal = pr.causal;
        p.scale_log2 = pr.scale * 1.4426950408889634f;
        p.wait_ns = wait_limit_ns();
        p.sel = mask ? reinterpret_cast<const SparseSel*>(ws + w.fwd_off + w.sel_off) : nullptr;
        p.sel_blocks = mask ? reinterpret_cast<const int32_t*>(ws + w.fwd_off + w.blocks_off) : nullptr;
        if (v_scale) {
            p.v_scale = static_cast<const uint32_t*>(v_scale);
            p.block_start = reinterpret_cast<const int32_t*>(ws + w.fwd_off + w.blocks_off);
        }
        return true;
    };
    // Plain forward (no block-sparse lists, no MXFP8 block table): the kernel
    // reads its CTA bounds and work items straight from the pinned staging
    // slot (through the slot's device mapping; every role reads items one
    // iteration ahead) and is launched from inside the staging call, so the
    // slot's reuse event follows it: no host-to-device copy in the stream.
    // With split-KV tables after the items, they are all copied as before.
    const bool direct = !mask && !v_scale && pr.N > 0;
    if (direct && !build()) return JFA_ERR_CUDA;
    bool launched = false;
    const ScheduleUpload upload = [&](const void* src_dev, size_t) {
        p.cta_start = static_cast<const int32_t*>(src_dev);
        p.items = reinterpret_cast<const WorkItem*>(static_cast<const char*>(src_dev) + kCtaStartBytes);
        launched = true;
        return timed_launch(kProfFwd, s, [&] { return launch_fwd(D, p, maps, P, s); });
    };
    int64_t n_groups = 0;
    const int64_t n = stage_schedule(pr.off, pr.B, pr.Lq, pr.H, pr.broadcast_q, pr.causal, 0, P, g_fwd_policy.load(),
                                     w, mask, ws + w.fwd_off, s, nullptr, may_split ? &n_groups : nullptr, &st,
                                     direct ? &upload : nullptr);
    if (n < 0) return st;
    if (n == 0) return JFA_OK;
    int64_t n_blocks = 0;
    if (v_scale && (st = stage_block_starts(pr.off, pr.B, ws + w.fwd_off + w.blocks_off, s, &n_blocks)) != JFA_OK)
        return st;
    if (!direct && !build()) return JFA_ERR_CUDA;
    if (n_groups > 0) {  // split-KV chunks write partials; the merge pass writes their O / LSE
        p.o_part = reinterpret_cast<float*>(ws + w.opart_off);
        p.lse_part = reinterpret_cast<float*>(ws + w.lpart_off);
        p.split_block0 = reinterpret_cast<const int32_t*>(ws + w.fwd_off + w.split_blk_off);
    }
    if (!launched && timed_launch(kProfFwd, s, [&] { return launch_fwd(D, p, maps, P, s); }) != cudaSuccess)
        return JFA_ERR_CUDA;
    if (n_groups > 0 && timed_launch(kProfMerge, s, [&] {
                            return launch_fwd_merge(D, reinterpret_cast<const SplitGroup*>(ws + w.fwd_off + w.split_off),
                                                    n_groups, p.o_part, p.lse_part, static_cast<uint16_t*>(o), lse,
                                                    pr.Lq, H, s);
                        }) != cudaSuccess)
        return JFA_ERR_CUDA;
    return JFA_OK;
}

extern "C" jfa_status jfa_fwd(const void* q, const void* k, const void* v, const int32_t* offsets_dev,
                              const int32_t* offsets_host, int B, int Lq, int H, int D, int broadcast_q, int causal,
                              float scale, void* o, float* lse, void* workspace, size_t workspace_bytes,
                              void* stream) {
    return fwd_impl(q, k, v, offsets_dev, offsets_host, nullptr, false, nullptr, B, Lq, H, D, broadcast_q, causal,
                    scale, o, lse, workspace, workspace_bytes, stream);
}

extern "C" jfa_status jfa_fwd_block_sparse(const void* q, const void* k, const void* v, const int32_t* offsets_dev,
                                           const int32_t* offsets_host, const uint8_t* kv_block_mask, int B, int Lq,
                                           int H, int D, int broadcast_q, float scale, void* o, float* lse,
                                           void* workspace, size_t workspace_bytes, void* stream) {
    if (!kv_block_mask) return JFA_ERR_INVALID_ARG;
    return fwd_impl(q, k, v, offsets_dev, offsets_host, kv_block_mask, false, nullptr, B, Lq, H, D, broadcast_q, 0,
                    scale, o, lse, workspace, workspace_bytes, stream);
}

extern "C" jfa_status jfa_fwd_mxfp8(const void* q, const void* k, const void* v8, const void* v_scale,
                                    const int32_t* offsets_dev, const int32_t* offsets_host, int B, int Lq, int H,
                                    int D, int broadcast_q, int causal, float scale, void* o, float* lse,
                                    void* workspace, size_t workspace_bytes, void* stream) {
    return fwd_impl(q, k, v8, offsets_dev, offsets_host, nullptr, true, v_scale, B, Lq, H, D, broadcast_q, causal,
                    scale, o, lse, workspace, workspace_bytes, stream);
}

extern "C" jfa_status jfa_quantize_v_mxfp8(const void* v, const int32_t* offsets_dev, const int32_t* offsets_host,
                                           int B, int H, int D, void* v8, void* v_scale, void* workspace,
                                           size_t workspace_bytes, void* stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    Problem pr;
    jfa_status st = check_common(B, 0, H, D, 0, 0, 1.0f, offsets_dev, offsets_host, s, &pr);
    if (st != JFA_OK) return st;
    if (!offsets_dev) return JFA_ERR_INVALID_ARG;
    const size_t need = kStatusBytes + sizeof(int32_t) * (static_cast<size_t>(B) + 1);
    if (!workspace || !aligned(workspace, 256) || workspace_bytes < need) return JFA_ERR_WORKSPACE;
    if (pr.N > 0 && (!v || !v8 || !v_scale)) return JFA_ERR_INVALID_ARG;
    if (!aligned(v, 16) || !aligned(v8, 16) || !aligned(v_scale, 16)) return JFA_ERR_UNSUPPORTED;
    if (pr.N == 0) return JFA_OK;
    int32_t* bs = reinterpret_cast<int32_t*>(static_cast<char*>(workspace) + kStatusBytes);
    int64_t n_blocks = 0;
    if ((st = stage_block_starts(pr.off, pr.B, bs, s, &n_blocks)) != JFA_OK) return st;
    if (timed_launch(kProfQuant, s, [&] {
            return launch_quant_v_mxfp8(static_cast<const uint16_t*>(v), offsets_dev, bs, pr.B, n_blocks, H, D,
                                        static_cast<uint8_t*>(v8), static_cast<uint32_t*>(v_scale), s);
        }) != cudaSuccess)
        return JFA_ERR_CUDA;
    return JFA_OK;
}

// Backward for jfa_bwd (mask == NULL) and jfa_bwd_block_sparse.
static jfa_status bwd_impl(const void* q, const void* k, const void* v, const void* o, const float* lse,
                           const void* dout, const int32_t* offsets_dev, const int32_t* offsets_host,
                           const uint8_t* mask, int B, int Lq, int H, int D, int broadcast_q, int causal, float scale,
                           float* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes, void* stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    Problem pr;
    jfa_status st = check_common(B, Lq, H, D, broadcast_q, causal, scale, offsets_dev, offsets_host, s, &pr);
    if (st != JFA_OK) return st;
    WsLayout w;
    if ((st = check_workspace(pr, workspace, workspace_bytes, &w)) != JFA_OK) return st;
    const int64_t q_rows = pr.broadcast_q ? pr.Lq : pr.N;
    const int64_t o_rows = pr.broadcast_q ? static_cast<int64_t>(pr.B) * pr.Lq : pr.N;
    if ((q_rows > 0 && (!q || !dq)) || (pr.N > 0 && (!k || !v || !dk || !dv)) ||
        (o_rows > 0 && (!o || !lse || !dout)))
        return JFA_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(dout, 16) ||
        !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16) || !aligned(lse, 4))
        return JFA_ERR_UNSUPPORTED;

    const size_t elems_kv = static_cast<size_t>(pr.N) * H * D;
    const size_t elems_q = static_cast<size_t>(q_rows) * H * D;
    char* ws = static_cast<char*>(workspace);
    if (o_rows == 0 || pr.N == 0) {
        if (q_rows > 0 && cudaMemsetAsync(dq, 0, elems_q * sizeof(float), s) != cudaSuccess) return JFA_ERR_CUDA;
        // no query rows: every key gets a zero gradient
        if (o_rows == 0 && elems_kv && (cudaMemsetAsync(dk, 0, elems_kv * 2, s) != cudaSuccess ||
                                        cudaMemsetAsync(dv, 0, elems_kv * 2, s) != cudaSuccess))
            return JFA_ERR_CUDA;
        return JFA_OK;
    }

    // Stream order: schedule copy (dense: done by the Delta pass itself),
    // zeroed dK/dV of unselected tiles (block-sparse), the Delta pre-pass
    // (which also zeroes dQ), then the main kernel.
    // Cluster Launch Control: the cost-sorted list (built as a one-CTA
    // schedule), one CTA per item; queues: one CTA per SM taking items from
    // its head group's queue at run time; otherwise a static deal to one CTA
    // per SM.
    const int policy = g_bwd_policy.load();
    const bool clc = policy == kSchedClc;
    const bool queue = policy == kSchedQueue;
    const int64_t n_items = count_items(pr, 1);
    const int P = clc ? 1 : ctas_for(n_items);

    float* delta = reinterpret_cast<float*>(ws + w.delta_off);
    PreParams pp;
    pp.o = static_cast<const uint16_t*>(o);
    pp.dout = static_cast<const uint16_t*>(dout);
    pp.delta = delta;
    pp.dq = dq;
    pp.dq_vec4 = static_cast<int64_t>(elems_q / 4);  // H * D is a multiple of 4
    pp.rows = o_rows * H;
    pp.B = pr.B;
    pp.Lq = pr.Lq;
    pp.H = H;
    pp.N = static_cast<int>(pr.N);
    pp.D = D;
    pp.broadcast_q = pr.broadcast_q;

    // Dense: the Delta pass, which runs right before the main kernel anyway,
    // moves the schedule from the pinned staging slot into the workspace, so
    // the stream holds no separate host-to-device copy.  (Block-sparse: the
    // zero-tile kernel reads the schedule region before the Delta pass, so
    // the schedule is copied as before.)
    bool pre_launched = false;
    const ScheduleUpload upload = [&](const void* src_dev, size_t bytes) {
        pp.sched_src = static_cast<const uint4*>(src_dev);
        pp.sched_dst = reinterpret_cast<uint4*>(ws + w.bwd_off);
        pp.sched_vec16 = static_cast<int64_t>(bytes / 16);
        pre_launched = true;
        return timed_launch(kProfPre, s, [&] { return launch_bwd_pre(pp, s); });
    };
    int64_t n_zero = 0;
    const int64_t n = stage_schedule(pr.off, pr.B, pr.Lq, pr.H, pr.broadcast_q, pr.causal, 1, P,
                                     policy, w, mask, ws + w.bwd_off, s, &n_zero, nullptr, &st,
                                     mask ? nullptr : &upload);
    if (n < 0) return st;
    if (n_zero > 0 && timed_launch(kProfZero, s, [&] {
                          return launch_zero_tiles(reinterpret_cast<const ZeroTile*>(ws + w.bwd_off + w.zero_off),
                                                   n_zero, static_cast<uint16_t*>(dk), static_cast<uint16_t*>(dv), H,
                                                   D, s);
                      }) != cudaSuccess)
        return JFA_ERR_CUDA;
    if (n == 0) return q_rows > 0 && cudaMemsetAsync(dq, 0, elems_q * sizeof(float), s) != cudaSuccess ? JFA_ERR_CUDA
                                                                                                 : JFA_OK;

    BwdMaps maps;
    if (!map_rows_bf16(&maps.q, q, q_rows, H, D, workspace) || !map_rows_bf16(&maps.k, k, pr.N, H, D, workspace) ||
        !map_rows_bf16(&maps.v, v, pr.N, H, D, workspace) || !map_rows_bf16(&maps.dout, dout, o_rows, H, D, workspace) ||
        !map_rows_f32(&maps.dq, dq, q_rows, H, D, workspace) || !map_rows_bf16(&maps.dk, dk, pr.N, H, D, workspace) ||
        !map_rows_bf16(&maps.dv, dv, pr.N, H, D, workspace))
        return JFA_ERR_CUDA;
    BwdParams p;
    p.cta_start = reinterpret_cast<const int32_t*>(ws + w.bwd_off);
    p.items = reinterpret_cast<const WorkItem*>(ws + w.bwd_off + kCtaStartBytes);
    p.lse = lse;
    p.delta = delta;
    p.dk = static_cast<uint16_t*>(dk);
    p.dv = static_cast<uint16_t*>(dv);
    p.status = reinterpret_cast<uint32_t*>(ws);
    p.Lq = pr.Lq;
    p.H = H;
    p.N = static_cast<int>(pr.N);
    p.broadcast_q = pr.broadcast_q;
    p.causal = pr.causal;
    p.clc = (clc || queue) ? 1 : 0;
    p.n_items = static_cast<int>(n);
    p.n_queues = queue ? queue_groups(pr.broadcast_q, H, P) : 0;
    p.queue = queue ? reinterpret_cast<int32_t*>(ws + w.bwd_off) + p.n_queues + 1 : nullptr;
    p.scale = pr.scale;
    p.scale_log2 = pr.scale * 1.4426950408889634f;
    p.wait_ns = wait_limit_ns();
    const int grid = clc ? static_cast<int>(n) : P;
    if (!pre_launched && timed_launch(kProfPre, s, [&] { return launch_bwd_pre(pp, s); }) != cudaSuccess)
        return JFA_ERR_CUDA;
    if (timed_launch(kProfBwd, s, [&] { return launch_bwd(D, p, maps, grid, s); }) != cudaSuccess) return JFA_ERR_CUDA;
    return JFA_OK;
}

extern "C" jfa_status jfa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                              const void* dout, const int32_t* offsets_dev, const int32_t* offsets_host, int B,
                              int Lq, int H, int D, int broadcast_q, int causal, float scale, float* dq, void* dk,
                              void* dv, void* workspace, size_t workspace_bytes, void* stream) {
    return bwd_impl(q, k, v, o, lse, dout, offsets_dev, offsets_host, nullptr, B, Lq, H, D, broadcast_q, causal, scale,
                    dq, dk, dv, workspace, workspace_bytes, stream);
}

extern "C" jfa_status jfa_bwd_block_sparse(const void* q, const void* k, const void* v, const void* o,
                                           const float* lse, const void* dout, const int32_t* offsets_dev,
                                           const int32_t* offsets_host, const uint8_t* kv_block_mask, int B, int Lq,
                                           int H, int D, int broadcast_q, float scale, float* dq, void* dk, void* dv,
                                           void* workspace, size_t workspace_bytes, void* stream) {
    if (!kv_block_mask) return JFA_ERR_INVALID_ARG;
    return bwd_impl(q, k, v, o, lse, dout, offsets_dev, offsets_host, kv_block_mask, B, Lq, H, D, broadcast_q, 0,
                    scale, dq, dk, dv, workspace, workspace_bytes, stream);
}

extern "C" int64_t jfa_num_kv_blocks(const int32_t* offsets_host, int B) {
    if (!offsets_host || B < 0) return -1;
    return num_kv_blocks(offsets_host, B);
}

extern "C" jfa_status jfa_device_status(void* workspace, void* stream) {
    if (!workspace) return JFA_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint32_t word = 0;
    if (cudaStreamSynchronize(s) != cudaSuccess) return JFA_ERR_CUDA;
    if (cudaMemcpy(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return JFA_ERR_CUDA;
    if (word != 0 && cudaMemset(workspace, 0, sizeof(word)) != cudaSuccess) return JFA_ERR_CUDA;
    return word ? JFA_ERR_DEVICE_TIMEOUT : JFA_OK;
}

extern "C" const char* jfa_status_string(jfa_status s) {
    switch (s) {
        case JFA_OK: return "JFA_OK";
        case JFA_ERR_INVALID_ARG: return "JFA_ERR_INVALID_ARG";
        case JFA_ERR_UNSUPPORTED: return "JFA_ERR_UNSUPPORTED";
        case JFA_ERR_WORKSPACE: return "JFA_ERR_WORKSPACE";
        case JFA_ERR_CUDA: return "JFA_ERR_CUDA";
        case JFA_ERR_DEVICE_TIMEOUT: return "JFA_ERR_DEVICE_TIMEOUT";
    }
    return "JFA_ERR_UNKNOWN";
}

extern "C" jfa_status jfa_profile_enable(int on) {
    Profiler& p = profiler();
    std::lock_guard<std::mutex> lock(p.mu);
    p.on = on != 0;
    return JFA_OK;
}

extern "C" jfa_status jfa_profile_read(double* ms, int* launches, int count) {
    Profiler& p = profiler();
    std::lock_guard<std::mutex> lock(p.mu);
    double t_ms[kProfKinds] = {};
    int n[kProfKinds] = {};
    jfa_status st = JFA_OK;
    for (auto& e : p.pending) {
        float t = 0.0f;
        if (cudaEventSynchronize(e.second.second) != cudaSuccess ||
            cudaEventElapsedTime(&t, e.second.first, e.second.second) != cudaSuccess)
            st = JFA_ERR_CUDA;
        t_ms[e.first] += t;
        n[e.first] += 1;
        p.pool.push_back(e.second.first);
        p.pool.push_back(e.second.second);
    }
    p.pending.clear();
    for (int k = 0; k < count && k < kProfKinds; ++k) {
        if (ms) ms[k] = t_ms[k];
        if (launches) launches[k] = n[k];
    }
    return st;
}
