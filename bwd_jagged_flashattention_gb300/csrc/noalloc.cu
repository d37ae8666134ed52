// noalloc.cu -- jfa_fwd_static_scratch: the forward pass for callers that
// cannot allocate memory.
//
// Some callers cannot hand the library a workspace: a plugin running inside
// an inference engine that owns all device memory and forbids allocation
// while it executes, code that runs with a fixed, pre-reserved memory pool,
// or a host program that must not touch any allocator on its hot path.
// This entry point needs nothing from them but the inputs and outputs.  Its
// scratch memory (the tile schedule and the kernel status word) lives in a
// fixed-size array in device global memory that the library declares at
// file scope; every GPU that loads the library holds those bytes until the
// process exits.  Host-side staging uses static buffers as well, so a call
// makes no allocation of any kind: no cudaMalloc/cudaFree, no pinned or
// heap memory.
//
// The array is shared by every call on a device and keeps the last call's
// contents.  Calls that overlap on the GPU (two streams, or two host threads
// whose launches run concurrently) race on it; serialise them.
//
// Set-up: the first call on each device looks up the array's device address
// with cudaGetSymbolAddress (a host-side name of a __device__ array is not a
// device address) and keeps it for the life of the process.  Make that first
// call before any stream capture.  The cached address does not survive
// cudaDeviceReset (the module may load elsewhere afterwards).
//
// The tile schedule is copied to the array from a host buffer that every call
// rewrites, so a call on a stream that is capturing is refused
// (JFA_ERR_UNSUPPORTED): a recorded copy would read whatever a later call
// left in that buffer.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <mutex>

#include "../../include/jfa.h"
#include "host_util.h"
#include "kernels.h"
#include "scheduler.h"

namespace jfa {
namespace {

// Scratch layout: [status word, 256 B][CTA bounds, 4 KiB][work items].
constexpr size_t kScratchBytes = size_t(1) << 20;  // 1 MiB per device
constexpr size_t kStatusBytes = 256;
constexpr size_t kStartsBytes = 4096;
constexpr int64_t kScratchMaxItems =
    static_cast<int64_t>((kScratchBytes - kStatusBytes - kStartsBytes) / sizeof(WorkItem));

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

// Host staging and schedule arrays (static: no heap use per call).
struct HostArena {
    alignas(64) unsigned char stage[kStartsBytes + kScratchMaxItems * sizeof(WorkItem)];
    WorkItem gen[kScratchMaxItems];
    int64_t order[kScratchMaxItems];
    int32_t owner[kScratchMaxItems];
    int32_t fill[kMaxCtas + 1];
    int64_t buckets[kCostBuckets + 2];
};
HostArena g_arena;
std::mutex g_mu;
void* g_scratch_addr[64] = {nullptr};

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// Device address of g_scratch on the current device, looked up once per
// device (with that device current) and cached; null on failure.  Callers
// hold g_mu.
char* scratch_address() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    if (!g_scratch_addr[dev]) {
        void* addr = nullptr;
        if (cudaGetSymbolAddress(&addr, g_scratch) != cudaSuccess || !addr) return nullptr;
        g_scratch_addr[dev] = addr;
    }
    return static_cast<char*>(g_scratch_addr[dev]);
}

bool map_rows_bf16(CUtensorMap* m, const void* base, int64_t rows, int H, int D, const void* fallback) {
    const uint64_t dims[2] = {static_cast<uint64_t>(H) * D, static_cast<uint64_t>(rows > 0 ? rows : 1)};
    const uint64_t strides[1] = {static_cast<uint64_t>(H) * D * 2};
    const uint32_t box[2] = {64, 128};
    return encode_tensor_map(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, rows > 0 ? base : fallback, dims, strides, box,
                             CU_TENSOR_MAP_SWIZZLE_128B);
}

}  // namespace
}  // namespace jfa

using namespace jfa;

extern "C" jfa_status jfa_fwd_static_scratch(const void* q, const void* k, const void* v, const int32_t* offsets_host,
                                             int B, int Lq, int H, int D, int broadcast_q, int causal, float scale,
                                             void* o, float* lse, void* stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (B < 0 || H <= 0 || Lq < 0 || !offsets_host || !std::isfinite(scale)) return JFA_ERR_INVALID_ARG;
    if (D != 64 && D != 128) return JFA_ERR_UNSUPPORTED;
    if (H > 255 || (broadcast_q && causal) || (broadcast_q && Lq > kMaxSeqLen)) return JFA_ERR_UNSUPPORTED;
    if (offsets_host[0] != 0) return JFA_ERR_INVALID_ARG;
    const int Lqb = broadcast_q ? Lq : 0;
    int64_t n_items = 0;
    for (int b = 0; b < B; ++b) {
        const int64_t len = static_cast<int64_t>(offsets_host[b + 1]) - offsets_host[b];
        if (len < 0) return JFA_ERR_INVALID_ARG;
        if (len > kMaxSeqLen) return JFA_ERR_UNSUPPORTED;
        const int64_t ntiles = broadcast_q ? (Lqb + 127) / 128 : (len + 127) / 128;
        n_items += static_cast<int64_t>(H) * ((ntiles + 1) / 2);
    }
    // The fixed scratch bounds the number of forward work items.
    if (n_items > kScratchMaxItems) return JFA_ERR_WORKSPACE;
    const int64_t N = offsets_host[B];
    const int64_t q_rows = broadcast_q ? Lqb : N;
    const int64_t o_rows = broadcast_q ? static_cast<int64_t>(B) * Lqb : N;
    if ((q_rows > 0 && !q) || (N > 0 && (!k || !v)) || (o_rows > 0 && (!o || !lse))) return JFA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
        (reinterpret_cast<uintptr_t>(lse) & 3))
        return JFA_ERR_UNSUPPORTED;
    if (o_rows == 0 || n_items == 0) return JFA_OK;

    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cap) != cudaSuccess) return JFA_ERR_CUDA;
    if (cap != cudaStreamCaptureStatusNone) return JFA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mu);
    char* scratch = scratch_address();
    if (!scratch) return JFA_ERR_CUDA;

    int P = device_sm_count();
    if (P <= 0) return JFA_ERR_CUDA;
    if (P > kMaxCtas) P = kMaxCtas;
    if (n_items < P) P = static_cast<int>(n_items);
    int32_t* starts = reinterpret_cast<int32_t*>(g_arena.stage);
    WorkItem* items = reinterpret_cast<WorkItem*>(g_arena.stage + kStartsBytes);
    const int64_t n = build_schedule_noalloc(offsets_host, B, Lqb, H, broadcast_q ? 1 : 0, causal ? 1 : 0, 0, P,
                                             items, starts, kScratchMaxItems, g_arena.gen, g_arena.order,
                                             g_arena.owner, g_arena.fill, g_arena.buckets);
    if (n < 0) return JFA_ERR_WORKSPACE;
    // Pageable source: the copy has consumed the staging buffer when it returns.
    if (cudaMemsetAsync(scratch, 0, sizeof(uint32_t), s) != cudaSuccess ||
        cudaMemcpyAsync(scratch + kStatusBytes, g_arena.stage, kStartsBytes + static_cast<size_t>(n) * sizeof(WorkItem),
                        cudaMemcpyHostToDevice, s) != cudaSuccess)
        return JFA_ERR_CUDA;

    FwdMaps maps;
    if (!map_rows_bf16(&maps.q, q, q_rows, H, D, scratch) || !map_rows_bf16(&maps.k, k, N, H, D, scratch) ||
        !map_rows_bf16(&maps.v, v, N, H, D, scratch) || !map_rows_bf16(&maps.o, o, o_rows, H, D, scratch))
        return JFA_ERR_CUDA;
    FwdParams p;
    p.status = reinterpret_cast<uint32_t*>(scratch);
    p.cta_start = reinterpret_cast<const int32_t*>(scratch + kStatusBytes);
    p.items = reinterpret_cast<const WorkItem*>(scratch + kStatusBytes + kStartsBytes);
    p.o = static_cast<uint16_t*>(o);
    p.lse = lse;
    p.Lq = Lqb;
    p.H = H;
    p.N = static_cast<int>(N);
    p.broadcast_q = broadcast_q ? 1 : 0;
    p.causal = causal ? 1 : 0;
    p.scale_log2 = (scale > 0.0f ? scale : 1.0f / std::sqrt(static_cast<float>(D))) * 1.4426950408889634f;
    p.wait_ns = wait_limit_ns();
    return launch_fwd(D, p, maps, P, s) == cudaSuccess ? JFA_OK : JFA_ERR_CUDA;
}

extern "C" jfa_status jfa_static_scratch_status(void* stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    std::lock_guard<std::mutex> lock(g_mu);
    char* scratch = scratch_address();
    if (!scratch || cudaStreamSynchronize(s) != cudaSuccess) return JFA_ERR_CUDA;
    uint32_t word = 0;
    if (cudaMemcpy(&word, scratch, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return JFA_ERR_CUDA;
    if (word != 0 && cudaMemset(scratch, 0, sizeof(word)) != cudaSuccess) return JFA_ERR_CUDA;
    return word ? JFA_ERR_DEVICE_TIMEOUT : JFA_OK;
}
