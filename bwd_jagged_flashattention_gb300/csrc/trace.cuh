// trace.cuh -- optional per-role event trace of the attention kernels.
//
// Compiled in only when JFA_TRACE is defined (a separate build used to study
// the pipelines); otherwise every JFA_TRACE_EVENT expands to nothing.  In a
// trace build, one thread per role of the first kTraceCtas CTAs appends
// (SM clock, event, role, two arguments) records to a device buffer that
// jfa_trace_read() copies out.
#pragma once
#include <cstdint>

namespace jfa {
constexpr int kTraceCtas = 4;
constexpr int kTraceRoles = 16;
constexpr int kTraceCap = 2048;  // records per (CTA, role)
}  // namespace jfa

#ifdef JFA_TRACE
#include <cuda_runtime.h>
namespace jfa {
// One buffer per translation unit (no relocatable device code needed).
// Only one thread per role records, so a plain shared-memory counter per
// role suffices and every record is a fire-and-forget store.
static __device__ unsigned long long g_trace[kTraceCtas][kTraceRoles][kTraceCap][2];
static __device__ unsigned int g_trace_n[kTraceCtas][kTraceRoles];
static __shared__ unsigned int s_trace_n[kTraceRoles];

__device__ __forceinline__ void trace_init() {
    if (threadIdx.x < kTraceRoles) s_trace_n[threadIdx.x] = 0;
}

__device__ __forceinline__ void trace_event(int ev, int role, int a, int b) {
    if (blockIdx.x >= kTraceCtas) return;
    const unsigned int i = s_trace_n[role]++;
    if (i >= kTraceCap) return;
    g_trace[blockIdx.x][role][i][0] = clock64();
    g_trace[blockIdx.x][role][i][1] = (static_cast<unsigned long long>(ev) << 48) |
                                      (static_cast<unsigned long long>(role & 0xFF) << 40) |
                                      (static_cast<unsigned long long>(a & 0xFFFFF) << 20) |
                                      static_cast<unsigned long long>(b & 0xFFFFF);
    g_trace_n[blockIdx.x][role] = i + 1;
}
// Calibration record: SM clock and the global nanosecond timer together.
__device__ __forceinline__ void trace_clock(int role) {
    if (blockIdx.x >= kTraceCtas) return;
    const unsigned int i = s_trace_n[role]++;
    if (i >= kTraceCap) return;
    unsigned long long ns;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(ns));
    g_trace[blockIdx.x][role][i][0] = clock64();
    g_trace[blockIdx.x][role][i][1] = (99ull << 48) | (static_cast<unsigned long long>(role & 0xFF) << 40) |
                                      (ns & ((1ull << 40) - 1));
    g_trace_n[blockIdx.x][role] = i + 1;
}
}  // namespace jfa
#define JFA_TRACE_INIT() ::jfa::trace_init()
#define JFA_TRACE_CLOCK(role) ::jfa::trace_clock(role)
#define JFA_TRACE_EVENT(ev, role, a, b) ::jfa::trace_event((ev), (role), (a), (b))
// Defines extern "C" int NAME(void* host, unsigned* counts): copies this
// unit's records and per-(CTA, role) counts, then clears the counts.
#define JFA_TRACE_DEFINE_READER(NAME)                                                                \
    extern "C" int NAME(void* host, unsigned* counts) {                                              \
        if (cudaDeviceSynchronize() != cudaSuccess) return 1;                                        \
        if (cudaMemcpyFromSymbol(host, ::jfa::g_trace, sizeof(::jfa::g_trace)) != cudaSuccess)       \
            return 2;                                                                                \
        if (cudaMemcpyFromSymbol(counts, ::jfa::g_trace_n, sizeof(::jfa::g_trace_n)) != cudaSuccess) \
            return 3;                                                                                \
        unsigned zero[::jfa::kTraceCtas * ::jfa::kTraceRoles] = {0};                                 \
        return cudaMemcpyToSymbol(::jfa::g_trace_n, zero, sizeof(zero)) == cudaSuccess ? 0 : 4;     \
    }
#else
#define JFA_TRACE_INIT() \
    do {                 \
    } while (0)
#define JFA_TRACE_EVENT(ev, role, a, b) \
    do {                                \
    } while (0)
#define JFA_TRACE_CLOCK(role) \
    do {                       \
    } while (0)
#define JFA_TRACE_DEFINE_READER(NAME)
#endif
