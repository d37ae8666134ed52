// host_util.h -- host-side helpers shared by the library's translation units:
// TMA tensor-map encoding (through the driver entry point, so the library
// needs no link-time libcuda) and device-property caching.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace jfa {

// Encode a 2D/3D tiled tensor map.  dims[0] is the innermost (contiguous)
// dimension; strides_bytes[i] is the byte stride of dimension i+1.
// Returns false if the driver rejects the map.
bool encode_tensor_map(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const void* base,
                       const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                       CUtensorMapSwizzle swizzle);

// Number of SMs of the current device (cached per device).
int device_sm_count();

// Limit of one barrier wait inside the kernels, in nanoseconds (process-wide;
// jfa_set_wait_limit sets it, 4 s by default).
uint64_t wait_limit_ns();
void set_wait_limit_ns(uint64_t ns);

}  // namespace jfa
