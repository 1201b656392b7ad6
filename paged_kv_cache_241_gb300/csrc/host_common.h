// host_common.h -- host-side helpers shared by the pkv entry points.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pkv.h"

namespace pkv {

// Number of SMs of the current device (cached per device).
int device_sm_count();

// Let `func` (a __global__ function) use `bytes` of dynamic shared memory on
// the current device (the attribute is per device; it is only ever raised)
// and store in *ctas_per_sm how many of its CTAs of `threads` threads fit on
// an SM with that much.  Cached per (kernel, device) and thread-safe.
// Returns false on a CUDA error.
bool kernel_smem_setup(const void *func, int threads, int bytes, int *ctas_per_sm);

// Encode a bf16 tiled tensor map (driver entry point resolved at run time).
// dims/strides follow cuTensorMapEncodeTiled: dims[0] is innermost, strides
// are in bytes for dims 1..rank-1.  Returns false on failure.
bool encode_bf16_map(CUtensorMap *map, const void *base, int rank, const uint64_t *dims,
                     const uint64_t *strides_bytes, const uint32_t *box, bool swizzle128);

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline pkv_status launch_status() {
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // namespace pkv
