// common.cuh -- shared host/device declarations of libfp8mm (not part of the public ABI).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "fp8mm.h"

namespace fp8mm {

// Per-device status word (defined in api.cu).  Kernels receive its device
// address as a parameter and record the first error with atomicCAS.
int* status_word_device_ptr();   // nullptr if it cannot be resolved

// Number of SMs of the current device (cached per device).
int num_sms();

// Build a 2-D tiled TMA descriptor through the driver entry point.
//   dtype: CU_TENSOR_MAP_DATA_TYPE_*; dims/box in elements (inner first);
//   row_stride_bytes: bytes between consecutive rows.
bool make_tma_2d(CUtensorMap* map, void* base, CUtensorMapDataType dtype, uint64_t inner, uint64_t outer,
                 uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swz);

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Upper bound on any single in-kernel wait before it gives up (ns).
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;

}  // namespace fp8mm
