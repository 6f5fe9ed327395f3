// common.cuh -- shared host/device declarations of libfp8mm (not part of the public ABI).
#pragma once

#include <cstdint>
#include <functional>
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

// One-time set-up per (key, current device): the first call for a pair runs
// `setup` and stores its result if it is >= 0 (a negative result is returned and
// not stored, so the next call tries again); later calls return the stored value.
// Thread-safe: two host threads launching at once run the set-up once.  `setup`
// must not call back into this function.
int once_per_device(const void* key, const std::function<int()>& setup);

// Raise `kernel`'s dynamic shared-memory limit to `bytes` once per device.
inline cudaError_t smem_opt_in(const void* kernel, int bytes) {
  const int r = once_per_device(kernel, [&]() {
    const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    return e == cudaSuccess ? 0 : -static_cast<int>(e);
  });
  return r < 0 ? static_cast<cudaError_t>(-r) : cudaSuccess;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Launch `kern` as a programmatic dependent of the work before it on the stream: its
// CTAs may start (set up, prefetch into L2) once that work lets its dependents launch,
// and read anything it produced only after griddepcontrol.wait, which every kernel
// launched this way executes first.  Every GEMM and the group / per-token quant
// kernels are launched so; the quant kernels and the small-M GEMMs let their own
// dependents launch when they start.  cluster_x > 0 adds a cluster of that size.
template <typename Kern, typename... Args>
cudaError_t launch_pdl(Kern kern, dim3 grid, dim3 block, size_t smem, cudaStream_t st, unsigned cluster_x,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  int n = 1;
  if (cluster_x > 0) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cluster_x;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    n = 2;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// Upper bound on any single in-kernel wait before it gives up (ns).
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;

// Limit of the pipeline waits of the GEMM and group-quant kernels launched from now
// on: kWaitTimeoutNs unless fp8mm_set_wait_timeout_ns set another (defined in api.cu).
uint64_t wait_timeout_ns();

}  // namespace fp8mm
