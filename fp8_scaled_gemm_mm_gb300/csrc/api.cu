// api.cu -- library-wide pieces of libfp8mm: the per-device status word, TMA
// descriptor construction through the driver entry point, status strings,
// and a self-test of the bounded in-kernel wait.
#include <cudaTypedefs.h>

#include <atomic>
#include <map>
#include <mutex>
#include <utility>

#include "common.cuh"
#include "ptx.cuh"

namespace fp8mm {

__device__ int g_status_word = 0;

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_mu;
int* g_status_ptr[kMaxDevices] = {};
int g_sms[kMaxDevices] = {};
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::mutex g_once_mu;   // separate from g_mu: set-ups may call num_sms() and the like
std::map<std::pair<const void*, int>, int> g_once;
std::atomic<uint64_t> g_wait_ns{kWaitTimeoutNs};
}  // namespace

uint64_t wait_timeout_ns() { return g_wait_ns.load(std::memory_order_relaxed); }

int once_per_device(const void* key, const std::function<int()>& setup) {
  int dev = 0;
  const cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return -static_cast<int>(e);
  std::lock_guard<std::mutex> lk(g_once_mu);
  const auto it = g_once.find({key, dev});
  if (it != g_once.end()) return it->second;
  const int r = setup();
  if (r >= 0) g_once[{key, dev}] = r;
  return r;
}

int* status_word_device_ptr() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_status_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
    g_status_ptr[dev] = static_cast<int*>(p);
  }
  return g_status_ptr[dev];
}

int num_sms() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_sms[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    g_sms[dev] = n;
  }
  return g_sms[dev];
}

bool make_tma_2d(CUtensorMap* map, void* base, CUtensorMapDataType dtype, uint64_t inner, uint64_t outer,
                 uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swz) {
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_encode) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
              cudaSuccess ||
          q != cudaDriverEntryPointSuccess || !fn)
        return false;
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
  }
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_stride_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, dtype, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// A barrier that nothing ever arrives on: the bounded wait must give up after
// `timeout_ns`, record FP8MM_ETIMEOUT and return.
__global__ void bounded_wait_selftest_kernel(int* status, uint64_t timeout_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(&bar, 0, &abort_flag, status, timeout_ns, FP8MM_ETIMEOUT);
  __syncthreads();
}

}  // namespace fp8mm

using namespace fp8mm;

extern "C" int fp8mm_get_device_status(int device, int clear) {
  int prev = -1;
  if (device >= 0) {
    if (cudaGetDevice(&prev) != cudaSuccess) return FP8MM_ECUDA;
    if (cudaSetDevice(device) != cudaSuccess) return FP8MM_ECUDA;
  }
  int value = FP8MM_ECUDA;
  int* p = status_word_device_ptr();
  if (p && cudaDeviceSynchronize() == cudaSuccess) {
    int v = 0;
    if (cudaMemcpy(&v, p, sizeof(int), cudaMemcpyDeviceToHost) == cudaSuccess) {
      value = v;
      if (clear) {
        int z = 0;
        if (cudaMemcpy(p, &z, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) value = FP8MM_ECUDA;
      }
    }
  }
  if (prev >= 0) cudaSetDevice(prev);
  return value;
}

extern "C" int fp8mm_selftest_bounded_wait(int64_t timeout_ns, fp8mm_stream_t stream) {
  if (timeout_ns <= 0 || timeout_ns > 10000000000ll) return FP8MM_EINVAL;
  int* status = status_word_device_ptr();
  if (!status) return FP8MM_ECUDA;
  bounded_wait_selftest_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      status, static_cast<uint64_t>(timeout_ns));
  return cudaGetLastError() == cudaSuccess ? FP8MM_OK : FP8MM_ECUDA;
}

extern "C" int fp8mm_set_wait_timeout_ns(int64_t timeout_ns) {
  if (timeout_ns < 0 || timeout_ns > static_cast<int64_t>(kWaitTimeoutNs)) return FP8MM_EINVAL;
  g_wait_ns.store(timeout_ns == 0 ? kWaitTimeoutNs : static_cast<uint64_t>(timeout_ns),
                       std::memory_order_relaxed);
  return FP8MM_OK;
}

extern "C" const char* fp8mm_status_string(int status) {
  switch (status) {
    case FP8MM_OK: return "FP8MM_OK";
    case FP8MM_EINVAL: return "FP8MM_EINVAL: invalid argument";
    case FP8MM_EALIGN: return "FP8MM_EALIGN: alignment requirement violated";
    case FP8MM_EUNSUPPORTED: return "FP8MM_EUNSUPPORTED: not supported by this build";
    case FP8MM_ECUDA: return "FP8MM_ECUDA: CUDA runtime or driver call failed";
    case FP8MM_ETIMEOUT: return "FP8MM_ETIMEOUT: a kernel-side bounded wait ran out";
    default: return "unknown fp8mm status";
  }
}

extern "C" int fp8mm_version(void) { return (1 << 16) | 0; }
