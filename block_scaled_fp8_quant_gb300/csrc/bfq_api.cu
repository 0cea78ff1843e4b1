// bfq_api.cu — host-side plumbing of the C ABI: version, status strings,
// per-device facts, the device error latch and the watchdog self-test.
#include <atomic>
#include <mutex>

#include "bfq_device.cuh"

namespace bfq {

__device__ int g_device_status = 0;
// Where take_status_kernel leaves the value it took from the latch.
__device__ int g_status_taken = 0;

namespace {
std::atomic<int> g_pdl{1};
constexpr int kMaxDevices = 64;
DeviceInfo g_info[kMaxDevices];
int* g_status_ptr[kMaxDevices];
std::mutex g_info_mu;
}  // namespace

bool pdl_enabled() { return g_pdl.load(std::memory_order_relaxed) != 0; }

int* device_status_ptr() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_info_mu);
  if (!g_status_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    g_status_ptr[dev] = (int*)p;
  }
  return g_status_ptr[dev];
}

bfq_status current_device(DeviceInfo* info) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return BFQ_ERR_CUDA;
  }
  {
    std::lock_guard<std::mutex> lock(g_info_mu);
    if (g_info[dev].ordinal == dev) {
      *info = g_info[dev];
      return BFQ_OK;
    }
  }
  DeviceInfo d;
  d.ordinal = dev;
  int optin = 0;
  if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev) !=
          cudaSuccess ||
      cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) !=
          cudaSuccess ||
      cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
          cudaSuccess) {
    cudaGetLastError();
    return BFQ_ERR_CUDA;
  }
  d.smem_optin = (size_t)optin;
  std::lock_guard<std::mutex> lock(g_info_mu);
  g_info[dev] = d;
  *info = d;
  return BFQ_OK;
}

// Waits on an mbarrier that no thread ever arrives on; the bounded wait gives
// up after timeout_ns, latches BFQ_ERR_TIMEOUT and the kernel returns.
__global__ void watchdog_selftest_kernel(int* status, uint64_t timeout_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) (void)mbar_wait(&bar, 0, &abort_flag, status, timeout_ns);
  __syncthreads();
}

// Reads and clears the latch in one atomic exchange, so that a timeout a
// kernel on another stream latches at the same moment is either returned now
// or kept for the next poll, never lost between a read and a clear.
__global__ void take_status_kernel(int* status, int* taken) { *taken = atomicExch(status, 0); }

}  // namespace bfq

using namespace bfq;

extern "C" int32_t bfq_version(void) { return 1 * 10000 + 0 * 100 + 0; }

extern "C" const char* bfq_status_string(bfq_status status) {
  switch (status) {
    case BFQ_OK: return "BFQ_OK";
    case BFQ_ERR_INVALID_ARG: return "BFQ_ERR_INVALID_ARG";
    case BFQ_ERR_UNSUPPORTED_SHAPE: return "BFQ_ERR_UNSUPPORTED_SHAPE";
    case BFQ_ERR_MISALIGNED: return "BFQ_ERR_MISALIGNED";
    case BFQ_ERR_FORMAT: return "BFQ_ERR_FORMAT";
    case BFQ_ERR_CUDA: return "BFQ_ERR_CUDA";
    case BFQ_ERR_TIMEOUT: return "BFQ_ERR_TIMEOUT";
    case BFQ_ERR_WORKSPACE: return "BFQ_ERR_WORKSPACE";
    case BFQ_ERR_DEVICE: return "BFQ_ERR_DEVICE";
    case BFQ_ERR_DEVICE_BOUNDS: return "BFQ_ERR_DEVICE_BOUNDS";
    default: return "BFQ_ERR_UNKNOWN";
  }
}

extern "C" int32_t bfq_set_programmatic_launch(int32_t enable) {
  return g_pdl.exchange(enable ? 1 : 0);
}

extern "C" bfq_status bfq_poll_device_status(void* stream) {
  cudaStream_t s = (cudaStream_t)stream;
  int* status = device_status_ptr();
  int* taken = nullptr;
  if (!status || cudaGetSymbolAddress((void**)&taken, g_status_taken) != cudaSuccess) {
    cudaGetLastError();
    return BFQ_ERR_CUDA;
  }
  int host = 0;
  take_status_kernel<<<1, 1, 0, s>>>(status, taken);
  if (cudaGetLastError() != cudaSuccess ||
      cudaMemcpyAsync(&host, taken, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess) {
    cudaGetLastError();
    return BFQ_ERR_CUDA;
  }
  return host == 0 ? (bfq_status)BFQ_OK : (bfq_status)host;
}

extern "C" bfq_status bfq_watchdog_selftest(int32_t timeout_us, void* stream) {
  if (timeout_us < 1 || timeout_us > 1000000) return BFQ_ERR_INVALID_ARG;
  DeviceInfo dev;
  bfq_status st = current_device(&dev);
  if (st != BFQ_OK) return st;
  int* status = device_status_ptr();
  if (!status) return BFQ_ERR_CUDA;
  watchdog_selftest_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(status,
                                                               (uint64_t)timeout_us * 1000ull);
  return launch_status(cudaGetLastError());
}
