// bfq_internal.h — declarations shared by the library's translation units.
#pragma once

#include <stddef.h>
#include <stdint.h>

#include <utility>

#include "bfq.h"

#ifndef __CUDACC__
#include <cuda_runtime_api.h>
#else
#include <cuda_runtime.h>
#endif

namespace bfq {

// Per-device facts the launch plans depend on (cached per device ordinal).
struct DeviceInfo {
  int ordinal = -1;
  int sm_count = 0;
  int cc_major = 0;
  int cc_minor = 0;
  size_t smem_optin = 0;
};

// Fills *info for the current device.  Returns BFQ_OK or BFQ_ERR_CUDA.
bfq_status current_device(DeviceInfo* info);

// Device address of the library's status word on the current device
// (looked up once per device).  NULL on failure.
int* device_status_ptr();

inline bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

inline bfq_status launch_status(cudaError_t e) {
  return e == cudaSuccess ? (bfq_status)BFQ_OK : (bfq_status)BFQ_ERR_CUDA;
}

inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Whether launches use programmatic stream serialization (process-wide,
// default on; bfq_set_programmatic_launch switches it for measurements).
bool pdl_enabled();

// Launch `kernel` on `stream` with programmatic stream serialization (the
// kernel may start before the previous one in the stream has finished; it
// waits in griddep_wait() before touching memory) and an optional cluster
// size along x.  With programmatic launch switched off the kernel is
// launched with plain stream order (griddep_wait() is then a no-op).
// `programmatic` false: plain stream order whatever the switch says.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_kernel(bool programmatic, void (*kernel)(KArgs...), dim3 grid,
                                 dim3 block, size_t smem, cudaStream_t stream,
                                 unsigned cluster_x, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  unsigned n = 0;
  if (programmatic && pdl_enabled()) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (cluster_x > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cluster_x;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, unsigned cluster_x, Args&&... args) {
  return launch_kernel(true, kernel, grid, block, smem, stream, cluster_x,
                       std::forward<Args>(args)...);
}

// silu(g) of every bf16 gate g (indexed by its 16 bits), evaluated once per
// device by the library's fp32 silu; built on the first call that is not
// being captured into a CUDA graph (the build synchronizes `stream` once).
// Null while `stream` is capturing and the table is not built yet.  Defined
// in quant_kernels.cu.
const float* silu_table(const DeviceInfo& dev, cudaStream_t stream);

// Columns of a column-major scale array for K elements per row.
inline int64_t scale_cols(int64_t K, int32_t fmt) {
  return fmt == BFQ_SCALE_UE8M0_PACKED ? cdiv(K / 128, 4) : K / 128;
}

inline bool valid_fmt(int32_t fmt) {
  return fmt == BFQ_SCALE_F32 || fmt == BFQ_SCALE_F32_POW2 || fmt == BFQ_SCALE_UE8M0_PACKED;
}

}  // namespace bfq
