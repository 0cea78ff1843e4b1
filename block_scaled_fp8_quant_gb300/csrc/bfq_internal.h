// bfq_internal.h — declarations shared by the library's translation units.
#pragma once

#include <stddef.h>
#include <stdint.h>

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

// Columns of a column-major scale array for K elements per row.
inline int64_t scale_cols(int64_t K, int32_t fmt) {
  return fmt == BFQ_SCALE_UE8M0_PACKED ? cdiv(K / 128, 4) : K / 128;
}

inline bool valid_fmt(int32_t fmt) {
  return fmt == BFQ_SCALE_F32 || fmt == BFQ_SCALE_F32_POW2 || fmt == BFQ_SCALE_UE8M0_PACKED;
}

}  // namespace bfq
