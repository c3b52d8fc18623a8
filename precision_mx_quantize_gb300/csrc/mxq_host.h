// Host-side helpers shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "mxq.h"

namespace mxq {

// Upper bound of every device-side wait, in nanoseconds.
uint64_t wait_timeout_ns();

// Number of SMs of the current device (cached per device).
int sm_count();

// cuTensorMapEncodeTiled obtained through the runtime's driver entry point;
// nullptr if unavailable.
PFN_cuTensorMapEncodeTiled_v12000 encode_tiled();

// Read and clear the device error word of each translation unit.
uint32_t take_quant_error();
uint32_t take_ablation_error();
uint32_t take_gemm_error();

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline mxq_status launch_status() {
  return cudaGetLastError() == cudaSuccess ? MXQ_OK : MXQ_ERR_CUDA;
}

}  // namespace mxq
