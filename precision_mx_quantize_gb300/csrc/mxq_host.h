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

// A 2-D tiled tensor map of `base` (dims d0 inner x d1, row stride in bytes,
// box0 x box1, element strides 1, no interleave, zero fill), encoded once per
// distinct argument set and device and then served from a small cache: the
// encoding depends only on these arguments, so a cached map is valid for any
// later call that passes the same ones.  Returns CUDA_SUCCESS or the
// encoder's error.
CUresult tensor_map_2d(CUtensorMap* out, CUtensorMapDataType dtype, const void* base, uint64_t d0,
                       uint64_t d1, uint64_t stride_bytes, uint32_t box0, uint32_t box1,
                       CUtensorMapSwizzle swizzle, CUtensorMapL2promotion l2);

// The same for a 3-D tensor (dims d0 inner, d1, d2; strides of dims 1 and 2
// in bytes; box box0 x box1 x box2).
CUresult tensor_map_3d(CUtensorMap* out, CUtensorMapDataType dtype, const void* base, uint64_t d0,
                       uint64_t d1, uint64_t d2, uint64_t stride1_bytes, uint64_t stride2_bytes,
                       uint32_t box0, uint32_t box1, uint32_t box2, CUtensorMapSwizzle swizzle,
                       CUtensorMapL2promotion l2);

// cudaFuncSetAttribute(MaxDynamicSharedMemorySize) for `kernel` on the
// current device, done once per (kernel, device, size).
bool ensure_dynamic_smem(const void* kernel, int bytes);

// The one-pass quantizer when either output is E5M2 (its own translation
// unit); arguments as mxq_quantize_dual_ex, status as the C entry points.
mxq_status quant_launch_dual_e5m2(const void* x, int64_t R, int64_t C, int fr, int hr,
                                  void* codes_r, uint8_t* scales_r, int fc, int hc, void* codes_c,
                                  uint8_t* scales_c, void* stream, int scale_layout);

// Read and clear the device error word of each translation unit.
uint32_t take_quant_error();
uint32_t take_quant_e5m2_error();
uint32_t take_ablation_error();
uint32_t take_gemm_error();

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline mxq_status launch_status() {
  return cudaGetLastError() == cudaSuccess ? MXQ_OK : MXQ_ERR_CUDA;
}

}  // namespace mxq
