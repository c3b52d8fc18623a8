// Library-wide entry points: version, status strings, error collection,
// wait limits and the host helpers the kernels' launchers share.
#include <atomic>
#include <mutex>

#include "mxq_common.cuh"
#include "mxq_host.h"

namespace mxq {

namespace {
std::atomic<uint64_t> g_timeout{2000000000ull};
__device__ uint32_t g_err_debug;

// One CTA waits on a barrier that nobody arrives on; the bounded wait runs
// out after limit_ns and records MXQ_ERR_TIMEOUT.
__global__ void expire_wait_kernel(uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
  }
  __syncthreads();
  const bool ok = mbar_wait(smem_u32(&bar), 0, limit_ns);
  if (!ok && threadIdx.x == 0) record_error(&g_err_debug, MXQ_ERR_TIMEOUT, SITE_DEBUG);
}

uint32_t take_debug_error() {
  uint32_t h = 0;
  if (cudaMemcpyFromSymbol(&h, g_err_debug, sizeof(h)) != cudaSuccess) return MXQ_ERR_CUDA;
  if (h) {
    const uint32_t z = 0;
    cudaMemcpyToSymbol(g_err_debug, &z, sizeof(z));
  }
  return h;
}
}  // namespace

uint64_t wait_timeout_ns() { return g_timeout.load(std::memory_order_relaxed); }

int sm_count() {
  static std::mutex mu;
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 1;
  if (dev >= 64) {
    int n = 1;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    return n;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (cached[dev] == 0) {
    int n = 1;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cached[dev] = n > 0 ? n : 1;
  }
  return cached[dev];
}

PFN_cuTensorMapEncodeTiled_v12000 encode_tiled() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

namespace {

struct TmapKey {
  const void* base;
  uint64_t d0, d1, d2, s1, s2;
  uint32_t box0, box1, box2;
  int rank, dtype, swizzle, l2, dev;
  bool operator==(const TmapKey& o) const {
    return base == o.base && d0 == o.d0 && d1 == o.d1 && d2 == o.d2 && s1 == o.s1 && s2 == o.s2 &&
           box0 == o.box0 && box1 == o.box1 && box2 == o.box2 && rank == o.rank &&
           dtype == o.dtype && swizzle == o.swizzle && l2 == o.l2 && dev == o.dev;
  }
};

struct TmapEntry {
  bool used;
  TmapKey key;
  CUtensorMap map;
};

constexpr int kTmapSlots = 512;   // direct-mapped; a collision just re-encodes
std::mutex g_tmap_mu;
TmapEntry g_tmap[kTmapSlots];

uint64_t mix(uint64_t h, uint64_t v) {
  h ^= v + 0x9E3779B97F4A7C15ull + (h << 6) + (h >> 2);
  return h;
}

// Encodes (or serves from the cache) a tiled tensor map of rank 2 or 3.
CUresult tensor_map_nd(CUtensorMap* out, const TmapKey& k) {
  uint64_t h = reinterpret_cast<uintptr_t>(k.base);
  for (uint64_t v : {k.d0, k.d1, k.d2, k.s1, k.s2, (uint64_t(k.box0) << 32) | k.box1,
                     uint64_t(k.box2), (uint64_t(k.dtype) << 48) | (uint64_t(k.swizzle) << 32) |
                                           (uint64_t(k.l2) << 16) | uint64_t(k.rank)})
    h = mix(h, v);
  h = mix(h, uint64_t(k.dev));
  TmapEntry& e = g_tmap[h % kTmapSlots];
  {
    std::lock_guard<std::mutex> lock(g_tmap_mu);
    if (e.used && e.key == k) {
      *out = e.map;
      return CUDA_SUCCESS;
    }
  }
  PFN_cuTensorMapEncodeTiled_v12000 encode = encode_tiled();
  if (!encode) return CUDA_ERROR_NOT_FOUND;
  const cuuint64_t dims[3] = {k.d0, k.d1, k.d2};
  const cuuint64_t strides[2] = {k.s1, k.s2};
  const cuuint32_t box[3] = {k.box0, k.box1, k.box2};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = encode(out, static_cast<CUtensorMapDataType>(k.dtype),
                            static_cast<cuuint32_t>(k.rank), const_cast<void*>(k.base), dims,
                            strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                            static_cast<CUtensorMapSwizzle>(k.swizzle),
                            static_cast<CUtensorMapL2promotion>(k.l2),
                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r == CUDA_SUCCESS) {
    std::lock_guard<std::mutex> lock(g_tmap_mu);
    e.used = true;
    e.key = k;
    e.map = *out;
  }
  return r;
}

}  // namespace

CUresult tensor_map_2d(CUtensorMap* out, CUtensorMapDataType dtype, const void* base, uint64_t d0,
                       uint64_t d1, uint64_t stride_bytes, uint32_t box0, uint32_t box1,
                       CUtensorMapSwizzle swizzle, CUtensorMapL2promotion l2) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return CUDA_ERROR_INVALID_CONTEXT;
  const TmapKey k{base, d0, d1, 1, stride_bytes, 0, box0, box1, 1, 2, static_cast<int>(dtype),
                  static_cast<int>(swizzle), static_cast<int>(l2), dev};
  return tensor_map_nd(out, k);
}

CUresult tensor_map_3d(CUtensorMap* out, CUtensorMapDataType dtype, const void* base, uint64_t d0,
                       uint64_t d1, uint64_t d2, uint64_t stride1_bytes, uint64_t stride2_bytes,
                       uint32_t box0, uint32_t box1, uint32_t box2, CUtensorMapSwizzle swizzle,
                       CUtensorMapL2promotion l2) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return CUDA_ERROR_INVALID_CONTEXT;
  const TmapKey k{base, d0, d1, d2, stride1_bytes, stride2_bytes, box0, box1, box2, 3,
                  static_cast<int>(dtype), static_cast<int>(swizzle), static_cast<int>(l2), dev};
  return tensor_map_nd(out, k);
}

bool ensure_dynamic_smem(const void* kernel, int bytes) {
  struct Done {
    const void* kernel;
    int dev, bytes;
  };
  static std::mutex mu;
  static Done done[256];
  static int n_done = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < n_done; ++i)
    if (done[i].kernel == kernel && done[i].dev == dev && done[i].bytes >= bytes) return true;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) !=
      cudaSuccess)
    return false;
  if (n_done < 256) done[n_done++] = Done{kernel, dev, bytes};
  return true;
}

}  // namespace mxq

using namespace mxq;

extern "C" int mxq_version(void) { return (0 << 16) | 1; }

extern "C" const char* mxq_status_str(int status) {
  switch (status) {
    case MXQ_OK: return "ok";
    case MXQ_ERR_ARG: return "invalid argument";
    case MXQ_ERR_ALIGN: return "misaligned pointer or dimension";
    case MXQ_ERR_UNSUPPORTED: return "unsupported request";
    case MXQ_ERR_CUDA: return "CUDA error";
    case MXQ_ERR_TIMEOUT: return "device-side wait timed out";
    case MXQ_ERR_WORKSPACE: return "workspace too small";
    case MXQ_ERR_BOUNDS: return "index out of bounds (bounds-checked build)";
    default: return "unknown status";
  }
}

extern "C" void mxq_set_wait_timeout_ns(uint64_t ns) {
  g_timeout.store(ns ? ns : 1, std::memory_order_relaxed);
}

extern "C" mxq_status mxq_check(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return MXQ_ERR_CUDA;
  }
  if (cudaGetLastError() != cudaSuccess) return MXQ_ERR_CUDA;
  const uint32_t words[5] = {take_quant_error(), take_quant_e5m2_error(), take_ablation_error(),
                             take_gemm_error(), take_debug_error()};
  for (uint32_t w : words)
    if (w) return static_cast<mxq_status>(w & 0xFFu);
  return MXQ_OK;
}

extern "C" mxq_status mxq_debug_expire_wait(uint64_t limit_ns, void* stream) {
  expire_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(limit_ns);
  return launch_status();
}
