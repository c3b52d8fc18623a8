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
  const uint32_t words[4] = {take_quant_error(), take_ablation_error(), take_gemm_error(),
                             take_debug_error()};
  for (uint32_t w : words)
    if (w) return static_cast<mxq_status>(w & 0xFFu);
  return MXQ_OK;
}

extern "C" mxq_status mxq_debug_expire_wait(uint64_t limit_ns, void* stream) {
  expire_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(limit_ns);
  return launch_status();
}
