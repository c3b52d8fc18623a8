// Device helpers shared by the MX kernels: shared-memory addresses,
// mbarriers with bounded waits, TMA and bulk copies, element conversions.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "mxq.h"

#define MXQ_DEV __device__ __forceinline__

namespace mxq {

// ---- error words --------------------------------------------------------
// Each translation unit owns one device error word; bit layout:
//   bits 0-7  : mxq_status of the first failure
//   bits 8-15 : site id of the wait that expired (or, in the bounds-checked
//               build, of the check that failed)
enum : uint32_t {
  SITE_QUANT_FULL = 1,
  SITE_QUANT_DRAIN = 2,
  SITE_GEMM_EMPTY = 3,
  SITE_GEMM_FULL = 4,
  SITE_GEMM_TMEM_FULL = 5,
  SITE_GEMM_TMEM_EMPTY = 6,
  SITE_GEMM_DRAIN = 7,
  SITE_DEBUG = 8,
  // bounds checks of the bounds-checked build (MXQ_DEBUG_BOUNDS)
  SITE_B_QUANT_TILE = 16,    // quantizer tile coordinates
  SITE_B_QUANT_TMA = 17,     // quantizer TMA coordinate alignment
  SITE_B_QUANT_SCALE = 18,   // row-major scale stores
  SITE_B_QUANT_SCALE_TC = 19,  // chunk-layout scale stores
  SITE_B_DQ_ROWS = 20,       // row-wise dequantizer loads / stores
  SITE_B_DQ_COLS = 21,       // column-wise dequantizer loads / stores
  SITE_B_GEMM_TILE = 22,     // GEMM tile coordinates
  SITE_B_GEMM_STORE = 23,    // GEMM epilogue stores of C / codes
  SITE_B_GEMM_QSCALE = 24,   // GEMM epilogue stores of output scales
  SITE_B_SF_CHUNKS = 25,     // scale re-layout stores
  SITE_B_GEMM_TMA = 26,      // GEMM TMA coordinates
};

MXQ_DEV void record_error(uint32_t* word, uint32_t status, uint32_t site) {
  atomicCAS(word, 0u, (status & 0xFFu) | ((site & 0xFFu) << 8));
}

// ---- bounds checks ------------------------------------------------------
// In the bounds-checked build (compiled with -DMXQ_DEBUG_BOUNDS into
// libmxq_debug.so) every global index a kernel computes from its arguments
// is checked, before the access, against the extent those arguments imply.
// A failed check records MXQ_ERR_BOUNDS and the site in the translation
// unit's error word (mxq_check reports it) and the access is skipped; no
// check traps.  In the normal build the checks compile away.
MXQ_DEV bool bounds_ok(bool ok, uint32_t* word, uint32_t site) {
  if (!ok) record_error(word, MXQ_ERR_BOUNDS, site);
  return ok;
}
#ifdef MXQ_DEBUG_BOUNDS
#define MXQ_IN_BOUNDS(cond, word, site) ::mxq::bounds_ok((cond), (word), (site))
#else
#define MXQ_IN_BOUNDS(cond, word, site) true
#endif

// ---- shared memory / mbarrier -------------------------------------------
MXQ_DEV uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

MXQ_DEV void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

MXQ_DEV void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

MXQ_DEV void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

MXQ_DEV void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

MXQ_DEV bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

MXQ_DEV uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait for the phase with the given parity to complete, giving up after
// limit_ns nanoseconds.  Returns false when the limit ran out.
MXQ_DEV bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_ns() - t0 > limit_ns) return false;
  }
  return true;
}

// ---- TMA / bulk copies ----------------------------------------------------
// 2-D tiled TMA load into this CTA's shared memory; completion is signalled
// on `bar` as transaction bytes.  x (innermost) * element size must be a
// multiple of 16 bytes.
MXQ_DEV void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int32_t x,
                         int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
      : "memory");
}

// Contiguous bulk copy global -> shared (16-byte aligned, size % 16 == 0).
MXQ_DEV void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

MXQ_DEV void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---- programmatic dependent launch --------------------------------------------
// Kernels launched with programmatic stream serialization may start while
// the previous kernel on the stream is still finishing.  Each such kernel
// sets up what needs no global memory (barriers, tensor memory, descriptor
// prefetch), then waits for the previous grid to complete and its writes to
// be visible before touching global memory, and lets the next kernel launch
// early.  Every CTA of these grids is resident at once, so a dependent grid
// waiting on free SMs can never hold up this one.
MXQ_DEV void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
MXQ_DEV void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---- shared exponents -------------------------------------------------------
// E8M0 byte from the magnitude bits of the block amax (fp32 layout):
// floor(log2 amax) - emax + 127 = biased_exponent - emax, clamped at 0
// (zero and subnormal maxima included); 255 for NaN / Inf.
MXQ_DEV uint32_t scale_of(uint32_t abits, uint32_t emax) {
  if (abits >= 0x7F800000u) return 255u;
  const uint32_t E = abits >> 23;
  return E > emax ? E - emax : 0u;
}

// 2^(127 - s), always a normal fp32 for the scales the quantizer produces
// (s <= 252); 1 for a NaN block whose codes are discarded.
MXQ_DEV float inv_scale(uint32_t s) {
  return s == 255u ? 1.0f : __uint_as_float((254u - s) << 23);
}

// ---- element conversions ----------------------------------------------------
// Four fp32 values -> four E4M3 codes (round to nearest even, saturating),
// a0 in the lowest byte.
MXQ_DEV uint32_t cvt_e4m3x4(float a0, float a1, float a2, float a3) {
  uint32_t r;
  asm("{\n\t.reg .b16 lo, hi;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n\t"
      "mov.b32 %0, {lo, hi};\n\t}"
      : "=r"(r)
      : "f"(a0), "f"(a1), "f"(a2), "f"(a3));
  return r;
}

// Four fp32 values -> four E5M2 codes (round to nearest even, saturating to
// the largest finite magnitude), a0 in the lowest byte.
MXQ_DEV uint32_t cvt_e5m2x4(float a0, float a1, float a2, float a3) {
  uint32_t r;
  asm("{\n\t.reg .b16 lo, hi;\n\t"
      "cvt.rn.satfinite.e5m2x2.f32 lo, %2, %1;\n\t"
      "cvt.rn.satfinite.e5m2x2.f32 hi, %4, %3;\n\t"
      "mov.b32 %0, {lo, hi};\n\t}"
      : "=r"(r)
      : "f"(a0), "f"(a1), "f"(a2), "f"(a3));
  return r;
}

// Eight fp32 values -> eight E2M1 codes packed in a word, a0 in the lowest
// nibble.
MXQ_DEV uint32_t cvt_e2m1x8(float a0, float a1, float a2, float a3, float a4, float a5, float a6,
                            float a7) {
  uint32_t r;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(r)
      : "f"(a0), "f"(a1), "f"(a2), "f"(a3), "f"(a4), "f"(a5), "f"(a6), "f"(a7));
  return r;
}

// max(|a|, |b|, |c|) propagating NaN.
MXQ_DEV float max3_abs_nan(float a, float b, float c) {
  float d;
  asm("max.NaN.abs.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Lane-wise max of the magnitudes of two bf16 pairs, propagating NaN (the
// sign bits of the result are meaningless).
MXQ_DEV uint32_t max_abs_bf16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.NaN.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

MXQ_DEV float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
MXQ_DEV float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

}  // namespace mxq
