// One-pass (row-wise + column-wise) MX quantizer with an E5M2 output on at
// least one side: the second MXFP8 element type in the kernel of
// quant_kernel.cuh, instantiated in a translation unit of its own so that its
// instantiations compile in parallel with the others.
//
// Formats: "Lumen：AMD原生大模型量化训练框架的技术突破与实践", §1 -- FP8 E4M3 and
// E5M2 as the quantized-training formats; E5M2 elements (emax 15, largest
// finite 57344) with E8M0 block scales per OCP MX v1.0.
#include "quant_kernel.cuh"

namespace mxq {

namespace {

template <int FR, bool HR, int FC, bool HC>
QuantKernel dual_k() {
  return mx_quant_kernel<true, true, FR, HR, FC, HC, 0>;
}

template <int FR, bool HR>
QuantKernel dual_by_fc(int fc, bool hc) {
  if (fc == MXQ_E4M3) return hc ? dual_k<FR, HR, MXQ_E4M3, true>() : dual_k<FR, HR, MXQ_E4M3, false>();
  if (fc == MXQ_E5M2) return hc ? dual_k<FR, HR, MXQ_E5M2, true>() : dual_k<FR, HR, MXQ_E5M2, false>();
  return hc ? dual_k<FR, HR, MXQ_E2M1, true>() : dual_k<FR, HR, MXQ_E2M1, false>();
}

template <int FR, bool HR>
QuantKernel dual_col_e5m2(bool hc) {
  return hc ? dual_k<FR, HR, MXQ_E5M2, true>() : dual_k<FR, HR, MXQ_E5M2, false>();
}

// The kernel for (fr, hr, fc, hc) with fr == E5M2 or fc == E5M2.
QuantKernel pick_dual_e5m2(int fr, bool hr, int fc, bool hc) {
  if (fr == MXQ_E5M2) return hr ? dual_by_fc<MXQ_E5M2, true>(fc, hc) : dual_by_fc<MXQ_E5M2, false>(fc, hc);
  if (fr == MXQ_E4M3) return hr ? dual_col_e5m2<MXQ_E4M3, true>(hc) : dual_col_e5m2<MXQ_E4M3, false>(hc);
  return hr ? dual_col_e5m2<MXQ_E2M1, true>(hc) : dual_col_e5m2<MXQ_E2M1, false>(hc);
}

}  // namespace

mxq_status quant_launch_dual_e5m2(const void* x, int64_t R, int64_t C, int fr, int hr,
                                  void* codes_r, uint8_t* scales_r, int fc, int hc, void* codes_c,
                                  uint8_t* scales_c, void* stream, int scale_layout) {
  if (fr != MXQ_E5M2 && fc != MXQ_E5M2) return MXQ_ERR_ARG;
  if (!valid_fmt(fr) || !valid_fmt(fc)) return MXQ_ERR_ARG;
  return quant_launch_k(pick_dual_e5m2(fr, hr != 0, fc, hc != 0), x, R, C, true, true, fr, codes_r,
                        scales_r, fc, codes_c, scales_c, 0u, 0u, stream, scale_layout);
}

uint32_t take_quant_e5m2_error() { return take_error_word(); }

}  // namespace mxq
