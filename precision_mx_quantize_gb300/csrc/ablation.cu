// Ablation quantizer: MX quantization with a random-sign Hadamard rotation
// and/or stochastic rounding, the two sources of randomness that
// "AMD顛覆行業認知！終于攻克FP4大模型訓練致命難題", §01, contrasts with its
// deterministic rotation.  Same kernel as the deterministic quantizer
// (quant_kernel.cuh), instantiated with the ABL flags; the random bits come
// from Philox4x32-10 inside the kernel, so the result depends only on the
// input, the sign mask and the seed.
#include "quant_kernel.cuh"

namespace mxq {

namespace {

template <bool ROW, int F, bool H, int ABL>
QuantKernel ablation_ptr() {
  if constexpr (ROW) return mx_quant_kernel<true, false, F, H, 0, false, ABL>;
  else return mx_quant_kernel<false, true, 0, false, F, H, ABL>;
}

template <bool ROW, int F>
QuantKernel ablation_for_fmt(bool had, bool sr) {
  if (had) return sr ? ablation_ptr<ROW, F, true, ABL_SIGN | ABL_SR>()
                     : ablation_ptr<ROW, F, true, ABL_SIGN>();
  return ablation_ptr<ROW, F, false, ABL_SR>();
}

template <bool ROW>
QuantKernel ablation_pick(int fmt, bool had, bool sr) {
  if (fmt == MXQ_E4M3) return ablation_for_fmt<ROW, MXQ_E4M3>(had, sr);
  if (fmt == MXQ_E5M2) return ablation_for_fmt<ROW, MXQ_E5M2>(had, sr);
  return ablation_for_fmt<ROW, MXQ_E2M1>(had, sr);
}

}  // namespace

uint32_t take_ablation_error() { return take_error_word(); }

}  // namespace mxq

using namespace mxq;

extern "C" mxq_status mxq_quantize_ablation(const void* x, int64_t rows, int64_t cols, int layout,
                                            int fmt, int hadamard, uint32_t sign_mask,
                                            int stochastic, uint64_t seed, void* codes,
                                            uint8_t* scales, void* stream) {
  if (layout != MXQ_ROWWISE && layout != MXQ_COLWISE_T) return MXQ_ERR_ARG;
  if (!hadamard && sign_mask != 0u) return MXQ_ERR_ARG;
  const bool row = layout == MXQ_ROWWISE;
  if (!hadamard && !stochastic) return mxq_quantize(x, rows, cols, layout, fmt, codes, scales, stream);
  if (!stochastic && sign_mask == 0u)
    return mxq_hadamard_quantize(x, rows, cols, layout, fmt, codes, scales, stream);
  const QuantKernel k = row ? ablation_pick<true>(fmt, hadamard != 0, stochastic != 0)
                            : ablation_pick<false>(fmt, hadamard != 0, stochastic != 0);
  return quant_launch_k(k, x, rows, cols, row, !row, fmt, codes, scales, fmt, codes, scales,
                        sign_mask, seed, stream);
}
