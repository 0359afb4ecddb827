// Instantiations of the quantize kernel for the 16-bit scale formats
// (LQ_SCALE_ROW_BF16: one bf16 scale per row, HyperQuant page, mma="int8"
// paragraph; LQ_SCALE_TILE_F16: fp16 tile scales, the page's KV-cache norms),
// in their own translation unit so that the build compiles them in parallel
// with the float32 ones.
#include "lq_quantize_kernel.cuh"

namespace lq {

namespace {

template <int LAT>
lq_status scaled16_for(QuantArgs& a, bool bf16, int sf, cudaStream_t st) {
  if (sf == LQ_SCALE_ROW_BF16)
    return bf16 ? launch_quantize_walk<LAT, true, LQ_SCALE_ROW_BF16>(a, st)
                : launch_quantize_walk<LAT, false, LQ_SCALE_ROW_BF16>(a, st);
  return bf16 ? launch_quantize_walk<LAT, true, LQ_SCALE_TILE_F16>(a, st)
              : launch_quantize_walk<LAT, false, LQ_SCALE_TILE_F16>(a, st);
}

}  // namespace

lq_status launch_quantize_scaled16(QuantArgs& a, int lattice, bool bf16, int sf, cudaStream_t st) {
  if (sf != LQ_SCALE_ROW_BF16 && sf != LQ_SCALE_TILE_F16) return LQ_ERR_ARG;
  switch (lattice) {
    case LQ_E8: return scaled16_for<LQ_E8>(a, bf16, sf, st);
    case LQ_D4: return scaled16_for<LQ_D4>(a, bf16, sf, st);
    case LQ_A2: return scaled16_for<LQ_A2>(a, bf16, sf, st);
    default:    return scaled16_for<LQ_Z1>(a, bf16, sf, st);
  }
}

}  // namespace lq
