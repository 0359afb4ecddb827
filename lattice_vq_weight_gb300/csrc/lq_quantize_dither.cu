// Instantiations of the quantize kernel with the subtractive Voronoi dither
// (HyperQuant page, "Key algorithmic ingredients": a subtractive dither keeps
// the KV cache's inner products unbiased), float32 or float16 tile scales, in
// their own translation unit so that the build compiles them in parallel.
#include "lq_quantize_kernel.cuh"

namespace lq {

namespace {

template <int LAT>
lq_status dithered_for(QuantArgs& a, bool bf16, int sf, cudaStream_t st) {
  if (sf == LQ_SCALE_TILE_F16)
    return bf16 ? launch_quantize_walk<LAT, true, LQ_SCALE_TILE_F16, true>(a, st)
                : launch_quantize_walk<LAT, false, LQ_SCALE_TILE_F16, true>(a, st);
  return bf16 ? launch_quantize_walk<LAT, true, LQ_SCALE_TILE_F32, true>(a, st)
              : launch_quantize_walk<LAT, false, LQ_SCALE_TILE_F32, true>(a, st);
}

}  // namespace

lq_status launch_quantize_dithered(QuantArgs& a, int lattice, bool bf16, int sf, cudaStream_t st) {
  if (sf != LQ_SCALE_TILE_F32 && sf != LQ_SCALE_TILE_F16) return LQ_ERR_ARG;
  switch (lattice) {
    case LQ_E8: return dithered_for<LQ_E8>(a, bf16, sf, st);
    case LQ_D4: return dithered_for<LQ_D4>(a, bf16, sf, st);
    case LQ_A2: return dithered_for<LQ_A2>(a, bf16, sf, st);
    default:    return dithered_for<LQ_Z1>(a, bf16, sf, st);
  }
}

}  // namespace lq
