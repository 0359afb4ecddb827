// Instantiations of the decode attention over caches quantized with the
// subtractive Voronoi dither (HyperQuant page, "Key algorithmic ingredients"),
// in their own translation unit so that the build compiles them in parallel.
#include "lq_kv_kernel.cuh"

namespace lq {
namespace kv {

lq_status launch_partial_dithered(const AttnArgs& a, int lattice, int group, bool h, unsigned grid, cudaStream_t s) {
  switch (lattice) {
    case LQ_E8: return launch_partial_groups<LQ_E8, 0>(a, group, h, grid, s);
    case LQ_D4: return launch_partial_groups<LQ_D4, 0>(a, group, h, grid, s);
    case LQ_A2: return launch_partial_groups<LQ_A2, 0>(a, group, h, grid, s);
    default:    return launch_partial_groups<LQ_Z1, 0>(a, group, h, grid, s);
  }
}

}  // namespace kv
}  // namespace lq
