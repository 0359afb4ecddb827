// Instantiations of the decode attention over Rice-coded K and V caches
// (HyperQuant page, KV-cache storage table: Rice bitstream + fp16 norms),
// in their own translation unit so that the build compiles them in parallel.
#include "lq_kv_kernel.cuh"

namespace lq {
namespace kv {

lq_status launch_partial_rice(const AttnArgs& a, int lattice, int group, bool h, unsigned grid, cudaStream_t s) {
  switch (lattice) {
    case LQ_E8: return launch_partial_groups<0, LQ_E8>(a, group, h, grid, s);
    case LQ_D4: return launch_partial_groups<0, LQ_D4>(a, group, h, grid, s);
    case LQ_A2: return launch_partial_groups<0, LQ_A2>(a, group, h, grid, s);
    default:    return launch_partial_groups<0, LQ_Z1>(a, group, h, grid, s);
  }
}

}  // namespace kv
}  // namespace lq
