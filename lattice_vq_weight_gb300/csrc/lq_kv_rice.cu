// Instantiations of the decode attention over Rice-coded K and V caches
// (HyperQuant page, KV-cache storage table: Rice bitstream + fp16 norms).
// The fully unrolled two-symbol decoders of K and V make each instantiation
// long to compile, so this file is compiled into eight objects, one per
// lattice and norm format (LQ_KV_RICE_PART = 0..7: lattice E8, D4, A2, Z1 =
// part / 2, fp16 norms = part % 2), which the build compiles in parallel.
#include "lq_kv_kernel.cuh"

#ifndef LQ_KV_RICE_PART
#error "compile with -DLQ_KV_RICE_PART=0..7 (one object per lattice and norm format)"
#endif

namespace lq {
namespace kv {

template <int RLAT, bool H>
lq_status launch_partial_rice_lh(const AttnArgs& a, int group, unsigned grid, cudaStream_t s) {
  switch (group) {
    case 1: return launch_partial_g<1, H, 0, RLAT>(a, grid, s);
    case 2: return launch_partial_g<2, H, 0, RLAT>(a, grid, s);
    case 4: return launch_partial_g<4, H, 0, RLAT>(a, grid, s);
    default: return launch_partial_g<8, H, 0, RLAT>(a, grid, s);
  }
}

namespace {
constexpr int kPartLattices[4] = {LQ_E8, LQ_D4, LQ_A2, LQ_Z1};
}  // namespace

template lq_status launch_partial_rice_lh<kPartLattices[LQ_KV_RICE_PART / 2], (LQ_KV_RICE_PART % 2) != 0>(
    const AttnArgs&, int, unsigned, cudaStream_t);

}  // namespace kv
}  // namespace lq
