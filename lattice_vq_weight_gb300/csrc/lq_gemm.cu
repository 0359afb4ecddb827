// Prefill GEMM from E8 codes (tcgen05).  Placeholder until the kernel lands.
#include <cstddef>
#include <cstdint>

#include "lq.h"

extern "C" size_t lq_gemm_workspace_size(int64_t M, int64_t K) {
  if (M <= 0 || K <= 0) return 0;
  return (size_t)M * (size_t)K * 2 + (size_t)M * 4 + 512;
}

extern "C" lq_status lq_gemm(int lattice, const int8_t* codes_dev, const float* scales_dev,
                             const int8_t* signs_dev, int64_t N, int64_t K, int tile,
                             const uint16_t* X_dev, int64_t M, float* Y_dev, void* workspace_dev,
                             int32_t* dev_status_dev, void* stream) {
  (void)lattice; (void)codes_dev; (void)scales_dev; (void)signs_dev; (void)N; (void)K; (void)tile;
  (void)X_dev; (void)M; (void)Y_dev; (void)workspace_dev; (void)dev_status_dev; (void)stream;
  return LQ_ERR_UNSUPPORTED;
}
