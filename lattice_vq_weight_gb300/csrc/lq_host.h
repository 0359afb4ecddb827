// Host-side helpers shared by the liblq entry points: argument checks, launch
// error mapping and grid sizing.  Internal to the library.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include "lq.h"

namespace lq {

// NVTX range around an entry point (seen by profilers; a no-op otherwise).
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};
#define LQ_NVTX_RANGE(name) ::lq::NvtxRange lq_nvtx_range_(name)

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

inline bool valid_lattice(int l) { return l == LQ_E8 || l == LQ_D4 || l == LQ_A2 || l == LQ_Z1; }

// Checks shared by quantize, dequantize and gemv: lattice, tile, shape.
inline lq_status validate_common(int lattice, int64_t rows, int64_t cols, int tile) {
  if (!valid_lattice(lattice)) return LQ_ERR_ARG;
  if (tile != 128 && tile != 256 && tile != 512 && tile != 1024 && tile != 2048) return LQ_ERR_UNSUPPORTED;
  if (rows < 0 || cols <= 0) return LQ_ERR_SHAPE;
  if (cols % tile != 0) return LQ_ERR_SHAPE;
  if (cols > (int64_t(1) << 20)) return LQ_ERR_SHAPE;
  if (rows > 0 && rows > (int64_t(1) << 40) / cols) return LQ_ERR_SHAPE;
  return LQ_OK;
}

// Map the last launch error (if any) to LQ_ERR_CUDA without clearing sticky errors twice.
inline lq_status check_launch() {
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? LQ_OK : LQ_ERR_CUDA;
}

inline int device_sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return sms;
}

template <typename K>
inline int occupancy_per_sm(K kernel, int threads, size_t smem = 0) {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, smem) != cudaSuccess) {
    cudaGetLastError();
    return 1;
  }
  return n > 0 ? n : 1;
}

// Persistent grid: at most one wave of resident CTAs, no more CTAs than the
// work needs.  When possible the total warp count is made a multiple of
// `warp_modulus` (so every warp keeps visiting the same column chunk), as long
// as that costs at most 1/16 of the resident CTAs.
inline int persistent_grid(int64_t units, int warps_per_cta, int warp_modulus, int per_sm) {
  const int sms = device_sm_count();
  if (sms <= 0) return 0;
  const int64_t resident = (int64_t)sms * per_sm;
  const int64_t needed = (units + warps_per_cta - 1) / warps_per_cta;
  int64_t g = needed < resident ? needed : resident;
  if (g == resident && warp_modulus > 1) {
    int64_t h = g;
    while (h > 0 && ((h * warps_per_cta) % warp_modulus) != 0) --h;
    if (h > 0 && h * 16 >= g * 15) g = h;
  }
  return (int)(g > 0 ? g : 1);
}

}  // namespace lq
