// Small host-only entry points of liblq: status strings, version, tile rule.
#include <cstdint>

#include "lq.h"

extern "C" const char* lq_status_string(int status) {
  switch (status) {
    case LQ_OK: return "ok";
    case LQ_ERR_ARG: return "invalid argument (null, misaligned pointer or bad enum)";
    case LQ_ERR_SHAPE: return "invalid or unsupported shape";
    case LQ_ERR_DTYPE: return "unsupported element type";
    case LQ_ERR_CUDA: return "CUDA runtime error";
    case LQ_ERR_UNSUPPORTED: return "not supported by this library";
    default: return "unknown status";
  }
}

extern "C" int lq_version(void) { return 100; }

// HyperQuant page, "Hadamard block size": the largest size in
// {256, 512, 1024, 2048} that is <= the request and divides in_features.
extern "C" int lq_pick_tile(int64_t cols, int requested) {
  static const int kSizes[4] = {256, 512, 1024, 2048};
  int best = 0;
  if (cols <= 0) return 0;
  for (int i = 0; i < 4; ++i)
    if (kSizes[i] <= requested && cols % kSizes[i] == 0) best = kSizes[i];
  return best;
}
