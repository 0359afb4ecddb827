// Activation side of the products computed from the codes, shared by the
// int8-code GEMV and the Rice-stream GEMV: the per-tile rotation of x into fp16
// (times a power of two per (row, tile)), the conversion of int8 codes to exact
// fp16 values and the m16n8k16 tensor-core step.  Internal.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "lq_device.cuh"
#include "lq_host.h"

namespace lq {

constexpr int kGemvMaxMats = LQ_GEMV_MAX_GROUP;

struct RotateArgs {
  const void* x;
  const int8_t* signs[kGemvMaxMats];
  float* y[kGemvMaxMats];
  int64_t y_elems[kGemvMaxMats];
  int n_mats;
  int64_t cols;
  int batch, tile, tiles_per_row;
  float post_scale;    // 1 / (2 sqrt(T))
  int a2;              // multiply odd coordinates by sqrt(3)
  __half* xh;          // [n_mats x batch x cols]: x~ times 2^e[row, tile], fp16
  float* xs;           // [n_mats x batch x tiles] = 2^-e
  int32_t* status;
};

// One thread per E consecutive columns of one activation row (E = 16 for
// tiles up to 512 columns, T/32 above): the tile spans T/E consecutive lanes,
// so the transform is log2(E) register stages plus log2(T/E) shuffle stages --
// a short dependent chain, since this kernel sits in front of every GEMV.
template <bool BF16, int E>
__global__ void __launch_bounds__(256) rotate_activation_kernel(RotateArgs a) {
  // launched early (programmatic dependent launch) behind the preceding
  // product, whose results x may be: wait for that grid first.  Then the
  // product that follows may start streaming codes (everything before this
  // launch is complete by now); it waits for this grid's results
  // (griddepcontrol.wait) before reading them
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  const int lane = threadIdx.x & 31;
  const int64_t gtid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t nthreads = (int64_t)gridDim.x * blockDim.x;
  for (int m = 0; m < a.n_mats; ++m)
    for (int64_t i = gtid; i < a.y_elems[m]; i += nthreads) a.y[m][i] = 0.f;

  // thread -> (matrix, activation row, E-column group); rows of x~ are
  // stored matrix-major: x~ row mb = m * batch + b
  const int64_t per_row = a.cols / E;
  const int64_t work = (int64_t)a.n_mats * a.batch * per_row;
  const int lpt = a.tile / E;                            // lanes per tile (<= 32)
  // every lane of a warp takes part in the shuffles; lanes past the end work on zeros
  const bool active = gtid < work;
  const int64_t mb = active ? gtid / per_row : 0;
  const int64_t col0 = active ? (gtid - mb * per_row) * E : 0;
  const int m = (int)(mb / a.batch);
  const int64_t b = mb - (int64_t)m * a.batch;
  float v[E];
  if (active) {
    const int8_t* sg = a.signs[m] + col0;
    if constexpr (BF16) load_bf16_signed<E>(reinterpret_cast<const __nv_bfloat16*>(a.x) + b * a.cols + col0, sg, v);
    else load_f32_signed<E>(reinterpret_cast<const float*>(a.x) + b * a.cols + col0, sg, v);
  } else {
#pragma unroll
    for (int c = 0; c < E; ++c) v[c] = 0.f;
  }
  fwht_tile<E>(v, lpt, lane);
  const float sc = a.post_scale;
  const float sc_odd = a.a2 ? sc * 1.7320508075688772f : sc;
  float mx = 0.f;
#pragma unroll
  for (int c = 0; c < E; ++c) {
    v[c] *= (c & 1) ? sc_odd : sc;
    mx = fmaxf(mx, fabsf(v[c]));
  }
  for (int m = 1; m < lpt; m <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, m));
  float f = 1.f;
  bool bad = false;
  if (!isfinite(mx)) {
    bad = active;
  } else if (mx > 0.f) {
    const int Ex = (int)((__float_as_uint(mx) >> 23) & 0xFFu) - 126;  // mx in [2^(Ex-1), 2^Ex)
    const int ex = max(-126, min(127, 15 - Ex));
    f = __uint_as_float((uint32_t)(ex + 127) << 23);
  }
  if (active) {
    uint4* dh = reinterpret_cast<uint4*>(a.xh + mb * a.cols + col0);
#pragma unroll
    for (int q = 0; q < E / 8; ++q) {
      uint32_t hw[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const __half2 h = __floats2half2_rn(v[8 * q + 2 * j] * f, v[8 * q + 2 * j + 1] * f);
        hw[j] = *reinterpret_cast<const uint32_t*>(&h);
      }
      dh[q] = make_uint4(hw[0], hw[1], hw[2], hw[3]);
    }
    if ((lane & (lpt - 1)) == 0) a.xs[mb * a.tiles_per_row + col0 / a.tile] = 1.0f / f;
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0) raise_flag(a.status, LQ_DEV_NONFINITE);
}

// int8 codes (4 per word) -> two f16x2 words holding the exact values: the
// offset byte u = c + 128 under the fp16 exponent of 1024 (bits 0x6400 | u are
// 1024 + u), minus 1152 -- the magic-number conversion of Kim et al. 2022
// ("Who Says Elephants Can't Run").
__device__ __forceinline__ void codes_to_f16x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ 0x80808080u;  // c + 128 as unsigned bytes
  const uint32_t l = __byte_perm(u, 0x64646464u, 0x4140);
  const uint32_t h = __byte_perm(u, 0x64646464u, 0x4342);
  const __half2 off = __half2half2(__ushort_as_half((unsigned short)0x6480));  // 1152
  const __half2 lv = __hsub2(*reinterpret_cast<const __half2*>(&l), off);
  const __half2 hv = __hsub2(*reinterpret_cast<const __half2*>(&h), off);
  lo = *reinterpret_cast<const uint32_t*>(&lv);
  hi = *reinterpret_cast<const uint32_t*>(&hv);
}

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

template <bool BF16, int E>
inline cudaError_t launch_rotation_pdl(const RotateArgs& r, unsigned grid, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(256);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, rotate_activation_kernel<BF16, E>, r);
}

// One thread per E activation columns of every (matrix, row) (a few CTAs),
// which also zero y; the small grid leaves the SMs free for the product
// launched right after it.  Both launches are programmatic dependent
// launches: the rotation's launch overlaps the end of the product before it,
// and the product's the rotation.  (A product that signals its dependents at
// its start, so that the next rotation waits on the SMs, measured 1 to 9 %
// slower at batch 4 and 16.)
inline lq_status launch_rotation(const RotateArgs& r, int xdtype, int64_t max_y, cudaStream_t s) {
  const int E = act_elems_for_tile(r.tile);
  const int64_t rot_threads = (int64_t)r.n_mats * r.batch * (r.cols / E);
  int64_t rgrid = (rot_threads + 255) / 256;
  const int64_t zgrid = (max_y + 256 * 16 - 1) / (256 * 16);
  if (rgrid < zgrid) rgrid = zgrid;
  if (rgrid < 1) rgrid = 1;
  const bool bf = (xdtype == LQ_BF16);
  const unsigned g = (unsigned)rgrid;
  cudaError_t e;
  if (E == 16) e = bf ? launch_rotation_pdl<true, 16>(r, g, s) : launch_rotation_pdl<false, 16>(r, g, s);
  else if (E == 32) e = bf ? launch_rotation_pdl<true, 32>(r, g, s) : launch_rotation_pdl<false, 32>(r, g, s);
  else e = bf ? launch_rotation_pdl<true, 64>(r, g, s) : launch_rotation_pdl<false, 64>(r, g, s);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return LQ_ERR_CUDA;
  }
  return LQ_OK;
}

}  // namespace lq
