// Quantize (tile RHT + lattice nearest point), dequantize and sign generation.
//
// HyperQuant page, "Key algorithmic ingredients": per-tile randomized Hadamard
// transform, then optimal low-dimensional lattice VQ (E8, D4, A2, Z1).
// Conway & Sloane, Sphere Packings, Lattices and Groups, ch. 20: nearest-point
// decoders.
//
// Work decomposition: a warp unit is one 2048-column chunk of one row; lane l
// owns columns [64 l, 64 l + 64) of the chunk (see lq_device.cuh).  Units are
// visited by a persistent grid of 8-warp CTAs, and each warp loads the raw
// data of its next unit before working on the current one.
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "lq_device.cuh"
#include "lq_host.h"

namespace lq {

// ------------------------------------------------------------------ signs
// SplitMix64 (Steele, Lea & Flood 2014): output k mixes seed + (k+1) * golden
// gamma through two xor-shift-multiply rounds; the sign is the top bit.
__global__ void make_signs_kernel(uint64_t seed, int64_t n, int8_t* signs) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  uint64_t z = seed + (uint64_t)(i + 1) * 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  z ^= z >> 31;
  signs[i] = (z >> 63) ? (int8_t)-1 : (int8_t)1;
}

// ------------------------------------------------------------------ loading
// Raw storage of one lane's 64 input columns.
template <bool BF16> struct LaneRaw;
template <> struct LaneRaw<true> { uint4 v[8]; };    // 64 bf16
template <> struct LaneRaw<false> { uint4 v[16]; };  // 64 fp32

template <bool BF16>
__device__ __forceinline__ void load_raw(LaneRaw<BF16>& r, const void* base) {
  const uint4* p = reinterpret_cast<const uint4*>(base);
#pragma unroll
  for (int i = 0; i < (BF16 ? 8 : 16); ++i) r.v[i] = __ldg(p + i);
}

// Sign masks of the lane's 64 columns.  bf16: one word per column pair with
// bits 15 and 31 set where the sign is -1.  fp32: the 64 sign bits in 2 words.
template <bool BF16> struct LaneSigns;
template <> struct LaneSigns<true> { uint32_t m[32]; };
template <> struct LaneSigns<false> { uint32_t bits[2]; };

template <bool BF16>
__device__ __forceinline__ void load_signs(LaneSigns<BF16>& s, const int8_t* signs_col0) {
  const uint4* p = reinterpret_cast<const uint4*>(signs_col0);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint4 v = __ldg(p + q);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      // word w[h] holds the signs of columns 16q + 4h .. 16q + 4h + 3
      if constexpr (BF16) {
        s.m[8 * q + 2 * h] = __byte_perm(w[h], 0u, 0x1404) & 0x80008000u;
        s.m[8 * q + 2 * h + 1] = __byte_perm(w[h], 0u, 0x3424) & 0x80008000u;
      } else {
        // bit 7 of each byte -> one bit per column
        uint32_t b = 0;
#pragma unroll
        for (int c = 0; c < 4; ++c) b |= ((w[h] >> (8 * c + 7)) & 1u) << c;
        const int col = 16 * q + 4 * h;
        s.bits[col >> 5] |= b << (col & 31);
      }
    }
  }
}

// Unpack raw input to fp32 pairs with the signs applied (exact).
template <bool BF16>
__device__ __forceinline__ void unpack_signed(const LaneRaw<BF16>& r, const LaneSigns<BF16>& s,
                                              float2 (&p)[32]) {
  if constexpr (BF16) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t w[4] = {r.v[i].x, r.v[i].y, r.v[i].z, r.v[i].w};
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const uint32_t x = w[h] ^ s.m[4 * i + h];
        p[4 * i + h] = make_float2(__uint_as_float(x << 16), __uint_as_float(x & 0xFFFF0000u));
      }
    }
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const uint32_t w[4] = {r.v[i].x, r.v[i].y, r.v[i].z, r.v[i].w};
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const int col = 4 * i + h;
        const uint32_t sb = ((s.bits[col >> 5] >> (col & 31)) & 1u) << 31;
        const float v = __uint_as_float(w[h] ^ sb);
        if (h & 1) p[col >> 1].y = v; else p[col >> 1].x = v;
      }
    }
  }
}

// ------------------------------------------------------------------ quantize
struct QuantArgs {
  const void* W;
  int64_t rows, cols, ldw;
  int tile, lanes_per_tile, tiles_per_row, chunks_per_row;
  float beta, sqrt_tile;
  const int8_t* signs;
  int8_t* codes;
  float* scales;
  int32_t* status;
  int64_t units;
};

template <int LAT, bool BF16>
__global__ void __launch_bounds__(256, 1) quantize_kernel(QuantArgs a) {
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  constexpr int kElemBytes = BF16 ? 2 : 4;

  LaneSigns<BF16> sg;
  int cached_chunk = -1;
  bool range = false, nonfinite = false;

  int64_t u = warp0;
  LaneRaw<BF16> raw, nxt;
  auto lane_col = [&](int64_t unit) -> int64_t {
    return (unit % a.chunks_per_row) * kChunkCols + (int64_t)lane * kLaneElems;
  };
  auto lane_ptr = [&](int64_t unit) -> const char* {
    const int64_t row = unit / a.chunks_per_row;
    return reinterpret_cast<const char*>(a.W) + (row * a.ldw + lane_col(unit)) * kElemBytes;
  };
  if (u < a.units && lane_col(u) < a.cols) load_raw<BF16>(raw, lane_ptr(u));

  for (; u < a.units; u += nwarps) {
    const int64_t un = u + nwarps;
    if (un < a.units && lane_col(un) < a.cols) load_raw<BF16>(nxt, lane_ptr(un));

    const int chunk = (int)(u % a.chunks_per_row);
    const int64_t row = u / a.chunks_per_row;
    const int64_t col0 = (int64_t)chunk * kChunkCols + (int64_t)lane * kLaneElems;
    const bool active = col0 < a.cols;
    if (chunk != cached_chunk) {
      if constexpr (!BF16) { sg.bits[0] = 0; sg.bits[1] = 0; }
      if (active) load_signs<BF16>(sg, a.signs + col0);
      cached_chunk = chunk;
    }

    float2 p[32];
    unpack_signed<BF16>(raw, sg, p);
    fwht64_local(p);
    fwht_cross_lanes(p, a.lanes_per_tile, lane);

    // U = sum u^2 over the tile; s = beta sqrt(U) / T; y = u / (s sqrt(T))
    float2 acc = make_float2(0.f, 0.f);
#pragma unroll
    for (int j = 0; j < 32; ++j) acc = fma2(p[j], p[j], acc);
    const float U = tile_lane_sum(acc.x + acc.y, a.lanes_per_tile);
    const bool finite = isfinite(U);
    float s = a.beta * sqrtf(U) * (1.0f / (float)a.tile);
    if (!finite) s = 0.f;
    const float k = (s > 0.f) ? 1.0f / (s * a.sqrt_tile) : 0.f;
    const float2 k2 = make_float2(k, k);
#pragma unroll
    for (int j = 0; j < 32; ++j) p[j] = mul2(p[j], k2);

    uint32_t w[16];
    bool r = false;
    decode_lane<LAT>(p, w, r);

    if (active) {
      range |= r;
      nonfinite |= !finite;
      uint4* dst = reinterpret_cast<uint4*>(a.codes + row * a.cols + col0);
#pragma unroll
      for (int q = 0; q < 4; ++q) dst[q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
      if ((lane & (a.lanes_per_tile - 1)) == 0)
        a.scales[row * a.tiles_per_row + col0 / a.tile] = s;
    }
    raw = nxt;
  }
  if (__any_sync(0xffffffffu, range) && lane == 0) raise_flag(a.status, LQ_DEV_RANGE);
  if (__any_sync(0xffffffffu, nonfinite) && lane == 0) raise_flag(a.status, LQ_DEV_NONFINITE);
}

// ------------------------------------------------------------------ dequantize
struct DequantArgs {
  const int8_t* codes;
  const float* scales;
  const int8_t* signs;
  int64_t rows, cols;
  int tile, lanes_per_tile, tiles_per_row, chunks_per_row;
  float inv_2sqrt_tile;
  void* out;
  int64_t units;
};

// W^ = D H (s p) / sqrt(T): codes -> (A2: odd coordinates x sqrt3) -> FWHT
// (integer-exact for the doubled codes) -> x s / (2 sqrt T) -> signs.
template <int LAT, bool OUT_BF16>
__global__ void __launch_bounds__(256, 1) dequantize_kernel(DequantArgs a) {
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t u = warp0; u < a.units; u += nwarps) {
    const int chunk = (int)(u % a.chunks_per_row);
    const int64_t row = u / a.chunks_per_row;
    const int64_t col0 = (int64_t)chunk * kChunkCols + (int64_t)lane * kLaneElems;
    const bool active = col0 < a.cols;
    float2 p[32];
    uint4 cw[4] = {};
    uint4 sw[4] = {};
    if (active) {
      const uint4* src = reinterpret_cast<const uint4*>(a.codes + row * a.cols + col0);
      const uint4* ssrc = reinterpret_cast<const uint4*>(a.signs + col0);
#pragma unroll
      for (int q = 0; q < 4; ++q) { cw[q] = __ldg(src + q); sw[q] = __ldg(ssrc + q); }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t w[4] = {cw[q].x, cw[q].y, cw[q].z, cw[q].w};
#pragma unroll
      for (int h = 0; h < 4; ++h) {
#pragma unroll
        for (int c = 0; c < 4; c += 2) {
          const float v0 = (float)(int8_t)(w[h] >> (8 * c));
          float v1 = (float)(int8_t)(w[h] >> (8 * c + 8));
          if constexpr (LAT == LQ_A2) v1 *= 1.7320508075688772f;
          p[(16 * q + 4 * h + c) >> 1] = make_float2(v0, v1);
        }
      }
    }
    fwht64_local(p);
    fwht_cross_lanes(p, a.lanes_per_tile, lane);
    if (!active) continue;
    const float f = a.scales[row * a.tiles_per_row + col0 / a.tile] * a.inv_2sqrt_tile;
    const float2 f2 = make_float2(f, f);
    float2 o[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) o[j] = mul2(p[j], f2);
    // apply signs: column c has sign byte c of the 64-byte sign run
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t w[4] = {sw[q].x, sw[q].y, sw[q].z, sw[q].w};
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const int col = 16 * q + 4 * h;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint32_t sbit = ((w[h] >> (8 * c + 7)) & 1u) << 31;
          float& v = ((col + c) & 1) ? o[(col + c) >> 1].y : o[(col + c) >> 1].x;
          v = __uint_as_float(__float_as_uint(v) ^ sbit);
        }
      }
    }
    if constexpr (OUT_BF16) {
      uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(a.out) + row * a.cols + col0);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        uint32_t w4[4];
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const __nv_bfloat162 b = __floats2bfloat162_rn(o[4 * q + h].x, o[4 * q + h].y);
          w4[h] = *reinterpret_cast<const uint32_t*>(&b);
        }
        dst[q] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
      }
    } else {
      float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(a.out) + row * a.cols + col0);
#pragma unroll
      for (int q = 0; q < 16; ++q)
        dst[q] = make_float4(o[2 * q].x, o[2 * q].y, o[2 * q + 1].x, o[2 * q + 1].y);
    }
  }
}

}  // namespace lq

using namespace lq;

// ------------------------------------------------------------------ host side
extern "C" lq_status lq_make_signs(uint64_t seed, int64_t cols, int8_t* signs_dev, void* stream) {
  if (cols < 0) return LQ_ERR_SHAPE;
  if (cols == 0) return LQ_OK;
  if (signs_dev == nullptr) return LQ_ERR_ARG;
  const int threads = 256;
  const int64_t blocks = (cols + threads - 1) / threads;
  make_signs_kernel<<<(unsigned)blocks, threads, 0, (cudaStream_t)stream>>>(seed, cols, signs_dev);
  return check_launch();
}

template <int LAT, bool BF16>
static lq_status launch_quantize(const QuantArgs& a, cudaStream_t st) {
  static int per_sm = 0;
  if (per_sm == 0) per_sm = occupancy_per_sm(quantize_kernel<LAT, BF16>, 256);
  const int grid = persistent_grid(a.units, 8, a.chunks_per_row, per_sm);
  if (grid <= 0) return LQ_ERR_CUDA;
  quantize_kernel<LAT, BF16><<<grid, 256, 0, st>>>(a);
  return check_launch();
}

extern "C" lq_status lq_quantize(int lattice, const void* W_dev, int wdtype, int64_t rows, int64_t cols,
                                 int64_t ldw, int tile, uint64_t seed, float beta, int8_t* codes_dev,
                                 float* scales_dev, int8_t* signs_dev, int32_t* dev_status_dev,
                                 void* stream) {
  lq_status st = validate_common(lattice, rows, cols, tile);
  if (st != LQ_OK) return st;
  if (wdtype != LQ_BF16 && wdtype != LQ_F32) return LQ_ERR_DTYPE;
  if (!(beta > 0.f) || !(beta < 1e30f)) return LQ_ERR_ARG;
  if (ldw < cols) return LQ_ERR_SHAPE;
  const int esize = (wdtype == LQ_BF16) ? 2 : 4;
  if (((ldw * esize) & 15) != 0) return LQ_ERR_SHAPE;
  if (signs_dev == nullptr || !aligned16(signs_dev)) return LQ_ERR_ARG;
  if (rows > 0) {
    if (W_dev == nullptr || codes_dev == nullptr || scales_dev == nullptr) return LQ_ERR_ARG;
    if (!aligned16(W_dev) || !aligned16(codes_dev) || !aligned4(scales_dev) ||
        (dev_status_dev != nullptr && !aligned4(dev_status_dev)))
      return LQ_ERR_ARG;
  }
  cudaStream_t s = (cudaStream_t)stream;
  st = lq_make_signs(seed, cols, signs_dev, stream);
  if (st != LQ_OK) return st;
  if (rows == 0) return LQ_OK;

  QuantArgs a;
  a.W = W_dev; a.rows = rows; a.cols = cols; a.ldw = ldw;
  a.tile = tile; a.lanes_per_tile = tile / kLaneElems; a.tiles_per_row = (int)(cols / tile);
  a.chunks_per_row = (int)((cols + kChunkCols - 1) / kChunkCols);
  a.beta = beta; a.sqrt_tile = sqrtf((float)tile);
  a.signs = signs_dev; a.codes = codes_dev; a.scales = scales_dev; a.status = dev_status_dev;
  a.units = rows * a.chunks_per_row;
  const bool bf = (wdtype == LQ_BF16);
  switch (lattice) {
    case LQ_E8: return bf ? launch_quantize<LQ_E8, true>(a, s) : launch_quantize<LQ_E8, false>(a, s);
    case LQ_D4: return bf ? launch_quantize<LQ_D4, true>(a, s) : launch_quantize<LQ_D4, false>(a, s);
    case LQ_A2: return bf ? launch_quantize<LQ_A2, true>(a, s) : launch_quantize<LQ_A2, false>(a, s);
    default:    return bf ? launch_quantize<LQ_Z1, true>(a, s) : launch_quantize<LQ_Z1, false>(a, s);
  }
}

template <int LAT, bool OB>
static lq_status launch_dequant(const DequantArgs& a, cudaStream_t st) {
  static int per_sm = 0;
  if (per_sm == 0) per_sm = occupancy_per_sm(dequantize_kernel<LAT, OB>, 256);
  const int grid = persistent_grid(a.units, 8, 1, per_sm);
  if (grid <= 0) return LQ_ERR_CUDA;
  dequantize_kernel<LAT, OB><<<grid, 256, 0, st>>>(a);
  return check_launch();
}

extern "C" lq_status lq_dequantize(int lattice, const int8_t* codes_dev, const float* scales_dev,
                                   const int8_t* signs_dev, int64_t rows, int64_t cols, int tile,
                                   void* What_dev, int out_dtype, void* stream) {
  lq_status st = validate_common(lattice, rows, cols, tile);
  if (st != LQ_OK) return st;
  if (out_dtype != LQ_BF16 && out_dtype != LQ_F32) return LQ_ERR_DTYPE;
  if (rows == 0) return LQ_OK;
  if (codes_dev == nullptr || scales_dev == nullptr || signs_dev == nullptr || What_dev == nullptr)
    return LQ_ERR_ARG;
  if (!aligned16(codes_dev) || !aligned16(signs_dev) || !aligned16(What_dev) || !aligned4(scales_dev))
    return LQ_ERR_ARG;
  DequantArgs a;
  a.codes = codes_dev; a.scales = scales_dev; a.signs = signs_dev; a.rows = rows; a.cols = cols;
  a.tile = tile; a.lanes_per_tile = tile / kLaneElems; a.tiles_per_row = (int)(cols / tile);
  a.chunks_per_row = (int)((cols + kChunkCols - 1) / kChunkCols);
  a.inv_2sqrt_tile = (float)(0.5 / sqrt((double)tile));
  a.out = What_dev;
  a.units = rows * a.chunks_per_row;
  const bool ob = (out_dtype == LQ_BF16);
  cudaStream_t s = (cudaStream_t)stream;
  switch (lattice) {
    case LQ_E8: return ob ? launch_dequant<LQ_E8, true>(a, s) : launch_dequant<LQ_E8, false>(a, s);
    case LQ_D4: return ob ? launch_dequant<LQ_D4, true>(a, s) : launch_dequant<LQ_D4, false>(a, s);
    case LQ_A2: return ob ? launch_dequant<LQ_A2, true>(a, s) : launch_dequant<LQ_A2, false>(a, s);
    default:    return ob ? launch_dequant<LQ_Z1, true>(a, s) : launch_dequant<LQ_Z1, false>(a, s);
  }
}
