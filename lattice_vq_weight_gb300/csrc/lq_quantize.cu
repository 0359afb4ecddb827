// Quantize entry points (tile RHT + lattice nearest point), dequantize and
// sign generation; the quantize kernel itself is in lq_quantize_kernel.cuh.
//
// HyperQuant page, "Key algorithmic ingredients": per-tile randomized Hadamard
// transform, then optimal low-dimensional lattice VQ (E8, D4, A2, Z1).
// Conway & Sloane, Sphere Packings, Lattices and Groups, ch. 20: nearest-point
// decoders.
//
// Work decomposition: a warp unit is one 2048-column chunk of one row; lane l
// loads columns [64 l, 64 l + 64) of the chunk (see lq_device.cuh).  Units are
// visited by a persistent grid of 4-warp CTAs, and each warp loads the raw
// data of its next unit before working on the current one.
#include "lq_quantize_kernel.cuh"

namespace lq {

struct SignsArgs {
  uint64_t seed[kQuantMaxMats];
  int64_t n[kQuantMaxMats];
  int8_t* out[kQuantMaxMats];
};

// ------------------------------------------------------------------ signs
// SplitMix64 (Steele, Lea & Flood 2014): output k mixes seed + (k+1) * golden
// gamma through two xor-shift-multiply rounds; the sign is the top bit.
// blockIdx.y selects the matrix of a group (each with its own seed).
__global__ void make_signs_kernel(SignsArgs a) {
  // the quantize kernel launched next may start now: it prefetches its input
  // and waits for these signs (griddepcontrol.wait) before reading them
  asm volatile("griddepcontrol.launch_dependents;");
  const int m = blockIdx.y;
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= a.n[m]) return;
  uint64_t z = a.seed[m] + (uint64_t)(i + 1) * 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  z ^= z >> 31;
  a.out[m][i] = (z >> 63) ? (int8_t)-1 : (int8_t)1;
}

// ------------------------------------------------------------------ row scales
// Per-row bf16 scale s_r = beta * RMS of the row (the tile Hadamards are
// orthonormal, so the RMS of the raw row is that of the rotated one), rounded
// to nearest-even.  One warp per row; 16-byte loads; per-lane partial sums of
// eight squares, then the warp sum.
struct RowScaleArgs {
  const void* W;
  int64_t rows, cols, ldw;
  float beta;
  uint16_t* out;
  int32_t* status;
};

constexpr int kRowScaleWarps = 8;

template <bool BF16>
__global__ void __launch_bounds__(kRowScaleWarps * 32) row_scale_kernel(RowScaleArgs a) {
  // the quantize kernel launched next may stage its input meanwhile
  asm volatile("griddepcontrol.launch_dependents;");
  const int64_t row = (int64_t)blockIdx.x * kRowScaleWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= a.rows) return;
  constexpr int kPer = BF16 ? 8 : 4;   // elements per 16-byte vector
  const uint4* src = reinterpret_cast<const uint4*>(reinterpret_cast<const char*>(a.W) +
                                                    row * a.ldw * (BF16 ? 2 : 4));
  const int64_t nvec = a.cols / kPer;
  float acc = 0.f;
  for (int64_t v = lane; v < nvec; v += 32) {
    const uint4 q = __ldg(src + v);
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
    float part = 0.f;
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      if constexpr (BF16) {
        const float lo = __uint_as_float(w[h] << 16), hi = __uint_as_float(w[h] & 0xFFFF0000u);
        part = fmaf(lo, lo, fmaf(hi, hi, part));
      } else {
        const float x = __uint_as_float(w[h]);
        part = fmaf(x, x, part);
      }
    }
    acc += part;
  }
  for (int o = 16; o; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (lane == 0) {
    float sc = a.beta * sqrtf(acc / (float)a.cols);
    if (!isfinite(sc)) {
      sc = 0.f;
      raise_flag(a.status, LQ_DEV_NONFINITE);
    }
    const __nv_bfloat16 b = __float2bfloat16_rn(sc);
    a.out[row] = *reinterpret_cast<const uint16_t*>(&b);
  }
}

// ------------------------------------------------------------------ dequantize
struct DequantArgs {
  const int8_t* codes;
  const void* scales;     // in format sfmt (LQ_SCALE_*)
  int sfmt;
  const int8_t* signs;
  int64_t rows, cols;
  int tile, lanes_per_tile, tiles_per_row, chunks_per_row;
  float inv_2sqrt_tile;
  void* out;
  int64_t units;
  int dither;             // subtract the subtractive dither of seed dither_seed (selects the DITHER kernel)
  uint64_t dither_seed;
};

// W^ = D H (s p) / sqrt(T): codes -> (A2: odd coordinates x sqrt3) -> FWHT
// (integer-exact for the doubled codes) -> x s / (2 sqrt T) -> signs; with a
// dither, p - u replaces p (2u in the doubled code units).
template <int LAT, bool OUT_BF16, bool DITHER>
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
    if (DITHER && active) {
#pragma unroll
      for (int gb = 0; gb < 8; ++gb) {
        float du[8];
        dither8<LAT>(a.dither_seed, (uint64_t)row * (uint64_t)a.cols + (uint64_t)(col0 + 8 * gb), du);
#pragma unroll
        for (int h = 0; h < 4; ++h)
          p[4 * gb + h] = sub2(p[4 * gb + h], make_float2(2.f * du[2 * h], 2.f * du[2 * h + 1]));
      }
    }
    fwht64_local(p);
    fwht_cross_lanes(p, a.lanes_per_tile, lane);
    if (!active) continue;
    const float f = load_scale(a.scales, a.sfmt, row, col0 / a.tile, a.tiles_per_row) * a.inv_2sqrt_tile;
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
namespace {

lq_status launch_signs(const SignsArgs& a, int n_mats, int64_t max_cols, cudaStream_t s) {
  if (max_cols <= 0) return LQ_OK;
  const int threads = 256;
  const int64_t blocks = (max_cols + threads - 1) / threads;
  make_signs_kernel<<<dim3((unsigned)blocks, (unsigned)n_mats), threads, 0, s>>>(a);
  return check_launch();
}


}  // namespace

extern "C" lq_status lq_make_signs(uint64_t seed, int64_t cols, int8_t* signs_dev, void* stream) {
  LQ_NVTX_RANGE("lq_make_signs");
  if (cols < 0) return LQ_ERR_SHAPE;
  if (cols == 0) return LQ_OK;
  if (signs_dev == nullptr) return LQ_ERR_ARG;
  SignsArgs a = {};
  a.seed[0] = seed;
  a.n[0] = cols;
  a.out[0] = signs_dev;
  return launch_signs(a, 1, cols, (cudaStream_t)stream);
}

template <int LAT, bool BF16>
static lq_status launch_quantize(QuantArgs& a, int sf, bool dither, cudaStream_t st) {
  if (dither) return launch_quantize_dithered(a, LAT, BF16, sf, st);
  if (sf != LQ_SCALE_TILE_F32) return launch_quantize_scaled16(a, LAT, BF16, sf, st);
  return launch_quantize_walk<LAT, BF16, LQ_SCALE_TILE_F32>(a, st);
}

namespace {

bool valid_scale_format(int f) {
  return f == LQ_SCALE_TILE_F32 || f == LQ_SCALE_ROW_BF16 || f == LQ_SCALE_TILE_F16;
}

// Checks of one matrix's arguments, in the order lq_quantize reports them.
lq_status validate_quantize(int lattice, const void* W_dev, int wdtype, int64_t rows, int64_t cols, int64_t ldw,
                            int tile, float beta, const int8_t* codes_dev, const void* scales_dev,
                            const int8_t* signs_dev, const int32_t* dev_status_dev, int sf = LQ_SCALE_TILE_F32) {
  lq_status st = validate_common(lattice, rows, cols, tile);
  if (st != LQ_OK) return st;
  if (wdtype != LQ_BF16 && wdtype != LQ_F32) return LQ_ERR_DTYPE;
  if (!valid_scale_format(sf)) return LQ_ERR_ARG;
  if (!(beta > 0.f) || !(beta < 1e30f)) return LQ_ERR_ARG;
  if (ldw < cols) return LQ_ERR_SHAPE;
  const int esize = (wdtype == LQ_BF16) ? 2 : 4;
  if (((ldw * esize) & 15) != 0) return LQ_ERR_SHAPE;
  if (signs_dev == nullptr || !aligned16(signs_dev)) return LQ_ERR_ARG;
  if (rows > 0) {
    if (W_dev == nullptr || codes_dev == nullptr || scales_dev == nullptr) return LQ_ERR_ARG;
    const uintptr_t salign = (sf == LQ_SCALE_TILE_F32) ? 3u : 1u;
    if (!aligned16(W_dev) || !aligned16(codes_dev) || (reinterpret_cast<uintptr_t>(scales_dev) & salign) != 0 ||
        (dev_status_dev != nullptr && !aligned4(dev_status_dev)))
      return LQ_ERR_ARG;
  }
  return LQ_OK;
}

// The quantize launch over n matrices (rows 0: skipped), after the signs
// launch when make_signs_too is set.
lq_status quantize_group(int lattice, int n, const void* const* W, int wdtype, const int64_t* rows,
                         const int64_t* cols, const int64_t* ldw, int tile, const uint64_t* seeds, float beta,
                         int8_t* const* codes, void* const* scales, int8_t* const* signs, int32_t* dev_status,
                         int sf, bool make_signs_too, cudaStream_t s, bool dither = false,
                         uint64_t dither_seed = 0) {
  SignsArgs sa = {};
  QuantArgs a = {};
  a.dither_seed = dither_seed;
  int64_t max_cols = 0, units = 0;
  int k = 0;
  const bool bf = (wdtype == LQ_BF16);
  for (int m = 0; m < n; ++m) {
    sa.seed[m] = seeds[m];
    sa.n[m] = cols[m];
    sa.out[m] = signs[m];
    if (cols[m] > max_cols) max_cols = cols[m];
    if (rows[m] == 0) continue;   // signs only
    // the input as 128-byte lines, one warp unit (2048 columns of a row) per copy
    if (!encode_row_lines_map(&a.maps[k], bf ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                              bf ? 2 : 4, W[m], rows[m], cols[m], ldw[m], bf ? 32 : 64))
      return LQ_ERR_CUDA;
    QuantMat& M = a.mat[k++];
    M.codes = codes[m]; M.scales = scales[m]; M.signs = signs[m];
    M.W = W[m]; M.ldw = ldw[m];
    M.rows = rows[m]; M.cols = cols[m];
    M.tiles_per_row = (int)(cols[m] / tile);
    M.chunks_per_row = (int)((cols[m] + kChunkCols - 1) / kChunkCols);
    M.row_groups = (rows[m] + kQuantWarps - 1) / kQuantWarps;
    M.cta_begin = units;
    units += M.row_groups * M.chunks_per_row;
  }
  if (units >= ((int64_t)1 << 40)) return LQ_ERR_SHAPE;
  if (make_signs_too) {
    const lq_status st = launch_signs(sa, n, max_cols, s);
    if (st != LQ_OK) return st;
  }
  if (k == 0) return LQ_OK;
  a.n_mats = k;
  a.tile = tile; a.tile_shift = __builtin_ctz((unsigned)tile);
  a.lanes_per_tile = tile / kLaneElems;
  a.beta = beta; a.sqrt_tile = sqrtf((float)tile); a.inv_tile = 1.0f / (float)tile;
  a.status = dev_status;
  a.cta_units = units;
  switch (lattice) {
    case LQ_E8: return bf ? launch_quantize<LQ_E8, true>(a, sf, dither, s) : launch_quantize<LQ_E8, false>(a, sf, dither, s);
    case LQ_D4: return bf ? launch_quantize<LQ_D4, true>(a, sf, dither, s) : launch_quantize<LQ_D4, false>(a, sf, dither, s);
    case LQ_A2: return bf ? launch_quantize<LQ_A2, true>(a, sf, dither, s) : launch_quantize<LQ_A2, false>(a, sf, dither, s);
    default:    return bf ? launch_quantize<LQ_Z1, true>(a, sf, dither, s) : launch_quantize<LQ_Z1, false>(a, sf, dither, s);
  }
}

// Rows per block of the per-row-scale quantize: the row-norm pass reads a
// block and the quantize pass reads it again, from L2 while the block stays
// well below its 129 MB.
constexpr int64_t kRowScaleBlockBytes = (int64_t)40 << 20;

}  // namespace

extern "C" lq_status lq_quantize(int lattice, const void* W_dev, int wdtype, int64_t rows, int64_t cols,
                                 int64_t ldw, int tile, uint64_t seed, float beta, int8_t* codes_dev,
                                 float* scales_dev, int8_t* signs_dev, int32_t* dev_status_dev,
                                 void* stream) {
  LQ_NVTX_RANGE("lq_quantize");
  const lq_status st = validate_quantize(lattice, W_dev, wdtype, rows, cols, ldw, tile, beta, codes_dev,
                                         scales_dev, signs_dev, dev_status_dev);
  if (st != LQ_OK) return st;
  void* sc = scales_dev;
  return quantize_group(lattice, 1, &W_dev, wdtype, &rows, &cols, &ldw, tile, &seed, beta, &codes_dev, &sc,
                        &signs_dev, dev_status_dev, LQ_SCALE_TILE_F32, true, (cudaStream_t)stream);
}

extern "C" lq_status lq_quantize_ex(int lattice, const void* W_dev, int wdtype, int64_t rows, int64_t cols,
                                    int64_t ldw, int tile, uint64_t seed, float beta, int scale_format,
                                    int8_t* codes_dev, void* scales_dev, int8_t* signs_dev,
                                    int32_t* dev_status_dev, void* stream) {
  LQ_NVTX_RANGE("lq_quantize_ex");
  lq_status st = validate_quantize(lattice, W_dev, wdtype, rows, cols, ldw, tile, beta, codes_dev, scales_dev,
                                   signs_dev, dev_status_dev, scale_format);
  if (st != LQ_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  if (scale_format != LQ_SCALE_ROW_BF16 || rows == 0)
    return quantize_group(lattice, 1, &W_dev, wdtype, &rows, &cols, &ldw, tile, &seed, beta, &codes_dev,
                          &scales_dev, &signs_dev, dev_status_dev, scale_format, true, s);
  st = lq_make_signs(seed, cols, signs_dev, stream);
  if (st != LQ_OK) return st;
  const int esize = (wdtype == LQ_BF16) ? 2 : 4;
  int64_t block = kRowScaleBlockBytes / (ldw * esize);
  if (block < 1) block = 1;
  for (int64_t r0 = 0; r0 < rows; r0 += block) {
    const int64_t nr = (rows - r0 < block) ? rows - r0 : block;
    RowScaleArgs ra;
    ra.W = reinterpret_cast<const char*>(W_dev) + r0 * ldw * esize;
    ra.rows = nr; ra.cols = cols; ra.ldw = ldw; ra.beta = beta;
    ra.out = reinterpret_cast<uint16_t*>(scales_dev) + r0;
    ra.status = dev_status_dev;
    const unsigned grid = (unsigned)((nr + kRowScaleWarps - 1) / kRowScaleWarps);
    if (wdtype == LQ_BF16) row_scale_kernel<true><<<grid, kRowScaleWarps * 32, 0, s>>>(ra);
    else row_scale_kernel<false><<<grid, kRowScaleWarps * 32, 0, s>>>(ra);
    st = check_launch();
    if (st != LQ_OK) return st;
    const void* Wb = ra.W;
    int8_t* cb = codes_dev + r0 * cols;
    void* sb = ra.out;
    st = quantize_group(lattice, 1, &Wb, wdtype, &nr, &cols, &ldw, tile, &seed, beta, &cb, &sb, &signs_dev,
                        dev_status_dev, LQ_SCALE_ROW_BF16, false, s);
    if (st != LQ_OK) return st;
  }
  return LQ_OK;
}

extern "C" lq_status lq_quantize_dithered(int lattice, const void* W_dev, int wdtype, int64_t rows, int64_t cols,
                                          int64_t ldw, int tile, uint64_t seed, uint64_t dither_seed, float beta,
                                          int scale_format, int8_t* codes_dev, void* scales_dev, int8_t* signs_dev,
                                          int32_t* dev_status_dev, void* stream) {
  LQ_NVTX_RANGE("lq_quantize_dithered");
  if (scale_format != LQ_SCALE_TILE_F32 && scale_format != LQ_SCALE_TILE_F16) return LQ_ERR_ARG;
  const lq_status st = validate_quantize(lattice, W_dev, wdtype, rows, cols, ldw, tile, beta, codes_dev,
                                         scales_dev, signs_dev, dev_status_dev, scale_format);
  if (st != LQ_OK) return st;
  return quantize_group(lattice, 1, &W_dev, wdtype, &rows, &cols, &ldw, tile, &seed, beta, &codes_dev,
                        &scales_dev, &signs_dev, dev_status_dev, scale_format, true, (cudaStream_t)stream, true,
                        dither_seed);
}

extern "C" lq_status lq_quantize_grouped(int lattice, int n, const void* const* W_dev, int wdtype,
                                         const int64_t* rows, const int64_t* cols, const int64_t* ldw, int tile,
                                         const uint64_t* seeds, float beta, int8_t* const* codes_dev,
                                         float* const* scales_dev, int8_t* const* signs_dev,
                                         int32_t* dev_status_dev, void* stream) {
  LQ_NVTX_RANGE("lq_quantize_grouped");
  if (n < 1 || n > kQuantMaxMats) return LQ_ERR_ARG;
  if (W_dev == nullptr || rows == nullptr || cols == nullptr || ldw == nullptr || seeds == nullptr ||
      codes_dev == nullptr || scales_dev == nullptr || signs_dev == nullptr)
    return LQ_ERR_ARG;
  for (int m = 0; m < n; ++m) {
    const lq_status st = validate_quantize(lattice, W_dev[m], wdtype, rows[m], cols[m], ldw[m], tile, beta,
                                           codes_dev[m], scales_dev[m], signs_dev[m], dev_status_dev);
    if (st != LQ_OK) return st;
  }
  void* sc[kQuantMaxMats];
  for (int m = 0; m < n; ++m) sc[m] = scales_dev[m];
  return quantize_group(lattice, n, W_dev, wdtype, rows, cols, ldw, tile, seeds, beta, codes_dev, sc, signs_dev,
                        dev_status_dev, LQ_SCALE_TILE_F32, true, (cudaStream_t)stream);
}

template <int LAT, bool OB, bool DITHER>
static lq_status launch_dequant_d(const DequantArgs& a, cudaStream_t st) {
  static int per_sm = 0;
  if (per_sm == 0) per_sm = occupancy_per_sm(dequantize_kernel<LAT, OB, DITHER>, 256);
  const int grid = persistent_grid(a.units, 8, 1, per_sm);
  if (grid <= 0) return LQ_ERR_CUDA;
  dequantize_kernel<LAT, OB, DITHER><<<grid, 256, 0, st>>>(a);
  return check_launch();
}

template <int LAT, bool OB>
static lq_status launch_dequant(const DequantArgs& a, cudaStream_t st) {
  return a.dither ? launch_dequant_d<LAT, OB, true>(a, st) : launch_dequant_d<LAT, OB, false>(a, st);
}

namespace {

lq_status dequantize_fmt(int lattice, const int8_t* codes_dev, const void* scales_dev, int sfmt,
                         const int8_t* signs_dev, int64_t rows, int64_t cols, int tile, void* What_dev,
                         int out_dtype, cudaStream_t s, bool dither = false, uint64_t dither_seed = 0) {
  lq_status st = validate_common(lattice, rows, cols, tile);
  if (st != LQ_OK) return st;
  if (out_dtype != LQ_BF16 && out_dtype != LQ_F32) return LQ_ERR_DTYPE;
  if (!valid_scale_format(sfmt)) return LQ_ERR_ARG;
  if (rows == 0) return LQ_OK;
  if (codes_dev == nullptr || scales_dev == nullptr || signs_dev == nullptr || What_dev == nullptr)
    return LQ_ERR_ARG;
  const uintptr_t salign = (sfmt == LQ_SCALE_TILE_F32) ? 3u : 1u;
  if (!aligned16(codes_dev) || !aligned16(signs_dev) || !aligned16(What_dev) ||
      (reinterpret_cast<uintptr_t>(scales_dev) & salign) != 0)
    return LQ_ERR_ARG;
  DequantArgs a;
  a.codes = codes_dev; a.scales = scales_dev; a.sfmt = sfmt; a.signs = signs_dev; a.rows = rows; a.cols = cols;
  a.tile = tile; a.lanes_per_tile = tile / kLaneElems; a.tiles_per_row = (int)(cols / tile);
  a.chunks_per_row = (int)((cols + kChunkCols - 1) / kChunkCols);
  a.inv_2sqrt_tile = (float)(0.5 / sqrt((double)tile));
  a.out = What_dev;
  a.units = rows * a.chunks_per_row;
  a.dither = dither ? 1 : 0;
  a.dither_seed = dither_seed;
  const bool ob = (out_dtype == LQ_BF16);
  switch (lattice) {
    case LQ_E8: return ob ? launch_dequant<LQ_E8, true>(a, s) : launch_dequant<LQ_E8, false>(a, s);
    case LQ_D4: return ob ? launch_dequant<LQ_D4, true>(a, s) : launch_dequant<LQ_D4, false>(a, s);
    case LQ_A2: return ob ? launch_dequant<LQ_A2, true>(a, s) : launch_dequant<LQ_A2, false>(a, s);
    default:    return ob ? launch_dequant<LQ_Z1, true>(a, s) : launch_dequant<LQ_Z1, false>(a, s);
  }
}

}  // namespace

extern "C" lq_status lq_dequantize(int lattice, const int8_t* codes_dev, const float* scales_dev,
                                   const int8_t* signs_dev, int64_t rows, int64_t cols, int tile,
                                   void* What_dev, int out_dtype, void* stream) {
  LQ_NVTX_RANGE("lq_dequantize");
  return dequantize_fmt(lattice, codes_dev, scales_dev, LQ_SCALE_TILE_F32, signs_dev, rows, cols, tile, What_dev,
                        out_dtype, (cudaStream_t)stream);
}

extern "C" lq_status lq_dequantize_ex(int lattice, const int8_t* codes_dev, const void* scales_dev,
                                      int scale_format, const int8_t* signs_dev, int64_t rows, int64_t cols,
                                      int tile, void* What_dev, int out_dtype, void* stream) {
  LQ_NVTX_RANGE("lq_dequantize_ex");
  return dequantize_fmt(lattice, codes_dev, scales_dev, scale_format, signs_dev, rows, cols, tile, What_dev,
                        out_dtype, (cudaStream_t)stream);
}

extern "C" lq_status lq_dequantize_dithered(int lattice, const int8_t* codes_dev, const void* scales_dev,
                                            int scale_format, const int8_t* signs_dev, uint64_t dither_seed,
                                            int64_t rows, int64_t cols, int tile, void* What_dev, int out_dtype,
                                            void* stream) {
  LQ_NVTX_RANGE("lq_dequantize_dithered");
  if (scale_format != LQ_SCALE_TILE_F32 && scale_format != LQ_SCALE_TILE_F16) return LQ_ERR_ARG;
  return dequantize_fmt(lattice, codes_dev, scales_dev, scale_format, signs_dev, rows, cols, tile, What_dev,
                        out_dtype, (cudaStream_t)stream, true, dither_seed);
}
