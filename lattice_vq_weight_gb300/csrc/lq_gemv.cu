// Decode-side GEMV: y = W^ x computed from the lattice codes.
//
// HyperQuant page, mma="bf16" paragraph: the product is accumulated from the
// codes as they are read (no decoded weight in memory); mma="int8" paragraph:
// the activation is rotated at each forward.
//
//   y[b, r] = sum_t s[r, t] * sum_i p[r, t, i] * x~[b, t, i],  x~ = H D x / sqrt(T).
//
// Two kernels:
//  1. rotate_activation_kernel: x~ per tile, times 1/2 (codes are 2p) and, for
//     A2, sqrt(3) on odd coordinates (the second A2 code is 2y/sqrt3); each
//     (row, tile) is scaled by a power of two into [2^14, 2^15) and rounded to
//     fp16 (11 significant bits, about 3e-4 normwise on y -- the precision of
//     the prefill GEMM's fp16 activations).  It also zeroes y.
//  2. gemv_kernel: warps stream 16-row groups of int8 codes with 16-byte loads,
//     turn them into exact fp16 values (magic-number conversion: the fp16 with
//     bits 0x6400 | u is 1024 + u for a byte u; the fast int8 -> fp16 conversion
//     of Kim et al., "Who Says Elephants Can't Run: Bringing Large Scale MoE
//     Models into Cloud Scale Production", 2022), and run m16n8k16 fp16 MMAs with fp32
//     accumulation against the activation.  One accumulator per tile is scaled by
//     s[r, t] * 2^-e[b, t] and summed; warps that split a row combine with
//     fp32 atomics.
// Both kernels take a group of up to kGemvMaxMats matrices that share the
// activation x (for example the q, k and v projections of a layer), each with
// its own signs, scales and output: one launch pair serves the whole group.
// Both are programmatic dependent launches: the rotation waits for the grid
// before it (whose output x may be), the GEMV prefetches codes during the
// rotation and waits for x~ before reading it.
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "lq_act.cuh"
#include "lq_device.cuh"
#include "lq_host.h"
#include "lq_tma.cuh"

namespace lq {

struct GemvMat {
  const void* scales;    // in the launch's scale format (gemv_kernel's SF)
  float* y;
  int64_t rows;
  int64_t groups;        // row groups of 16 RG rows
  int64_t step_begin;    // first step of this matrix in the group's step order
};

struct GemvArgs {
  CUtensorMap maps[kGemvMaxMats];   // codes of each matrix, boxes of 64 columns x 16 RG rows
  GemvMat mat[kGemvMaxMats];
  int n_mats;
  int64_t cols;
  int tile, tiles_per_row, batch;
  const __half* xh;      // [n_mats x batch x cols]
  const float* xs;       // [n_mats x batch x tiles]
  int64_t steps;         // total steps (row group, 64-column slice) of all matrices
  int64_t warps;         // warps of the persistent grid
  int32_t* status;       // LQ_DEV_TIMEOUT if a code copy never landed
};

constexpr long long kGemvWaitCycles = 2000000000ll;   // about a second

// Work: a step is one 64-column slice of one group of 16 RG rows; the steps of
// all matrices are ordered matrix, row group, column.  Steps come in pairs
// (a "box": 128 columns of the group, copied as one unit), and warp w of the
// persistent grid takes the contiguous box range [w B / W, (w+1) B / W), so
// every warp streams the same number of code bytes whatever the tile size or
// the matrices' shapes.  The per-tile scale is applied when a tile ends or
// the range ends (the tile sum splits linearly), and a warp flushes its
// per-row sums whenever its range leaves a row group -- with plain stores
// when it covered the whole row, else with fp32 atomics.
//
// Fragment mapping (g = lane/4, q4 = lane%4): within a step the thread uses
// 16 code bytes of rows rg and rg+8 of each 16-row block (rg a permutation of
// g, see below) at columns 16 q4 .. 16 q4 + 15; MMA k-chunk c uses bytes 4c .. 4c+3, i.e. k-slots (2 q4, 2 q4+1,
// 2 q4+8, 2 q4+9) hold columns 16 q4 + 4c + (0, 1, 2, 3).  The activation
// fragment of column n = g uses the same permutation, so the dot products are
// unchanged.
//
// Codes arrive by TMA: one 2-D box per box unit (128 columns x 16 RG rows,
// a full 128-byte line of each row, 128-byte swizzle) into a ring of S stages
// per warp, issued by lane 0 S - 1 boxes ahead and counted on the stage's
// mbarrier; rows past the matrix read as zeros.  With the swizzle (16-byte
// chunk c of row r at chunk c ^ (r & 7)) a quarter warp reads 8 distinct
// chunk positions, so the 16-byte loads are conflict-free.  The ring is filled
// before griddepcontrol.wait: codes do not depend on the activation kernel
// that precedes this one, so with programmatic dependent launch the code
// stream starts while that kernel is still running.
template <int NB, int RG, int S, int SF>
__global__ void __launch_bounds__(128, NB == 1 ? 4 : 3) gemv_kernel(const __grid_constant__ GemvArgs a) {
  constexpr int kBoxBytes = 16 * RG * 128;
  constexpr int kWarps = 4;
  static_assert((S & (S - 1)) == 0, "ring size must be a power of two");
  extern __shared__ __align__(1024) uint8_t gemv_smem_raw[];
  // 1024-byte alignment of every stage (the swizzle pattern repeats every 8 rows)
  uint8_t* gemv_smem = gemv_smem_raw + ((1024u - (smem_addr(gemv_smem_raw) & 1023u)) & 1023u);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2, q4 = lane & 3;
  // matrix row (within each 8-row half of a 16-row block) of MMA fragment row
  // g: rows 2j and 2j + 1 of the fragment, read by one quarter warp, sit 4 rows
  // apart, so that the swizzle puts their chunks on different banks
  const int rg = (g >> 1) | ((g & 1) << 2);
  uint8_t* ring = gemv_smem + warp * S * kBoxBytes;
  uint64_t* bar = reinterpret_cast<uint64_t*>(gemv_smem + kWarps * S * kBoxBytes) + warp * S;
  const int64_t w = (int64_t)blockIdx.x * (blockDim.x >> 5) + warp;
  const int64_t boxes = a.steps >> 1;
  const int64_t b0 = w * boxes / a.warps;
  const int64_t b1 = (w + 1) * boxes / a.warps;
  const int64_t i0 = 2 * b0;
  const int64_t n_box = b1 - b0;
  const int64_t n_it = 2 * n_box;
  const int steps = a.tile >> 6;                 // steps per tile (power of two)
  const int per_grp = a.tiles_per_row * steps;          // steps per row group (even)

  if (lane == 0) {
#pragma unroll
    for (int i = 0; i < S; ++i) mbar_init1(&bar[i], 1);
    mbar_init_fence();
  }
  __syncwarp();

  const bool xok0 = g < a.batch;
  const bool xok1 = NB > 1 && 8 + g < a.batch;
  const int64_t xoff0 = (int64_t)(xok0 ? g : 0) * a.cols + 16 * q4;
  const int64_t xoff1 = (int64_t)(xok1 ? 8 + g : 0) * a.cols + 16 * q4;
  const int64_t xmat = (int64_t)a.batch * a.cols;      // x~ elements per matrix

  // Position of a step: matrix, row group and step s within the group (the
  // group's steps run along k: s covers columns 64 s .. 64 s + 63), advanced
  // one step at a time (divisions only at start).
  const int steps_log2 = __ffs(steps) - 1;
  struct Cursor {
    int m, grp, s;
  };
  auto start_cursor = [&]() {
    Cursor c;
    c.m = 0;
    while (c.m + 1 < a.n_mats && i0 >= a.mat[c.m + 1].step_begin) ++c.m;
    const int64_t local = i0 - a.mat[c.m].step_begin;
    c.grp = (int)(local / per_grp);
    c.s = (int)(local - (int64_t)c.grp * per_grp);
    return c;
  };
  auto advance = [&](Cursor& c, int by) {
    c.s += by;
    if (c.s == per_grp) {
      c.s = 0;
      if (++c.grp == a.mat[c.m].groups) { c.grp = 0; ++c.m; }
    }
  };
  Cursor ci = start_cursor();   // next box to issue (always at an even step)
  Cursor cb = ci;               // next box whose activations to load
  Cursor cm = ci;               // step being computed
  auto issue = [&](int64_t ib) {
    if (ib < n_box) {
      if (lane == 0) {
        const int st = (int)(ib & (S - 1));
        mbar_expect_tx(&bar[st], kBoxBytes);
        tma_load_2d(ring + st * kBoxBytes, &a.maps[ci.m], &bar[st], ci.s * 64, ci.grp * 16 * RG);
      }
      advance(ci, 2);
    }
  };
  // activations of both steps of box ib (loaded one box ahead of their use)
  auto load_xbox = [&](int64_t ib, uint4 (&h)[2][NB][2]) {
    if (ib < n_box) {
      const __half* xb = a.xh + (int64_t)cb.m * xmat + (int64_t)cb.s * 64;
#pragma unroll
      for (int sub = 0; sub < 2; ++sub) {
        if (xok0) {
          h[sub][0][0] = __ldg(reinterpret_cast<const uint4*>(xb + xoff0 + 64 * sub));
          h[sub][0][1] = __ldg(reinterpret_cast<const uint4*>(xb + xoff0 + 64 * sub) + 1);
        }
        if constexpr (NB > 1) {
          if (xok1) {
            h[sub][1][0] = __ldg(reinterpret_cast<const uint4*>(xb + xoff1 + 64 * sub));
            h[sub][1][1] = __ldg(reinterpret_cast<const uint4*>(xb + xoff1 + 64 * sub) + 1);
          }
        }
      }
      advance(cb, 2);
    }
  };

  // code prefetch first (independent of the preceding kernel), then wait for it
#pragma unroll
  for (int ib = 0; ib < S - 1; ++ib) issue(ib);
  asm volatile("griddepcontrol.wait;" ::: "memory");

  float yacc[RG][NB][4], acc[RG][NB][4];
#pragma unroll
  for (int i = 0; i < RG; ++i)
#pragma unroll
    for (int n = 0; n < NB; ++n)
#pragma unroll
      for (int c = 0; c < 4; ++c) yacc[i][n][c] = acc[i][n][c] = 0.f;
  uint4 xA[2][NB][2], xB[2][NB][2];
#pragma unroll
  for (int sub = 0; sub < 2; ++sub)
#pragma unroll
    for (int n = 0; n < NB; ++n)
      xA[sub][n][0] = xA[sub][n][1] = xB[sub][n][0] = xB[sub][n][1] = make_uint4(0, 0, 0, 0);
  load_xbox(0, xA);
  int cur_grp = -1, cur_m = -1, steps_in_grp = 0;
  bool timed_out = false;
  // scales of the tile being accumulated: s[r, t] for the thread's rows and
  // 2^-e[b, t] for its batch columns, loaded when the tile starts
  float scur[RG][2], fcur[NB][2];

  auto flush = [&]() {
    const bool whole_row = steps_in_grp == per_grp;
    float* y = a.mat[cur_m].y;
    const int64_t rows = a.mat[cur_m].rows;
#pragma unroll
    for (int i = 0; i < RG; ++i)
#pragma unroll
      for (int n = 0; n < NB; ++n)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int64_t r = (int64_t)cur_grp * 16 * RG + 16 * i + 8 * (c >> 1) + rg;
          const int bb = n * 8 + 2 * q4 + (c & 1);
          if (r < rows && bb < a.batch) {
            float* dst = y + (int64_t)bb * rows + r;
            if (whole_row) *dst = yacc[i][n][c]; else atomicAdd(dst, yacc[i][n][c]);
          }
          yacc[i][n][c] = 0.f;
        }
  };

  // swizzled 16-byte chunk of the thread in rows 8 h + rg of a block: column
  // chunk 4 sub + q4 sits at chunk (4 sub + q4) ^ rg (every block starts at a
  // multiple of 8 rows)
  const int off0 = 128 * rg + 16 * ((0 + q4) ^ rg);
  const int off1 = 128 * rg + 16 * ((4 + q4) ^ rg);

  // one 64-column step: codes of the box at sub-step `sub`, activations xh
  auto do_step = [&](const uint8_t* box, int sub, const uint4 (&xh)[NB][2], int64_t it) {
    const int grp = cm.grp;
    const int m = cm.m;
    const int t = cm.s >> steps_log2;
    const bool tile_start = (cm.s & (steps - 1)) == 0 || it == 0;
    const bool tile_end = (cm.s & (steps - 1)) == steps - 1 || it == n_it - 1;
    advance(cm, 1);
    if (grp != cur_grp || m != cur_m) {
      if (cur_grp >= 0) flush();
      cur_grp = grp;
      cur_m = m;
      steps_in_grp = 0;
    }
    ++steps_in_grp;
    if (tile_start) {
      const float* xs = a.xs + (int64_t)m * a.batch * a.tiles_per_row + t;
      const void* scales = a.mat[m].scales;
      const int64_t rows = a.mat[m].rows;
#pragma unroll
      for (int n = 0; n < NB; ++n)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int bb = n * 8 + 2 * q4 + h;
          fcur[n][h] = (bb < a.batch) ? __ldg(xs + (int64_t)bb * a.tiles_per_row) : 0.f;
        }
#pragma unroll
      for (int i = 0; i < RG; ++i)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int64_t r = (int64_t)grp * 16 * RG + 16 * i + 8 * h + rg;
          scur[i][h] = (r < rows) ? load_scale_t<SF>(scales, r, t, a.tiles_per_row) : 0.f;
        }
    }
    const uint8_t* slot = box + (sub ? off1 : off0);
    uint4 cw[RG][2];
#pragma unroll
    for (int i = 0; i < RG; ++i) {
      cw[i][0] = *reinterpret_cast<const uint4*>(slot + 128 * (16 * i));
      cw[i][1] = *reinterpret_cast<const uint4*>(slot + 128 * (16 * i + 8));
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint32_t bh[NB][2];
#pragma unroll
      for (int n = 0; n < NB; ++n) {
        const uint4& H = xh[n][c >> 1];
        bh[n][0] = (c & 1) ? H.z : H.x;
        bh[n][1] = (c & 1) ? H.w : H.y;
      }
#pragma unroll
      for (int i = 0; i < RG; ++i) {
        const uint32_t wa = (c == 0) ? cw[i][0].x : (c == 1) ? cw[i][0].y : (c == 2) ? cw[i][0].z : cw[i][0].w;
        const uint32_t wb = (c == 0) ? cw[i][1].x : (c == 1) ? cw[i][1].y : (c == 2) ? cw[i][1].z : cw[i][1].w;
        uint32_t a0, a2, a1, a3;
        codes_to_f16x2(wa, a0, a2);
        codes_to_f16x2(wb, a1, a3);
#pragma unroll
        for (int n = 0; n < NB; ++n) {
          mma16816(acc[i][n], a0, a1, a2, a3, bh[n][0], bh[n][1]);
        }
      }
    }
    if (tile_end) {
#pragma unroll
      for (int i = 0; i < RG; ++i)
#pragma unroll
        for (int n = 0; n < NB; ++n) {
          yacc[i][n][0] = fmaf(acc[i][n][0], scur[i][0] * fcur[n][0], yacc[i][n][0]);
          yacc[i][n][1] = fmaf(acc[i][n][1], scur[i][0] * fcur[n][1], yacc[i][n][1]);
          yacc[i][n][2] = fmaf(acc[i][n][2], scur[i][1] * fcur[n][0], yacc[i][n][2]);
          yacc[i][n][3] = fmaf(acc[i][n][3], scur[i][1] * fcur[n][1], yacc[i][n][3]);
#pragma unroll
          for (int c = 0; c < 4; ++c) acc[i][n][c] = 0.f;
        }
    }
  };

  // one box: refill the ring, prefetch the next box's activations, compute
  // both steps with the activations X (the next box's go to Xn)
  auto do_box = [&](int64_t ib, const uint4 (&X)[2][NB][2], uint4 (&Xn)[2][NB][2]) -> bool {
    // the stage refilled now was read for the previous box: order those reads
    // before the copy that overwrites it
    fence_proxy_async_smem();
    __syncwarp();
    issue(ib + S - 1);
    load_xbox(ib + 1, Xn);
    const int st = (int)(ib & (S - 1));
    if (!mbar_wait_bounded(&bar[st], (uint32_t)((ib / S) & 1), kGemvWaitCycles)) return false;
    const uint8_t* box = ring + st * kBoxBytes;
    do_step(box, 0, X[0], 2 * ib);
    do_step(box, 1, X[1], 2 * ib + 1);
    return true;
  };

  int64_t ib = 0;
  for (; ib < n_box; ib += 2) {
    // boxes in pairs, so that the two activation register sets alternate
    if (!do_box(ib, xA, xB)) { timed_out = true; break; }
    if (ib + 1 < n_box && !do_box(ib + 1, xB, xA)) { ++ib; timed_out = true; break; }
  }
  if (timed_out) {
    // copies issued for boxes ib .. ib + S - 1 may still be in flight: let them land
    for (int64_t j = ib; j < n_box && j < ib + S; ++j)
      mbar_wait_bounded(&bar[j & (S - 1)], (uint32_t)((j / S) & 1), kGemvWaitCycles);
    if (lane == 0) raise_flag(a.status, LQ_DEV_TIMEOUT);
    return;
  }
  if (cur_grp >= 0) flush();
}

}  // namespace lq

using namespace lq;

namespace {

constexpr size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

struct GemvWorkspace {
  size_t xh, xs, total;
};

GemvWorkspace gemv_workspace_layout(int n_mats, int batch, int64_t cols, int tile) {
  GemvWorkspace w;
  const size_t rows = (size_t)n_mats * (size_t)batch;
  w.xh = 0;
  w.xs = align256(rows * (size_t)cols * 2);
  w.total = w.xs + align256(rows * (size_t)(cols / tile) * 4);
  return w;
}

// Minimum steps per warp: below it the ring fill and flush of a warp cost more
// than its share of the stream.
constexpr int64_t kMinStepsPerWarp = 4;

template <int NB, int RG, int SF>
lq_status launch_gemv(const GemvArgs& a0, cudaStream_t st) {
  constexpr int S = 2;                       // ring stages (boxes) per warp
  constexpr int kWarps = 4;
  constexpr size_t smem = (size_t)kWarps * S * (16 * RG * 128) + (size_t)kWarps * S * 8 + 1024;
  GemvArgs a = a0;
  static int per_sm = 0;
  if (per_sm == 0) {
    if (cudaFuncSetAttribute(gemv_kernel<NB, RG, S, SF>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess) {
      cudaGetLastError();
      return LQ_ERR_CUDA;
    }
    per_sm = occupancy_per_sm(gemv_kernel<NB, RG, S, SF>, kWarps * 32, smem);
  }
  const int sms = device_sm_count();
  if (sms <= 0) return LQ_ERR_CUDA;
  const int64_t steps_per_grp = (int64_t)a.tiles_per_row * (a.tile >> 6);
  int64_t total = 0;
  for (int m = 0; m < a.n_mats; ++m) {
    a.mat[m].groups = (a.mat[m].rows + 16 * RG - 1) / (16 * RG);
    a.mat[m].step_begin = total;
    total += a.mat[m].groups * steps_per_grp;
  }
  a.steps = total;
  int64_t ctas = (int64_t)sms * per_sm;
  const int64_t need = (total + kWarps * kMinStepsPerWarp - 1) / (kWarps * kMinStepsPerWarp);
  if (ctas > need) ctas = need;
  if (ctas < 1) ctas = 1;
  a.warps = ctas * kWarps;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)ctas);
  cfg.blockDim = dim3(kWarps * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, gemv_kernel<NB, RG, S, SF>, a) != cudaSuccess) {
    cudaGetLastError();
    return LQ_ERR_CUDA;
  }
  return LQ_OK;
}

// Validation and both launches for a group of n matrices sharing x.
lq_status gemv_group(int lattice, int n, const int8_t* const* codes_dev, const void* const* scales_dev,
                     const int8_t* const* signs_dev, const int64_t* rows, int64_t cols, int tile,
                     const void* x_dev, int xdtype, int batch, float* const* y_dev, void* workspace_dev,
                     int32_t* dev_status_dev, cudaStream_t s, int sfmt = LQ_SCALE_TILE_F32) {
  if (n < 1 || n > kGemvMaxMats) return LQ_ERR_ARG;
  if (sfmt != LQ_SCALE_TILE_F32 && sfmt != LQ_SCALE_ROW_BF16 && sfmt != LQ_SCALE_TILE_F16) return LQ_ERR_ARG;
  const uintptr_t salign = (sfmt == LQ_SCALE_TILE_F32) ? 3u : 1u;
  if (codes_dev == nullptr || scales_dev == nullptr || signs_dev == nullptr || rows == nullptr ||
      y_dev == nullptr)
    return LQ_ERR_ARG;
  lq_status st = validate_common(lattice, 0, cols, tile);
  if (st != LQ_OK) return st;
  if (xdtype != LQ_BF16 && xdtype != LQ_F32) return LQ_ERR_DTYPE;
  if (batch < 1 || batch > 16) return LQ_ERR_SHAPE;
  int64_t total_rows = 0;
  for (int m = 0; m < n; ++m) {
    st = validate_common(lattice, rows[m], cols, tile);
    if (st != LQ_OK) return st;
    total_rows += rows[m];
  }
  if (total_rows == 0) return LQ_OK;
  if (x_dev == nullptr || workspace_dev == nullptr) return LQ_ERR_ARG;
  if (!aligned16(x_dev) || !aligned16(workspace_dev) || (dev_status_dev != nullptr && !aligned4(dev_status_dev)))
    return LQ_ERR_ARG;
  for (int m = 0; m < n; ++m) {
    if (signs_dev[m] == nullptr || !aligned16(signs_dev[m])) return LQ_ERR_ARG;
    if (rows[m] == 0) continue;
    if (codes_dev[m] == nullptr || scales_dev[m] == nullptr || y_dev[m] == nullptr) return LQ_ERR_ARG;
    if (!aligned16(codes_dev[m]) || (reinterpret_cast<uintptr_t>(scales_dev[m]) & salign) != 0 ||
        !aligned4(y_dev[m]))
      return LQ_ERR_ARG;
  }
  const GemvWorkspace lay = gemv_workspace_layout(n, batch, cols, tile);
  char* ws = reinterpret_cast<char*>(workspace_dev);
  // matrices without rows take no part (the kernels see only the others)
  int idx[kGemvMaxMats];
  int ne = 0;
  for (int m = 0; m < n; ++m)
    if (rows[m] > 0) idx[ne++] = m;

  RotateArgs r = {};
  r.x = x_dev; r.n_mats = ne; r.cols = cols; r.batch = batch; r.tile = tile;
  r.tiles_per_row = (int)(cols / tile);
  r.post_scale = (float)(0.5 / sqrt((double)tile));
  r.a2 = (lattice == LQ_A2);
  r.xh = reinterpret_cast<__half*>(ws + lay.xh);
  r.xs = reinterpret_cast<float*>(ws + lay.xs);
  r.status = dev_status_dev;
  int64_t max_y = 0;
  for (int j = 0; j < ne; ++j) {
    r.signs[j] = signs_dev[idx[j]];
    r.y[j] = y_dev[idx[j]];
    r.y_elems[j] = (int64_t)batch * rows[idx[j]];
    if (r.y_elems[j] > max_y) max_y = r.y_elems[j];
  }
  st = launch_rotation(r, xdtype, max_y, s);
  if (st != LQ_OK) return st;

  GemvArgs g = {};
  constexpr int kRowsPerStep = 32;   // 16 RG rows (RG = 2 in every instantiation below)
  for (int j = 0; j < ne; ++j) {
    if (!encode_codes_map(&g.maps[j], codes_dev[idx[j]], rows[idx[j]], cols, kRowsPerStep)) return LQ_ERR_CUDA;
    g.mat[j].scales = scales_dev[idx[j]];
    g.mat[j].y = y_dev[idx[j]];
    g.mat[j].rows = rows[idx[j]];
  }
  g.n_mats = ne;
  g.cols = cols; g.tile = tile; g.tiles_per_row = (int)(cols / tile); g.batch = batch;
  g.xh = r.xh; g.xs = r.xs; g.status = dev_status_dev;
  if (sfmt == LQ_SCALE_ROW_BF16)
    return batch <= 8 ? launch_gemv<1, 2, LQ_SCALE_ROW_BF16>(g, s) : launch_gemv<2, 2, LQ_SCALE_ROW_BF16>(g, s);
  if (sfmt == LQ_SCALE_TILE_F16)
    return batch <= 8 ? launch_gemv<1, 2, LQ_SCALE_TILE_F16>(g, s) : launch_gemv<2, 2, LQ_SCALE_TILE_F16>(g, s);
  return batch <= 8 ? launch_gemv<1, 2, LQ_SCALE_TILE_F32>(g, s) : launch_gemv<2, 2, LQ_SCALE_TILE_F32>(g, s);
}

}  // namespace

extern "C" size_t lq_gemv_workspace_size(int batch, int64_t cols, int tile) {
  if (batch <= 0 || cols <= 0 || tile <= 0) return 0;
  return gemv_workspace_layout(1, batch, cols, tile).total;
}

extern "C" size_t lq_gemv_grouped_workspace_size(int n, int batch, int64_t cols, int tile) {
  if (n <= 0 || batch <= 0 || cols <= 0 || tile <= 0) return 0;
  return gemv_workspace_layout(n, batch, cols, tile).total;
}

extern "C" lq_status lq_gemv(int lattice, const int8_t* codes_dev, const float* scales_dev,
                             const int8_t* signs_dev, int64_t rows, int64_t cols, int tile,
                             const void* x_dev, int xdtype, int batch, float* y_dev,
                             void* workspace_dev, int32_t* dev_status_dev, void* stream) {
  LQ_NVTX_RANGE("lq_gemv");
  lq_status st = validate_common(lattice, rows, cols, tile);
  if (st != LQ_OK) return st;
  if (xdtype != LQ_BF16 && xdtype != LQ_F32) return LQ_ERR_DTYPE;
  if (batch < 1 || batch > 16) return LQ_ERR_SHAPE;
  if (rows == 0) return LQ_OK;
  if (codes_dev == nullptr || scales_dev == nullptr || signs_dev == nullptr || x_dev == nullptr ||
      y_dev == nullptr || workspace_dev == nullptr)
    return LQ_ERR_ARG;
  const void* sc = scales_dev;
  return gemv_group(lattice, 1, &codes_dev, &sc, &signs_dev, &rows, cols, tile, x_dev, xdtype, batch,
                    &y_dev, workspace_dev, dev_status_dev, (cudaStream_t)stream);
}

extern "C" lq_status lq_gemv_ex(int lattice, const int8_t* codes_dev, const void* scales_dev, int scale_format,
                                const int8_t* signs_dev, int64_t rows, int64_t cols, int tile, const void* x_dev,
                                int xdtype, int batch, float* y_dev, void* workspace_dev,
                                int32_t* dev_status_dev, void* stream) {
  LQ_NVTX_RANGE("lq_gemv_ex");
  lq_status st = validate_common(lattice, rows, cols, tile);
  if (st != LQ_OK) return st;
  if (xdtype != LQ_BF16 && xdtype != LQ_F32) return LQ_ERR_DTYPE;
  if (batch < 1 || batch > 16) return LQ_ERR_SHAPE;
  if (rows == 0) return LQ_OK;
  if (codes_dev == nullptr || scales_dev == nullptr || signs_dev == nullptr || x_dev == nullptr ||
      y_dev == nullptr || workspace_dev == nullptr)
    return LQ_ERR_ARG;
  return gemv_group(lattice, 1, &codes_dev, &scales_dev, &signs_dev, &rows, cols, tile, x_dev, xdtype, batch,
                    &y_dev, workspace_dev, dev_status_dev, (cudaStream_t)stream, scale_format);
}

extern "C" lq_status lq_gemv_grouped(int lattice, int n, const int8_t* const* codes_dev,
                                     const float* const* scales_dev, const int8_t* const* signs_dev,
                                     const int64_t* rows, int64_t cols, int tile, const void* x_dev, int xdtype,
                                     int batch, float* const* y_dev, void* workspace_dev,
                                     int32_t* dev_status_dev, void* stream) {
  LQ_NVTX_RANGE("lq_gemv_grouped");
  if (n < 1 || n > kGemvMaxMats || scales_dev == nullptr) return LQ_ERR_ARG;
  const void* sc[kGemvMaxMats];
  for (int m = 0; m < n; ++m) sc[m] = scales_dev[m];
  return gemv_group(lattice, n, codes_dev, sc, signs_dev, rows, cols, tile, x_dev, xdtype, batch, y_dev,
                    workspace_dev, dev_status_dev, (cudaStream_t)stream);
}

// ---------------------------------------------------------------------------
// lq_gemv_noalloc: the same product for callers that cannot allocate device
// memory themselves.  Its workspace is a fixed array in this library's device
// image (allocated once per GPU when the library's module is loaded and kept
// until the process exits).  Host code must not use the array's name as a
// device address; the address is looked up with cudaGetSymbolAddress the first
// time a device is used, and again whenever the device's current context is no
// longer the one the address was looked up in (after cudaDeviceReset the
// module is loaded anew and the array may move).
static __device__ __align__(256) unsigned char g_gemv_noalloc_scratch[LQ_GEMV_NOALLOC_MAX_WORKSPACE];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxDevices] = {};
CUcontext g_scratch_ctx[kMaxDevices] = {};

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);

// The driver's current context of the calling thread (nullptr if unknown).
CUcontext current_context() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(p);
    else
      cudaGetLastError();
  });
  CUcontext c = nullptr;
  if (fn == nullptr || fn(&c) != CUDA_SUCCESS) return nullptr;
  return c;
}

// Device address of the scratch array on the current device, looked up once
// per device and context.
lq_status noalloc_scratch(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return LQ_ERR_CUDA;
  }
  const CUcontext ctx = current_context();
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_ptr[dev] == nullptr || ctx == nullptr || ctx != g_scratch_ctx[dev]) {
    // the lookup also makes the device's primary context current if no
    // context was current yet
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_gemv_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return LQ_ERR_CUDA;
    }
    g_scratch_ptr[dev] = p;
    g_scratch_ctx[dev] = current_context();
  }
  *out = g_scratch_ptr[dev];
  return LQ_OK;
}

}  // namespace

extern "C" lq_status lq_gemv_noalloc(int lattice, const int8_t* codes_dev, const float* scales_dev,
                                     const int8_t* signs_dev, int64_t rows, int64_t cols, int tile,
                                     const void* x_dev, int xdtype, int batch, float* y_dev,
                                     int32_t* dev_status_dev, void* stream) {
  LQ_NVTX_RANGE("lq_gemv_noalloc");
  lq_status st = validate_common(lattice, rows, cols, tile);
  if (st != LQ_OK) return st;
  if (batch < 1 || batch > 16) return LQ_ERR_SHAPE;
  if (lq_gemv_workspace_size(batch, cols, tile) > (size_t)LQ_GEMV_NOALLOC_MAX_WORKSPACE) return LQ_ERR_SHAPE;
  void* scratch = nullptr;
  st = noalloc_scratch(&scratch);
  if (st != LQ_OK) return st;
  return lq_gemv(lattice, codes_dev, scales_dev, signs_dev, rows, cols, tile, x_dev, xdtype, batch, y_dev,
                 scratch, dev_status_dev, stream);
}
