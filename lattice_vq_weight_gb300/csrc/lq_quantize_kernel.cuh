// The quantize kernel (tile RHT + lattice nearest point) and its launch
// templates, shared by the translation units that instantiate it
// (lq_quantize.cu: float32 tile scales, one matrix or a group; lq_quantize_fmt.cu:
// the 16-bit scale formats; lq_quantize_dither.cu: the subtractive dither).
//
// HyperQuant page, "Key algorithmic ingredients": per-tile randomized Hadamard
// transform, then optimal low-dimensional lattice VQ (E8, D4, A2, Z1).
// Conway & Sloane, Sphere Packings, Lattices and Groups, ch. 20: nearest-point
// decoders.
//
// Work decomposition.  A warp unit is one 2048-column chunk of one row, and a
// CTA unit the same chunk of four consecutive rows of one matrix (one per
// warp), so the four warps of a CTA share the chunk's signs.  A persistent
// grid strides over CTA units, numbered matrix by matrix, row group by row
// group, chunk fastest; a grid that is a multiple of the chunks per row keeps
// every CTA on one chunk of a matrix.
//
// Staging.  Each warp's input arrives by one TMA copy per unit (lane 0 issues
// it, an mbarrier counts its bytes) into a two-stage ring: the matrix is read
// as lines of 128 bytes with the 128-byte swizzle, one line per lane for bf16
// (two for fp32), so each lane reads its own 64 columns back with
// conflict-free 16-byte loads.  The copy of the next unit is in flight while
// the current one is transformed.
//
// Registers.  Lane l holds columns [64 l, 64 l + 64) of the chunk as float2
// p[32], p[j].x = column j and p[j].y = column j + 32: five butterfly stages
// run as packed f32x2 pairs, the stage between the halves as scalars.  Tile
// bits 6 and 7 (or 6 alone for 128-column tiles) sit in the lane index; one
// pass through shared memory swaps them with register bits 3 and 4, so their
// stages run in registers too, every 8-column block stays in one lane, and
// .x / .y hold two different blocks for the decoders (lq_device.cuh); larger
// tiles' remaining bits cross lanes with shuffles.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "lq_device.cuh"
#include "lq_host.h"
#include "lq_tma.cuh"

namespace lq {

constexpr int kQuantMaxMats = LQ_QUANTIZE_MAX_GROUP;
constexpr int kQuantWarps = 4;
constexpr int kQuantThreads = kQuantWarps * 32;
constexpr long long kQuantWaitCycles = 2000000000ll;   // about a second: a TMA copy that never lands

// One matrix of a quantize launch.  Its CTA units are cta_begin ..
// cta_begin + row_groups * chunks_per_row - 1.
struct QuantMat {
  int8_t* codes;
  void* scales;             // in the launch's scale format
  const int8_t* signs;
  const void* W;            // the input (read by the fix-up of deferred tiles)
  int64_t ldw;              // its row stride in elements
  int64_t rows, cols;
  int64_t cta_begin, row_groups;
  int tiles_per_row, chunks_per_row;
};

struct QuantArgs {
  CUtensorMap maps[kQuantMaxMats];   // the matrices' input, see encode_row_lines_map
  QuantMat mat[kQuantMaxMats];
  int n_mats;
  int tile, tile_shift, lanes_per_tile;
  float beta, sqrt_tile, inv_tile;
  int32_t* status;
  int64_t cta_units;        // CTA units of all matrices
  uint64_t dither_seed;     // subtractive dither (DITHER instantiations only)
};

// Shared memory of a CTA: the chunk's sign masks, the parity-fix selectors,
// the mbarriers and, per warp, two stages of raw input.  A stage also serves
// as the buffer of the butterfly exchange once its input is in registers.
template <bool BF16> struct QuantSmem {
  static constexpr int kBoxBytes = BF16 ? 4096 : 8192;               // one warp unit of input
  static constexpr int kStageBytes = BF16 ? 5120 : 8192;             // >= the exchange's 280 16-byte slots
  static constexpr int kMaskBytes = 16 * 32 * 16;                    // uint4 [16][32]
  static constexpr int kSelOffset = kMaskBytes;                      // uint2 [9]
  static constexpr int kBarOffset = kSelOffset + 128;                // uint64 [warps][2]
  static constexpr int kStageOffset = 10240;                         // 1024-aligned
  static constexpr int kBytes = kStageOffset + kQuantWarps * 2 * kStageBytes;
  static constexpr int kDynamic = kBytes + 1024;                     // room to align the base
  static_assert(kBarOffset + kQuantWarps * 2 * 8 <= kStageOffset, "layout");
  static_assert(kStageBytes % 1024 == 0, "stages keep the 1024-byte alignment of the swizzle");
};

// ------------------------------------------------------------------ exchange
// Swap of EX lane bits (tile bits 6, 7) with register bits 3, 4 of p (float2
// index bits 3, 4) through shared memory, in two halves (float2 index bit 2)
// of 8 16-byte slots per lane.  A slot holds p[j], p[j + 1] (j even) and is
// named (u, h): xj<EX>(u, h) is its j; the low EX bits of u are the exchanged
// register bits, the others spectators.  Slot of the value with lane group G,
// spectator ux, lane bits a and register bits c:
//   (G >> (3 - EX)) * kBlk + ux * kUxSpan + (G & (X - 1)) * Q + a + 9 c,
// additive in a and c, so every access is a per-lane base plus a constant,
// and conflict-free for 16-byte accesses both when a varies (writes) and when
// c varies (reads): the slots of the 8 lanes of a phase differ modulo 8.
template <int EX> struct Xchg {
  static constexpr int Q = 1 << EX;          // lanes whose bits are swapped
  static constexpr int X = 8 >> EX;          // spectator values per half
  static constexpr int kUxSpan = 9 * Q - 1;
  static constexpr int kBlk = X * kUxSpan;
  static constexpr int kSlots = 4 * kBlk;
};
static_assert(Xchg<1>::kSlots * 16 <= 5120 && Xchg<2>::kSlots * 16 <= 5120, "exchange slots fit a stage");

template <int EX>
__device__ __forceinline__ constexpr int xj(int u, int h) {
  // EX = 2: u = (c3, c4, c1) low to high; EX = 1: u = (c3, c1, c4); h = c2
  return EX == 2 ? (((u >> 2) << 1) | (h << 2) | ((u & 3) << 3))
                 : ((((u >> 1) & 1) << 1) | (h << 2) | ((u & 1) << 3) | ((u >> 2) << 4));
}

template <int EX>
__device__ __forceinline__ void exchange_tile_bits(float2 (&p)[32], uint32_t buf, int lane) {
  using XC = Xchg<EX>;
  const int q = lane & (XC::Q - 1), G = lane >> EX;
  const uint32_t g = (uint32_t)((G >> (3 - EX)) * XC::kBlk + (G & (XC::X - 1)) * XC::Q);
  const uint32_t wb = buf + (g + (uint32_t)q) * 16u;
  const uint32_t rb = buf + (g + 9u * (uint32_t)q) * 16u;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    __syncwarp();
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const uint32_t off = (uint32_t)(((u >> EX) * XC::kUxSpan + 9 * (u & (XC::Q - 1))) * 16);
      const int j = xj<EX>(u, h);
      asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(wb + off), "f"(p[j].x), "f"(p[j].y),
                   "f"(p[j + 1].x), "f"(p[j + 1].y) : "memory");
    }
    __syncwarp();
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const uint32_t off = (uint32_t)(((u >> EX) * XC::kUxSpan + (u & (XC::Q - 1))) * 16);
      const int j = xj<EX>(u, h);
      asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                   : "=f"(p[j].x), "=f"(p[j].y), "=f"(p[j + 1].x), "=f"(p[j + 1].y)
                   : "r"(rb + off) : "memory");
    }
  }
  __syncwarp();
  // the swapped tile bits now sit in float2 index bits 3 (and 4)
#pragma unroll
  for (int hp = 8; hp < (8 << EX); hp <<= 1) {
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      if ((j & hp) == 0) {
        const float2 x0 = p[j], x1 = p[j + hp];
        p[j] = add2(x0, x1);
        p[j + hp] = sub2(x0, x1);
      }
    }
  }
}

// Column (within the chunk) of coordinate 0 of register block (g, h) of a lane
// after the exchange: p[8 g + i].x (h = 0) or .y (h = 1) is column
// block_col + i.
template <int EX>
__device__ __forceinline__ int block_col(int lane, int g, int h) {
  return EX == 2 ? 8 * (lane & 3) + 32 * h + 64 * ((lane & ~3) + g)
                 : 8 * (lane & 1) + 64 * (lane & ~1) + 32 * h + 64 * (g & 1) + 16 * (g >> 1);
}

// Codes of one 8-coordinate register block (consecutive coordinates y) with
// the scalar decoders of lq_device.cuh: one E8 block, two D4 blocks, four A2
// blocks or eight Z1 values; CHECK adds the exact int8 range check.
template <int LAT, bool CHECK>
__device__ __forceinline__ uint2 decode_block8(const float2 (&y4)[4], bool& r) {
  if constexpr (LAT == LQ_E8) {
    const BlockCodes8 b = decode_e8<CHECK>(y4, r);
    return make_uint2(b.w0, b.w1);
  } else if constexpr (LAT == LQ_D4) {
    const float2 a0[2] = {y4[0], y4[1]}, a1[2] = {y4[2], y4[3]};
    return make_uint2(decode_d4<CHECK>(a0, r), decode_d4<CHECK>(a1, r));
  } else if constexpr (LAT == LQ_A2) {
    return make_uint2(decode_a2_pair<CHECK>(y4[0], r) | (decode_a2_pair<CHECK>(y4[1], r) << 16),
                      decode_a2_pair<CHECK>(y4[2], r) | (decode_a2_pair<CHECK>(y4[3], r) << 16));
  } else {
    return make_uint2(decode_z1_quad<CHECK>(y4[0], y4[1], r), decode_z1_quad<CHECK>(y4[2], y4[3], r));
  }
}

// The scalar decoders with the exact int8 range check over a lane's 64
// values (blocks regrouped as consecutive 8-coordinate pairs), out of line: for
// E8 and Z1 with 16-bit scales or the dither it only runs for a lane holding a
// value of 62.5 or more (an outlier that survived the transform), so its
// registers are kept out of the fast path's allocation.
template <int LAT, int EX>
__device__ __noinline__ void decode_lane_checked(const float2 (&p)[32], float k, int lane, int8_t* dst, bool active,
                                                 bool& r) {
#pragma unroll
  for (int g = 0; g < 4; ++g) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float y[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) y[i] = (h ? p[8 * g + i].y : p[8 * g + i].x) * k;
      const float2 y4[4] = {make_float2(y[0], y[1]), make_float2(y[2], y[3]), make_float2(y[4], y[5]),
                            make_float2(y[6], y[7])};
      const uint2 w = decode_block8<LAT, true>(y4, r);
      if (active) *reinterpret_cast<uint2*>(dst + block_col<EX>(lane, g, h)) = w;
    }
  }
}

// Instantiations that defer the tiles their packed decoders cannot take (a
// value of 62.5 or more in a lane) to fix_deferred at the end of the warp's
// unit: E8 and Z1 with float32 tile scales and no dither.
template <int LAT, int SF, bool DITHER>
constexpr bool kDeferTiles = (LAT == LQ_E8 || LAT == LQ_Z1) && SF == LQ_SCALE_TILE_F32 && !DITHER;

__device__ __forceinline__ bool tile_lane_any(bool v, int lanes_per_tile) {
  uint32_t x = v ? 1u : 0u;
  for (int m = 1; m < lanes_per_tile; m <<= 1) x |= __shfl_xor_sync(0xffffffffu, x, m);
  return x != 0u;
}

// One deferred tile (row, t) of matrix M again from its input (an L2 hit: the
// unit was just copied in): signs, the Walsh-Hadamard transform (E columns per
// lane over T / E lanes), the scale and the range-checked scalar decoders.
template <int LAT, bool BF16, int E>
__device__ __forceinline__ void fix_tile(const QuantArgs& a, const QuantMat& M, int64_t row, int t, int lane,
                                         bool& range) {
  const int lpt = a.tile / E;
  const bool act = lane < lpt;
  const int64_t col0 = (int64_t)t * a.tile + (int64_t)lane * E;
  float v[E];
  if (act) {
    if constexpr (BF16) load_bf16_signed<E>(reinterpret_cast<const __nv_bfloat16*>(M.W) + row * M.ldw + col0,
                                            M.signs + col0, v);
    else load_f32_signed<E>(reinterpret_cast<const float*>(M.W) + row * M.ldw + col0, M.signs + col0, v);
  } else {
#pragma unroll
    for (int c = 0; c < E; ++c) v[c] = 0.f;
  }
  fwht_tile<E>(v, lpt, lane);
  float u2 = 0.f;
#pragma unroll
  for (int c = 0; c < E; ++c) u2 = fmaf(v[c], v[c], u2);
  for (int o = 16; o; o >>= 1) u2 += __shfl_xor_sync(0xffffffffu, u2, o);
  const bool finite = isfinite(u2);
  float s = finite ? a.beta * sqrtf(u2) * a.inv_tile : 0.f;
  const float k = (s > 0.f) ? 1.0f / (s * a.sqrt_tile) : 0.f;
  bool r = false;
#pragma unroll
  for (int b = 0; b < E / 8; ++b) {
    float2 y4[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) y4[i] = make_float2(v[8 * b + 2 * i] * k, v[8 * b + 2 * i + 1] * k);
    const uint2 w = finite ? decode_block8<LAT, true>(y4, r) : make_uint2(0u, 0u);
    if (act) *reinterpret_cast<uint2*>(M.codes + row * M.cols + col0 + 8 * b) = w;
  }
  if (lane == 0) reinterpret_cast<float*>(M.scales)[row * M.tiles_per_row + t] = s;
  range |= r;
}

// The deferred tiles of a warp's unit (row, chunk): bit l of dm is set for the
// first lane l of each.
template <int LAT, bool BF16, bool XL>
__device__ __forceinline__ void fix_deferred(const QuantArgs& a, const QuantMat& M, int64_t row, int chunk,
                                             unsigned dm, int lane, bool& range) {
  const int E = XL ? act_elems_for_tile(a.tile) : 16;
  while (dm != 0u) {
    const int src = __ffs((int)dm) - 1;
    dm &= dm - 1u;
    const int t = (int)(((int64_t)chunk * kChunkCols + (int64_t)src * kLaneElems) >> a.tile_shift);
    if (E == 16) fix_tile<LAT, BF16, 16>(a, M, row, t, lane, range);
    else if constexpr (XL) {
      if (E == 32) fix_tile<LAT, BF16, 32>(a, M, row, t, lane, range);
      else fix_tile<LAT, BF16, 64>(a, M, row, t, lane, range);
    }
  }
}

// ------------------------------------------------------------------ quantize
// EX = tile bits exchanged through shared memory: 1 for 128-column tiles, 2
// above.  XL: tiles of 512 ... 2048 columns, whose bits above 7 cross lanes
// with shuffles (a separate instantiation: the shuffle loop's registers would
// otherwise crowd the 128- and 256-column kernels).
// DITHER: subtractive dither (lq_device.cuh) added to y before the decode.
template <int LAT, bool BF16, int EX, bool XL, int SF, bool DITHER = false>
__global__ void __launch_bounds__(kQuantThreads, (BF16 && !XL) ? 4 : 3)
    quantize_kernel(const __grid_constant__ QuantArgs a) {
  using SM = QuantSmem<BF16>;
  extern __shared__ uint8_t quant_smem_raw[];
  // aligned by pointer arithmetic on the shared array, so that accesses stay
  // known shared-memory accesses
  uint8_t* smem = quant_smem_raw + ((1024u - (smem_addr(quant_smem_raw) & 1023u)) & 1023u);
  uint4* mtab = reinterpret_cast<uint4*>(smem);                       // [16][32] sign masks
  uint2* fixsel = reinterpret_cast<uint2*>(smem + SM::kSelOffset);    // [9]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + SM::kBarOffset) + 2 * warp;
  uint8_t* stage_base = smem + SM::kStageOffset + warp * 2 * SM::kStageBytes;

  if (threadIdx.x < 9) fixsel[threadIdx.x] = parity_fix_selector(threadIdx.x);
  if (lane == 0) {
    mbar_init1(&bar[0], 1);
    mbar_init1(&bar[1], 1);
    mbar_init_fence();
  }
  __syncthreads();

  // (matrix, row, chunk) of CTA unit cu for this warp
  struct Unit {
    int m, chunk;
    int64_t row;
    bool valid;   // the unit exists and its row is inside the matrix
  };
  auto locate = [&](int64_t cu, Unit& u) {
    u.valid = false;
    if (cu >= a.cta_units) return;
    while (u.m + 1 < a.n_mats && cu >= a.mat[u.m + 1].cta_begin) ++u.m;
    const QuantMat& M = a.mat[u.m];
    const int64_t local = cu - M.cta_begin;
    const int64_t rg = local < 0x7FFFFFFF ? (int64_t)((uint32_t)local / (uint32_t)M.chunks_per_row)
                                          : local / M.chunks_per_row;
    u.chunk = (int)(local - rg * M.chunks_per_row);
    u.row = rg * kQuantWarps + warp;
    u.valid = u.row < M.rows;
  };
  auto issue = [&](const Unit& u, int st) {
    if (lane == 0 && u.valid) {
      mbar_expect_tx(&bar[st], SM::kBoxBytes);
      tma_load_3d(stage_base + st * SM::kStageBytes, &a.maps[u.m], &bar[st], 0, u.chunk * (BF16 ? 32 : 64),
                  (int)u.row);
    }
  };

  bool range = false, nonfinite = false, timed_out = false;
  uint32_t phase = 0;          // bit s: parity of stage s's next completion
  bool pending[2] = {false, false};
  int key_m = -1, key_chunk = -1;
  int st = 0;
  int64_t cu = blockIdx.x;
  Unit cur;
  cur.m = 0;
  locate(cu, cur);
  issue(cur, 0);
  pending[0] = cur.valid;
  // the signs (and the per-row scales) come from the kernel launched before
  asm volatile("griddepcontrol.wait;" ::: "memory");

  for (; cu < a.cta_units; cu += gridDim.x) {
    Unit nxt = cur;
    locate(cu + gridDim.x, nxt);
    // the other stage was read, and written by the exchange, for the previous
    // unit: order those accesses before the copy that refills it
    fence_proxy_async_smem();
    __syncwarp();
    if (!timed_out) {
      issue(nxt, st ^ 1);
      pending[st ^ 1] = nxt.valid;
    }

    const QuantMat& M = a.mat[cur.m];
    if (cur.m != key_m || cur.chunk != key_chunk) {
      // sign masks of this chunk: entry (q, l) holds bit 31 set where the sign
      // of column 64 l + 4 q + i (i = 0..3) is -1; for bf16 input these are the
      // masks of the low and high halves of column pairs 2 q and 2 q + 1
      __syncthreads();
      for (int e = threadIdx.x; e < 16 * 32; e += kQuantThreads) {
        const int q = e >> 5, l = e & 31;
        const int64_t col = (int64_t)cur.chunk * kChunkCols + 64 * l + 4 * q;
        uint32_t w = 0;
        if (col < M.cols) w = *reinterpret_cast<const uint32_t*>(M.signs + col);
        mtab[e] = make_uint4((w << 24) & 0x80000000u, (w << 16) & 0x80000000u, (w << 8) & 0x80000000u,
                             w & 0x80000000u);
      }
      __syncthreads();
      key_m = cur.m;
      key_chunk = cur.chunk;
    }

    if (cur.valid && !timed_out) {
      if (!mbar_wait_bounded(&bar[st], (phase >> st) & 1u, kQuantWaitCycles)) {
        timed_out = true;
      } else {
        phase ^= 1u << st;
        pending[st] = false;
      }
    }
    if (cur.valid && !timed_out) {
      const uint8_t* raw = stage_base + st * SM::kStageBytes;
      const int64_t col0 = (int64_t)cur.chunk * kChunkCols + (int64_t)lane * kLaneElems;
      const bool active = col0 < M.cols;

      // ---- load, signs, bf16 -> fp32 (exact)
      float2 p[32];
      if constexpr (BF16) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint4 v = *reinterpret_cast<const uint4*>(raw + 128 * lane + 16 * (i ^ (lane & 7)));
          const uint4 m0 = mtab[(2 * i) * 32 + lane], m1 = mtab[(2 * i + 1) * 32 + lane];
          const uint32_t w[4] = {v.x, v.y, v.z, v.w};
          const uint32_t ml[4] = {m0.x, m0.z, m1.x, m1.z}, mh[4] = {m0.y, m0.w, m1.y, m1.w};
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            // word 4 i + h = columns c = 8 i + 2 h (low half) and c + 1
            const float lo = __uint_as_float(imad(w[h], 65536u, ml[h]));
            const float hi = __uint_as_float((w[h] & 0xFFFF0000u) ^ mh[h]);
            const int c = 8 * i + 2 * h;
            if (c < 32) { p[c].x = lo; p[c + 1].x = hi; }
            else { p[c - 32].y = lo; p[c - 31].y = hi; }
          }
        }
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int line = 2 * lane + (i >> 3);
          const uint4 v = *reinterpret_cast<const uint4*>(raw + 128 * line + 16 * ((i & 7) ^ (line & 7)));
          const uint4 m = mtab[i * 32 + lane];
          const uint32_t w[4] = {v.x ^ m.x, v.y ^ m.y, v.z ^ m.z, v.w ^ m.w};
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            const int c = 4 * i + h;
            if (c < 32) p[c].x = __uint_as_float(w[h]);
            else p[c - 32].y = __uint_as_float(w[h]);
          }
        }
      }

      // ---- Hadamard: register bits 0..4 (packed), the halves, the exchanged bits, shuffles
#pragma unroll
      for (int hp = 1; hp < 32; hp <<= 1) {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          if ((j & hp) == 0) {
            const float2 x0 = p[j], x1 = p[j + hp];
            p[j] = add2(x0, x1);
            p[j + hp] = sub2(x0, x1);
          }
        }
      }
#pragma unroll
      for (int j = 0; j < 32; ++j) p[j] = make_float2(p[j].x + p[j].y, p[j].x - p[j].y);
      exchange_tile_bits<EX>(p, smem_addr(raw), lane);
      if constexpr (XL) for (int mm = 1 << EX; mm < a.lanes_per_tile; mm <<= 1) {
        const float sgn = (lane & mm) ? -1.0f : 1.0f;
        const float2 sg2 = make_float2(sgn, sgn);
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          float2 o;
          o.x = __shfl_xor_sync(0xffffffffu, p[j].x, mm);
          o.y = __shfl_xor_sync(0xffffffffu, p[j].y, mm);
          p[j] = fma2(p[j], sg2, o);
        }
      }

      // ---- scale: U = sum u^2 over the tile; s = beta sqrt(U) / T; y = u / (s sqrt(T))
      float2 acc = make_float2(0.f, 0.f);
#pragma unroll
      for (int j = 0; j < 32; ++j) acc = fma2(p[j], p[j], acc);
      const float lane_u2 = acc.x + acc.y;
      const float U = tile_lane_sum(lane_u2, a.lanes_per_tile);
      const bool finite = isfinite(U);
      float s;
      bool over = false;
      __half s16;
      if constexpr (SF == LQ_SCALE_ROW_BF16) {
        s = __uint_as_float((uint32_t)reinterpret_cast<const unsigned short*>(M.scales)[cur.row] << 16);
      } else {
        s = a.beta * sqrtf(U) * a.inv_tile;
        if (!finite) s = 0.f;
        if constexpr (SF == LQ_SCALE_TILE_F16) {
          s16 = __float2half_rn(s);
          s = __half2float(s16);
          over = isinf(s);
          if (over) s = 0.f;
        }
      }
      if (!finite) {
#pragma unroll
        for (int j = 0; j < 32; ++j) p[j] = make_float2(0.f, 0.f);   // the tile's codes are zeros
      }
      float k = (s > 0.f) ? 1.0f / (s * a.sqrt_tile) : 0.f;

      int8_t* dst = M.codes + cur.row * M.cols + (int64_t)cur.chunk * kChunkCols;
      if constexpr (DITHER) {
        // y + u (u the dither draw of each element's counter row * cols + col)
        // for tiles with a scale; the decoders then see y with k = 1
        const float2 k2 = make_float2(k, k);
#pragma unroll
        for (int j = 0; j < 32; ++j) p[j] = mul2(p[j], k2);
        if (k > 0.f) {
          const uint64_t c_row = (uint64_t)cur.row * (uint64_t)M.cols + (uint64_t)cur.chunk * kChunkCols;
#pragma unroll
          for (int g = 0; g < 4; ++g) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              float u[8];
              dither8<LAT>(a.dither_seed, c_row + (uint64_t)block_col<EX>(lane, g, h), u);
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                if (h == 0) p[8 * g + i].x += u[i];
                else p[8 * g + i].y += u[i];
              }
            }
          }
        }
        k = 1.f;
      }

      // ---- decode.  Every |y| of the lane below 62.5 keeps every code inside
      // int8 and allows the packed fast decoders; the lane's sum of y^2 decides
      // that for free in most cases, the lane maximum otherwise.
      bool small = !DITHER && lane_u2 * (k * k) < 3906.25f;
      if (!small) {
        float mx = 0.f;
#pragma unroll
        for (int j = 0; j < 32; ++j) mx = fmaxf(mx, fmaxf(fabsf(p[j].x), fabsf(p[j].y)));
        small = mx * k < 62.5f;
      }
      const float2 k2 = make_float2(k, k);
      bool r = false;
      // Deferred tiles (float32 scales, no dither): a tile with a lane that
      // cannot use the packed decoders gets no codes here; fix_deferred redoes
      // it after the unit, from the input, with the range-checked decoders.
      // Called there, with the unit's registers dead, that decoder costs the
      // fast path nothing (inline in the decode it cost about 6 %).
      bool tile_deferred = false;
      if constexpr (kDeferTiles<LAT, SF, DITHER>) {
        if (__any_sync(0xffffffffu, !small)) tile_deferred = tile_lane_any(!small, a.lanes_per_tile);
      }
      if constexpr (LAT == LQ_E8 || LAT == LQ_Z1) {
        if (small) {
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            const float2 u[8] = {p[8 * g], p[8 * g + 1], p[8 * g + 2], p[8 * g + 3],
                                 p[8 * g + 4], p[8 * g + 5], p[8 * g + 6], p[8 * g + 7]};
            uint2 cP, cQ;
            if constexpr (LAT == LQ_E8) decode_e8_pair(u, k2, fixsel, cP, cQ);
            else decode_z1_pair(u, k2, cP, cQ);
            if (active) {
              *reinterpret_cast<uint2*>(dst + block_col<EX>(lane, g, 0)) = cP;
              *reinterpret_cast<uint2*>(dst + block_col<EX>(lane, g, 1)) = cQ;
            }
          }
        } else if constexpr (!kDeferTiles<LAT, SF, DITHER>) {
          float2 pc[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) pc[j] = p[j];
          decode_lane_checked<LAT, EX>(pc, k, lane, dst, active, r);
        }
      } else {
        // D4, A2: the scalar decoders, with the exact int8 range check unless
        // the lane is known to be small
#pragma unroll
        for (int g = 0; g < 4; ++g) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            float y[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) y[i] = (h ? p[8 * g + i].y : p[8 * g + i].x) * k;
            const float2 y4[4] = {make_float2(y[0], y[1]), make_float2(y[2], y[3]), make_float2(y[4], y[5]),
                                  make_float2(y[6], y[7])};
            uint2 w;
            if (small) w = decode_block8<LAT, false>(y4, r);
            else w = decode_block8<LAT, true>(y4, r);
            if (active) *reinterpret_cast<uint2*>(dst + block_col<EX>(lane, g, h)) = w;
          }
        }
      }

      if (active) {
        range |= r | over;
        nonfinite |= !finite;
        if ((lane & (a.lanes_per_tile - 1)) == 0) {
          const int64_t si = cur.row * M.tiles_per_row + (col0 >> a.tile_shift);
          if constexpr (SF == LQ_SCALE_TILE_F32) {
            if (!tile_deferred) reinterpret_cast<float*>(M.scales)[si] = s;
          }
          if constexpr (SF == LQ_SCALE_TILE_F16) reinterpret_cast<__half*>(M.scales)[si] = s16;
        }
      }
      if constexpr (kDeferTiles<LAT, SF, DITHER>) {
        const unsigned dm =
            __ballot_sync(0xffffffffu, tile_deferred && active && (lane & (a.lanes_per_tile - 1)) == 0);
        if (dm != 0u) fix_deferred<LAT, BF16, XL>(a, M, cur.row, cur.chunk, dm, lane, range);
      }
    }
    cur = nxt;
    st ^= 1;
  }
  // copies still in flight (only after a timeout) land before the CTA exits
  for (int s2 = 0; s2 < 2; ++s2)
    if (pending[s2]) mbar_wait_bounded(&bar[s2], (phase >> s2) & 1u, kQuantWaitCycles);
  if (__any_sync(0xffffffffu, range) && lane == 0) raise_flag(a.status, LQ_DEV_RANGE);
  if (__any_sync(0xffffffffu, nonfinite) && lane == 0) raise_flag(a.status, LQ_DEV_NONFINITE);
  if (__any_sync(0xffffffffu, timed_out) && lane == 0) raise_flag(a.status, LQ_DEV_TIMEOUT);
}

template <int LAT, bool BF16, int EX, bool XL, int SF, bool DITHER = false>
inline lq_status launch_quantize_ex(QuantArgs& a, cudaStream_t st) {
  constexpr int smem = QuantSmem<BF16>::kDynamic;
  static int per_sm = 0;
  if (per_sm == 0) {
    if (cudaFuncSetAttribute(quantize_kernel<LAT, BF16, EX, XL, SF, DITHER>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) {
      cudaGetLastError();
      return LQ_ERR_CUDA;
    }
    per_sm = occupancy_per_sm(quantize_kernel<LAT, BF16, EX, XL, SF, DITHER>, kQuantThreads, smem);
  }
  // a CTA count that is a multiple of every matrix's chunks per row keeps
  // each CTA on one chunk (one set of signs) within a matrix
  int64_t modulus = 1;
  for (int m = 0; m < a.n_mats; ++m) {
    const int64_t c = a.mat[m].chunks_per_row;
    int64_t x = modulus, y = c;
    while (y) {
      const int64_t t = x % y;
      x = y;
      y = t;
    }
    modulus = modulus / x * c;
    if (modulus > 64) { modulus = 1; break; }
  }
  const int grid = persistent_grid(a.cta_units, 1, (int)modulus, per_sm);
  if (grid <= 0) return LQ_ERR_CUDA;
  // programmatic dependent launch after the signs (or row-norm) kernel
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kQuantThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, quantize_kernel<LAT, BF16, EX, XL, SF, DITHER>, a) != cudaSuccess) {
    cudaGetLastError();
    return LQ_ERR_CUDA;
  }
  return LQ_OK;
}

template <int LAT, bool BF16, int SF, bool DITHER = false>
inline lq_status launch_quantize_walk(QuantArgs& a, cudaStream_t st) {
  lq_status r;
  if (a.lanes_per_tile == 2) r = launch_quantize_ex<LAT, BF16, 1, false, SF, DITHER>(a, st);
  else if (a.lanes_per_tile == 4) r = launch_quantize_ex<LAT, BF16, 2, false, SF, DITHER>(a, st);
  else r = launch_quantize_ex<LAT, BF16, 2, true, SF, DITHER>(a, st);

  return r;
}

// Launch with a 16-bit scale format (LQ_SCALE_ROW_BF16 or LQ_SCALE_TILE_F16),
// defined in lq_quantize_fmt.cu.
lq_status launch_quantize_scaled16(QuantArgs& a, int lattice, bool bf16, int sf, cudaStream_t st);

// Launch with the subtractive dither (scale format LQ_SCALE_TILE_F32 or
// LQ_SCALE_TILE_F16), defined in lq_quantize_dither.cu.
lq_status launch_quantize_dithered(QuantArgs& a, int lattice, bool bf16, int sf, cudaStream_t st);

}  // namespace lq
