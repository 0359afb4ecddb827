// The quantize kernel (tile RHT + lattice nearest point) and its launch
// templates, shared by the translation units that instantiate it
// (lq_quantize.cu: float32 tile scales, single and grouped walks;
// lq_quantize_fmt.cu: the 16-bit scale formats).
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
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "lq_device.cuh"
#include "lq_host.h"

namespace lq {

constexpr int kQuantMaxMats = LQ_QUANTIZE_MAX_GROUP;

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

// bf16 pair masks of one lane kept in shared memory: uint4 q of lane l at
// msk[q * 32 + l] holds the masks of column pairs 4q .. 4q+3 (conflict-free).
__device__ __forceinline__ void store_sign_masks(uint4* msk, int lane, const int8_t* signs_col0) {
  const uint4* p = reinterpret_cast<const uint4*>(signs_col0);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint4 v = __ldg(p + q);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      // sign words 2hh, 2hh+1 of this 16-byte run cover column pairs 8q + 4hh .. +3
      const uint32_t a = w[2 * hh], b = w[2 * hh + 1];
      msk[(2 * q + hh) * 32 + lane] = make_uint4(__byte_perm(a, 0u, 0x1404) & 0x80008000u,
                                                 __byte_perm(a, 0u, 0x3424) & 0x80008000u,
                                                 __byte_perm(b, 0u, 0x1404) & 0x80008000u,
                                                 __byte_perm(b, 0u, 0x3424) & 0x80008000u);
    }
  }
}

__device__ __forceinline__ void unpack_bf16_smem_signs(const LaneRaw<true>& r, const uint4* msk, int lane,
                                                       float2 (&p)[32]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint4 m = msk[i * 32 + lane];
    const uint32_t w[4] = {r.v[i].x ^ m.x, r.v[i].y ^ m.y, r.v[i].z ^ m.z, r.v[i].w ^ m.w};
#pragma unroll
    for (int h = 0; h < 4; ++h)
      p[4 * i + h] = make_float2(__uint_as_float(w[h] << 16), __uint_as_float(w[h] & 0xFFFF0000u));
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

// ------------------------------------------------------------------ staging
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait0() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// ------------------------------------------------------------------ quantize
// One matrix of a quantize launch.  Its warp units (row, 2048-column chunk)
// are numbered row * chunks_per_row + chunk and taken four at a time by the
// four warps of a CTA: CTA unit k of the matrix (global CTA unit cta_begin + k)
// holds warp units 4k .. 4k + 3, those past the matrix's end doing nothing.
// The grid strides over CTA units, so every warp of a CTA is always in the
// same matrix.  A warp unit's row is local / chunks_per_row, computed as the
// high half of local * cpr_recip with cpr_recip = ceil(2^64 / chunks_per_row)
// (exact for every local below 2^64 / chunks_per_row; 0 marks one chunk per
// row), so the kernel divides nothing.
struct QuantMat {
  const void* W;
  int8_t* codes;
  float* scales;
  const int8_t* signs;
  int64_t rows, cols, ldw;
  int64_t cta_begin;
  uint64_t cpr_recip;
  int tiles_per_row, chunks_per_row;
};

struct QuantArgs {
  QuantMat mat[kQuantMaxMats];
  int n_mats;
  int tile, tile_shift, lanes_per_tile;
  float beta, sqrt_tile, inv_tile;
  int32_t* status;
  int64_t cta_units;  // CTA units of all matrices
  uint64_t dither_seed;   // subtractive dither (DITHER instantiations only)
};

constexpr int kQuantThreads = 128;

// Shared memory per warp: two stages of raw input (each lane copies its own
// 64 columns with cp.async and later reads back only its own copies) and, for
// bf16, the lane's sign masks.  Once a stage has been read into registers it
// doubles as the buffer of the butterfly exchange below, so a stage holds at
// least the exchange's 284 16-byte slots.
template <bool BF16> struct QuantSmem {
  static constexpr int kRawVec = BF16 ? 8 : 16;             // 16-byte vectors per lane per stage
  static constexpr int kStageVec = BF16 ? 288 : 512;        // uint4 per warp per stage
  static constexpr int kRawWords = 2 * kStageVec;           // uint4 per warp, both stages
  static constexpr int kMaskWords = BF16 ? 8 * 32 : 0;      // uint4 per warp
  static constexpr int kPerWarp = kRawWords + kMaskWords;
};

// Butterfly stages of tile bits 6 .. 6+MP-1 without shuffles.  After the six
// register stages, lane bits 0 .. MP-1 of a lane hold tile bits 6 .. and its
// register index bits 3 .. 3+MP-1 hold tile bits 3 ..; one pass through shared
// memory swaps the two, so those stages run in registers as well and every
// 8-coordinate block (tile bits 0 .. 2) stays in one lane.  The pass goes in
// two halves (register bit 2) of 32 values per lane.  Slot of the value with
// lane group G, spectator register bits ux, lane bits a and register bits c:
//   (G >> (3 - MP)) * kBlk + ux * kUxSpan + (G & (X - 1)) * Q + a + 9 c,
// additive in a and c, so every access is a per-lane base plus a constant,
// and conflict-free for 16-byte accesses both when a varies (writes) and when
// c varies (reads): the slots of the 8 lanes of a phase differ modulo 8.
template <int MP> struct Xchg {
  static constexpr int Q = 1 << MP;          // lanes whose bits are swapped
  static constexpr int X = 8 >> MP;          // spectator register values per half
  static constexpr int kUxSpan = 9 * Q - 1;
  static constexpr int kBlk = X * kUxSpan;
  static constexpr int kSlots = 4 * kBlk;
};
static_assert(Xchg<2>::kSlots <= 288 && Xchg<3>::kSlots <= 288, "exchange slots");

template <int MP>
__device__ __forceinline__ void exchange_tile_bits(float2 (&p)[32], uint32_t buf, int lane) {
  using XC = Xchg<MP>;
  const int q = lane & (XC::Q - 1), G = lane >> MP;
  const uint32_t g = (uint32_t)((G >> (3 - MP)) * XC::kBlk + (G & (XC::X - 1)) * XC::Q);
  const uint32_t wb = buf + (g + (uint32_t)q) * 16u;
  const uint32_t rb = buf + (g + 9u * (uint32_t)q) * 16u;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    __syncwarp();
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const uint32_t off = (uint32_t)(((u >> MP) * XC::kUxSpan + 9 * (u & (XC::Q - 1))) * 16);
      const float2 v0 = p[4 * u + 2 * h], v1 = p[4 * u + 2 * h + 1];
      asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(wb + off), "f"(v0.x), "f"(v0.y),
                   "f"(v1.x), "f"(v1.y) : "memory");
    }
    __syncwarp();
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const uint32_t off = (uint32_t)(((u >> MP) * XC::kUxSpan + (u & (XC::Q - 1))) * 16);
      float2 v0, v1;
      asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v0.x), "=f"(v0.y), "=f"(v1.x), "=f"(v1.y)
                   : "r"(rb + off) : "memory");
      p[4 * u + 2 * h] = v0;
      p[4 * u + 2 * h + 1] = v1;
    }
  }
  __syncwarp();
  // the swapped tile bits now sit in register index bits 3 .. 3+MP-1 (float2 bits 2 ..)
#pragma unroll
  for (int hp = 4; hp < (4 << MP); hp <<= 1) {
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

// GROUPED = false: one matrix (a.mat[0]); a warp takes warp units w, w + W,
// w + 2W, ... (W = warps of the grid), advanced without divisions.
// GROUPED = true: the CTA-unit walk over several matrices described above.
// Both walks feed the same per-unit body; they are separate instantiations
// because the single-matrix walk keeps fewer values live across the decode.
// Residency: 4 CTAs per SM (128 registers) for the single-matrix walk, 3 (168
// registers) for the grouped walk -- each measured faster than the other
// choice for its walk.
// DITHER: subtractive dither (lq_device.cuh) added to y before the decode.
template <int LAT, bool BF16, int MP, bool GROUPED, int SF, bool DITHER = false>
__global__ void __launch_bounds__(kQuantThreads, GROUPED ? 3 : 4) quantize_kernel(QuantArgs a) {
  static_assert(!GROUPED || SF == LQ_SCALE_TILE_F32, "grouped calls store float32 tile scales");
  static_assert(!(GROUPED && DITHER), "the dither runs on the single-matrix walk");
  using SM = QuantSmem<BF16>;
  extern __shared__ uint4 quant_smem[];
  const int lane = threadIdx.x & 31;
  uint4* wsm = quant_smem + (threadIdx.x >> 5) * SM::kPerWarp;
  uint4* raw_sm = wsm;                          // [stage][vec][lane]
  uint4* msk = wsm + SM::kRawWords;             // bf16 sign masks [q][lane]
  const uint32_t raw_s = (uint32_t)__cvta_generic_to_shared(raw_sm);
  constexpr int kElemBytes = BF16 ? 2 : 4;

  LaneSigns<false> sg;     // fp32 input keeps its 64 sign bits in registers
  int cached_chunk = -1, cached_m = -1;
  bool range = false, nonfinite = false;

  // copy the lane's 64 input columns of unit (row, chunk) of M into stage st
  auto stage_in = [&](bool valid, const QuantMat& M, int64_t row, int chunk, int st) {
    const int64_t c = (int64_t)chunk * kChunkCols + (int64_t)lane * kLaneElems;
    if (valid && row < M.rows && c < M.cols) {
      const char* src = reinterpret_cast<const char*>(M.W) + (row * M.ldw + c) * kElemBytes;
#pragma unroll
      for (int i = 0; i < SM::kRawVec; ++i)
        cp_async16(raw_s + (uint32_t)((st * SM::kStageVec + i * 32 + lane) * 16), src + 16 * i);
    }
    cp_async_commit();
  };

  // quantize unit (row, chunk) of matrix m, whose input is in stage st
  auto process = [&](const QuantMat& M, int m, int64_t row, int chunk, int st) {
    const int64_t col0 = (int64_t)chunk * kChunkCols + (int64_t)lane * kLaneElems;
    const bool active = col0 < M.cols;
    if (chunk != cached_chunk || m != cached_m) {
      if constexpr (BF16) {
        if (active) store_sign_masks(msk, lane, M.signs + col0);
      } else {
        sg.bits[0] = 0;
        sg.bits[1] = 0;
        if (active) load_signs<false>(sg, M.signs + col0);
      }
      cached_chunk = chunk;
      cached_m = m;
    }
    cp_async_wait1();   // this unit's copies have landed

    float2 p[32];
    {
      LaneRaw<BF16> raw;
#pragma unroll
      for (int i = 0; i < SM::kRawVec; ++i) raw.v[i] = raw_sm[st * SM::kStageVec + i * 32 + lane];
      if constexpr (BF16) unpack_bf16_smem_signs(raw, msk, lane, p);
      else unpack_signed<false>(raw, sg, p);
    }
    fwht64_local(p);
    if constexpr (MP > 0) exchange_tile_bits<MP>(p, raw_s + (uint32_t)(st * SM::kStageVec * 16), lane);
    // lane bits not exchanged (MP = 0: all of them; tiles of 1024 and 2048
    // columns: tile bits 9 .. on lane bits 3 ..) cross lanes with shuffles
    for (int mm = (MP == 0 ? 1 : 8); mm < a.lanes_per_tile; mm <<= 1) {
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

    // U = sum u^2 over the tile; s = beta sqrt(U) / T; y = u / (s sqrt(T))
    float2 acc = make_float2(0.f, 0.f);
#pragma unroll
    for (int j = 0; j < 32; ++j) acc = fma2(p[j], p[j], acc);
    const float U = tile_lane_sum(acc.x + acc.y, a.lanes_per_tile);
    const bool finite = isfinite(U);
    // s: the value of the stored scale (the codes are decoded against it)
    float s;
    bool over = false;
    __half s16;
    if constexpr (SF == LQ_SCALE_ROW_BF16) {
      // written by the row-norm kernel that precedes this one
      s = __uint_as_float((uint32_t)reinterpret_cast<const unsigned short*>(M.scales)[row] << 16);
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
    const float k = (s > 0.f) ? 1.0f / (s * a.sqrt_tile) : 0.f;
    const float2 k2 = make_float2(k, k);
#pragma unroll
    for (int j = 0; j < 32; ++j) p[j] = mul2(p[j], k2);

    constexpr int Q = 1 << MP;
    if constexpr (DITHER) {
      // y + u for tiles with a scale (a zero scale keeps y = 0 and zero codes);
      // register block g holds the 8 columns 8 q + 8 Q gx + 64 ga (see the store)
      if (k > 0.f) {
        const uint64_t c_row = (uint64_t)row * (uint64_t)M.cols + (uint64_t)chunk * kChunkCols +
                               (uint64_t)((lane >> MP) * (64 * Q) + 8 * (lane & (Q - 1)));
#pragma unroll
        for (int gb = 0; gb < 8; ++gb) {
          float u[8];
          dither8<LAT>(a.dither_seed, c_row + (uint64_t)((gb >> MP) * (8 * Q) + 64 * (gb & (Q - 1))), u);
#pragma unroll
          for (int h = 0; h < 4; ++h) p[4 * gb + h] = add2(p[4 * gb + h], make_float2(u[2 * h], u[2 * h + 1]));
        }
      }
    }
    // every |y| of the lane below 62.5 keeps every code inside int8, and the
    // per-block range check is left out; the lane's sum of y^2 decides that
    // for free in most cases (not with a dither, which moves y), the lane
    // maximum otherwise
    const float lane_y2 = (acc.x + acc.y) * (k * k);
    bool small = !DITHER && lane_y2 < 3906.25f;
    if (!small) {
      float mx = 0.f;
#pragma unroll
      for (int j = 0; j < 32; ++j) mx = fmaxf(mx, fmaxf(fabsf(p[j].x), fabsf(p[j].y)));
      small = mx < 62.5f;
    }
    uint32_t w[16];
    bool r = false;
    if (small) decode_lane<LAT, false>(p, w, r);
    else decode_lane<LAT, true>(p, w, r);

    if (active) {
      range |= r | over;
      nonfinite |= !finite;
      // register block u holds tile columns 8 q + 8 Q ux + 64 a (q = lane bits,
      // ux = u >> MP, a = u & (Q - 1)) of the tile group G = lane >> MP
      int8_t* dst = M.codes + row * M.cols + (int64_t)chunk * kChunkCols + (lane >> MP) * (64 * Q) +
                    8 * (lane & (Q - 1));
#pragma unroll
      for (int u = 0; u < 8; ++u)
        *reinterpret_cast<uint2*>(dst + (u >> MP) * (8 * Q) + 64 * (u & (Q - 1))) = make_uint2(w[2 * u], w[2 * u + 1]);
      if ((lane & (a.lanes_per_tile - 1)) == 0) {
        const int64_t si = row * M.tiles_per_row + (col0 >> a.tile_shift);
        if constexpr (SF == LQ_SCALE_TILE_F32) M.scales[si] = s;
        if constexpr (SF == LQ_SCALE_TILE_F16) reinterpret_cast<__half*>(M.scales)[si] = s16;
      }
    }
  };

  int stage = 0;
  if constexpr (!GROUPED) {
    const QuantMat& M = a.mat[0];
    const int64_t warp0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    // unit u = row * chunks_per_row + chunk grows by nwarps per step
    const int64_t d_row = nwarps / M.chunks_per_row;
    const int d_chunk = (int)(nwarps % M.chunks_per_row);
    int64_t row = warp0 / M.chunks_per_row;
    int chunk = (int)(warp0 % M.chunks_per_row);
    stage_in(true, M, row, chunk, 0);
    // the signs come from the kernel launched just before this one
    asm volatile("griddepcontrol.wait;" ::: "memory");
    while (row < M.rows) {
      int64_t nrow = row + d_row;
      int nchunk = chunk + d_chunk;
      if (nchunk >= M.chunks_per_row) { nchunk -= M.chunks_per_row; ++nrow; }
      stage_in(true, M, nrow, nchunk, stage ^ 1);
      process(M, 0, row, chunk, stage);
      row = nrow;
      chunk = nchunk;
      stage ^= 1;
    }
  } else {
    // (matrix, row, chunk) of a CTA unit's warp unit for this warp
    struct Pos {
      int m, chunk;
      int64_t row;
    };
    const int wic = threadIdx.x >> 5;   // warp in the CTA
    auto locate = [&](int64_t cu, Pos& p) {
      while (p.m + 1 < a.n_mats && cu >= a.mat[p.m + 1].cta_begin) ++p.m;
      const QuantMat& M = a.mat[p.m];
      const uint64_t local = (uint64_t)(cu - M.cta_begin) * (kQuantThreads / 32) + (uint64_t)wic;
      const uint64_t r = M.cpr_recip ? __umul64hi(local, M.cpr_recip) : local;
      p.row = (int64_t)r;
      p.chunk = (int)(local - r * (uint64_t)M.chunks_per_row);
    };
    int64_t cu = blockIdx.x;
    Pos cur;
    cur.m = 0;
    cur.row = 0;
    cur.chunk = 0;
    if (cu < a.cta_units) locate(cu, cur);
    stage_in(cu < a.cta_units, a.mat[cur.m], cur.row, cur.chunk, 0);
    asm volatile("griddepcontrol.wait;" ::: "memory");
    for (; cu < a.cta_units; cu += gridDim.x) {
      const int64_t cn = cu + gridDim.x;
      Pos nxt = cur;
      if (cn < a.cta_units) locate(cn, nxt);
      stage_in(cn < a.cta_units, a.mat[nxt.m], nxt.row, nxt.chunk, stage ^ 1);
      const QuantMat& M = a.mat[cur.m];
      if (cur.row < M.rows) process(M, cur.m, cur.row, cur.chunk, stage);   // else past the matrix's end
      cur = nxt;
      stage ^= 1;
    }
  }
  cp_async_wait0();
  if (__any_sync(0xffffffffu, range) && lane == 0) raise_flag(a.status, LQ_DEV_RANGE);
  if (__any_sync(0xffffffffu, nonfinite) && lane == 0) raise_flag(a.status, LQ_DEV_NONFINITE);
}

inline int64_t gcd64(int64_t x, int64_t y) {
  while (y) {
    const int64_t t = x % y;
    x = y;
    y = t;
  }
  return x;
}

template <int LAT, bool BF16, int MP, bool GROUPED, int SF, bool DITHER = false>
inline lq_status launch_quantize_mp(QuantArgs& a, cudaStream_t st) {
  constexpr size_t smem = (size_t)(kQuantThreads / 32) * QuantSmem<BF16>::kPerWarp * sizeof(uint4);
  static int per_sm = 0;
  if (per_sm == 0) {
    if (cudaFuncSetAttribute(quantize_kernel<LAT, BF16, MP, GROUPED, SF, DITHER>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) {
      cudaGetLastError();
      return LQ_ERR_CUDA;
    }
    per_sm = occupancy_per_sm(quantize_kernel<LAT, BF16, MP, GROUPED, SF, DITHER>, kQuantThreads, smem);
  }
  // a warp count that is a multiple of every matrix's chunks per row keeps
  // each warp on one chunk (one set of signs) within a matrix
  int64_t modulus = 1;
  for (int m = 0; m < a.n_mats; ++m) {
    const int64_t c = a.mat[m].chunks_per_row;
    modulus = modulus / gcd64(modulus, c) * c;
    if (modulus > 64) { modulus = 1; break; }
  }
  const int grid = persistent_grid(a.cta_units * (kQuantThreads / 32), kQuantThreads / 32, (int)modulus, per_sm);
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
  if (cudaLaunchKernelEx(&cfg, quantize_kernel<LAT, BF16, MP, GROUPED, SF, DITHER>, a) != cudaSuccess) {
    cudaGetLastError();
    return LQ_ERR_CUDA;
  }
  return LQ_OK;
}

// MP = tile bits exchanged through shared memory: log2(tile / 64), at most 3.
// A 128-column tile has a single cross-lane stage, cheaper as a shuffle (MP = 0).
template <int LAT, bool BF16, bool GROUPED, int SF, bool DITHER = false>
inline lq_status launch_quantize_walk(QuantArgs& a, cudaStream_t st) {
  if (a.lanes_per_tile == 2) return launch_quantize_mp<LAT, BF16, 0, GROUPED, SF, DITHER>(a, st);
  if (a.lanes_per_tile == 4) return launch_quantize_mp<LAT, BF16, 2, GROUPED, SF, DITHER>(a, st);
  return launch_quantize_mp<LAT, BF16, 3, GROUPED, SF, DITHER>(a, st);
}

// Launch of the single-matrix walk with a 16-bit scale format
// (LQ_SCALE_ROW_BF16 or LQ_SCALE_TILE_F16), defined in lq_quantize_fmt.cu.
lq_status launch_quantize_scaled16(QuantArgs& a, int lattice, bool bf16, int sf, cudaStream_t st);

// Launch of the single-matrix walk with the subtractive dither (scale format
// LQ_SCALE_TILE_F32 or LQ_SCALE_TILE_F16), defined in lq_quantize_dither.cu.
lq_status launch_quantize_dithered(QuantArgs& a, int lattice, bool bf16, int sf, cudaStream_t st);

}  // namespace lq
