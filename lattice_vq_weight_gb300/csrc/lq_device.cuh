// Device building blocks shared by the liblq kernels: packed fp32 pair
// arithmetic, the per-lane/ cross-lane fast Walsh-Hadamard transform, and the
// nearest-point decoders of the E8, D4, A2 and Z1 lattices.
//
// Data layout used by every kernel that rotates a 2048-column chunk of a row:
// lane l of a warp owns the 64 consecutive columns [64 l, 64 l + 64) of the
// chunk, held as float2 p[32] (p[j] = columns 2j, 2j+1).  A tile of T columns
// is spread over T/64 consecutive lanes, so the Hadamard index bits 0..5 live
// in registers and bits 6.. in the lane index.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>

#include "lq.h"

namespace lq {

constexpr int kWarp = 32;
constexpr int kLaneElems = 64;                  // columns owned by one lane
constexpr int kChunkCols = kWarp * kLaneElems;  // 2048 columns per warp unit

// x + 1.5 * 2^23 rounds x (|x| < 2^22) to the nearest integer, ties to even,
// and leaves that integer in the low mantissa bits: bits = 0x4B400000 + rint(x).
constexpr float kRoundMagic = 12582912.0f;
constexpr uint32_t kRoundMagicBits = 0x4B400000u;

// ---------------------------------------------------------------- f32x2 ops
// sm_100+ packed fp32 pair arithmetic (one instruction for two lanes of work).
__device__ __forceinline__ unsigned long long as_u64(float2 a) {
  return *reinterpret_cast<unsigned long long*>(&a);
}
__device__ __forceinline__ float2 as_f2(unsigned long long a) {
  return *reinterpret_cast<float2*>(&a);
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
  unsigned long long r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(as_u64(a)), "l"(as_u64(b)));
  return as_f2(r);
}
__device__ __forceinline__ float2 sub2(float2 a, float2 b) {
  unsigned long long r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(as_u64(a)), "l"(as_u64(b)));
  return as_f2(r);
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
  unsigned long long r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(as_u64(a)), "l"(as_u64(b)));
  return as_f2(r);
}
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  unsigned long long r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(as_u64(a)), "l"(as_u64(b)), "l"(as_u64(c)));
  return as_f2(r);
}

// ---------------------------------------------------------------- status word
__device__ __forceinline__ void raise_flag(int32_t* status, int32_t bit) {
  if (status != nullptr) atomicOr(status, bit);
}

// ---------------------------------------------------------------- FWHT
// Unnormalised Walsh-Hadamard transform (Sylvester order, entry
// (-1)^popcount(i & j)) of the 64 register-resident columns: 6 butterfly
// stages, the first inside each float2, the rest between float2 pairs.
__device__ __forceinline__ void fwht64_local(float2 (&p)[32]) {
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const float a = p[j].x, b = p[j].y;
    p[j] = make_float2(a + b, a - b);
  }
#pragma unroll
  for (int hp = 1; hp < 32; hp <<= 1) {
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      if ((j & hp) == 0) {
        const float2 a = p[j], b = p[j + hp];
        p[j] = add2(a, b);
        p[j + hp] = sub2(a, b);
      }
    }
  }
}

// Remaining butterfly stages across the lanes of one tile: the partner of lane
// l in the stage for index bit 6 + log2(m) is lane l ^ m.  The lane whose bit
// is clear keeps a + b, the other keeps a - b (a = lower index).
__device__ __forceinline__ void fwht_cross_lanes(float2 (&p)[32], int lanes_per_tile, int lane) {
  for (int m = 1; m < lanes_per_tile; m <<= 1) {
    const float sg = (lane & m) ? -1.0f : 1.0f;
    const float2 sg2 = make_float2(sg, sg);
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      float2 q;
      q.x = __shfl_xor_sync(0xffffffffu, p[j].x, m);
      q.y = __shfl_xor_sync(0xffffffffu, p[j].y, m);
      p[j] = fma2(p[j], sg2, q);
    }
  }
}

// Sum over the lanes of one tile (lanes_per_tile is a power of two <= 32).
__device__ __forceinline__ float tile_lane_sum(float v, int lanes_per_tile) {
  for (int m = 1; m < lanes_per_tile; m <<= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
  return v;
}
__device__ __forceinline__ float tile_lane_max(float v, int lanes_per_tile) {
  for (int m = 1; m < lanes_per_tile; m <<= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, m));
  return v;
}

// Unnormalised Walsh-Hadamard transform of one tile spread over `lpt`
// consecutive lanes (lpt a power of two <= 32) holding E consecutive columns
// each: log2(E) register stages, then log2(lpt) shuffle stages.  Used for
// activations (E = 16 up to 512-column tiles, E = T/32 above), where a short
// dependent chain matters more than lanes.
template <int E>
__device__ __forceinline__ void fwht_tile(float (&v)[E], int lpt, int lane) {
#pragma unroll
  for (int h = 1; h < E; h <<= 1)
#pragma unroll
    for (int c = 0; c < E; ++c)
      if ((c & h) == 0) {
        const float x0 = v[c], x1 = v[c + h];
        v[c] = x0 + x1;
        v[c + h] = x0 - x1;
      }
  for (int m = 1; m < lpt; m <<= 1) {
    const float sgn = (lane & m) ? -1.0f : 1.0f;
#pragma unroll
    for (int c = 0; c < E; ++c) v[c] = fmaf(v[c], sgn, __shfl_xor_sync(0xffffffffu, v[c], m));
  }
}

// E consecutive bf16 (or fp32) activations with the column signs applied (exact).
template <int E>
__device__ __forceinline__ void apply_signs(const int8_t* signs, float (&v)[E]) {
#pragma unroll
  for (int q = 0; q < E / 16; ++q) {
    const uint4 sw = __ldg(reinterpret_cast<const uint4*>(signs) + q);
    const uint32_t sg[4] = {sw.x, sw.y, sw.z, sw.w};
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      const uint32_t sbit = ((sg[c >> 2] >> (8 * (c & 3) + 7)) & 1u) << 31;
      v[16 * q + c] = __uint_as_float(__float_as_uint(v[16 * q + c]) ^ sbit);
    }
  }
}
template <int E>
__device__ __forceinline__ void load_bf16_signed(const void* src, const int8_t* signs, float (&v)[E]) {
  const uint4* p = reinterpret_cast<const uint4*>(src);
#pragma unroll
  for (int i = 0; i < E / 8; ++i) {
    const uint4 q = __ldg(p + i);
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      v[8 * i + 2 * h] = __uint_as_float(w[h] << 16);
      v[8 * i + 2 * h + 1] = __uint_as_float(w[h] & 0xFFFF0000u);
    }
  }
  apply_signs<E>(signs, v);
}
template <int E>
__device__ __forceinline__ void load_f32_signed(const void* src, const int8_t* signs, float (&v)[E]) {
  const float4* p = reinterpret_cast<const float4*>(src);
#pragma unroll
  for (int i = 0; i < E / 4; ++i) {
    const float4 q = __ldg(p + i);
    v[4 * i] = q.x; v[4 * i + 1] = q.y; v[4 * i + 2] = q.z; v[4 * i + 3] = q.w;
  }
  apply_signs<E>(signs, v);
}

// Columns per thread for the activation transforms: a tile must fit one warp.
__host__ __device__ constexpr int act_elems_for_tile(int tile) { return tile <= 512 ? 16 : tile / 32; }

// ---------------------------------------------------------------- scales
// Stored scale of (row, tile t) in one of the LQ_SCALE_* formats (lq.h):
// float32 [rows x tiles], bfloat16 [rows] or float16 [rows x tiles].
__device__ __forceinline__ float load_scale(const void* base, int fmt, int64_t row, int64_t t,
                                            int64_t tiles_per_row) {
  if (fmt == LQ_SCALE_ROW_BF16)
    return __uint_as_float((uint32_t)__ldg(reinterpret_cast<const unsigned short*>(base) + row) << 16);
  if (fmt == LQ_SCALE_TILE_F16)
    return __half2float(__ldg(reinterpret_cast<const __half*>(base) + row * tiles_per_row + t));
  return __ldg(reinterpret_cast<const float*>(base) + row * tiles_per_row + t);
}

// The same with the format fixed at compile time (for hot loops).
template <int SF>
__device__ __forceinline__ float load_scale_t(const void* base, int64_t row, int64_t t, int64_t tiles_per_row) {
  if constexpr (SF == LQ_SCALE_ROW_BF16)
    return __uint_as_float((uint32_t)__ldg(reinterpret_cast<const unsigned short*>(base) + row) << 16);
  else if constexpr (SF == LQ_SCALE_TILE_F16)
    return __half2float(__ldg(reinterpret_cast<const __half*>(base) + row * tiles_per_row + t));
  else
    return __ldg(reinterpret_cast<const float*>(base) + row * tiles_per_row + t);
}

// ---------------------------------------------------------------- code packing
// Low bytes of four ints into one word (byte i = low byte of ci).
__device__ __forceinline__ uint32_t pack4(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3) {
  return __byte_perm(__byte_perm(c0, c1, 0x0040), __byte_perm(c2, c3, 0x0040), 0x5410);
}

// Add `step` (+-2) to byte k (0..7) of the code pair (w0: bytes 0-3, w1: 4-7)
// when `fix` is set.  Bytes are moved to offset binary first so that the add
// cannot carry into a neighbour unless the code itself leaves int8, which the
// range check reports.
__device__ __forceinline__ void add_to_byte(uint32_t& w0, uint32_t& w1, bool fix, int k, int step) {
  const uint32_t delta = fix ? (uint32_t)(step * (1 << (8 * (k & 3)))) : 0u;
  const uint32_t d0 = (k < 4) ? delta : 0u;
  const uint32_t d1 = (k < 4) ? 0u : delta;
  w0 = ((w0 ^ 0x80808080u) + d0) ^ 0x80808080u;
  w1 = ((w1 ^ 0x80808080u) + d1) ^ 0x80808080u;
}

// ---------------------------------------------------------------- decoders
// Each decoder takes the scaled coordinates y of one lattice block and writes
// the int8 codes (doubled coordinates).  Rounding is x + kRoundMagic, which is
// round-half-even; for f = rint(y), e = y - f is exact and bits(t) - 0x4B400000
// is f as an integer.
//
// Worst-coordinate search packs (|e|, index, sign) into one integer key:
// rotl(bits(e), 1) moves the sign to bit 0 and keeps |e| monotone in bits
// 4..31 (|e| <= 1/2, so the top bit is clear); bits 1..3 hold the index,
// ordered so that ties of |e| (to 2^-20 relative) go to the lowest index.
//
// Range: a code is 2 rint(y) plus at most 3 in magnitude, so a block whose
// coordinates all satisfy |y| < 62.5 cannot leave int8.  Blocks above that
// recompute their codes as 32-bit integers and report |code| > 127.

struct BlockCodes8 { uint32_t w0, w1; };

// Keys are non-negative floats when their bit patterns are read as fp32 (bit
// 31 is clear and the exponent field never reaches 255), so the three-input
// float min/max of sm_100+ orders them exactly like unsigned integers.
__device__ __forceinline__ uint32_t key_max3(uint32_t a, uint32_t b, uint32_t c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(__uint_as_float(a)), "f"(__uint_as_float(b)), "f"(__uint_as_float(c)));
  return __float_as_uint(r);
}
__device__ __forceinline__ uint32_t key_min3(uint32_t a, uint32_t b, uint32_t c) {
  float r;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(__uint_as_float(a)), "f"(__uint_as_float(b)), "f"(__uint_as_float(c)));
  return __float_as_uint(r);
}

__device__ __forceinline__ int rint_int(uint32_t tbits) { return (int)(tbits - kRoundMagicBits); }

// E8 = D8 u (D8 + 1/2).  Coset D8: f = rint(y), parity of sum(f), fix the
// coordinate with the largest |e| when odd.  Coset D8 + 1/2 shares the
// rounding: rint(y - 1/2) + 1/2 = f + copysign(1/2, e), residual
// e' = e - copysign(1/2, e), |e'| = 1/2 - |e|, and its parity differs from
// sum(f) by the number of negative e.  So
//   dA = sum e^2              (+ 1 - 2 max|e| when sum f is odd)
//   dB = sum e^2 + 2 - sum|e| (+ 2 min|e|     when sum f + #neg is odd)
// and the D8 candidate is kept when dA <= dB.
// a * b + c on the integer multiply-add path
__device__ __forceinline__ uint32_t imad(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t r;
  asm("mad.lo.u32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
  return r;
}

template <bool CHECK>
__device__ __forceinline__ BlockCodes8 decode_e8(const float2 (&y)[4], bool& range) {
  const float2 M2 = make_float2(kRoundMagic, kRoundMagic);
  float2 t[4], e[4];
  float2 sq = make_float2(0.f, 0.f);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    t[j] = add2(y[j], M2);
    e[j] = sub2(y[j], sub2(t[j], M2));
    sq = fma2(e[j], e[j], sq);
  }
  const float dA0 = sq.x + sq.y;
  uint32_t px = 0, sx = 0, key[8];
  float sabs = 0.f;
  uint32_t tb[8], eb[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float ei = (i & 1) ? e[i >> 1].y : e[i >> 1].x;
    tb[i] = __float_as_uint((i & 1) ? t[i >> 1].y : t[i >> 1].x);
    eb[i] = __float_as_uint(ei);
    px ^= tb[i];
    sx ^= eb[i];
    sabs += fabsf(ei);
    const uint32_t rot = __funnelshift_l(eb[i], eb[i], 1);
    key[i] = (rot & 0xFFFFFFF1u) | (uint32_t)((7 - i) << 1);
  }
  // One key per coordinate serves both searches: the largest key is the worst
  // D8 residual (lowest index on ties); the smallest is the worst D8+1/2
  // residual (highest index on exact ties -- an equally distant point).
  const uint32_t keyA = max(key_max3(key[0], key[1], key[2]), key_max3(key[3], key[4], key_max3(key[5], key[6], key[7])));
  const uint32_t keyB = min(key_min3(key[0], key[1], key[2]), key_min3(key[3], key[4], key_min3(key[5], key[6], key[7])));
  const bool oddA = (px & 1u) != 0;
  const bool oddB = ((px ^ (sx >> 31)) & 1u) != 0;
  const float maxe = __uint_as_float((keyA >> 1) & 0x7FFFFFF8u);
  const float mine = __uint_as_float((keyB >> 1) & 0x7FFFFFF8u);
  const float dA = oddA ? dA0 + fmaf(-2.f, maxe, 1.f) : dA0;
  const float dB = (dA0 + 2.f - sabs) + (oddB ? 2.f * mine : 0.f);
  const bool takeB = dB < dA;
  // code byte: 2 f for D8; for D8 + 1/2, 2 f + 1 - 2 [e < 0] (the sign of e is
  // bit 0 of the key) -- built with two multiply-adds
  const uint32_t bs = takeB ? 1u : 0u;
  uint32_t c[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) c[i] = imad(tb[i], 2u, imad(key[i] & bs, 0xFFFFFFFEu, bs));
  BlockCodes8 r;
  r.w0 = pack4(c[0], c[1], c[2], c[3]);
  r.w1 = pack4(c[4], c[5], c[6], c[7]);
  // parity fix of the chosen coset
  const uint32_t kk = takeB ? keyB : keyA;
  const int k = 7 - (int)((kk >> 1) & 7u);
  const bool neg = (kk & 1u) != 0;
  // D8: rounding the other way moves toward y, +1 when e >= 0.
  // D8 + 1/2: e' = e - copysign(1/2, e) has the opposite sign of e.
  const int step = takeB ? (neg ? 2 : -2) : (neg ? -2 : 2);
  const bool fix = takeB ? oddB : oddA;
  add_to_byte(r.w0, r.w1, fix, k, step);
  if constexpr (CHECK) {
    float bmax = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) bmax = fmaxf(bmax, fmaxf(fabsf(y[j].x), fabsf(y[j].y)));
    if (!(bmax < 62.5f)) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int adj = takeB ? (((int32_t)eb[i] >> 31) | 1) : 0;
        const int ci = 2 * rint_int(tb[i]) + adj + ((fix && i == k) ? step : 0);
        range |= (ci > 127) || (ci < -127);
      }
    }
  }
  return r;
}

// D4 = {x in Z^4 : sum even}: round, fix the worst coordinate when odd.
template <bool CHECK>
__device__ __forceinline__ uint32_t decode_d4(const float2 (&y)[2], bool& range) {
  const float2 M2 = make_float2(kRoundMagic, kRoundMagic);
  uint32_t tb[4], px = 0, keyA = 0;
  float bmax = 0.f;
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const float2 t = add2(y[j], M2);
    const float2 e = sub2(y[j], sub2(t, M2));
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int i = 2 * j + h;
      tb[i] = __float_as_uint(h ? t.y : t.x);
      const uint32_t eb = __float_as_uint(h ? e.y : e.x);
      px ^= tb[i];
      bmax = fmaxf(bmax, fabsf(h ? y[j].y : y[j].x));
      const uint32_t rot = __funnelshift_l(eb, eb, 1);
      keyA = max(keyA, (rot & 0xFFFFFFF1u) | (uint32_t)((7 - i) << 1));
    }
  }
  uint32_t w = pack4(tb[0] + tb[0], tb[1] + tb[1], tb[2] + tb[2], tb[3] + tb[3]);
  uint32_t unused = 0;
  const int k = 7 - (int)((keyA >> 1) & 7u);
  const int step = (keyA & 1u) ? -2 : 2;
  const bool fix = (px & 1u) != 0;
  add_to_byte(w, unused, fix, k, step);
  if (CHECK && !(bmax < 62.5f)) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int ci = 2 * rint_int(tb[i]) + ((fix && i == k) ? step : 0);
      range |= (ci > 127) || (ci < -127);
    }
  }
  return w;
}

// A2 = R u (R + (1/2, sqrt3/2)), R = Z x sqrt3 Z.  In the coordinates
// (y0, z = y1/sqrt3) both cosets are integer grids: squared distance
// e0^2 + 3 ez^2 for R, (1/2-|e0|)^2 + 3 (1/2-|ez|)^2 for the shifted coset
// (R kept on equal distance).  Codes (2x, 2y/sqrt3) = (2 f0, 2 fz) or
// (2 f0 +- 1, 2 fz +- 1), the +-1 toward the coordinate.  Returns 2 bytes.
template <bool CHECK>
__device__ __forceinline__ uint32_t decode_a2_pair(float2 y, bool& range) {
  const float z = y.y * 0.57735026918962576f;  // 1/sqrt(3)
  const float2 v = make_float2(y.x, z);
  const float2 M2 = make_float2(kRoundMagic, kRoundMagic);
  const float2 t = add2(v, M2);
  const float2 e = sub2(v, sub2(t, M2));
  const float a0 = fabsf(e.x), a1 = fabsf(e.y);
  const float dA = fmaf(3.f * e.y, e.y, e.x * e.x);
  const float b0 = 0.5f - a0, b1 = 0.5f - a1;
  const float dB = fmaf(3.f * b1, b1, b0 * b0);
  const bool takeB = dB < dA;
  const uint32_t bmask = takeB ? 0xFFFFFFFFu : 0u;
  const uint32_t t0 = __float_as_uint(t.x), t1 = __float_as_uint(t.y);
  const uint32_t s0 = ((uint32_t)((int32_t)__float_as_uint(e.x) >> 31) | 1u) & bmask;
  const uint32_t s1 = ((uint32_t)((int32_t)__float_as_uint(e.y) >> 31) | 1u) & bmask;
  const uint32_t c0 = t0 + t0 + s0;
  const uint32_t c1 = t1 + t1 + s1;
  if (CHECK && !(fmaxf(fabsf(y.x), fabsf(z)) < 62.5f)) {
    const int i0 = 2 * rint_int(t0) + (int)s0, i1 = 2 * rint_int(t1) + (int)s1;
    range |= (i0 > 127) || (i0 < -127) || (i1 > 127) || (i1 < -127);
  }
  return (c0 & 0xFFu) | ((c1 & 0xFFu) << 8);
}

// Z: c = 2 rint(y) for four coordinates.
template <bool CHECK>
__device__ __forceinline__ uint32_t decode_z1_quad(float2 a, float2 b, bool& range) {
  const float2 M2 = make_float2(kRoundMagic, kRoundMagic);
  const float2 t0 = add2(a, M2), t1 = add2(b, M2);
  const uint32_t u0 = __float_as_uint(t0.x), u1 = __float_as_uint(t0.y);
  const uint32_t u2 = __float_as_uint(t1.x), u3 = __float_as_uint(t1.y);
  const float m = fmaxf(fmaxf(fabsf(a.x), fabsf(a.y)), fmaxf(fabsf(b.x), fabsf(b.y)));
  if (CHECK && !(m < 62.5f)) {
    const int mx = max(max(abs(rint_int(u0)), abs(rint_int(u1))), max(abs(rint_int(u2)), abs(rint_int(u3))));
    range |= (2 * mx > 127);
  }
  return pack4(u0 + u0, u1 + u1, u2 + u2, u3 + u3);
}

// Decode the 64 register-resident coordinates of one lane into 16 code words
// (word w = columns 4w .. 4w+3).  CHECK adds the exact int8 range check; it
// can be left out when every |y| of the lane is known to be below 62.5.
template <int LAT, bool CHECK>
__device__ __forceinline__ void decode_lane(const float2 (&p)[32], uint32_t (&w)[16], bool& range) {
  if constexpr (LAT == LQ_E8) {
#pragma unroll
    for (int b = 0; b < 8; ++b) {
      const float2 y[4] = {p[4 * b], p[4 * b + 1], p[4 * b + 2], p[4 * b + 3]};
      const BlockCodes8 r = decode_e8<CHECK>(y, range);
      w[2 * b] = r.w0;
      w[2 * b + 1] = r.w1;
    }
  } else if constexpr (LAT == LQ_D4) {
#pragma unroll
    for (int b = 0; b < 16; ++b) {
      const float2 y[2] = {p[2 * b], p[2 * b + 1]};
      w[b] = decode_d4<CHECK>(y, range);
    }
  } else if constexpr (LAT == LQ_A2) {
#pragma unroll
    for (int b = 0; b < 16; ++b) {
      const uint32_t lo = decode_a2_pair<CHECK>(p[2 * b], range);
      const uint32_t hi = decode_a2_pair<CHECK>(p[2 * b + 1], range);
      w[b] = lo | (hi << 16);
    }
  } else {
#pragma unroll
    for (int b = 0; b < 16; ++b) w[b] = decode_z1_quad<CHECK>(p[2 * b], p[2 * b + 1], range);
  }
}

// ---------------------------------------------------------------- pair decoders
// The quantize kernel holds the 64 coordinates of a lane as float2 p[32] with
// p[j].x = column j and p[j].y = column j + 32 (after its transform: two
// different lattice blocks), so one f32x2 instruction works on coordinate i of
// two blocks at once.  These decoders take u[i] = p[8 g + i] (i = 0..7) and
// the scale k (y = u k): block P in the .x halves, block Q in the .y halves.
//
// Fast-path precondition: every |y| < 62.5.  Then rint(y) lies in [-62, 62]
// and every code in [-127, 127], and the codes are built four to a word in
// "offset binary" (code + 128 per byte, every byte in [1, 255] at every step),
// so that 32-bit adds and subtracts never carry from one byte into the next;
// one XOR with 0x80808080 at the end gives the int8 codes.

// y + kRoundMagic64 (|y| < 2^22) rounds y to the nearest integer (ties to
// even) and leaves rint(y) + 64 in the low byte of its bits.
constexpr float kRoundMagic64 = 12582976.0f;   // 1.5 * 2^23 + 64

// PTX prmt in its default mode: byte n of the result is byte (sel_n & 7) of
// {b, a}, or, when bit 3 of the selector nibble sel_n is set, that byte's sign
// bit replicated over all 8 bits.  (The __byte_perm intrinsic keeps only the
// low three bits of each nibble, so the sign mode needs the instruction itself.)
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// Bytes 0 of four words into one word.
__device__ __forceinline__ uint32_t pack_low4(uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  return prmt(prmt(a, b, 0x0040u), prmt(c, d, 0x0040u), 0x5410u);
}
// 0xFF in byte i where word i is negative (its sign bit replicated), else 0.
__device__ __forceinline__ uint32_t pack_sign4(uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  return prmt(prmt(a, b, 0x00FBu), prmt(c, d, 0x00FBu), 0x5410u);
}

// PRMT selectors that turn a word of per-coordinate fix bytes into the fix of
// one coordinate as a signed 32-bit number: entry i (0..7) keeps byte i & 3 of
// the fix word of code word i >> 2 at its place, zero below it and its sign
// replicated above it (.x: selector for word 0, coordinates 0..3; .y: word 1,
// coordinates 4..7; the other word gets zero); entry 8 is no fix at all.
// Nibble 4 selects a zero byte (byte 0 of the zero operand), nibble p byte p,
// nibble 8 | p the sign of byte p.
__device__ __forceinline__ uint2 parity_fix_selector(int i) {
  const int p = i & 3;
  const uint32_t one = p == 0 ? 0x8880u : p == 1 ? 0x9914u : p == 2 ? 0xA244u : 0x3444u;
  if (i >= 8) return make_uint2(0x4444u, 0x4444u);
  return i < 4 ? make_uint2(one, 0x4444u) : make_uint2(0x4444u, one);
}

// Codes of one E8 block from its packed rounding bytes F0, F1 (rint(y) + 64 of
// coordinates 0..3 and 4..7), packed residual signs N0, N1 (0xFF where
// y < rint(y)), the largest and smallest key (|e| with the low three mantissa
// bits replaced by 7 - i) and lhs = 2 - sum |e|.  E8 = D8 u (D8 + 1/2) decoded
// as in decode_e8: the D8 point is f = rint(y) with the worst coordinate
// (largest |e|, lowest index on ties) rounded the other way when sum f is odd;
// the D8 + 1/2 point is floor(y) + 1/2 with its worst coordinate (smallest |e|)
// moved across when sum floor(y) is odd.  Their squared distances minus
// sum e^2 are dA = [odd A] (1 - 2 max|e|) and dB = 2 - sum|e| + [odd B] 2 min|e|,
// and D8 is kept when dA <= dB.  Per byte, in offset binary: D8 code 2F
// (F = rint(y) + 64), D8 + 1/2 code 2F + 1 - 2[e < 0]; the parity fix adds +-2
// at the chosen coordinate (toward y: +2 - 4[e < 0] for D8, -2 + 4[e < 0] for
// D8 + 1/2).
__device__ __forceinline__ uint2 e8_block_codes(uint32_t F0, uint32_t F1, uint32_t N0, uint32_t N1, uint32_t kA,
                                                uint32_t kB, float lhs, const uint2* fixsel) {
  // bit 0 of each byte: parity of F_i + F_(i+4); bit 4: of the two signs.  The
  // byte sum (top byte of the product) then has the parity of sum F (= that of
  // sum rint(y): 8 * 64 is even) in bit 0 and that of the count of negative
  // residuals in bit 4.
  const uint32_t par = imad(((F0 ^ F1) & 0x01010101u) | ((N0 ^ N1) & 0x10101010u), 0x01010101u, 0u) >> 24;
  const bool oddA = (par & 1u) != 0;
  const bool oddB = ((par ^ (par >> 4)) & 1u) != 0;
  const float dA = oddA ? fmaf(-2.f, __uint_as_float(kA), 1.f) : 0.f;
  const float dB = oddB ? fmaf(2.f, __uint_as_float(kB), lhs) : lhs;
  const bool takeB = dB < dA;
  const uint32_t kk = takeB ? kB : kA;
  const bool fix = takeB ? oddB : oddA;
  const uint2 sel = fixsel[fix ? 7 - (int)(kk & 7u) : 8];
  const uint32_t bm = takeB ? 0xFFFFFFFFu : 0u;
  const uint32_t fixbytes = 0x02020202u ^ (bm & 0xFCFCFCFCu);   // +2 (D8) or -2 (D8 + 1/2) where e >= 0
  uint2 r;
  r.x = ((F0 + F0 + (bm & 0x01010101u)) - (N0 & bm & 0x02020202u) +
         prmt(fixbytes ^ (N0 & 0xFCFCFCFCu), 0u, sel.x)) ^ 0x80808080u;
  r.y = ((F1 + F1 + (bm & 0x01010101u)) - (N1 & bm & 0x02020202u) +
         prmt(fixbytes ^ (N1 & 0xFCFCFCFCu), 0u, sel.y)) ^ 0x80808080u;
  return r;
}

// Rounding bits, residual bits and key of coordinate i of two blocks side by
// side (.x block P, .y block Q): t = u k + magic and e = u k - rint(y) are each
// one fused multiply-add of the exact product.
struct E8Coord {
  uint32_t tP, tQ, eP, eQ, kP, kQ;
};
__device__ __forceinline__ E8Coord e8_coord(float2 u, float2 k2, int i) {
  const float2 MG = make_float2(kRoundMagic64, kRoundMagic64);
  const float2 t = fma2(u, k2, MG);
  const float2 e = fma2(u, k2, sub2(MG, t));   // MG - t = -rint(y), exact
  E8Coord c;
  c.tP = __float_as_uint(t.x);
  c.tQ = __float_as_uint(t.y);
  c.eP = __float_as_uint(e.x);
  c.eQ = __float_as_uint(e.y);
  c.kP = (c.eP & 0x7FFFFFF8u) | (uint32_t)(7 - i);
  c.kQ = (c.eQ & 0x7FFFFFF8u) | (uint32_t)(7 - i);
  return c;
}
__device__ __forceinline__ float2 key_pair(const E8Coord& c) {
  return make_float2(__uint_as_float(c.kP), __uint_as_float(c.kQ));
}

// Fast E8 decode of two blocks side by side (see above), y = u k never formed.
// The coordinates are taken four at a time and reduced at once (packed bytes,
// partial key extremes and sums), which keeps few temporaries alive.
__device__ __forceinline__ void decode_e8_pair(const float2 (&u)[8], float2 k2, const uint2* fixsel, uint2& cP,
                                               uint2& cQ) {
  uint32_t FP[2], FQ[2], NP[2], NQ[2];
  uint32_t mxP = 0, mxQ = 0, mnP = 0, mnQ = 0;
  float2 s = make_float2(0.f, 0.f);
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const E8Coord c0 = e8_coord(u[4 * h], k2, 4 * h), c1 = e8_coord(u[4 * h + 1], k2, 4 * h + 1);
    const E8Coord c2 = e8_coord(u[4 * h + 2], k2, 4 * h + 2), c3 = e8_coord(u[4 * h + 3], k2, 4 * h + 3);
    FP[h] = pack_low4(c0.tP, c1.tP, c2.tP, c3.tP);
    FQ[h] = pack_low4(c0.tQ, c1.tQ, c2.tQ, c3.tQ);
    NP[h] = pack_sign4(c0.eP, c1.eP, c2.eP, c3.eP);
    NQ[h] = pack_sign4(c0.eQ, c1.eQ, c2.eQ, c3.eQ);
    // sum |e| of each block from the keys (each within 7 ulps of |e|)
    const float2 sh = add2(add2(key_pair(c0), key_pair(c1)), add2(key_pair(c2), key_pair(c3)));
    if (h == 0) {
      s = sh;
      mxP = key_max3(c0.kP, c1.kP, c2.kP);
      mxQ = key_max3(c0.kQ, c1.kQ, c2.kQ);
      mnP = key_min3(c0.kP, c1.kP, c2.kP);
      mnQ = key_min3(c0.kQ, c1.kQ, c2.kQ);
      mxP = __float_as_uint(fmaxf(__uint_as_float(mxP), __uint_as_float(c3.kP)));
      mxQ = __float_as_uint(fmaxf(__uint_as_float(mxQ), __uint_as_float(c3.kQ)));
      mnP = __float_as_uint(fminf(__uint_as_float(mnP), __uint_as_float(c3.kP)));
      mnQ = __float_as_uint(fminf(__uint_as_float(mnQ), __uint_as_float(c3.kQ)));
    } else {
      s = add2(s, sh);
      mxP = key_max3(key_max3(mxP, c0.kP, c1.kP), c2.kP, c3.kP);
      mxQ = key_max3(key_max3(mxQ, c0.kQ, c1.kQ), c2.kQ, c3.kQ);
      mnP = key_min3(key_min3(mnP, c0.kP, c1.kP), c2.kP, c3.kP);
      mnQ = key_min3(key_min3(mnQ, c0.kQ, c1.kQ), c2.kQ, c3.kQ);
    }
  }
  const float2 lhs = sub2(make_float2(2.f, 2.f), s);
  cP = e8_block_codes(FP[0], FP[1], NP[0], NP[1], mxP, mnP, lhs.x, fixsel);
  cQ = e8_block_codes(FQ[0], FQ[1], NQ[0], NQ[1], mxQ, mnQ, lhs.y, fixsel);
}

// Fast Z1 decode of two 8-coordinate groups side by side: c = 2 rint(y).
__device__ __forceinline__ void decode_z1_pair(const float2 (&u)[8], float2 k2, uint2& cP, uint2& cQ) {
  const float2 MG = make_float2(kRoundMagic64, kRoundMagic64);
  uint32_t tP[8], tQ[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float2 t = fma2(u[i], k2, MG);
    tP[i] = __float_as_uint(t.x);
    tQ[i] = __float_as_uint(t.y);
  }
  const uint32_t P0 = pack_low4(tP[0], tP[1], tP[2], tP[3]), P1 = pack_low4(tP[4], tP[5], tP[6], tP[7]);
  const uint32_t Q0 = pack_low4(tQ[0], tQ[1], tQ[2], tQ[3]), Q1 = pack_low4(tQ[4], tQ[5], tQ[6], tQ[7]);
  cP = make_uint2((P0 + P0) ^ 0x80808080u, (P1 + P1) ^ 0x80808080u);
  cQ = make_uint2((Q0 + Q0) ^ 0x80808080u, (Q1 + Q1) ^ 0x80808080u);
}

// ---------------------------------------------------------------- dither
// Subtractive dither (Zamir & Feder, "On lattice quantization noise", 1996):
// element (r, k) of a [rows x cols] matrix draws w = (top 24 bits of SplitMix64
// output r * cols + k from state seed) / 2^24 -- the generator of the signs
// (Steele, Lea & Flood 2014) -- and the draws of one lattice block, scaled to
// a box that tiles space under a sublattice (E8, D4: side 2; A2: 1 x sqrt 3;
// Z: 1), are reduced into the Voronoi cell: u = z - Q(z).
__device__ __forceinline__ float dither_w(uint64_t seed, uint64_t counter) {
  uint64_t z = seed + (counter + 1) * 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  // the generator's last step, z ^= z >> 31, leaves bits 63 .. 40 unchanged
  // (it only flips bits below 33), so the top 24 bits are read before it
  return (float)(uint32_t)(z >> 40) * (1.0f / 16777216.0f);
}

__device__ __forceinline__ float code_byte(uint32_t w, int k) { return (float)(int8_t)(w >> (8 * k)); }

// Dither u (point coordinates) of the 8 consecutive elements whose first has
// counter c0 (one E8 block, two D4 blocks, four A2 pairs or eight Z values).
template <int LAT>
__device__ __forceinline__ void dither8(uint64_t seed, uint64_t c0, float (&u)[8]) {
  float z[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) z[i] = dither_w(seed, c0 + (uint64_t)i);
  bool unused = false;
  if constexpr (LAT == LQ_E8) {
    const float2 y[4] = {make_float2(2.f * z[0], 2.f * z[1]), make_float2(2.f * z[2], 2.f * z[3]),
                         make_float2(2.f * z[4], 2.f * z[5]), make_float2(2.f * z[6], 2.f * z[7])};
    const BlockCodes8 c = decode_e8<false>(y, unused);
#pragma unroll
    for (int i = 0; i < 8; ++i) u[i] = 2.f * z[i] - 0.5f * code_byte(i < 4 ? c.w0 : c.w1, i & 3);
  } else if constexpr (LAT == LQ_D4) {
#pragma unroll
    for (int b = 0; b < 2; ++b) {
      const float2 y[2] = {make_float2(2.f * z[4 * b], 2.f * z[4 * b + 1]),
                           make_float2(2.f * z[4 * b + 2], 2.f * z[4 * b + 3])};
      const uint32_t c = decode_d4<false>(y, unused);
#pragma unroll
      for (int i = 0; i < 4; ++i) u[4 * b + i] = 2.f * z[4 * b + i] - 0.5f * code_byte(c, i);
    }
  } else if constexpr (LAT == LQ_A2) {
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const float2 y = make_float2(z[2 * b], 1.7320508075688772f * z[2 * b + 1]);
      const uint32_t c = decode_a2_pair<false>(y, unused);
      u[2 * b] = y.x - 0.5f * code_byte(c, 0);
      u[2 * b + 1] = y.y - 0.8660254037844386f * code_byte(c, 1);
    }
  } else {
#pragma unroll
    for (int b = 0; b < 2; ++b) {
      const uint32_t c = decode_z1_quad<false>(make_float2(z[4 * b], z[4 * b + 1]),
                                               make_float2(z[4 * b + 2], z[4 * b + 3]), unused);
#pragma unroll
      for (int i = 0; i < 4; ++i) u[4 * b + i] = z[4 * b + i] - 0.5f * code_byte(c, i);
    }
  }
}

}  // namespace lq
