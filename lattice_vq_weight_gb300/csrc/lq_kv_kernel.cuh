// The decode-attention partial kernel over a lattice-quantized KV cache and
// its launch templates, shared by the translation units that instantiate it
// (lq_kv.cu: int8 codes; lq_kv_dither.cu: the subtractive dither;
// lq_kv_rice.cu: Rice-coded caches).  The method and the data flow are
// described at the top of lq_kv.cu.
#pragma once

#include <cmath>
#include <cuda_fp16.h>

#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "lq_device.cuh"
#include "lq_host.h"
#include "lq_rice.cuh"

namespace lq {
namespace kv {

constexpr int D = 128;              // head_dim handled here
constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;

struct AttnArgs {
  const int8_t* kc;
  const void* ks;        // [tokens x kv_heads], format sfmt (LQ_SCALE_TILE_F32 / _F16)
  const int8_t* ksg;
  const int8_t* vc;
  const void* vs;
  const int8_t* vsg;
  int sfmt;
  uint64_t kdseed, vdseed;   // subtractive dither seeds (DLAT instantiations)
  // Rice-coded caches (RLAT instantiations): streams, their lengths in words,
  // and the bit offset of each (token, kv head) segment
  const uint32_t* krs;
  const uint32_t* vrs;
  int64_t knw, vnw;
  const uint32_t* koff;
  const uint32_t* voff;
  const void* q;
  int qbf16;
  int64_t tokens;
  int kv_heads, group, splits;
  int a2;
  float* part;        // [kv_heads x splits x group x (2 + D)]: m, l, acc[D]
  float* qrot;        // [q_heads x D]: rotated, scaled queries
  float* out;         // [q_heads x D]
};

__device__ __forceinline__ float code_f(uint32_t w, int k) { return (float)(int8_t)(w >> (8 * k)); }

// Rows of the per-warp dither transpose (padded: conflict-free 16-byte
// accesses both by token rows and by dimension columns).
constexpr int kDvStride = D + 4;

// Dither of one cached vector in the doubled code units the kernel uses
// (2u; A2 odd coordinates 2u / sqrt 3): element (token, kvh * D + i) of the
// [tokens x kv_heads * D] cache.
template <int LAT>
__device__ __forceinline__ void dither8_codes(uint64_t seed, uint64_t c0, float (&du)[8]) {
  dither8<LAT>(seed, c0, du);
#pragma unroll
  for (int i = 0; i < 8; ++i) du[i] *= (LAT == LQ_A2 && (i & 1)) ? 1.1547005383792515f : 2.f;
}

// Per-warp Rice buffers, rows of 33 words (conflict-free 4-byte accesses by
// rows and by columns): the first 32 stream words of the chunk's K and of its
// V segments, word k of token t at k * 33 + t (33 rows: a window read at word
// 31 touches row 32), and the decoded V code words, word q of token t at
// t * 33 + q.
constexpr int kRiceStride = D / 4 + 1;
constexpr int kRiceStageWords = 33 * kRiceStride;
constexpr int kRiceWarpWords = 2 * kRiceStageWords + 32 * kRiceStride;
constexpr size_t kDvSmem = (size_t)kWarps * 32 * kDvStride * sizeof(float);
constexpr size_t kRiceSmem = (size_t)kWarps * kRiceWarpWords * sizeof(uint32_t);

// Decode the Rice segment at bit `pos` (D codes) into 32 code words at row,
// word q at row[q * STRIDE].
template <int LAT, int STRIDE = 1>
__device__ __forceinline__ void decode_segment(const uint32_t* stream, int64_t nwords, uint64_t pos, uint32_t* row) {
  constexpr int n = rice::Fmt<LAT>::n;
  rice::BitReader rd;
  rd.init(stream, nwords, pos);
  const int K = (int)rd.get(rice::kKBits);
#pragma unroll 1
  for (int q = 0; q < D / 16; ++q) {
    uint32_t wv[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int j = 0; j < 16; j += n) {
      int c[n];
      rice::decode_block<LAT>(rd, K, c);
#pragma unroll
      for (int e = 0; e < n; ++e) wv[(j + e) >> 2] |= ((uint32_t)c[e] & 0xFFu) << (8 * ((j + e) & 3));
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) row[(4 * q + e) * STRIDE] = wv[e];
  }
}

// DLAT = 0: caches without dither; otherwise the lattice of dithered caches,
// whose reconstruction is s (p - u): each score loses q~ . u of its token and
// the value sum the weighted dither of each token (transposed through shared
// memory, dynamic: kWarps x 32 x kDvStride floats).
// RLAT = 0: int8 codes; otherwise the lattice of Rice-coded caches: each lane
// decodes its token's K and V segments from per-warp staging buffers (dynamic:
// kWarps x kRiceWarpWords words), K into registers for the scores and V into a
// shared-memory row read back by dimension for the value sum.
template <int G, bool F16S, int DLAT, int RLAT>
__global__ void __launch_bounds__(kThreads, G <= 4 ? 4 : 2) attn_partial_kernel(AttnArgs a) {
  static_assert(DLAT == 0 || RLAT == 0, "dither and Rice caches are separate variants");
  __shared__ __align__(16) float qr[G][D];         // rotated, scaled queries
  __shared__ float wm[kWarps][G], wl[kWarps][G];
  __shared__ __align__(16) float wacc[kWarps][G][D];
  extern __shared__ __align__(16) float dv_smem[];
  const int kvh = blockIdx.x / a.splits, split = blockIdx.x % a.splits;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t ld = (int64_t)a.kv_heads * D;
  const int64_t j0 = split * a.tokens / a.splits, j1 = (split + 1) * a.tokens / a.splits;

  // the group's rotated queries
  for (int e = threadIdx.x; e < G * D / 4; e += blockDim.x)
    reinterpret_cast<float4*>(&qr[0][0])[e] =
        reinterpret_cast<const float4*>(a.qrot + (int64_t)kvh * a.group * D)[e];
  __syncthreads();

  float m[G], l[G], acc[G][4];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    m[g] = -INFINITY;
    l[g] = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) acc[g][k] = 0.f;
  }

  for (int64_t c0 = j0 + (int64_t)warp * 32; c0 < j1; c0 += kWarps * 32) {
    // issue every load of the chunk first: this lane's token's 128 K codes and
    // scales (lane = token), and its 4 V codes of each of the chunk's tokens
    // (lane = dimensions 4 lane .. 4 lane + 3)
    const int64_t j = c0 + lane;
    const bool ok = j < j1;
    const int nt = (j1 - c0) < 32 ? (int)(j1 - c0) : 32;
    uint4 kw[D / 16];
    float s_k = 0.f, s_v = 0.f;
    uint32_t kcw[RLAT != 0 ? D / 4 : 1];
    uint32_t* vrows = nullptr;
    if constexpr (RLAT != 0) {
      // stage the first 32 words of every token's K and V segments (one
      // coalesced copy per token and cache), then each lane decodes its own
      // token's segments with the two-symbol decoder: K into registers, V into
      // its row of vrows; a lane whose segment does not decode within the
      // staged words (or overflows a window) falls back to the sequential
      // reader on the stream in global memory
      uint32_t* kst = reinterpret_cast<uint32_t*>(dv_smem) + (size_t)warp * kRiceWarpWords;
      uint32_t* vst = kst + kRiceStageWords;
      vrows = vst + kRiceStageWords;
      const int64_t seg = j * a.kv_heads + kvh;
      const uint32_t ko = ok ? __ldg(a.koff + seg) : 0u, vo = ok ? __ldg(a.voff + seg) : 0u;
      __syncwarp();                                  // the previous chunk's reads of the buffers are done
#pragma unroll 1
      for (int t = 0; t < nt; ++t) {
        const uint32_t gk = __shfl_sync(0xffffffffu, ko >> 5, t) + (uint32_t)lane;
        const uint32_t gv = __shfl_sync(0xffffffffu, vo >> 5, t) + (uint32_t)lane;
        const bool ik = (int64_t)gk < a.knw, iv = (int64_t)gv < a.vnw;
        rice::cp_async4(kst + lane * kRiceStride + t, a.krs + (ik ? gk : 0u), ik ? 4u : 0u);
        rice::cp_async4(vst + lane * kRiceStride + t, a.vrs + (iv ? gv : 0u), iv ? 4u : 0u);
      }
      rice::cp_async_commit();
      rice::cp_async_wait<0>();
      __syncwarp();
      uint32_t* vrow = vrows + lane * kRiceStride;
      if (ok) {
        auto kwin = [&](uint32_t pos) {
          const uint32_t w = min(pos >> 5, 31u);
          return __funnelshift_r(kst[w * kRiceStride + lane], kst[(w + 1) * kRiceStride + lane], pos);
        };
        auto vwin = [&](uint32_t pos) {
          const uint32_t w = min(pos >> 5, 31u);
          return __funnelshift_r(vst[w * kRiceStride + lane], vst[(w + 1) * kRiceStride + lane], pos);
        };
        // V first (into its row), then K into registers: the two decodes do
        // not hold their outputs in registers at the same time
        uint32_t pos = vo & 31u;
        const rice::RiceK rv = rice::rice_k(vwin(pos) & 7u);
        pos += rice::kKBits;
        uint32_t um = rice::decode_codes_fast<RLAT, D>(vwin, pos, rv, [&](int q, uint32_t w) { vrow[q] = w; });
        if (um > 31u || (pos >> 5) + 1u > 31u) decode_segment<RLAT>(a.vrs, a.vnw, vo, vrow);
        pos = ko & 31u;
        const rice::RiceK rk = rice::rice_k(kwin(pos) & 7u);
        pos += rice::kKBits;
        um = rice::decode_codes_fast<RLAT, D>(kwin, pos, rk, [&](int q, uint32_t w) { kcw[q] = w; });
        if (um > 31u || (pos >> 5) + 1u > 31u) {
          // this lane's staged K column is free now: the sequential reader's scratch
          decode_segment<RLAT, kRiceStride>(a.krs, a.knw, ko, kst + lane);
#pragma unroll
          for (int q = 0; q < D / 4; ++q) kcw[q] = kst[q * kRiceStride + lane];
        }
      } else {
#pragma unroll
        for (int q = 0; q < D / 4; ++q) vrow[q] = 0u;
      }
      __syncwarp();
    }
    if (ok) {
      if constexpr (RLAT != 0) {
#pragma unroll
        for (int q = 0; q < D / 16; ++q) kw[q] = make_uint4(kcw[4 * q], kcw[4 * q + 1], kcw[4 * q + 2], kcw[4 * q + 3]);
      } else {
        const uint4* kp = reinterpret_cast<const uint4*>(a.kc + j * ld + (int64_t)kvh * D);
#pragma unroll
        for (int q = 0; q < D / 16; ++q) kw[q] = __ldg(kp + q);
      }
      if constexpr (F16S) {
        s_k = __half2float(__ldg(reinterpret_cast<const __half*>(a.ks) + j * a.kv_heads + kvh));
        s_v = __half2float(__ldg(reinterpret_cast<const __half*>(a.vs) + j * a.kv_heads + kvh));
      } else {
        s_k = __ldg(reinterpret_cast<const float*>(a.ks) + j * a.kv_heads + kvh);
        s_v = __ldg(reinterpret_cast<const float*>(a.vs) + j * a.kv_heads + kvh);
      }
    } else {
#pragma unroll
      for (int q = 0; q < D / 16; ++q) kw[q] = make_uint4(0, 0, 0, 0);
    }
    uint32_t vw[32];
    if constexpr (RLAT != 0) {
#pragma unroll
      for (int t = 0; t < 32; ++t) vw[t] = vrows[t * kRiceStride + lane];
    } else {
      const uint32_t* vp = reinterpret_cast<const uint32_t*>(a.vc + c0 * ld + (int64_t)kvh * D) + lane;
#pragma unroll
      for (int t = 0; t < 32; ++t) vw[t] = (t < nt) ? __ldg(vp + t * (ld / 4)) : 0u;
    }

    // scores
    float sc[G];
#pragma unroll
    for (int g = 0; g < G; ++g) sc[g] = 0.f;
#pragma unroll
    for (int q = 0; q < D / 16; ++q) {
      const uint32_t w[4] = {kw[q].x, kw[q].y, kw[q].z, kw[q].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float c0f = code_f(w[e], 0), c1f = code_f(w[e], 1), c2f = code_f(w[e], 2), c3f = code_f(w[e], 3);
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float4 qv = *reinterpret_cast<const float4*>(&qr[g][16 * q + 4 * e]);
          sc[g] = fmaf(c0f, qv.x, fmaf(c1f, qv.y, fmaf(c2f, qv.z, fmaf(c3f, qv.w, sc[g]))));
        }
      }
    }
    if constexpr (DLAT != 0) {
      // this lane's token: scores lose q~ . u (K dither); the V dither goes to
      // the warp's transpose buffer, row = lane
      float* dvrow = dv_smem + ((size_t)warp * 32 + lane) * kDvStride;
      const uint64_t cbase = (uint64_t)j * (uint64_t)ld + (uint64_t)kvh * D;
#pragma unroll 1
      for (int gb = 0; gb < D / 8; ++gb) {
        float du[8], dvv[8];
        if (ok) {
          dither8_codes<DLAT>(a.kdseed, cbase + 8 * gb, du);
          dither8_codes<DLAT>(a.vdseed, cbase + 8 * gb, dvv);
        } else {
#pragma unroll
          for (int i = 0; i < 8; ++i) du[i] = dvv[i] = 0.f;
        }
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float4 q0 = *reinterpret_cast<const float4*>(&qr[g][8 * gb]);
          const float4 q1 = *reinterpret_cast<const float4*>(&qr[g][8 * gb + 4]);
          float d = q0.x * du[0] + q0.y * du[1] + q0.z * du[2] + q0.w * du[3];
          d += q1.x * du[4] + q1.y * du[5] + q1.z * du[6] + q1.w * du[7];
          sc[g] -= d;
        }
        *reinterpret_cast<float4*>(dvrow + 8 * gb) = make_float4(dvv[0], dvv[1], dvv[2], dvv[3]);
        *reinterpret_cast<float4*>(dvrow + 8 * gb + 4) = make_float4(dvv[4], dvv[5], dvv[6], dvv[7]);
      }
      __syncwarp();
    }
    // online softmax over this chunk
    float p[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float s = ok ? sc[g] * s_k : -INFINITY;
      float cm = s;
      for (int o = 16; o; o >>= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, o));
      const float mn = fmaxf(m[g], cm);
      const float r = __expf(m[g] - mn);         // 0 when m was -inf
      p[g] = ok ? __expf(s - mn) : 0.f;
      l[g] = l[g] * r + p[g];                   // per-lane partial sum
      m[g] = mn;
#pragma unroll
      for (int k = 0; k < 4; ++k) acc[g][k] *= r;
      p[g] *= s_v;                              // the value scale of this lane's token
    }
    // values over the chunk's tokens (codes of missing tokens are zero, and so
    // are their weights)
#pragma unroll
    for (int t = 0; t < 32; ++t) {
      const uint32_t w = vw[t];
      float v0 = code_f(w, 0), v1 = code_f(w, 1), v2 = code_f(w, 2), v3 = code_f(w, 3);
      if constexpr (DLAT != 0) {
        const float4 dq = *reinterpret_cast<const float4*>(dv_smem + ((size_t)warp * 32 + t) * kDvStride + 4 * lane);
        v0 -= dq.x; v1 -= dq.y; v2 -= dq.z; v3 -= dq.w;
      }
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float pt = __shfl_sync(0xffffffffu, p[g], t);
        acc[g][0] = fmaf(pt, v0, acc[g][0]);
        acc[g][1] = fmaf(pt, v1, acc[g][1]);
        acc[g][2] = fmaf(pt, v2, acc[g][2]);
        acc[g][3] = fmaf(pt, v3, acc[g][3]);
      }
    }
    if constexpr (DLAT != 0 || RLAT != 0) __syncwarp();   // the next chunk rewrites the shared rows
  }
  // merge the four warps
#pragma unroll
  for (int g = 0; g < G; ++g) {
    float ls = l[g];
    for (int o = 16; o; o >>= 1) ls += __shfl_xor_sync(0xffffffffu, ls, o);
    if (lane == 0) {
      wm[warp][g] = m[g];
      wl[warp][g] = ls;
    }
    *reinterpret_cast<float4*>(&wacc[warp][g][4 * lane]) = make_float4(acc[g][0], acc[g][1], acc[g][2], acc[g][3]);
  }
  __syncthreads();
  for (int g = 0; g < G; ++g) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, wm[w][g]);
    float* dst = a.part + (((int64_t)kvh * a.splits + split) * G + g) * (2 + D);
    for (int i = threadIdx.x; i < D; i += blockDim.x) {
      float s = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) s += (wm[w][g] == -INFINITY) ? 0.f : wacc[w][g][i] * __expf(wm[w][g] - M);
      dst[2 + i] = s;
    }
    if (threadIdx.x == 0) {
      float L = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) L += (wm[w][g] == -INFINITY) ? 0.f : wl[w][g] * __expf(wm[w][g] - M);
      dst[0] = M;
      dst[1] = L;
    }
  }
}


// Launch of one instantiation with the dynamic shared memory it needs.
template <int G, bool H, int DLAT, int RLAT>
lq_status launch_partial_g(const AttnArgs& a, unsigned grid, cudaStream_t s) {
  constexpr size_t smem = DLAT ? kDvSmem : RLAT ? kRiceSmem : 0;
  if constexpr (smem > 0) {
    static bool attr = false;
    if (!attr) {
      if (cudaFuncSetAttribute(attn_partial_kernel<G, H, DLAT, RLAT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)smem) != cudaSuccess) {
        cudaGetLastError();
        return LQ_ERR_CUDA;
      }
      attr = true;
    }
  }
  attn_partial_kernel<G, H, DLAT, RLAT><<<grid, kThreads, smem, s>>>(a);
  return LQ_OK;
}

template <int DLAT, int RLAT>
lq_status launch_partial_groups(const AttnArgs& a, int group, bool h, unsigned grid, cudaStream_t s) {
  switch (group) {
    case 1: return h ? launch_partial_g<1, true, DLAT, RLAT>(a, grid, s) : launch_partial_g<1, false, DLAT, RLAT>(a, grid, s);
    case 2: return h ? launch_partial_g<2, true, DLAT, RLAT>(a, grid, s) : launch_partial_g<2, false, DLAT, RLAT>(a, grid, s);
    case 4: return h ? launch_partial_g<4, true, DLAT, RLAT>(a, grid, s) : launch_partial_g<4, false, DLAT, RLAT>(a, grid, s);
    default: return h ? launch_partial_g<8, true, DLAT, RLAT>(a, grid, s) : launch_partial_g<8, false, DLAT, RLAT>(a, grid, s);
  }
}

// The dithered (lq_kv_dither.cu) and Rice-coded (lq_kv_rice.cu) variants,
// instantiated in translation units of their own.
lq_status launch_partial_dithered(const AttnArgs& a, int lattice, int group, bool h, unsigned grid, cudaStream_t s);
// Rice-coded caches of lattice RLAT with fp16 (H) or fp32 norms: explicitly
// instantiated in lq_kv_rice.cu, which is compiled once per (lattice, norm
// format) pair; launch_partial_rice (lq_kv.cu) picks the instantiation.
template <int RLAT, bool H>
lq_status launch_partial_rice_lh(const AttnArgs& a, int group, unsigned grid, cudaStream_t s);
lq_status launch_partial_rice(const AttnArgs& a, int lattice, int group, bool h, unsigned grid, cudaStream_t s);

}  // namespace kv
}  // namespace lq
