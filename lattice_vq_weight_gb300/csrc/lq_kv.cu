// Decode attention over a lattice-quantized KV cache, computed from the codes.
//
// HyperQuant page, KV-cache section: the cache keeps lattice codes plus one
// norm per vector after a random sign rotation, and attention runs on the
// quantized K/V.  A cache [tokens x kv_heads * head_dim] quantized by
// lq_quantize with tile = head_dim holds, for token j and kv head h, the codes
// c and the scale s of k^ = D H (s c~ / 2) / sqrt(d)  (c~: A2 odd coordinates
// times sqrt 3), so with x~ = H D q / sqrt(d):
//     q . k^ = (s / 2) x~ . c~        (one rotation of q per head, then dot
//                                       products with the raw codes)
//     sum_j p_j v^_j = D H (sum_j p_j s_j c~_j) / (2 sqrt d)
//                                      (accumulate codes in the rotated domain,
//                                       rotate back once per head)
// Kernel 1 rotates the queries.  Kernel 2 (one CTA per kv head and token
// range, four warps): each warp takes 32 tokens at a time -- lane = token for
// the scores (128 codes against the group's rotated queries), an online
// softmax, then lane = 4 dimensions for the value sum over those 32 tokens.
// Kernel 3 merges the ranges and rotates the result back.
#include <cmath>

#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "lq_device.cuh"
#include "lq_host.h"

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

// In-place unnormalised Walsh-Hadamard transform of v[0 .. D) in shared memory
// (Sylvester order), all threads of the block.
__device__ __forceinline__ void block_fwht(float* v) {
  for (int h = 1; h < D; h <<= 1) {
    __syncthreads();
    for (int i = threadIdx.x; i < D / 2; i += blockDim.x) {
      const int lo = (i / h) * 2 * h + (i % h);
      const float a = v[lo], b = v[lo + h];
      v[lo] = a + b;
      v[lo + h] = a - b;
    }
  }
  __syncthreads();
}

// One block per query head: x~ = H D q / sqrt(d), times 1/2 (codes are
// doubled), sqrt 3 on A2 odd coordinates and the softmax scale 1/sqrt(d).
__global__ void __launch_bounds__(D) rotate_query_kernel(AttnArgs a) {
  __shared__ float v[D];
  const int qh = blockIdx.x, kvh = qh / a.group, i = threadIdx.x;
  const int64_t qi = (int64_t)qh * D + i;
  const float x = a.qbf16 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(a.q)[qi])
                          : reinterpret_cast<const float*>(a.q)[qi];
  v[i] = x * (float)a.ksg[kvh * D + i];
  block_fwht(v);
  a.qrot[qi] = v[i] * (0.5f / (float)D) * ((a.a2 && (i & 1)) ? 1.7320508075688772f : 1.f);
}

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

// DLAT = 0: caches without dither; otherwise the lattice of dithered caches,
// whose reconstruction is s (p - u): each score loses q~ . u of its token and
// the value sum the weighted dither of each token (transposed through shared
// memory, dynamic: kWarps x 32 x kDvStride floats).
template <int G, bool F16S, int DLAT>
__global__ void __launch_bounds__(kThreads, G <= 4 ? 4 : 2) attn_partial_kernel(AttnArgs a) {
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
    if (ok) {
      const uint4* kp = reinterpret_cast<const uint4*>(a.kc + j * ld + (int64_t)kvh * D);
#pragma unroll
      for (int q = 0; q < D / 16; ++q) kw[q] = __ldg(kp + q);
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
    const uint32_t* vp = reinterpret_cast<const uint32_t*>(a.vc + c0 * ld + (int64_t)kvh * D) + lane;
    uint32_t vw[32];
#pragma unroll
    for (int t = 0; t < 32; ++t) vw[t] = (t < nt) ? __ldg(vp + t * (ld / 4)) : 0u;

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
    if constexpr (DLAT != 0) __syncwarp();   // the next chunk rewrites the transpose buffer
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

// One block per query head: merge the token ranges (weights exp(m_s - M) of
// every range computed once, in parallel), rotate back, apply signs.
constexpr int kMaxSplits = 4096;

__global__ void __launch_bounds__(D) attn_combine_kernel(AttnArgs a, int G) {
  __shared__ float r[D];
  __shared__ float wgt[kMaxSplits];
  __shared__ float red[D / 32];
  const int qh = blockIdx.x, kvh = qh / a.group, g = qh % a.group;
  const int i = threadIdx.x, lane = i & 31, warp = i >> 5;
  const float* base = a.part + ((int64_t)kvh * a.splits * G + g) * (2 + D);
  const int64_t stride = (int64_t)G * (2 + D);
  float M = -INFINITY;
  for (int s = i; s < a.splits; s += D) M = fmaxf(M, base[s * stride]);
  for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  if (lane == 0) red[warp] = M;
  __syncthreads();
  M = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
  __syncthreads();
  float L = 0.f;
  for (int s = i; s < a.splits; s += D) {
    const float ms = base[s * stride];
    const float e = (ms == -INFINITY) ? 0.f : __expf(ms - M);
    wgt[s] = e;
    L += e * base[s * stride + 1];
  }
  for (int o = 16; o; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
  if (lane == 0) red[warp] = L;
  __syncthreads();
  L = red[0] + red[1] + red[2] + red[3];
  float acc = 0.f;
  for (int s = 0; s < a.splits; ++s) acc = fmaf(wgt[s], base[s * stride + 2 + i], acc);
  r[i] = acc * ((a.a2 && (i & 1)) ? 1.7320508075688772f : 1.f) / (2.f * sqrtf((float)D) * L);
  block_fwht(r);
  a.out[(int64_t)qh * D + i] = r[i] * (float)a.vsg[kvh * D + i];
}

// Dense rotation of every D-column block: y = M x with M = R or R^T (R [D x D]
// row-major, fp32).  M^T is staged in shared memory (64 KB) so that lane j
// reads M[j][i] conflict-free; each warp rotates one block at a time, lane j
// computing outputs j, j + 32, j + 64, j + 96.
struct RotArgs {
  const float* R;
  int transpose;
  const void* X;
  int xbf16;
  int64_t rows, blocks_per_row, ldx, ldy;
  float* Y;
};

__global__ void __launch_bounds__(256) rotate_blocks_kernel(RotArgs a) {
  extern __shared__ float rot_smem[];
  float* mt = rot_smem;                 // mt[i * D + j] = M[j][i]
  float* xs = rot_smem + D * D;         // one D-vector per warp
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int e = threadIdx.x; e < D * D; e += blockDim.x) {
    const int i = e / D, j = e % D;
    mt[e] = a.transpose ? a.R[i * D + j] : a.R[j * D + i];   // M[j][i]
  }
  __syncthreads();
  float* xw = xs + warp * D;
  const int64_t nvec = a.rows * a.blocks_per_row;
  for (int64_t v = (int64_t)blockIdx.x * (blockDim.x >> 5) + warp; v < nvec;
       v += (int64_t)gridDim.x * (blockDim.x >> 5)) {
    const int64_t r = v / a.blocks_per_row, b = v - r * a.blocks_per_row;
    const int64_t xo = r * a.ldx + b * D;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int i = lane + 32 * k;
      xw[i] = a.xbf16 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(a.X)[xo + i])
                      : reinterpret_cast<const float*>(a.X)[xo + i];
    }
    __syncwarp();
    float y[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
    for (int i = 0; i < D; ++i) {
      const float xi = xw[i];
#pragma unroll
      for (int k = 0; k < 4; ++k) y[k] = fmaf(mt[i * D + lane + 32 * k], xi, y[k]);
    }
    float* yo = a.Y + r * a.ldy + b * D;
#pragma unroll
    for (int k = 0; k < 4; ++k) yo[lane + 32 * k] = y[k];
    __syncwarp();
  }
}

}  // namespace kv
}  // namespace lq

using namespace lq;
using namespace lq::kv;

namespace {

// floats of the per-range partial results, rounded up to 64 (the rotated
// queries that follow them are read as float4)
size_t part_floats(int kv_heads, int splits, int group) {
  const size_t n = (size_t)kv_heads * splits * group * (2 + D);
  return (n + 63) & ~(size_t)63;
}

int attn_splits(int64_t tokens, int kv_heads) {
  const int sms = device_sm_count();
  // about four CTAs per SM and at least 128 tokens (one chunk per warp) per range
  int64_t want = sms > 0 ? (4LL * sms + kv_heads - 1) / kv_heads : 1;
  const int64_t by_tokens = (tokens + 127) / 128;
  if (want > by_tokens) want = by_tokens;
  if (want < 1) want = 1;
  if (want > kMaxSplits) want = kMaxSplits;
  return (int)want;
}

}  // namespace

extern "C" size_t lq_attention_workspace_size(int64_t tokens, int kv_heads, int q_heads, int head_dim) {
  if (tokens <= 0 || kv_heads <= 0 || q_heads <= 0 || head_dim != D || q_heads % kv_heads != 0) return 0;
  const int splits = attn_splits(tokens, kv_heads);
  return (part_floats(kv_heads, splits, q_heads / kv_heads) + (size_t)q_heads * D) * sizeof(float);
}

namespace {

constexpr size_t kDvSmem = (size_t)kWarps * 32 * kDvStride * sizeof(float);

template <int G, bool H, int LAT>
lq_status launch_partial_dithered_g(const AttnArgs& a, unsigned grid, cudaStream_t s) {
  static bool attr = false;
  if (!attr) {
    if (cudaFuncSetAttribute(attn_partial_kernel<G, H, LAT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kDvSmem) != cudaSuccess) {
      cudaGetLastError();
      return LQ_ERR_CUDA;
    }
    attr = true;
  }
  attn_partial_kernel<G, H, LAT><<<grid, kThreads, kDvSmem, s>>>(a);
  return LQ_OK;
}

template <int LAT>
lq_status launch_partial_dithered(const AttnArgs& a, int group, bool h, unsigned grid, cudaStream_t s) {
  switch (group) {
    case 1: return h ? launch_partial_dithered_g<1, true, LAT>(a, grid, s) : launch_partial_dithered_g<1, false, LAT>(a, grid, s);
    case 2: return h ? launch_partial_dithered_g<2, true, LAT>(a, grid, s) : launch_partial_dithered_g<2, false, LAT>(a, grid, s);
    case 4: return h ? launch_partial_dithered_g<4, true, LAT>(a, grid, s) : launch_partial_dithered_g<4, false, LAT>(a, grid, s);
    default: return h ? launch_partial_dithered_g<8, true, LAT>(a, grid, s) : launch_partial_dithered_g<8, false, LAT>(a, grid, s);
  }
}

lq_status attention_fmt(int lattice, const int8_t* k_codes_dev, const void* k_scales_dev,
                        const int8_t* k_signs_dev, const int8_t* v_codes_dev, const void* v_scales_dev,
                        const int8_t* v_signs_dev, int sfmt, int64_t tokens, int kv_heads, int q_heads, int head_dim,
                        const void* q_dev, int qdtype, float* out_dev, void* workspace_dev, size_t workspace_bytes,
                        void* stream, bool dither = false, uint64_t k_dither_seed = 0, uint64_t v_dither_seed = 0) {
  if (!valid_lattice(lattice)) return LQ_ERR_ARG;
  if (sfmt != LQ_SCALE_TILE_F32 && sfmt != LQ_SCALE_TILE_F16) return LQ_ERR_ARG;
  const uintptr_t salign = (sfmt == LQ_SCALE_TILE_F32) ? 3u : 1u;
  if (head_dim != D) return LQ_ERR_UNSUPPORTED;
  if (qdtype != LQ_BF16 && qdtype != LQ_F32) return LQ_ERR_DTYPE;
  if (tokens <= 0 || kv_heads <= 0 || q_heads <= 0 || q_heads % kv_heads != 0) return LQ_ERR_SHAPE;
  const int group = q_heads / kv_heads;
  if (group != 1 && group != 2 && group != 4 && group != 8) return LQ_ERR_UNSUPPORTED;
  if (tokens > (int64_t(1) << 31)) return LQ_ERR_SHAPE;
  if (k_codes_dev == nullptr || k_scales_dev == nullptr || k_signs_dev == nullptr || v_codes_dev == nullptr ||
      v_scales_dev == nullptr || v_signs_dev == nullptr || q_dev == nullptr || out_dev == nullptr ||
      workspace_dev == nullptr)
    return LQ_ERR_ARG;
  if (!aligned16(k_codes_dev) || !aligned16(v_codes_dev) || (reinterpret_cast<uintptr_t>(k_scales_dev) & salign) ||
      (reinterpret_cast<uintptr_t>(v_scales_dev) & salign) ||
      !aligned4(out_dev) || !aligned4(workspace_dev))
    return LQ_ERR_ARG;
  if (workspace_bytes < lq_attention_workspace_size(tokens, kv_heads, q_heads, head_dim)) return LQ_ERR_SHAPE;
  AttnArgs a;
  a.kc = k_codes_dev; a.ks = k_scales_dev; a.ksg = k_signs_dev;
  a.vc = v_codes_dev; a.vs = v_scales_dev; a.vsg = v_signs_dev;
  a.sfmt = sfmt;
  a.kdseed = k_dither_seed;
  a.vdseed = v_dither_seed;
  a.q = q_dev; a.qbf16 = (qdtype == LQ_BF16);
  a.tokens = tokens; a.kv_heads = kv_heads; a.group = group;
  a.splits = attn_splits(tokens, kv_heads);
  a.a2 = (lattice == LQ_A2);
  a.part = reinterpret_cast<float*>(workspace_dev);
  a.qrot = a.part + part_floats(kv_heads, a.splits, group);
  a.out = out_dev;
  cudaStream_t s = (cudaStream_t)stream;
  if (!aligned16(workspace_dev)) return LQ_ERR_ARG;
  rotate_query_kernel<<<(unsigned)q_heads, D, 0, s>>>(a);
  const unsigned grid = (unsigned)(kv_heads * a.splits);
  const bool h = (sfmt == LQ_SCALE_TILE_F16);
  lq_status st = LQ_OK;
  if (dither) {
    switch (lattice) {
      case LQ_E8: st = launch_partial_dithered<LQ_E8>(a, group, h, grid, s); break;
      case LQ_D4: st = launch_partial_dithered<LQ_D4>(a, group, h, grid, s); break;
      case LQ_A2: st = launch_partial_dithered<LQ_A2>(a, group, h, grid, s); break;
      default:    st = launch_partial_dithered<LQ_Z1>(a, group, h, grid, s); break;
    }
    if (st != LQ_OK) return st;
  } else {
    switch (group) {
      case 1: h ? attn_partial_kernel<1, true, 0><<<grid, kThreads, 0, s>>>(a)
                : attn_partial_kernel<1, false, 0><<<grid, kThreads, 0, s>>>(a); break;
      case 2: h ? attn_partial_kernel<2, true, 0><<<grid, kThreads, 0, s>>>(a)
                : attn_partial_kernel<2, false, 0><<<grid, kThreads, 0, s>>>(a); break;
      case 4: h ? attn_partial_kernel<4, true, 0><<<grid, kThreads, 0, s>>>(a)
                : attn_partial_kernel<4, false, 0><<<grid, kThreads, 0, s>>>(a); break;
      default: h ? attn_partial_kernel<8, true, 0><<<grid, kThreads, 0, s>>>(a)
                 : attn_partial_kernel<8, false, 0><<<grid, kThreads, 0, s>>>(a); break;
    }
  }
  st = check_launch();
  if (st != LQ_OK) return st;
  attn_combine_kernel<<<(unsigned)q_heads, D, 0, s>>>(a, group);
  return check_launch();
}

}  // namespace

extern "C" lq_status lq_attention_decode(int lattice, const int8_t* k_codes_dev, const float* k_scales_dev,
                                         const int8_t* k_signs_dev, const int8_t* v_codes_dev,
                                         const float* v_scales_dev, const int8_t* v_signs_dev, int64_t tokens,
                                         int kv_heads, int q_heads, int head_dim, const void* q_dev, int qdtype,
                                         float* out_dev, void* workspace_dev, size_t workspace_bytes,
                                         void* stream) {
  LQ_NVTX_RANGE("lq_attention_decode");
  return attention_fmt(lattice, k_codes_dev, k_scales_dev, k_signs_dev, v_codes_dev, v_scales_dev, v_signs_dev,
                       LQ_SCALE_TILE_F32, tokens, kv_heads, q_heads, head_dim, q_dev, qdtype, out_dev,
                       workspace_dev, workspace_bytes, stream);
}

extern "C" lq_status lq_attention_decode_ex(int lattice, const int8_t* k_codes_dev, const void* k_scales_dev,
                                            const int8_t* k_signs_dev, const int8_t* v_codes_dev,
                                            const void* v_scales_dev, const int8_t* v_signs_dev, int scale_format,
                                            int64_t tokens, int kv_heads, int q_heads, int head_dim,
                                            const void* q_dev, int qdtype, float* out_dev, void* workspace_dev,
                                            size_t workspace_bytes, void* stream) {
  LQ_NVTX_RANGE("lq_attention_decode_ex");
  return attention_fmt(lattice, k_codes_dev, k_scales_dev, k_signs_dev, v_codes_dev, v_scales_dev, v_signs_dev,
                       scale_format, tokens, kv_heads, q_heads, head_dim, q_dev, qdtype, out_dev, workspace_dev,
                       workspace_bytes, stream);
}

extern "C" lq_status lq_attention_decode_dithered(int lattice, const int8_t* k_codes_dev, const void* k_scales_dev,
                                                  const int8_t* k_signs_dev, uint64_t k_dither_seed,
                                                  const int8_t* v_codes_dev, const void* v_scales_dev,
                                                  const int8_t* v_signs_dev, uint64_t v_dither_seed, int scale_format,
                                                  int64_t tokens, int kv_heads, int q_heads, int head_dim,
                                                  const void* q_dev, int qdtype, float* out_dev, void* workspace_dev,
                                                  size_t workspace_bytes, void* stream) {
  LQ_NVTX_RANGE("lq_attention_decode_dithered");
  return attention_fmt(lattice, k_codes_dev, k_scales_dev, k_signs_dev, v_codes_dev, v_scales_dev, v_signs_dev,
                       scale_format, tokens, kv_heads, q_heads, head_dim, q_dev, qdtype, out_dev, workspace_dev,
                       workspace_bytes, stream, true, k_dither_seed, v_dither_seed);
}

extern "C" lq_status lq_rotate_blocks(const float* R_dev, int transpose, int head_dim, const void* X_dev,
                                      int xdtype, int64_t rows, int64_t cols, int64_t ldx, float* Y_dev,
                                      int64_t ldy, void* stream) {
  LQ_NVTX_RANGE("lq_rotate_blocks");
  if (head_dim != D) return LQ_ERR_UNSUPPORTED;
  if (xdtype != LQ_BF16 && xdtype != LQ_F32) return LQ_ERR_DTYPE;
  if (rows < 0 || cols <= 0 || cols % D != 0 || ldx < cols || ldy < cols) return LQ_ERR_SHAPE;
  if (rows == 0) return LQ_OK;
  if (R_dev == nullptr || X_dev == nullptr || Y_dev == nullptr) return LQ_ERR_ARG;
  if (!aligned4(R_dev) || !aligned4(Y_dev) || !aligned4(X_dev)) return LQ_ERR_ARG;
  RotArgs a;
  a.R = R_dev; a.transpose = transpose != 0; a.X = X_dev; a.xbf16 = (xdtype == LQ_BF16);
  a.rows = rows; a.blocks_per_row = cols / D; a.ldx = ldx; a.ldy = ldy; a.Y = Y_dev;
  const size_t smem = (size_t)(D * D + 8 * D) * sizeof(float);
  static bool attr = false;
  if (!attr) {
    if (cudaFuncSetAttribute(rotate_blocks_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess) {
      cudaGetLastError();
      return LQ_ERR_CUDA;
    }
    attr = true;
  }
  const int sms = device_sm_count();
  if (sms <= 0) return LQ_ERR_CUDA;
  const int64_t nvec = rows * (cols / D);
  int64_t grid = (nvec + 7) / 8;
  if (grid > (int64_t)sms * 3) grid = (int64_t)sms * 3;
  rotate_blocks_kernel<<<(unsigned)grid, 256, smem, (cudaStream_t)stream>>>(a);
  return check_launch();
}
