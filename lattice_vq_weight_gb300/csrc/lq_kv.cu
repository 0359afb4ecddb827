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
// Kernel 1 rotates the queries.  Kernel 2 (attn_partial_kernel in
// lq_kv_kernel.cuh; one CTA per kv head and token range, four warps): each
// warp takes 32 tokens at a time -- lane = token for the scores (128 codes
// against the group's rotated queries), an online softmax, then lane = 4
// dimensions for the value sum over those 32 tokens; its variants subtract a
// subtractive dither or decode Rice-coded caches on chip.  Kernel 3 merges
// the ranges and rotates the result back.
#include "lq_kv_kernel.cuh"

namespace lq {
namespace kv {

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

// The Rice-coded caches' partial attention of one lattice and norm format
// (the instantiations live in the objects built from lq_kv_rice.cu).
lq_status launch_partial_rice(const AttnArgs& a, int lattice, int group, bool h, unsigned grid, cudaStream_t s) {
  switch (lattice) {
    case LQ_E8: return h ? launch_partial_rice_lh<LQ_E8, true>(a, group, grid, s)
                         : launch_partial_rice_lh<LQ_E8, false>(a, group, grid, s);
    case LQ_D4: return h ? launch_partial_rice_lh<LQ_D4, true>(a, group, grid, s)
                         : launch_partial_rice_lh<LQ_D4, false>(a, group, grid, s);
    case LQ_A2: return h ? launch_partial_rice_lh<LQ_A2, true>(a, group, grid, s)
                         : launch_partial_rice_lh<LQ_A2, false>(a, group, grid, s);
    default:    return h ? launch_partial_rice_lh<LQ_Z1, true>(a, group, grid, s)
                         : launch_partial_rice_lh<LQ_Z1, false>(a, group, grid, s);
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

// K and V caches held as Rice streams (lq_rice_encode with tile = head_dim).
struct RiceKV {
  const uint32_t* krs;
  int64_t knw;
  const uint32_t* koff;
  const uint32_t* vrs;
  int64_t vnw;
  const uint32_t* voff;
};

lq_status attention_fmt(int lattice, const int8_t* k_codes_dev, const void* k_scales_dev,
                        const int8_t* k_signs_dev, const int8_t* v_codes_dev, const void* v_scales_dev,
                        const int8_t* v_signs_dev, int sfmt, int64_t tokens, int kv_heads, int q_heads, int head_dim,
                        const void* q_dev, int qdtype, float* out_dev, void* workspace_dev, size_t workspace_bytes,
                        void* stream, bool dither = false, uint64_t k_dither_seed = 0, uint64_t v_dither_seed = 0,
                        const RiceKV* rice = nullptr) {
  if (!valid_lattice(lattice)) return LQ_ERR_ARG;
  if (sfmt != LQ_SCALE_TILE_F32 && sfmt != LQ_SCALE_TILE_F16) return LQ_ERR_ARG;
  const uintptr_t salign = (sfmt == LQ_SCALE_TILE_F32) ? 3u : 1u;
  if (head_dim != D) return LQ_ERR_UNSUPPORTED;
  if (qdtype != LQ_BF16 && qdtype != LQ_F32) return LQ_ERR_DTYPE;
  if (tokens <= 0 || kv_heads <= 0 || q_heads <= 0 || q_heads % kv_heads != 0) return LQ_ERR_SHAPE;
  const int group = q_heads / kv_heads;
  if (group != 1 && group != 2 && group != 4 && group != 8) return LQ_ERR_UNSUPPORTED;
  if (tokens > (int64_t(1) << 31)) return LQ_ERR_SHAPE;
  if (k_scales_dev == nullptr || k_signs_dev == nullptr || v_scales_dev == nullptr || v_signs_dev == nullptr ||
      q_dev == nullptr || out_dev == nullptr || workspace_dev == nullptr)
    return LQ_ERR_ARG;
  if (rice != nullptr) {
    if (rice->krs == nullptr || rice->koff == nullptr || rice->vrs == nullptr || rice->voff == nullptr ||
        !aligned4(rice->krs) || !aligned4(rice->koff) || !aligned4(rice->vrs) || !aligned4(rice->voff) ||
        rice->knw <= 0 || rice->vnw <= 0)
      return LQ_ERR_ARG;
  } else if (k_codes_dev == nullptr || v_codes_dev == nullptr || !aligned16(k_codes_dev) || !aligned16(v_codes_dev)) {
    return LQ_ERR_ARG;
  }
  if ((reinterpret_cast<uintptr_t>(k_scales_dev) & salign) || (reinterpret_cast<uintptr_t>(v_scales_dev) & salign) ||
      !aligned4(out_dev) || !aligned4(workspace_dev))
    return LQ_ERR_ARG;
  if (workspace_bytes < lq_attention_workspace_size(tokens, kv_heads, q_heads, head_dim)) return LQ_ERR_SHAPE;
  AttnArgs a;
  a.kc = k_codes_dev; a.ks = k_scales_dev; a.ksg = k_signs_dev;
  a.vc = v_codes_dev; a.vs = v_scales_dev; a.vsg = v_signs_dev;
  a.sfmt = sfmt;
  a.kdseed = k_dither_seed;
  a.vdseed = v_dither_seed;
  a.krs = rice ? rice->krs : nullptr; a.knw = rice ? rice->knw : 0; a.koff = rice ? rice->koff : nullptr;
  a.vrs = rice ? rice->vrs : nullptr; a.vnw = rice ? rice->vnw : 0; a.voff = rice ? rice->voff : nullptr;
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
  if (dither) st = launch_partial_dithered(a, lattice, group, h, grid, s);
  else if (rice != nullptr) st = launch_partial_rice(a, lattice, group, h, grid, s);
  else st = launch_partial_groups<0, 0>(a, group, h, grid, s);
  if (st != LQ_OK) return st;
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

extern "C" lq_status lq_attention_decode_rice(int lattice, const uint32_t* k_stream_dev, size_t k_stream_bytes,
                                              const uint32_t* k_offsets_dev, const void* k_scales_dev,
                                              const int8_t* k_signs_dev, const uint32_t* v_stream_dev,
                                              size_t v_stream_bytes, const uint32_t* v_offsets_dev,
                                              const void* v_scales_dev, const int8_t* v_signs_dev, int scale_format,
                                              int64_t tokens, int kv_heads, int q_heads, int head_dim,
                                              const void* q_dev, int qdtype, float* out_dev, void* workspace_dev,
                                              size_t workspace_bytes, void* stream) {
  LQ_NVTX_RANGE("lq_attention_decode_rice");
  if (tokens > 0 && kv_heads > 0 && (uint64_t)tokens * (uint64_t)kv_heads * D > ((uint64_t)1 << 28))
    return LQ_ERR_SHAPE;   // the format's 32-bit bit offsets cover at most 2^28 weights per stream
  RiceKV r;
  r.krs = k_stream_dev; r.knw = (int64_t)(k_stream_bytes / 4); r.koff = k_offsets_dev;
  r.vrs = v_stream_dev; r.vnw = (int64_t)(v_stream_bytes / 4); r.voff = v_offsets_dev;
  return attention_fmt(lattice, nullptr, k_scales_dev, k_signs_dev, nullptr, v_scales_dev, v_signs_dev, scale_format,
                       tokens, kv_heads, q_heads, head_dim, q_dev, qdtype, out_dev, workspace_dev, workspace_bytes,
                       stream, false, 0, 0, &r);
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
