// Prefill GEMM from lattice codes on the 5th-generation tensor cores (tcgen05).
//
// HyperQuant page, mma="int8" paragraph: the decoded codes feed a tensor-core
// GEMM on every forward, the activation is rotated first, and no decoded
// weight is ever written to memory -- best for prefill / large batch.
//
//   Y[m, n] = sum_t s[n, t] * (X~_t[m] . p[n, t]),   X~ = H D X / sqrt(T).
//
// Two kernels:
//  1. gemm_prep_kernel:  X~ as fp16 (each token row scaled by a power of two
//     g_m so that |X~ g_m| < 2^15; A2 odd coordinates times sqrt 3), one
//     power-of-two factor f_n per weight row so that |p s f_n| < 2^15, and a
//     zeroed Y when several CTAs add into the same output.
//  2. gemm_kernel: persistent, warp-specialised CTA (one per SM) computing a
//     128 (weight rows) x 256 (tokens) output tile with
//       tcgen05.mma.cta_group::1.kind::f16  (A = decoded weights, B = X~, D fp32 in TMEM)
//     warp 0      TMA producer of int8 code tiles [128 x 64] (8-stage ring: the
//                 codes come from HBM, so this ring is the deep one)
//     warp 14     TMA producer of X~ tiles [256 x 64] (4-stage ring, mostly L2)
//     warp 1      allocates TMEM, one lane issues the MMAs
//     warps 2..9  decoders in two groups of four warps taking alternate K
//                 stages (four 16-code chunks per thread per stage): codes ->
//                 fp16 (c * s[n,t] * f_n / 2) written to a 2-stage ring of A
//                 tiles in the 128-byte-swizzled K-major layout, group g
//                 always into slot g
//     warps 10..13 epilogue: tcgen05.ld of the accumulator, Y = D / (f_n g_m)
//   Each ring has its own full/empty mbarriers, so code loads run far ahead of
//   the MMAs.  TMEM holds two 256-column accumulators so the epilogue of one
//   tile overlaps the main loop of the next.  Every mbarrier wait is bounded
//   (about a second of clock cycles); on expiry the kernel records
//   LQ_DEV_TIMEOUT and winds down.
// The GEMM is a programmatic dependent launch of the prep kernel: its
// prologue and the code producer run while the prep finishes, every other
// warp waits for the prep's results first.
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "lq_device.cuh"
#include "lq_host.h"

namespace lq {
namespace gemm {

constexpr int BM = 128;            // weight rows per tile (MMA M)
constexpr int BN = 256;            // tokens per tile (MMA N)
constexpr int BK = 64;             // K per pipeline stage
constexpr int kCodeStages = 8;     // int8 code ring (TMA -> decoders)
constexpr int kXStages = 4;        // X~ ring (TMA -> MMA): covers the L2 latency of a 32 KB tile
constexpr int kAStages = 2;        // decoded-weight ring (decoders -> MMA)
constexpr int kCodeBytes = BM * BK;          // int8 codes per stage:   8 KB
constexpr int kABytes = BM * BK * 2;         // fp16 decoded weights:   16 KB
constexpr int kXBytes = BN * BK * 2;         // fp16 activations:       32 KB
constexpr int kDecodeWarps = 8;
constexpr int kEpiWarp0 = 2 + kDecodeWarps;         // four epilogue warps
constexpr int kXWarp = kEpiWarp0 + 4;               // X~ producer
constexpr int kThreads = (kXWarp + 1) * 32;
constexpr int kDecodeGroups = 2;                    // decoder groups taking alternate K stages
constexpr int kGroupWarps = kDecodeWarps / kDecodeGroups;
constexpr int kGroupThreads = kGroupWarps * 32;
constexpr int kDecodePasses = BM * BK / 16 / kGroupThreads;  // 16-code chunks per thread per stage
static_assert(kDecodePasses * kGroupThreads * 16 == BM * BK, "a decoder group covers the code tile");
static_assert(kAStages % kDecodeGroups == 0, "each decoder group keeps to its own A slots");
constexpr int kEpiThreads = 128;
constexpr uint32_t kTmemCols = 512;          // two 256-column fp32 accumulators
constexpr long long kWaitCycles = 2000000000ll;  // about one second
// Wait limit of the wait-expiry self-test instantiation (about 0.1 ms).
constexpr long long kSelfTestWaitCycles = 200000ll;

struct Smem {
  // stage buffers come first and are 1024-byte aligned (128-byte swizzle atoms)
  alignas(1024) uint8_t x[kXStages][kXBytes];
  alignas(1024) uint8_t a[kAStages][kABytes];
  alignas(1024) uint8_t codes[kCodeStages][kCodeBytes];
  alignas(8) uint64_t full_c[kCodeStages];    // code tile landed
  alignas(8) uint64_t empty_c[kCodeStages];   // decoders finished reading it
  alignas(8) uint64_t full_x[kXStages];       // X~ tile landed
  alignas(8) uint64_t empty_x[kXStages];      // MMAs finished reading it
  alignas(8) uint64_t full_a[kAStages];       // decoders wrote the A tile
  alignas(8) uint64_t empty_a[kAStages];      // MMAs finished reading it
  alignas(8) uint64_t tmem_full[2];           // accumulator ready for the epilogue
  alignas(8) uint64_t tmem_empty[2];          // epilogue drained the accumulator
  alignas(8) uint64_t drain;                  // all issued MMAs complete (teardown)
  uint32_t tmem_base;
  int timeout;
};

struct Args {
  int64_t M, N, K;
  int tile, tiles_per_row;
  int n_tiles, m_tiles, splits, stages_per_split, k_stages;
  int64_t units;
  const void* scales;     // [N x K/T] or [N], in gemm_kernel's format SF
  const float* f;         // [N]   row factors 2^e
  const float* inv_g;     // [M]   1 / g_m
  float* Y32;             // [M x N] float32 output, or the float32 sums of the K splits
  __nv_bfloat16* Ybf;     // [M x N] bf16 output written directly (one K split), else null
  int32_t* status;
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait: false when the limit expired (the caller records the timeout)
// or when another thread of the CTA already recorded one.
template <long long LIMIT = kWaitCycles>
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* timeout_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*timeout_flag) return false;
    if (clock64() - t0 > LIMIT) {
      *timeout_flag = 1;
      return false;
    }
  }
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];"
      ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y)
      : "memory");
}

// Shared-memory matrix descriptor for tcgen05: K-major, 128-byte swizzle,
// 8-row atoms of 1024 bytes (stride byte offset), descriptor version 1.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t addr) {
  uint64_t d = 0;
  d |= (uint64_t)((addr >> 4) & 0x3FFFu);          // start address
  d |= (uint64_t)1u << 16;                          // leading byte offset (unused for this layout)
  d |= (uint64_t)(1024u >> 4) << 32;                // stride byte offset
  d |= (uint64_t)1u << 46;                          // descriptor version
  d |= (uint64_t)2u << 61;                          // 128-byte swizzle
  return d;
}

// Instruction descriptor: D f32, A/B f16, both K-major, N = 256, M = 128.
constexpr uint32_t kIdesc = (1u << 4) | (0u << 7) | (0u << 10) | ((uint32_t)(BN >> 3) << 17) |
                            ((uint32_t)(BM >> 4) << 24);

__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n"
      ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(kIdesc), "r"(accumulate));
}
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
               ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }


// 32 consecutive accumulator columns of this warp's 32 TMEM lanes, without
// waiting (tmem_wait_ld waits for every load the thread has issued).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// int8 codes (4 per word) -> f16x2 words (exact: the magic-number conversion of
// Kim et al. 2022, "Who Says Elephants Can't Run"), then times the fp16 scale.
__device__ __forceinline__ uint32_t code_pair_f16(uint32_t u, uint32_t sel, __half2 sf) {
  const uint32_t h = __byte_perm(u, 0x64646464u, sel);
  const __half2 off = __half2half2(__ushort_as_half((unsigned short)0x6480));  // 1152
  const __half2 v = __hmul2(__hsub2(*reinterpret_cast<const __half2*>(&h), off), sf);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// Storage type of one scale in format SF and its value.
template <int SF> struct ScaleType { using T = float; };
template <> struct ScaleType<LQ_SCALE_ROW_BF16> { using T = unsigned short; };
template <> struct ScaleType<LQ_SCALE_TILE_F16> { using T = __half; };
template <int SF>
__device__ __forceinline__ float scale_value(const typename ScaleType<SF>::T* p) {
  if constexpr (SF == LQ_SCALE_ROW_BF16) return __uint_as_float((uint32_t)__ldg(p) << 16);
  else if constexpr (SF == LQ_SCALE_TILE_F16) return __half2float(__ldg(p));
  else return __ldg(p);
}

// SF: the scale format (LQ_SCALE_*), fixed at compile time for the decode loop.
// SELF_TEST: the wait-expiry self-test (lq_gemm_wait_expiry_test): the X~
// producer issues no copies and every pipeline wait gives up after
// kSelfTestWaitCycles, so the MMA issuer's first wait on an X~ tile expires and
// the timeout path below runs.  Never instantiated for lq_gemm / lq_gemm_ex.
template <int SF, bool SELF_TEST = false>
__global__ void __launch_bounds__(kThreads, 1)
gemm_kernel(const __grid_constant__ CUtensorMap map_codes, const __grid_constant__ CUtensorMap map_x, Args a) {
  constexpr long long kLimit = SELF_TEST ? kSelfTestWaitCycles : kWaitCycles;
  extern __shared__ uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  volatile int* timeout = &sm.timeout;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kCodeStages; ++i) {
      mbar_init(&sm.full_c[i], 1);
      mbar_init(&sm.empty_c[i], kGroupWarps);    // one arrival per warp of the decoder group
    }
    for (int i = 0; i < kXStages; ++i) {
      mbar_init(&sm.full_x[i], 1);
      mbar_init(&sm.empty_x[i], 1);
    }
    for (int i = 0; i < kAStages; ++i) {
      mbar_init(&sm.full_a[i], kGroupWarps);
      mbar_init(&sm.empty_a[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sm.tmem_full[i], 1);
      mbar_init(&sm.tmem_empty[i], kEpiThreads / 32);   // one arrival per epilogue warp
    }
    mbar_init(&sm.drain, 1);
    sm.timeout = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 ::"r"(smem_u32(&sm.tmem_base)), "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  // launched as a programmatic dependent of the prep kernel: everything but
  // the code stream (written before the prep kernel started) waits for its
  // X~, factors and zeroed Y; the code producer fills its ring meanwhile
  if (warp != 0) asm volatile("griddepcontrol.wait;" ::: "memory");

  // unit u -> (n tile, m tile, K split) and its K-stage range
  auto unit_range = [&](int64_t u, int& nt, int& mt, int& k0, int& k1) {
    nt = (int)(u % a.n_tiles);
    const int64_t rest = u / a.n_tiles;
    mt = (int)(rest % a.m_tiles);
    const int sp = (int)(rest / a.m_tiles);
    k0 = sp * a.stages_per_split;
    k1 = min(a.k_stages, k0 + a.stages_per_split);
  };

  if (warp == 0 || warp == kXWarp) {
    // ------------------------------------------------------------ TMA producers
    // warp 0 streams code tiles, the last warp streams X~ tiles; each owns one ring.
    if (lane == 0) {
      const bool codes_side = (warp == 0);
      const int depth = codes_side ? kCodeStages : kXStages;
      uint64_t* full = codes_side ? sm.full_c : sm.full_x;
      uint64_t* empty = codes_side ? sm.empty_c : sm.empty_x;
      const uint32_t bytes = codes_side ? kCodeBytes : kXBytes;
      int s = 0;
      uint32_t ph = 0;
      int64_t issued = 0;
      for (int64_t u = blockIdx.x; u < a.units && !*timeout; u += gridDim.x) {
        int nt, mt, k0, k1;
        unit_range(u, nt, mt, k0, k1);
        for (int ks = k0; ks < k1; ++ks) {
          if (!mbar_wait<kLimit>(&empty[s], ph ^ 1, timeout)) break;
          if (SELF_TEST && !codes_side) {
            // the self-test's X~ producer never fills its ring
          } else {
            mbar_arrive_expect_tx(&full[s], bytes);
            if (codes_side) tma_load_2d(sm.codes[s], &map_codes, &full[s], ks * BK, nt * BM);
            else tma_load_2d(sm.x[s], &map_x, &full[s], ks * BK, mt * BN);
            ++issued;
          }
          if (++s == depth) { s = 0; ph ^= 1; }
        }
      }
      if (*timeout) {
        // let the copies already in flight land before the CTA exits (bounded)
        for (int i = 0; i < depth && i < issued; ++i) {
          if (--s < 0) { s = depth - 1; ph ^= 1; }
          const long long t0 = clock64();
          while (!mbar_try_wait(&full[s], ph) && clock64() - t0 < kWaitCycles) {
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int sa = 0, sx = 0;
      uint32_t pha = 0, phx = 0;
      int it = 0;
      for (int64_t u = blockIdx.x; u < a.units && !*timeout; u += gridDim.x, ++it) {
        int nt, mt, k0, k1;
        unit_range(u, nt, mt, k0, k1);
        const int acc = it & 1;
        const uint32_t acc_ph = (uint32_t)((it >> 1) & 1);
        if (!mbar_wait<kLimit>(&sm.tmem_empty[acc], acc_ph ^ 1, timeout)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem + (uint32_t)(acc * BN);
        bool ok = true;
        for (int ks = k0; ks < k1; ++ks) {
          if (!mbar_wait<kLimit>(&sm.full_a[sa], pha, timeout) || !mbar_wait<kLimit>(&sm.full_x[sx], phx, timeout)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(sm.a[sa]);
          const uint32_t x_addr = smem_u32(sm.x[sx]);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            mma_f16(d_tmem, sw128_desc(a_addr + kk * 32), sw128_desc(x_addr + kk * 32),
                    (ks > k0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(&sm.empty_a[sa]);
          mma_commit(&sm.empty_x[sx]);
          if (++sa == kAStages) { sa = 0; pha ^= 1; }
          if (++sx == kXStages) { sx = 0; phx ^= 1; }
        }
        if (!ok) break;
        mma_commit(&sm.tmem_full[acc]);
      }
    }
  } else if (warp < kEpiWarp0) {
    // ------------------------------------------------------------ decoders
    // kDecodeGroups groups of warps take turns over the K stages (group g the
    // stages whose CTA-wide index is g modulo the group count, which use the A
    // slots congruent to g), so each group has several MMA stage times to
    // decode its tile and the groups overlap.
    const int dgrp = (warp - 2) / kGroupWarps;
    const int d = threadIdx.x - 64 - dgrp * kGroupThreads;   // 0 .. kGroupThreads - 1
    const int rsub = d >> 2;                 // row within a pass
    const int c4 = d & 3;                    // 16-code chunk within the 64-code stage row
    const int stages_per_t = a.tile / BK;
    int64_t i = 0;                           // CTA-wide stage index
    for (int64_t u = blockIdx.x; u < a.units && !*timeout; u += gridDim.x) {
      int nt, mt, k0, k1;
      unit_range(u, nt, mt, k0, k1);
      constexpr int P = kDecodePasses;
      constexpr int kRowsPerPass = kGroupThreads / 4;
      // per pass: the row's first tile scale (the row's scale for the per-row format)
      using ST = typename ScaleType<SF>::T;
      constexpr int kTileStep = (SF == LQ_SCALE_ROW_BF16) ? 0 : 1;
      float fr[P];
      const ST* srow[P];
#pragma unroll
      for (int p = 0; p < P; ++p) {
        // rows past N (a ragged last weight tile) decode the TMA's zero fill
        // with a zero factor, reading the scales of row 0
        const int64_t row = (int64_t)nt * BM + kRowsPerPass * p + rsub;
        const bool in = row < a.N;
        fr[p] = in ? 0.5f * __ldg(a.f + row) : 0.f;
        srow[p] = reinterpret_cast<const ST*>(a.scales) + (in ? row : 0) * (kTileStep ? a.tiles_per_row : 1);
      }
      // scales of the current tile and (prefetched) of the next one
      float s_cur[P], s_nxt[P];
      int t_cur = k0 / stages_per_t;
#pragma unroll
      for (int p = 0; p < P; ++p) s_cur[p] = scale_value<SF>(srow[p] + kTileStep * t_cur);
#pragma unroll
      for (int p = 0; p < P; ++p)
        s_nxt[p] = (t_cur + 1 < a.tiles_per_row) ? scale_value<SF>(srow[p] + kTileStep * (t_cur + 1)) : 0.f;
      __half2 sf[P];
#pragma unroll
      for (int p = 0; p < P; ++p) sf[p] = __float2half2_rn(s_cur[p] * fr[p]);
      for (int ks = k0; ks < k1; ++ks, ++i) {
        if ((int)(i % kDecodeGroups) != dgrp) continue;    // another group's stage
        const int t = ks / stages_per_t;
        if (t != t_cur) {
          // the next tile's scales were loaded ahead; a group that skipped a
          // whole tile loads them now
#pragma unroll
          for (int p = 0; p < P; ++p) {
            const float sv = (t == t_cur + 1) ? s_nxt[p] : scale_value<SF>(srow[p] + kTileStep * t);
            sf[p] = __float2half2_rn(sv * fr[p]);
            s_nxt[p] = (t + 1 < a.tiles_per_row) ? scale_value<SF>(srow[p] + kTileStep * (t + 1)) : 0.f;
          }
          t_cur = t;
        }
        const int sc = (int)(i % kCodeStages), sa = (int)(i % kAStages);
        const uint32_t phc = (uint32_t)((i / kCodeStages) & 1), pha = (uint32_t)((i / kAStages) & 1);
        // warp-uniform waits: the warp arrives once per barrier below
        if (!__all_sync(0xffffffffu, mbar_wait<kLimit>(&sm.full_c[sc], phc, timeout))) break;
        if (!__all_sync(0xffffffffu, mbar_wait<kLimit>(&sm.empty_a[sa], pha ^ 1, timeout))) break;
        const uint8_t* cbase = sm.codes[sc];
        uint8_t* abase = sm.a[sa];
#pragma unroll
        for (int p = 0; p < P; ++p) {
          const int r = kRowsPerPass * p + rsub;
          const uint4 cw = *reinterpret_cast<const uint4*>(cbase + r * BK + 16 * c4);
          const uint32_t w[4] = {cw.x ^ 0x80808080u, cw.y ^ 0x80808080u, cw.z ^ 0x80808080u, cw.w ^ 0x80808080u};
          uint32_t o[8];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            o[2 * q] = code_pair_f16(w[q], 0x4140, sf[p]);
            o[2 * q + 1] = code_pair_f16(w[q], 0x4342, sf[p]);
          }
          // 128-byte swizzle: 16-byte chunk j of row r sits at chunk j ^ (r & 7)
          const int j0 = 2 * c4, j1 = 2 * c4 + 1;
          *reinterpret_cast<uint4*>(abase + r * 128 + ((j0 ^ (r & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
          *reinterpret_cast<uint4*>(abase + r * 128 + ((j1 ^ (r & 7)) << 4)) = make_uint4(o[4], o[5], o[6], o[7]);
        }
        // each thread orders its A writes before the tensor cores' reads; the
        // warp then arrives once on each barrier
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&sm.empty_c[sc]);           // this warp's code reads are done
          mbar_arrive(&sm.full_a[sa]);            // its part of the A tile is written
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;            // TMEM lane quarter this warp may access
    const int row_in_tile = quarter * 32 + lane;
    int it = 0;
    for (int64_t u = blockIdx.x; u < a.units; u += gridDim.x, ++it) {
      if (__any_sync(0xffffffffu, *timeout != 0)) break;
      int nt, mt, k0, k1;
      unit_range(u, nt, mt, k0, k1);
      const int acc = it & 1;
      const uint32_t acc_ph = (uint32_t)((it >> 1) & 1);
      const bool ready = mbar_wait<kLimit>(&sm.tmem_full[acc], acc_ph, timeout);
      if (!__all_sync(0xffffffffu, ready)) break;
      tc_fence_after();
      const int64_t n = (int64_t)nt * BM + row_in_tile;
      const bool row_in = n < a.N;                 // false in a ragged last weight tile
      const float inv_f = row_in ? 1.0f / __ldg(a.f + n) : 0.f;
      const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * BN);
      const bool atomic = a.splits > 1;
      // 32 columns per TMEM load, the next load in flight while a chunk is
      // written out; 1/g_m of the chunk's tokens loaded once per lane and
      // broadcast by shuffles
      const int64_t m_base = (int64_t)mt * BN;
      auto write_chunk = [&](const uint32_t (&r)[32], int c0, float g_lane) {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int64_t m = m_base + c0 + j;
          const float g = __shfl_sync(0xffffffffu, g_lane, j);
          if (row_in && m < a.M) {
            const float v = __uint_as_float(r[j]) * inv_f * g;
            if (atomic) atomicAdd(a.Y32 + m * a.N + n, v);
            else if (a.Ybf != nullptr) a.Ybf[m * a.N + n] = __float2bfloat16_rn(v);
            else a.Y32[m * a.N + n] = v;
          }
        }
      };
      auto g_of = [&](int c0) {
        const int64_t m = m_base + c0 + lane;
        return m < a.M ? __ldg(a.inv_g + m) : 0.f;
      };
      uint32_t ra[32], rb[32];
      __syncwarp();                                // tcgen05.ld is warp-collective
      tmem_ld32(taddr, ra);
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += 64) {
        const float ga = g_of(c0), gb = g_of(c0 + 32);
        tmem_wait_ld();                            // columns c0 .. c0 + 31 in ra
        tmem_ld32(taddr + (uint32_t)(c0 + 32), rb);
        write_chunk(ra, c0, ga);
        tmem_wait_ld();                            // columns c0 + 32 .. c0 + 63 in rb
        if (c0 + 64 < BN) tmem_ld32(taddr + (uint32_t)(c0 + 64), ra);
        write_chunk(rb, c0 + 32, gb);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.tmem_empty[acc]);
    }
  }

  // ---------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    if (lane == 0) {
      // every MMA this thread issued has completed once this commit arrives
      mma_commit(&sm.drain);
      const long long t0 = clock64();
      while (!mbar_try_wait(&sm.drain, 0) && clock64() - t0 < kWaitCycles) {
      }
    }
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
  }
  if (threadIdx.x == 0 && sm.timeout) raise_flag(a.status, LQ_DEV_TIMEOUT);
}

// ---------------------------------------------------------------- prep kernel
struct PrepArgs {
  const __nv_bfloat16* X;    // [M x K]
  const int8_t* signs;       // [K]
  int64_t M, N, K;
  int tile, lanes_per_tile, tiles_per_row, chunks_per_row;
  float inv_sqrt_tile;
  int a2;
  __half* Xt;                // [M x K]
  float* inv_g;              // [M]
  const void* scales;        // [N x K/T] or [N], format sfmt
  int sfmt;
  float* f;                  // [N]
  float* Y;                  // zeroed when zero_y
  int zero_y;
  int32_t* status;
};

// Blocks [0, M): one token row each (max |x| over the row, then the rotation
// with E columns per thread).  Blocks [M, M + ceil(N/16)): weight-row
// factors, one warp per row.
constexpr int kPrepThreads = 512;
constexpr int kPrepWarps = kPrepThreads / 32;

template <int E>
__global__ void __launch_bounds__(kPrepThreads) gemm_prep_kernel(PrepArgs a) {
  __shared__ float red[kPrepWarps];
  __shared__ float row_g;
  // the GEMM may be scheduled now (it waits for this grid's results)
  asm volatile("griddepcontrol.launch_dependents;");
  if (blockIdx.x >= a.M) {
    const int64_t n = (int64_t)(blockIdx.x - a.M) * kPrepWarps + (threadIdx.x >> 5);
    const int ln = threadIdx.x & 31;
    if (n >= a.N) return;
    float mx = 0.f;
    if (a.sfmt == LQ_SCALE_TILE_F32) {
      const float* sc = reinterpret_cast<const float*>(a.scales) + n * a.tiles_per_row;
      for (int t = ln; t < a.tiles_per_row; t += 32) mx = fmaxf(mx, __ldg(sc + t));
    } else {
      for (int t = ln; t < a.tiles_per_row; t += 32) mx = fmaxf(mx, load_scale(a.scales, a.sfmt, n, t, a.tiles_per_row));
    }
    for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    // |p s| <= 63.5 s; choose f = 2^e with 63.5 * max(s) * f in [2^14, 2^15)
    float fv = 1.f;
    if (mx > 0.f && isfinite(mx)) {
      const float top = 63.5f * mx;
      const int eb = (int)((__float_as_uint(top) >> 23) & 0xFFu) - 126;  // top in [2^(eb-1), 2^eb)
      const int ex = max(-126, min(127, 15 - eb));
      fv = __uint_as_float((uint32_t)(ex + 127) << 23);
    }
    if (ln == 0) a.f[n] = fv;
    return;
  }
  const int64_t m = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const __nv_bfloat16* xr = a.X + m * a.K;
  // pass 1: max |x| over the row
  float mx = 0.f;
  for (int64_t i = (int64_t)threadIdx.x * 8; i < a.K; i += kPrepThreads * 8) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(xr + i));
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int h = 0; h < 4; ++h)
      mx = fmaxf(mx, fmaxf(fabsf(__uint_as_float(w[h] << 16)), fabsf(__uint_as_float(w[h] & 0xFFFF0000u))));
  }
  for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if (lane == 0) red[warp] = mx;
  __syncthreads();
  if (threadIdx.x == 0) {
    float v = 0.f;
    for (int i = 0; i < kPrepWarps; ++i) v = fmaxf(v, red[i]);
    // |x~| <= sqrt(T) max|x| (times sqrt 3 for A2): g = 2^e with that bound in [2^13, 2^14]
    float gv = 1.f;
    if (!isfinite(v)) {
      raise_flag(a.status, LQ_DEV_NONFINITE);
    } else if (v > 0.f) {
      const float top = v * (1.0f / a.inv_sqrt_tile) * (a.a2 ? 1.7320508f : 1.f);
      const int eb = (int)((__float_as_uint(top) >> 23) & 0xFFu) - 126;
      const int ex = max(-126, min(127, 14 - eb));
      gv = __uint_as_float((uint32_t)(ex + 127) << 23);
    }
    row_g = gv;
    a.inv_g[m] = 1.0f / gv;
  }
  __syncthreads();
  const float g = row_g;
  if (a.zero_y) {
    for (int64_t i = threadIdx.x; i < a.N; i += kPrepThreads) a.Y[m * a.N + i] = 0.f;
  }
  // pass 2: rotate, E consecutive columns per thread (a tile spans T/E lanes of
  // one warp)
  const int lpt = a.tile / E;
  const int64_t groups = a.K / E;
  const float sc = a.inv_sqrt_tile * g;
  const float sc_odd = a.a2 ? sc * 1.7320508075688772f : sc;
  for (int64_t base = 0; base < groups; base += kPrepThreads) {
    const int64_t j = base + threadIdx.x;
    const bool active = j < groups;            // groups is a multiple of lpt: whole tiles
    const int64_t col0 = (active ? j : 0) * E;
    float v[E];
    if (active) {
      load_bf16_signed<E>(xr + col0, a.signs + col0, v);
    } else {
#pragma unroll
      for (int c = 0; c < E; ++c) v[c] = 0.f;
    }
    fwht_tile<E>(v, lpt, lane);
    if (active) {
      uint4* dst = reinterpret_cast<uint4*>(a.Xt + m * a.K + col0);
#pragma unroll
      for (int q = 0; q < E / 8; ++q) {
        uint32_t hw[4];
#pragma unroll
        for (int j2 = 0; j2 < 4; ++j2) {
          const __half2 h = __floats2half2_rn(v[8 * q + 2 * j2] * sc, v[8 * q + 2 * j2 + 1] * sc_odd);
          hw[j2] = *reinterpret_cast<const uint32_t*>(&h);
        }
        dst[q] = make_uint4(hw[0], hw[1], hw[2], hw[3]);
      }
    }
  }
}

// bf16 output of a K-split launch: Y = bf16(the float32 sums), nearest even.
__global__ void __launch_bounds__(256) gemm_to_bf16_kernel(const float* __restrict__ src,
                                                            __nv_bfloat16* __restrict__ dst, int64_t n) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; 4 * i < n; i += stride) {
    if (4 * i + 4 <= n) {
      const float4 v = __ldg(reinterpret_cast<const float4*>(src) + i);
      const __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
      uint2 o;
      o.x = *reinterpret_cast<const uint32_t*>(&lo);
      o.y = *reinterpret_cast<const uint32_t*>(&hi);
      *reinterpret_cast<uint2*>(dst + 4 * i) = o;
    } else {
      for (int64_t j = 4 * i; j < n; ++j) dst[j] = __float2bfloat16_rn(src[j]);
    }
  }
}

}  // namespace gemm
}  // namespace lq

using namespace lq;
using namespace lq::gemm;

namespace {

constexpr size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

struct GemmWorkspace {
  size_t xt, inv_g, f, acc, total;
};

// X~ fp16 [M x K], 1/g [M], f [N], and for a bf16 output the float32 sums
// [M x N] that the K splits add into.
GemmWorkspace gemm_layout(int64_t M, int64_t N, int64_t K, bool bf16_out) {
  GemmWorkspace w;
  w.xt = 0;
  w.inv_g = align256((size_t)M * (size_t)K * 2);
  w.f = w.inv_g + align256((size_t)M * 4);
  w.acc = w.f + align256((size_t)N * 4);
  w.total = w.acc + (bf16_out ? align256((size_t)M * (size_t)N * 4) : 0);
  return w;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
    else
      cudaGetLastError();
  });
  return fn;
}

bool make_map_2d(CUtensorMap* map, CUtensorMapDataType dt, size_t esize, const void* base, uint64_t inner,
                 uint64_t outer, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {inner * esize};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Split K so that the work units fill the GPU without a long tail.
int choose_splits(int64_t tiles, int k_stages, int sms) {
  int best = 1;
  double best_eff = 0.0;
  for (int s = 1; s <= 8; ++s) {
    if (k_stages / s < 8) break;
    const int64_t units = tiles * s;
    const double waves = (double)units / sms;
    const double eff = waves / (double)((units + sms - 1) / sms) - 0.01 * (s - 1);
    if (eff > best_eff + 1e-9) { best_eff = eff; best = s; }
  }
  return best;
}

}  // namespace

extern "C" size_t lq_gemm_workspace_size(int64_t M, int64_t N, int64_t K, int ydtype) {
  if (M <= 0 || N <= 0 || K <= 0 || (ydtype != LQ_F32 && ydtype != LQ_BF16)) return 0;
  return gemm_layout(M, N, K, ydtype == LQ_BF16).total;
}

namespace {

lq_status gemm_fmt(int lattice, const int8_t* codes_dev, const void* scales_dev, int sfmt, const int8_t* signs_dev,
                   int64_t N, int64_t K, int tile, const uint16_t* X_dev, int64_t M, void* Y_dev, int ydtype,
                   void* workspace_dev, int32_t* dev_status_dev, void* stream, bool self_test = false) {
  if (sfmt != LQ_SCALE_TILE_F32 && sfmt != LQ_SCALE_ROW_BF16 && sfmt != LQ_SCALE_TILE_F16) return LQ_ERR_ARG;
  if (ydtype != LQ_F32 && ydtype != LQ_BF16) return LQ_ERR_DTYPE;
  const bool bf16_out = ydtype == LQ_BF16;
  const uintptr_t salign = (sfmt == LQ_SCALE_TILE_F32) ? 3u : 1u;
  lq_status st = validate_common(lattice, N, K, tile);
  if (st != LQ_OK) return st;
  if (M < 0) return LQ_ERR_SHAPE;
  if (K % BK != 0) return LQ_ERR_SHAPE;       // implied by K % tile == 0
  if (M > (int64_t(1) << 31) || N > (int64_t(1) << 31)) return LQ_ERR_SHAPE;
  if (M == 0 || N == 0) return LQ_OK;
  if (codes_dev == nullptr || scales_dev == nullptr || signs_dev == nullptr || X_dev == nullptr ||
      Y_dev == nullptr || workspace_dev == nullptr)
    return LQ_ERR_ARG;
  if (!aligned16(codes_dev) || !aligned16(signs_dev) || !aligned16(X_dev) || !aligned16(Y_dev) ||
      (reinterpret_cast<uintptr_t>(workspace_dev) & 255u) != 0 ||
      (reinterpret_cast<uintptr_t>(scales_dev) & salign) != 0 ||
      (dev_status_dev != nullptr && !aligned4(dev_status_dev)))
    return LQ_ERR_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  const int sms = device_sm_count();
  if (sms <= 0) return LQ_ERR_CUDA;

  const GemmWorkspace lay = gemm_layout(M, N, K, bf16_out);
  char* ws = reinterpret_cast<char*>(workspace_dev);
  __half* Xt = reinterpret_cast<__half*>(ws + lay.xt);
  float* inv_g = reinterpret_cast<float*>(ws + lay.inv_g);
  float* f = reinterpret_cast<float*>(ws + lay.f);

  Args a;
  a.M = M; a.N = N; a.K = K; a.tile = tile; a.tiles_per_row = (int)(K / tile);
  a.n_tiles = (int)((N + BM - 1) / BM);
  a.m_tiles = (int)((M + BN - 1) / BN);
  a.k_stages = (int)(K / BK);
  a.splits = choose_splits((int64_t)a.n_tiles * a.m_tiles, a.k_stages, sms);
  a.stages_per_split = (a.k_stages + a.splits - 1) / a.splits;
  a.splits = (a.k_stages + a.stages_per_split - 1) / a.stages_per_split;
  a.units = (int64_t)a.n_tiles * a.m_tiles * a.splits;
  a.scales = scales_dev; a.f = f; a.inv_g = inv_g; a.status = dev_status_dev;
  // float32 output: the kernel writes (or, split along K, adds into) Y.  bf16
  // output: one split writes bf16 directly; several add into float32 sums in
  // the workspace that a last kernel rounds to bf16.
  const bool via_acc = bf16_out && a.splits > 1;
  a.Y32 = bf16_out ? (via_acc ? reinterpret_cast<float*>(ws + lay.acc) : nullptr) : reinterpret_cast<float*>(Y_dev);
  a.Ybf = (bf16_out && !via_acc) ? reinterpret_cast<__nv_bfloat16*>(Y_dev) : nullptr;

  PrepArgs p;
  p.X = reinterpret_cast<const __nv_bfloat16*>(X_dev); p.signs = signs_dev; p.M = M; p.N = N; p.K = K;
  p.tile = tile; p.lanes_per_tile = tile / kLaneElems; p.tiles_per_row = (int)(K / tile);
  p.chunks_per_row = (int)((K + kChunkCols - 1) / kChunkCols);
  p.inv_sqrt_tile = (float)(1.0 / sqrt((double)tile));
  p.a2 = (lattice == LQ_A2);
  p.Xt = Xt; p.inv_g = inv_g; p.scales = scales_dev; p.sfmt = sfmt; p.f = f; p.Y = a.Y32; p.zero_y = a.splits > 1;
  p.status = dev_status_dev;
  const int64_t prep_blocks = M + (N + kPrepWarps - 1) / kPrepWarps;
  const int E = act_elems_for_tile(tile);
  if (E == 16) gemm_prep_kernel<16><<<(unsigned)prep_blocks, kPrepThreads, 0, s>>>(p);
  else if (E == 32) gemm_prep_kernel<32><<<(unsigned)prep_blocks, kPrepThreads, 0, s>>>(p);
  else gemm_prep_kernel<64><<<(unsigned)prep_blocks, kPrepThreads, 0, s>>>(p);
  st = check_launch();
  if (st != LQ_OK) return st;

  CUtensorMap map_codes, map_x;
  if (!make_map_2d(&map_codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, codes_dev, (uint64_t)K, (uint64_t)N, BK, BM,
                   CU_TENSOR_MAP_SWIZZLE_NONE))
    return LQ_ERR_CUDA;
  if (!make_map_2d(&map_x, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, Xt, (uint64_t)K, (uint64_t)M, BK, BN,
                   CU_TENSOR_MAP_SWIZZLE_128B))
    return LQ_ERR_CUDA;

  const size_t smem = sizeof(Smem) + 1024;
  static_assert(sizeof(Smem) + 1024 <= 227 * 1024, "shared memory budget");
  static bool attr_set = false;
  if (!attr_set) {
    if (cudaFuncSetAttribute(gemm_kernel<LQ_SCALE_TILE_F32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess ||
        cudaFuncSetAttribute(gemm_kernel<LQ_SCALE_ROW_BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess ||
        cudaFuncSetAttribute(gemm_kernel<LQ_SCALE_TILE_F16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess ||
        cudaFuncSetAttribute(gemm_kernel<LQ_SCALE_TILE_F32, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess) {
      cudaGetLastError();
      return LQ_ERR_CUDA;
    }
    attr_set = true;
  }
  const int64_t grid = a.units < sms ? a.units : sms;
  // programmatic dependent launch behind the prep kernel
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  auto kern = self_test                       ? gemm_kernel<LQ_SCALE_TILE_F32, true>
              : (sfmt == LQ_SCALE_ROW_BF16) ? gemm_kernel<LQ_SCALE_ROW_BF16>
              : (sfmt == LQ_SCALE_TILE_F16) ? gemm_kernel<LQ_SCALE_TILE_F16>
                                            : gemm_kernel<LQ_SCALE_TILE_F32>;
  if (cudaLaunchKernelEx(&cfg, kern, map_codes, map_x, a) != cudaSuccess) {
    cudaGetLastError();
    return LQ_ERR_CUDA;
  }
  if (!via_acc) return LQ_OK;
  const int64_t n_out = M * N;
  const int64_t cvt_blocks = std::min<int64_t>((n_out / 4 + 255) / 256 + 1, (int64_t)sms * 8);
  gemm_to_bf16_kernel<<<(unsigned)cvt_blocks, 256, 0, s>>>(a.Y32, reinterpret_cast<__nv_bfloat16*>(Y_dev), n_out);
  return check_launch();
}

}  // namespace

extern "C" lq_status lq_gemm(int lattice, const int8_t* codes_dev, const float* scales_dev,
                             const int8_t* signs_dev, int64_t N, int64_t K, int tile,
                             const uint16_t* X_dev, int64_t M, void* Y_dev, int ydtype, void* workspace_dev,
                             int32_t* dev_status_dev, void* stream) {
  LQ_NVTX_RANGE("lq_gemm");
  return gemm_fmt(lattice, codes_dev, scales_dev, LQ_SCALE_TILE_F32, signs_dev, N, K, tile, X_dev, M, Y_dev, ydtype,
                  workspace_dev, dev_status_dev, stream);
}

extern "C" lq_status lq_gemm_ex(int lattice, const int8_t* codes_dev, const void* scales_dev, int scale_format,
                                const int8_t* signs_dev, int64_t N, int64_t K, int tile, const uint16_t* X_dev,
                                int64_t M, void* Y_dev, int ydtype, void* workspace_dev, int32_t* dev_status_dev,
                                void* stream) {
  LQ_NVTX_RANGE("lq_gemm_ex");
  return gemm_fmt(lattice, codes_dev, scales_dev, scale_format, signs_dev, N, K, tile, X_dev, M, Y_dev, ydtype,
                  workspace_dev, dev_status_dev, stream);
}

extern "C" lq_status lq_gemm_wait_expiry_test(int lattice, const int8_t* codes_dev, const float* scales_dev,
                                              const int8_t* signs_dev, int64_t N, int64_t K, int tile,
                                              const uint16_t* X_dev, int64_t M, void* Y_dev, int ydtype,
                                              void* workspace_dev, int32_t* dev_status_dev, void* stream) {
  LQ_NVTX_RANGE("lq_gemm_wait_expiry_test");
  if (dev_status_dev == nullptr) return LQ_ERR_ARG;
  return gemm_fmt(lattice, codes_dev, scales_dev, LQ_SCALE_TILE_F32, signs_dev, N, K, tile, X_dev, M, Y_dev, ydtype,
                  workspace_dev, dev_status_dev, stream, true);
}
