// Rice format of lattice codes: encoder, decoder and the GEMV that reads the
// stream directly.
//
// HyperQuant page, "Key algorithmic ingredients": the bits the lattice fixes
// are dropped without loss and the remaining integers Rice coded; mma="bf16"
// paragraph: the weight is stored as that stream (~4 bps) and the GEMV reads
// it without an int8 copy.  Rice codes:
// R. F. Rice, JPL Publication 79-22 (1979).
//
// Format (see include/lq.h): per (row, tile) one segment -- K in 3 bits, then
// per block [parity bit] and the zigzag Rice codes of the halved codes, the
// last one without its implied low bit for E8 and D4.  Bits are LSB-first in
// 32-bit words; segment offsets (bits) are stored per (row, tile).
//
// Kernels: one thread per segment for the encoder passes (lengths, then bits
// with atomicOr into the zeroed stream) and the decoder; a three-pass scan turns
// lengths into offsets.  The GEMV gives each lane one row of a 32-row group:
// the lane decodes its row 64 columns at a time, from a shared-memory ring
// that the warp fills with coalesced background copies of the rows' stream,
// into the fragment layout of the int8-code GEMV, and the warp runs fp16 MMAs.
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "lq_act.cuh"
#include "lq_device.cuh"
#include "lq_host.h"
#include "lq_rice.cuh"

namespace lq {
namespace rice {

// Block of n codes -> parity bit and n zigzag symbols; `bad` when the codes do
// not have the pinned bits the format strips.
template <int LAT>
__device__ __forceinline__ void strip(const int (&c)[Fmt<LAT>::n], uint32_t& k, uint32_t (&z)[Fmt<LAT>::n],
                                      bool& bad) {
  constexpr int n = Fmt<LAT>::n;
  k = (uint32_t)c[0] & 1u;
  int u[n];
  int sum = 0;
#pragma unroll
  for (int i = 0; i < n; ++i) {
    if (((uint32_t)c[i] & 1u) != (Fmt<LAT>::parity ? k : 0u)) bad = true;
    u[i] = c[i] >> 1;
    sum += u[i];
  }
  if constexpr (Fmt<LAT>::even_sum) {
    if (sum & 1) bad = true;
    u[n - 1] >>= 1;
  }
#pragma unroll
  for (int i = 0; i < n; ++i) z[i] = zigzag(u[i]);
}

// n codes as bytes at p (aligned to n bytes).
template <int n>
__device__ __forceinline__ void store_block(uint8_t* p, const int (&c)[n]) {
  if constexpr (n == 8) {
    const uint32_t lo = ((uint32_t)c[0] & 0xFFu) | (((uint32_t)c[1] & 0xFFu) << 8) |
                        (((uint32_t)c[2] & 0xFFu) << 16) | ((uint32_t)c[3] << 24);
    const uint32_t hi = ((uint32_t)c[4] & 0xFFu) | (((uint32_t)c[5] & 0xFFu) << 8) |
                        (((uint32_t)c[6] & 0xFFu) << 16) | ((uint32_t)c[7] << 24);
    *reinterpret_cast<uint2*>(p) = make_uint2(lo, hi);
  } else if constexpr (n == 4) {
    *reinterpret_cast<uint32_t*>(p) = ((uint32_t)c[0] & 0xFFu) | (((uint32_t)c[1] & 0xFFu) << 8) |
                                      (((uint32_t)c[2] & 0xFFu) << 16) | ((uint32_t)c[3] << 24);
  } else if constexpr (n == 2) {
    *reinterpret_cast<uint16_t*>(p) = (uint16_t)(((uint32_t)c[0] & 0xFFu) | (((uint32_t)c[1] & 0xFFu) << 8));
  } else {
    *p = (uint8_t)c[0];
  }
}

// Writer into a zeroed stream: whole words and the partial last word by atomicOr
// (a segment's first and last words are shared with its neighbours).
struct BitWriter {
  uint32_t* w;
  int64_t word;
  uint64_t acc;
  int nacc;
  __device__ __forceinline__ void init(uint32_t* words, uint64_t pos) {
    w = words;
    word = (int64_t)(pos >> 5);
    nacc = (int)(pos & 31u);
    acc = 0;
  }
  __device__ __forceinline__ void put(uint32_t v, int nbits) {   // nbits <= 32
    acc |= (uint64_t)v << nacc;
    nacc += nbits;
    if (nacc >= 32) {
      if ((uint32_t)acc) atomicOr(w + word, (uint32_t)acc);
      ++word;
      acc >>= 32;
      nacc -= 32;
    }
  }
  __device__ __forceinline__ void rice(uint32_t z, int K) {
    uint32_t q = z >> K;
    while (q >= 32) { put(0xFFFFFFFFu, 32); q -= 32; }
    put((1u << q) - 1u, (int)q + 1);                 // q ones and a zero (q <= 31)
    if (K) put(z & ((1u << K) - 1u), K);
  }
  __device__ __forceinline__ void flush() {
    if (nacc > 0 && (uint32_t)acc) atomicOr(w + word, (uint32_t)acc);
  }
};

struct SegArgs {
  const int8_t* codes;
  int64_t rows, cols;
  int tile, tiles_per_row;
  int64_t segments;
  uint32_t* len;         // [segments] bits
  uint8_t* kpar;         // [segments] chosen K
  const uint32_t* off;   // [segments] bit offsets (write pass)
  uint32_t* stream;
  int32_t* status;
};

// Codes of segment i, 16 bytes at a time: f(c[16]).
template <typename F>
__device__ __forceinline__ void for_each_chunk(const SegArgs& a, int64_t i, F f) {
  const int64_t r = i / a.tiles_per_row;
  const int t = (int)(i - r * a.tiles_per_row);
  const uint4* src = reinterpret_cast<const uint4*>(a.codes + r * a.cols + (int64_t)t * a.tile);
  for (int q = 0; q < a.tile / 16; ++q) {
    const uint4 v = __ldg(src + q);
    const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
    int c[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) c[j] = (int)(int8_t)(wv[j >> 2] >> (8 * (j & 3)));
    f(c);
  }
}

// Pass 1: the length of every segment for every K, keep the shortest.
template <int LAT>
__global__ void __launch_bounds__(256) seg_length_kernel(SegArgs a) {
  constexpr int n = Fmt<LAT>::n;
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= a.segments) return;
  uint32_t sh[kKMax + 1] = {};
  uint32_t nsym = 0;
  bool bad = false;
  for_each_chunk(a, i, [&](const int (&c)[16]) {
#pragma unroll
    for (int j = 0; j < 16; j += n) {
      int blk[n];
#pragma unroll
      for (int e = 0; e < n; ++e) blk[e] = c[j + e];
      uint32_t k, z[n];
      strip<LAT>(blk, k, z, bad);
#pragma unroll
      for (int e = 0; e < n; ++e)
#pragma unroll
        for (int K = 0; K <= kKMax; ++K) sh[K] += z[e] >> K;
      nsym += n;
    }
  });
  uint32_t best = 0xFFFFFFFFu;
  int bk = 0;
#pragma unroll
  for (int K = 0; K <= kKMax; ++K) {
    const uint32_t l = sh[K] + nsym * (uint32_t)(1 + K);
    if (l < best) { best = l; bk = K; }
  }
  const uint32_t blocks = (uint32_t)(a.tile / n);
  a.len[i] = (uint32_t)kKBits + (Fmt<LAT>::parity ? blocks : 0u) + best;
  a.kpar[i] = (uint8_t)bk;
  if (bad) raise_flag(a.status, LQ_DEV_FORMAT);
}

// Pass 3: write every segment's bits at its offset.
template <int LAT>
__global__ void __launch_bounds__(256) seg_write_kernel(SegArgs a) {
  constexpr int n = Fmt<LAT>::n;
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= a.segments) return;
  const int K = a.kpar[i];
  BitWriter wr;
  wr.init(a.stream, a.off[i]);
  wr.put((uint32_t)K, kKBits);
  bool bad = false;
  for_each_chunk(a, i, [&](const int (&c)[16]) {
#pragma unroll
    for (int j = 0; j < 16; j += n) {
      int blk[n];
#pragma unroll
      for (int e = 0; e < n; ++e) blk[e] = c[j + e];
      uint32_t k, z[n];
      strip<LAT>(blk, k, z, bad);
      if (Fmt<LAT>::parity) wr.put(k, 1);
#pragma unroll
      for (int e = 0; e < n; ++e) wr.rice(z[e], K);
    }
  });
  wr.flush();
}

// Exclusive scan of the segment lengths (three passes; 4096 values per block).
constexpr int kScanThreads = 1024;
constexpr int kScanPer = 4;
constexpr int64_t kScanBlock = (int64_t)kScanThreads * kScanPer;

__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t* warp_sums, uint32_t& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    uint32_t s = warp_sums[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    warp_sums[lane] = s;
  }
  __syncthreads();
  total = warp_sums[31];
  const uint32_t before = warp > 0 ? warp_sums[warp - 1] : 0u;
  __syncthreads();
  return before + x - v;
}

__global__ void __launch_bounds__(kScanThreads) scan_local_kernel(const uint32_t* len, uint32_t* off,
                                                                  uint32_t* block_sums, int64_t n) {
  __shared__ uint32_t ws[32];
  const int64_t base = blockIdx.x * kScanBlock + (int64_t)threadIdx.x * kScanPer;
  uint32_t v[kScanPer], s = 0;
#pragma unroll
  for (int j = 0; j < kScanPer; ++j) {
    v[j] = (base + j < n) ? len[base + j] : 0u;
    s += v[j];
  }
  uint32_t total;
  uint32_t run = block_exclusive_scan(s, ws, total);
#pragma unroll
  for (int j = 0; j < kScanPer; ++j) {
    if (base + j < n) off[base + j] = run;
    run += v[j];
  }
  if (threadIdx.x == 0) block_sums[blockIdx.x] = total;
}

__global__ void __launch_bounds__(kScanThreads) scan_sums_kernel(uint32_t* block_sums, int64_t nb) {
  __shared__ uint32_t ws[32];
  const int64_t base = (int64_t)threadIdx.x * kScanPer;
  uint32_t v[kScanPer], s = 0;
#pragma unroll
  for (int j = 0; j < kScanPer; ++j) {
    v[j] = (base + j < nb) ? block_sums[base + j] : 0u;
    s += v[j];
  }
  uint32_t total;
  uint32_t run = block_exclusive_scan(s, ws, total);
#pragma unroll
  for (int j = 0; j < kScanPer; ++j) {
    if (base + j < nb) block_sums[base + j] = run;
    run += v[j];
  }
}

__global__ void __launch_bounds__(kScanThreads) scan_add_kernel(uint32_t* off, const uint32_t* block_sums,
                                                                const uint32_t* len, int64_t n,
                                                                uint64_t* total_bits) {
  const int64_t base = blockIdx.x * kScanBlock + (int64_t)threadIdx.x * kScanPer;
  const uint32_t add = block_sums[blockIdx.x];
#pragma unroll
  for (int j = 0; j < kScanPer; ++j) {
    if (base + j < n) {
      off[base + j] += add;
      if (base + j == n - 1 && total_bits != nullptr) *total_bits = (uint64_t)off[base + j] + len[base + j];
    }
  }
}

// Decoder: one thread per segment.
struct DecArgs {
  const uint32_t* stream;
  int64_t nwords;
  const uint32_t* off;
  int64_t rows, cols;
  int tile, tiles_per_row;
  int64_t segments;
  int8_t* codes;
};

template <int LAT>
__global__ void __launch_bounds__(256) seg_decode_kernel(DecArgs a) {
  constexpr int n = Fmt<LAT>::n;
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= a.segments) return;
  const int64_t r = i / a.tiles_per_row;
  const int t = (int)(i - r * a.tiles_per_row);
  BitReader rd;
  rd.init(a.stream, a.nwords, a.off[i]);
  const int K = (int)rd.get(kKBits);
  uint4* dst = reinterpret_cast<uint4*>(a.codes + r * a.cols + (int64_t)t * a.tile);
  for (int q = 0; q < a.tile / 16; ++q) {
    uint32_t wv[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int j = 0; j < 16; j += n) {
      int c[n];
      decode_block<LAT>(rd, K, c);
#pragma unroll
      for (int e = 0; e < n; ++e) wv[(j + e) >> 2] |= ((uint32_t)c[e] & 0xFFu) << (8 * ((j + e) & 3));
    }
    dst[q] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
  }
}

// ---------------------------------------------------------------- GEMV
struct GemvRiceArgs {
  const uint32_t* stream;
  int64_t nwords;
  const uint32_t* off;     // [rows x tiles]
  const float* scales;
  int64_t rows, cols;
  int tile, tiles_per_row, batch;
  const __half* xh;
  const float* xs;
  float* y;
  int64_t items;           // row groups of 32 x tiles
  int64_t warps;
};

// Per row of a warp's 32-row group, a ring of two 32-word chunks of the row's
// part of the stream: the region starts at the 32-word line holding the row's
// first segment, and word w of it (w from the region's start; s = the word of
// the segment's first bit) sits at ring index (w - s) & 63, so that rows that
// have decoded the same number of codes read distinct banks.  Index 64 holds a
// copy of index 0, so that a two-word window read never wraps.  The odd row
// stride (65 words) spreads the rows over the banks.
constexpr int kRingWords = 65;

// Items are (32-row group, tile) pairs; warp w takes [w I / W, (w+1) I / W).
// Lane l decodes row 32 grp + l, 64 codes per step, into the shared-memory
// slots of the int8-code GEMV's fragment layout (slot (2i + h) * 32 + 4 g + q
// holds columns 16 q .. 16 q + 15 of row 16 i + 8 h + g; here chunk q of row
// g is stored at q ^ (g >> 1), which makes both the decoder's 16-byte stores
// and the fragment loads conflict-free), and the warp runs fp16 MMAs on them.
//
// The decoder takes two Rice symbols from one 32-bit window of the lane's
// ring: a symbol's unary run and closing zero are counted as the popcount of
// x ^ (x + 1), its K low bits follow, and the window is shifted on.  Four
// decoded values are packed into one word and un-zigzagged bytewise.  A step
// is redone from the stream in global memory with the sequential reader when a
// pair of symbols (with a block's parity bit) does not fit in its window, or
// when the step read words whose chunk had not landed.  Chunks are copied by
// the whole warp, one row's 32 words per instruction, as the rows' positions
// free ring slots.
template <int LAT, int NB>
__global__ void __launch_bounds__(128, 4) gemv_rice_kernel(const GemvRiceArgs a) {
  constexpr int n = Fmt<LAT>::n;
  __shared__ uint32_t rings[4][32 * kRingWords];
  __shared__ uint4 slots[4][128];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint32_t* ring = rings[warp];
  uint32_t* myring = ring + lane * kRingWords;
  uint4* slot = slots[warp];
  const int g = lane >> 2, q4 = lane & 3;
  const int di = lane >> 4, dh = (lane >> 3) & 1, dg = lane & 7;   // the row this lane decodes
  uint4* myslot = slot + (2 * di + dh) * 32 + 4 * dg;
  const int mysw = dg >> 1;
  const int rdsw = g >> 1;
  // 8 codes (columns 8 j .. 8 j + 7 of this lane's row) as two words: chunk
  // (j >> 1) ^ (g >> 1), half (j & 1) ^ h of the chunk -- the half swap makes
  // the 8-byte stores of a half warp conflict-free; the reader undoes it.
  auto store_half = [&](uint4* base, int j, uint32_t lo, uint32_t hi) {
    reinterpret_cast<uint2*>(base + ((j >> 1) ^ mysw))[(j & 1) ^ dh] = make_uint2(lo, hi);
  };
  const int64_t w = (int64_t)blockIdx.x * (blockDim.x >> 5) + warp;
  const int64_t i0 = w * a.items / a.warps, i1 = (w + 1) * a.items / a.warps;
  const int steps = a.tile >> 6;
  const bool xok0 = g < a.batch;
  const bool xok1 = NB > 1 && 8 + g < a.batch;
  const __half* xh0 = a.xh + (int64_t)(xok0 ? g : 0) * a.cols + 16 * q4;
  const __half* xh1 = a.xh + (int64_t)(xok1 ? 8 + g : 0) * a.cols + 16 * q4;

  asm volatile("griddepcontrol.wait;" ::: "memory");

  float yacc[2][NB][4];
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int nb = 0; nb < NB; ++nb)
#pragma unroll
      for (int c = 0; c < 4; ++c) yacc[i][nb][c] = 0.f;
  int64_t grp = i0 / a.tiles_per_row;
  int t = (int)(i0 - grp * a.tiles_per_row);
  int64_t cur_grp = -1;
  int tiles_in_grp = 0;

  // The lane's region of the stream: base word wb (a multiple of 32), the
  // segment's first word s (0..31) from wb, the bit position posr from word
  // wb + s; chunks [0, ic) issued, [0, landed) landed.
  uint32_t wb = 0, s = 0, posr = 0;
  int ic = 0, landed = 0;
  bool row_ok = false;

  auto flush = [&](int64_t fg, bool whole_row) {
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
      for (int nb = 0; nb < NB; ++nb)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int64_t r = fg * 32 + 16 * i + 8 * (c >> 1) + g;
          const int bb = nb * 8 + 2 * q4 + (c & 1);
          if (r < a.rows && bb < a.batch) {
            float* dst = a.y + (int64_t)bb * a.rows + r;
            if (whole_row) *dst = yacc[i][nb][c]; else atomicAdd(dst, yacc[i][nb][c]);
          }
          yacc[i][nb][c] = 0.f;
        }
  };

  // Issue the chunks each row's position has room for: [ic, chunk + 2), one
  // or two per row, one warp-wide copy instruction per chunk.
  auto issue = [&]() {
    __syncwarp();
    const int want = row_ok ? (int)(((posr >> 5) + s) >> 5) + 2 : 0;
    const int nc = min(max(want - ic, 0), 2);
    unsigned m = __ballot_sync(0xFFFFFFFFu, nc > 0);
    const unsigned m2 = __ballot_sync(0xFFFFFFFFu, nc > 1);
    const uint32_t my_gw = wb + 32u * (uint32_t)ic;                  // the first chunk's first stream word
    const uint32_t my_ix = (32u * (uint32_t)ic - s) & 63u;          // its ring index
    while (m != 0u) {
      const int r = __ffs((int)m) - 1;
      m &= m - 1u;
      const uint32_t gw = __shfl_sync(0xFFFFFFFFu, my_gw, r) + (uint32_t)lane;
      const uint32_t ix = (__shfl_sync(0xFFFFFFFFu, my_ix, r) + (uint32_t)lane) & 63u;
      uint32_t* rrow = ring + r * kRingWords;
      const bool in = (int64_t)gw < a.nwords;
      const uint32_t* src = a.stream + (in ? gw : 0u);
      cp_async4(rrow + ix, src, in ? 4u : 0u);
      if (ix == 0u) cp_async4(rrow + 64, src, in ? 4u : 0u);
      if ((m2 >> r) & 1u) {   // the next chunk too: ring index + 32
        const uint32_t gw2 = gw + 32u;
        const uint32_t ix2 = ix ^ 32u;
        const bool in2 = (int64_t)gw2 < a.nwords;
        const uint32_t* src2 = a.stream + (in2 ? gw2 : 0u);
        cp_async4(rrow + ix2, src2, in2 ? 4u : 0u);
        if (ix2 == 0u) cp_async4(rrow + 64, src2, in2 ? 4u : 0u);
      }
    }
    ic += nc;
  };

  for (int64_t it = i0; it < i1; ++it) {
    const bool newgrp = grp != cur_grp;
    if (newgrp) {
      if (cur_grp >= 0) flush(cur_grp, tiles_in_grp == a.tiles_per_row);
      cur_grp = grp;
      tiles_in_grp = 0;
    }
    const int64_t my_row = grp * 32 + lane;
    row_ok = my_row < a.rows;
    const uint32_t o = row_ok ? __ldg(a.off + my_row * a.tiles_per_row + t) : 0u;
    // a segment that does not start where the lane stands restarts its region
    const bool restart = newgrp || (row_ok && o != (wb + s) * 32u + posr);
    if (restart) {
      wb = (o >> 5) & ~31u;
      s = (o >> 5) & 31u;
      posr = o & 31u;
      ic = 0;
    }
    if (__any_sync(0xFFFFFFFFu, restart)) {
      issue();
      cp_async_commit();
      cp_async_wait<0>();
      __syncwarp();
      landed = ic;
    }
    RiceK rk = rice_k(0);
    float acc[2][NB][4];
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
      for (int nb = 0; nb < NB; ++nb)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[i][nb][c] = 0.f;

    for (int st = 0; st < steps; ++st) {
      const int64_t k0 = (int64_t)t * a.tile + st * 64;
      uint4 xhv[NB][2];
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) xhv[nb][0] = xhv[nb][1] = make_uint4(0, 0, 0, 0);
      if (xok0) {
        xhv[0][0] = __ldg(reinterpret_cast<const uint4*>(xh0 + k0));
        xhv[0][1] = __ldg(reinterpret_cast<const uint4*>(xh0 + k0) + 1);
      }
      if constexpr (NB > 1) {
        if (xok1) {
          xhv[1][0] = __ldg(reinterpret_cast<const uint4*>(xh1 + k0));
          xhv[1][1] = __ldg(reinterpret_cast<const uint4*>(xh1 + k0) + 1);
        }
      }
      cp_async_wait<1>();
      __syncwarp();

      // ---- decode 64 codes of this lane's row
      const uint32_t posr0 = posr;
      auto window = [&](uint32_t pos) {
        const uint32_t* p = myring + ((pos >> 5) & 63u);
        return __funnelshift_r(p[0], p[1], pos);
      };
      if (st == 0) {   // the segment's K
        rk = rice_k(window(posr) & 7u);
        posr += kKBits;
      }
      {
        uint32_t half_lo = 0;
        // columns 8 j .. 8 j + 7 (code words 2 j, 2 j + 1): 16-byte chunk j >> 1, half (j & 1) ^ dh
        const uint32_t umax = decode_codes_fast<LAT, 64>(window, posr, rk, [&](int q, uint32_t w) {
          if ((q & 1) == 0) half_lo = w;
          else store_half(myslot, q >> 1, half_lo, w);
        });
        const uint32_t last_word = (posr >> 5) + s + 1u;   // highest stream word (from wb) the windows read
        const bool bad = row_ok && (umax > 31u || last_word >= (uint32_t)landed * 32u);
        if (!row_ok) {
#pragma unroll
          for (int j = 0; j < 8; ++j) store_half(myslot, j, 0u, 0u);
        }
        if (bad) {
          // the sequential reader on the stream in global memory
          BitReader rd;
          rd.init(a.stream, a.nwords, (uint64_t)(wb + s) * 32u + posr0);
          if (st == 0) rk = rice_k(rd.get(kKBits));
#pragma unroll 1
          for (int j = 0; j < 64 / n; ++j) {
            int c[n];
            decode_block<LAT>(rd, (int)rk.K, c);
#pragma unroll
            for (int e = 0; e < n; ++e) {
              const int col = j * n + e;
              reinterpret_cast<uint8_t*>(myslot + (((col >> 4) ^ mysw)))[(8 * (((col >> 3) & 1) ^ dh)) + (col & 7)] =
                  (uint8_t)c[e];
            }
          }
          posr = (uint32_t)((uint64_t)rd.word * 32u + (uint64_t)rd.b - (uint64_t)(wb + s) * 32u);
        }
      }
      __syncwarp();

      // ---- MMA on the 32 x 64 codes
      uint4 cwv[2][2];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        cwv[i][0] = slot[(2 * i) * 32 + 4 * g + (q4 ^ rdsw)];
        const uint4 sw = slot[(2 * i + 1) * 32 + 4 * g + (q4 ^ rdsw)];
        cwv[i][1] = make_uint4(sw.z, sw.w, sw.x, sw.y);   // rows 8 + g: halves stored swapped
      }
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t bh[NB][2];
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
          const uint4& H = xhv[nb][c >> 1];
          bh[nb][0] = (c & 1) ? H.z : H.x;
          bh[nb][1] = (c & 1) ? H.w : H.y;
        }
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const uint32_t wa = (c == 0) ? cwv[i][0].x : (c == 1) ? cwv[i][0].y : (c == 2) ? cwv[i][0].z : cwv[i][0].w;
          const uint32_t wbw = (c == 0) ? cwv[i][1].x : (c == 1) ? cwv[i][1].y : (c == 2) ? cwv[i][1].z : cwv[i][1].w;
          uint32_t a0, a2, a1, a3;
          codes_to_f16x2(wa, a0, a2);
          codes_to_f16x2(wbw, a1, a3);
#pragma unroll
          for (int nb = 0; nb < NB; ++nb) {
            mma16816(acc[i][nb], a0, a1, a2, a3, bh[nb][0], bh[nb][1]);
          }
        }
      }
      // next chunks for the rows that have room
      landed = ic;
      issue();
      cp_async_commit();
    }
    // per-tile scale
    float fx[NB][2];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int bb = nb * 8 + 2 * q4 + h;
        fx[nb][h] = (bb < a.batch) ? __ldg(a.xs + (int64_t)bb * a.tiles_per_row + t) : 0.f;
      }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      float sr[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int64_t r = grp * 32 + 16 * i + 8 * h + g;
        sr[h] = (r < a.rows) ? __ldg(a.scales + r * a.tiles_per_row + t) : 0.f;
      }
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) {
        yacc[i][nb][0] = fmaf(acc[i][nb][0], sr[0] * fx[nb][0], yacc[i][nb][0]);
        yacc[i][nb][1] = fmaf(acc[i][nb][1], sr[0] * fx[nb][1], yacc[i][nb][1]);
        yacc[i][nb][2] = fmaf(acc[i][nb][2], sr[1] * fx[nb][0], yacc[i][nb][2]);
        yacc[i][nb][3] = fmaf(acc[i][nb][3], sr[1] * fx[nb][1], yacc[i][nb][3]);
      }
    }
    ++tiles_in_grp;
    if (++t == a.tiles_per_row) { t = 0; ++grp; }
  }
  if (cur_grp >= 0) flush(cur_grp, tiles_in_grp == a.tiles_per_row);
  cp_async_wait<0>();
}

}  // namespace rice
}  // namespace lq

using namespace lq;
using namespace lq::rice;

namespace {

constexpr size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

// Largest rows * cols a stream can hold: segment offsets are 32-bit bit counts.
constexpr int64_t kMaxWeights = int64_t(1) << 28;

lq_status check_shape(int lattice, int64_t rows, int64_t cols, int tile) {
  lq_status st = validate_common(lattice, rows, cols, tile);
  if (st != LQ_OK) return st;
  if (rows > 0 && rows > kMaxWeights / cols) return LQ_ERR_SHAPE;
  return LQ_OK;
}

int lattice_dim(int lattice) { return lattice == LQ_E8 ? 8 : lattice == LQ_D4 ? 4 : lattice == LQ_A2 ? 2 : 1; }

struct RiceWorkspace {
  size_t len, kpar, sums, total;
};

RiceWorkspace rice_layout(int64_t rows, int64_t cols, int tile) {
  const size_t segs = (size_t)rows * (size_t)(cols / tile);
  const size_t nblocks = (segs + kScanBlock - 1) / kScanBlock;
  RiceWorkspace w;
  w.len = 0;
  w.kpar = align256(segs * 4);
  w.sums = w.kpar + align256(segs);
  w.total = w.sums + align256(nblocks * 4);
  return w;
}

template <template <int> class KER, typename A>
lq_status launch_per_segment(int lattice, const A& a, int64_t segments, cudaStream_t s) {
  const unsigned grid = (unsigned)((segments + 255) / 256);
  switch (lattice) {
    case LQ_E8: KER<LQ_E8>::launch(grid, a, s); break;
    case LQ_D4: KER<LQ_D4>::launch(grid, a, s); break;
    case LQ_A2: KER<LQ_A2>::launch(grid, a, s); break;
    default:    KER<LQ_Z1>::launch(grid, a, s); break;
  }
  return check_launch();
}
template <int LAT> struct LenK { static void launch(unsigned g, const SegArgs& a, cudaStream_t s) { seg_length_kernel<LAT><<<g, 256, 0, s>>>(a); } };
template <int LAT> struct WriteK { static void launch(unsigned g, const SegArgs& a, cudaStream_t s) { seg_write_kernel<LAT><<<g, 256, 0, s>>>(a); } };
template <int LAT> struct DecK { static void launch(unsigned g, const DecArgs& a, cudaStream_t s) { seg_decode_kernel<LAT><<<g, 256, 0, s>>>(a); } };

template <int LAT, int NB>
lq_status launch_gemv_rice(GemvRiceArgs g, cudaStream_t s) {
  static int per_sm = 0;
  if (per_sm == 0) per_sm = occupancy_per_sm(gemv_rice_kernel<LAT, NB>, 128);
  const int sms = device_sm_count();
  if (sms <= 0 || per_sm <= 0) return LQ_ERR_CUDA;
  int64_t ctas = (int64_t)sms * per_sm;
  const int64_t need = (g.items + 3) / 4;
  if (ctas > need) ctas = need;
  if (ctas < 1) ctas = 1;
  g.warps = ctas * 4;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)ctas);
  cfg.blockDim = dim3(128);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, gemv_rice_kernel<LAT, NB>, g) != cudaSuccess) {
    cudaGetLastError();
    return LQ_ERR_CUDA;
  }
  return LQ_OK;
}

}  // namespace

extern "C" size_t lq_rice_stream_bound(int lattice, int64_t rows, int64_t cols, int tile) {
  if (check_shape(lattice, rows, cols, tile) != LQ_OK) return 0;
  const int nd = lattice_dim(lattice);
  const bool parity = (lattice == LQ_E8 || lattice == LQ_A2);
  // with the shortest K no symbol is longer than with K = 7: 8 bits (|code| <= 128)
  const uint64_t bits = (uint64_t)rows * (uint64_t)(cols / tile) * kKBits + (uint64_t)rows * (uint64_t)cols * 8u +
                        (parity ? (uint64_t)rows * (uint64_t)(cols / nd) : 0u);
  return (size_t)(((bits + 31) / 32) * 4 + 16);
}

extern "C" size_t lq_rice_workspace_size(int64_t rows, int64_t cols, int tile) {
  if (rows <= 0 || cols <= 0 || tile <= 0) return 0;
  return rice_layout(rows, cols, tile).total;
}

extern "C" lq_status lq_rice_encode(int lattice, const int8_t* codes_dev, int64_t rows, int64_t cols, int tile,
                                    uint32_t* stream_dev, size_t stream_bytes, uint32_t* tile_offsets_dev,
                                    uint64_t* total_bits_dev, void* workspace_dev, int32_t* dev_status_dev,
                                    void* stream) {
  LQ_NVTX_RANGE("lq_rice_encode");
  lq_status st = check_shape(lattice, rows, cols, tile);
  if (st != LQ_OK) return st;
  if (stream_dev == nullptr || tile_offsets_dev == nullptr || total_bits_dev == nullptr) return LQ_ERR_ARG;
  if (stream_bytes < lq_rice_stream_bound(lattice, rows, cols, tile)) return LQ_ERR_SHAPE;
  if (!aligned16(stream_dev) || !aligned4(tile_offsets_dev) ||
      (reinterpret_cast<uintptr_t>(total_bits_dev) & 7u) != 0 ||
      (dev_status_dev != nullptr && !aligned4(dev_status_dev)))
    return LQ_ERR_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  if (cudaMemsetAsync(stream_dev, 0, stream_bytes, s) != cudaSuccess ||
      cudaMemsetAsync(total_bits_dev, 0, sizeof(uint64_t), s) != cudaSuccess) {
    cudaGetLastError();
    return LQ_ERR_CUDA;
  }
  if (rows == 0) return LQ_OK;
  if (codes_dev == nullptr || workspace_dev == nullptr) return LQ_ERR_ARG;
  if (!aligned16(codes_dev) || (reinterpret_cast<uintptr_t>(workspace_dev) & 255u) != 0) return LQ_ERR_ARG;
  const RiceWorkspace lay = rice_layout(rows, cols, tile);
  char* ws = reinterpret_cast<char*>(workspace_dev);
  SegArgs a;
  a.codes = codes_dev; a.rows = rows; a.cols = cols; a.tile = tile; a.tiles_per_row = (int)(cols / tile);
  a.segments = rows * (cols / tile);
  a.len = reinterpret_cast<uint32_t*>(ws + lay.len);
  a.kpar = reinterpret_cast<uint8_t*>(ws + lay.kpar);
  a.off = tile_offsets_dev;
  a.stream = stream_dev;
  a.status = dev_status_dev;
  st = launch_per_segment<LenK>(lattice, a, a.segments, s);
  if (st != LQ_OK) return st;
  uint32_t* sums = reinterpret_cast<uint32_t*>(ws + lay.sums);
  const int64_t nblocks = (a.segments + kScanBlock - 1) / kScanBlock;
  scan_local_kernel<<<(unsigned)nblocks, kScanThreads, 0, s>>>(a.len, tile_offsets_dev, sums, a.segments);
  scan_sums_kernel<<<1, kScanThreads, 0, s>>>(sums, nblocks);
  scan_add_kernel<<<(unsigned)nblocks, kScanThreads, 0, s>>>(tile_offsets_dev, sums, a.len, a.segments,
                                                             total_bits_dev);
  st = check_launch();
  if (st != LQ_OK) return st;
  return launch_per_segment<WriteK>(lattice, a, a.segments, s);
}

extern "C" lq_status lq_rice_decode(int lattice, const uint32_t* stream_dev, size_t stream_bytes,
                                    const uint32_t* tile_offsets_dev, int64_t rows, int64_t cols, int tile,
                                    int8_t* codes_dev, void* stream) {
  LQ_NVTX_RANGE("lq_rice_decode");
  lq_status st = check_shape(lattice, rows, cols, tile);
  if (st != LQ_OK) return st;
  if (rows == 0) return LQ_OK;
  if (stream_dev == nullptr || tile_offsets_dev == nullptr || codes_dev == nullptr) return LQ_ERR_ARG;
  if (!aligned4(stream_dev) || !aligned4(tile_offsets_dev) || !aligned16(codes_dev)) return LQ_ERR_ARG;
  DecArgs a;
  a.stream = stream_dev; a.nwords = (int64_t)(stream_bytes / 4); a.off = tile_offsets_dev;
  a.rows = rows; a.cols = cols; a.tile = tile; a.tiles_per_row = (int)(cols / tile);
  a.segments = rows * (cols / tile); a.codes = codes_dev;
  return launch_per_segment<DecK>(lattice, a, a.segments, (cudaStream_t)stream);
}

extern "C" lq_status lq_gemv_rice(int lattice, const uint32_t* stream_dev, size_t stream_bytes,
                                  const uint32_t* tile_offsets_dev, const float* scales_dev,
                                  const int8_t* signs_dev, int64_t rows, int64_t cols, int tile, const void* x_dev,
                                  int xdtype, int batch, float* y_dev, void* workspace_dev,
                                  int32_t* dev_status_dev, void* stream) {
  LQ_NVTX_RANGE("lq_gemv_rice");
  lq_status st = check_shape(lattice, rows, cols, tile);
  if (st != LQ_OK) return st;
  if (xdtype != LQ_BF16 && xdtype != LQ_F32) return LQ_ERR_DTYPE;
  if (batch < 1 || batch > 16) return LQ_ERR_SHAPE;
  if (rows == 0) return LQ_OK;
  if (stream_dev == nullptr || tile_offsets_dev == nullptr || scales_dev == nullptr || signs_dev == nullptr ||
      x_dev == nullptr || y_dev == nullptr || workspace_dev == nullptr)
    return LQ_ERR_ARG;
  if (!aligned4(stream_dev) || !aligned4(tile_offsets_dev) || !aligned4(scales_dev) || !aligned16(signs_dev) ||
      !aligned16(x_dev) || !aligned4(y_dev) || !aligned16(workspace_dev) ||
      (dev_status_dev != nullptr && !aligned4(dev_status_dev)))
    return LQ_ERR_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  // the workspace holds the rotated activation exactly as for lq_gemv
  const size_t half_bytes = align256((size_t)batch * (size_t)cols * 2);
  char* ws = reinterpret_cast<char*>(workspace_dev);
  RotateArgs r = {};
  r.x = x_dev; r.n_mats = 1; r.cols = cols; r.batch = batch; r.tile = tile;
  r.tiles_per_row = (int)(cols / tile);
  r.post_scale = (float)(0.5 / sqrt((double)tile));
  r.a2 = (lattice == LQ_A2);
  r.xh = reinterpret_cast<__half*>(ws);
  r.xs = reinterpret_cast<float*>(ws + half_bytes);
  r.status = dev_status_dev;
  r.signs[0] = signs_dev;
  r.y[0] = y_dev;
  r.y_elems[0] = (int64_t)batch * rows;
  st = launch_rotation(r, xdtype, r.y_elems[0], s);
  if (st != LQ_OK) return st;
  GemvRiceArgs g;
  g.stream = stream_dev; g.nwords = (int64_t)(stream_bytes / 4); g.off = tile_offsets_dev; g.scales = scales_dev;
  g.rows = rows; g.cols = cols; g.tile = tile; g.tiles_per_row = (int)(cols / tile); g.batch = batch;
  g.xh = r.xh; g.xs = r.xs; g.y = y_dev;
  g.items = ((rows + 31) / 32) * g.tiles_per_row;
  g.warps = 1;
  const bool two = batch > 8;
  switch (lattice) {
    case LQ_E8: return two ? launch_gemv_rice<LQ_E8, 2>(g, s) : launch_gemv_rice<LQ_E8, 1>(g, s);
    case LQ_D4: return two ? launch_gemv_rice<LQ_D4, 2>(g, s) : launch_gemv_rice<LQ_D4, 1>(g, s);
    case LQ_A2: return two ? launch_gemv_rice<LQ_A2, 2>(g, s) : launch_gemv_rice<LQ_A2, 1>(g, s);
    default:    return two ? launch_gemv_rice<LQ_Z1, 2>(g, s) : launch_gemv_rice<LQ_Z1, 1>(g, s);
  }
}
