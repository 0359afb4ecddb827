// Rice format of lattice codes: the format constants, the sequential decoder
// and the two-symbol fast decoder, shared by the stream kernels (lq_rice.cu)
// and the decode attention over a Rice-coded KV cache (lq_kv_kernel.cuh).
// Format: see include/lq.h.
// R. F. Rice, JPL Publication 79-22 (1979).
#pragma once

#include <cstdint>

#include "lq.h"

namespace lq {
namespace rice {

constexpr int kKBits = 3;
constexpr int kKMax = 7;

template <int LAT> struct Fmt;
template <> struct Fmt<LQ_E8> { static constexpr int n = 8; static constexpr bool parity = true;  static constexpr bool even_sum = true; };
template <> struct Fmt<LQ_D4> { static constexpr int n = 4; static constexpr bool parity = false; static constexpr bool even_sum = true; };
template <> struct Fmt<LQ_A2> { static constexpr int n = 2; static constexpr bool parity = true;  static constexpr bool even_sum = false; };
template <> struct Fmt<LQ_Z1> { static constexpr int n = 1; static constexpr bool parity = false; static constexpr bool even_sum = false; };

__device__ __forceinline__ uint32_t zigzag(int u) { return ((uint32_t)u << 1) ^ (uint32_t)(u >> 31); }
__device__ __forceinline__ int unzigzag(uint32_t z) { return (int)(z >> 1) ^ -(int)(z & 1u); }

// Sequential reader over the stream, 64-bit window; words past `nwords` read
// as 0.  The next four words wait in registers (loaded four words before the
// window needs them), so a refill never waits for memory in the decode chain.
struct BitReader {
  const uint32_t* w;
  int64_t nwords;
  int64_t word;      // stream word of the window's low half
  uint64_t win;
  int b;             // next bit inside the window, 0 .. 31 between calls
  uint32_t ahead[4]; // stream words word + 2 .. word + 5

  __device__ __forceinline__ uint32_t at(int64_t i) const { return i < nwords ? __ldg(w + i) : 0u; }
  __device__ __forceinline__ void init(const uint32_t* words, int64_t n, uint64_t pos) {
    w = words;
    nwords = n;
    word = (int64_t)(pos >> 5);
    b = (int)(pos & 31u);
    win = (uint64_t)at(word) | ((uint64_t)at(word + 1) << 32);
#pragma unroll
    for (int k = 0; k < 4; ++k) ahead[k] = at(word + 2 + k);
  }
  // one refill step: enough whenever b < 64
  __device__ __forceinline__ void refill1() {
    if (b >= 32) {
      win = (win >> 32) | ((uint64_t)ahead[0] << 32);
      ahead[0] = ahead[1];
      ahead[1] = ahead[2];
      ahead[2] = ahead[3];
      ahead[3] = at(word + 6);
      ++word;
      b -= 32;
    }
  }
  __device__ __forceinline__ void refill() {
    while (b >= 32) {
      win = (win >> 32) | ((uint64_t)ahead[0] << 32);
      ahead[0] = ahead[1];
      ahead[1] = ahead[2];
      ahead[2] = ahead[3];
      ahead[3] = at(word + 6);
      ++word;
      b -= 32;
    }
  }
  __device__ __forceinline__ uint32_t get(int nbits) {   // nbits <= 32
    const uint32_t v = (uint32_t)(win >> b) & (uint32_t)((1ull << nbits) - 1ull);
    b += nbits;   // at most 31 + 32
    refill1();
    return v;
  }
  __device__ __forceinline__ uint32_t rice(int K) {
    // common case: the run of ones, its closing zero and the K low bits all lie
    // in the window's next 32 bits (b <= 31 between calls)
    const uint32_t lo = (uint32_t)(win >> b);
    if (~lo != 0u) {
      const int t = __ffs((int)~lo) - 1;           // ones before the first zero
      if (t + 1 + K <= 32) {
        const uint32_t v = ((uint32_t)t << K) | ((uint32_t)((uint64_t)lo >> (t + 1)) & ((1u << K) - 1u));
        b += t + 1 + K;   // at most 31 + 32
        refill1();
        return v;
      }
    }
    uint32_t q = 0;
    while (true) {
      const uint64_t x = ~(win >> b);            // valid bits inverted; the vacated top bits read as 1
      const int t = x ? __ffsll((long long)x) - 1 : 64;   // ones before the first zero
      if (t < 64 - b) {
        q += (uint32_t)t;
        b += t + 1;
        refill();
        break;
      }
      q += (uint32_t)(64 - b);
      b = 64;
      refill();
    }
    return (q << K) | get(K);
  }
};

// Decode one block into n codes.
template <int LAT>
__device__ __forceinline__ void decode_block(BitReader& rd, int K, int (&c)[Fmt<LAT>::n]) {
  constexpr int n = Fmt<LAT>::n;
  const int k = Fmt<LAT>::parity ? (int)rd.get(1) : 0;
  int u[n];
  int sum = 0;
#pragma unroll
  for (int i = 0; i < n; ++i) {
    u[i] = unzigzag(rd.rice(K));
    if (i < n - 1) sum += u[i];
  }
  if constexpr (Fmt<LAT>::even_sum) u[n - 1] = 2 * u[n - 1] + (sum & 1);
#pragma unroll
  for (int i = 0; i < n; ++i) c[i] = 2 * u[i] + k;
}

// One 4-byte global -> shared copy in the background (`bytes` 4, or 0 to
// write a zero without reading).
__device__ __forceinline__ void cp_async4(uint32_t* dst, const uint32_t* src, uint32_t bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(
                   static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
               "l"(src), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ---------------------------------------------------------------- fast decode
// The Rice parameter of a segment and the constants the fast decoder derives
// from it.
struct RiceK {
  uint32_t K, kone, kmask, kk;   // K, 2^K, 2^K - 1, 2^K in each byte
};
__device__ __forceinline__ RiceK rice_k(uint32_t K) {
  RiceK r;
  r.K = K;
  r.kone = 1u << K;
  r.kmask = r.kone - 1u;
  r.kk = r.kone * 0x01010101u;
  return r;
}

// Four zigzag values (plus kone each) in bytes -> four codes 2 u + k in bytes:
// per byte u2 = v ^ (0 - (v & 1)) is twice the signed value, ORed with the
// block's parity bit (kp: 0x01 in each byte of a block with odd codes).
__device__ __forceinline__ uint32_t codes_from_zigzag4(uint32_t vb0, uint32_t vb1, uint32_t vb2, uint32_t vb3,
                                                       uint32_t kk, uint32_t kp) {
  const uint32_t vw = ((vb3 * 256u + vb2) * 65536u + (vb1 * 256u + vb0)) - kk;
  const uint32_t m = (vw & 0x01010101u) * 0xFFu;
  return (vw ^ m) | kp;
}

// The last code of an even-sum block (E8, D4) in byte 3 of `w`: the format
// stores half of its halved value; the halved value is 2 * that + the parity
// of the sum of the block's other halved values.  `w0` is the block's other
// code word for E8 (zero for D4).  Bit 1 of a code is the parity of its halved
// value, so the parity of the sum is bit 1 of the XOR of the other codes,
// summed into bit 25 by one multiply.
template <bool TWO_WORDS>
__device__ __forceinline__ uint32_t fix_last_code(uint32_t w0, uint32_t w) {
  const uint32_t t = TWO_WORDS ? ((w0 ^ w) & 0x02020202u) : (w & 0x00020202u);
  const uint32_t p = t * 0x01010101u;                 // bit 25: parity (E8: XOR bit 1 of code 7 too)
  const uint32_t a = w << 1;                          // code 7 doubled in byte 3 (bit 24: junk)
  const uint32_t sel = (w & 0x01FFFFFFu) | (a & 0xFE000000u);
  const uint32_t q = TWO_WORDS ? (p ^ w ^ a) : (p ^ a);  // bit 25: the sum parity, less what sel holds
  return sel ^ (q & 0x02000000u);
}

// Fast decode of NCODES codes (whole blocks) starting at bit `pos` of a
// segment, two Rice symbols per 32-bit window: a symbol's unary run and
// closing zero are counted as the popcount of x ^ (x + 1), its K low bits
// follow, and the window shifts on; four values are packed into one word and
// un-zigzagged bytewise.  window(pos) returns the 32 stream bits from pos;
// emit(q, w) receives code word q (codes 4 q .. 4 q + 3 as bytes).  Returns
// the most bits one window gave: above 31 a pair (with a block's parity bit)
// did not fit its window and the codes are invalid (the caller decodes again
// with the sequential reader).
template <int LAT, int NCODES, class Win, class Emit>
__device__ __forceinline__ uint32_t decode_codes_fast(const Win& window, uint32_t& pos, const RiceK& rk,
                                                      const Emit& emit) {
  constexpr int n = Fmt<LAT>::n;
  static_assert(NCODES % 8 == 0, "whole blocks, whole code words");
  uint32_t vb[4];
  uint32_t x = 0, pw = 0, umax = 0, kp = 0, prev = 0;
#pragma unroll
  for (int sy = 0; sy < NCODES; ++sy) {
    const int i = sy % n;
    if ((sy & 1) == 0) {
      x = window(pos);
      pw = pos;
      if (Fmt<LAT>::parity && i == 0) {
        // the block's parity bit in each of its code bytes (A2: two blocks per word)
        if constexpr (n >= 4) {
          kp = (x & 1u) * 0x01010101u;
        } else {
          const uint32_t kb = (x & 1u) * (0x0101u << (8 * (sy & 3)));
          kp = (sy & 3) == 0 ? kb : (kp | kb);
        }
        x >>= 1;
        pos += 1;
      }
    }
    const uint32_t p1 = __popc(x ^ (x + 1u));          // run of ones + its closing zero
    const uint32_t y1 = __funnelshift_rc(x, 0u, p1);   // x >> p1 (0 when p1 = 32)
    vb[sy & 3] = p1 * rk.kone + (y1 & rk.kmask);       // zigzag value + kone
    x = y1 >> rk.K;
    pos += p1 + rk.K;
    if ((sy & 1) == 1) umax = max(umax, pos - pw);
    if ((sy & 3) == 3) {
      uint32_t cword = codes_from_zigzag4(vb[0], vb[1], vb[2], vb[3], rk.kk, kp);
      if constexpr (LAT == LQ_E8) {
        if ((sy & 7) == 7) cword = fix_last_code<true>(prev, cword);
      } else if constexpr (LAT == LQ_D4) {
        cword = fix_last_code<false>(0u, cword);
      }
      emit(sy >> 2, cword);
      prev = cword;
    }
  }
  return umax;
}

}  // namespace rice
}  // namespace lq
