// Rice format of lattice codes: the format constants and the sequential
// decoder, shared by the stream kernels (lq_rice.cu) and the decode attention
// over a Rice-coded KV cache (lq_kv.cu).  Format: see include/lq.h.
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

}  // namespace rice
}  // namespace lq
