// Rate / SNR calibration of the lattice quantizer.
//
// HyperQuant page, usage section and "bps" table: the quantizer runs on a
// continuous bits-per-scalar axis; rates are related to the SNRs they reach
// by measurement, and the lattice scale is set from a target SNR.
//
//  - lq_beta_for_snr: high-resolution closed form.  The error per coordinate of
//    a lattice quantizer with cell volume V and normalised second moment G at
//    scale s is G V^(2/n) s^2 (Conway & Sloane ch. 2 and 21); with s = beta RMS
//    the SNR is 1 / (G V^(2/n) beta^2).
//  - lq_calibrate_bps: bisection on log2(beta) over [-8, 4] (24 halvings) of the
//    bit-stripped Rice rate of the caller's sample, each probe a quantize plus
//    Rice encode on the GPU (a probe whose codes leave int8 counts as above the
//    target); then the SNR of the final scale from a dequantize and one
//    reduction kernel.
#include <cmath>

#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "lq_device.cuh"
#include "lq_host.h"

namespace lq {

struct ErrArgs {
  const void* W;
  int64_t rows, cols, ldw;
  const float* What;
  double* sums;     // [0] sum w^2, [1] sum (w - w^)^2
};

template <bool BF16>
__global__ void __launch_bounds__(256) error_sums_kernel(ErrArgs a) {
  const int64_t n = a.rows * a.cols;
  double s0 = 0.0, s1 = 0.0;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / a.cols, c = i - r * a.cols;
    float w;
    if constexpr (BF16) w = __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(a.W)[r * a.ldw + c]);
    else w = reinterpret_cast<const float*>(a.W)[r * a.ldw + c];
    const double wd = (double)w, e = wd - (double)a.What[i];
    s0 += wd * wd;
    s1 += e * e;
  }
  for (int o = 16; o; o >>= 1) {
    s0 += __shfl_xor_sync(0xffffffffu, s0, o);
    s1 += __shfl_xor_sync(0xffffffffu, s1, o);
  }
  if ((threadIdx.x & 31) == 0) {
    atomicAdd(a.sums, s0);
    atomicAdd(a.sums + 1, s1);
  }
}

}  // namespace lq

using namespace lq;

namespace {

constexpr size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

// normalised second moments (Conway & Sloane table 2.3) and cell volumes at the
// scales the quantizer uses (E8, D4: minimal norm^2 2; A2: minimal distance 1)
void lattice_constants(int lattice, double& G, double& V, int& n) {
  switch (lattice) {
    case LQ_E8: G = 929.0 / 12960.0; V = 1.0; n = 8; break;
    case LQ_D4: G = 0.0766032; V = 2.0; n = 4; break;
    case LQ_A2: G = 5.0 / (36.0 * std::sqrt(3.0)); V = std::sqrt(3.0) / 2.0; n = 2; break;
    default:    G = 1.0 / 12.0; V = 1.0; n = 1; break;
  }
}

struct CalibLayout {
  size_t codes, scales, signs, stream, stream_bytes, offs, total, rice_ws, what, sums, status, end;
};

CalibLayout calib_layout(int lattice, int64_t rows, int64_t cols, int tile) {
  CalibLayout L;
  const size_t n = (size_t)rows * (size_t)cols, tiles = (size_t)rows * (size_t)(cols / tile);
  size_t p = 0;
  L.codes = p; p += align256(n);
  L.scales = p; p += align256(tiles * 4);
  L.signs = p; p += align256((size_t)cols);
  L.stream_bytes = lq_rice_stream_bound(lattice, rows, cols, tile);
  L.stream = p; p += align256(L.stream_bytes);
  L.offs = p; p += align256(tiles * 4);
  L.total = p; p += 256;
  L.rice_ws = p; p += align256(lq_rice_workspace_size(rows, cols, tile));
  L.what = p; p += align256(n * 4);
  L.sums = p; p += 256;
  L.status = p; p += 256;
  L.end = p;
  return L;
}

}  // namespace

extern "C" double lq_beta_for_snr(int lattice, double snr_db) {
  if (!valid_lattice(lattice)) return 0.0;
  double G, V;
  int n;
  lattice_constants(lattice, G, V, n);
  return std::sqrt(std::pow(10.0, -snr_db / 10.0) / (G * std::pow(V, 2.0 / n)));
}

extern "C" lq_status lq_error_sums(const void* W_dev, int wdtype, int64_t rows, int64_t cols, int64_t ldw,
                                   const float* What_dev, double* sums_dev, void* stream) {
  LQ_NVTX_RANGE("lq_error_sums");
  if (wdtype != LQ_BF16 && wdtype != LQ_F32) return LQ_ERR_DTYPE;
  if (rows < 0 || cols <= 0 || ldw < cols) return LQ_ERR_SHAPE;
  if (sums_dev == nullptr || (reinterpret_cast<uintptr_t>(sums_dev) & 7u) != 0) return LQ_ERR_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  if (cudaMemsetAsync(sums_dev, 0, 2 * sizeof(double), s) != cudaSuccess) {
    cudaGetLastError();
    return LQ_ERR_CUDA;
  }
  if (rows == 0) return LQ_OK;
  if (W_dev == nullptr || What_dev == nullptr) return LQ_ERR_ARG;
  ErrArgs a;
  a.W = W_dev; a.rows = rows; a.cols = cols; a.ldw = ldw; a.What = What_dev; a.sums = sums_dev;
  const int sms = device_sm_count();
  if (sms <= 0) return LQ_ERR_CUDA;
  const int64_t want = (rows * cols + 255) / 256;
  const unsigned grid = (unsigned)(want < (int64_t)sms * 8 ? want : (int64_t)sms * 8);
  if (wdtype == LQ_BF16) error_sums_kernel<true><<<grid, 256, 0, s>>>(a);
  else error_sums_kernel<false><<<grid, 256, 0, s>>>(a);
  return check_launch();
}

extern "C" size_t lq_calibrate_workspace_size(int lattice, int64_t rows, int64_t cols, int tile) {
  if (validate_common(lattice, rows, cols, tile) != LQ_OK || rows <= 0) return 0;
  if (lq_rice_stream_bound(lattice, rows, cols, tile) == 0) return 0;
  return calib_layout(lattice, rows, cols, tile).end;
}

extern "C" lq_status lq_calibrate_bps(int lattice, int tile, double target_bps, const void* W_dev, int wdtype,
                                      int64_t rows, int64_t cols, int64_t ldw, uint64_t seed, void* workspace_dev,
                                      size_t workspace_bytes, double* result, void* stream) {
  LQ_NVTX_RANGE("lq_calibrate_bps");
  lq_status st = validate_common(lattice, rows, cols, tile);
  if (st != LQ_OK) return st;
  if (rows <= 0) return LQ_ERR_SHAPE;
  if (!(target_bps > 0.0) || result == nullptr || W_dev == nullptr || workspace_dev == nullptr) return LQ_ERR_ARG;
  if ((reinterpret_cast<uintptr_t>(workspace_dev) & 255u) != 0) return LQ_ERR_ARG;
  const size_t need = lq_calibrate_workspace_size(lattice, rows, cols, tile);
  if (need == 0) return LQ_ERR_SHAPE;
  if (workspace_bytes < need) return LQ_ERR_SHAPE;
  const CalibLayout L = calib_layout(lattice, rows, cols, tile);
  char* ws = reinterpret_cast<char*>(workspace_dev);
  int8_t* codes = reinterpret_cast<int8_t*>(ws + L.codes);
  float* scales = reinterpret_cast<float*>(ws + L.scales);
  int8_t* signs = reinterpret_cast<int8_t*>(ws + L.signs);
  uint32_t* rstream = reinterpret_cast<uint32_t*>(ws + L.stream);
  uint32_t* offs = reinterpret_cast<uint32_t*>(ws + L.offs);
  uint64_t* total = reinterpret_cast<uint64_t*>(ws + L.total);
  void* rice_ws = ws + L.rice_ws;
  float* what = reinterpret_cast<float*>(ws + L.what);
  double* sums = reinterpret_cast<double*>(ws + L.sums);
  int32_t* status = reinterpret_cast<int32_t*>(ws + L.status);
  cudaStream_t s = (cudaStream_t)stream;
  if (cudaMemsetAsync(status, 0, sizeof(int32_t), s) != cudaSuccess) {
    cudaGetLastError();
    return LQ_ERR_CUDA;
  }

  // Rice bits of the sample quantized at beta and the probe's status bits
  // (synchronises the stream).
  int32_t probe_status = 0;
  auto bits_at = [&](float beta, uint64_t& bits) -> lq_status {
    if (cudaMemsetAsync(status, 0, sizeof(int32_t), s) != cudaSuccess) {
      cudaGetLastError();
      return LQ_ERR_CUDA;
    }
    lq_status e = lq_quantize(lattice, W_dev, wdtype, rows, cols, ldw, tile, seed, beta, codes, scales, signs,
                              status, stream);
    if (e != LQ_OK) return e;
    e = lq_rice_encode(lattice, codes, rows, cols, tile, rstream, L.stream_bytes, offs, total, rice_ws, status,
                       stream);
    if (e != LQ_OK) return e;
    if (cudaMemcpyAsync(&bits, total, sizeof(uint64_t), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaMemcpyAsync(&probe_status, status, sizeof(int32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess) {
      cudaGetLastError();
      return LQ_ERR_CUDA;
    }
    return LQ_OK;
  };

  // a probe whose codes leave int8 counts as above the target rate
  const double target_bits = target_bps * (double)rows * (double)cols;
  double lo = -8.0, hi = 4.0;
  for (int i = 0; i < 24; ++i) {
    const double mid = 0.5 * (lo + hi);
    uint64_t bits = 0;
    st = bits_at((float)std::pow(2.0, mid), bits);
    if (st != LQ_OK) return st;
    if ((probe_status & LQ_DEV_RANGE) || (double)bits > target_bits) lo = mid; else hi = mid;
  }
  const float beta = (float)std::pow(2.0, hi);
  uint64_t bits = 0;
  st = bits_at(beta, bits);
  if (st != LQ_OK) return st;
  st = lq_dequantize(lattice, codes, scales, signs, rows, cols, tile, what, LQ_F32, stream);
  if (st != LQ_OK) return st;
  st = lq_error_sums(W_dev, wdtype, rows, cols, ldw, what, sums, stream);
  if (st != LQ_OK) return st;
  double h[2] = {0.0, 0.0};
  const int32_t dev_status = probe_status;
  if (cudaMemcpyAsync(h, sums, sizeof(h), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess) {
    cudaGetLastError();
    return LQ_ERR_CUDA;
  }
  result[0] = (double)beta;
  result[1] = (double)bits / ((double)rows * (double)cols);
  result[2] = 10.0 * std::log10(h[0] / h[1]);
  // the final scale must quantize the sample without leaving int8 or the format
  if (dev_status & (LQ_DEV_RANGE | LQ_DEV_NONFINITE | LQ_DEV_FORMAT)) return LQ_ERR_UNSUPPORTED;
  return LQ_OK;
}
