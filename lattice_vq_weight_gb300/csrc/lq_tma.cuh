// Tensor-memory-accelerator (TMA) copies and shared-memory mbarriers for the
// kernels that stage their input with one bulk tensor copy per warp unit, and
// the host-side encoder of their tensor maps.  Internal to the library.
#pragma once

#include <cstdint>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

namespace lq {

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init1(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count));
}

// Make initialised mbarriers visible to the copy engine (and to the CTA after
// the barrier that follows).
__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase of the given parity to complete, giving up after about
// `limit` clock cycles (returns false then).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, long long limit) {
  if (mbar_test(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_test(bar, parity)) {
    if (clock64() - t0 > limit) return false;
  }
  return true;
}

// Order this thread's earlier generic-proxy accesses of shared memory before
// later async-proxy (TMA) accesses of the same bytes.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 3-D tiled bulk tensor copy global -> shared (this CTA), completing on `bar`.
__device__ __forceinline__ void tma_load_3d(void* dst, const void* map, uint64_t* bar, int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], "
      "[%2];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_addr(bar)), "r"(x), "r"(y), "r"(z)
      : "memory");
}

// 2-D tiled bulk tensor copy global -> shared (this CTA), completing on `bar`.
__device__ __forceinline__ void tma_load_2d(void* dst, const void* map, uint64_t* bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];"
      ::"r"(smem_addr(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_addr(bar)), "r"(x), "r"(y)
      : "memory");
}

// ------------------------------------------------------------------ host
typedef CUresult (*TensorMapEncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                           const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                           CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                           CUtensorMapFloatOOBfill);

// The driver's cuTensorMapEncodeTiled, looked up once through the runtime
// (the library links no driver library).
inline TensorMapEncodeTiledFn tensor_map_encoder() {
  static TensorMapEncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<TensorMapEncodeTiledFn>(p);
    else
      cudaGetLastError();
  });
  return fn;
}

// A row-major [rows x ld] matrix of `esize`-byte elements (first `cols`
// columns used) viewed as [rows][cols / e][e] with e = 128 bytes of elements,
// copied in boxes of {e, lines, 1} with the 128-byte swizzle: line k of a box
// lands at byte 128 k of the (1024-byte aligned) destination with its 16-byte
// chunk c at chunk c ^ (k & 7).  Out-of-range lines read as zeros.
inline bool encode_row_lines_map(CUtensorMap* map, CUtensorMapDataType dt, int esize, const void* base,
                                 int64_t rows, int64_t cols, int64_t ld, int lines) {
  TensorMapEncodeTiledFn fn = tensor_map_encoder();
  if (fn == nullptr) return false;
  const cuuint64_t e = (cuuint64_t)(128 / esize);
  const cuuint64_t dims[3] = {e, (cuuint64_t)(cols / (int64_t)e), (cuuint64_t)rows};
  const cuuint64_t strides[2] = {128, (cuuint64_t)(ld * esize)};
  const cuuint32_t box[3] = {(cuuint32_t)e, (cuuint32_t)lines, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, dt, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// int8 codes [rows x cols] (row stride cols) copied in boxes of 128 columns x
// `box_rows` rows, one 128-byte line per row with the 128-byte swizzle (16-byte
// chunk c of row r at chunk c ^ (r & 7); 1024-byte aligned destination); rows
// past the matrix read as zeros.
inline bool encode_codes_map(CUtensorMap* map, const void* codes, int64_t rows, int64_t cols, int box_rows) {
  TensorMapEncodeTiledFn fn = tensor_map_encoder();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols};
  const cuuint32_t box[2] = {128, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(codes), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace lq
