// Launch helpers of the tcgen05 grouped-verify kernel (instantiated per FP8 format by
// verify_e4m3.cu and verify_e5m2.cu, compiled in parallel).
#pragma once

#include <atomic>

#include "verify_kernel.cuh"

namespace pfkv {

constexpr int kVerifyThreads = kVerifyWarps * 32;

template <int D, int KV, int NM>
static cudaError_t verify_one(const CUtensorMap& tmk, const CUtensorMap& tmv, const DecodeParams& p, dim3 grid,
                              cudaStream_t stream, int* ctas_out) {
  using S = VerifyShape<D, NM>;
  static std::atomic<uint64_t> done_mask{0};
  const int smem = S::SMEM + 1024;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = uint64_t(1) << (dev & 63);
  if (!(done_mask.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(verify_kernel<D, KV, NM>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    done_mask.fetch_or(bit, std::memory_order_acq_rel);
  }
  if (ctas_out != nullptr) {
    int n = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, verify_kernel<D, KV, NM>, kVerifyThreads, smem);
    *ctas_out = (e == cudaSuccess && n > 0) ? n : 1;
    return e;
  }
  return launch_pdl(verify_kernel<D, KV, NM>, grid, dim3(kVerifyThreads), smem, stream, tmk, tmv, p);
}

template <int D, int KV>
static cudaError_t verify_nm(int nmax, const CUtensorMap& tmk, const CUtensorMap& tmv, const DecodeParams& p,
                             dim3 grid, cudaStream_t stream, int* ctas_out) {
  if (nmax <= 32) return verify_one<D, KV, 32>(tmk, tmv, p, grid, stream, ctas_out);
  if (nmax <= 48) return verify_one<D, KV, 48>(tmk, tmv, p, grid, stream, ctas_out);
  return verify_one<D, KV, 64>(tmk, tmv, p, grid, stream, ctas_out);
}

}  // namespace pfkv
