// Launch helpers of the decode kernel for one cache dtype (instantiated by
// decode_fp16.cu, decode_e4m3.cu and decode_e5m2.cu, compiled in parallel).
#pragma once

#include <atomic>

#include "decode_kernel.cuh"

namespace pfkv {

// The opt-in shared-memory limit is set once per device and instantiation
// (to the largest request this library makes), not on every launch.
template <int D, int KV, int NT>
static cudaError_t ensure_smem_attr() {
  static std::atomic<uint64_t> done_mask{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = uint64_t(1) << (dev & 63);
  if (done_mask.load(std::memory_order_acquire) & bit) return cudaSuccess;
  const int smem = decode_smem_bytes<D, KV, NT>(8) + 1024;  // 8 consumer warps: the largest CTA
  e = cudaFuncSetAttribute(decode_kernel<D, KV, NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess) done_mask.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

template <int D, int KV, int NT>
static cudaError_t launch_one(const CUtensorMap& tmk, const CUtensorMap& tmv, const DecodeParams& p, dim3 grid,
                              cudaStream_t stream) {
  const int ncw = p.nrg * p.nts;
  const int smem = decode_smem_bytes<D, KV, NT>(ncw) + 1024;
  cudaError_t e = ensure_smem_attr<D, KV, NT>();
  if (e != cudaSuccess) return e;
  return launch_pdl(decode_kernel<D, KV, NT>, grid, dim3((ncw + 1) * 32), smem, stream, tmk, tmv, p);
}

template <int D, int KV, int NT>
static int ctas_one(int ncw) {
  const int smem = decode_smem_bytes<D, KV, NT>(ncw) + 1024;
  auto kern = decode_kernel<D, KV, NT>;
  if (ensure_smem_attr<D, KV, NT>() != cudaSuccess) return 1;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, (ncw + 1) * 32, smem) != cudaSuccess) return 1;
  return n > 0 ? n : 1;
}

// The persistent grid (one row tile per warp): its shared memory grows with the batch (lengths and
// item prefix), up to kMaxPersistSeqs sequences.
template <int D, int KV>
static cudaError_t ensure_persist_attr() {
  static std::atomic<uint64_t> done_mask{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = uint64_t(1) << (dev & 63);
  if (done_mask.load(std::memory_order_acquire) & bit) return cudaSuccess;
  const int smem = persist_smem_bytes<D, KV, 1>(4, kMaxPersistSeqs) + 1024;  // one row group x 4 slices
  e = cudaFuncSetAttribute(decode_persist_kernel<D, KV, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess) done_mask.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

template <int D, int KV>
static cudaError_t launch_persist_one(const CUtensorMap& tmk, const CUtensorMap& tmv, const DecodeParams& p,
                                      int ctas, cudaStream_t stream) {
  const int ncw = p.nrg * p.nts;
  const int smem = persist_smem_bytes<D, KV, 1>(ncw, p.num_seqs) + 1024;
  cudaError_t e = ensure_persist_attr<D, KV>();
  if (e != cudaSuccess) return e;
  return launch_pdl(decode_persist_kernel<D, KV, 1>, dim3(ctas), dim3((ncw + 1) * 32), smem, stream, tmk, tmv, p);
}

template <int D, int KV>
static int persist_ctas_one(int ncw, int num_seqs) {
  const int smem = persist_smem_bytes<D, KV, 1>(ncw, num_seqs) + 1024;
  if (ensure_persist_attr<D, KV>() != cudaSuccess) return 1;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_persist_kernel<D, KV, 1>, (ncw + 1) * 32, smem) !=
      cudaSuccess)
    return 1;
  return n > 0 ? n : 1;
}

template <int KV>
cudaError_t launch_persist_kv(const DecodeLaunch& cfg, const CUtensorMap& tmk, const CUtensorMap& tmv,
                              const DecodeParams& p, int ctas, cudaStream_t stream) {
  if (cfg.nt != 1) return cudaErrorInvalidValue;
  return cfg.head_dim == 128 ? launch_persist_one<128, KV>(tmk, tmv, p, ctas, stream)
                             : launch_persist_one<256, KV>(tmk, tmv, p, ctas, stream);
}

template <int KV>
int persist_ctas_kv(const DecodeLaunch& cfg, int ncw, int num_seqs) {
  return cfg.head_dim == 128 ? persist_ctas_one<128, KV>(ncw, num_seqs) : persist_ctas_one<256, KV>(ncw, num_seqs);
}

template <int KV>
cudaError_t launch_decode_kv(const DecodeLaunch& cfg, const CUtensorMap& tmk, const CUtensorMap& tmv,
                             const DecodeParams& p, dim3 grid, cudaStream_t stream) {
  if (cfg.head_dim == 128) {
    return cfg.nt == 1 ? launch_one<128, KV, 1>(tmk, tmv, p, grid, stream)
                       : launch_one<128, KV, 2>(tmk, tmv, p, grid, stream);
  }
  return cfg.nt == 1 ? launch_one<256, KV, 1>(tmk, tmv, p, grid, stream)
                     : launch_one<256, KV, 2>(tmk, tmv, p, grid, stream);
}

template <int KV>
int decode_ctas_kv(const DecodeLaunch& cfg, int ncw) {
  if (cfg.head_dim == 128) return cfg.nt == 1 ? ctas_one<128, KV, 1>(ncw) : ctas_one<128, KV, 2>(ncw);
  return cfg.nt == 1 ? ctas_one<256, KV, 1>(ncw) : ctas_one<256, KV, 2>(ncw);
}

}  // namespace pfkv
