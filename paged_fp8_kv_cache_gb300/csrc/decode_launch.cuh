// Launch helpers of the decode kernel for one cache dtype (instantiated by
// decode_fp16.cu, decode_e4m3.cu and decode_e5m2.cu, compiled in parallel).
#pragma once

#include "decode_kernel.cuh"

namespace pfkv {

template <int D, int KV, int NT>
static cudaError_t launch_one(const CUtensorMap& tmk, const CUtensorMap& tmv, const DecodeParams& p, dim3 grid,
                              cudaStream_t stream) {
  const int ncw = p.nrg * p.nts;
  const int smem = decode_smem_bytes<D, KV, NT>(ncw) + 1024;
  auto kern = decode_kernel<D, KV, NT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, (ncw + 1) * 32, smem, stream>>>(tmk, tmv, p);
  return cudaGetLastError();
}

template <int D, int KV, int NT>
static int ctas_one(int ncw) {
  const int smem = decode_smem_bytes<D, KV, NT>(ncw) + 1024;
  auto kern = decode_kernel<D, KV, NT>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) return 1;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, (ncw + 1) * 32, smem) != cudaSuccess) return 1;
  return n > 0 ? n : 1;
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
int decode_smem_kv(const DecodeLaunch& cfg, int ncw) {
  if (cfg.head_dim == 128)
    return (cfg.nt == 1 ? decode_smem_bytes<128, KV, 1>(ncw) : decode_smem_bytes<128, KV, 2>(ncw)) + 1024;
  return (cfg.nt == 1 ? decode_smem_bytes<256, KV, 1>(ncw) : decode_smem_bytes<256, KV, 2>(ncw)) + 1024;
}

template <int KV>
int decode_ctas_kv(const DecodeLaunch& cfg, int ncw) {
  if (cfg.head_dim == 128) return cfg.nt == 1 ? ctas_one<128, KV, 1>(ncw) : ctas_one<128, KV, 2>(ncw);
  return cfg.nt == 1 ? ctas_one<256, KV, 1>(ncw) : ctas_one<256, KV, 2>(ncw);
}

}  // namespace pfkv
