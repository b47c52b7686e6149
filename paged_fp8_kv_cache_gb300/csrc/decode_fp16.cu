// Decode kernels for the fp16 cache (head_dim 128/256 x 1 or 2 row tiles per warp).
#include "decode_launch.cuh"

namespace pfkv {

cudaError_t launch_decode_fp16(const DecodeLaunch& cfg, const CUtensorMap& tmk, const CUtensorMap& tmv,
                                const DecodeParams& p, dim3 grid, cudaStream_t stream) {
  return launch_decode_kv<kKvFp16>(cfg, tmk, tmv, p, grid, stream);
}

int decode_ctas_fp16(const DecodeLaunch& cfg, int ncw) { return decode_ctas_kv<kKvFp16>(cfg, ncw); }

cudaError_t launch_decode_persist_fp16(const DecodeLaunch& cfg, const CUtensorMap& tmk, const CUtensorMap& tmv,
                                       const DecodeParams& p, int ctas, cudaStream_t stream) {
  return launch_persist_kv<kKvFp16>(cfg, tmk, tmv, p, ctas, stream);
}

int decode_persist_ctas_fp16(const DecodeLaunch& cfg, int ncw, int num_seqs) {
  return persist_ctas_kv<kKvFp16>(cfg, ncw, num_seqs);
}

}  // namespace pfkv
