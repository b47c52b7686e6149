// tcgen05 grouped-verify kernels for the E4M3 cache (head_dim 128/256 x 32/48/64 padded rows).
#include "verify_launch.cuh"

namespace pfkv {

cudaError_t launch_verify_e4m3(int head_dim, int nmax, const CUtensorMap& tmk, const CUtensorMap& tmv,
                              const DecodeParams& p, dim3 grid, cudaStream_t stream, int* ctas_out) {
  return head_dim == 128 ? verify_nm<128, kKvE4m3>(nmax, tmk, tmv, p, grid, stream, ctas_out)
                         : verify_nm<256, kKvE4m3>(nmax, tmk, tmv, p, grid, stream, ctas_out);
}

}  // namespace pfkv
