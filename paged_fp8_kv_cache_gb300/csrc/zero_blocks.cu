// kv_cache_zero_blocks: clear every byte of the listed blocks in the K and V
// pools (all KV heads, all page offsets), so that a block handed to a new
// sequence carries nothing of its previous owner ("1Cat-vLLM 1.5.0",
// "Reliability and correctness fixes": newly reused KV blocks are zeroed
// before attention; the zeroing runs on the device, with no host staging).
//
// A block is one contiguous chunk of num_kv_heads * page_size * head_dim
// elements per pool. Grid = (chunks of 32 KB per block, listed blocks): each
// CTA writes one 32 KB chunk of the block in both pools with 16-byte vector
// stores, so a warp instruction covers 512 contiguous bytes. HBM-bound: the
// bytes written are the whole work.
#include "pfkv_internal.h"

namespace pfkv {

constexpr int kZeroThreads = 256;
constexpr int kZeroChunk = 32 * 1024;  // bytes per CTA and pool

__global__ void __launch_bounds__(kZeroThreads) zero_blocks_kernel(unsigned char* __restrict__ k_cache,
                                                                   unsigned char* __restrict__ v_cache,
                                                                   const int32_t* __restrict__ block_ids,
                                                                   long long block_bytes, int num_blocks,
                                                                   unsigned* err) {
  const int id = block_ids[blockIdx.y];
  if (id < 0) return;  // "no block": skipped
  if (id >= num_blocks) {
    if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(err, kDevErrBlockId);
    return;
  }
  const long long base = static_cast<long long>(id) * block_bytes;
  const long long start = static_cast<long long>(blockIdx.x) * kZeroChunk;
  const long long stop = min(start + kZeroChunk, block_bytes);
  const uint4 z = make_uint4(0u, 0u, 0u, 0u);
  for (long long o = start + 16LL * threadIdx.x; o < stop; o += 16LL * kZeroThreads) {
    *reinterpret_cast<uint4*>(k_cache + base + o) = z;
    *reinterpret_cast<uint4*>(v_cache + base + o) = z;
  }
}

cudaError_t launch_zero_blocks(void* k_cache, void* v_cache, const int32_t* block_ids, int n_ids, long long block_bytes,
                               int num_blocks, unsigned* err, cudaStream_t stream) {
  const long long chunks = (block_bytes + kZeroChunk - 1) / kZeroChunk;
  if (chunks > 0x7fffffffLL) return cudaErrorInvalidValue;
  // grid.y holds the listed blocks (at most 65535 per launch)
  for (int first = 0; first < n_ids; first += 65535) {
    const int n = min(65535, n_ids - first);
    zero_blocks_kernel<<<dim3(static_cast<unsigned>(chunks), static_cast<unsigned>(n)), kZeroThreads, 0, stream>>>(
        static_cast<unsigned char*>(k_cache), static_cast<unsigned char*>(v_cache), block_ids + first, block_bytes,
        num_blocks, err);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace pfkv
