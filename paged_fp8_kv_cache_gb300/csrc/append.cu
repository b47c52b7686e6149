// kv_cache_append: quantise new fp16 K/V tokens with a static per-tensor
// scale (or one per KV head) and write them into their cache pages (the KV
// write path of the fork, "1Cat-vLLM": FP8 KV cache with static scales, no
// online scale computation; pages of 16 or 2048 tokens, "SM70 release
// profile and acceleration status").
//
// One thread moves 8 consecutive head-dim elements of one (token, KV head)
// for both K and V: two 16-byte loads of fp16, two 8-byte stores of FP8
// codes (or two 16-byte stores for an fp16 cache). Consecutive threads
// cover consecutive elements, so loads and stores are coalesced.
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "pfkv_internal.h"

namespace pfkv {

template <int KV>
__device__ __forceinline__ uint2 quantise8(const uint4 src, float scale) {
  const __half2* h = reinterpret_cast<const __half2*>(&src);
  constexpr __nv_fp8_interpretation_t fmt = (KV == kKvE4m3) ? __NV_E4M3 : __NV_E5M2;
  uint32_t packed[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    uint32_t word = 0;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const float2 f = __half22float2(h[2 * i + j]);
      // IEEE round-to-nearest division (no fast-math), then RNE + satfinite
      const __nv_fp8_storage_t lo = __nv_cvt_float_to_fp8(__fdiv_rn(f.x, scale), __NV_SATFINITE, fmt);
      const __nv_fp8_storage_t hi = __nv_cvt_float_to_fp8(__fdiv_rn(f.y, scale), __NV_SATFINITE, fmt);
      word |= (uint32_t(lo) | (uint32_t(hi) << 8)) << (16 * j);
    }
    packed[i] = word;
  }
  return make_uint2(packed[0], packed[1]);
}

template <int KV>
__global__ void __launch_bounds__(256) append_kernel(const __half* __restrict__ k_new, const __half* __restrict__ v_new,
                                                     unsigned char* __restrict__ k_cache,
                                                     unsigned char* __restrict__ v_cache,
                                                     const int64_t* __restrict__ slots, int n_tok, int num_kv_heads,
                                                     int head_dim, int page_size, int num_blocks,
                                                     const float* __restrict__ k_scale,
                                                     const float* __restrict__ v_scale, int scale_stride,
                                                     unsigned* err) {
  // An attention kernel launched next with programmatic stream serialisation may start its
  // launch now: it waits (griddepcontrol.wait) for this grid to complete, and its writes to be
  // visible, before it reads the cache.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int chunks = head_dim / 8;
  const int64_t per_tok = static_cast<int64_t>(num_kv_heads) * chunks;
  const int64_t total = per_tok * n_tok;
  float ks = 1.f, vs = 1.f;
  if (KV != kKvFp16) {
    ks = *k_scale;
    vs = *v_scale;
  }
  const int64_t capacity = static_cast<int64_t>(num_blocks) * page_size;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t tok = i / per_tok;
    const int64_t rem = i - tok * per_tok;
    const int h = static_cast<int>(rem / chunks);
    const int ch = static_cast<int>(rem - static_cast<int64_t>(h) * chunks);
    const int64_t slot = slots[tok];
    if (slot < 0) continue;
    if (slot >= capacity) {
      atomicOr(err, kDevErrSlot);
      continue;
    }
    const int64_t blk = slot / page_size, off = slot - blk * page_size;
    if (KV != kKvFp16 && scale_stride != 0) {  // one scale per KV head
      ks = k_scale[h];
      vs = v_scale[h];
    }
    const int64_t src = (tok * num_kv_heads + h) * head_dim + ch * 8;
    const int64_t dst = ((blk * num_kv_heads + h) * page_size + off) * head_dim + ch * 8;
    const uint4 kv = *reinterpret_cast<const uint4*>(k_new + src);
    const uint4 vv = *reinterpret_cast<const uint4*>(v_new + src);
    if constexpr (KV == kKvFp16) {
      *reinterpret_cast<uint4*>(k_cache + dst * 2) = kv;
      *reinterpret_cast<uint4*>(v_cache + dst * 2) = vv;
    } else {
      *reinterpret_cast<uint2*>(k_cache + dst) = quantise8<KV>(kv, ks);
      *reinterpret_cast<uint2*>(v_cache + dst) = quantise8<KV>(vv, vs);
    }
  }
}

cudaError_t launch_append(const __half* k_new, const __half* v_new, void* k_cache, void* v_cache, const int64_t* slots,
                          int n_tok, int num_kv_heads, int head_dim, int page_size, int num_blocks, int kv,
                          const float* k_scale, const float* v_scale, int scale_stride, unsigned* err,
                          int num_sms, cudaStream_t stream) {
  const int64_t total = static_cast<int64_t>(n_tok) * num_kv_heads * (head_dim / 8);
  const int threads = 256;
  int64_t blocks = (total + threads - 1) / threads;
  const int64_t cap = static_cast<int64_t>(num_sms > 0 ? num_sms : 1) * 64;
  if (blocks > cap) blocks = cap;  // grid-stride beyond 64 CTAs per SM
  if (blocks < 1) blocks = 1;
  auto* kc = static_cast<unsigned char*>(k_cache);
  auto* vc = static_cast<unsigned char*>(v_cache);
  switch (kv) {
    case kKvFp16:
      append_kernel<kKvFp16><<<static_cast<int>(blocks), threads, 0, stream>>>(
          k_new, v_new, kc, vc, slots, n_tok, num_kv_heads, head_dim, page_size, num_blocks, k_scale, v_scale, scale_stride, err);
      break;
    case kKvE4m3:
      append_kernel<kKvE4m3><<<static_cast<int>(blocks), threads, 0, stream>>>(
          k_new, v_new, kc, vc, slots, n_tok, num_kv_heads, head_dim, page_size, num_blocks, k_scale, v_scale, scale_stride, err);
      break;
    default:
      append_kernel<kKvE5m2><<<static_cast<int>(blocks), threads, 0, stream>>>(
          k_new, v_new, kc, vc, slots, n_tok, num_kv_heads, head_dim, page_size, num_blocks, k_scale, v_scale, scale_stride, err);
      break;
  }
  return cudaGetLastError();
}

}  // namespace pfkv
