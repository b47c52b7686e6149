// LSE merge of split-KV partial results (the combine step of the split
// long-context decode route, "1Cat-vLLM 1.5.0", "Flash-V100 long-context
// improvements"):
//   M = max_s lse_s, w_s = exp(lse_s - M),
//   out = sum_s w_s o_s / sum_s w_s, lse = M + ln(sum_s w_s).
// Each thread owns 4 consecutive head-dim elements of one row; the row's
// part LSEs are read by every thread of the row (they stay in L1).
#include <cuda_fp16.h>
#include <math_constants.h>

#include "pfkv_internal.h"

namespace pfkv {

__global__ void __launch_bounds__(256) lse_merge_kernel(__half* __restrict__ out, float* __restrict__ lse,
                                                        const float* __restrict__ o_parts,
                                                        const float* __restrict__ lse_parts, int rows, int num_parts,
                                                        int head_dim, const int32_t* __restrict__ seq_lens,
                                                        int rows_per_seq, int split_tokens, int len_cap) {
  const int q4 = head_dim / 4;
  const int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
  if (idx >= static_cast<int64_t>(rows) * q4) return;
  const int r = static_cast<int>(idx / q4);
  const int d = static_cast<int>(idx - static_cast<int64_t>(r) * q4) * 4;
  int n = num_parts;
  if (seq_lens != nullptr) {
    int len = seq_lens[r / rows_per_seq];
    len = len < 0 ? 0 : (len > len_cap ? len_cap : len);
    n = len > 0 ? (len + split_tokens - 1) / split_tokens : 1;
    if (n <= 1) return;  // written directly by the decode kernel
  }
  const float* lp = lse_parts + static_cast<int64_t>(r) * num_parts;
  float M = -CUDART_INF_F;
  for (int s = 0; s < n; ++s) M = fmaxf(M, lp[s]);
  float W = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (M != -CUDART_INF_F) {
    const float* op = o_parts + static_cast<int64_t>(r) * num_parts * head_dim + d;
    for (int s = 0; s < n; ++s) {
      const float l = lp[s];
      if (l == -CUDART_INF_F) continue;
      const float w = expf(l - M);
      W += w;
      const float4 v = *reinterpret_cast<const float4*>(op + static_cast<int64_t>(s) * head_dim);
      acc.x += w * v.x;
      acc.y += w * v.y;
      acc.z += w * v.z;
      acc.w += w * v.w;
    }
  }
  const bool has = (M != -CUDART_INF_F) && (W > 0.f);
  const float inv = has ? 1.f / W : 0.f;
  const __half2 h01 = __floats2half2_rn(acc.x * inv, acc.y * inv);
  const __half2 h23 = __floats2half2_rn(acc.z * inv, acc.w * inv);
  uint2 packed;
  packed.x = *reinterpret_cast<const uint32_t*>(&h01);
  packed.y = *reinterpret_cast<const uint32_t*>(&h23);
  *reinterpret_cast<uint2*>(out + static_cast<int64_t>(r) * head_dim + d) = packed;
  if (d == 0 && lse != nullptr) lse[r] = has ? M + logf(W) : -CUDART_INF_F;
}

cudaError_t launch_lse_merge(__half* out, float* lse, const float* o_parts, const float* lse_parts, int rows,
                             int num_parts, int head_dim, const int32_t* seq_lens, int rows_per_seq,
                             int split_tokens, int max_seq_len, int max_len_cap, cudaStream_t stream) {
  (void)max_seq_len;
  const int64_t total = static_cast<int64_t>(rows) * (head_dim / 4);
  if (total == 0) return cudaSuccess;
  const int threads = 256;
  const int64_t blocks = (total + threads - 1) / threads;
  lse_merge_kernel<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(
      out, lse, o_parts, lse_parts, rows, num_parts, head_dim, seq_lens, rows_per_seq > 0 ? rows_per_seq : 1,
      split_tokens > 0 ? split_tokens : 1, max_len_cap);
  return cudaGetLastError();
}

}  // namespace pfkv
