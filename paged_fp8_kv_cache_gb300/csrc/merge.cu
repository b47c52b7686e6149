// LSE merge of split-KV partial results (the combine step of the split
// long-context decode route, "1Cat-vLLM 1.5.0", "Flash-V100 long-context
// improvements"):
//   M = max_s lse_s, w_s = exp(lse_s - M),
//   out = sum_s w_s o_s / sum_s w_s, lse = M + ln(sum_s w_s).
//
// One CTA per output row, of 1, 2, 4 or 8 warps (at least one per 8 parts of
// the call, so that a row costs one memory round trip up to 64 parts, and
// calls with many rows of few parts fit on the GPU in one wave); the row's
// parts are spread over the warps, each warp keeping a running maximum. When launched after the decode
// kernel with programmatic stream serialisation, the grid starts while the
// decode kernel drains and waits (griddepcontrol.wait) before touching the
// partials.
#include <cuda_fp16.h>
#include <math_constants.h>

#include "mask_span.h"
#include "pfkv_internal.h"

namespace pfkv {

template <int D, int NW>
__global__ void __launch_bounds__(NW * 32) lse_merge_kernel(__half* __restrict__ out, float* __restrict__ lse,
                                                            const float* __restrict__ o_parts,
                                                            const float* __restrict__ lse_parts, int rows,
                                                            int num_parts, const MergeRows mr) {
  // One CTA (NW warps) per row. Warp w takes parts w, w+NW, ...; each lane owns D/32
  // consecutive output elements. A warp issues the loads (LSE and output) of up to kBatch of
  // its parts at once and keeps a running maximum with sums rescaled to it, so a row costs
  // one memory round trip; the NW warps' results are then rescaled to the row maximum and
  // added through shared memory.
  constexpr int PER = D / 32;  // 4 or 8 floats per lane
  constexpr int kBatch = 8;
  __shared__ float s_m[NW];
  __shared__ float s_w[NW];
  __shared__ float4 s_acc[NW][D / 4];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int r = blockIdx.x;
  int n = num_parts;
  if (mr.seq_lens != nullptr) {
    // The sequence lengths are read before this grid's dependency wait: they are an input of
    // the decode call, complete before the decode kernel ran, and this grid starts only once
    // every CTA of the decode kernel has passed its own wait (the partials are not).
    const int rows_per_seq = mr.T * mr.num_q_heads;
    int len = mr.seq_lens[r / rows_per_seq];
    len = len < 0 ? 0 : (len > mr.len_cap ? mr.len_cap : len);
    const int t = (r / mr.num_q_heads) % mr.T;
    const SlabSpan sp = slab_span(len, mr.T, t / mr.slab_tokens, mr.slab_tokens, mr.causal, mr.window, mr.tile);
    n = span_splits(sp, mr.split_tokens);
    if (n <= 1) return;  // written directly by the attention kernel (uniform across the CTA)
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const float* lp = lse_parts + static_cast<int64_t>(r) * num_parts;
  const float* op = o_parts + static_cast<int64_t>(r) * num_parts * D + lane * PER;
  float Mw = -CUDART_INF_F, Ww = 0.f;  // this warp's running maximum and weight sum
  float acc[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) acc[i] = 0.f;
  for (int s0 = warp; s0 < n; s0 += NW * kBatch) {
    float4 v[kBatch][PER / 4];
    float l[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int s = s0 + NW * u;
      l[u] = -CUDART_INF_F;
      if (s < n) {
        l[u] = lp[s];
#pragma unroll
        for (int i = 0; i < PER / 4; ++i)
          v[u][i] = *reinterpret_cast<const float4*>(op + static_cast<int64_t>(s) * D + 4 * i);
      }
    }
    float bm = -CUDART_INF_F;
#pragma unroll
    for (int u = 0; u < kBatch; ++u) bm = fmaxf(bm, l[u]);
    const float nm = fmaxf(Mw, bm);
    if (nm == -CUDART_INF_F) continue;  // nothing visible yet (uniform across the warp)
    const float sc = (Mw == -CUDART_INF_F) ? 0.f : expf(Mw - nm);
    Ww *= sc;
#pragma unroll
    for (int i = 0; i < PER; ++i) acc[i] *= sc;
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      if (s0 + NW * u < n && l[u] != -CUDART_INF_F) {
        const float w = expf(l[u] - nm);
        Ww += w;
#pragma unroll
        for (int i = 0; i < PER / 4; ++i) {
          acc[4 * i + 0] += w * v[u][i].x;
          acc[4 * i + 1] += w * v[u][i].y;
          acc[4 * i + 2] += w * v[u][i].z;
          acc[4 * i + 3] += w * v[u][i].w;
        }
      }
    }
    Mw = nm;
  }
#pragma unroll
  for (int i = 0; i < PER / 4; ++i)
    s_acc[warp][lane * (PER / 4) + i] = make_float4(acc[4 * i], acc[4 * i + 1], acc[4 * i + 2], acc[4 * i + 3]);
  if (lane == 0) {
    s_m[warp] = Mw;
    s_w[warp] = Ww;
  }
  __syncthreads();
  // the D / 4 float4 outputs (D = 128: 32, D = 256: 64), one per thread while the CTA has them
  for (int t = threadIdx.x; t < D / 4; t += NW * 32) {
    float M = s_m[0];
#pragma unroll
    for (int w = 1; w < NW; ++w) M = fmaxf(M, s_m[w]);
    float Wt = 0.f;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    if (M != -CUDART_INF_F) {
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        const float f = (s_m[w] == -CUDART_INF_F) ? 0.f : expf(s_m[w] - M);
        Wt += f * s_w[w];
        const float4 x = s_acc[w][t];
        a.x += f * x.x;
        a.y += f * x.y;
        a.z += f * x.z;
        a.w += f * x.w;
      }
    }
    const bool has = (M != -CUDART_INF_F) && (Wt > 0.f);
    const float inv = has ? 1.f / Wt : 0.f;
    const __half2 h01 = __floats2half2_rn(a.x * inv, a.y * inv);
    const __half2 h23 = __floats2half2_rn(a.z * inv, a.w * inv);
    uint2 packed;
    packed.x = *reinterpret_cast<const uint32_t*>(&h01);
    packed.y = *reinterpret_cast<const uint32_t*>(&h23);
    *reinterpret_cast<uint2*>(out + static_cast<int64_t>(r) * D + 4 * t) = packed;
    if (t == 0 && lse != nullptr) lse[r] = has ? M + logf(Wt) : -CUDART_INF_F;
  }
}

// Warps per row: one per 8 parts (kBatch), at most 8.
template <int D>
cudaError_t launch_merge_d(const cudaLaunchConfig_t& base, __half* out, float* lse, const float* o_parts,
                           const float* lse_parts, int rows, int num_parts, const MergeRows& mr) {
  cudaLaunchConfig_t cfg = base;
  if (num_parts <= 8) {
    cfg.blockDim = dim3(32);
    return cudaLaunchKernelEx(&cfg, lse_merge_kernel<D, 1>, out, lse, o_parts, lse_parts, rows, num_parts, mr);
  }
  if (num_parts <= 16) {
    cfg.blockDim = dim3(64);
    return cudaLaunchKernelEx(&cfg, lse_merge_kernel<D, 2>, out, lse, o_parts, lse_parts, rows, num_parts, mr);
  }
  if (num_parts <= 32) {
    cfg.blockDim = dim3(128);
    return cudaLaunchKernelEx(&cfg, lse_merge_kernel<D, 4>, out, lse, o_parts, lse_parts, rows, num_parts, mr);
  }
  cfg.blockDim = dim3(256);
  return cudaLaunchKernelEx(&cfg, lse_merge_kernel<D, 8>, out, lse, o_parts, lse_parts, rows, num_parts, mr);
}

// Generic head dims (multiples of 4 up to 1024, standalone entry point only):
// one thread per 4 output elements.
__global__ void __launch_bounds__(256) lse_merge_generic_kernel(__half* __restrict__ out, float* __restrict__ lse,
                                                                const float* __restrict__ o_parts,
                                                                const float* __restrict__ lse_parts, int rows,
                                                                int num_parts, int head_dim) {
  const int q4 = head_dim / 4;
  const int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
  if (idx >= static_cast<int64_t>(rows) * q4) return;
  const int r = static_cast<int>(idx / q4);
  const int d = static_cast<int>(idx - static_cast<int64_t>(r) * q4) * 4;
  const float* lp = lse_parts + static_cast<int64_t>(r) * num_parts;
  float M = -CUDART_INF_F;
  for (int s = 0; s < num_parts; ++s) M = fmaxf(M, lp[s]);
  float W = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (M != -CUDART_INF_F) {
    const float* op = o_parts + static_cast<int64_t>(r) * num_parts * head_dim + d;
    for (int s = 0; s < num_parts; ++s) {
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
                             int num_parts, int head_dim, const MergeRows& mr, cudaStream_t stream) {
  if (rows == 0) return cudaSuccess;
  if (head_dim != 128 && head_dim != 256) {
    const int64_t total = static_cast<int64_t>(rows) * (head_dim / 4);
    const int64_t blocks = (total + 255) / 256;
    lse_merge_generic_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(out, lse, o_parts, lse_parts, rows,
                                                                               num_parts, head_dim);
    return cudaGetLastError();
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(rows));
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (head_dim == 128) return launch_merge_d<128>(cfg, out, lse, o_parts, lse_parts, rows, num_parts, mr);
  return launch_merge_d<256>(cfg, out, lse, o_parts, lse_parts, rows, num_parts, mr);
}

}  // namespace pfkv
