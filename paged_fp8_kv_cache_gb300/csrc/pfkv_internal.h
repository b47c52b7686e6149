// Internal interface between the C-ABI host code and the kernel translation units.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

namespace pfkv {

enum KvKind : int { kKvFp16 = 0, kKvE4m3 = 1, kKvE5m2 = 2 };

// must equal the PFKV_DEVERR_* bits of include/pfkv.h
constexpr unsigned kDevErrSlot = 0x1u;
constexpr unsigned kDevErrBlockId = 0x2u;
constexpr unsigned kDevErrSeqLen = 0x4u;
constexpr unsigned kDevErrTimeout = 0x8u;

// sequences of one call that the persistent decode grid takes (lengths and item prefix in shared memory)
constexpr int kMaxPersistSeqs = 1024;

struct DecodeParams {
  const __half* q;
  __half* out;
  float* lse;
  const int32_t* block_table;
  const int32_t* seq_lens;
  const float* k_scale;
  const float* v_scale;
  int scale_stride;  // 0: one scale per pool; 1: one per KV head (k_scale[kvh])
  float* o_part;
  float* lse_part;
  unsigned* err;
  int max_blocks;
  int num_seqs;
  int T;
  int num_q_heads;
  int num_kv_heads;
  int G;
  int page_size;
  int page_shift;
  int num_blocks;
  int max_seq_len;
  int split_tokens;
  int num_splits;
  int nrg;  // row groups (of 8*NT rows) per CTA
  int nts;  // consumer warps per row group (key slices)
  float softmax_scale;
  // mask and query slabs (mask_span.h): grid.y = num_kv_heads * num_slabs
  int causal;       // 1: query t sees no key after its own position
  int window;       // > 0: query t sees no key W or more positions before its own (0: no window)
  int slab_tokens;  // query tokens per CTA
  int num_slabs;    // ceil(T / slab_tokens)
  // persistent decode grid: the next unclaimed range (zeroed by the call before the launch)
  int* work_ctr;
};

struct DecodeLaunch {
  int head_dim;
  int kv;
  int nt;  // n-tiles of 8 query rows per consumer warp (1 or 2)
};

// Launch with programmatic stream serialisation: the grid may start while the
// previous kernel on the stream drains; the kernel executes griddepcontrol.wait
// before reading anything that kernel could have written.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, int smem, cudaStream_t stream,
                              Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// decode_fp16.cu / decode_e4m3.cu / decode_e5m2.cu: the mma.sync decode kernel per cache
// dtype; *_ctas_* returns the CTAs of a configuration that fit on one SM.
cudaError_t launch_decode_fp16(const DecodeLaunch&, const CUtensorMap&, const CUtensorMap&, const DecodeParams&, dim3,
                               cudaStream_t);
cudaError_t launch_decode_e4m3(const DecodeLaunch&, const CUtensorMap&, const CUtensorMap&, const DecodeParams&, dim3,
                               cudaStream_t);
cudaError_t launch_decode_e5m2(const DecodeLaunch&, const CUtensorMap&, const CUtensorMap&, const DecodeParams&, dim3,
                               cudaStream_t);
int decode_ctas_fp16(const DecodeLaunch&, int ncw);
int decode_ctas_e4m3(const DecodeLaunch&, int ncw);
int decode_ctas_e5m2(const DecodeLaunch&, int ncw);
// The persistent grid of the same kernel (one row tile per warp, one query slab, at most
// kMaxPersistSeqs sequences): ctas CTAs take the ranges from p.work_ctr, which must read 0.
cudaError_t launch_decode_persist_fp16(const DecodeLaunch&, const CUtensorMap&, const CUtensorMap&,
                                       const DecodeParams&, int ctas, cudaStream_t);
cudaError_t launch_decode_persist_e4m3(const DecodeLaunch&, const CUtensorMap&, const CUtensorMap&,
                                       const DecodeParams&, int ctas, cudaStream_t);
cudaError_t launch_decode_persist_e5m2(const DecodeLaunch&, const CUtensorMap&, const CUtensorMap&,
                                       const DecodeParams&, int ctas, cudaStream_t);
int decode_persist_ctas_fp16(const DecodeLaunch&, int ncw, int num_seqs);
int decode_persist_ctas_e4m3(const DecodeLaunch&, int ncw, int num_seqs);
int decode_persist_ctas_e5m2(const DecodeLaunch&, int ncw, int num_seqs);

// verify_e4m3.cu / verify_e5m2.cu: tcgen05 grouped verify (FP8 caches). nmax = rows padded
// to 32/48/64. With ctas_out non-null nothing is launched: it receives the CTAs per SM.
cudaError_t launch_verify_e4m3(int head_dim, int nmax, const CUtensorMap& tmk, const CUtensorMap& tmv,
                               const DecodeParams& p, dim3 grid, cudaStream_t stream, int* ctas_out);
cudaError_t launch_verify_e5m2(int head_dim, int nmax, const CUtensorMap& tmk, const CUtensorMap& tmv,
                               const DecodeParams& p, dim3 grid, cudaStream_t stream, int* ctas_out);

// How many parts each row of an attention call has (rows of sequence b = r / (T * Hq), query
// token (r / Hq) % T): the split ranges of its slab (mask_span.h); rows with one part are
// skipped (the attention kernel wrote them).
struct MergeRows {
  const int32_t* seq_lens;  // null: every row has num_parts parts
  int T, num_q_heads, slab_tokens, causal, window, tile, split_tokens, len_cap;
};

// merge.cu: combine per-range partials.
cudaError_t launch_lse_merge(__half* out, float* lse, const float* o_parts, const float* lse_parts, int rows,
                             int num_parts, int head_dim, const MergeRows& mr, cudaStream_t stream);

// zero_blocks.cu
cudaError_t launch_zero_blocks(void* k_cache, void* v_cache, const int32_t* block_ids, int n_ids, long long block_bytes,
                               int num_blocks, unsigned* err, cudaStream_t stream);

// append.cu
cudaError_t launch_append(const __half* k_new, const __half* v_new, void* k_cache, void* v_cache,
                          const int64_t* slots, int n_tok, int num_kv_heads, int head_dim, int page_size,
                          int num_blocks, int kv, const float* k_scale, const float* v_scale, int scale_stride,
                          unsigned* err, int num_sms, cudaStream_t stream);

}  // namespace pfkv
