// Internal interface between the C-ABI host code and the kernel translation units.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pfkv {

enum KvKind : int { kKvFp16 = 0, kKvE4m3 = 1, kKvE5m2 = 2 };

// must equal the PFKV_DEVERR_* bits of include/pfkv.h
constexpr unsigned kDevErrSlot = 0x1u;
constexpr unsigned kDevErrBlockId = 0x2u;
constexpr unsigned kDevErrSeqLen = 0x4u;
constexpr unsigned kDevErrTimeout = 0x8u;

struct DecodeParams {
  const __half* q;
  __half* out;
  float* lse;
  const int32_t* block_table;
  const int32_t* seq_lens;
  const float* k_scale;
  const float* v_scale;
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
};

struct DecodeLaunch {
  int head_dim;
  int kv;
  int nt;  // n-tiles of 8 query rows per consumer warp (1 or 2)
};

// decode_*.cu
cudaError_t launch_decode(const DecodeLaunch& cfg, const CUtensorMap& tmk, const CUtensorMap& tmv,
                          const DecodeParams& p, dim3 grid, cudaStream_t stream);
// Dynamic shared memory and threads per CTA of a decode configuration.
int decode_smem_request(const DecodeLaunch& cfg, int ncw);
// CTAs of this configuration that fit on one SM (cached per device).
int decode_ctas_per_sm(const DecodeLaunch& cfg, int ncw);

// merge.cu: combine per-range partials. If seq_lens is non-null, row r of
// sequence b = r / (T * num_q_heads) has ceil(seq_len / split_tokens) parts
// (rows with one part are skipped: the decode kernel wrote them); otherwise
// every row has num_parts parts.
cudaError_t launch_lse_merge(__half* out, float* lse, const float* o_parts, const float* lse_parts, int rows,
                             int num_parts, int head_dim, const int32_t* seq_lens, int rows_per_seq,
                             int split_tokens, int max_seq_len, int max_len_cap, cudaStream_t stream);

// append.cu
cudaError_t launch_append(const __half* k_new, const __half* v_new, void* k_cache, void* v_cache,
                          const int64_t* slots, int n_tok, int num_kv_heads, int head_dim, int page_size,
                          int num_blocks, int kv, const float* k_scale, const float* v_scale, unsigned* err,
                          cudaStream_t stream);

}  // namespace pfkv
