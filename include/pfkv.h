/*
 * pfkv: paged FP8 KV-cache decode attention for NVIDIA GB300 (sm_103a).
 *
 * C ABI of libpfkv.so. Plain pointers and sizes only; every device pointer
 * is owned by the caller. The library never allocates or frees device
 * memory, never synchronises a stream and never reads device memory from the
 * host on these entry points (the diagnostic pfkv_device_errors() is the one
 * exception, and says so). All work is enqueued on the caller's stream.
 *
 * Where the operations come from. The pages describing the method are the
 * release notes and docs of an SM70 serving fork:
 *   [R1] "1Cat-vLLM" (README), sections "What is new in 1.0.0" and
 *        "Optional experimental feature: FP8 KV cache";
 *   [R2] "1Cat-vLLM 1.5.0" (release notes), sections "Production DFlash2 on
 *        V100", "Flash-V100 long-context improvements" and "Reliability and
 *        correctness fixes";
 *   [R3] "SM70 release profile and acceleration status", the profile
 *        paragraph (2048-token KV blocks) and the override table.
 * Each entry point below names the passage that defines its operation.
 *
 * Cache layout (a reading; the pages give none): one pool per K and V,
 * [num_blocks][num_kv_heads][page_size][head_dim], row-major, one byte per
 * element for FP8 and two for fp16. Element (block, kvh, off, d) is at
 * ((block * num_kv_heads + kvh) * page_size + off) * head_dim + d.
 * A sequence's key j lives in block block_table[b][j / page_size] at offset
 * j % page_size.
 *
 * Errors. Arguments are validated on the host before anything is enqueued;
 * a bad argument returns PFKV_ERR_INVALID_ARG, a shape the kernels do not
 * implement returns PFKV_ERR_UNSUPPORTED (there is no fallback path), a
 * failed launch returns PFKV_ERR_CUDA. Values that live in device memory
 * (block ids, slots, sequence lengths) are checked by the kernels: a bad
 * value sets a bit in a per-device error word (see pfkv_device_errors), the
 * offending access is skipped or redirected to a valid address, and the
 * kernels never trap.
 */
#ifndef PFKV_H
#define PFKV_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__) || defined(__clang__)
#define PFKV_API __attribute__((visibility("default")))
#else
#define PFKV_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Opaque stream handle: a cudaStream_t (CUstream_st*). NULL = legacy default stream. */
typedef struct CUstream_st* pfkv_stream_t;

typedef enum {
  PFKV_OK = 0,
  PFKV_ERR_INVALID_ARG = 1,  /* null pointer, negative size, Hq % Hkv != 0, ... */
  PFKV_ERR_UNSUPPORTED = 2,  /* head_dim / page_size / num_q_tokens / dtype not implemented */
  PFKV_ERR_WORKSPACE = 3,    /* workspace missing or smaller than pfkv_decode_workspace_bytes() */
  PFKV_ERR_CUDA = 4,         /* a CUDA runtime/driver call or a launch failed */
  PFKV_ERR_DEVICE_CHECK = 5  /* returned by pfkv_device_errors() when a kernel flagged bad data */
} pfkv_status;

typedef enum {
  PFKV_KV_FP16 = 0,      /* no quantisation: the cache holds the fp16 bits */
  PFKV_KV_FP8_E4M3 = 1,  /* E4M3 "fn": bias 7, max 448, no inf, NaN = S.1111.111 */
  PFKV_KV_FP8_E5M2 = 2   /* E5M2: bias 15, max 57344, IEEE-style inf/NaN */
} pfkv_kv_dtype;

/*
 * OR this flag into the dtype argument of pfkv_kv_cache_append,
 * pfkv_paged_attention_decode or pfkv_paged_attention_decode_static_scratch
 * with an FP8 cache to pass one static scale per KV head: k_scale and v_scale
 * then point to num_kv_heads floats each, and KV head h is quantised,
 * decoded and scaled with k_scale[h] / v_scale[h]. (The pages use one
 * per-tensor scale per pool; per-head scales are the generalisation of it.)
 * pfkv_decode_plan, pfkv_decode_workspace_bytes and pfkv_kv_cache_zero_blocks
 * accept and ignore the flag; with an fp16 cache it is an invalid argument.
 */
#define PFKV_KV_SCALES_PER_HEAD 0x100

/* Bits of the per-device error word (pfkv_device_errors). */
#define PFKV_DEVERR_SLOT      0x1u  /* append: slot >= num_blocks * page_size (token skipped) */
#define PFKV_DEVERR_BLOCK_ID  0x2u  /* decode: block_table entry outside [0, num_blocks) (block 0 read instead);
                                       zero_blocks: listed id >= num_blocks (skipped) */
#define PFKV_DEVERR_SEQ_LEN   0x4u  /* decode: seq_len < 0 or > min(max_seq_len, max_blocks_per_seq * page_size) (clamped) */
#define PFKV_DEVERR_TIMEOUT   0x8u  /* decode: a pipeline wait exceeded its iteration limit (CTA abandoned its work) */

/* Capability bits (pfkv_capabilities). */
#define PFKV_CAP_KV_FP16        0x001u
#define PFKV_CAP_KV_FP8_E4M3    0x002u
#define PFKV_CAP_KV_FP8_E5M2    0x004u
#define PFKV_CAP_HEAD_DIM_128   0x010u
#define PFKV_CAP_HEAD_DIM_256   0x020u
#define PFKV_CAP_PAGE_16        0x100u
#define PFKV_CAP_PAGE_2048      0x200u
#define PFKV_CAP_PAGE_POW2_ANY  0x400u  /* any power-of-two page size from 16 to 2048 */
#define PFKV_CAP_Q_TOKENS_1_8   0x1000u /* 1..8 causal query tokens per sequence */
#define PFKV_CAP_Q_TOKENS_1_16  0x4000u /* 1..16 causal query tokens (a q16 verify), rows <= 64 */
#define PFKV_CAP_SPLIT_KV       0x2000u /* split-KV partitions + LSE merge kernel */
#define PFKV_CAP_SCALES_PER_HEAD 0x8000u /* PFKV_KV_SCALES_PER_HEAD: one FP8 scale per KV head */
#define PFKV_CAP_NON_CAUSAL     0x10000u /* pfkv_paged_attention without PFKV_MASK_CAUSAL */
#define PFKV_CAP_SLIDING_WINDOW 0x20000u /* pfkv_paged_attention with window > 0 (prefix tiles skipped) */
#define PFKV_CAP_PREFILL        0x40000u /* pfkv_paged_attention with up to 8192 query tokens per sequence */

/* The mask argument of pfkv_paged_attention (a bit set). */
#define PFKV_MASK_CAUSAL 0x1  /* query t sees no key after its own position */

/*
 * pfkv_kv_cache_append -- quantise new K/V tokens and write them into their
 * pages (the KV write path named next to the attention extension in [R1];
 * static per-tensor scales, never computed online, [R1] "Optional
 * experimental feature: FP8 KV cache"; 16- or 2048-token pages, [R3]).
 *
 * For token i (0 <= i < n_tok) with slot = slot_mapping[i] >= 0, block =
 * slot / page_size, off = slot % page_size, for every KV head h and d:
 *   FP8:  cache[block][h][off][d] = fp8_rne_satfinite(float(x) / *scale)
 *         (fp16 widened to float, IEEE round-to-nearest division by the
 *         float scale, then round-to-nearest-even to the FP8 format with
 *         saturation to its largest finite value);
 *   FP16: cache[block][h][off][d] = x (bit copy).
 * A negative slot skips the token. A slot >= num_blocks * page_size skips
 * the token and sets PFKV_DEVERR_SLOT. Distinct tokens must name distinct
 * slots (otherwise which one lands is unspecified).
 *
 *   k_new, v_new   device, fp16 [n_tok][num_kv_heads][head_dim], 16-byte aligned
 *   k_cache, v_cache device pools as described above, 16-byte aligned
 *   slot_mapping   device, int64 [n_tok]
 *   k_scale, v_scale device, one float each (num_kv_heads each with
 *                  PFKV_KV_SCALES_PER_HEAD); ignored (may be NULL) for FP16
 *   head_dim       a multiple of 8 (any value up to 1024)
 * n_tok == 0 enqueues nothing and returns PFKV_OK.
 */
PFKV_API pfkv_status pfkv_kv_cache_append(const void* k_new, const void* v_new,
                                 void* k_cache, void* v_cache,
                                 const int64_t* slot_mapping, int n_tok,
                                 int num_kv_heads, int head_dim, int page_size,
                                 int num_blocks, pfkv_kv_dtype dtype,
                                 const float* k_scale, const float* v_scale,
                                 pfkv_stream_t stream);

/*
 * pfkv_kv_cache_zero_blocks -- clear every byte of the listed blocks in both
 * pools (all KV heads, all page offsets), so that a block handed to a new
 * sequence holds nothing of its previous owner ([R2] "Reliability and
 * correctness fixes": newly reused KV blocks are zeroed before attention, on
 * the device, with no host staging). The zero byte is +0 in every cache
 * dtype.
 *
 *   k_cache, v_cache device pools as described above, 16-byte aligned
 *   block_ids      device, int32 [n_ids]; a negative id is skipped; an id >=
 *                  num_blocks is skipped and sets PFKV_DEVERR_BLOCK_ID;
 *                  repeated ids are allowed
 *   head_dim       up to 1024, with rows of a multiple of 16 bytes (a
 *                  multiple of 16 for FP8, of 8 for fp16)
 * n_ids == 0 enqueues nothing and returns PFKV_OK. Blocks not listed are not
 * written.
 */
PFKV_API pfkv_status pfkv_kv_cache_zero_blocks(void* k_cache, void* v_cache,
                                      const int32_t* block_ids, int n_ids,
                                      int num_kv_heads, int head_dim, int page_size,
                                      int num_blocks, pfkv_kv_dtype dtype,
                                      pfkv_stream_t stream);

/*
 * pfkv_decode_plan -- the split-KV partition pfkv_paged_attention_decode
 * will use for these arguments (same arguments, same result, on the current
 * device). Long contexts are cut into *num_splits ranges of *split_tokens
 * keys (the last one shorter) that independent CTAs process; their partial
 * results are combined by the LSE merge (the long-context E4M3 route of
 * [R2] "Flash-V100 long-context improvements"). num_splits_request > 0
 * forces that many ranges for a max_seq_len-long sequence (rounded so every
 * range is a multiple of 64 keys); 0 lets the library choose from the SM
 * count and occupancy. A sequence of length n uses ceil(n / split_tokens)
 * ranges (at least 1).
 */
PFKV_API pfkv_status pfkv_decode_plan(int num_seqs, int num_q_tokens, int num_q_heads,
                             int num_kv_heads, int head_dim, int page_size,
                             pfkv_kv_dtype dtype, int max_seq_len,
                             int num_splits_request, int* num_splits,
                             int* split_tokens);

/*
 * pfkv_decode_workspace_bytes -- bytes of scratch pfkv_paged_attention_decode
 * needs for these arguments (0 when no sequence is split). Layout, for
 * S = *num_splits of pfkv_decode_plan and rows = num_seqs * num_q_tokens *
 * num_q_heads:
 *   float o_part[rows][S][head_dim]   at offset 0
 *   float lse_part[rows][S]           right after it
 *   int   range_counter               at the next 16-byte boundary, then
 *                                     12 bytes of padding
 * Row index = (b * num_q_tokens + t) * num_q_heads + h. For a row whose
 * sequence was split, o_part[row][s] is the attention output of range s
 * normalised by its own weight sum and lse_part[row][s] its natural-log
 * LSE (-inf when the range holds no key visible to the row); rows of
 * sequences that were not split are not written. range_counter serves the
 * persistent grid that large ragged decode batches run on (one wave of CTAs
 * taking the key ranges that exist, one after another, instead of one CTA
 * per range of the longest allowed sequence): the call zeroes it on the
 * stream before that grid starts, and afterwards it holds the number of
 * key ranges the grid processed. Nothing in the workspace needs to start
 * at zero.
 */
PFKV_API size_t pfkv_decode_workspace_bytes(int num_seqs, int num_q_tokens, int num_q_heads,
                                   int num_kv_heads, int head_dim, int page_size,
                                   pfkv_kv_dtype dtype, int max_seq_len,
                                   int num_splits_request);

/*
 * pfkv_paged_attention_decode -- paged decode attention over an FP8 (or
 * fp16) KV cache, and its grouped causal multi-token form used to verify
 * speculative drafts ([R2] "Flash-V100 long-context improvements": batched
 * FP8 decode reusing page IDs with 128-bit cache loads, long-context E4M3
 * routing, grouped q8 verifier; [R2] "Production DFlash2 on V100": exact
 * grouped q8 verification over FP8 KV, 7 drafts + 1 = 8 query tokens).
 *
 * For sequence b (N = seq_lens[b] keys, which already include the T query
 * tokens), query token t < T (position N - T + t), query head h, with
 * g = num_q_heads / num_kv_heads and kvh = h / g:
 *   s_j = softmax_scale * *k_scale * sum_d q[d] * dec(K[j][d])  for j <= N-T+t
 *   out = *v_scale * sum_j exp(s_j - m) dec(V[j]) / sum_j exp(s_j - m)
 *   lse = m + ln(sum_j exp(s_j - m)),  m = max_j s_j
 * where dec() is the exact FP8 (or fp16) value of a cache element. A row
 * that sees no key gets out = 0 and lse = -inf.
 *
 *   out            device, fp16 [num_seqs * T][num_q_heads][head_dim], 8-byte aligned
 *   lse            device, float [num_seqs * T][num_q_heads], 4-byte aligned
 *   q              device, fp16 [num_seqs * T][num_q_heads][head_dim], 16-byte aligned
 *   k_cache, v_cache device pools (see top of file); 16-byte aligned
 *   block_table    device, int32 [num_seqs][max_blocks_per_seq]; entries past
 *                  a sequence's last page are never read
 *   seq_lens       device, int32 [num_seqs]
 *   k_scale, v_scale device floats, one each (num_kv_heads each with
 *                  PFKV_KV_SCALES_PER_HEAD); ignored (may be NULL) for FP16 caches
 *   max_seq_len    host upper bound on seq_lens (sizes the split plan)
 *   num_splits     see pfkv_decode_plan (0 = automatic)
 *   workspace      device scratch of at least pfkv_decode_workspace_bytes()
 *                  (256-byte aligned; may be NULL when that is 0)
 * Supported: head_dim 128 or 256; page_size a power of two in [16, 2048];
 * 1 <= num_q_tokens <= 16 (e.g. 15 drafts + 1 for a q16 verify);
 * num_q_heads % num_kv_heads == 0 and num_q_tokens * g <= 64.
 *
 * Arithmetic (within 2e-3 of the exact out and 1e-4 of the exact lse on
 * unit-scale inputs): cache values are decoded exactly; logits are fp32
 * sums; the softmax weights enter the PV product rounded to fp16, while their
 * sums stay fp32. With an FP8 cache and more than 16 rows per KV head
 * (num_q_tokens * g) the kernel runs on the 5th-generation tensor cores and
 * Q enters them as three E4M3 terms per element (each row scaled by a power
 * of two), whose sum equals the fp16 value to within half an E4M3 subnormal
 * step of the scaled row.
 */
PFKV_API pfkv_status pfkv_paged_attention_decode(void* out, float* lse, const void* q,
                                        const void* k_cache, const void* v_cache,
                                        const int32_t* block_table, int max_blocks_per_seq,
                                        const int32_t* seq_lens, int num_seqs,
                                        int num_q_tokens, int num_q_heads, int num_kv_heads,
                                        int head_dim, int page_size, int num_blocks,
                                        pfkv_kv_dtype dtype, const float* k_scale,
                                        const float* v_scale, float softmax_scale,
                                        int max_seq_len, int num_splits,
                                        void* workspace, size_t workspace_bytes,
                                        pfkv_stream_t stream);

/*
 * pfkv_paged_attention -- the same paged attention with a choice of mask and
 * any number of query tokens per sequence: the non-causal sliding-window
 * draft attention ([R2] "Production DFlash2 on V100": non-causal
 * sliding-window draft attention; [R2] "Flash-V100 long-context
 * improvements": the draft's sliding-window attention skips the prefix tiles
 * it does not use) and the chunked prefill over the paged FP8 cache ([R2]
 * "Flash-V100 long-context improvements": the long-prefill GQA path that
 * packs the heads of a group into wider tensor-core work; [R3] the prefill
 * chunk budgets of the profile).
 *
 * Arguments, layouts and results as pfkv_paged_attention_decode, plus:
 *   mask    PFKV_MASK_CAUSAL, or 0 for a non-causal block of queries
 *   window  0 (none), or W > 0: query t sees no key W or more positions
 *           before its own
 * For query t at position p = N - T + t the visible keys are lo <= j <= hi
 * with hi = p (causal) or N - 1 (not), lo = max(0, p - W + 1) (window) or 0.
 * (A reading: the pages name the mask but do not define it; the window
 * bounds how far back a query looks, the causal bit how far forward.) Keys
 * wholly before every query's window are never read, so the cost of a
 * windowed call does not grow with the context.
 * Supported: 1 <= num_q_tokens <= 8192 and a group of at most 64 query heads
 * per KV head; the T tokens are processed in slabs of up to 64 rows (tokens x
 * heads of the group) per CTA. num_splits, the workspace and its layout are
 * as for the decode, sized by pfkv_attention_plan /
 * pfkv_attention_workspace_bytes (same arguments plus mask and window); a
 * row's split partials cover the ranges of its slab only.
 */
PFKV_API pfkv_status pfkv_paged_attention(void* out, float* lse, const void* q,
                                 const void* k_cache, const void* v_cache,
                                 const int32_t* block_table, int max_blocks_per_seq,
                                 const int32_t* seq_lens, int num_seqs, int num_q_tokens,
                                 int num_q_heads, int num_kv_heads, int head_dim,
                                 int page_size, int num_blocks, pfkv_kv_dtype dtype,
                                 const float* k_scale, const float* v_scale,
                                 float softmax_scale, int mask, int window,
                                 int max_seq_len, int num_splits, void* workspace,
                                 size_t workspace_bytes, pfkv_stream_t stream);

/* pfkv_attention_plan / pfkv_attention_workspace_bytes -- pfkv_decode_plan and
 * pfkv_decode_workspace_bytes for pfkv_paged_attention (same meaning; the
 * mask and window change the key span a CTA covers). */
PFKV_API pfkv_status pfkv_attention_plan(int num_seqs, int num_q_tokens, int num_q_heads,
                                int num_kv_heads, int head_dim, int page_size,
                                pfkv_kv_dtype dtype, int mask, int window, int max_seq_len,
                                int num_splits_request, int* num_splits, int* split_tokens);
PFKV_API size_t pfkv_attention_workspace_bytes(int num_seqs, int num_q_tokens, int num_q_heads,
                                      int num_kv_heads, int head_dim, int page_size,
                                      pfkv_kv_dtype dtype, int mask, int window,
                                      int max_seq_len, int num_splits_request);

/*
 * pfkv_paged_attention_decode_static_scratch -- pfkv_paged_attention_decode
 * for callers that cannot allocate device memory. (An addition of this
 * library: the pages have no counterpart.)
 *
 * Who needs it: code that runs inside another engine's memory pool, which
 * has already reserved nearly all device memory (typically for its own KV
 * cache) so that a cudaMalloc would fail, or a latency-critical serving loop
 * in which cudaMalloc / cudaFree would implicitly synchronise the device.
 *
 * Same arguments and results as pfkv_paged_attention_decode, without the
 * workspace: the split partials go to a fixed 32 MiB array compiled into the
 * library's device image (every GPU that loads the library holds it until
 * the process exits). Nothing is allocated or freed, by this call or by
 * anything it calls.
 *  - Size limit: if pfkv_decode_workspace_bytes() for these arguments exceeds
 *    32 MiB (33554432 bytes) the call returns PFKV_ERR_WORKSPACE and enqueues
 *    nothing. The workloads of this library need at most about 16 MB.
 *  - Set-up: the first call on each device looks up the array's device
 *    address (cudaGetSymbolAddress, with that device current) and caches it
 *    (a call after cudaDeviceReset, in the device's new context, looks it up
 *    again); make that first call before any stream capture.
 *  - Sharing: every call on a device uses the same array, and it keeps the
 *    last call's contents (nothing in it needs to start at zero). Calls whose
 *    work overlaps on the GPU (other streams, or another thread's calls)
 *    race on it: order them on one stream or synchronise between them.
 */
PFKV_API pfkv_status pfkv_paged_attention_decode_static_scratch(
    void* out, float* lse, const void* q, const void* k_cache, const void* v_cache,
    const int32_t* block_table, int max_blocks_per_seq, const int32_t* seq_lens,
    int num_seqs, int num_q_tokens, int num_q_heads, int num_kv_heads, int head_dim,
    int page_size, int num_blocks, pfkv_kv_dtype dtype, const float* k_scale,
    const float* v_scale, float softmax_scale, int max_seq_len, int num_splits,
    pfkv_stream_t stream);

/*
 * pfkv_lse_merge -- combine per-range partial attention results into the
 * final output (the merge step of the split long-context route of [R2]
 * "Flash-V100 long-context improvements"). For each row r:
 *   M = max_s lse_parts[r][s]; w_s = exp(lse_parts[r][s] - M)
 *   out[r] = sum_s w_s o_parts[r][s] / sum_s w_s;  lse[r] = M + ln sum_s w_s
 * Parts with lse = -inf carry no weight; a row whose parts are all -inf
 * gets out = 0, lse = -inf.
 *
 *   out        device, fp16 [rows][head_dim]
 *   lse        device, float [rows] (may be NULL)
 *   o_parts    device, float [rows][num_parts][head_dim]
 *   lse_parts  device, float [rows][num_parts]
 *   head_dim   a multiple of 4, at most 1024
 */
PFKV_API pfkv_status pfkv_lse_merge(void* out, float* lse, const float* o_parts,
                           const float* lse_parts, int rows, int num_parts,
                           int head_dim, pfkv_stream_t stream);

/*
 * pfkv_device_errors -- read (and optionally clear) the error word of the
 * current device. Synchronises the device first (diagnostic use only).
 * Returns PFKV_OK if no bit is set, PFKV_ERR_DEVICE_CHECK otherwise; *flags
 * receives the PFKV_DEVERR_* bits (may be NULL).
 */
PFKV_API pfkv_status pfkv_device_errors(uint32_t* flags, int clear);

/* Bitmask of PFKV_CAP_* the library implements (cf. the route capability
 * report of [R3]). */
PFKV_API uint32_t pfkv_capabilities(void);

/* Human-readable name of a status code. */
PFKV_API const char* pfkv_status_string(pfkv_status status);

/* Message describing the last non-OK status returned on this host thread. */
PFKV_API const char* pfkv_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* PFKV_H */
