// C ABI of libpfkv.so (declared in include/pfkv.h): argument validation,
// split-KV planning, TMA descriptor set-up and kernel launches on the
// caller's stream. Nothing here allocates device memory or synchronises.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <unordered_map>

#include "../../include/pfkv.h"
#include "frag_layout.h"
#include "mask_span.h"
#include "pfkv_internal.h"

namespace pfkv {

__device__ unsigned g_pfkv_err;  // per-device error word (PFKV_DEVERR_* bits)

namespace {

thread_local std::string g_last_error;

pfkv_status fail(pfkv_status st, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
pfkv_status fail(pfkv_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

pfkv_status cuda_fail(cudaError_t e, const char* what) {
  return fail(PFKV_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int g_sm_count[kMaxDevices];
unsigned* g_err_ptr[kMaxDevices];
unsigned long long g_err_ctx[kMaxDevices];  // context the cached error-word address belongs to
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
PFN_cuCtxGetId_v12000 g_ctx_id = nullptr;

struct TmKey {
  const void* ptr;
  int dev, kv, head_dim, page_size;
  long long rows;
  bool operator==(const TmKey& o) const {
    return ptr == o.ptr && dev == o.dev && kv == o.kv && head_dim == o.head_dim && page_size == o.page_size &&
           rows == o.rows;
  }
};
struct TmHash {
  size_t operator()(const TmKey& k) const {
    size_t h = std::hash<const void*>()(k.ptr);
    h ^= std::hash<long long>()(k.rows * 1315423911LL + k.head_dim * 31 + k.page_size * 7 + k.kv + k.dev * 101);
    return h;
  }
};
std::unordered_map<TmKey, CUtensorMap, TmHash> g_tmaps;
std::unordered_map<long long, int> g_occ;  // (device, kv, D, nt, ncw) -> CTAs per SM

cudaError_t current_device(int* dev) {
  cudaError_t e = cudaGetDevice(dev);
  if (e != cudaSuccess) return e;
  if (*dev < 0 || *dev >= kMaxDevices) return cudaErrorInvalidDevice;
  return cudaSuccess;
}

cudaError_t sm_count(int dev, int* n) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_sm_count[dev] == 0) {
    cudaError_t e = cudaDeviceGetAttribute(&g_sm_count[dev], cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
  }
  *n = g_sm_count[dev];
  return cudaSuccess;
}

// Unique id of the current CUDA context (0 if the driver cannot tell). A device symbol's address
// belongs to the context the module was loaded in: after cudaDeviceReset the device gets a new
// primary context, and addresses cached for the old one must be looked up again.
unsigned long long context_id() {
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_ctx_current == nullptr || g_ctx_id == nullptr) {
    void* f1 = nullptr;
    void* f2 = nullptr;
    cudaDriverEntryPointQueryResult q1, q2;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 4000, cudaEnableDefault, &q1) != cudaSuccess ||
        q1 != cudaDriverEntryPointSuccess ||
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault, &q2) != cudaSuccess ||
        q2 != cudaDriverEntryPointSuccess)
      return 0;
    g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f1);
    g_ctx_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(f2);
  }
  CUcontext c = nullptr;
  unsigned long long id = 0;
  if (g_ctx_current(&c) != CUDA_SUCCESS || c == nullptr || g_ctx_id(c, &id) != CUDA_SUCCESS) return 0;
  return id;
}

cudaError_t err_word(int dev, unsigned** p) {
  const unsigned long long ctx = context_id();
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_err_ptr[dev] == nullptr || g_err_ctx[dev] != ctx) {
    void* a = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&a, g_pfkv_err);
    if (e != cudaSuccess) return e;
    g_err_ptr[dev] = static_cast<unsigned*>(a);
    g_err_ctx[dev] = ctx;
  }
  *p = g_err_ptr[dev];
  return cudaSuccess;
}

pfkv_status get_encoder() {
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_encode) return PFKV_OK;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
  if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || fn == nullptr)
    return fail(PFKV_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
  g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  return PFKV_OK;
}

// Tensor map over a cache pool viewed as rows of head_dim elements:
// [num_blocks * Hkv * page_size rows][head_dim], 128-byte boxes of
// min(page_size, 64) rows, 128-byte swizzle.
pfkv_status tensor_map(int dev, const void* pool, int kv, int head_dim, int page_size, long long rows,
                       CUtensorMap* out) {
  TmKey key{pool, dev, kv, head_dim, page_size, rows};
  {
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_tmaps.find(key);
    if (it != g_tmaps.end()) {
      *out = it->second;
      return PFKV_OK;
    }
  }
  pfkv_status st = get_encoder();
  if (st != PFKV_OK) return st;
  const int elt = kv == kKvFp16 ? 2 : 1;
  CUtensorMap m;
  cuuint64_t gdim[2] = {static_cast<cuuint64_t>(head_dim), static_cast<cuuint64_t>(rows)};
  cuuint64_t gstride[1] = {static_cast<cuuint64_t>(head_dim) * elt};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(kBoxBytes / elt),
                       static_cast<cuuint32_t>(page_size < kTileKeys ? page_size : kTileKeys)};
  cuuint32_t estride[2] = {1, 1};
  CUresult r = g_encode(&m, elt == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_UINT16, 2,
                        const_cast<void*>(pool), gdim, gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(PFKV_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_tmaps.size() > 256) g_tmaps.clear();
    g_tmaps[key] = m;
  }
  *out = m;
  return PFKV_OK;
}

int kv_of(pfkv_kv_dtype d) {
  return d == PFKV_KV_FP16 ? kKvFp16 : (d == PFKV_KV_FP8_E4M3 ? kKvE4m3 : kKvE5m2);
}

bool valid_dtype(pfkv_kv_dtype d) {
  return d == PFKV_KV_FP16 || d == PFKV_KV_FP8_E4M3 || d == PFKV_KV_FP8_E5M2;
}

// A dtype argument is a cache format, optionally ORed with PFKV_KV_SCALES_PER_HEAD (FP8 only).
bool split_dtype(pfkv_kv_dtype in, pfkv_kv_dtype* fmt, int* scale_stride) {
  const unsigned v = static_cast<unsigned>(in);
  *fmt = static_cast<pfkv_kv_dtype>(v & ~static_cast<unsigned>(PFKV_KV_SCALES_PER_HEAD));
  *scale_stride = (v & PFKV_KV_SCALES_PER_HEAD) ? 1 : 0;
  return valid_dtype(*fmt) && !(*scale_stride && *fmt == PFKV_KV_FP16);
}

bool is_pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

int log2i(int x) {
  int s = 0;
  while ((1 << s) < x) ++s;
  return s;
}

constexpr int kMaxQTokens = 8192;  // query tokens per sequence of one call (a prefill chunk)
constexpr int kMaxRows = 64;       // query rows per CTA (a slab of tokens x the group's heads)

struct Plan {
  DecodeLaunch cfg;
  int nrg, nts, ncw;  // mma.sync decode kernel: row groups x key slices of consumer warps
  bool tc;            // tcgen05 grouped-verify kernel (FP8 cache, more than 16 rows per KV head)
  int nmax;           // its padded row count (32, 48, 64)
  int tile;           // keys per pipeline tile (split ranges are multiples of it)
  int splits, split_tokens;
  int causal, window;          // the mask (window 0 when it cannot bind: at least max_seq_len)
  int slab_tokens, num_slabs;  // query tokens per CTA
};

int ctas_per_sm(int dev, const DecodeLaunch& cfg, int ncw, bool tc, int nmax) {
  const long long key =
      ((((static_cast<long long>(dev) * 4 + cfg.kv) * 512 + cfg.head_dim) * 4 + cfg.nt) * 64 + ncw) * 256 +
      (tc ? nmax : 0);
  {
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_occ.find(key);
    if (it != g_occ.end()) return it->second;
  }
  int n = 1;
  if (tc) {
    CUtensorMap unused;
    std::memset(&unused, 0, sizeof(unused));
    DecodeParams none;
    std::memset(&none, 0, sizeof(none));
    if (cfg.kv == kKvE4m3)
      launch_verify_e4m3(cfg.head_dim, nmax, unused, unused, none, dim3(1), nullptr, &n);
    else
      launch_verify_e5m2(cfg.head_dim, nmax, unused, unused, none, dim3(1), nullptr, &n);
  } else {
    n = cfg.kv == kKvFp16 ? decode_ctas_fp16(cfg, ncw)
                          : (cfg.kv == kKvE4m3 ? decode_ctas_e4m3(cfg, ncw) : decode_ctas_e5m2(cfg, ncw));
  }
  std::lock_guard<std::mutex> lk(g_mu);
  g_occ[key] = n;
  return n;
}

// Shape checks shared by plan / workspace / attention.
pfkv_status check_shape(int num_seqs, int T, int Hq, int Hkv, int D, int P, pfkv_kv_dtype dtype, int mask,
                        int window, int max_seq_len, int num_splits) {
  if (num_seqs < 0 || Hq <= 0 || Hkv <= 0 || max_seq_len < 0 || num_splits < 0 || window < 0)
    return fail(PFKV_ERR_INVALID_ARG,
                "negative size (num_seqs=%d Hq=%d Hkv=%d max_seq_len=%d num_splits=%d window=%d)", num_seqs, Hq,
                Hkv, max_seq_len, num_splits, window);
  if (Hq % Hkv != 0) return fail(PFKV_ERR_INVALID_ARG, "num_q_heads %d not a multiple of num_kv_heads %d", Hq, Hkv);
  if (!valid_dtype(dtype)) return fail(PFKV_ERR_INVALID_ARG, "unknown kv dtype %d", static_cast<int>(dtype));
  if (mask & ~PFKV_MASK_CAUSAL) return fail(PFKV_ERR_INVALID_ARG, "unknown mask bits 0x%x", mask);
  if (T < 1 || T > kMaxQTokens) return fail(PFKV_ERR_UNSUPPORTED, "num_q_tokens %d outside 1..%d", T, kMaxQTokens);
  if (D != 128 && D != 256) return fail(PFKV_ERR_UNSUPPORTED, "head_dim %d (supported: 128, 256)", D);
  if (!is_pow2(P) || P < 16 || P > 2048)
    return fail(PFKV_ERR_UNSUPPORTED, "page_size %d (supported: powers of two 16..2048)", P);
  if (Hq / Hkv > kMaxRows) return fail(PFKV_ERR_UNSUPPORTED, "group size %d > %d", Hq / Hkv, kMaxRows);
  if (static_cast<long long>(num_seqs) * T * Hq > 0x7fffffffLL)
    return fail(PFKV_ERR_UNSUPPORTED, "num_seqs * num_q_tokens * num_q_heads exceeds 2^31");
  return PFKV_OK;
}

// Zeroes the persistent decode grid's range counter. Launched with programmatic serialisation
// between the previous kernel on the stream (e.g. the step's append, which releases its
// dependents at once) and the persistent grid (which waits for this one): unlike a memset node it
// lets both launches overlap the kernel before.
__global__ void zero_counter_kernel(int* ctr) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (threadIdx.x == 0) *ctr = 0;
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

pfkv_status make_plan(int num_seqs, int T, int Hq, int Hkv, int D, int P, pfkv_kv_dtype dtype, int mask, int window,
                      int max_seq_len, int num_splits_request, Plan* pl) {
  pfkv_status st = check_shape(num_seqs, T, Hq, Hkv, D, P, dtype, mask, window, max_seq_len, num_splits_request);
  if (st != PFKV_OK) return st;
  const int G = Hq / Hkv;
  // query slabs: every token in one CTA when its rows fit, else slabs of 64 / G tokens
  pl->slab_tokens = T * G <= kMaxRows ? T : kMaxRows / G;
  pl->num_slabs = (T + pl->slab_tokens - 1) / pl->slab_tokens;
  if (static_cast<long long>(Hkv) * pl->num_slabs > 65535)
    return fail(PFKV_ERR_UNSUPPORTED, "num_kv_heads * query slabs = %lld > 65535",
                static_cast<long long>(Hkv) * pl->num_slabs);
  pl->causal = (mask & PFKV_MASK_CAUSAL) ? 1 : 0;
  pl->window = window >= max_seq_len ? 0 : window;  // a window of at least every length never binds
  const int R = pl->slab_tokens * G;
  pl->cfg.head_dim = D;
  pl->cfg.kv = kv_of(dtype);
  pl->cfg.nt = R <= 8 ? 1 : 2;
  const int rows_w = 8 * pl->cfg.nt;
  pl->nrg = (R + rows_w - 1) / rows_w;
  pl->nts = pl->nrg == 1 ? 4 : 2;
  pl->ncw = pl->nrg * pl->nts;
  pl->tc = (dtype != PFKV_KV_FP16) && R > 16;
  pl->nmax = R <= 32 ? 32 : (R <= 48 ? 48 : 64);
  pl->tile = pl->tc ? 128 : kTileKeys;
  // the longest key span of a slab: the sequence, or with a window the window plus the tokens
  // a slab's rows spread over (all T without the causal bound) plus the tile alignment
  long long span = max_seq_len;
  if (pl->window > 0) {
    const long long w = static_cast<long long>(pl->causal ? pl->slab_tokens : T) + pl->window + pl->tile;
    if (w < span) span = w;
  }
  const int tiles = span > 0 ? static_cast<int>((span + pl->tile - 1) / pl->tile) : 1;
  int want;
  if (num_splits_request > 0) {
    want = num_splits_request;
  } else {
    int dev, sms;
    cudaError_t e = current_device(&dev);
    if (e == cudaSuccess) e = sm_count(dev, &sms);
    if (e != cudaSuccess) return cuda_fail(e, "device query");
    const int units = num_seqs > 0 ? num_seqs * Hkv * pl->num_slabs : 1;
    const int occ = ctas_per_sm(dev, pl->cfg, pl->ncw, pl->tc, pl->nmax);
    int base = (sms * occ + units - 1) / units;
    // Long ranges at full occupancy: one CTA per SM with ranges twice as long measured faster
    // (128K-key decode: 38 ranges 54 us, 76 ranges 58 us; with 4096 keys, 5 tiles per range,
    // the three CTAs per SM stay ahead).
    const bool long_ranges = !pl->tc && occ > 1 && tiles >= 24 * base;
    if (long_ranges) base = (sms + units - 1) / units;
    // Bound the keys per CTA so ragged batches balance (when sequences outnumber the SMs, each
    // range is a unit of work of the wave); the bound grows with the row count because every
    // range costs an fp32 partial per row, and doubles for the tcgen05 kernel (one CTA per
    // SM, with a fixed start-up and first-tile cost worth ~8 tiles: two waves of half-length
    // ranges cost more than one wave).
    const int max_keys = (pl->tc ? 2 : 1) * (R * 256 > 2048 ? R * 256 : 2048);
    const int need = (long_ranges && units < sms) ? 1 : static_cast<int>((span + max_keys - 1) / max_keys);
    const int k = base > 0 ? (need + base - 1) / base : 1;
    want = base * (k > 1 ? k : 1);
    // Tensor-core calls with units for a wave or more already (prefill chunks: a unit per query
    // slab): the ranges only shorten the CTAs of the last wave, and each costs a partial per
    // row and a merge term. Take the count, up to the bound, whose waves are fullest per unit of
    // work, each range past the first counted 1.15 % dearer (2048-token chunk over 128K keys,
    // 820 units: 9671 / 9299 / 9605 / 9464 / 9443 us at 1 / 2 / 3 / 4 / 5 ranges).
    if (pl->tc && units >= sms * occ && want > 1) {
      const long long slots = static_cast<long long>(sms) * occ;
      double best = 0.0;
      int pick = 1;
      for (int s = 1; s <= want; ++s) {
        const long long waves = (static_cast<long long>(units) * s + slots - 1) / slots;
        const double cost = static_cast<double>(waves) / s * (1.0 + 0.0115 * (s - 1));
        if (s == 1 || cost < best) {
          best = cost;
          pick = s;
        }
      }
      want = pick;
    }
  }
  if (want < 1) want = 1;
  if (want > tiles) want = tiles;
  const int tiles_per_split = (tiles + want - 1) / want;
  pl->split_tokens = tiles_per_split * pl->tile;
  pl->splits = (tiles + tiles_per_split - 1) / tiles_per_split;
  return PFKV_OK;
}

// Split partials (o_part, lse_part), then the persistent grid's range counter at the next
// 16-byte boundary.
size_t counter_offset(const Plan& pl, int num_seqs, int T, int Hq, int D) {
  const size_t rows = static_cast<size_t>(num_seqs) * T * Hq;
  const size_t o = rows * pl.splits * D * sizeof(float);
  const size_t l = rows * pl.splits * sizeof(float);
  return (o + l + 15) & ~static_cast<size_t>(15);
}

size_t workspace_for(const Plan& pl, int num_seqs, int T, int Hq, int D) {
  if (pl.splits <= 1) return 0;
  return counter_offset(pl, num_seqs, T, Hq, D) + 16;
}

// The decode entry points keep their contract: causal, no window, 1..16 query tokens whose rows
// (tokens x group heads) fit one CTA.
pfkv_status check_decode_tokens(int T, int Hq, int Hkv) {
  if (T < 1 || T > 16) return fail(PFKV_ERR_UNSUPPORTED, "num_q_tokens %d outside 1..16", T);
  if (Hkv > 0 && Hq % Hkv == 0 && T * (Hq / Hkv) > kMaxRows)
    return fail(PFKV_ERR_UNSUPPORTED, "num_q_tokens * group size = %d > %d rows per KV head", T * (Hq / Hkv),
                kMaxRows);
  return PFKV_OK;
}

pfkv_status plan_impl(int num_seqs, int num_q_tokens, int num_q_heads, int num_kv_heads, int head_dim, int page_size,
                      pfkv_kv_dtype dtype_arg, int mask, int window, int max_seq_len, int num_splits_request,
                      int* num_splits, int* split_tokens) {
  pfkv_kv_dtype dtype;
  int unused_stride;
  if (!split_dtype(dtype_arg, &dtype, &unused_stride))
    return fail(PFKV_ERR_INVALID_ARG, "unknown kv dtype %d", static_cast<int>(dtype_arg));
  Plan pl;
  pfkv_status st = make_plan(num_seqs, num_q_tokens, num_q_heads, num_kv_heads, head_dim, page_size, dtype, mask,
                             window, max_seq_len, num_splits_request, &pl);
  if (st != PFKV_OK) return st;
  if (num_splits) *num_splits = pl.splits;
  if (split_tokens) *split_tokens = pl.split_tokens;
  return PFKV_OK;
}

size_t workspace_impl(int num_seqs, int num_q_tokens, int num_q_heads, int num_kv_heads, int head_dim, int page_size,
                      pfkv_kv_dtype dtype_arg, int mask, int window, int max_seq_len, int num_splits_request) {
  pfkv_kv_dtype dtype;
  int unused_stride;
  if (!split_dtype(dtype_arg, &dtype, &unused_stride)) return 0;
  Plan pl;
  if (make_plan(num_seqs, num_q_tokens, num_q_heads, num_kv_heads, head_dim, page_size, dtype, mask, window,
                max_seq_len, num_splits_request, &pl) != PFKV_OK)
    return 0;
  return workspace_for(pl, num_seqs, num_q_tokens, num_q_heads, head_dim);
}

pfkv_status attention_impl(void* out, float* lse, const void* q, const void* k_cache, const void* v_cache,
                           const int32_t* block_table, int max_blocks_per_seq, const int32_t* seq_lens, int num_seqs,
                           int num_q_tokens, int num_q_heads, int num_kv_heads, int head_dim, int page_size,
                           int num_blocks, pfkv_kv_dtype dtype_arg, const float* k_scale, const float* v_scale,
                           float softmax_scale, int mask, int window, int max_seq_len, int num_splits,
                           void* workspace, size_t workspace_bytes, pfkv_stream_t stream) {
  pfkv_kv_dtype dtype;
  int scale_stride;
  if (!split_dtype(dtype_arg, &dtype, &scale_stride))
    return fail(PFKV_ERR_INVALID_ARG, "unknown kv dtype %d", static_cast<int>(dtype_arg));
  Plan pl;
  pfkv_status st = make_plan(num_seqs, num_q_tokens, num_q_heads, num_kv_heads, head_dim, page_size, dtype, mask,
                             window, max_seq_len, num_splits, &pl);
  if (st != PFKV_OK) return st;
  if (num_seqs == 0) return PFKV_OK;
  if (!out || !lse || !q || !k_cache || !v_cache || !block_table || !seq_lens)
    return fail(PFKV_ERR_INVALID_ARG, "null pointer");
  if (dtype != PFKV_KV_FP16 && (!k_scale || !v_scale)) return fail(PFKV_ERR_INVALID_ARG, "null scale pointer");
  if (num_blocks <= 0 || max_blocks_per_seq <= 0)
    return fail(PFKV_ERR_INVALID_ARG, "num_blocks=%d max_blocks_per_seq=%d", num_blocks, max_blocks_per_seq);
  const long long rows = static_cast<long long>(num_blocks) * num_kv_heads * page_size;
  if (rows > 0x7fffffffLL) return fail(PFKV_ERR_UNSUPPORTED, "cache pool of %lld rows exceeds 2^31", rows);
  if (static_cast<long long>(max_blocks_per_seq) * page_size > 0x7fffffffLL)
    return fail(PFKV_ERR_UNSUPPORTED, "max_blocks_per_seq * page_size exceeds 2^31");
  if ((reinterpret_cast<uintptr_t>(k_cache) | reinterpret_cast<uintptr_t>(v_cache)) & 15)
    return fail(PFKV_ERR_INVALID_ARG, "cache pools must be 16-byte aligned");
  if (reinterpret_cast<uintptr_t>(q) & 15)
    return fail(PFKV_ERR_INVALID_ARG, "q must be 16-byte aligned");  // the verify kernel reads 16-byte pieces
  if (reinterpret_cast<uintptr_t>(out) & 7) return fail(PFKV_ERR_INVALID_ARG, "out must be 8-byte aligned");
  if (reinterpret_cast<uintptr_t>(lse) & 3) return fail(PFKV_ERR_INVALID_ARG, "lse must be 4-byte aligned");
  const size_t need = workspace_for(pl, num_seqs, num_q_tokens, num_q_heads, head_dim);
  if (need > 0) {
    if (!workspace || workspace_bytes < need)
      return fail(PFKV_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need, workspace_bytes);
    if (reinterpret_cast<uintptr_t>(workspace) & 15)
      return fail(PFKV_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
  }
  int dev;
  unsigned* err;
  cudaError_t e = current_device(&dev);
  if (e == cudaSuccess) e = err_word(dev, &err);
  if (e != cudaSuccess) return cuda_fail(e, "device set-up");

  CUtensorMap tmk, tmv;
  const int kv = kv_of(dtype);
  st = tensor_map(dev, k_cache, kv, head_dim, page_size, rows, &tmk);
  if (st != PFKV_OK) return st;
  st = tensor_map(dev, v_cache, kv, head_dim, page_size, rows, &tmv);
  if (st != PFKV_OK) return st;

  DecodeParams p;
  p.q = static_cast<const __half*>(q);
  p.out = static_cast<__half*>(out);
  p.lse = lse;
  p.block_table = block_table;
  p.seq_lens = seq_lens;
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.scale_stride = scale_stride;
  const size_t nrows = static_cast<size_t>(num_seqs) * num_q_tokens * num_q_heads;
  p.o_part = need ? static_cast<float*>(workspace) : nullptr;
  p.lse_part = need ? static_cast<float*>(workspace) + nrows * pl.splits * head_dim : nullptr;
  p.err = err;
  p.max_blocks = max_blocks_per_seq;
  p.num_seqs = num_seqs;
  p.T = num_q_tokens;
  p.num_q_heads = num_q_heads;
  p.num_kv_heads = num_kv_heads;
  p.G = num_q_heads / num_kv_heads;
  p.page_size = page_size;
  p.page_shift = log2i(page_size);
  p.num_blocks = num_blocks;
  p.max_seq_len = max_seq_len;
  p.split_tokens = pl.split_tokens;
  p.num_splits = pl.splits;
  p.nrg = pl.nrg;
  p.nts = pl.nts;
  p.softmax_scale = softmax_scale;
  p.causal = pl.causal;
  p.window = pl.window;
  p.slab_tokens = pl.slab_tokens;
  p.num_slabs = pl.num_slabs;
  p.work_ctr = nullptr;

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  dim3 grid(pl.splits, num_kv_heads * pl.num_slabs, num_seqs);
  // A grid of more than two waves, sized for the longest sequence the call allows, holds many
  // CTAs without work when the batch is ragged (each still takes an SM slot for a few
  // microseconds): one-slab decode then runs as one wave of CTAs that claim the ranges that exist.
  int persist_ctas = 0;
  if (!pl.tc && pl.num_slabs == 1 && pl.cfg.nt == 1 && pl.splits > 1 && num_seqs <= kMaxPersistSeqs) {
    int sms;
    e = sm_count(dev, &sms);
    if (e != cudaSuccess) return cuda_fail(e, "device query");
    const long long ctas = static_cast<long long>(num_seqs) * num_kv_heads * pl.splits;
    const int occ = ctas_per_sm(dev, pl.cfg, pl.ncw, false, 0);
    if (ctas > 2LL * sms * occ) {
      const int pocc = kv == kKvFp16 ? decode_persist_ctas_fp16(pl.cfg, pl.ncw, num_seqs)
                                     : (kv == kKvE4m3 ? decode_persist_ctas_e4m3(pl.cfg, pl.ncw, num_seqs)
                                                      : decode_persist_ctas_e5m2(pl.cfg, pl.ncw, num_seqs));
      persist_ctas = static_cast<int>(std::min<long long>(static_cast<long long>(sms) * pocc, ctas));
    }
  }
  if (persist_ctas > 0) {
    p.work_ctr = reinterpret_cast<int*>(static_cast<char*>(workspace) +
                                        counter_offset(pl, num_seqs, num_q_tokens, num_q_heads, head_dim));
    e = launch_pdl(zero_counter_kernel, dim3(1), dim3(32), 0, s, p.work_ctr);
    if (e != cudaSuccess) return cuda_fail(e, "range counter reset");
    e = kv == kKvFp16 ? launch_decode_persist_fp16(pl.cfg, tmk, tmv, p, persist_ctas, s)
                      : (kv == kKvE4m3 ? launch_decode_persist_e4m3(pl.cfg, tmk, tmv, p, persist_ctas, s)
                                       : launch_decode_persist_e5m2(pl.cfg, tmk, tmv, p, persist_ctas, s));
  } else if (pl.tc) {
    e = kv == kKvE4m3 ? launch_verify_e4m3(head_dim, pl.nmax, tmk, tmv, p, grid, s, nullptr)
                      : launch_verify_e5m2(head_dim, pl.nmax, tmk, tmv, p, grid, s, nullptr);
  } else {
    e = kv == kKvFp16 ? launch_decode_fp16(pl.cfg, tmk, tmv, p, grid, s)
                      : (kv == kKvE4m3 ? launch_decode_e4m3(pl.cfg, tmk, tmv, p, grid, s)
                                       : launch_decode_e5m2(pl.cfg, tmk, tmv, p, grid, s));
  }
  if (e != cudaSuccess) return cuda_fail(e, "attention launch");
  if (pl.splits > 1) {
    const long long cap_ll = static_cast<long long>(max_blocks_per_seq) * page_size;
    MergeRows mr;
    mr.seq_lens = seq_lens;
    mr.T = num_q_tokens;
    mr.num_q_heads = num_q_heads;
    mr.slab_tokens = pl.slab_tokens;
    mr.causal = pl.causal;
    mr.window = pl.window;
    mr.tile = pl.tile;
    mr.split_tokens = pl.split_tokens;
    mr.len_cap = static_cast<int>(cap_ll < max_seq_len ? cap_ll : max_seq_len);
    e = launch_lse_merge(p.out, lse, p.o_part, p.lse_part, static_cast<int>(nrows), pl.splits, head_dim, mr, s);
    if (e != cudaSuccess) return cuda_fail(e, "merge launch");
  }
  return PFKV_OK;
}

}  // namespace
}  // namespace pfkv

using namespace pfkv;

extern "C" {

const char* pfkv_status_string(pfkv_status s) {
  switch (s) {
    case PFKV_OK: return "PFKV_OK";
    case PFKV_ERR_INVALID_ARG: return "PFKV_ERR_INVALID_ARG";
    case PFKV_ERR_UNSUPPORTED: return "PFKV_ERR_UNSUPPORTED";
    case PFKV_ERR_WORKSPACE: return "PFKV_ERR_WORKSPACE";
    case PFKV_ERR_CUDA: return "PFKV_ERR_CUDA";
    case PFKV_ERR_DEVICE_CHECK: return "PFKV_ERR_DEVICE_CHECK";
  }
  return "PFKV_UNKNOWN_STATUS";
}

const char* pfkv_last_error(void) { return g_last_error.c_str(); }

uint32_t pfkv_capabilities(void) {
  return PFKV_CAP_KV_FP16 | PFKV_CAP_KV_FP8_E4M3 | PFKV_CAP_KV_FP8_E5M2 | PFKV_CAP_HEAD_DIM_128 |
         PFKV_CAP_HEAD_DIM_256 | PFKV_CAP_PAGE_16 | PFKV_CAP_PAGE_2048 | PFKV_CAP_PAGE_POW2_ANY |
         PFKV_CAP_Q_TOKENS_1_8 | PFKV_CAP_Q_TOKENS_1_16 | PFKV_CAP_SPLIT_KV |
         PFKV_CAP_SCALES_PER_HEAD | PFKV_CAP_NON_CAUSAL | PFKV_CAP_SLIDING_WINDOW | PFKV_CAP_PREFILL;
}

pfkv_status pfkv_device_errors(uint32_t* flags, int clear) {
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
  unsigned v = 0;
  e = cudaMemcpyFromSymbol(&v, g_pfkv_err, sizeof(v));
  if (e != cudaSuccess) return cuda_fail(e, "read error word");
  if (clear) {
    const unsigned zero = 0;
    e = cudaMemcpyToSymbol(g_pfkv_err, &zero, sizeof(zero));
    if (e != cudaSuccess) return cuda_fail(e, "clear error word");
  }
  if (flags) *flags = v;
  return v ? fail(PFKV_ERR_DEVICE_CHECK, "device error word 0x%x", v) : PFKV_OK;
}

pfkv_status pfkv_kv_cache_append(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                                 const int64_t* slot_mapping, int n_tok, int num_kv_heads, int head_dim,
                                 int page_size, int num_blocks, pfkv_kv_dtype dtype_arg, const float* k_scale,
                                 const float* v_scale, pfkv_stream_t stream) {
  if (n_tok < 0 || num_kv_heads <= 0 || head_dim <= 0 || page_size <= 0 || num_blocks <= 0)
    return fail(PFKV_ERR_INVALID_ARG, "bad size (n_tok=%d Hkv=%d D=%d P=%d num_blocks=%d)", n_tok, num_kv_heads,
                head_dim, page_size, num_blocks);
  pfkv_kv_dtype dtype;
  int scale_stride;
  if (!split_dtype(dtype_arg, &dtype, &scale_stride))
    return fail(PFKV_ERR_INVALID_ARG, "unknown kv dtype %d", static_cast<int>(dtype_arg));
  if (head_dim % 8 != 0 || head_dim > 1024)
    return fail(PFKV_ERR_UNSUPPORTED, "head_dim %d (must be a multiple of 8, at most 1024)", head_dim);
  if (n_tok == 0) return PFKV_OK;
  if (!k_new || !v_new || !k_cache || !v_cache || !slot_mapping)
    return fail(PFKV_ERR_INVALID_ARG, "null pointer");
  if (dtype != PFKV_KV_FP16 && (!k_scale || !v_scale)) return fail(PFKV_ERR_INVALID_ARG, "null scale pointer");
  if ((reinterpret_cast<uintptr_t>(k_new) | reinterpret_cast<uintptr_t>(v_new) |
       reinterpret_cast<uintptr_t>(k_cache) | reinterpret_cast<uintptr_t>(v_cache)) & 15)
    return fail(PFKV_ERR_INVALID_ARG, "K/V and cache pointers must be 16-byte aligned");
  int dev, sms;
  unsigned* err;
  cudaError_t e = current_device(&dev);
  if (e == cudaSuccess) e = err_word(dev, &err);
  if (e == cudaSuccess) e = sm_count(dev, &sms);
  if (e != cudaSuccess) return cuda_fail(e, "device set-up");
  e = launch_append(static_cast<const __half*>(k_new), static_cast<const __half*>(v_new), k_cache, v_cache,
                    slot_mapping, n_tok, num_kv_heads, head_dim, page_size, num_blocks, kv_of(dtype), k_scale, v_scale,
                    scale_stride, err, sms, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PFKV_OK : cuda_fail(e, "append launch");
}

pfkv_status pfkv_kv_cache_zero_blocks(void* k_cache, void* v_cache, const int32_t* block_ids, int n_ids,
                                      int num_kv_heads, int head_dim, int page_size, int num_blocks,
                                      pfkv_kv_dtype dtype_arg, pfkv_stream_t stream) {
  if (n_ids < 0 || num_kv_heads <= 0 || head_dim <= 0 || page_size <= 0 || num_blocks <= 0)
    return fail(PFKV_ERR_INVALID_ARG, "bad size (n_ids=%d Hkv=%d D=%d P=%d num_blocks=%d)", n_ids, num_kv_heads,
                head_dim, page_size, num_blocks);
  pfkv_kv_dtype dtype;
  int unused_stride;
  if (!split_dtype(dtype_arg, &dtype, &unused_stride))
    return fail(PFKV_ERR_INVALID_ARG, "unknown kv dtype %d", static_cast<int>(dtype_arg));
  // every cache row a whole number of 16-byte stores
  const int row_bytes = head_dim * (dtype == PFKV_KV_FP16 ? 2 : 1);
  if (row_bytes % 16 != 0 || head_dim > 1024)
    return fail(PFKV_ERR_UNSUPPORTED, "head_dim %d (rows of a multiple of 16 bytes, at most 1024 elements)",
                head_dim);
  if (n_ids == 0) return PFKV_OK;
  if (!k_cache || !v_cache || !block_ids) return fail(PFKV_ERR_INVALID_ARG, "null pointer");
  if ((reinterpret_cast<uintptr_t>(k_cache) | reinterpret_cast<uintptr_t>(v_cache)) & 15)
    return fail(PFKV_ERR_INVALID_ARG, "cache pointers must be 16-byte aligned");
  const long long elt = dtype == PFKV_KV_FP16 ? 2 : 1;
  const long long block_bytes = static_cast<long long>(num_kv_heads) * page_size * head_dim * elt;
  int dev;
  unsigned* err;
  cudaError_t e = current_device(&dev);
  if (e == cudaSuccess) e = err_word(dev, &err);
  if (e != cudaSuccess) return cuda_fail(e, "device set-up");
  e = launch_zero_blocks(k_cache, v_cache, block_ids, n_ids, block_bytes, num_blocks, err,
                         reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PFKV_OK : cuda_fail(e, "zero_blocks launch");
}


pfkv_status pfkv_attention_plan(int num_seqs, int num_q_tokens, int num_q_heads, int num_kv_heads, int head_dim,
                                int page_size, pfkv_kv_dtype dtype, int mask, int window, int max_seq_len,
                                int num_splits_request, int* num_splits, int* split_tokens) {
  return plan_impl(num_seqs, num_q_tokens, num_q_heads, num_kv_heads, head_dim, page_size, dtype, mask, window,
                   max_seq_len, num_splits_request, num_splits, split_tokens);
}

size_t pfkv_attention_workspace_bytes(int num_seqs, int num_q_tokens, int num_q_heads, int num_kv_heads,
                                      int head_dim, int page_size, pfkv_kv_dtype dtype, int mask, int window,
                                      int max_seq_len, int num_splits_request) {
  return workspace_impl(num_seqs, num_q_tokens, num_q_heads, num_kv_heads, head_dim, page_size, dtype, mask, window,
                        max_seq_len, num_splits_request);
}

pfkv_status pfkv_paged_attention(void* out, float* lse, const void* q, const void* k_cache, const void* v_cache,
                                 const int32_t* block_table, int max_blocks_per_seq, const int32_t* seq_lens,
                                 int num_seqs, int num_q_tokens, int num_q_heads, int num_kv_heads, int head_dim,
                                 int page_size, int num_blocks, pfkv_kv_dtype dtype, const float* k_scale,
                                 const float* v_scale, float softmax_scale, int mask, int window, int max_seq_len,
                                 int num_splits, void* workspace, size_t workspace_bytes, pfkv_stream_t stream) {
  return attention_impl(out, lse, q, k_cache, v_cache, block_table, max_blocks_per_seq, seq_lens, num_seqs,
                        num_q_tokens, num_q_heads, num_kv_heads, head_dim, page_size, num_blocks, dtype, k_scale,
                        v_scale, softmax_scale, mask, window, max_seq_len, num_splits, workspace, workspace_bytes,
                        stream);
}

pfkv_status pfkv_decode_plan(int num_seqs, int num_q_tokens, int num_q_heads, int num_kv_heads, int head_dim,
                             int page_size, pfkv_kv_dtype dtype, int max_seq_len, int num_splits_request,
                             int* num_splits, int* split_tokens) {
  pfkv_status st = check_decode_tokens(num_q_tokens, num_q_heads, num_kv_heads);
  if (st != PFKV_OK) return st;
  return plan_impl(num_seqs, num_q_tokens, num_q_heads, num_kv_heads, head_dim, page_size, dtype, PFKV_MASK_CAUSAL,
                   0, max_seq_len, num_splits_request, num_splits, split_tokens);
}

size_t pfkv_decode_workspace_bytes(int num_seqs, int num_q_tokens, int num_q_heads, int num_kv_heads, int head_dim,
                                   int page_size, pfkv_kv_dtype dtype, int max_seq_len, int num_splits_request) {
  if (check_decode_tokens(num_q_tokens, num_q_heads, num_kv_heads) != PFKV_OK) return 0;
  return workspace_impl(num_seqs, num_q_tokens, num_q_heads, num_kv_heads, head_dim, page_size, dtype,
                        PFKV_MASK_CAUSAL, 0, max_seq_len, num_splits_request);
}

pfkv_status pfkv_paged_attention_decode(void* out, float* lse, const void* q, const void* k_cache, const void* v_cache,
                                        const int32_t* block_table, int max_blocks_per_seq, const int32_t* seq_lens,
                                        int num_seqs, int num_q_tokens, int num_q_heads, int num_kv_heads,
                                        int head_dim, int page_size, int num_blocks, pfkv_kv_dtype dtype,
                                        const float* k_scale, const float* v_scale, float softmax_scale,
                                        int max_seq_len, int num_splits, void* workspace, size_t workspace_bytes,
                                        pfkv_stream_t stream) {
  pfkv_status st = check_decode_tokens(num_q_tokens, num_q_heads, num_kv_heads);
  if (st != PFKV_OK) return st;
  return attention_impl(out, lse, q, k_cache, v_cache, block_table, max_blocks_per_seq, seq_lens, num_seqs,
                        num_q_tokens, num_q_heads, num_kv_heads, head_dim, page_size, num_blocks, dtype, k_scale,
                        v_scale, softmax_scale, PFKV_MASK_CAUSAL, 0, max_seq_len, num_splits, workspace,
                        workspace_bytes, stream);
}

pfkv_status pfkv_lse_merge(void* out, float* lse, const float* o_parts, const float* lse_parts, int rows,
                           int num_parts, int head_dim, pfkv_stream_t stream) {
  if (rows < 0 || num_parts <= 0 || head_dim <= 0)
    return fail(PFKV_ERR_INVALID_ARG, "bad size (rows=%d parts=%d D=%d)", rows, num_parts, head_dim);
  if (head_dim % 4 != 0 || head_dim > 1024)
    return fail(PFKV_ERR_UNSUPPORTED, "head_dim %d (multiple of 4, at most 1024)", head_dim);
  if (rows == 0) return PFKV_OK;
  if (!out || !o_parts || !lse_parts) return fail(PFKV_ERR_INVALID_ARG, "null pointer");
  if ((reinterpret_cast<uintptr_t>(o_parts) & 15) || (reinterpret_cast<uintptr_t>(out) & 7))
    return fail(PFKV_ERR_INVALID_ARG, "o_parts must be 16-byte and out 8-byte aligned");
  if (static_cast<long long>(rows) * num_parts * head_dim > (1LL << 40))
    return fail(PFKV_ERR_INVALID_ARG, "too large");
  MergeRows every_row = {};  // no sequence lengths: every row has num_parts parts
  cudaError_t e = launch_lse_merge(static_cast<__half*>(out), lse, o_parts, lse_parts, rows, num_parts, head_dim,
                                   every_row, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PFKV_OK : cuda_fail(e, "merge launch");
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Decode without caller-provided scratch.
//
// Some callers cannot allocate device memory: for example a plugin running
// inside another engine whose memory pool reserved nearly all of the GPU for
// its KV cache up front (a fresh cudaMalloc would fail), or a latency-critical
// serving loop where cudaMalloc/cudaFree would implicitly synchronise the
// device. For them the split partials live in a fixed array that is part of
// this library's device image: every GPU that loads the library holds
// kPfkvStaticScratchBytes of it until the process exits.
namespace {

constexpr size_t kPfkvStaticScratchBytes = size_t(32) << 20;  // 32 MiB
static __device__ __align__(256) unsigned char g_pfkv_static_scratch[kPfkvStaticScratchBytes];
void* g_static_scratch_ptr[kMaxDevices];
unsigned long long g_static_scratch_ctx[kMaxDevices];

// Device address of the array on the current device. In host code the
// array's name is only a host-side stand-in, never a device address: it is
// looked up once per device (with that device current) and cached, and looked
// up again if the device's context changed since (after a cudaDeviceReset).
pfkv_status static_scratch_address(void** out) {
  int dev;
  cudaError_t e = current_device(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  const unsigned long long ctx = context_id();
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_static_scratch_ptr[dev] == nullptr || g_static_scratch_ctx[dev] != ctx) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_pfkv_static_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(static scratch)");
    g_static_scratch_ptr[dev] = p;
    g_static_scratch_ctx[dev] = ctx;
  }
  *out = g_static_scratch_ptr[dev];
  return PFKV_OK;
}

}  // namespace

extern "C" pfkv_status pfkv_paged_attention_decode_static_scratch(
    void* out, float* lse, const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
    int max_blocks_per_seq, const int32_t* seq_lens, int num_seqs, int num_q_tokens, int num_q_heads,
    int num_kv_heads, int head_dim, int page_size, int num_blocks, pfkv_kv_dtype dtype, const float* k_scale,
    const float* v_scale, float softmax_scale, int max_seq_len, int num_splits, pfkv_stream_t stream) {
  const size_t need = pfkv_decode_workspace_bytes(num_seqs, num_q_tokens, num_q_heads, num_kv_heads, head_dim,
                                                  page_size, dtype, max_seq_len, num_splits);
  if (need > kPfkvStaticScratchBytes)
    return fail(PFKV_ERR_WORKSPACE,
                "this call needs %zu bytes of split scratch; the built-in array holds %zu (use fewer splits, "
                "fewer sequences or pfkv_paged_attention_decode with your own workspace)",
                need, kPfkvStaticScratchBytes);
  void* scratch = nullptr;
  pfkv_status st = static_scratch_address(&scratch);
  if (st != PFKV_OK) return st;
  return pfkv_paged_attention_decode(out, lse, q, k_cache, v_cache, block_table, max_blocks_per_seq, seq_lens,
                                     num_seqs, num_q_tokens, num_q_heads, num_kv_heads, head_dim, page_size,
                                     num_blocks, dtype, k_scale, v_scale, softmax_scale, max_seq_len, num_splits,
                                     scratch, kPfkvStaticScratchBytes, stream);
}
