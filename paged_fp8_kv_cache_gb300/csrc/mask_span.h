// The keys one CTA of the attention kernels covers, shared by the kernels, the merge kernel and
// the host plan (host and device code).
//
// A sequence of N keys has T query tokens at positions p_t = N - T + t. Query t sees the keys
// lo_t <= j <= hi_t with
//   hi_t = p_t when causal (over its own drafts), N - 1 when not (a draft block attending to all
//          of its own tokens: the non-causal draft attention of "1Cat-vLLM 1.5.0", "Production
//          DFlash2 on V100");
//   lo_t = max(0, p_t - W + 1) with a sliding window of W keys (the draft's sliding-window
//          attention, same page, "Flash-V100 long-context improvements"), 0 without (W = 0).
// The T tokens are cut into slabs of slab_tokens consecutive tokens (one slab for a decode or a
// verify, many for a prefill chunk); a CTA takes the g query heads of one KV head for the tokens
// of one slab. lo_t and hi_t grow with t, so a slab's visible keys lie in [lo of its first
// token, hi of its last]. Its split ranges start at that lower bound rounded down to the
// kernel's tile (so tiles stay page-aligned) -- the tiles wholly before a window are never
// read -- and are split_tokens keys long.
#pragma once

#if defined(__CUDACC__)
#define PFKV_HD __host__ __device__ __forceinline__
#else
#define PFKV_HD inline
#endif

namespace pfkv {

struct SlabSpan {
  int ts0, ts1;  // query tokens [ts0, ts1) of the slab
  int lo, hi;    // its visible keys lie in [lo, hi] (none when hi < lo)
  int base;      // lo rounded down to the tile: where range 0 starts
};

PFKV_HD SlabSpan slab_span(int N, int T, int slab, int slab_tokens, int causal, int window, int tile) {
  SlabSpan s;
  s.ts0 = slab * slab_tokens;
  s.ts1 = (s.ts0 + slab_tokens < T) ? s.ts0 + slab_tokens : T;
  const int p0 = N - T + s.ts0, p1 = N - T + s.ts1 - 1;
  s.hi = (causal && p1 < N - 1) ? p1 : N - 1;
  s.lo = (window > 0 && p0 - window + 1 > 0) ? p0 - window + 1 : 0;
  s.base = s.lo & ~(tile - 1);
  return s;
}

// Split ranges of a slab (at least 1: an empty slab still has one CTA writing its empty rows).
PFKV_HD int span_splits(SlabSpan s, int split_tokens) {
  return s.hi >= s.lo ? (s.hi - s.base + split_tokens) / split_tokens : 1;
}

// Visible-key bounds of query token t.
PFKV_HD int key_hi(int N, int T, int t, int causal) {
  const int p = N - T + t;
  return (causal && p < N - 1) ? p : N - 1;
}
PFKV_HD int key_lo(int N, int T, int t, int window) {
  const int p = N - T + t;
  return (window > 0 && p - window + 1 > 0) ? p - window + 1 : 0;
}

}  // namespace pfkv
