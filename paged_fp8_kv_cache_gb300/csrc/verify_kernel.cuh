// Grouped causal-verify attention on the 5th-generation tensor cores
// (tcgen05 + TMEM) for FP8 caches: the g*T query rows of one KV head
// (e.g. 6 heads x 8 speculative tokens = 48 rows, "1Cat-vLLM 1.5.0",
// "Production DFlash2 on V100" / "Flash-V100 long-context improvements":
// exact grouped q8 verification over FP8 KV) form a real dense tile.
//
// One CTA = one (key range, KV head, query slab, sequence), 14 warps (the slab
// is all T tokens of a verify, or up to 64 rows of a prefill chunk; the mask --
// causal or not, sliding window -- bounds each row's keys from both sides, and
// a CTA's range starts at its slab's lowest visible key: mask_span.h):
//   warp 0      producers: TMA tile copies of 128-key FP8 K (lane 0) and V
//               (lane 1) tiles into two shared-memory rings (same tensor maps
//               as the decode kernel);
//   warp 1      MMA issuer (one lane) and TMEM owner;
//   warps 2-9   softmax: each thread owns one key of the tile (its TMEM lane)
//               and half of the query rows; it pulls the key's logits from
//               TMEM into registers (releasing the single S^T buffer to the
//               next tile's MMAs), masks, exponentiates against a per-row
//               reference maximum and writes P^T (fp16) into a swizzled
//               shared-memory B operand; at the end it reads O^T back from
//               TMEM and writes the output;
//   warps 10-13 V converter: each thread owns one TMEM lane = one or two
//               head-dim elements and writes them for all keys of the tile,
//               FP8 -> fp16 (exact), as the A operand of O^T = V^T P^T
//               (two TMEM buffers where they fit, so tile i+1 is converted
//               while the MMAs of tile i run).
// S^T = K Q^T runs on FP8 directly (tcgen05.mma kind::f8f6f4, M = 128 keys):
// the K tile is the A operand exactly as TMA left it in shared memory, and Q
// is the sum of three E4M3 terms per element (row r scaled by 2^e_r so that
// its largest element is at most 448; the terms are the successive
// round-to-nearest residuals, so their sum is the fp16 Q element to within
// half an E4M3 subnormal step). The terms are stacked along N (one MMA of
// N = 3 x rows per 32 head-dim elements reads the K tile once); the softmax
// adds the three columns. O^T = V^T P^T runs on kind::f16 (M = 128 head-dim
// elements, N = rows). Rows are padded to 32/48/64.
// The tensor pipe costs about the same per MMA instruction for any N up to
// ~144 at these shapes, so the instruction count, not the FLOPs, is what
// the MMA schedule minimises.
// Online softmax: every row keeps a reference maximum m; p is formed against
// it in one pass. A tile whose logits exceed m by more than kRescaleLog2
// triggers an exact update (the tile's row maxima are reduced across the 128
// keys, its first-pass terms are taken back out of the fp32 row sums, the
// sums and the O^T accumulators are rescaled and the tile is redone); the
// first tile goes straight to the update. Every wait is an mbarrier wait
// with a time limit, so every path of every role ends; TMEM is freed by the
// MMA warp once the softmax warps, its last readers, have signalled.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <math_constants.h>
#include <stdint.h>

#include "device_utils.cuh"
#include "frag_layout.h"
#include "mask_span.h"
#include "pfkv_internal.h"
#include "verify_layout.h"

namespace pfkv {

constexpr float kRescaleLog2 = 8.f;
// Reference maximum of a row that has seen no visible key yet: finite, so that logit minus
// reference is +1e30 for a visible key (forcing an update) and -inf for a masked one (p = 0).
constexpr float kNoRef = -1e30f;
constexpr int kQTerms = 3;
constexpr int kSoftmaxWarps = 8;
constexpr int kVerifyWarps = 14;

template <int D, int NMAX_>
struct VerifyShape {
  static constexpr int KT = 128;                         // keys per tile (MMA M)
  static constexpr int NBOX = D / kBoxBytes;             // 128-byte boxes per FP8 key row
  static constexpr int SUB = KT * kBoxBytes;             // one box column of a tile (16 KB)
  static constexpr int KV_TILE = NBOX * SUB;             // K (or V) bytes per tile
  static constexpr int NMAX = NMAX_;                     // padded query rows (MMA N): 32, 48 or 64
  static constexpr int HN = NMAX / 2;                    // rows per softmax warp
  static constexpr int NQ = kQTerms * NMAX;               // B rows of S^T: term t of row r is row t*NMAX + r
  static constexpr int Q_BLK = NQ * 128;                 // one 128-dim block of the stacked Q terms
  static constexpr int Q_BYTES = NBOX * Q_BLK;
  static constexpr int PT_BYTES = (KT / 64) * NMAX * 128;  // one P^T buffer (fp16, K-major, 64-key blocks)
  static constexpr int MT = D / 128;                     // O^T M-tiles
  static constexpr int TMEM_COLS = 512;
  // S^T accumulators: up to 48 rows the three Q terms are stacked along N (one MMA of N = 3 x
  // rows per 32 head-dim elements; the softmax adds the three column groups); at 64 rows terms 0
  // and 1 are stacked (one MMA of N = 2 x rows) and term 2 accumulates onto term 1's columns (one
  // MMA of N = rows): two column groups, which leave room for two V^T operands
  static constexpr bool TWO_S = (NMAX == 64);
  static constexpr int NS_COLS = TWO_S ? 2 * NMAX : NQ;
  static constexpr int COL_S = 0;                        // NS_COLS: S^T
  static constexpr int COL_O = NS_COLS;                  // MT x NMAX: O^T
  static constexpr int COL_AV = ((COL_O + MT * NMAX + 31) / 32) * 32;  // NAV x AV_COLS: V^T operands
  static constexpr int AV_COLS = MT * KT / 2;            // one V^T operand (fp16 pairs)
  static constexpr int NAV = COL_AV + 2 * AV_COLS <= TMEM_COLS ? 2 : 1;
  static_assert(COL_AV + NAV * AV_COLS <= TMEM_COLS, "TMEM budget");
  // The V^T operands are written and consumed in units of UK keys, in two buffers of UNIT_COLS
  // columns (M-tile mt of a unit at column mt * UK / 2): whole 128-key tiles where two fit, 64-key
  // halves where TMEM holds a single 128-key operand (64 rows at D = 256), so that the converter
  // always writes one buffer while the O^T MMAs read the other.
  static constexpr int UPT = NAV == 2 ? 1 : 2;  // conversion units per tile
  static constexpr int UK = KT / UPT;           // keys per unit
  static constexpr int UNIT_COLS = MT * UK / 2;
  static constexpr int NHB = 2;                 // unit buffers
  static_assert(NQ <= 256, "MMA N");
  static_assert(HN % 8 == 0, "softmax rows come in TMEM loads of 8 columns");
  // misc: m_ref, alpha, sc2r, rscale, wred[4], lsum[4], m_use, thr, dx (NMAX floats each),
  // out_row (NMAX ints), vote flags, TMEM slot, barriers
  static constexpr int MISC_WORDS = 16 * NMAX;
  static constexpr int MISC_BYTES = MISC_WORDS * 4 + 64 + 32 * 8;
  static constexpr int kSmemLimit = 227 * 1024;
  static constexpr int FIT = (kSmemLimit - 1024 - Q_BYTES - 2 * PT_BYTES - MISC_BYTES) / KV_TILE;
  static constexpr int NK = FIT / 2 > 4 ? 4 : FIT / 2;
  static constexpr int NV = FIT - NK > 4 ? 4 : FIT - NK;
  static_assert(NK >= 2 && NV >= 2, "shared memory budget");
  static_assert(2 * NK + 2 * NV + 12 <= 32, "mbarrier slots");
  // shared memory map (offsets from the 1 KB-aligned base)
  static constexpr int OFF_KRING = 0;
  static constexpr int OFF_VRING = OFF_KRING + NK * KV_TILE;
  static constexpr int OFF_Q = OFF_VRING + NV * KV_TILE;
  static constexpr int OFF_PT = OFF_Q + Q_BYTES;  // 2 buffers
  static constexpr int OFF_MISC = OFF_PT + 2 * PT_BYTES;
  static constexpr int SMEM = OFF_MISC + MISC_BYTES;
};

__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t saddr) {
  // K-major operand, 128-byte swizzle, 8-row groups 1024 bytes apart
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFF);
  d |= static_cast<uint64_t>(1) << 16;
  d |= static_cast<uint64_t>(1024 >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// M = 128, N = n, f16 x f16 -> f32, both operands K-major.
__device__ __forceinline__ uint32_t umma_idesc_f16(int n) {
  return (1u << 4) | (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(128 >> 4) << 24);
}

// M = 128, N = n, A: FP8 codes (afmt 0 = E4M3, 1 = E5M2), B: E4M3, f32 accumulators, both K-major.
__device__ __forceinline__ uint32_t umma_idesc_f8(int n, uint32_t afmt) {
  return (1u << 4) | (afmt << 7) | (0u << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
         (static_cast<uint32_t>(128 >> 4) << 24);
}

// D (TMEM) (+)= A (TMEM) * B (shared memory), f16 operands
__device__ __forceinline__ void umma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate));
}

// D (TMEM) (+)= A (shared memory) * B (shared memory), FP8 operands
__device__ __forceinline__ void umma_ss_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate));
}

__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}

__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&v)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(v[0]),
               "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
               : "memory");
}

__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&v)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7])
               : "r"(taddr)
               : "memory");
}

__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

template <bool B>
struct BoolTag {
  static constexpr bool value = B;
};

__device__ __forceinline__ void st_shared_u16(uint32_t addr, uint32_t low16) {
  asm volatile("st.shared.b16 [%0], %1;" ::"r"(addr), "h"(static_cast<unsigned short>(low16)) : "memory");
}

// two FP8 codes (low byte -> low half) to an fp16 pair
template <int KV>
__device__ __forceinline__ uint32_t fp8x2_to_f16x2(uint32_t two) {
  if constexpr (KV == kKvE4m3) {
    return e4m3x2_to_f16x2(two);
  } else {
    return __byte_perm(two, 0u, 0x1404);  // [0, b0, 0, b1]
  }
}

// Exponent e with 2^e * mx <= 448 (the largest E4M3 value, 1.75 * 2^8) and 2^(e+1) * mx > 448,
// for a finite mx > 0; 0 otherwise. Exact: read off the bits of mx.
__device__ __forceinline__ int e4m3_row_exponent(float mx) {
  const uint32_t u = __float_as_uint(mx);
  const int be = static_cast<int>((u >> 23) & 0xFF);
  if (!(mx > 0.f) || be == 0xFF) return 0;
  if (be == 0) return 0;  // below the fp32 normal range: cannot come from an fp16 input
  const int E = be - 127;
  const uint32_t frac = u & 0x7FFFFF;  // mantissa bits of 1.f
  return (frac <= 0x600000u) ? 8 - E : 7 - E;  // 1.f <= 1.75 ?
}

// x0, x1 (exactly representable sums of at most three E4M3 values once scaled) as three
// successive round-to-nearest E4M3 residual terms; term k of the pair in the low/high byte of t[k].
__device__ __forceinline__ void split3_e4m3(float x0, float x1, uint32_t (&t)[kQTerms]) {
#pragma unroll
  for (int k = 0; k < kQTerms; ++k) {
    const __nv_fp8x2_storage_t c = __nv_cvt_float2_to_fp8x2(make_float2(x0, x1), __NV_SATFINITE, __NV_E4M3);
    t[k] = c;
    const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(c, __NV_E4M3);
    const float2 back = __half22float2(*reinterpret_cast<const __half2*>(&hr));
    x0 -= back.x;  // exact: the residual is a multiple of the input's quantum
    x1 -= back.y;
  }
}

// 14 warps: the busiest SM sub-partition holds 4 of them, which caps a thread at 128 registers
template <int D, int KV, int NMAX_>
__global__ void __launch_bounds__(kVerifyWarps * 32, 1)
    verify_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                  const DecodeParams p) {
  using S = VerifyShape<D, NMAX_>;
  constexpr int KT = S::KT, NBOX = S::NBOX, NK = S::NK, NV = S::NV, NMAX = S::NMAX, MT = S::MT, HN = S::HN;
  extern __shared__ unsigned char smem_raw[];
  // 1 KB-aligned base, formed by pointer arithmetic on the shared array so that every pointer
  // derived from it stays a shared-memory pointer (32-bit shared loads and stores)
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);

  const int split = blockIdx.x, b = blockIdx.z;
  // KV head major (CTAs running together share one head's keys in L2), longest slabs first
  const int kvh = blockIdx.y / p.num_slabs;
  const int slab = p.num_slabs - 1 - static_cast<int>(blockIdx.y) % p.num_slabs;

  // launched with programmatic stream serialisation: wait for the preceding grid first
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // Up to 48 rows the slab's Q rows (fp16) are copied into the P^T buffers, not yet in use, with
  // asynchronous 16-byte copies issued by every thread at once, so that the prologue waits for one
  // memory round trip instead of one per row of each warp (a slab's query tokens do not depend
  // on the sequence length). (The 64-row kernels keep per-warp loads: their register-bound code
  // measured slower with any change to the prologue.)
  constexpr bool QSTAGE = NMAX <= 48;
  if constexpr (QSTAGE) {
    static_assert(NMAX * D * 2 <= 2 * S::PT_BYTES, "Q staging fits the P^T buffers");
    const int ts0q = slab * p.slab_tokens;
    const int rows = (min(ts0q + p.slab_tokens, p.T) - ts0q) * p.G;
    constexpr int CH = D / 8;  // 16-byte chunks per row
    for (int idx = threadIdx.x; idx < rows * CH; idx += blockDim.x) {
      const int r = idx / CH, c = idx - r * CH;
      const int tl = r / p.G, j = r - tl * p.G;
      const __half* src =
          p.q + ((static_cast<size_t>(b) * p.T + ts0q + tl) * p.num_q_heads + kvh * p.G + j) * D + c * 8;
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem + S::OFF_PT + r * (D * 2) + c * 16)),
                   "l"(src)
                   : "memory");
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  }
  int N = p.seq_lens[b];
  {
    const int cap = min(p.max_seq_len, p.max_blocks * p.page_size);
    if (N < 0 || N > cap) {
      if (threadIdx.x == 0 && split == 0 && blockIdx.y == 0) atomicOr(p.err, kDevErrSeqLen);
      N = N < 0 ? 0 : cap;
    }
  }
  const SlabSpan sp = slab_span(N, p.T, slab, p.slab_tokens, p.causal, p.window, KT);
  const int nsplit_b = span_splits(sp, p.split_tokens);
  if (split >= nsplit_b) {
    if constexpr (QSTAGE) asm volatile("cp.async.wait_all;" ::: "memory");  // no copy lands after the CTA left
    return;
  }
  const int R = (sp.ts1 - sp.ts0) * p.G;  // query rows of this slab
  const int t0 = sp.base + split * p.split_tokens;
  const int t1 = sp.hi >= sp.lo ? min(sp.hi + 1, t0 + p.split_tokens) : t0;
  const int ntiles = t1 > t0 ? (t1 - t0 + KT - 1) / KT : 0;

  float* m_ref = reinterpret_cast<float*>(smem + S::OFF_MISC);  // [NMAX] reference max (log2 units)
  float* alpha_s = m_ref + NMAX;                                 // [NMAX] rescale factors
  float* sc2r = alpha_s + NMAX;                                  // [NMAX] logit scale of row r (log2 units)
  float* rscale = sc2r + NMAX;                                   // [NMAX] output scale v_scale / L
  float* wred = rscale + NMAX;                                   // [4][NMAX] per-quadrant maxima
  float* lsum = wred + 4 * NMAX;                                 // [4][NMAX] per-quadrant row sums
  // the reference as the logits use it: m_ref, or 0 while a row has none (kNoRef); and the
  // threshold above which a logit forces an update: kRescaleLog2, or -inf while it has none
  float* m_use = lsum + 4 * NMAX;                                // [NMAX]
  float* thr = m_use + NMAX;                                     // [NMAX]
  float* dx_s = thr + NMAX;                                      // [NMAX] old m_use - new m_use
  int* out_row = reinterpret_cast<int*>(dx_s + NMAX);            // [NMAX] output row of row r
  int* flag = out_row + NMAX;                                    // [3] rescale votes
  uint32_t* tslot = reinterpret_cast<uint32_t*>(flag + 4);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::OFF_MISC + S::MISC_WORDS * 4 + 64);
  uint64_t* kfull = bars;              // [NK] producer -> MMA (K tile landed)
  uint64_t* kempty = kfull + NK;       // [NK] MMA commit: S^T MMAs done reading the K tile
  uint64_t* vfull = kempty + NK;       // [NV] producer -> V converter
  uint64_t* vempty = vfull + NV;       // [NV] V converter -> producer
  uint64_t* av_full = vempty + NV;     // [NHB] V converter -> MMA (V^T unit written)
  uint64_t* av_free = av_full + 2;     // [NHB] MMA commit: O^T MMAs done with a V^T unit
  uint64_t* s_full = av_free + 2;      // MMA commit: S^T ready
  uint64_t* s_free = s_full + 1;       // softmax -> MMA: S^T read into registers
  uint64_t* pt_full = s_free + 1;      // [2] softmax -> MMA: P^T written
  uint64_t* pt_free = pt_full + 2;     // [2] MMA commit: O^T MMAs of the tile done (P^T buffer free)
  uint64_t* swg_bar = pt_free + 2;     // softmax warps' rendezvous (bounded waits, unlike bar.sync)
  uint64_t* tmem_done = swg_bar + 1;   // softmax warps -> MMA warp: last TMEM read done

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tid = threadIdx.x;

  if (tid == 0) {
    for (int s = 0; s < NK; ++s) {
      mbar_init(&kfull[s], 1);
      mbar_init(&kempty[s], 1);
    }
    for (int s = 0; s < NV; ++s) {
      mbar_init(&vfull[s], 1);
      mbar_init(&vempty[s], 4);  // one arrival per V-converter warp
    }
    for (int i = 0; i < S::NHB; ++i) {
      mbar_init(&av_full[i], 4);  // one arrival per V-converter warp
      mbar_init(&av_free[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&pt_full[i], kSoftmaxWarps);
      mbar_init(&pt_free[i], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(s_free, kSoftmaxWarps);
    mbar_init(swg_bar, kSoftmaxWarps);
    mbar_init(tmem_done, kSoftmaxWarps);
    fence_barrier_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tslot)),
                 "r"(S::TMEM_COLS));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  // the pool's scale, or this KV head's
  const float kscale = p.k_scale[kvh * p.scale_stride], vscale = p.v_scale[kvh * p.scale_stride];
  const float sc2 = p.softmax_scale * kscale * 1.4426950408889634f;
  // Q -> three E4M3 terms in shared memory (K-major, 128B swizzle), one warp per row; padded rows zero
  if constexpr (QSTAGE) {
    asm volatile("cp.async.wait_all;" ::: "memory");
    __syncthreads();  // every thread's Q copies have landed
  }
  {
    constexpr int PER_LANE = D / 32;  // 8 (D = 256) or 4 (D = 128) consecutive dims per lane
    for (int r = warp; r < NMAX; r += kVerifyWarps) {
      float x[PER_LANE];
      float mx = 0.f;
      if (r < R) {
        const int tl = r / p.G, j = r - tl * p.G;
        const __half* src = QSTAGE ? reinterpret_cast<const __half*>(smem + S::OFF_PT + r * (D * 2)) + lane * PER_LANE
                                   : p.q + ((static_cast<size_t>(b) * p.T + sp.ts0 + tl) * p.num_q_heads + kvh * p.G + j) * D +
                                         lane * PER_LANE;
        if constexpr (PER_LANE == 8) {
          const uint4 v = *reinterpret_cast<const uint4*>(src);
          const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
            x[2 * i] = f.x;
            x[2 * i + 1] = f.y;
          }
        } else {
          const uint2 v = *reinterpret_cast<const uint2*>(src);
          const uint32_t w[2] = {v.x, v.y};
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
            x[2 * i] = f.x;
            x[2 * i + 1] = f.y;
          }
        }
#pragma unroll
        for (int i = 0; i < PER_LANE; ++i) mx = fmaxf(mx, fabsf(x[i]));
      } else {
#pragma unroll
        for (int i = 0; i < PER_LANE; ++i) x[i] = 0.f;
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      const int e = e4m3_row_exponent(mx);
      const float up = __int_as_float((127 + e) << 23);    // 2^e (e in [-8, 32] for fp16 rows)
      const float down = __int_as_float((127 - e) << 23);  // 2^-e
      if (lane == 0) sc2r[r] = sc2 * down;
      uint32_t tw[kQTerms][PER_LANE / 4];  // per term: PER_LANE codes as 32-bit words
#pragma unroll
      for (int i = 0; i < PER_LANE; i += 4) {
        uint32_t lo[kQTerms], hi[kQTerms];
        split3_e4m3(x[i] * up, x[i + 1] * up, lo);
        split3_e4m3(x[i + 2] * up, x[i + 3] * up, hi);
#pragma unroll
        for (int k = 0; k < kQTerms; ++k) tw[k][i / 4] = (lo[k] & 0xFFFFu) | (hi[k] << 16);
      }
      const int d0 = lane * PER_LANE;
      // term k of row r is B row k * NMAX + r (NMAX is a multiple of 8: same swizzle phase)
      const int off = (d0 >> 7) * S::Q_BLK + r * 128 + (((((d0 & 127) >> 4) ^ r) & 7) << 4) + (d0 & 15);
#pragma unroll
      for (int k = 0; k < kQTerms; ++k) {
        unsigned char* dst = smem + S::OFF_Q + k * NMAX * 128 + off;
        if constexpr (PER_LANE == 8) {
          *reinterpret_cast<uint2*>(dst) = make_uint2(tw[k][0], tw[k][1]);
        } else {
          *reinterpret_cast<uint32_t*>(dst) = tw[k][0];
        }
      }
    }
    for (int i = tid; i < NMAX; i += blockDim.x) {
      m_ref[i] = kNoRef;
      m_use[i] = 0.f;
      thr[i] = -CUDART_INF_F;
    }
    if (tid == 0) flag[0] = flag[1] = flag[2] = 0;
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;
  bool alive = true;

  if (warp == 0) {
    // ---------------------------------------------------------------- producers (lanes 0 and 1)
    // Lane 0 copies the K tiles, lane 1 the V tiles, each into its own ring and each sleeping
    // in its own slot waits: the two divergent paths of the warp progress independently, so a
    // V copy never waits behind a K slot (freed by the S^T MMAs) nor the reverse. Each lane
    // reads the block-table entries it needs itself (a page id is reused while its page lasts).
    if (ntiles > 0 && lane < 2) {
      const int which = lane;  // 0: K, 1: V
      const CUtensorMap* map = which == 0 ? &tmk : &tmv;
      prefetch_tensormap(map);
      uint64_t* fullb = which == 0 ? kfull : vfull;
      uint64_t* emptyb = which == 0 ? kempty : vempty;
      const int depth = which == 0 ? NK : NV;
      unsigned char* ring = smem + (which == 0 ? S::OFF_KRING : S::OFF_VRING);
      const int P = p.page_size;
      const int* bt = p.block_table + static_cast<size_t>(b) * p.max_blocks;
      int cur_page = -1, cur_id = 0;
      auto page_id = [&](int pidx) -> int {
        if (pidx != cur_page) {
          cur_page = pidx;
          cur_id = bt[pidx];
          if (static_cast<unsigned>(cur_id) >= static_cast<unsigned>(p.num_blocks)) {
            atomicOr(p.err, kDevErrBlockId);
            cur_id = 0;
          }
        }
        return cur_id;
      };
      int it = 0;
      for (; it < ntiles; ++it) {
        const int tile_start = t0 + it * KT;
        const int valid = min(KT, t1 - tile_start);
        // rows of the tile's 64-row boxes (P >= 64) or pages (P < 64); at most 8
        int rows[8], box_rows, nbox_rows;
        if (P >= kTileKeys) {
          nbox_rows = (valid + kTileKeys - 1) / kTileKeys;
          box_rows = kTileKeys;
#pragma unroll
          for (int hf = 0; hf < 8; ++hf) {
            const int key = tile_start + hf * kTileKeys;
            rows[hf] = 0;
            if (hf < 2 && hf < nbox_rows)
              rows[hf] = (page_id(key >> p.page_shift) * p.num_kv_heads + kvh) * P + (key & (P - 1));
          }
        } else {
          nbox_rows = (valid + P - 1) >> p.page_shift;
          box_rows = P;
          const int pfirst = tile_start >> p.page_shift;
#pragma unroll
          for (int pg = 0; pg < 8; ++pg) {
            rows[pg] = 0;
            if (pg < nbox_rows) {
              int id = bt[pfirst + pg];  // independent loads: one round trip per tile
              if (static_cast<unsigned>(id) >= static_cast<unsigned>(p.num_blocks)) {
                atomicOr(p.err, kDevErrBlockId);
                id = 0;
              }
              rows[pg] = (id * p.num_kv_heads + kvh) * P;
            }
          }
        }
        // slot of tile it-depth released (its previous phase, of tile it-2*depth, was waited
        // for by this lane; the next one needs this lane's own copy of tile it)
        if (it >= depth && !mbar_wait(&emptyb[it % depth], ((it / depth) - 1) & 1)) {
          atomicOr(p.err, kDevErrTimeout);
          break;
        }
        unsigned char* dst = ring + (it % depth) * S::KV_TILE;
        mbar_arrive_expect_tx(&fullb[it % depth], NBOX * nbox_rows * box_rows * kBoxBytes);
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          if (r < nbox_rows) {
#pragma unroll
            for (int bx = 0; bx < NBOX; ++bx)
              tma_load_2d(dst + bx * S::SUB + r * box_rows * kBoxBytes, map, &fullb[it % depth], bx * kBoxBytes,
                          rows[r]);
          }
        }
      }
      // do not leave while copies may still land in this CTA's shared memory
      for (int jt = max(0, it - depth); jt < it; ++jt)
        if (!mbar_wait(&fullb[jt % depth], (jt / depth) & 1)) {
          atomicOr(p.err, kDevErrTimeout);
          break;
        }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0 && ntiles > 0) {
      constexpr int NHB = S::NHB;
      const uint32_t idesc_qk = umma_idesc_f8(S::NS_COLS, KV == kKvE4m3 ? 0u : 1u);
      const uint32_t idesc_qk1 = umma_idesc_f8(NMAX, KV == kKvE4m3 ? 0u : 1u);  // term 2 alone (64 rows)
      const uint32_t idesc_pv = umma_idesc_f16(NMAX);
      // descriptors of the operands' first k-slices; a k-step adds its byte offset / 16 to the
      // start-address field (every operand lies below 256 KB, so the 14-bit field never carries)
      const uint64_t q_desc = umma_desc_sw128(smem_u32(smem + S::OFF_Q));
      const uint64_t k_desc = umma_desc_sw128(smem_u32(smem + S::OFF_KRING));
      const uint64_t pt_desc = umma_desc_sw128(smem_u32(smem + S::OFF_PT));
      // With one S^T buffer the issue order is fixed, and the tensor pipe executes in issue
      // order: S^T(0), S^T(1), then per tile i, once P^T(i) and V^T(i) are written: S^T(i+2)
      // (its K tile landed and the softmax read S^T(i+1) out, which it does right after
      // finishing tile i), then O^T(i). S^T of the tile after next thus never queues behind a
      // tile's 16 O^T MMAs; O^T(i) is only needed two tiles later (P^T and V^T are double
      // buffered). Blocking waits wake as soon as the phase completes. Each parity wait is
      // sound: this thread saw the previous phase of that barrier, and its next phase needs an
      // MMA this thread has not issued yet.
      // (Issuing the O^T MMAs from a second warp was measured slower: that warp's sub-partition
      // also runs a V converter, which then fell behind.)
      bool ok = true;
      auto issue_s = [&](int sn) {
        const uint64_t ka = k_desc + static_cast<uint64_t>(((sn % NK) * S::KV_TILE) >> 4);
#pragma unroll
        for (int ks = 0; ks < D / 32; ++ks) {  // 32 FP8 dims = 32 bytes of a swizzled row per MMA
          const uint32_t koff = ((ks >> 2) * S::SUB + (ks & 3) * 32) >> 4;
          const uint32_t qoff = ((ks >> 2) * S::Q_BLK + (ks & 3) * 32) >> 4;
          umma_ss_f8(tbase + S::COL_S, ka + koff, q_desc + qoff, idesc_qk, ks > 0 ? 1u : 0u);
          if constexpr (S::TWO_S) {
            // term 2 of every row (B rows 2 * NMAX + r) onto term 1's columns
            umma_ss_f8(tbase + S::COL_S + NMAX, ka + koff, q_desc + qoff + static_cast<uint32_t>((2 * NMAX * 128) >> 4),
                       idesc_qk1, 1u);
          }
        }
        umma_commit(s_full);
        umma_commit(&kempty[sn % NK]);
      };
      ok = mbar_wait(&kfull[0], 0);
      if (ok) {
        tc_fence_after();
        issue_s(0);
      }
      if (ok && ntiles > 1) {
        ok = mbar_wait(&kfull[1 % NK], (1 / NK) & 1) && mbar_wait(s_free, 0);
        if (ok) {
          tc_fence_after();
          issue_s(1);
        }
      }
      constexpr int UPT = S::UPT;
      for (int on = 0; on < ntiles && ok; ++on) {
        // conversion units UPT*on .. UPT*on + UPT-1 of tile on; each parity wait on a unit buffer
        // is sound for the same reason as above (units u - NHB, u, u + NHB of a buffer are waited
        // for in order)
        ok = mbar_wait(&av_full[(UPT * on) % NHB], ((UPT * on) / NHB) & 1) && mbar_wait(&pt_full[on & 1], (on >> 1) & 1);
        if (!ok) break;
        const int sn = on + 2;
        if (sn < ntiles) {
          ok = mbar_wait(&kfull[sn % NK], (sn / NK) & 1) && mbar_wait(s_free, (sn - 1) & 1);
          if (!ok) break;
          tc_fence_after();
          issue_s(sn);
        }
        tc_fence_after();
        const uint64_t pt = pt_desc + static_cast<uint64_t>(((on & 1) * S::PT_BYTES) >> 4);
#pragma unroll
        for (int h = 0; h < UPT; ++h) {
          const int u = UPT * on + h;
          if (h > 0) {
            ok = mbar_wait(&av_full[u % NHB], (u / NHB) & 1);
            if (!ok) break;
            tc_fence_after();
          }
          const uint32_t av = tbase + S::COL_AV + (u % NHB) * S::UNIT_COLS;
#pragma unroll
          for (int kh = 0; kh < S::UK / 16; ++kh) {
            const int ks = h * (S::UK / 16) + kh;  // 16-key step of the tile
            const uint32_t poff = ((ks >> 2) * NMAX * 128 + (ks & 3) * 32) >> 4;
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
              umma_ts(tbase + S::COL_O + mt * NMAX, av + mt * (S::UK / 2) + 8 * kh, pt + poff, idesc_pv,
                      (on > 0 || ks > 0) ? 1u : 0u);
          }
          umma_commit(&av_free[u % NHB]);
        }
        if (!ok) break;
        umma_commit(&pt_free[on & 1]);
      }
      if (!ok) atomicOr(p.err, kDevErrTimeout);
    }
    __syncwarp();
  } else if (warp >= 10) {
    // ---------------------------------------------------------------- V converter (warps 10-13)
    // TMEM lane L of O^T M-tile mt holds head-dim element 2L + mt (D = 256) or L (D = 128);
    // its columns hold the tile's keys as fp16 pairs.
    const int q = warp & 3;
    const int lane_row = 32 * q + lane;
    const uint32_t tq = tbase + (static_cast<uint32_t>(32 * q) << 16);
    const int dim = (D == 256) ? 2 * lane_row : lane_row;
    const int vbx = dim >> 7, vbyte = dim & 127;
    // byte offset of this thread's element(s) in key rows j = 0..7 of an 8-row group
    int voff[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) voff[j] = vbx * S::SUB + swz_offset(j, vbyte >> 4) + (vbyte & 15);
    for (int it = 0; it < ntiles && alive; ++it) {
      const int s = it % NV;
      if (!mbar_wait(&vfull[s], (it / NV) & 1)) {
        alive = false;
        break;
      }
      const unsigned char* Vs = smem + S::OFF_VRING + s * S::KV_TILE;
      const int valid = min(KT, t1 - (t0 + it * KT));
      uint32_t av = 0;
      // a full tile and the range's last, partial one take separate copies of the loop, so that
      // the full tiles carry no per-key range checks; keys k_lo .. k_lo + UK - 1 go to one buffer
      auto convert_unit = [&](auto tail_tag, int k_lo) {
        constexpr bool kTail = decltype(tail_tag)::value;
#pragma unroll 1
        for (int k0 = k_lo; k0 < k_lo + S::UK; k0 += 32) {
          const unsigned char* vrow = Vs + k0 * kBoxBytes;  // rows k0.. of the tile (k0 % 8 == 0)
          uint32_t v0[16], v1[16];
#pragma unroll
          for (int kk = 0; kk < 32; kk += 2) {
            const int oa = voff[kk & 7] + ((kk >> 3) << 10);
            const int ob = voff[(kk + 1) & 7] + ((kk >> 3) << 10);
            uint32_t wa, wb;
            if constexpr (D == 256) {
              wa = *reinterpret_cast<const uint16_t*>(vrow + oa);  // dims 2L, 2L+1 of key k0+kk
              wb = *reinterpret_cast<const uint16_t*>(vrow + ob);
            } else {
              wa = vrow[oa];
              wb = vrow[ob];
            }
            if constexpr (kTail) {  // stale bytes past the range end must not reach the MMA
              if (k0 + kk >= valid) wa = 0u;
              if (k0 + kk + 1 >= valid) wb = 0u;
            }
            if constexpr (KV == kKvE5m2 && D == 256) {
              // an E5M2 code is the high byte of the fp16 with the same value: the fp16 pairs
              // (key k, key k+1) of dims 2L and 2L+1 are byte moves, bytes 2-3 of wa being zero
              v0[kk >> 1] = __byte_perm(wa, wb, 0x4202);  // [0, a.b0, 0, b.b0]
              v1[kk >> 1] = __byte_perm(wa, wb, 0x5212);  // [0, a.b1, 0, b.b1]
            } else {
              const uint32_t X = __byte_perm(wa, wb, 0x5140);  // [a.b0, b.b0, a.b1, b.b1]
              v0[kk >> 1] = fp8x2_to_f16x2<KV>(X);
              v1[kk >> 1] = fp8x2_to_f16x2<KV>(X >> 16);
            }
          }
          tmem_st16(av + ((k0 - k_lo) >> 1), v0);
          if constexpr (MT == 2) tmem_st16(av + S::UK / 2 + ((k0 - k_lo) >> 1), v1);
        }
      };
      for (int h = 0; h < S::UPT; ++h) {
        const int u = S::UPT * it + h;  // conversion unit h of tile it
        // unit buffer u % NHB is free once the O^T MMAs of unit u - NHB are done (sound: this
        // thread saw that barrier's previous phase, of unit u - 2*NHB, before converting u - NHB)
        if (u >= S::NHB && !mbar_wait(&av_free[u % S::NHB], ((u / S::NHB) - 1) & 1)) {
          alive = false;
          break;
        }
        tc_fence_after();
        av = tq + S::COL_AV + (u % S::NHB) * S::UNIT_COLS;
        if (valid < KT) {
          convert_unit(BoolTag<true>{}, h * S::UK);
        } else {
          convert_unit(BoolTag<false>{}, h * S::UK);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&av_full[u % S::NHB]);
      }
      if (!alive) break;
      if (lane == 0) mbar_arrive(&vempty[s]);
    }
    if (!alive && lane == 0) atomicOr(p.err, kDevErrTimeout);
  } else {
    // ---------------------------------------------------------------- softmax + epilogue (warps 2-9)
    const int sw = warp - 2;           // 0..7 within the softmax warps
    const int q = warp & 3;            // TMEM lane quadrant
    const int rbase = (sw >> 2) * HN;  // this warp's rows: rbase .. rbase + HN - 1
    const int key_lane = 32 * q + lane;
    const int sidx = sw * 32 + lane;   // 0..255: the row owned in the per-row steps
    const uint32_t tq = tbase + (static_cast<uint32_t>(32 * q) << 16);
    // shared addresses of this thread's P^T element (its key) in rows rbase + 8i + j of buffer 0:
    // rbase and 8i are multiples of 8, so row & 7 = j and the swizzle depends on j alone
    uint32_t pta[8];
    {
      const int kk = key_lane & 63;
      const uint32_t pt0 = smem_u32(smem + S::OFF_PT + (key_lane >> 6) * NMAX * 128);
#pragma unroll
      for (int j = 0; j < 8; ++j) pta[j] = pt0 + static_cast<uint32_t>(sw128_elem(rbase + j, kk));
    }
    uint32_t swg_phase = 0;
    // the softmax warps meet; a wait that runs out marks the CTA's work as failed
    auto swg_sync = [&]() {
      __syncwarp();
      if (lane == 0) mbar_arrive(swg_bar);
      if (!mbar_wait(swg_bar, swg_phase & 1)) alive = false;
      ++swg_phase;
    };
    float l_part[HN];  // this thread's (key lane's) share of its rows' sums, fp32
#pragma unroll
    for (int r = 0; r < HN; ++r) l_part[r] = 0.f;
    // Row r of the slab is query token ts0 + r / G at position pos0 + r / G; it sees key kp iff
    // r >= rmin(kp) (causal: kp is not after it) and r < rmax(kp) (window: kp is less than W
    // positions before it). Every row sees [lo_all, hi_all] (the slab's first token's upper and
    // last token's lower bound).
    const int pos0 = N - p.T + sp.ts0;
    const int hi_all = key_hi(N, p.T, sp.ts0, p.causal);
    const int lo_all = key_lo(N, p.T, sp.ts1 - 1, p.window);
    auto load8 = [](const float* src, float (&m)[8]) {
      const float4 a = *reinterpret_cast<const float4*>(src);
      const float4 c = *reinterpret_cast<const float4*>(src + 4);
      m[0] = a.x;
      m[1] = a.y;
      m[2] = a.z;
      m[3] = a.w;
      m[4] = c.x;
      m[5] = c.y;
      m[6] = c.z;
      m[7] = c.w;
    };
    // 2^x for x = s - m_use (base-2 units), capped so that a logit that outgrew its reference
    // stays finite (the tile is then redone). A row without a reference yet (m_use = 0) has the
    // threshold -inf, so any visible key of it forces the update, whose factor for that row is
    // 2^(kNoRef - m) = 0; the tile is then redone against the new reference.
    auto pexp = [](float x) -> float { return fast_exp2(fminf(x, 15.f)); };
    for (int it = 0; it < ntiles && alive; ++it) {
      const int sb = it & 1;
      if (!mbar_wait(s_full, it & 1)) {
        alive = false;
        break;
      }
      tc_fence_after();
      const int tile_start = t0 + it * KT;
      const int kp = tile_start + key_lane;  // absolute key position
      // The rows that see this key are rmin <= r < rmax: rows r >= G * (kp - pos0) have kp at or
      // before their position, rows r < G * (kp + W - pos0) have it within their window (clamped
      // to [0, 64]: a slab has at most 64 rows); none past the range end. Padding rows follow the
      // same rule (they are never written out; a row that sees nothing gets p = 0).
      const long long dk = static_cast<long long>(kp) - pos0;
      const int rmin = p.causal ? static_cast<int>(max(0LL, min(64LL, p.G * dk))) : 0;
      const int rmax = kp >= t1 ? 0 : (p.window > 0 ? static_cast<int>(max(0LL, min(64LL, p.G * (dk + p.window)))) : 64);
      const bool all_vis =  // CTA-uniform: every row sees every key of the tile
          (tile_start + KT <= t1) && (tile_start + KT - 1 <= hi_all) && (tile_start >= lo_all);
      // this key's logits of rows rbase .. rbase+HN-1 (sum of the three Q-term columns) less
      // the rows' references, x = s - m_use in base-2 units, -inf where masked; then the S^T
      // buffer goes back to the MMA warp. And whether any x exceeds its row's threshold.
      float x[HN];
      bool exceed = false;
#pragma unroll
      for (int c = 0; c < HN; c += 8) {
        uint32_t v0[8], v1[8], v2[8];
        float sc[8], mu[8], th[8];
        const uint32_t col = tq + S::COL_S + rbase + c;
        tmem_ld8(col, v0);
        tmem_ld8(col + NMAX, v1);
        if constexpr (!S::TWO_S) tmem_ld8(col + 2 * NMAX, v2);
        load8(sc2r + rbase + c, sc);
        load8(m_use + rbase + c, mu);
        load8(thr + rbase + c, th);
        tmem_wait_ld();
        if (all_vis) {  // CTA-uniform: every row sees every key of the tile
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float raw = S::TWO_S ? __uint_as_float(v0[j]) + __uint_as_float(v1[j])
                                       : (__uint_as_float(v0[j]) + __uint_as_float(v1[j])) + __uint_as_float(v2[j]);
            x[c + j] = fmaf(raw, sc[j], -mu[j]);
            exceed |= x[c + j] > th[j];
          }
        } else {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int r = rbase + c + j;
            const bool vis = r >= rmin && r < rmax;
            const float raw = S::TWO_S ? __uint_as_float(v0[j]) + __uint_as_float(v1[j])
                                       : (__uint_as_float(v0[j]) + __uint_as_float(v1[j])) + __uint_as_float(v2[j]);
            x[c + j] = vis ? fmaf(raw, sc[j], -mu[j]) : -CUDART_INF_F;
            exceed |= x[c + j] > th[j];
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(s_free);
      // Vote on the update now and meet after the pass (which assumes no update): the
      // rendezvous then costs nothing unless the warps are far apart. (Three rotating flags:
      // the one cleared below, of tile it-1, was read by every thread before it voted on this
      // tile, and is voted on again only after the next rendezvous, which the clearing thread
      // must reach first.)
      if (it > 0) {
        if (__any_sync(0xffffffffu, exceed) && lane == 0) atomicOr(&flag[it % 3], 1);
        __syncwarp();
        if (lane == 0) mbar_arrive(swg_bar);
      }
      // P^T buffer sb is free once the O^T MMAs of tile it-2 are done (sound: this thread saw
      // that barrier's previous phase, of tile it-4, at tile it-2)
      if (it >= 2 && !mbar_wait(&pt_free[sb], ((it >> 1) - 1) & 1)) {
        alive = false;
        break;
      }
      const uint32_t ptb = sb * S::PT_BYTES;  // P^T buffer sb
      bool update = (it == 0);  // the first tile has no references yet
      bool did_pass = false;
#pragma unroll 1
      for (int round = 0; round < 2; ++round) {
        if (update) {
          // exact update: this tile's row maxima over its 128 keys; this tile's first-pass
          // terms (same formula, same values) taken back out of the row sums
#pragma unroll
          for (int c = 0; c < HN; c += 8) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              float mx = x[c + j];
#pragma unroll
              for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
              if (lane == 0) wred[q * NMAX + rbase + c + j] = mx;
              if (did_pass) l_part[c + j] -= pexp(x[c + j]);
            }
          }
          swg_sync();
          if (sidx < NMAX) {
            const int r = sidx;
            const float mu_old = m_use[r];
            // the tile's row maximum of s (x + m_use: -inf if every key is masked)
            const float mt =
                fmaxf(fmaxf(wred[r], wred[NMAX + r]), fmaxf(wred[2 * NMAX + r], wred[3 * NMAX + r])) + mu_old;
            const float mo = m_ref[r];
            const float mn = fmaxf(mo, mt);
            // the reference only moves up; rows with nothing visible so far keep kNoRef
            const bool none = !(mn > kNoRef);
            const float mu_new = none ? 0.f : mn;
            alpha_s[r] = fast_exp2(mo - mn);
            m_ref[r] = mn;
            m_use[r] = mu_new;
            thr[r] = none ? -CUDART_INF_F : kRescaleLog2;
            dx_s[r] = mu_old - mu_new;
          }
          swg_sync();
#pragma unroll
          for (int c = 0; c < HN; c += 8) {
            float a[8], d[8];
            load8(alpha_s + rbase + c, a);
            load8(dx_s + rbase + c, d);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              l_part[c + j] *= a[j];
              x[c + j] += d[j];  // against the new reference (-inf stays -inf)
            }
          }
          if (it > 0) {
            // rescale the O^T columns once the previous tile's MMAs are done (sound: this
            // thread saw that barrier's previous phase, of tile it-3, at the top of tile it-1)
            if (!mbar_wait(&pt_free[(it - 1) & 1], ((it - 1) >> 1) & 1)) alive = false;
            tc_fence_after();
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
              for (int c = 0; c < HN; c += 8) {
                uint32_t v[8];
                float a[8];
                const uint32_t addr = tq + S::COL_O + mt * NMAX + rbase + c;
                tmem_ld8(addr, v);
                load8(alpha_s + rbase + c, a);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 8; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) * a[j]);
                tmem_st8(addr, v);
              }
            }
            tmem_wait_st();
          }
        }
        // one pass: P^T and the row sums against the current references
#pragma unroll
        for (int c = 0; c < HN; c += 8) {
#pragma unroll
          for (int j = 0; j < 8; j += 2) {
            const float p0 = pexp(x[c + j]), p1 = pexp(x[c + j + 1]);
            l_part[c + j] += p0;
            l_part[c + j + 1] += p1;
            const __half2 h = __floats2half2_rn(p0, p1);
            const uint32_t hw = *reinterpret_cast<const uint32_t*>(&h);
            st_shared_u16(pta[j] + ptb + c * 128, hw);
            st_shared_u16(pta[j + 1] + ptb + c * 128, hw >> 16);
          }
        }
        did_pass = true;
        if (update) break;  // after an update no logit exceeds its reference
        if (!mbar_wait(swg_bar, swg_phase & 1)) alive = false;  // the vote cast before the pass
        ++swg_phase;
        update = flag[it % 3] != 0;
        if (sidx == 0) flag[(it + 2) % 3] = 0;
        if (!update) break;
      }
      if (!alive) break;
      tc_fence_before();
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(&pt_full[sb]);
    }
    if (!alive && lane == 0) atomicOr(p.err, kDevErrTimeout);

    // ------------------------------------------------------------ epilogue
    // All MMAs done: pt_free of the last tile's buffer (sound: this thread saw its previous
    // phase, of tile ntiles-3) is committed after every earlier MMA.
    if (ntiles > 0 && alive && !mbar_wait(&pt_free[(ntiles - 1) & 1], ((ntiles - 1) >> 1) & 1)) alive = false;
    tc_fence_after();
    // row sums over the 128 keys
#pragma unroll
    for (int j = 0; j < HN; ++j) {
      float v = l_part[j];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
      if (lane == 0) lsum[q * NMAX + rbase + j] = v;
    }
    swg_sync();
    const bool final_out = (nsplit_b == 1);
    if (sidx < R) {  // per row: output scale, output row, LSE
      const int r = sidx;
      const float L = lsum[r] + lsum[NMAX + r] + lsum[2 * NMAX + r] + lsum[3 * NMAX + r];
      const float M = m_ref[r];
      const bool has = alive && ntiles > 0 && (M != kNoRef) && (L > 0.f);
      const int tl = r / p.G, jj = r - tl * p.G;
      const int grow = (b * p.T + sp.ts0 + tl) * p.num_q_heads + kvh * p.G + jj;
      rscale[r] = has ? vscale / L : 0.f;
      out_row[r] = grow;
      const float lse_val = has ? (M + log2f(L)) * 0.6931471805599453f : -CUDART_INF_F;
      if (final_out) {
        p.lse[grow] = lse_val;
      } else {
        p.lse_part[static_cast<size_t>(grow) * p.num_splits + split] = lse_val;
      }
    }
    swg_sync();
    // this thread's TMEM lane = head-dim element(s) of O^T; its rows: rbase .. rbase + HN - 1
#pragma unroll
    for (int c = 0; c < HN; c += 8) {
      if (rbase + c >= R) break;
      uint32_t v[MT][8];
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        if (ntiles > 0) {
          tmem_ld8(tq + S::COL_O + mt * NMAX + rbase + c, v[mt]);
        } else {
#pragma unroll
          for (int j = 0; j < 8; ++j) v[mt][j] = 0u;
        }
      }
      if (ntiles > 0) tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int r = rbase + c + j;
        if (r >= R) break;
        const float sc = rscale[r];
        const size_t grow = static_cast<size_t>(out_row[r]);
        if constexpr (MT == 2) {
          const float o0 = sc != 0.f ? __uint_as_float(v[0][j]) * sc : 0.f;
          const float o1 = sc != 0.f ? __uint_as_float(v[1][j]) * sc : 0.f;
          const int d0 = 2 * key_lane;
          if (final_out) {
            *reinterpret_cast<__half2*>(p.out + grow * D + d0) = __floats2half2_rn(o0, o1);
          } else {
            *reinterpret_cast<float2*>(p.o_part + (grow * p.num_splits + split) * D + d0) = make_float2(o0, o1);
          }
        } else {
          const float o0 = sc != 0.f ? __uint_as_float(v[0][j]) * sc : 0.f;
          if (final_out) {
            p.out[grow * D + key_lane] = __float2half_rn(o0);
          } else {
            p.o_part[(grow * p.num_splits + split) * D + key_lane] = o0;
          }
        }
      }
    }
    // last TMEM access of this warp done: the MMA warp may free TMEM
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(tmem_done);
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  }
  if (warp == 1) {
    // Free TMEM once the softmax warps (the last readers; the MMAs they waited for and the V
    // converters' stores precede their reads) are done. Every softmax path arrives once, and
    // their own waits are bounded, so this wait ends; a few limits' worth covers them.
    bool got = false;
    for (int k = 0; k < 4 && !got; ++k) got = mbar_wait(tmem_done, 0);
    if (!got && lane == 0) atomicOr(p.err, kDevErrTimeout);
    tc_fence_after();
    __syncwarp();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tbase), "r"(S::TMEM_COLS));
  }
}

}  // namespace pfkv
