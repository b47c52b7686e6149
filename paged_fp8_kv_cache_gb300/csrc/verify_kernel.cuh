// Grouped causal-verify attention on the 5th-generation tensor cores
// (tcgen05 + TMEM) for FP8 caches: the g*T query rows of one KV head
// (e.g. 6 heads x 8 speculative tokens = 48 rows, "1Cat-vLLM 1.5.0",
// "Production DFlash2 on V100" / "Flash-V100 long-context improvements":
// exact grouped q8 verification over FP8 KV) form a real dense tile.
//
// One CTA = one (key range, KV head, sequence), 14 warps:
//   warp 0      producer: TMA tile copies of 128-key FP8 K/V tiles into a
//               shared-memory ring (same tensor maps as the decode kernel);
//   warp 1      MMA issuer (one lane) and TMEM owner;
//   warps 2-5   K converter: each thread owns one TMEM lane = one key of the
//               tile and turns its K row (FP8 -> fp16, exact) into the A
//               operand of S^T = K Q^T, written with tcgen05.st;
//   warps 6-9   softmax: each thread owns one key of the tile; it reads the
//               key's logits for all rows from TMEM, masks, exponentiates
//               against a per-row reference maximum and writes P^T (fp16)
//               into a swizzled shared-memory B operand; at the end it reads
//               O^T back from TMEM and writes the output;
//   warps 10-13 V converter: each thread owns one TMEM lane = one or two
//               head-dim elements and writes them for all keys of the tile
//               as the A operand of O^T = V^T P^T.
// MMAs: M = 128 (keys for S^T, head-dim elements for O^T), N = rows padded
// to a multiple of 16, K = 16 per instruction, f16 inputs, f32 accumulators
// in TMEM. Online softmax: every row keeps a reference maximum m; p is formed
// against it in one pass. A tile whose logits exceed m by more than
// kRescaleLog2 triggers an exact update (the tile's true row maxima are
// reduced across the 128 keys; the running sums and the O^T accumulators are
// rescaled and the tile is redone against the new references); the first
// tile always does. Every wait is an mbarrier wait with a poll limit, so
// every path of every role ends, and TMEM is freed after a CTA-wide barrier.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <math_constants.h>
#include <stdint.h>

#include "device_utils.cuh"
#include "frag_layout.h"
#include "pfkv_internal.h"

namespace pfkv {

constexpr float kRescaleLog2 = 8.f;

template <int D, int NMAX_>
struct VerifyShape {
  static constexpr int KT = 128;                         // keys per tile (MMA M)
  static constexpr int NBOX = D / kBoxBytes;             // 128-byte boxes per FP8 key row
  static constexpr int SUB = KT * kBoxBytes;             // one box column of a tile (16 KB)
  static constexpr int KV_TILE = NBOX * SUB;             // K (or V) bytes per tile
  static constexpr int NMAX = NMAX_;                     // padded query rows (MMA N): 32, 48 or 64
  static constexpr int Q_BYTES = (D / 64) * NMAX * 128;  // Q as K-major 128B-swizzled blocks of 64 dims
  static constexpr int PT_BYTES = (KT / 64) * NMAX * 128;  // one P^T buffer (K-major, 64-key blocks)
  static constexpr int MT = D / 128;                     // O^T M-tiles
  static constexpr int TMEM_COLS = 512;
  static constexpr int COL_S = 0;                        // 2 x NMAX: S^T double buffer
  static constexpr int COL_O = 2 * NMAX;                 // MT x NMAX: O^T
  static constexpr int COL_AK = ((COL_O + MT * NMAX + 31) / 32) * 32;  // D/2: K as A operand (fp16 pairs)
  static constexpr int COL_AV = COL_AK + D / 2;          // MT x KT/2: V^T as A operand
  static_assert(COL_AV + MT * KT / 2 <= TMEM_COLS, "TMEM budget");
  // misc: m_ref, alpha, wred[4], lsum[4], m_prev (NMAX floats each), flags, TMEM slot, barriers
  static constexpr int MISC_BYTES = 11 * NMAX * 4 + 64 + 32 * 8;
  // Separate K and V rings. V tiles are held longest (the V operand of tile i+1 can only be
  // written once the PV MMAs of tile i are done), so the V ring gets whatever depth the
  // remaining shared memory allows (2..4 tiles).
  static constexpr int kSmemLimit = 227 * 1024;
  static constexpr int NK = KV_TILE <= 16384 ? 3 : 2;
  static constexpr int NV_FIT = (kSmemLimit - 1024 - NK * KV_TILE - Q_BYTES - 2 * PT_BYTES - MISC_BYTES) / KV_TILE;
  static constexpr int NV = NV_FIT > 4 ? 4 : NV_FIT;
  static_assert(NV >= 2, "shared memory budget");
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

// D (TMEM) (+)= A (TMEM) * B (shared memory)
__device__ __forceinline__ void umma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate));
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

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]),
        "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// byte offset of 16-bit element (row, k) in a K-major 128B-swizzled block of 64-element rows
__device__ __forceinline__ int sw128_elem(int row, int k) {
  return row * 128 + ((((k >> 3) ^ row) & 7) << 4) + ((k & 7) << 1);
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

template <int D, int KV, int NMAX_>
__global__ void __launch_bounds__(448, 1)
    verify_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                  const DecodeParams p) {
  using S = VerifyShape<D, NMAX_>;
  constexpr int KT = S::KT, NBOX = S::NBOX, NK = S::NK, NV = S::NV, NMAX = S::NMAX, MT = S::MT;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int R = p.T * p.G;
  const int NP = (R + 15) & ~15;  // MMA N

  // launched with programmatic stream serialisation: wait for the preceding grid first
  asm volatile("griddepcontrol.wait;" ::: "memory");
  int N = p.seq_lens[b];
  {
    const int cap = min(p.max_seq_len, p.max_blocks * p.page_size);
    if (N < 0 || N > cap) {
      if (threadIdx.x == 0 && split == 0 && kvh == 0) atomicOr(p.err, kDevErrSeqLen);
      N = N < 0 ? 0 : cap;
    }
  }
  const int nsplit_b = N > 0 ? (N + p.split_tokens - 1) / p.split_tokens : 1;
  if (split >= nsplit_b) return;
  const int t0 = split * p.split_tokens;
  const int t1 = min(N, t0 + p.split_tokens);
  const int ntiles = t1 > t0 ? (t1 - t0 + KT - 1) / KT : 0;

  float* m_ref = reinterpret_cast<float*>(smem + S::OFF_MISC);  // [NMAX] reference max (log2 units)
  float* alpha_s = m_ref + NMAX;                                 // [NMAX] rescale factors
  float* wred = alpha_s + NMAX;                                  // [4][NMAX] per-warp maxima
  float* lsum = wred + 4 * NMAX;                                 // [4][NMAX] per-warp row sums
  float* m_prev = lsum + 4 * NMAX;                               // [NMAX] references before an update
  int* flag = reinterpret_cast<int*>(m_prev + NMAX);             // [3] rescale votes
  uint32_t* tslot = reinterpret_cast<uint32_t*>(flag + 4);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::OFF_MISC + 11 * NMAX * 4 + 64);
  uint64_t* kfull = bars;              // [NK] producer -> K converter
  uint64_t* kempty = kfull + NK;       // [NK] K converter -> producer
  uint64_t* vfull = kempty + NK;       // [NV] producer -> V converter
  uint64_t* vempty = vfull + NV;       // [NV] V converter -> producer
  uint64_t* ak_full = vempty + NV;     // K converter -> MMA (K operand written)
  uint64_t* av_full = ak_full + 1;     // V converter -> MMA (V operand written)
  uint64_t* ak_free = av_full + 1;     // MMA commit: S^T MMAs done with the K operand
  uint64_t* s_full = ak_free + 1;      // [2] MMA commit: S^T ready
  uint64_t* s_free = s_full + 2;       // [2] softmax -> MMA: S^T read
  uint64_t* pt_full = s_free + 2;      // [2] softmax -> MMA: P^T written
  uint64_t* pt_free = pt_full + 2;     // [2] MMA commit: O^T MMAs done reading P^T buffer
  uint64_t* o_done = pt_free + 2;      // MMA commit: O^T MMAs of a tile done
  uint64_t* swg_bar = o_done + 1;      // softmax warpgroup rendezvous (bounded waits, unlike bar.sync)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tid = threadIdx.x;

  if (tid == 0) {
    for (int s = 0; s < NK; ++s) {
      mbar_init(&kfull[s], 1);
      mbar_init(&kempty[s], 4);  // one arrival per K-converter warp
    }
    for (int s = 0; s < NV; ++s) {
      mbar_init(&vfull[s], 1);
      mbar_init(&vempty[s], 4);  // one arrival per V-converter warp
    }
    mbar_init(ak_full, 4);
    mbar_init(av_full, 4);
    mbar_init(ak_free, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_free[i], 4);
      mbar_init(&pt_full[i], 4);
      mbar_init(&pt_free[i], 1);
    }
    mbar_init(o_done, 1);
    mbar_init(swg_bar, 4);
    fence_barrier_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tslot)),
                 "r"(S::TMEM_COLS));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  // Q -> shared memory (K-major, 128B swizzle), padded rows zero; softmax state
  {
    unsigned char* sq = smem + S::OFF_Q;
    for (int idx = tid; idx < NMAX * (D / 8); idx += blockDim.x) {
      const int r = idx / (D / 8);
      const int d8 = (idx - r * (D / 8)) * 8;  // 8 consecutive dims = one 16-byte chunk
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (r < R) {
        const int t = r / p.G, j = r - t * p.G;
        v = *reinterpret_cast<const uint4*>(p.q + ((static_cast<size_t>(b) * p.T + t) * p.num_q_heads + kvh * p.G + j) * D + d8);
      }
      *reinterpret_cast<uint4*>(sq + (d8 >> 6) * NMAX * 128 + sw128_elem(r, d8 & 63)) = v;
    }
    for (int i = tid; i < NMAX; i += blockDim.x) m_ref[i] = -CUDART_INF_F;
    if (tid == 0) flag[0] = flag[1] = flag[2] = 0;
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;

  const float kscale = *p.k_scale, vscale = *p.v_scale;
  const float sc2 = p.softmax_scale * kscale * 1.4426950408889634f;
  bool alive = true;

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    if (ntiles > 0) {
      if (lane == 0) {
        prefetch_tensormap(&tmk);
        prefetch_tensormap(&tmv);
      }
      const int P = p.page_size;
      const int* bt = p.block_table + static_cast<size_t>(b) * p.max_blocks;
      const int page_last = (t1 - 1) >> p.page_shift;
      // 32 lanes fetch 32 consecutive page ids at a time; lane 0 reads them by shuffle
      int chunk_base = -(1 << 30);
      int my_id = 0;
      auto page_id = [&](int pidx) -> int {
        if (pidx < chunk_base || pidx >= chunk_base + 32) {
          chunk_base = pidx;
          const int mine = chunk_base + lane;
          my_id = 0;
          if (mine <= page_last) {
            my_id = bt[mine];
            if (static_cast<unsigned>(my_id) >= static_cast<unsigned>(p.num_blocks)) {
              atomicOr(p.err, kDevErrBlockId);
              my_id = 0;
            }
          }
        }
        return __shfl_sync(0xffffffffu, my_id, pidx - chunk_base);
      };
      // rows of the tile's 64-row boxes (P >= 64) or pages (P < 64); at most 8
      auto wait_slot = [&](uint64_t* bar, int it, int depth) -> bool {
        if (it < depth) return true;
        bool got = true;
        if (lane == 0) got = mbar_wait(&bar[it % depth], ((it / depth) - 1) & 1);
        return __shfl_sync(0xffffffffu, got, 0);
      };
      for (int it = 0; it < ntiles && alive; ++it) {
        const int tile_start = t0 + it * KT;
        const int valid = min(KT, t1 - tile_start);
        int rows[8], box_rows, nbox_rows;
        if (P >= kTileKeys) {
          nbox_rows = (valid + kTileKeys - 1) / kTileKeys;
          box_rows = kTileKeys;
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            const int key = tile_start + hf * kTileKeys;
            rows[hf] = 0;
            if (hf < nbox_rows) rows[hf] = (page_id(key >> p.page_shift) * p.num_kv_heads + kvh) * P + (key & (P - 1));
          }
        } else {
          nbox_rows = (valid + P - 1) >> p.page_shift;
          box_rows = P;
          const int pfirst = tile_start >> p.page_shift;
#pragma unroll
          for (int pg = 0; pg < 8; ++pg) {
            rows[pg] = 0;
            if (pg < nbox_rows) rows[pg] = (page_id(pfirst + pg) * p.num_kv_heads + kvh) * P;
          }
        }
        const uint32_t bytes = NBOX * nbox_rows * box_rows * kBoxBytes;
        // K tile, then V tile, each into its own ring
        for (int which = 0; which < 2; ++which) {
          uint64_t* fullb = which == 0 ? kfull : vfull;
          uint64_t* emptyb = which == 0 ? kempty : vempty;
          const int depth = which == 0 ? NK : NV;
          if (!wait_slot(emptyb, it, depth)) {
            if (lane == 0) atomicOr(p.err, kDevErrTimeout);
            alive = false;
            break;
          }
          unsigned char* dst = smem + (which == 0 ? S::OFF_KRING : S::OFF_VRING) + (it % depth) * S::KV_TILE;
          const CUtensorMap* map = which == 0 ? &tmk : &tmv;
          if (lane == 0) {
            mbar_arrive_expect_tx(&fullb[it % depth], bytes);
            for (int r = 0; r < nbox_rows; ++r) {
#pragma unroll
              for (int bx = 0; bx < NBOX; ++bx)
                tma_load_2d(dst + bx * S::SUB + r * box_rows * kBoxBytes, map, &fullb[it % depth], bx * kBoxBytes,
                            rows[r]);
            }
          }
        }
      }
      // do not leave while copies may still land in this CTA's shared memory
      if (lane == 0) {
        for (int it = max(0, ntiles - NK); it < ntiles; ++it)
          if (!mbar_wait(&kfull[it % NK], (it / NK) & 1)) {
            atomicOr(p.err, kDevErrTimeout);
            break;
          }
        for (int it = max(0, ntiles - NV); it < ntiles; ++it)
          if (!mbar_wait(&vfull[it % NV], (it / NV) & 1)) {
            atomicOr(p.err, kDevErrTimeout);
            break;
          }
      }
      __syncwarp();
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0 && ntiles > 0) {
      const uint32_t idesc = umma_idesc_f16(NP);
      const uint32_t q_base = smem_u32(smem + S::OFF_Q);
      const uint32_t pt_base = smem_u32(smem + S::OFF_PT);
      // Issue whichever MMA group is ready: S^T of the next tile (its K operand written, its
      // S buffer released by the softmax) or O^T of the oldest tile whose V operand and P^T
      // are written. Neither waits behind the other.
      int sn = 0, on = 0;
      bool ok = true;
      uint64_t last = global_ns();
      while (on < ntiles) {
        bool progress = false;
        if (sn < ntiles && mbar_test(ak_full, sn & 1) &&
            (sn < 2 || mbar_test(&s_free[sn & 1], ((sn >> 1) - 1) & 1))) {
          tc_fence_after();
          const uint32_t d_t = tbase + S::COL_S + (sn & 1) * NMAX;
#pragma unroll 1
          for (int ks = 0; ks < D / 16; ++ks) {
            const uint64_t bd = umma_desc_sw128(q_base + (ks >> 2) * NMAX * 128 + (ks & 3) * 32);
            umma_ts(d_t, tbase + S::COL_AK + 8 * ks, bd, idesc, ks > 0 ? 1u : 0u);
          }
          umma_commit(&s_full[sn & 1]);
          umma_commit(ak_free);
          ++sn;
          progress = true;
        }
        if (on < sn && mbar_test(av_full, on & 1) && mbar_test(&pt_full[on & 1], (on >> 1) & 1)) {
          tc_fence_after();
          const uint32_t pt = pt_base + (on & 1) * S::PT_BYTES;
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
#pragma unroll 1
            for (int ks = 0; ks < KT / 16; ++ks) {
              const uint64_t bd = umma_desc_sw128(pt + (ks >> 2) * NMAX * 128 + (ks & 3) * 32);
              umma_ts(tbase + S::COL_O + mt * NMAX, tbase + S::COL_AV + mt * (KT / 2) + 8 * ks, bd, idesc,
                      (on > 0 || ks > 0) ? 1u : 0u);
            }
          }
          umma_commit(&pt_free[on & 1]);
          umma_commit(o_done);
          ++on;
          progress = true;
        }
        if (progress) {
          last = global_ns();
        } else {
          if (global_ns() - last > kWaitLimitNs) {
            ok = false;
            break;
          }
          __nanosleep(32);
        }
      }
      if (!ok) atomicOr(p.err, kDevErrTimeout);
    }
    __syncwarp();
  } else if (warp < 6) {
    // ---------------------------------------------------------------- K converter (warps 2-5)
    const int q = warp & 3;              // TMEM lane quadrant of this warp
    const int key_row = 32 * q + lane;   // this thread's key of the tile = its TMEM lane
    const uint32_t tq = tbase + (static_cast<uint32_t>(32 * q) << 16);
    for (int it = 0; it < ntiles; ++it) {
      const int s = it % NK;
      if (!mbar_wait(&kfull[s], (it / NK) & 1) || (it > 0 && !mbar_wait(ak_free, (it - 1) & 1))) {
        alive = false;
        break;
      }
      tc_fence_after();
      const unsigned char* Ks = smem + S::OFF_KRING + s * S::KV_TILE;
#pragma unroll
      for (int bx = 0; bx < NBOX; ++bx) {
#pragma unroll
        for (int cp = 0; cp < 4; ++cp) {  // two 16-byte chunks = 32 codes = 16 fp16 pairs = 16 columns
          uint32_t u[16];
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            const uint4 v = lds128(Ks + bx * S::SUB + swz_offset(key_row, 2 * cp + cc));
            const uint32_t x[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              u[cc * 8 + 2 * j] = fp8x2_to_f16x2<KV>(x[j]);            // dims 4j, 4j+1 of the chunk
              u[cc * 8 + 2 * j + 1] = fp8x2_to_f16x2<KV>(x[j] >> 16);  // dims 4j+2, 4j+3
            }
          }
          tmem_st16(tq + S::COL_AK + bx * 64 + cp * 16, u);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(ak_full);
        mbar_arrive(&kempty[s]);
      }
    }
    if (!alive && lane == 0) atomicOr(p.err, kDevErrTimeout);
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
    for (int it = 0; it < ntiles; ++it) {
      const int s = it % NV;
      if (!mbar_wait(&vfull[s], (it / NV) & 1) || (it > 0 && !mbar_wait(o_done, (it - 1) & 1))) {
        alive = false;
        break;
      }
      tc_fence_after();
      const unsigned char* Vs = smem + S::OFF_VRING + s * S::KV_TILE;
      const int valid = min(KT, t1 - (t0 + it * KT));
      const bool tail = valid < KT;
#pragma unroll 1
      for (int k0 = 0; k0 < KT; k0 += 32) {
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
          if (tail) {  // stale bytes past the range end must not reach the MMA
            if (k0 + kk >= valid) wa = 0u;
            if (k0 + kk + 1 >= valid) wb = 0u;
          }
          const uint32_t X = __byte_perm(wa, wb, 0x5140);  // [a.b0, b.b0, a.b1, b.b1]
          v0[kk >> 1] = fp8x2_to_f16x2<KV>(X);
          v1[kk >> 1] = fp8x2_to_f16x2<KV>(X >> 16);
        }
        tmem_st16(tq + S::COL_AV + (k0 >> 1), v0);
        if constexpr (MT == 2) tmem_st16(tq + S::COL_AV + KT / 2 + (k0 >> 1), v1);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(av_full);
        mbar_arrive(&vempty[s]);
      }
    }
    if (!alive && lane == 0) atomicOr(p.err, kDevErrTimeout);
  } else {
    // ---------------------------------------------------------------- softmax + epilogue (warps 6-9)
    const int q = warp & 3;
    const int sw = warp - 6;  // 0..3 within the softmax warpgroup
    const int key_lane = 32 * q + lane;
    const uint32_t tq = tbase + (static_cast<uint32_t>(32 * q) << 16);
    uint32_t swg_phase = 0;
    // the 4 softmax warps meet; a wait that runs out marks the CTA's work as failed
    auto swg_sync = [&]() {
      __syncwarp();
      if (lane == 0) mbar_arrive(swg_bar);
      if (!mbar_wait(swg_bar, swg_phase & 1)) alive = false;
      ++swg_phase;
    };
    float l_part[NMAX];  // this thread's (key lane's) share of every row sum, fp32
#pragma unroll
    for (int r = 0; r < NMAX; ++r) l_part[r] = 0.f;
    const int tlim_base = N - p.T;  // row r sees keys <= N - T + r / G
    for (int it = 0; it < ntiles && alive; ++it) {
      const int sb = it & 1;
      if (!mbar_wait(&s_full[sb], (it >> 1) & 1)) {
        alive = false;
        break;
      }
      tc_fence_after();
      // P^T buffer sb is free once the O^T MMAs of tile it-2 are done (its own barrier:
      // o_done may already be a phase further, which a parity wait cannot tell apart)
      if (it >= 2 && !mbar_wait(&pt_free[sb], ((it >> 1) - 1) & 1)) {
        alive = false;
        break;
      }
      const uint32_t s_col = tq + S::COL_S + sb * NMAX;
      const int tile_start = t0 + it * KT;
      const int kp = tile_start + key_lane;  // absolute key position
      const bool in_range = kp < t1;
      // row r sees this key iff r / G >= kp - (N - T), i.e. r >= G * (kp - (N - T))
      const int rmin = p.G * (kp - tlim_base);
      const bool all_vis = (tile_start + KT <= t1) && (tile_start + KT - 1 <= tlim_base);  // CTA-uniform
      // logits of 16 rows (columns c0..c0+15) of this thread's key, scaled to base 2 and masked
      auto load_s2 = [&](int c0, float (&s2)[16]) {
        uint32_t v[16];
        tmem_ld16(s_col + c0, v);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int r = c0 + j;
          const bool vis = all_vis || (in_range && (r >= R || r >= rmin));
          s2[j] = vis ? __uint_as_float(v[j]) * sc2 : -CUDART_INF_F;
        }
      };
      auto load_m = [&](const float* src, int c0, float (&m)[16]) {
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const float4 mv = *reinterpret_cast<const float4*>(src + c0 + 4 * q4);
          m[4 * q4] = mv.x;
          m[4 * q4 + 1] = mv.y;
          m[4 * q4 + 2] = mv.z;
          m[4 * q4 + 3] = mv.w;
        }
      };
      // 2^(s - m) against a reference m; 0 while a row has no reference yet, and capped so
      // that a logit that outgrew its reference (the tile is then redone) stays finite
      auto pexp = [](float s2, float m) -> float {
        return m == -CUDART_INF_F ? 0.f : fast_exp2(fminf(s2 - m, 15.f));
      };
      unsigned char* pt = smem + S::OFF_PT + sb * S::PT_BYTES + (key_lane >> 6) * NMAX * 128;
      const int kk = key_lane & 63;
      // one pass: P^T and the row sums against the current references; note outgrown rows
      bool exceed = false;
#pragma unroll
      for (int c0 = 0; c0 < NMAX; c0 += 16) {
        if (c0 < NP) {
          float s2[16], m[16];
          load_s2(c0, s2);
          load_m(m_ref, c0, m);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            exceed |= (s2[j] > m[j] + kRescaleLog2);
            const float pr = pexp(s2[j], m[j]);
            l_part[c0 + j] += pr;
            *reinterpret_cast<__half*>(pt + sw128_elem(c0 + j, kk)) = __float2half_rn(pr);
          }
        }
      }
      // exact update of the reference maxima when any logit outgrew its row's
      // (three rotating flags: the one cleared here, of tile it-1, was read by every
      // thread before it reached this tile's rendezvous, and is voted on again only
      // after the next rendezvous, which the clearing thread must reach first)
      if (__any_sync(0xffffffffu, exceed) && lane == 0) atomicOr(&flag[it % 3], 1);
      swg_sync();
      const bool rescale = flag[it % 3] != 0;
      if (threadIdx.x == 6 * 32) flag[(it + 2) % 3] = 0;
      if (rescale) {
#pragma unroll
        for (int c0 = 0; c0 < NMAX; c0 += 16) {
          if (c0 < NP) {
            float s2[16];
            load_s2(c0, s2);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              float mx = s2[j];
#pragma unroll
              for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
              if (lane == 0) wred[sw * NMAX + c0 + j] = mx;
            }
          }
        }
        swg_sync();
        if (key_lane < NP) {
          const int r = key_lane;
          const float mt = fmaxf(fmaxf(wred[r], wred[NMAX + r]), fmaxf(wred[2 * NMAX + r], wred[3 * NMAX + r]));
          const float mo = m_ref[r];
          const float mn = fmaxf(mo, mt);
          // the reference only moves up; rows with nothing visible so far keep -inf
          alpha_s[r] = (mo == -CUDART_INF_F) ? 0.f : fast_exp2(mo - mn);
          m_prev[r] = mo;
          m_ref[r] = mn;
        }
        swg_sync();
        // take this tile's first-pass terms back out (same formula, same values), rescale the
        // earlier tiles' share, then redo the tile against the new references
#pragma unroll
        for (int c0 = 0; c0 < NMAX; c0 += 16) {
          if (c0 < NP) {
            float s2[16], m[16];
            load_s2(c0, s2);
            load_m(m_prev, c0, m);
#pragma unroll
            for (int j = 0; j < 16; ++j) l_part[c0 + j] = (l_part[c0 + j] - pexp(s2[j], m[j])) * alpha_s[c0 + j];
          }
        }
        if (it > 0) {
          // rescale the O^T columns once the previous tile's MMAs are done (sound: the wait
          // on pt_free at the top of this tile established that tile it-2's were)
          if (!mbar_wait(o_done, (it - 1) & 1)) alive = false;
          tc_fence_after();
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
            for (int c0 = 0; c0 < NMAX; c0 += 16) {
              if (c0 < NP) {
                uint32_t v[16];
                const uint32_t a = tq + S::COL_O + mt * NMAX + c0;
                tmem_ld16(a, v);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 16; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) * alpha_s[c0 + j]);
                tmem_st16(a, v);
              }
            }
          }
          tmem_wait_st();
        }
#pragma unroll
        for (int c0 = 0; c0 < NMAX; c0 += 16) {
          if (c0 < NP) {
            float s2[16], m[16];
            load_s2(c0, s2);
            load_m(m_ref, c0, m);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const float pr = pexp(s2[j], m[j]);
              l_part[c0 + j] += pr;
              *reinterpret_cast<__half*>(pt + sw128_elem(c0 + j, kk)) = __float2half_rn(pr);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_free[sb]);  // S^T buffer sb fully read
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(&pt_full[sb]);
    }
    if (!alive && lane == 0) atomicOr(p.err, kDevErrTimeout);

    // ------------------------------------------------------------ epilogue
    // All MMAs done. (Not a wait on o_done for the last tile: a parity wait for phase k is
    // only sound once phase k-1 has completed, and nothing here orders the PV MMAs of tile
    // ntiles-2 before this point. pt_free of the last tile's buffer is sound -- this thread
    // saw its previous phase, of tile ntiles-3 -- and its commit covers every earlier MMA.)
    if (ntiles > 0 && alive && !mbar_wait(&pt_free[(ntiles - 1) & 1], ((ntiles - 1) >> 1) & 1)) alive = false;
    tc_fence_after();
    // row sums over the 128 keys
#pragma unroll
    for (int r = 0; r < NMAX; ++r) {
      float v = l_part[r];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
      if (lane == 0) lsum[sw * NMAX + r] = v;
    }
    swg_sync();
    const bool final_out = (nsplit_b == 1);
    // this thread's TMEM lane = head-dim element(s) of O^T
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      const int d_out = (MT == 2) ? 2 * key_lane + mt : key_lane;
#pragma unroll
      for (int c0 = 0; c0 < NMAX; c0 += 16) {
        if (c0 >= NP) continue;
        uint32_t v[16];
        if (ntiles > 0) {
          tmem_ld16(tq + S::COL_O + mt * NMAX + c0, v);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int j = 0; j < 16; ++j) v[j] = 0u;
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int r = c0 + j;
          if (r >= R) continue;
          const float L = lsum[r] + lsum[NMAX + r] + lsum[2 * NMAX + r] + lsum[3 * NMAX + r];
          const float M = m_ref[r];
          const bool has = alive && ntiles > 0 && (M != -CUDART_INF_F) && (L > 0.f);
          const float o = has ? __uint_as_float(v[j]) * vscale / L : 0.f;
          const int t = r / p.G, jj = r - t * p.G;
          const size_t grow = (static_cast<size_t>(b) * p.T + t) * p.num_q_heads + kvh * p.G + jj;
          const float lse_val = has ? (M + log2f(L)) * 0.6931471805599453f : -CUDART_INF_F;
          if (final_out) {
            p.out[grow * D + d_out] = __float2half_rn(o);
            if (d_out == 0) p.lse[grow] = lse_val;
          } else {
            p.o_part[(grow * p.num_splits + split) * D + d_out] = o;
            if (d_out == 0) p.lse_part[grow * p.num_splits + split] = lse_val;
          }
        }
      }
    }
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  }
  // all roles done with TMEM before it is released
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tbase), "r"(S::TMEM_COLS));
}

}  // namespace pfkv
