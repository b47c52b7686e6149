// Paged decode / grouped causal-verify attention over an FP8 (or fp16)
// KV cache: the split-KV partial kernel.
//
// One CTA handles one (key range, KV head, query slab, sequence). Its rows
// are the query rows (query token t of the slab, head of the group) that
// share the KV head -- all T * g rows for ordinary GQA decode and for the
// grouped q8 verifier ("1Cat-vLLM 1.5.0", "Flash-V100 long-context
// improvements": grouped q8 verifier, page-ID reuse, 128-bit cache loads,
// long-context split route), up to 64 rows of a prefill chunk's slab. The
// mask (causal or not, sliding window) bounds each row's keys from both
// sides; a CTA's key range starts at its slab's lowest visible key, so the
// tiles before a window are never read (mask_span.h).
//
// Warp roles:
//  * one producer warp: walks the key range 64 keys at a time, reads each
//    page id from the block table once and issues TMA tile copies of the K
//    and V rows (FP8 bytes, 128-byte swizzle) into a ring of shared-memory
//    stages, signalling an mbarrier per stage;
//  * NRG x NTS consumer warps: row group rg (8*NT query rows) x token slice
//    ts. Each consumer handles, per stage, the 16-key groups ts, ts+NTS, ...
//    For a group it converts the FP8 K bytes to fp16 in registers (exact),
//    computes S^T = K Q^T with mma.sync (16 keys x 8 rows x 16 dims per
//    instruction, fp32 accumulate), masks by causal limit and sequence end,
//    updates its running max / sum (online softmax, base-2 exponent), moves
//    P^T into MMA operand form with movmatrix and accumulates O^T = V^T P^T
//    with V converted in registers the same way.
// At the end the NTS partial states of each row group are combined through
// shared memory and written either as the final output (fp16 out + fp32
// LSE) when the sequence has a single key range, or as a normalised fp32
// partial plus its LSE for the merge kernel.
//
// Two grids run this work. decode_kernel: one CTA per (range, KV head, slab,
// sequence) of the longest sequence the call allows; CTAs past a shorter
// sequence's ranges return at once. decode_persist_kernel (ragged batches of
// one-slab calls): one wave of CTAs that take the ranges that exist, one
// after another, from a counter -- the CTAs of a batch of short sequences
// never sit in an SM slot without work.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <math_constants.h>
#include <stdint.h>

#include "device_utils.cuh"
#include "frag_layout.h"
#include "mask_span.h"
#include "pfkv_internal.h"

namespace pfkv {

template <int D, int KV>
struct DecodeShape {
  static constexpr int ELT = (KV == kKvFp16) ? 2 : 1;
  static constexpr int ROWB = D * ELT;
  static constexpr int NBOX = ROWB / kBoxBytes;
  static constexpr int KV_STAGE = NBOX * kSubTileBytes;  // K (or V) bytes of one stage
  static constexpr int STAGE = 2 * KV_STAGE;
  static constexpr int NS = STAGE <= 16384 ? 4 : (STAGE <= 32768 ? 3 : 2);  // pipeline depth
  static constexpr int KSTEPS = D / 16;
  static constexpr int MTILES = D / 16;                  // PV m-tiles over the head dim
};

// Dynamic shared memory needed by one CTA (without the 1 KB alignment slack).
template <int D, int KV, int NT>
constexpr int decode_smem_bytes(int ncw) {
  using S = DecodeShape<D, KV>;
  const int obuf = ncw * 8 * NT * D * 4;
  const int ring = S::NS * S::STAGE;
  const int body = obuf > ring ? obuf : ring;
  return body + ncw * 8 * NT * 8 /* m, l */ + 2 * S::NS * 8 /* barriers */;
}

// The persistent kernel: ring | (m, l) | full[NS], empty[NS] | item_full[2], item_free[2], the
// consumers' rendezvous | item slots[2] | lengths[B] | ranges[B] | item prefix[B + 1]. (Its
// combine buffer is the ring slot of each item's last stage.)
template <int D, int KV, int NT>
constexpr int persist_smem_bytes(int ncw, int num_seqs) {
  using S = DecodeShape<D, KV>;
  return S::NS * S::STAGE + ncw * 8 * NT * 8 + (2 * S::NS + 5) * 8 + 8 + (3 * num_seqs + 1) * 4;
}

// One unit of work: a key range of one (sequence, KV head, slab).
struct DecodeItem {
  int b, kvh, slab, split, N;
  SlabSpan sp;
  int nsplit, t0, t1, ntiles;
};

// Sequence length validated against what the block table can address (clamped; flagged when
// `report`).
__device__ __forceinline__ int checked_len(const DecodeParams& p, int N, bool report) {
  const int cap = min(p.max_seq_len, p.max_blocks * p.page_size);
  if (N < 0 || N > cap) {
    if (report) atomicOr(p.err, kDevErrSeqLen);
    N = N < 0 ? 0 : cap;
  }
  return N;
}

__device__ __forceinline__ DecodeItem make_item(const DecodeParams& p, int b, int kvh, int slab, int split, int N) {
  DecodeItem it;
  it.b = b;
  it.kvh = kvh;
  it.slab = slab;
  it.split = split;
  it.N = N;
  it.sp = slab_span(N, p.T, slab, p.slab_tokens, p.causal, p.window, kTileKeys);
  it.nsplit = span_splits(it.sp, p.split_tokens);
  it.t0 = it.sp.base + split * p.split_tokens;
  it.t1 = it.sp.hi >= it.sp.lo ? min(it.sp.hi + 1, it.t0 + p.split_tokens) : it.t0;
  it.ntiles = it.t1 > it.t0 ? (it.t1 - it.t0 + kTileKeys - 1) / kTileKeys : 0;
  return it;
}

// Producer warp: issue the TMA copies of one item's tiles into the ring. g counts the stages
// filled so far (across items): stage g is slot g % NS_, phase g / NS_. pguess / pre_id: the
// block-table entries of 32 pages from page pguess, fetched ahead (pguess = -1: none).
template <int D, int KV, int NS_>
__device__ __forceinline__ bool produce_item(const CUtensorMap& tmk, const CUtensorMap& tmv, const DecodeParams& p,
                                             unsigned char* smem, uint64_t* full, uint64_t* empty,
                                             const DecodeItem& item, int& g, int pguess, int pre_id, int lane) {
  using S = DecodeShape<D, KV>;
  constexpr int ELT = S::ELT, NBOX = S::NBOX;
  const int kvh = item.kvh;
  const int ntiles = item.ntiles;
  if (ntiles <= 0) return true;
  const int P = p.page_size;
  const int* bt = p.block_table + static_cast<size_t>(item.b) * p.max_blocks;
  const int page_last = (item.t1 - 1) >> p.page_shift;
  const int pfirst0 = item.t0 >> p.page_shift;
  // The lanes hold the ids of pages chunk_base .. chunk_base + 31 (the first chunk fetched ahead
  // when it did not depend on the length), and the raw ids of the next 32 pages, loaded one
  // chunk ahead: moving to the next chunk never waits on the table (with 16-token pages a chunk
  // lasts 8 tiles). An id outside the pool is flagged when its chunk becomes current and block 0
  // is read instead.
  auto load_raw = [&](int first) -> int {
    const int mine = first + lane;
    return mine <= page_last ? bt[mine] : 0;
  };
  auto checked = [&](int raw, int first) -> int {
    if (first + lane > page_last) return 0;
    if (static_cast<unsigned>(raw) >= static_cast<unsigned>(p.num_blocks)) {
      atomicOr(p.err, kDevErrBlockId);
      return 0;
    }
    return raw;
  };
  int chunk_base = pfirst0;
  int my_id = checked(pguess == pfirst0 ? pre_id : load_raw(pfirst0), pfirst0);
  int next_raw = load_raw(pfirst0 + 32);
  auto page_id = [&](int pidx) -> int {
    if (pidx < chunk_base || pidx >= chunk_base + 32) {
      my_id = pidx == chunk_base + 32 ? checked(next_raw, pidx) : checked(load_raw(pidx), pidx);
      chunk_base = pidx;
      next_raw = load_raw(chunk_base + 32);
    }
    return __shfl_sync(0xffffffffu, my_id, pidx - chunk_base);
  };
  for (int it = 0; it < ntiles; ++it, ++g) {
    const int s = g % NS_;
    // slot s is free once the consumers released stage g - NS_ (sound: this warp waited for that
    // barrier's previous phase, of stage g - 2 * NS_, before filling stage g - NS_)
    if (g >= NS_) {
      bool got = true;
      if (lane == 0) got = mbar_wait(&empty[s], ((g / NS_) - 1) & 1);
      got = __shfl_sync(0xffffffffu, got, 0);
      if (!got) {
        if (lane == 0) atomicOr(p.err, kDevErrTimeout);
        return false;
      }
    }
    unsigned char* kdst = smem + s * S::STAGE;
    unsigned char* vdst = kdst + S::KV_STAGE;
    const int tile_start = item.t0 + it * kTileKeys;
    if (P >= kTileKeys) {
      const int blk = page_id(tile_start >> p.page_shift);
      const int row = (blk * p.num_kv_heads + kvh) * P + (tile_start & (P - 1));
      if (lane == 0) {
        mbar_arrive_expect_tx(&full[s], 2 * S::KV_STAGE);
#pragma unroll
        for (int bx = 0; bx < NBOX; ++bx) {
          tma_load_2d(kdst + bx * kSubTileBytes, &tmk, &full[s], bx * (kBoxBytes / ELT), row);
          tma_load_2d(vdst + bx * kSubTileBytes, &tmv, &full[s], bx * (kBoxBytes / ELT), row);
        }
      }
    } else {
      const int valid = min(kTileKeys, item.t1 - tile_start);
      const int npages = (valid + P - 1) >> p.page_shift;
      const int pfirst = tile_start >> p.page_shift;
      if (lane == 0) mbar_arrive_expect_tx(&full[s], 2 * NBOX * npages * P * kBoxBytes);
      for (int pg = 0; pg < npages; ++pg) {
        const int blk = page_id(pfirst + pg);
        const int row = (blk * p.num_kv_heads + kvh) * P;
        if (lane == 0) {
#pragma unroll
          for (int bx = 0; bx < NBOX; ++bx) {
            tma_load_2d(kdst + bx * kSubTileBytes + pg * P * kBoxBytes, &tmk, &full[s], bx * (kBoxBytes / ELT),
                        row);
            tma_load_2d(vdst + bx * kSubTileBytes + pg * P * kBoxBytes, &tmv, &full[s], bx * (kBoxBytes / ELT),
                        row);
          }
        }
      }
    }
  }
  return true;
}

// Producer warp, after its last item: do not leave while copies may still land in this CTA's
// shared memory (stages older than the last NS_ were released by the consumers, so they landed).
template <int NS_>
__device__ __forceinline__ void drain_copies(const DecodeParams& p, uint64_t* full, int g, int lane) {
  if (lane == 0) {
    for (int x = max(0, g - NS_); x < g; ++x) {
      if (!mbar_wait(&full[x % NS_], (x / NS_) & 1)) {
        atomicOr(p.err, kDevErrTimeout);
        break;
      }
    }
  }
  __syncwarp();
}

// The consumer warps meet: a named barrier in the one-item kernel (non-aligned form: a warp
// counts once, after all of its threads have arrived); in the persistent kernel an mbarrier with
// a bounded wait (a consumer warp that gave up on an item never arrives, and the others must not
// wait for it forever).
template <bool PERSIST>
struct ConsumerSync {
  uint64_t* bar;
  uint32_t phase;
  int nthreads;
  __device__ __forceinline__ bool sync(int lane) {
    if constexpr (!PERSIST) {
      asm volatile("barrier.sync 1, %0;" ::"r"(nthreads) : "memory");
      return true;
    } else {
      __syncwarp();
      if (lane == 0) mbar_arrive(bar);
      const bool ok = mbar_wait(bar, phase & 1);
      ++phase;
      return ok;
    }
  }
};

// Consumer warps: one item's tiles, then the combine of the key slices and its outputs. g counts
// the stages consumed so far (across items). The one-item kernel passes its combine buffer (the
// ring, reused); the persistent kernel holds on to the item's last stage and combines in its slot,
// releasing it to the producer afterwards (obuf null). Returns false if a wait ran out.
template <int D, int KV, int NT, int NS_, bool PERSIST>
__device__ __forceinline__ bool consume_item(const DecodeParams& p, unsigned char* smem, float* obuf, float2* ml_buf,
                                             uint64_t* full, uint64_t* empty, const DecodeItem& item, int& g,
                                             ConsumerSync<PERSIST>& csync, int warp, int lane, int ncw) {
  using S = DecodeShape<D, KV>;
  constexpr int ELT = S::ELT, NBOX = S::NBOX, KSTEPS = S::KSTEPS, MTILES = S::MTILES;
  constexpr int ROWS_W = 8 * NT;  // query rows per consumer warp
  const int b = item.b, kvh = item.kvh, split = item.split, N = item.N;
  const SlabSpan sp = item.sp;
  const int nsplit_b = item.nsplit, t0 = item.t0, t1 = item.t1, ntiles = item.ntiles;
  const int R = (sp.ts1 - sp.ts0) * p.G;  // query rows of this slab
  const int rg = warp / p.nts, ts = warp % p.nts;
  const int g8 = lane >> 2, c = lane & 3;
  const int row_base = rg * ROWS_W;

  float kscale = 1.f, vscale = 1.f;
  if (KV != kKvFp16) {  // the pool's scale, or this KV head's
    kscale = p.k_scale[kvh * p.scale_stride];
    vscale = p.v_scale[kvh * p.scale_stride];
  }
  // logits in base-2 units: s2 = acc * softmax_scale * k_scale * log2(e)
  const float sc2 = p.softmax_scale * kscale * 1.4426950408889634f;

  // Q^T fragments (B operand of S^T = K Q^T), kept in registers.
  uint32_t qf[KSTEPS][NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int row = row_base + nt * 8 + g8;
    const __half* qrow = nullptr;
    if (row < R) {
      const int tl = row / p.G, j = row - tl * p.G;
      qrow = p.q + ((static_cast<size_t>(b) * p.T + sp.ts0 + tl) * p.num_q_heads + kvh * p.G + j) * D;
    }
#pragma unroll
    for (int ks = 0; ks < KSTEPS; ++ks) {
      if (qrow) {
        const uint2 v = *reinterpret_cast<const uint2*>(qrow + qk_elem(ELT, ks, c));
        qf[ks][nt][0] = v.x;
        qf[ks][nt][1] = v.y;
      } else {
        qf[ks][nt][0] = qf[ks][nt][1] = 0u;
      }
    }
  }

  // Keys every row of the slab sees: [max_lo, min_hi] (the bounds grow with the query token, so
  // they are its first token's upper and last token's lower bound). Groups inside it need no
  // masking; elsewhere each row's own bounds follow from its query token (padding rows past R
  // take the slab's last token: they are never written out).
  const int min_hi = key_hi(N, p.T, sp.ts0, p.causal);
  const int max_lo = key_lo(N, p.T, sp.ts1 - 1, p.window);

  float o[MTILES][NT][4];
#pragma unroll
  for (int i = 0; i < MTILES; ++i)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int k = 0; k < 4; ++k) o[i][nt][k] = 0.f;
  float m_run[NT][2], l_run[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      m_run[nt][e] = -CUDART_INF_F;
      l_run[nt][e] = 0.f;
    }

  bool alive = true;
  const int groups_per_stage = kTileKeys / 16;
  for (int it = 0; it < ntiles; ++it, ++g) {
    const int s = g % NS_;
    if (!mbar_wait(&full[s], (g / NS_) & 1)) {
      if (lane == 0) atomicOr(p.err, kDevErrTimeout);
      alive = false;
      g += ntiles - it;  // the stage count stays in step with the producer's
      break;
    }
    const unsigned char* Ks = smem + s * S::STAGE;
    const unsigned char* Vs = Ks + S::KV_STAGE;
    const int tile_start = t0 + it * kTileKeys;
    const int valid = min(kTileKeys, t1 - tile_start);

    for (int grp = ts; grp < groups_per_stage; grp += p.nts) {
      if (grp * 16 >= valid) break;
      const int key0 = tile_start + grp * 16;  // absolute position of key row 0 of this group

      // ---- S^T = K Q^T (NACC independent accumulator chains, summed afterwards)
      constexpr int NACC = NT == 1 ? 2 : 1;
      float sacc2[NACC][NT][4];
#pragma unroll
      for (int a = 0; a < NACC; ++a)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int k = 0; k < 4; ++k) sacc2[a][nt][k] = 0.f;
      const int r0 = grp * 16 + g8;
#pragma unroll
      for (int bx = 0; bx < NBOX; ++bx) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const unsigned char* kb = Ks + bx * kSubTileBytes;
          const uint4 k0 = lds128(kb + swz_offset(r0, k_chunk(c, h)));
          const uint4 k1 = lds128(kb + swz_offset(r0 + 8, k_chunk(c, h)));
          const uint32_t w0[4] = {k0.x, k0.y, k0.z, k0.w};
          const uint32_t w1[4] = {k1.x, k1.y, k1.z, k1.w};
          if constexpr (ELT == 1) {
#pragma unroll
            for (int w = 0; w < 4; ++w) {
              const int ks = (2 * bx + h) * 4 + w;
              uint32_t a0, a1, a2, a3;
              if constexpr (KV == kKvE4m3) {
                a0 = e4m3x2_to_f16x2(w0[w]);
                a1 = e4m3x2_to_f16x2(w1[w]);
                a2 = e4m3x2_to_f16x2(w0[w] >> 16);
                a3 = e4m3x2_to_f16x2(w1[w] >> 16);
              } else {
                a0 = e5m2_bytes_to_f16x2<0, 1>(w0[w]);
                a1 = e5m2_bytes_to_f16x2<0, 1>(w1[w]);
                a2 = e5m2_bytes_to_f16x2<2, 3>(w0[w]);
                a3 = e5m2_bytes_to_f16x2<2, 3>(w1[w]);
              }
#pragma unroll
              for (int nt = 0; nt < NT; ++nt)
                mma_16816(sacc2[w % NACC][nt], a0, a1, a2, a3, qf[ks][nt][0], qf[ks][nt][1]);
            }
          } else {
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const int ks = (2 * bx + h) * 2 + u;
#pragma unroll
              for (int nt = 0; nt < NT; ++nt)
                mma_16816(sacc2[u % NACC][nt], w0[2 * u], w1[2 * u], w0[2 * u + 1], w1[2 * u + 1], qf[ks][nt][0],
                          qf[ks][nt][1]);
            }
          }
        }
      }
      float sacc[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          float v = sacc2[0][nt][k];
#pragma unroll
          for (int a = 1; a < NACC; ++a) v += sacc2[a][nt][k];
          sacc[nt][k] = v;
        }

      // ---- scale, mask, running max
      const bool need_mask = (key0 + 15 > min_hi) || (key0 < max_lo);
      const int keyA = key0 + g8, keyB = keyA + 8;
      float mx[NT][2];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float sa = sacc[nt][e] * sc2, sb = sacc[nt][2 + e] * sc2;
          if (need_mask) {
            const int row = row_base + nt * 8 + 2 * c + e;
            const int tok = row < R ? sp.ts0 + row / p.G : sp.ts1 - 1;
            const int khi = key_hi(N, p.T, tok, p.causal);
            const int klo = key_lo(N, p.T, tok, p.window);
            if (keyA > khi || keyA < klo) sa = -CUDART_INF_F;
            if (keyB > khi || keyB < klo) sb = -CUDART_INF_F;
          }
          sacc[nt][e] = sa;
          sacc[nt][2 + e] = sb;
          mx[nt][e] = fmaxf(sa, sb);
        }
#pragma unroll
      for (int off = 4; off < 32; off <<= 1)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e) mx[nt][e] = fmaxf(mx[nt][e], __shfl_xor_sync(0xffffffffu, mx[nt][e], off));

      bool changed = false;
      float alpha[NT][2], muse[NT][2];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float mnew = fmaxf(m_run[nt][e], mx[nt][e]);
          muse[nt][e] = (mnew == -CUDART_INF_F) ? 0.f : mnew;
          alpha[nt][e] = fast_exp2(m_run[nt][e] - muse[nt][e]);  // 0 when the old max was -inf
          changed |= (mnew != m_run[nt][e]);
          m_run[nt][e] = mnew;
        }
      if (__any_sync(0xffffffffu, changed)) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            l_run[nt][e] *= alpha[nt][e];
#pragma unroll
            for (int i = 0; i < MTILES; ++i) {
              o[i][nt][e] *= alpha[nt][e];
              o[i][nt][2 + e] *= alpha[nt][e];
            }
          }
      }

      // ---- P = exp2(s - m), then P^T fragments via movmatrix
      uint32_t pb[NT][2];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        float pv[4];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          pv[e] = fast_exp2(sacc[nt][e] - muse[nt][e]);
          pv[2 + e] = fast_exp2(sacc[nt][2 + e] - muse[nt][e]);
          l_run[nt][e] += pv[e] + pv[2 + e];
        }
        pb[nt][0] = movmatrix_trans(pack_half2(pv[0], pv[1]));  // keys 0..7 of the group
        pb[nt][1] = movmatrix_trans(pack_half2(pv[2], pv[3]));  // keys 8..15
      }

      // ---- O^T += V^T P^T
      const bool v_tail = (grp * 16 + 16 > valid);
#pragma unroll
      for (int bx = 0; bx < NBOX; ++bx) {
        const unsigned char* vb = Vs + bx * kSubTileBytes;
        uint4 vr[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int r = grp * 16 + pv_key(c, i);
          vr[i] = lds128(vb + swz_offset(r, g8));
          if (v_tail && (r >= valid)) vr[i] = make_uint4(0u, 0u, 0u, 0u);  // stale bytes past the sequence end
        }
        const uint32_t W0[4] = {vr[0].x, vr[0].y, vr[0].z, vr[0].w};
        const uint32_t W1[4] = {vr[1].x, vr[1].y, vr[1].z, vr[1].w};
        const uint32_t W2[4] = {vr[2].x, vr[2].y, vr[2].z, vr[2].w};
        const uint32_t W3[4] = {vr[3].x, vr[3].y, vr[3].z, vr[3].w};
        if constexpr (ELT == 1) {
#pragma unroll
          for (int w = 0; w < 4; ++w) {
#pragma unroll
            for (int sh = 0; sh < 2; ++sh) {
              const int mt = bx * 8 + 2 * w + sh;
              // bytes (2sh, 2sh+1) of the word: element pair (d0, d0+1) of m-tile mt
              const uint32_t X = __byte_perm(W0[w], W1[w], sh ? 0x7362 : 0x5140);  // [k0 d0, k1 d0, k0 d1, k1 d1]
              const uint32_t Y = __byte_perm(W2[w], W3[w], sh ? 0x7362 : 0x5140);
              uint32_t a0, a1, a2, a3;
              if constexpr (KV == kKvE4m3) {
                a0 = e4m3x2_to_f16x2(X);
                a1 = e4m3x2_to_f16x2(X >> 16);
                a2 = e4m3x2_to_f16x2(Y);
                a3 = e4m3x2_to_f16x2(Y >> 16);
              } else {
                a0 = e5m2_bytes_to_f16x2<0, 1>(X);
                a1 = e5m2_bytes_to_f16x2<2, 3>(X);
                a2 = e5m2_bytes_to_f16x2<0, 1>(Y);
                a3 = e5m2_bytes_to_f16x2<2, 3>(Y);
              }
#pragma unroll
              for (int nt = 0; nt < NT; ++nt) mma_16816(o[mt][nt], a0, a1, a2, a3, pb[nt][0], pb[nt][1]);
            }
          }
        } else {
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            const int mt = bx * 4 + w;
            const uint32_t a0 = __byte_perm(W0[w], W1[w], 0x5410);
            const uint32_t a1 = __byte_perm(W0[w], W1[w], 0x7632);
            const uint32_t a2 = __byte_perm(W2[w], W3[w], 0x5410);
            const uint32_t a3 = __byte_perm(W2[w], W3[w], 0x7632);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) mma_16816(o[mt][nt], a0, a1, a2, a3, pb[nt][0], pb[nt][1]);
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0 && !(PERSIST && it == ntiles - 1)) mbar_arrive(&empty[s]);
  }

  const int rows_cta = min(R, p.nrg * ROWS_W);  // at most 64 (4 row groups of 16)
  const bool final_out = (nsplit_b == 1);
  const int ctid = warp * 32 + lane;  // consumer thread index
  if constexpr (PERSIST) {
    if (!alive) return false;
    if (ntiles == 0) {  // no key visible (a range of a sequence with no keys): out 0, lse -inf
      for (int idx = ctid; idx < rows_cta * (D / 4); idx += ncw * 32) {
        const int r = idx / (D / 4), d = (idx - r * (D / 4)) * 4;
        const int tl = r / p.G, j = r - tl * p.G;
        const size_t grow = (static_cast<size_t>(b) * p.T + sp.ts0 + tl) * p.num_q_heads + kvh * p.G + j;
        if (final_out) {
          *reinterpret_cast<uint2*>(p.out + grow * D + d) = make_uint2(0u, 0u);
          if (d == 0) p.lse[grow] = -CUDART_INF_F;
        } else {
          *reinterpret_cast<float4*>(p.o_part + (grow * p.num_splits + split) * D + d) = make_float4(0.f, 0.f, 0.f, 0.f);
          if (d == 0) p.lse_part[grow * p.num_splits + split] = -CUDART_INF_F;
        }
      }
      return true;
    }
    obuf = reinterpret_cast<float*>(smem + ((g - 1) % NS_) * S::STAGE);
  }

  // let the merge kernel (launched with programmatic serialisation) start while this CTA finishes
  if constexpr (!PERSIST) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  // ------------------------------------------------------------------ combine the token slices
  // full row sums of this warp
#pragma unroll
  for (int off = 4; off < 32; off <<= 1)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) l_run[nt][e] += __shfl_xor_sync(0xffffffffu, l_run[nt][e], off);

  // all consumers are done with the stage(s) that become the combine buffer
  alive = csync.sync(lane) && alive;

  float* my_o = obuf + static_cast<size_t>(warp) * ROWS_W * D;
  if (g8 == 0) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e)
        ml_buf[warp * ROWS_W + nt * 8 + 2 * c + e] = make_float2(alive ? m_run[nt][e] : -CUDART_INF_F, l_run[nt][e]);
  }
#pragma unroll
  for (int i = 0; i < MTILES; ++i) {
    const int d0 = pv_elem(ELT, i, g8);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float* rowp = my_o + (nt * 8 + 2 * c + e) * D;
        *reinterpret_cast<float2*>(rowp + d0) = make_float2(o[i][nt][e], o[i][nt][2 + e]);
      }
  }
  alive = csync.sync(lane) && alive;

  const int nts = p.nts;  // 2 or 4
  constexpr int QD = D / 4;
  const int items = rows_cta * QD;  // (row, 4 consecutive dims) items
  if (items <= ncw * 32) {
    // At most one item per consumer thread: each thread combines its item's slices itself
    // (the slices of an item are loaded together: one shared-memory round trip).
    const int idx = ctid;
    if (idx < items) {
      const int r = idx / QD;
      const int d = (idx - r * QD) * 4;
      const int rgr = r / ROWS_W, rr = r - rgr * ROWS_W;
      float2 ml[4];
      float4 v[4];
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        ml[t] = make_float2(-CUDART_INF_F, 0.f);
        v[t] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (t < nts) {
          const int wi = rgr * nts + t;
          ml[t] = ml_buf[wi * ROWS_W + rr];
          v[t] = *reinterpret_cast<const float4*>(obuf + (static_cast<size_t>(wi) * ROWS_W + rr) * D + d);
        }
      }
      const float M = fmaxf(fmaxf(ml[0].x, ml[1].x), fmaxf(ml[2].x, ml[3].x));
      float L = 0.f;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      if (M != -CUDART_INF_F) {
#pragma unroll
        for (int t = 0; t < 4; ++t) {  // slices past nts have weight 0
          const float w = (ml[t].x == -CUDART_INF_F) ? 0.f : fast_exp2(ml[t].x - M);
          L += w * ml[t].y;
          acc.x += w * v[t].x;
          acc.y += w * v[t].y;
          acc.z += w * v[t].z;
          acc.w += w * v[t].w;
        }
      }
      const bool has = (M != -CUDART_INF_F) && (L > 0.f);
      const float inv = has ? vscale / L : 0.f;
      const int tl = r / p.G, j = r - tl * p.G;
      const size_t grow = (static_cast<size_t>(b) * p.T + sp.ts0 + tl) * p.num_q_heads + kvh * p.G + j;
      // natural-log LSE from base-2 running values
      const float lse_val = has ? (M + log2f(L)) * 0.6931471805599453f : -CUDART_INF_F;
      if (final_out) {
        __half2 h01 = __floats2half2_rn(acc.x * inv, acc.y * inv);
        __half2 h23 = __floats2half2_rn(acc.z * inv, acc.w * inv);
        uint2 packed;
        packed.x = *reinterpret_cast<uint32_t*>(&h01);
        packed.y = *reinterpret_cast<uint32_t*>(&h23);
        *reinterpret_cast<uint2*>(p.out + grow * D + d) = packed;
        if (d == 0) p.lse[grow] = lse_val;
      } else {
        float* dst = p.o_part + (grow * p.num_splits + split) * D + d;
        *reinterpret_cast<float4*>(dst) = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
        if (d == 0) p.lse_part[grow * p.num_splits + split] = lse_val;
      }
    }
  } else {
    // Several items per thread (e.g. 6 rows of 256 dims over 4 warps): first, per row (one thread
    // each), the slices' weights 2^(m_t - M) folded with v_scale / L into four coefficients, the
    // row's LSE and the offset of its output row; then every item is a 4-term weighted sum of the
    // slices, with no per-item chain of exponentials, division and logarithm.
    __shared__ float4 s_coef[64];
    __shared__ long long s_orow[64];
    if (ctid < rows_cta) {
      const int r = ctid;
      const int rgr = r / ROWS_W, rr = r - rgr * ROWS_W;
      float2 ml[4];
#pragma unroll
      for (int t = 0; t < 4; ++t) ml[t] = t < nts ? ml_buf[(rgr * nts + t) * ROWS_W + rr] : make_float2(-CUDART_INF_F, 0.f);
      const float M = fmaxf(fmaxf(ml[0].x, ml[1].x), fmaxf(ml[2].x, ml[3].x));
      float w[4];
      float L = 0.f;
#pragma unroll
      for (int t = 0; t < 4; ++t) {  // slices past nts, and empty ones, have weight 0
        w[t] = (ml[t].x == -CUDART_INF_F) ? 0.f : fast_exp2(ml[t].x - M);
        L += w[t] * ml[t].y;
      }
      const bool has = (M != -CUDART_INF_F) && (L > 0.f);
      const float inv = has ? vscale / L : 0.f;
      s_coef[r] = make_float4(w[0] * inv, w[1] * inv, w[2] * inv, w[3] * inv);
      const int tl = r / p.G, j = r - tl * p.G;
      const long long grow = (static_cast<long long>(b) * p.T + sp.ts0 + tl) * p.num_q_heads + kvh * p.G + j;
      const float lse_val = has ? (M + log2f(L)) * 0.6931471805599453f : -CUDART_INF_F;
      if (final_out) {
        s_orow[r] = grow * D;
        p.lse[grow] = lse_val;
      } else {
        s_orow[r] = (grow * p.num_splits + split) * D;
        p.lse_part[grow * p.num_splits + split] = lse_val;
      }
    }
    alive = csync.sync(lane) && alive;
    for (int idx = ctid; idx < items; idx += ncw * 32) {
      const int r = idx / QD;
      const int d = (idx - r * QD) * 4;
      const int rgr = r / ROWS_W, rr = r - rgr * ROWS_W;
      const float4 cf = s_coef[r];
      const float cw[4] = {cf.x, cf.y, cf.z, cf.w};
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        if (t < nts) {
          const float4 v = *reinterpret_cast<const float4*>(obuf + (static_cast<size_t>(rgr * nts + t) * ROWS_W + rr) * D + d);
          acc.x += cw[t] * v.x;
          acc.y += cw[t] * v.y;
          acc.z += cw[t] * v.z;
          acc.w += cw[t] * v.w;
        }
      }
      const long long off = s_orow[r] + d;
      if (final_out) {
        __half2 h01 = __floats2half2_rn(acc.x, acc.y);
        __half2 h23 = __floats2half2_rn(acc.z, acc.w);
        uint2 packed;
        packed.x = *reinterpret_cast<uint32_t*>(&h01);
        packed.y = *reinterpret_cast<uint32_t*>(&h23);
        *reinterpret_cast<uint2*>(p.out + off) = packed;
      } else {
        *reinterpret_cast<float4*>(p.o_part + off) = acc;
      }
    }
  }
  if constexpr (PERSIST) {  // this warp has read the combine buffer: the slot goes back to the ring
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[(g - 1) % NS_]);
  }
  return alive;
}

// One CTA per (key range, KV head, slab, sequence).
template <int D, int KV, int NT>
__global__ void __launch_bounds__(NT == 1 ? 160 : 288, NT == 1 ? 2 : 1)
    decode_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                  const DecodeParams p) {
  using S = DecodeShape<D, KV>;
  constexpr int NS = S::NS;
  constexpr int ROWS_W = 8 * NT;

  extern __shared__ unsigned char smem_raw[];
  // 1 KB-aligned base, formed by pointer arithmetic on the shared array so that every pointer
  // derived from it stays a shared-memory pointer (32-bit shared loads and stores)
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);

  const int split = blockIdx.x, b = blockIdx.z;
  // KV head major (CTAs running together share one head's keys in L2), longest slabs first
  const int kvh = blockIdx.y / p.num_slabs;
  const int slab = p.num_slabs - 1 - static_cast<int>(blockIdx.y) % p.num_slabs;
  const int ncw = p.nrg * p.nts;

  // launched with programmatic stream serialisation: wait for the preceding
  // grid (which may produce q, the cache or the tables) before any global read
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // Without a window the range's first page does not depend on the sequence length: the
  // producer warp fetches the block-table entries of its first 32 pages now, so that the load
  // overlaps the sequence-length load (entries stay inside the table row; they are validated
  // once the length is known). With a window the fetch waits for the length.
  const int pguess = p.window > 0 ? -1 : (split * p.split_tokens) >> p.page_shift;
  int pre_id = 0;
  if ((threadIdx.x >> 5) == ncw && pguess >= 0) {
    const int m = pguess + (threadIdx.x & 31);
    if (m < p.max_blocks) pre_id = p.block_table[static_cast<size_t>(b) * p.max_blocks + m];
  }
  const int N = checked_len(p, p.seq_lens[b], threadIdx.x == 0 && split == 0 && blockIdx.y == 0);
  const DecodeItem item = make_item(p, b, kvh, slab, split, N);
  if (split >= item.nsplit) return;

  const int body_bytes = decode_smem_bytes<D, KV, NT>(ncw) - ncw * ROWS_W * 8 - 2 * NS * 8;
  float2* ml_buf = reinterpret_cast<float2*>(smem + body_bytes);  // [ncw][ROWS_W] (m, l)
  uint64_t* full = reinterpret_cast<uint64_t*>(ml_buf + ncw * ROWS_W);
  uint64_t* empty = full + NS;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], ncw);
    }
    fence_barrier_init();
  }
  __syncthreads();

  int g = 0;
  if (warp == ncw) {
    // ------------------------------------------------------------------ producer
    // The whole warp walks the tiles; its 32 lanes fetch 32 consecutive page ids of the range at
    // a time (one coalesced load instead of a chain of dependent ones) and lane 0 issues the
    // copies, reading ids by shuffle.
    if (item.ntiles > 0) {
      if (lane == 0) {
        prefetch_tensormap(&tmk);
        prefetch_tensormap(&tmv);
      }
      produce_item<D, KV, NS>(tmk, tmv, p, smem, full, empty, item, g, pguess, pre_id, lane);
      drain_copies<NS>(p, full, g, lane);
    }
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    return;
  }
  // ------------------------------------------------------------------ consumers
  // the combine buffer [ncw][ROWS_W][D] reuses the stage ring
  ConsumerSync<false> csync{nullptr, 0u, ncw * 32};
  consume_item<D, KV, NT, NS, false>(p, smem, reinterpret_cast<float*>(smem), ml_buf, full, empty, item, g, csync,
                                     warp, lane, ncw);
}

// sequences whose last ranges the persistent grid orders by length
constexpr int kSortSeqs = 256;

// One wave of CTAs over the items that have work: the (sequence, KV head, range) triples, full
// ranges first (see decode_item below); CTA c starts with item c and then takes item numbers
// from a counter the call zeroed. The producer warp claims them and hands each to the
// consumer warps through a two-slot mailbox; the copy ring runs on across items.
// (head dim 128: registers for three CTAs per SM, as many as its shared memory allows)
template <int D, int KV, int NT>
__global__ void __launch_bounds__(NT == 1 ? 160 : 288, NT == 1 ? (D == 128 ? 3 : 2) : 1)
    decode_persist_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                          const DecodeParams p) {
  using S = DecodeShape<D, KV>;
  constexpr int NS = S::NS;
  constexpr int ROWS_W = 8 * NT;
  // one row group of 4 key slices; its combine buffer [4][ROWS_W][D] fits a stage
  static_assert(4 * ROWS_W * D * 4 <= S::STAGE, "combine buffer larger than a stage");

  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int ncw = p.nrg * p.nts;
  const int B = p.num_seqs;
  float2* ml_buf = reinterpret_cast<float2*>(smem + NS * S::STAGE);  // [ncw][ROWS_W]
  uint64_t* full = reinterpret_cast<uint64_t*>(ml_buf + ncw * ROWS_W);
  uint64_t* empty = full + NS;
  uint64_t* item_full = empty + NS;    // [2] producer -> consumers: mailbox slot written
  uint64_t* item_free = item_full + 2;  // [2] consumers -> producer: mailbox slot read
  uint64_t* cons_bar = item_free + 2;   // the consumer warps' rendezvous
  int* item_slot = reinterpret_cast<int*>(cons_bar + 1);  // [2] mailbox
  int* lens = item_slot + 2;                              // [B] validated lengths
  int* nsp = lens + B;                                    // [B] ranges per KV head of sequence b
  int* prefix = nsp + B;                                  // [B + 1] first leading item of sequence b

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], ncw);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&item_full[i], 1);
      mbar_init(&item_free[i], ncw);
    }
    mbar_init(cons_bar, ncw);
    fence_barrier_init();
  }
  // the lengths, the range counts, and the prefix of the leading items per sequence (warp 0, 32
  // sequences at a time)
  if (warp == 0) {
    int run = 0;
    for (int base = 0; base < B; base += 32) {
      const int bb = base + lane;
      int n = 0, cnt = 0, ns = 1;
      if (bb < B) {
        n = checked_len(p, p.seq_lens[bb], blockIdx.x == 0);
        ns = span_splits(slab_span(n, p.T, 0, p.slab_tokens, p.causal, p.window, kTileKeys), p.split_tokens);
        cnt = (ns - 1) * p.num_kv_heads;
      }
      int incl = cnt;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += v;
      }
      if (bb < B) {
        lens[bb] = n;
        nsp[bb] = ns;
        prefix[bb + 1] = run + incl;
      }
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) prefix[0] = 0;
  }
  __syncthreads();
  // Items: first every range but the last of each (sequence, KV head) -- full split_tokens
  // ranges -- numbered sequence-major from prefix[b]; then the last ranges, Hkv per sequence,
  // whose lengths vary, longest first (for up to kSortSeqs sequences; sequence order beyond),
  // so that the CTAs finish on short items.
  const int leading = prefix[B];
  const int total = leading + B * p.num_kv_heads;
  __shared__ int s_last[kSortSeqs], s_order[kSortSeqs];  // last-range keys; sequences by it
  const bool sorted = B <= kSortSeqs;
  if (sorted) {
    for (int bb = threadIdx.x; bb < B; bb += blockDim.x) {
      const SlabSpan sp = slab_span(lens[bb], p.T, 0, p.slab_tokens, p.causal, p.window, kTileKeys);
      s_last[bb] = sp.hi >= sp.lo ? sp.hi - sp.base - (nsp[bb] - 1) * p.split_tokens + 1 : 0;
    }
    __syncthreads();
    for (int bb = threadIdx.x; bb < B; bb += blockDim.x) {  // rank: longer first, ties by index
      const int mine = s_last[bb];
      int rank = 0;
      for (int o = 0; o < B; ++o) {
        const int t = s_last[o];
        rank += (t > mine || (t == mine && o < bb)) ? 1 : 0;
      }
      s_order[rank] = bb;
    }
    __syncthreads();
  }
  auto decode_item = [&](int i) -> DecodeItem {
    if (i >= leading) {
      const int j = i - leading;
      const int jb = j / p.num_kv_heads;
      const int bb = sorted ? s_order[jb] : jb;
      return make_item(p, bb, j - jb * p.num_kv_heads, 0, nsp[bb] - 1, lens[bb]);
    }
    // the last sequence whose first leading item is <= i
    int lo = 0, hi = B - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (prefix[mid] <= i) {
        lo = mid;
      } else {
        hi = mid - 1;
      }
    }
    const int per = nsp[lo] - 1;  // leading ranges per KV head (at least 1 here)
    const int local = i - prefix[lo];
    return make_item(p, lo, local / per, 0, local % per, lens[lo]);
  };

  int g = 0;
  if (warp == ncw) {
    // ------------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensormap(&tmk);
      prefetch_tensormap(&tmv);
    }
    for (int k = 0;; ++k) {
      // The first item is the CTA's own index; later ones are claimed once the previous item's
      // copies are all issued (the consumers still have a ring of stages to work through while
      // the claim and the first page ids are fetched). Each CTA that had a first item makes one
      // claim past the end, so the counter ends at the number of items.
      int i = static_cast<int>(blockIdx.x);
      if (k > 0) {
        if (lane == 0) i = static_cast<int>(gridDim.x) + atomicAdd(p.work_ctr, 1);
        i = __shfl_sync(0xffffffffu, i, 0);
      }
      // mailbox slot k & 1 is free once the consumers read item k - 2 (sound: this warp waited for
      // that barrier's previous phase, of item k - 4, before writing item k - 2)
      if (k >= 2) {
        bool got = true;
        if (lane == 0) got = mbar_wait(&item_free[k & 1], ((k >> 1) - 1) & 1);
        if (!__shfl_sync(0xffffffffu, got, 0)) {
          if (lane == 0) atomicOr(p.err, kDevErrTimeout);
          break;
        }
      }
      if (lane == 0) {
        item_slot[k & 1] = i < total ? i : -1;
        mbar_arrive(&item_full[k & 1]);
      }
      if (i >= total) break;
      const DecodeItem item = decode_item(i);
      if (!produce_item<D, KV, NS>(tmk, tmv, p, smem, full, empty, item, g, -1, 0, lane)) break;
    }
    drain_copies<NS>(p, full, g, lane);
    return;
  }
  // ------------------------------------------------------------------ consumers
  ConsumerSync<true> csync{cons_bar, 0u, ncw * 32};
  for (int k = 0;; ++k) {
    // item k's mailbox slot (sound: this warp waited for its previous phase, of item k - 2)
    if (!mbar_wait(&item_full[k & 1], (k >> 1) & 1)) {
      if (lane == 0) atomicOr(p.err, kDevErrTimeout);
      break;
    }
    const int i = item_slot[k & 1];
    __syncwarp();
    if (lane == 0) mbar_arrive(&item_free[k & 1]);
    if (i < 0) break;
    const DecodeItem item = decode_item(i);
    if (!consume_item<D, KV, NT, NS, true>(p, smem, nullptr, ml_buf, full, empty, item, g, csync, warp, lane, ncw)) {
      if (lane == 0) atomicOr(p.err, kDevErrTimeout);
      break;
    }
  }
  // every item of this CTA written: the merge kernel may start
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

}  // namespace pfkv
