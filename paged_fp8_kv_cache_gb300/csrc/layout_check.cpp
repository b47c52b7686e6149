// Host-side check of the decode kernel's fragment / shared-memory layout
// (frag_layout.h). Built with the host compiler and run by the CPU test
// suite; exits non-zero with a message on the first violation.
//
// Checked for fp8 (1-byte) and fp16 (2-byte) caches, head_dim 128 and 256:
//  * the QK k <-> element map of every k-step is a bijection onto 16
//    elements and the k-steps together cover the head dim exactly once;
//  * the bytes each lane loads for its K fragment are exactly the elements
//    the map assigns to it, and likewise for the PV (V) fragments and the
//    output element map;
//  * every shared-memory address stays inside its 64 x 128 B sub-tile;
//  * 16-byte loads are bank-conflict free: each group of 8 lanes (one
//    shared-memory wavefront) touches 8 distinct 16-byte bank groups.
#include <cstdio>
#include <cstdlib>
#include <set>
#include <vector>

#include "frag_layout.h"
#include "verify_layout.h"

using namespace pfkv;

static int g_fail = 0;
#define CHECK(cond, ...)                 \
  do {                                   \
    if (!(cond)) {                       \
      std::fprintf(stderr, __VA_ARGS__); \
      std::fprintf(stderr, "\n");        \
      g_fail = 1;                        \
      return;                            \
    }                                    \
  } while (0)

static void check_layout(int elt, int D) {
  const int nbox = D * elt / kBoxBytes;
  const int ksteps = D / 16;
  // QK map: bijection per k-step, disjoint cover of [0, D)
  std::set<int> all;
  for (int ks = 0; ks < ksteps; ++ks) {
    std::set<int> one;
    for (int k = 0; k < 16; ++k) {
      const int e = qk_logical_elem(elt, ks, k);
      CHECK(e >= 0 && e < D, "elt %d D %d: k-step %d k %d -> element %d out of range", elt, D, ks, k, e);
      one.insert(e);
      all.insert(e);
    }
    CHECK(one.size() == 16, "elt %d D %d: k-step %d maps to %zu elements", elt, D, ks, one.size());
  }
  CHECK(static_cast<int>(all.size()) == D, "elt %d D %d: QK map covers %zu elements", elt, D, all.size());

  // K fragment loads: lane c, box bx, half h -> chunk bytes; element of each word
  const int kpc = ksteps_per_chunk(elt);
  for (int c = 0; c < 4; ++c)
    for (int bx = 0; bx < nbox; ++bx)
      for (int h = 0; h < 2; ++h)
        for (int w = 0; w < kpc; ++w) {
          const int ks = (2 * bx + h) * kpc + w;
          const int byte = bx * kBoxBytes + k_chunk(c, h) * 16 + (elt == 1 ? 4 * w : 8 * w);
          const int elem = byte / elt;
          CHECK(elem == qk_elem(elt, ks, c), "elt %d D %d: K word of lane c=%d ks=%d at element %d, map says %d", elt,
                D, c, ks, elem, qk_elem(elt, ks, c));
          // logical k = 2c + e (e = 0, 1) and 2c + 8 + e are the 4 consecutive elements
          for (int e = 0; e < 2; ++e) {
            CHECK(qk_logical_elem(elt, ks, 2 * c + e) == elem + e, "elt %d: low pair mismatch", elt);
            CHECK(qk_logical_elem(elt, ks, 2 * c + 8 + e) == elem + 2 + e, "elt %d: high pair mismatch", elt);
          }
        }

  // PV / output map: pv_elem(mt, g) and +1 cover [0, D) once
  std::set<int> pv;
  for (int mt = 0; mt < D / 16; ++mt)
    for (int g = 0; g < 8; ++g) {
      const int e = pv_elem(elt, mt, g);
      CHECK(e >= 0 && e + 1 < D + 1, "pv element out of range");
      CHECK(pv.insert(e).second && pv.insert(e + 1).second, "elt %d D %d: pv element %d repeated", elt, D, e);
    }
  CHECK(static_cast<int>(pv.size()) == D, "elt %d D %d: PV map covers %zu", elt, D, pv.size());
  // V chunk g of box bx, word w: elements the kernel feeds to m-tile mt
  for (int bx = 0; bx < nbox; ++bx)
    for (int g = 0; g < 8; ++g)
      for (int w = 0; w < 4; ++w) {
        if (elt == 1) {
          for (int sh = 0; sh < 2; ++sh) {
            const int mt = bx * 8 + 2 * w + sh;
            const int elem = bx * kBoxBytes + g * 16 + 4 * w + 2 * sh;
            CHECK(elem == pv_elem(elt, mt, g), "fp8 V word mismatch bx %d g %d w %d sh %d", bx, g, w, sh);
          }
        } else {
          const int mt = bx * 4 + w;
          const int elem = (bx * kBoxBytes + g * 16 + 4 * w) / 2;
          CHECK(elem == pv_elem(elt, mt, g), "fp16 V word mismatch bx %d g %d w %d", bx, g, w);
        }
      }

  // keys of the PV fragment: {2c, 2c+1, 2c+8, 2c+9}, disjoint across c, covering 0..15
  std::set<int> keys;
  for (int c = 0; c < 4; ++c)
    for (int i = 0; i < 4; ++i) CHECK(keys.insert(pv_key(c, i)).second, "pv key repeated");
  CHECK(keys.size() == 16, "pv keys do not cover 16");

  // shared-memory bounds and bank conflicts of the 16-byte loads
  for (int grp = 0; grp < kTileKeys / 16; ++grp) {
    // K: rows grp*16 + g (and + 8), chunk 2c + h
    for (int half = 0; half < 2; ++half)
      for (int h = 0; h < 2; ++h)
        for (int quarter = 0; quarter < 4; ++quarter) {
          std::set<int> banks;
          for (int l = 8 * quarter; l < 8 * quarter + 8; ++l) {
            const int g = l >> 2, c = l & 3;
            const int row = grp * 16 + g + 8 * half;
            const int off = swz_offset(row, k_chunk(c, h));
            CHECK(off >= 0 && off + 16 <= kSubTileBytes, "K offset %d out of the sub-tile", off);
            banks.insert((off >> 4) & 7);
          }
          CHECK(banks.size() == 8, "K load grp %d half %d h %d quarter %d: %zu bank groups", grp, half, h, quarter,
                banks.size());
        }
    // V: rows grp*16 + pv_key(c, i), chunk g
    for (int i = 0; i < 4; ++i)
      for (int quarter = 0; quarter < 4; ++quarter) {
        std::set<int> banks;
        for (int l = 8 * quarter; l < 8 * quarter + 8; ++l) {
          const int g = l >> 2, c = l & 3;
          const int row = grp * 16 + pv_key(c, i);
          const int off = swz_offset(row, g);
          CHECK(off >= 0 && off + 16 <= kSubTileBytes, "V offset %d out of the sub-tile", off);
          banks.insert((off >> 4) & 7);
        }
        CHECK(banks.size() == 8, "V load grp %d i %d quarter %d: %zu bank groups", grp, i, quarter, banks.size());
      }
  }
}

// Pages smaller than a stage: page pg of a stage lands at row pg * P of each
// sub-tile, which must keep the 1024-byte alignment the swizzle assumes.
static void check_small_pages() {
  for (int P = 16; P < kTileKeys; P *= 2)
    for (int pg = 0; pg < kTileKeys / P; ++pg) {
      const int off = pg * P * kBoxBytes;
      CHECK(off % 1024 == 0, "page %d of size %d lands at %d (not 1024-aligned)", pg, P, off);
      CHECK(off + P * kBoxBytes <= kSubTileBytes, "page %d of size %d overflows the sub-tile", pg, P);
    }
}

// The grouped verifier's P^T buffer (verify_layout.h), for 32, 48 and 64 padded rows:
//  * (row, key) -> byte offset is a bijection onto the buffer's 2 x nmax x 128 bytes;
//  * the softmax threads' hoisted addressing holds: for rbase in {0, nmax/2} and c a multiple of
//    8, row rbase + c + j of a key is its row rbase + j shifted by c * 128 bytes (the swizzle
//    phase of a row is its index mod 8);
//  * one warp's stores of one row (32 consecutive keys of a 64-key block) touch 16 distinct
//    4-byte banks, two lanes per word: one shared-memory wavefront.
static void check_pt_layout() {
  for (int nmax : {32, 48, 64}) {
    const int bytes = 2 * nmax * 128;
    std::vector<int> seen(bytes / 2, 0);
    for (int row = 0; row < nmax; ++row)
      for (int key = 0; key < 128; ++key) {
        const int off = pt_elem(nmax, row, key);
        CHECK(off >= 0 && off + 2 <= bytes && off % 2 == 0, "P^T nmax %d: (row %d, key %d) at %d", nmax, row, key,
              off);
        CHECK(seen[off / 2]++ == 0, "P^T nmax %d: (row %d, key %d) reuses byte %d", nmax, row, key, off);
      }
    for (int rbase : {0, nmax / 2})
      for (int key = 0; key < 128; ++key)
        for (int c = 0; c < nmax / 2; c += 8)
          for (int j = 0; j < 8; ++j)
            CHECK(pt_elem(nmax, rbase + c + j, key) == pt_elem(nmax, rbase + j, key) + 128 * c,
                  "P^T nmax %d: hoisted address of row %d, key %d", nmax, rbase + c + j, key);
    for (int row = 0; row < nmax; ++row)
      for (int first = 0; first < 128; first += 32) {
        std::set<int> words, banks;
        for (int lane = 0; lane < 32; ++lane) {
          const int w = pt_elem(nmax, row, first + lane) / 4;
          words.insert(w);
          banks.insert(w % 32);
        }
        CHECK(words.size() == 16 && banks.size() == 16, "P^T nmax %d: row %d keys %d.. span %zu words, %zu banks",
              nmax, row, first, words.size(), banks.size());
      }
  }
}

int main() {
  for (int elt = 1; elt <= 2; ++elt)
    for (int D : {128, 256}) check_layout(elt, D);
  check_small_pages();
  check_pt_layout();
  if (g_fail) return 1;
  std::printf("layout ok\n");
  return 0;
}
