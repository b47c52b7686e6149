// Fragment and shared-memory layout of the decode kernel's K/V tiles.
//
// Plain C++ (usable from host code): the decode kernel uses these functions
// to address shared memory and global Q, and csrc/layout_check.cpp
// verifies on the host that every mapping is a bijection, stays in bounds
// and is free of shared-memory bank conflicts.
//
// Tiles. One pipeline stage holds TT = 64 consecutive keys of one
// (sequence, KV head). A key's row of K (D elements, ELT bytes each) is
// split into NBOX = D*ELT/128 boxes of 128 bytes; box bx of the 64 rows
// forms a sub-tile of 64 x 128 bytes written by one (or, for small pages,
// several) TMA tile copies with the 128-byte swizzle, under which the
// 16-byte chunk x of row r is stored at chunk x ^ (r & 7).
//
// Warp-level products (mma.m16n8k16, f16 inputs, f32 accumulators).
// Lanes are named (g, c) = (lane / 4, lane % 4).
//
//  S^T = K Q^T : M = 16 keys, N = 8 query rows, K = 16 head-dim elements.
//    A (keys x dims):   lane (g, c) supplies key rows g and g + 8. For its
//                       logical k in {2c, 2c+1, 2c+8, 2c+9} of k-step ks it
//                       reads 4 consecutive elements of the row starting at
//                       qk_elem(ELT, ks, c) (fp8) -- the k <-> element map
//                       differs from the identity, which is harmless because
//                       Q^T (B) is read with the same map.
//    B (dims x rows):   Q rows, same element map; one 8-byte global load
//                       per (k-step, n-tile).
//  O^T = V^T P^T : M = 16 head-dim elements, N = 8 query rows, K = 16 keys.
//    A (dims x keys):   lane (g, c) supplies keys {2c, 2c+1, 2c+8, 2c+9} of
//                       the 16-key group (identity map: the P^T fragments are
//                       the S^T accumulators moved with movmatrix.trans, which
//                       keeps key indices), and the 16-byte chunk g of every
//                       box of those key rows. Output m-tile mt covers the
//                       elements pv_elem(ELT, mt, g) (row g of the tile) and
//                       pv_elem(...) + 1 (row g + 8).
#pragma once

#ifdef __CUDACC__
#define PFKV_HD __host__ __device__ __forceinline__
#else
#define PFKV_HD inline
#endif

namespace pfkv {

constexpr int kTileKeys = 64;   // keys per pipeline stage
constexpr int kBoxBytes = 128;  // swizzle span and TMA box width in bytes
constexpr int kSubTileBytes = kTileKeys * kBoxBytes;  // one box column of a stage

// Byte offset inside a 64 x 128 B sub-tile of chunk `chunk` (0..7) of row `row`.
PFKV_HD int swz_offset(int row, int chunk) { return row * kBoxBytes + ((chunk ^ (row & 7)) << 4); }

// Number of QK k-steps whose A fragments one 16-byte K chunk provides.
PFKV_HD int ksteps_per_chunk(int elt) { return elt == 1 ? 4 : 2; }

// K chunk (box bx, half h) read by lane c, as a chunk index within the box.
PFKV_HD int k_chunk(int c, int h) { return 2 * c + h; }

// First element (of 4 consecutive, fp8; of 2 + 2, fp16) of a key row that
// lane c feeds into k-step ks. k-steps are numbered chunk-major:
// ks = (2*bx + h) * ksteps_per_chunk + w.
PFKV_HD int qk_elem(int elt, int ks, int c) {
  const int kpc = ksteps_per_chunk(elt);
  const int chunk_id = ks / kpc;  // 2*bx + h
  const int w = ks % kpc;
  const int bx = chunk_id >> 1, h = chunk_id & 1;
  const int elems_per_box = kBoxBytes / elt;
  const int elems_per_chunk = 16 / elt;
  return bx * elems_per_box + k_chunk(c, h) * elems_per_chunk + 4 * w;
}

// Element index of logical k (0..15) of k-step ks for lane c = k/2 % 4:
// k in {2c, 2c+1} -> qk_elem + (k - 2c); k in {2c+8, 2c+9} -> qk_elem + 2 + (k - 2c - 8).
PFKV_HD int qk_logical_elem(int elt, int ks, int k) {
  const int c = (k & 7) >> 1;
  const int hi = k >= 8;
  return qk_elem(elt, ks, c) + 2 * hi + (k & 1);
}

// PV m-tile mt (0 .. D/16-1): element of its row g (row g + 8 is this + 1).
PFKV_HD int pv_elem(int elt, int mt, int g) {
  const int per_box = (kBoxBytes / elt) / 16;  // m-tiles per box: 8 (fp8), 4 (fp16)
  const int bx = mt / per_box, i = mt % per_box;
  return bx * (kBoxBytes / elt) + g * (16 / elt) + 2 * i;
}

// Keys (0..15 within the 16-key group) whose V rows lane c loads, in the
// order of the PV A fragment: {2c, 2c+1, 2c+8, 2c+9}.
PFKV_HD int pv_key(int c, int i) { return 2 * c + (i & 1) + 8 * (i >> 1); }

}  // namespace pfkv
