// Shared-memory layout of the grouped verifier's P^T operand (the B operand of
// O^T = V^T P^T on the 5th-generation tensor cores): per P^T buffer, the
// 128 keys of a tile in two 64-key blocks of NMAX rows, each row 64 fp16
// elements (128 bytes) in the K-major 128-byte-swizzled form, 8-row groups
// 1024 bytes apart. Host and device: the CPU layout check (layout_check.cpp)
// verifies the properties the kernel relies on.
#pragma once

#include "frag_layout.h"

namespace pfkv {

// byte offset of 16-bit element (row, k) in a K-major 128B-swizzled block of 64-element rows
PFKV_HD int sw128_elem(int row, int k) { return row * 128 + ((((k >> 3) ^ row) & 7) << 4) + ((k & 7) << 1); }

// byte offset of P^T element (row, key) in one buffer of nmax rows: 64-key blocks of nmax * 128 bytes
PFKV_HD int pt_elem(int nmax, int row, int key) { return (key >> 6) * nmax * 128 + sw128_elem(row, key & 63); }

}  // namespace pfkv
