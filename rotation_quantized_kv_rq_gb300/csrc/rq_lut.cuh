// Code-pair lookup tables shared by the attention kernels: one shared-memory load turns an
// index byte that carries two codes into the half2 of their centroids.
//
// Entry e of a table is the half2 (c[code_a], c[code_b]) of the two codes index byte e carries:
//   T4 (4-bit):  code_a = e & 15,                       code_b = e >> 4
//   T1 (3-bit):  code_a = (e & 3) | (e >> 4 & 1) << 2,   code_b = (e >> 2 & 3) | (e >> 5 & 1) << 2
//   T2 (3-bit):  code_a = (e >> 4 & 3) | (e & 1) << 2,   code_b = (e >> 6 & 3) | (e >> 1 & 1) << 2
//   U1 (2-bit):  code_a = e & 3,                        code_b = e >> 4 & 3
//   U2 (2-bit):  code_a = e >> 2 & 3,                   code_b = e >> 6 & 3
// The 3-bit tables fit the split storage of a 32-dim group (low bits in W0 / W1, high bits in
// W2): bit-selecting nibbles of W0 / W1 and W2 gives bytes whose T1 / T2 entries are pairs of
// dims, see the kernels.  Row e of the 64 KB table holds 64 words: for 3- and 4-bit codes word
// l (l < 32) is the first table's entry for lane l and word 32 + l the second table's (T2; a
// copy of T4 for 4-bit); for 2-bit codes words 2l, 2l + 1 are lane l's U1 and U2 entries, so
// one 8-byte load gets both (both tables' entries of an index byte are always wanted together
// at 2 bits).  Either way every lane reads its own banks, so no lookup ever conflicts.
#pragma once
#include <cuda_fp16.h>
#include <stdint.h>

namespace rq {
namespace lut {

constexpr int kBytes = 256 * 256;  // 256 index bytes x (2 tables x 32 lanes x 4 B)

// Fills the table at `table` (16-byte aligned) from the centroids cb[2^BITS] (already in shared
// memory): each row holds 2 distinct words, written as 16-byte stores of four copies, a warp
// covering 512 consecutive bytes (two rows) per store.  Threads tid = 0 .. nthreads - 1.
template <int BITS>
__device__ __forceinline__ void fill(uint32_t* table, const float* cb, int tid, int nthreads) {
  uint4* t4 = reinterpret_cast<uint4*>(table);
  if constexpr (BITS == 2) {  // (U1, U2) pairs of lanes 2m, 2m + 1 per 16-byte store
    for (int i = tid; i < 256 * 16; i += nthreads) {
      const int e = i >> 4;
      const __half2 h1 = __floats2half2_rn(cb[e & 3], cb[(e >> 4) & 3]);
      const __half2 h2 = __floats2half2_rn(cb[(e >> 2) & 3], cb[(e >> 6) & 3]);
      const uint32_t w1 = *reinterpret_cast<const uint32_t*>(&h1), w2 = *reinterpret_cast<const uint32_t*>(&h2);
      t4[i] = make_uint4(w1, w2, w1, w2);
    }
  } else {
  for (int i = tid; i < 256 * 16; i += nthreads) {
    const int e = i >> 4, second = (i >> 3) & 1;
    int ca, cbx;
    if (BITS == 4) {
      ca = e & 15;
      cbx = e >> 4;
    } else if (!second) {
      ca = (e & 3) | ((e >> 4) & 1) << 2;
      cbx = ((e >> 2) & 3) | ((e >> 5) & 1) << 2;
    } else {
      ca = ((e >> 4) & 3) | (e & 1) << 2;
      cbx = ((e >> 6) & 3) | ((e >> 1) & 1) << 2;
    }
    const __half2 hv = __floats2half2_rn(cb[ca], cb[cbx]);
    const uint32_t w = *reinterpret_cast<const uint32_t*>(&hv);
    t4[i] = make_uint4(w, w, w, w);
  }
  }
}

// The table starts at a 64 KB-aligned shared address A, so an entry's address A + e * 256 +
// (lane's offset) has byte 0 = the lane's offset (lane * 4, + 128 for the second table; lane * 8,
// + 4 for U2, at 2 bits), byte 1 = e and bytes 2-3 = A's: one byte permute of (x, key) with
// key = A | offset forms it, with no add.
template <int BITS>
__device__ __forceinline__ uint32_t key(uint32_t table_saddr, int lane, int second) {
  return BITS == 2 ? table_saddr | ((uint32_t)lane * 8u) | (second ? 4u : 0u)
                   : table_saddr | ((uint32_t)lane * 4u) | (second ? 128u : 0u);
}
// Half2 of the two codes in byte j (0..3, a compile-time constant after unrolling) of index
// word x, from the table that `key` selects.
__device__ __forceinline__ uint32_t get(uint32_t x, int j, uint32_t k) {
  uint32_t addr, v;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(addr) : "r"(x), "r"(k), "r"(0x7604u | ((uint32_t)j << 4)));
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

// 2-bit codes: the (U1, U2) pair of byte j of index word x, with key = key<2>(A, lane, 0).
__device__ __forceinline__ void get2(uint32_t x, int j, uint32_t k, uint32_t& u1, uint32_t& u2) {
  uint32_t addr;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(addr) : "r"(x), "r"(k), "r"(0x7604u | ((uint32_t)j << 4)));
  asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(u1), "=r"(u2) : "r"(addr));
}

}  // namespace lut
}  // namespace rq
