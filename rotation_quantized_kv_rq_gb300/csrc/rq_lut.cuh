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
// dims, see the kernels.  Row e of the 64 KB table holds 64 words: word l (l < 32) is the first
// table's entry for lane l, word 32 + l the second table's (T2 for 3-bit, U2 for 2-bit; a copy
// of T4 for 4-bit) -- every lane reads its own bank, so no lookup ever conflicts.
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
  for (int i = tid; i < 256 * 16; i += nthreads) {
    const int e = i >> 4, second = (i >> 3) & 1;
    int ca, cbx;
    if (BITS == 4) {
      ca = e & 15;
      cbx = e >> 4;
    } else if (BITS == 2) {
      ca = second ? (e >> 2) & 3 : e & 3;
      cbx = second ? (e >> 6) & 3 : (e >> 4) & 3;
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

// The table starts at a 64 KB-aligned shared address A, so an entry's address
// A + e * 256 + lane * 4 (+ 128) has byte 0 = lane * 4 (+ 128), byte 1 = e and bytes 2-3 = A's:
// one byte permute of (x, key) with key = A | lane * 4 (+ 128) forms it, with no add.
__device__ __forceinline__ uint32_t key(uint32_t table_saddr, int lane, int second) {
  return table_saddr | ((uint32_t)lane * 4u) | (second ? 128u : 0u);
}
// Half2 of the two codes in byte j (0..3, a compile-time constant after unrolling) of index
// word x, from the table that `key` selects.
__device__ __forceinline__ uint32_t get(uint32_t x, int j, uint32_t k) {
  uint32_t addr, v;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(addr) : "r"(x), "r"(k), "r"(0x7604u | ((uint32_t)j << 4)));
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

}  // namespace lut
}  // namespace rq
