// Fused quantize-pack-append ("SGLang 1-Bit Turbo" README, section "RotorQuant KV Cache
// Compression": norm, fixed data-oblivious rotation -- 2D Givens pairs or 4D quaternion
// blocks -- then Lloyd-Max scalar codes, bit-packed into the paged cache; section "TurboQuant
// KV Cache Compression" for the dense random rotation).
//
// Structured rotations (planar / iso): work item = one (token, kv head).  A half-warp takes
// items in a grid-stride loop: its lanes 0-7 encode the K vector and lanes 8-15 the V vector,
// lane l owning dimensions 16l..16l+15 -- eight whole Givens pairs or four whole quaternion
// blocks -- so the rotation is lane-local and only the squared norm is reduced (xor-shuffles
// within the eight lanes).  Each lane reads 32 bytes, the next item's loaded while the current
// one is coded, and writes its share of the packed codes in one store.  Per item: 512 bytes of
// fp16 in, 2 * (16 * bits + 2) bytes out.
//
// Dense rotation: Y = X R^T for a tile of 32 vectors of one (kv head, K or V) is a small GEMM
// (32 x 128 x 128) on the tensor cores, two CTAs per SM so that one's GEMM overlaps the other's
// coding.  X is fp16 and exact as an operand; R (fp32) is split
// as R = hi + lo with hi = fp16(R), lo = fp16(R - hi), both multiplied into one fp32
// accumulator.  That carries R to ~6e-8 per entry, but the tensor cores' fp32 accumulation is
// not correctly rounded, so a coordinate whose u lies within kFixBand of a boundary is
// recomputed exactly -- a compensated fp32 dot product (error-free products and sums) against
// the fp32 R, shared by the vector's half-warp -- before it is coded.  Codes then differ from
// the fp64 definition only as rarely as the structured kernel's.  The coding epilogue is the
// one the structured kernel uses, on Y staged in shared memory.
#include <cuda_fp16.h>

#include "rq_codec.cuh"
#include "rq_internal.h"
#include "../../include/rq.h"

namespace rq {
namespace {

using namespace codec;

constexpr int kAppendThreads = 256;
constexpr int kAppendCtasPerSm = 3;  // 85 registers a thread: a lane's 16 parameters, inputs and outputs

// slot -> (page, offset): a shift and a mask for the usual power-of-two page sizes (decided once
// per thread; the division is a longer instruction sequence), else a division.
struct PageSplit {
  int P, shift;  // shift < 0: P is not a power of two
  __device__ explicit PageSplit(int page_size) : P(page_size), shift(-1) {
    if ((page_size & (page_size - 1)) == 0) {  // page sizes are at most 256
      shift = 0;
      while ((1 << shift) < page_size) ++shift;
    }
  }
  __device__ __forceinline__ void operator()(int slot, int& page, int& off) const {
    if (shift >= 0) {
      page = slot >> shift;
      off = slot & (P - 1);
    } else {
      page = slot / P;
      off = slot - page * P;
    }
  }
};

// ---------------------------------------------------------------------------------------
// Structured rotations
// ---------------------------------------------------------------------------------------
// A half-warp takes one item (token t, kv head h) at a time: lanes 0-7 of the half code its K
// vector and lanes 8-15 its V vector, lane l owning dims 16l .. 16l + 15 (eight Givens pairs or
// four quaternion blocks, so the rotation stays lane-local).  Per vector: one 3-step shuffle
// reduction of the squared norm, then each lane codes its 16 dims and writes its share of the
// packed bytes as one store: 4-bit, the 8-byte unit of its 16-dim group (K: bytes 8l.., V: the
// unit's token-pair slot); 2-bit, its 4-byte unit likewise; 3-bit, the low-bit word of half l & 1
// of 32-dim group l >> 1, with the group's high-bit word W2 assembled from the two lanes of the
// group by one shuffle and stored by the even lane.

// The 16 codes of a lane, from its rotated coordinates y and 1 / norm, as the words it stores:
// 4-bit, w0 = dims 0-7 and w1 = dims 8-15 as nibbles; 2-bit, w0 = 16 two-bit fields; 3-bit,
// w0 = the 16 low-bit fields and w1 = the lane's high bits at their W2 positions for half hh.
// The code is the select-tree search of code_of, whose decisions are the code's bits (most
// significant first); each decision is set straight into its packed position.
template <int BITS>
__device__ __forceinline__ void code16(const float (&y)[16], float rcp, const float (&b)[15], int hh,
                                       uint32_t& w0, uint32_t& w1) {
  w0 = 0u;
  w1 = 0u;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float u = y[i] * rcp;
    if constexpr (BITS == 4) {
      const bool s3 = u > b[7];
      const bool s2 = u > (s3 ? b[11] : b[3]);
      const bool s1 = u > (s3 ? (s2 ? b[13] : b[9]) : (s2 ? b[5] : b[1]));
      const float m0 = s3 ? (s2 ? (s1 ? b[14] : b[12]) : (s1 ? b[10] : b[8]))
                          : (s2 ? (s1 ? b[6] : b[4]) : (s1 ? b[2] : b[0]));
      const bool s0 = u > m0;
      uint32_t& w = i < 8 ? w0 : w1;
      const int sh = 4 * (i & 7);
      if (s0) w |= 1u << sh;
      if (s1) w |= 2u << sh;
      if (s2) w |= 4u << sh;
      if (s3) w |= 8u << sh;
    } else if constexpr (BITS == 2) {
      const bool s1 = u > b[1];
      const bool s0 = u > (s1 ? b[2] : b[0]);
      if (s0) w0 |= 1u << (2 * i);
      if (s1) w0 |= 2u << (2 * i);
    } else {
      // dim 16 hh + i with i = 4k + r: low bits at 2i of W_hh, high bit at 8k + 2hh + {4,5,0,1}[r]
      const int k = i >> 2, r = i & 3;
      const int pos = 8 * k + 2 * hh + (r < 2 ? 4 + r : r - 2);
      const bool s2 = u > b[3];
      const bool s1 = u > (s2 ? b[5] : b[1]);
      const bool s0 = u > (s2 ? (s1 ? b[6] : b[4]) : (s1 ? b[2] : b[0]));
      if (s0) w0 |= 1u << (2 * i);
      if (s1) w0 |= 2u << (2 * i);
      if (s2) w1 |= 1u << pos;
    }
  }
}

template <int BITS>
__global__ void __launch_bounds__(kAppendThreads, kAppendCtasPerSm)
append_kernel(Geometry g, const __half* __restrict__ k, const __half* __restrict__ v,
              const int32_t* __restrict__ slots, int n, uint8_t* __restrict__ pages,
              int32_t* __restrict__ status) {
  constexpr int vb = BITS * 16;
  float bnd[15];
  load_boundaries<BITS>(bnd, g.boundaries);

  const int lane = threadIdx.x & 31;
  const int kind = (lane >> 3) & 1;  // 0: K, 1: V
  const int l = lane & 7;            // dims 16l .. 16l + 15
  const int hkv = g.num_kv_heads;
  const long long items = (long long)n * hkv;
  const long long halves = (long long)gridDim.x * (kAppendThreads / 16);  // half-warps of the grid
  const float* rot = kind ? g.rot_v : g.rot_k;
  const long long pool_slots = (long long)g.num_pages * g.page_size;
  const PageSplit split(g.page_size);

  long long item = (long long)blockIdx.x * (kAppendThreads / 16) + (threadIdx.x >> 4);
  // item = t * Hkv + h: divided once, then advanced by the stride without dividing; when the
  // stride is a multiple of Hkv the half-warp's head never changes and its rotation parameters
  // are loaded once
  int t = (int)(item / hkv), h = (int)(item % hkv);
  const int stride_t = (int)(halves / hkv), stride_h = (int)(halves % hkv);
  float pr[16];
  auto load_params = [&](int hh) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float4 p4 = __ldg(reinterpret_cast<const float4*>(rot + (size_t)hh * kHeadDim + 16 * l + 4 * q));
      pr[4 * q] = p4.x, pr[4 * q + 1] = p4.y, pr[4 * q + 2] = p4.z, pr[4 * q + 3] = p4.w;
    }
  };
  load_params(h);
  // every lane of the warp runs every iteration (shuffles): an item past the end stores nothing
  const long long first = (long long)blockIdx.x * (kAppendThreads / 16) + (threadIdx.x & ~31) / 16;
  const long long iters = first < items ? (items - first + halves - 1) / halves : 0;
  // the item's slot and 32 bytes, loaded an iteration ahead
  int slot_n = -1;
  uint4 raw0_n = make_uint4(0u, 0u, 0u, 0u), raw1_n = raw0_n;
  auto fetch = [&](long long itm, int tt, int hh) {
    slot_n = -1;
    if (itm < items) {
      slot_n = __ldg(slots + tt);
      const uint4* src = reinterpret_cast<const uint4*>((kind ? v : k) + ((size_t)tt * hkv + hh) * kHeadDim + 16 * l);
      raw0_n = __ldg(src);
      raw1_n = __ldg(src + 1);
    }
  };
  fetch(item, t, h);
  for (long long it = 0; it < iters; ++it, item += halves) {
    const bool live = item < items;
    const int slot = slot_n;
    const uint4 raw0 = raw0_n, raw1 = raw1_n;
    if (stride_h != 0 && it > 0 && live) load_params(h);
    const int h_cur = h;
    t += stride_t;
    h += stride_h;
    if (h >= hkv) {
      h -= hkv;
      ++t;
    }
    fetch(item + halves, t, h);

    const bool bad = (long long)slot >= pool_slots;
    if (bad && l == 0 && kind == 0 && status) atomicOr(status, RQ_STATUS_BAD_SLOT);
    const bool store = live && slot >= 0 && !bad;
    float x[16];
    {
      const uint32_t w[8] = {raw0.x, raw0.y, raw0.z, raw0.w, raw1.x, raw1.y, raw1.z, raw1.w};
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[e]));
        x[2 * e] = f.x;
        x[2 * e + 1] = f.y;
      }
    }
    // The squared norm in the order of the 16-lane codec (rq_codec.cuh, which the decode step's
    // append uses): this lane's halves are that codec's lanes 2l and 2l + 1, whose butterfly
    // pairs lanes 8, 4, 2 and then 1 apart -- here lanes 4, 2, 1 apart for each half, then the
    // two halves -- so both write bitwise the same norm.
    float sa = 0.f, sb = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      sa += x[e] * x[e];
      sb += x[8 + e] * x[8 + e];
    }
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) {
      sa += __shfl_xor_sync(0xffffffffu, sa, o);
      sb += __shfl_xor_sync(0xffffffffu, sb, o);
    }
    const float nrm = __fsqrt_rn(sa + sb);
    float y[16];
    {
      float y8[8], x8[8], p8[8];
#pragma unroll
      for (int hv = 0; hv < 2; ++hv) {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          x8[e] = x[8 * hv + e];
          p8[e] = pr[8 * hv + e];
        }
        rotate8(y8, x8, p8, g.mode);
#pragma unroll
        for (int e = 0; e < 8; ++e) y[8 * hv + e] = y8[e];
      }
    }
    uint32_t w0, w1;
    code16<BITS>(y, inv_norm(nrm), bnd, l & 1, w0, w1);
    uint32_t w2 = 0u;
    if constexpr (BITS == 3) w2 = w1 | __shfl_xor_sync(0xffffffffu, w1, 1);  // the group's high bits
    if (store) {
      int page, off;
      split(slot, page, off);
      uint8_t* chunk = pages + ((size_t)page * hkv + h_cur) * (size_t)g.page_bytes;
      uint8_t* dst = chunk + (size_t)kind * g.page_size * vb + (size_t)off * vb;
      const int pair = off >> 1, hvt = off & 1;
      if constexpr (BITS == 4) {
        uint8_t* at = kind == 0 ? dst + 8 * l
                                : chunk + (size_t)g.page_size * vb + pair * 128 + 16 * (l ^ ((2 * pair) & 7)) + 8 * hvt;
        *reinterpret_cast<uint2*>(at) = make_uint2(w0, w1);
      } else if constexpr (BITS == 2) {
        uint8_t* at = kind == 0 ? dst + 4 * l
                                : chunk + (size_t)g.page_size * vb + pair * 64 + 8 * (l ^ (4 * ((pair >> 1) & 1))) + 4 * hvt;
        *reinterpret_cast<uint32_t*>(at) = w0;
      } else {
        *reinterpret_cast<uint32_t*>(dst + 12 * (l >> 1) + 4 * (l & 1)) = w0;
        if ((l & 1) == 0) *reinterpret_cast<uint32_t*>(dst + 12 * (l >> 1) + 8) = w2;
      }
      if (l == 0) {
        const __half n16 = __float2half_rn(nrm);
        *reinterpret_cast<__half*>(chunk + (size_t)2 * g.page_size * vb + (size_t)kind * 2 * g.page_size + 2 * off) = n16;
        if (status && __hisinf(n16)) atomicOr(status, RQ_STATUS_NORM_OVERFLOW);
      }
    }
  }
}

// ---------------------------------------------------------------------------------------
// Dense rotation (tensor cores)
// ---------------------------------------------------------------------------------------
// Two CTAs per SM, so that one CTA's GEMM overlaps the other's coding (each CTA alternates the
// two with barriers in between).
constexpr int kDenseRows = 32;                 // vectors per tile
constexpr int kDenseThreads = 256;             // 8 warps: 2 row tiles x 4 column quarters
constexpr int kDenseWarps = kDenseThreads / 32;
constexpr int kDenseCtasPerSm = 2;
constexpr int kYStride = 136;                  // floats per staged Y row (conflict-free float2 stores)
constexpr int kSmemR = 0;                      // fp16 [2 (hi, lo)][128][128], 16-byte chunks swizzled
constexpr int kSmemX = kSmemR + 2 * 128 * 128 * 2;            // fp16 [2 buffers][32][128], swizzled
constexpr int kSmemY = kSmemX + 2 * kDenseRows * 128 * 2;     // fp32 [32][136]
constexpr int kDenseSmem = kSmemY + kDenseRows * kYStride * 4;  // 99,328 bytes; the fp32 R of the
                                                                // exact recompute is read from L2

// A 256-byte row of 16 chunks (8 fp16 each) stores chunk c at position c ^ (row mod 8), so the
// eight rows one ldmatrix phase reads fall in eight different 16-byte bank groups.
__device__ __forceinline__ uint32_t swz(int row, int chunk) { return (uint32_t)(row * 256 + ((chunk ^ (row & 7)) << 4)); }

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

// Tile t covers tokens kDenseRows * blk .. + kDenseRows - 1 of kv head hk % Hkv, K (hk < Hkv) or V, with
// hk = t % (2 Hkv) and blk = t / (2 Hkv).  Rows past n are zero-filled.
__device__ __forceinline__ void issue_x(uint32_t xs, int hk, long long blk, const Geometry& g, const __half* k,
                                       const __half* v, int n, uint8_t* xs_generic) {
  const int hkv = g.num_kv_heads;
  const int kind = hk >= hkv, h = kind ? hk - hkv : hk;
  const __half* src = kind ? v : k;
  for (int i = threadIdx.x; i < kDenseRows * 16; i += kDenseThreads) {
    const int r = i >> 4, c = i & 15;
    const long long t = blk * kDenseRows + r;
    if (t < n) {
      cp_async16(xs + swz(r, c), src + ((size_t)t * hkv + h) * kHeadDim + 8 * c);
    } else {
      *reinterpret_cast<uint4*>(xs_generic + swz(r, c)) = make_uint4(0u, 0u, 0u, 0u);
    }
  }
}

template <int BITS>
__global__ void __launch_bounds__(kDenseThreads, kDenseCtasPerSm)
append_dense_kernel(Geometry g, const __half* __restrict__ k, const __half* __restrict__ v,
                    const int32_t* __restrict__ slots, int n, uint8_t* __restrict__ pages,
                    int32_t* __restrict__ status) {
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t base = (uint32_t)__cvta_generic_to_shared(smem);
  float* Ys = reinterpret_cast<float*>(smem + kSmemY);
  float bnd[15];
  load_boundaries<BITS>(bnd, g.boundaries);

  const int hkv = g.num_kv_heads;
  const long long nblk = ((long long)n + kDenseRows - 1) / kDenseRows;
  const long long tiles = 2LL * hkv * nblk;
  const long long pool_slots = (long long)g.num_pages * g.page_size;
  const PageSplit split(g.page_size);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gq = lane >> 2, tq = lane & 3;
  const int mt = warp & 1, nq = warp >> 1;  // rows 16mt.., columns 32nq..
  const int half = lane >> 4, j = lane & 15;

  long long tile = blockIdx.x;
  if (tile >= tiles) return;
  // (hk, blk) of the tile, advanced by the grid stride without dividing
  const int h2 = 2 * hkv;
  int hk = (int)(tile % h2);
  long long blk = tile / h2;
  const int stride_hk = (int)(gridDim.x % h2);
  const long long stride_blk = gridDim.x / h2;
  auto advance = [&](int& a, long long& b) {
    a += stride_hk;
    b += stride_blk;
    if (a >= h2) {
      a -= h2;
      ++b;
    }
  };
  int buf = 0, cur_hk = -1;
  issue_x(base + kSmemX, hk, blk, g, k, v, n, smem + kSmemX);
  cp_async_commit();
  for (; tile < tiles; tile += gridDim.x) {
    const int kind = hk >= hkv, h = kind ? hk - hkv : hk;
    const float* r32 = g.dense32 + ((size_t)kind * hkv + h) * 128 * 128;  // fp32 R rows (exact recompute)
    if (hk != cur_hk) {  // stage R of this (K or V, head); the previous tile is done with it
      const uint4* src = reinterpret_cast<const uint4*>(g.dense16 + ((size_t)kind * hkv + h) * 2 * 128 * 128);
      for (int i = threadIdx.x; i < 2 * 128 * 16; i += kDenseThreads) {
        const int hl = i >> 11, row = (i >> 4) & 127, c = i & 15;
        *reinterpret_cast<uint4*>(smem + kSmemR + hl * 32768 + swz(row, c)) = __ldg(src + i);
      }
      cur_hk = hk;
    }
    const long long next = tile + gridDim.x;
    int hk_next = hk;
    long long blk_next = blk;
    advance(hk_next, blk_next);
    const uint32_t xs_next = base + kSmemX + (uint32_t)((buf ^ 1) * kDenseRows * 256);
    if (next < tiles) issue_x(xs_next, hk_next, blk_next, g, k, v, n, smem + kSmemX + (buf ^ 1) * kDenseRows * 256);
    cp_async_commit();
    cp_async_wait1();
    __syncthreads();  // this tile's X (and R, if restaged) visible to every warp

    const uint32_t xs = base + kSmemX + (uint32_t)(buf * kDenseRows * 256);
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
#pragma unroll 2
    for (int ks = 0; ks < 8; ++ks) {
      uint32_t a[4];
      // matrices: rows 0-7 / 8-15 of the row tile, k chunks 2ks / 2ks+1 -> a0, a1, a2, a3
      ldsm_x4(a, xs + swz(16 * mt + (lane & 15), 2 * ks + (lane >> 4)));
#pragma unroll
      for (int np = 0; np < 2; ++np) {
        const int nrow = 8 * (4 * nq + 2 * np + (lane >> 4)) + (lane & 7);
        const int kc = 2 * ks + ((lane >> 3) & 1);
#pragma unroll
        for (int hl = 0; hl < 2; ++hl) {
          uint32_t b[4];  // b0, b1 of n-tile 2np, then of 2np + 1
          ldsm_x4(b, base + kSmemR + hl * 32768 + swz(nrow, kc));
          mma16816(acc[2 * np], a, b[0], b[1]);
          mma16816(acc[2 * np + 1], a, b[2], b[3]);
        }
      }
    }
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      const int col = 32 * nq + 8 * nt + 2 * tq;
      *reinterpret_cast<float2*>(Ys + (16 * mt + gq) * kYStride + col) = make_float2(acc[nt][0], acc[nt][1]);
      *reinterpret_cast<float2*>(Ys + (16 * mt + gq + 8) * kYStride + col) = make_float2(acc[nt][2], acc[nt][3]);
    }
    __syncthreads();

    // Coding: a half-warp per vector, lane j on dims 8j..8j+7 (2 kDenseWarps vectors per pass).
    const uint8_t* xg = smem + kSmemX + buf * kDenseRows * 256;
#pragma unroll 1
    for (int pass = 0; pass < kDenseRows / (2 * kDenseWarps); ++pass) {
      const int r = 2 * kDenseWarps * pass + 2 * warp + half;
      const long long t = blk * kDenseRows + r;
      int slot = t < n ? __ldg(slots + t) : -1;
      const bool bad = (long long)slot >= pool_slots;
      if (bad && j == 0 && status) atomicOr(status, RQ_STATUS_BAD_SLOT);
      const bool store = slot >= 0 && !bad;
      if (!store) slot = 0;
      const uint4 raw = *reinterpret_cast<const uint4*>(xg + swz(r, j));
      float y[8];
      {
        const float4 y0 = *reinterpret_cast<const float4*>(Ys + r * kYStride + 8 * j);
        const float4 y1 = *reinterpret_cast<const float4*>(Ys + r * kYStride + 8 * j + 4);
        y[0] = y0.x, y[1] = y0.y, y[2] = y0.z, y[3] = y0.w, y[4] = y1.x, y[5] = y1.y, y[6] = y1.z, y[7] = y1.w;
      }
      int code[8];
      float nrm;
      dense_codes<BITS>(code, nrm, raw, y, bnd, r32, store, lane);
      int page, off;
      split(slot, page, off);
      uint8_t* chunk = pages + ((size_t)page * hkv + h) * (size_t)g.page_bytes;
      pack_store<BITS>(code, nrm, chunk, g.page_size, kind, off, j, store, status);
    }
    __syncthreads();  // X buffer and Y free for the next tile
    buf ^= 1;
    hk = hk_next;
    blk = blk_next;
  }
}

template <int BITS>
cudaError_t launch_append_bits(const Geometry& g, const __half* k, const __half* v, const int32_t* slots, int n,
                               uint8_t* pages, int32_t* status, cudaStream_t stream, int sms) {
  if (g.mode == RQ_DENSE) {
    const long long tiles = 2LL * g.num_kv_heads * ((n + kDenseRows - 1) / kDenseRows);
    // whole multiples of the 2 Hkv (K/V, head) groups, so a CTA keeps one R staged
    const int resident = kDenseCtasPerSm * sms;
    int ctas = resident >= 2 * g.num_kv_heads ? resident / (2 * g.num_kv_heads) * (2 * g.num_kv_heads) : resident;
    if (tiles < ctas) ctas = (int)tiles;
    append_dense_kernel<BITS><<<ctas, kDenseThreads, kDenseSmem, stream>>>(g, k, v, slots, n, pages, status);
  } else {
    const long long items = (long long)n * g.num_kv_heads;
    long long blocks = (items + kAppendThreads / 16 - 1) / (kAppendThreads / 16);  // an item per half-warp
    const long long max_blocks = (long long)sms * kAppendCtasPerSm;
    if (blocks > max_blocks) blocks = max_blocks;
    append_kernel<BITS><<<(unsigned)blocks, kAppendThreads, 0, stream>>>(g, k, v, slots, n, pages, status);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t append_prepare() {
  cudaError_t e = cudaFuncSetAttribute(append_dense_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, kDenseSmem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(append_dense_kernel<3>, cudaFuncAttributeMaxDynamicSharedMemorySize, kDenseSmem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(append_dense_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, kDenseSmem);
  return e;
}

cudaError_t launch_append(const Geometry& g, const void* k, const void* v, const int32_t* slots, int n,
                          uint8_t* pages, int32_t* status, cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  static int sms_of[64] = {};  // per device; benign race: every writer stores the same value
  int dev = 0;
  cudaGetDevice(&dev);
  int sms = dev >= 0 && dev < 64 ? sms_of[dev] : 0;
  if (sms <= 0) {
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) sms = 132;
    if (dev >= 0 && dev < 64) sms_of[dev] = sms;
  }
  const __half* kh = (const __half*)k;
  const __half* vh = (const __half*)v;
  if (g.bits == 4) return launch_append_bits<4>(g, kh, vh, slots, n, pages, status, stream, sms);
  if (g.bits == 3) return launch_append_bits<3>(g, kh, vh, slots, n, pages, status, stream, sms);
  return launch_append_bits<2>(g, kh, vh, slots, n, pages, status, stream, sms);
}

}  // namespace rq
