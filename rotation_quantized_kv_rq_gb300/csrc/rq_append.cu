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
// Dense rotation: Y = X R^T for a tile of 128 vectors of one (kv head, K or V) is a GEMM
// (128 x 128 x 128) on the 5th-generation tensor cores (tcgen05, f32 accumulators in tensor
// memory).  X is fp16 and exact as an operand; R (fp32) is split as R = hi + lo with
// hi = fp16(R), lo = fp16(R - hi), both multiplied into one fp32 accumulator.  That carries R to
// ~6e-8 per entry, but the tensor cores' fp32 accumulation is not correctly rounded, so a
// coordinate whose u lies within kFixBand of a boundary is recomputed exactly -- a compensated
// fp32 dot product (error-free products and sums) against the fp32 R -- before it is coded.
// Codes then differ from the fp64 definition only as rarely as the structured kernel's.
#include <cuda_fp16.h>

#include "rq_codec.cuh"
#include "rq_tc.cuh"
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
// Dense rotation on the 5th-generation tensor cores (tcgen05).  A CTA (one per SM) takes
// 128-vector tiles of one (K or V, kv head), whose R_hi, R_lo it stages once:
//   * 2 loader warps stage X (fp16, 128 x 128) with cp.async into a two-buffer ring, in the
//     K-major 128-byte-swizzled operand layout;
//   * one thread issues Y = X R_hi^T + X R_lo^T (M 128 x N 128 x K 128, f32 accumulate) into
//     tensor memory, two tiles' Y in 256 columns;
//   * 16 coding warps: thread (row, part) reads 32 coordinates of its vector's Y from tensor
//     memory (the lane is the row), forms the norm from X (the partial sums of squares of the
//     16 eight-dim chunks combined in the half-warp codec's order, so the fp16 norm is the
//     decode step's bit for bit), codes, and writes its part of the packed vector.  A
//     coordinate whose u lies within kFixBand of a boundary is recomputed exactly by its whole
//     warp (a compensated fp32 dot product against R's fp32 row, 4 terms a lane) and re-coded.
// ---------------------------------------------------------------------------------------
namespace dtc {
constexpr int kRows = 128;                        // vectors per tile: M of the MMA
constexpr int kCodeWarps = 16;                    // warps 0-15: coding
constexpr int kParts = kCodeWarps / 4;            // coding threads per vector (row)
constexpr int kPartDims = 128 / kParts;           // dims each codes
constexpr int kLoadWarps = 2;                     // warps 16-17: X loads
constexpr int kThreads = 32 * (kCodeWarps + kLoadWarps + 1);  // + warp 18: MMA issue
constexpr int kCodeThreads = 32 * kCodeWarps, kLoadThreads = 32 * kLoadWarps;
constexpr uint32_t kR = 0;                        // R_hi, R_lo: fp16 [2][2 atoms of 16 KB]
constexpr uint32_t kX = 65536;                    // X: fp16 [2 buffers][2 atoms of 16 KB]
constexpr uint32_t kSS = kX + 65536;              // partial sums of squares: f32 [2][16 chunks][128 rows]
constexpr uint32_t kBar = kSS + 2 * kRows * 16 * 4;
constexpr uint32_t kBarXFull = 0, kBarXEmpty = 16, kBarYFull = 32, kBarYEmpty = 48, kBarDrain = 64;
constexpr uint32_t kTmemSlot = 72, kAbort = 76;
constexpr uint32_t kTab = kBar + 128;             // the binned code table: u32 [kCodeBins][2]
constexpr int kSmem = (int)kTab + kCodeBins * 8 + 1024;  // + slack to align the window to 1024 bytes
constexpr uint32_t kTmemCols = 256;
}  // namespace dtc

__device__ __forceinline__ void cp_async16_tc(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

// y_i = sum_m x_m R[i][m], exactly enough to be correctly rounded in all but pathological
// cases (error-free products and sums, errors carried in a second word), by a whole warp: lane
// l takes dims 4l .. 4l + 3 of x (fp16, row `xrow` of a staged X tile) and of R's fp32 row.
__device__ __forceinline__ float dot_compensated_warp(const uint8_t* xatoms, int xrow, const float* rrow, int lane) {
  const uint2 raw = *reinterpret_cast<const uint2*>(xatoms + (lane >> 4) * 16384 + tc::sw128(xrow, (lane >> 1) & 7) +
                                                    8 * (lane & 1));
  const float2 x01 = __half22float2(*reinterpret_cast<const __half2*>(&raw.x));
  const float2 x23 = __half22float2(*reinterpret_cast<const __half2*>(&raw.y));
  const float x[4] = {x01.x, x01.y, x23.x, x23.y};
  const float4 r4 = __ldg(reinterpret_cast<const float4*>(rrow + 4 * lane));
  const float rr[4] = {r4.x, r4.y, r4.z, r4.w};
  float s = 0.f, c = 0.f;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float p = x[e] * rr[e];
    const float pe = fmaf(x[e], rr[e], -p);  // x * r = p + pe exactly
    const float t = s + p;
    const float z = t - s;
    c += ((s - (t - z)) + (p - z)) + pe;     // s + p = t + (that) exactly
    s = t;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
    const float c2 = __shfl_xor_sync(0xffffffffu, c, o);
    const float t = s + s2;
    const float z = t - s;
    c += c2 + ((s - (t - z)) + (s2 - z));
    s = t;
  }
  return s + c;
}

template <int BITS>
__global__ void __launch_bounds__(dtc::kThreads, 1)
append_dense_tc_kernel(Geometry g, const __half* __restrict__ k, const __half* __restrict__ v,
                       const int32_t* __restrict__ slots, int n, uint8_t* __restrict__ pages,
                       int32_t* __restrict__ status) {
  using namespace dtc;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = (uint32_t)__cvta_generic_to_shared(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const sm = smem_raw + (base - raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int hkv = g.num_kv_heads, npairs = 2 * hkv;
  const int cpp = (int)gridDim.x / npairs;  // CTAs per (K or V, head): the launch makes it >= 1
  const int pair = (int)blockIdx.x / cpp, sub = (int)blockIdx.x % cpp;
  const int nblk = (n + kRows - 1) / kRows;
  const int my_tiles = (pair < npairs && sub < nblk) ? (nblk - 1 - sub) / cpp + 1 : 0;
  if (my_tiles == 0) return;  // uniform over the CTA, before any barrier or allocation
  const int kind = pair >= hkv, h = kind ? pair - hkv : pair;
  const __half* const src = kind ? v : k;
  const float* const r32 = g.dense32 + ((size_t)kind * hkv + h) * 128 * 128;  // fp32 R rows (exact recompute)
  const uint32_t mb = base + kBar;
  volatile int* const abort_flag = reinterpret_cast<volatile int*>(sm + kBar + kAbort);
  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(mb + kBarXFull + 8 * i, kLoadThreads);
      tc::mbar_init(mb + kBarXEmpty + 8 * i, kCodeThreads);
      tc::mbar_init(mb + kBarYFull + 8 * i, 1);
      tc::mbar_init(mb + kBarYEmpty + 8 * i, kCodeThreads);
    }
    tc::mbar_init(mb + kBarDrain, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kCodeWarps + kLoadWarps) tc::tmem_alloc(mb + kTmemSlot, kTmemCols);  // whole warp
  {  // R_hi, R_lo ([2][128][128] row-major fp16) in the K-major swizzled layout, rows = output dims
    const uint4* rsrc = reinterpret_cast<const uint4*>(g.dense16 + ((size_t)kind * hkv + h) * 2 * 128 * 128);
    for (int i = tid; i < 2 * 128 * 16; i += kThreads) {
      const int hl = i >> 11, row = (i >> 4) & 127, c = i & 15;
      *reinterpret_cast<uint4*>(sm + kR + hl * 32768 + (c >> 3) * 16384 + tc::sw128(row, c & 7)) = __ldg(rsrc + i);
    }
  }
  const uint2* const tab = g.code_table ? reinterpret_cast<const uint2*>(sm + kTab) : nullptr;
  if (tab)
    for (int i = tid; i < kCodeBins; i += kThreads)
      reinterpret_cast<uint2*>(sm + kTab)[i] = __ldg(reinterpret_cast<const uint2*>(g.code_table) + i);
  tc::fence_async_smem();  // read by the tensor core (async proxy)
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sm + kBar + kTmemSlot);

  if (warp < kCodeWarps) {
    // ================= coding: thread = (row, part ch of the dims) =================
    const int row = 32 * (warp & 3) + lane, ch = warp >> 2;  // dims kPartDims ch .. + kPartDims - 1
    const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
    // the four warps of a lane quarter (warp % 4: the same 32 rows, a quarter of the dims each)
    // exchange their rows' partial sums of squares at named barrier 1 + warp % 4
    const uint32_t quarter_bar = 1u + (uint32_t)(warp & 3);
    float bnd[15];
    load_boundaries<BITS>(bnd, g.boundaries);
    const PageSplit split(g.page_size);
    const long long pool_slots = (long long)g.num_pages * g.page_size;
    constexpr int vb = BITS * 16;
    bool ok = true;
    for (int i = 0; i < my_tiles && ok; ++i) {
      const int b = i & 1;
      const long long t = (long long)(sub + i * cpp) * kRows + row;
      int slot = t < n ? __ldg(slots + t) : -1;
      const bool bad = (long long)slot >= pool_slots;
      if (bad && ch == 0 && status) atomicOr(status, RQ_STATUS_BAD_SLOT);
      const bool store = slot >= 0 && !bad;
      if (!store) slot = 0;
      ok = tc::role_wait(mb + kBarXFull + 8 * b, (uint32_t)((i >> 1) & 1), abort_flag) &&
           tc::role_wait(mb + kBarYFull + 8 * b, (uint32_t)((i >> 1) & 1), abort_flag);
      {  // agree across the quarter's coding warps (they meet at a named barrier below)
        uint32_t all_ok;
        asm volatile("{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.and.pred q, %2, %3, p;\n selp.u32 %0, 1, 0, q;\n}"
                     : "=r"(all_ok)
                     : "r"((uint32_t)ok), "r"(quarter_bar), "n"(kCodeThreads / 4)
                     : "memory");
        ok = all_ok != 0;
      }
      if (!ok) break;
      tc::fence_after_sync();
      const uint8_t* const xatoms = sm + kX + b * 32768;
      // the norm: partial sums of squares of the 8-dim chunks (each in order), combined as the
      // half-warp codec's butterfly (xor 8, 4, 2, 1) combines its lanes' sums
      float* const ss = reinterpret_cast<float*>(sm + kSS) + b * 16 * kRows + row;  // chunk c at ss[c * kRows]
#pragma unroll
      for (int cc0 = 0; cc0 < kPartDims / 8; ++cc0) {
        const int cc = (kPartDims / 8) * ch + cc0;  // the 8-dim chunk of the vector
        const uint4 w4 = *reinterpret_cast<const uint4*>(xatoms + (cc >> 3) * 16384 + tc::sw128(row, cc & 7));
        const uint32_t w[4] = {w4.x, w4.y, w4.z, w4.w};
        float x[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[e]));
          x[2 * e] = f.x;
          x[2 * e + 1] = f.y;
        }
        float ps = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) ps += x[e] * x[e];
        ss[cc * kRows] = ps;
      }
      asm volatile("bar.sync %0, %1;" ::"r"(quarter_bar), "n"(kCodeThreads / 4) : "memory");  // the row's sums are in
      float a8[8];
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) a8[jj] = ss[jj * kRows] + ss[(jj + 8) * kRows];
      const float b0 = a8[0] + a8[4], b1 = a8[1] + a8[5], b2 = a8[2] + a8[6], b3 = a8[3] + a8[7];
      const float nrm = __fsqrt_rn((b0 + b2) + (b1 + b3));
      const float rcp = inv_norm(nrm);

      int page = 0, off = 0;
      split(slot, page, off);
      uint8_t* const chunk = pages + ((size_t)page * hkv + h) * (size_t)g.page_bytes;
      uint8_t* const dst = chunk + (size_t)kind * g.page_size * vb + (size_t)off * vb;
      uint8_t* const vsec = chunk + (size_t)g.page_size * vb;
      const int vpair = off >> 1, hv = off & 1;
      uint32_t w2 = 0u;  // 3-bit: the high bits of the current 32-dim group
      static_assert(kPartDims == 32, "two 16-dim units a thread");
      float yy[2][16];  // both units' y, loaded together (one wait)
      tc::tmem_ld16(tmem + lane_off + 128 * b + 32 * ch, yy[0]);
      tc::tmem_ld16(tmem + lane_off + 128 * b + 32 * ch + 16, yy[1]);
      tc::tmem_wait_ld();
#pragma unroll
      for (int q0 = 0; q0 < 2; ++q0) {  // coordinates 16 q .. 16 q + 15
        const int q = 2 * ch + q0;       // the 16-dim unit of the vector
        const float(&y)[16] = yy[q0];
        int code[16];
        uint32_t todo = 0;
        if (tab) {  // the same codes and the same coordinates to recompute as the select tree
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            bool near;
            code[e] = code_of_table(y[e] * rcp, tab, near);
            if (near && store) todo |= 1u << e;
          }
        } else {
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            float dm;
            code[e] = code_of_margin<BITS>(y[e] * rcp, bnd, dm);
            if (dm < kFixBand && store) todo |= 1u << e;
          }
        }
        while (__any_sync(0xffffffffu, todo != 0)) {  // exact recompute, one coordinate at a time
          const uint32_t want = __ballot_sync(0xffffffffu, todo != 0);
          const int leader = __ffs(want) - 1;
          const int e_lead = __shfl_sync(0xffffffffu, todo ? __ffs(todo) - 1 : 0, leader);
          const float yi = dot_compensated_warp(xatoms, 32 * (warp & 3) + leader, r32 + (16 * q + e_lead) * 128, lane);
          if (lane == leader) {
            const int c = code_of<BITS>(yi * rcp, bnd);
#pragma unroll
            for (int e = 0; e < 16; ++e)
              if (e == e_lead) code[e] = c;
            todo &= ~(1u << e_lead);
          }
        }
        if (store) {
          const int u = q;
          if constexpr (BITS == 4) {
            uint32_t lo = 0, hi = 0;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              lo |= (uint32_t)code[e] << (4 * e);
              hi |= (uint32_t)code[8 + e] << (4 * e);
            }
            uint8_t* at = kind == 0 ? dst + 8 * u : vsec + vpair * 128 + 16 * (u ^ ((2 * vpair) & 7)) + 8 * hv;
            *reinterpret_cast<uint2*>(at) = make_uint2(lo, hi);
          } else if constexpr (BITS == 2) {
            uint32_t wd = 0;
#pragma unroll
            for (int e = 0; e < 16; ++e) wd |= (uint32_t)code[e] << (2 * e);
            uint8_t* at = kind == 0 ? dst + 4 * u : vsec + vpair * 64 + 8 * (u ^ (4 * ((vpair >> 1) & 1))) + 4 * hv;
            *reinterpret_cast<uint32_t*>(at) = wd;
          } else {
            // group grp = u / 2, half hq = u % 2: the low bits are word hq of the group, the high
            // bits of dim i = 16 hq + 4 kk + r go to bit 8 kk + 2 hq + {4, 5, 0, 1}[r] of W2
            const int grp = u >> 1, hq = u & 1;
            uint32_t lo = 0;
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              lo |= (uint32_t)(code[e] & 3) << (2 * e);
              const int kk = e >> 2, r = e & 3;
              w2 |= (uint32_t)(code[e] >> 2) << (8 * kk + 2 * hq + (r < 2 ? 4 + r : r - 2));
            }
            *reinterpret_cast<uint32_t*>(dst + 12 * grp + 4 * hq) = lo;
            if (hq == 1) {
              *reinterpret_cast<uint32_t*>(dst + 12 * grp + 8) = w2;
              w2 = 0u;
            }
          }
        }
      }
      tc::fence_before_sync();
      tc::mbar_arrive(mb + kBarYEmpty + 8 * b);  // this tile's Y has been read
      tc::mbar_arrive(mb + kBarXEmpty + 8 * b);  // and its X (norms, recomputes)
      if (store && ch == 0) {
        const __half n16 = __float2half_rn(nrm);
        *reinterpret_cast<__half*>(chunk + (size_t)2 * g.page_size * vb + (size_t)kind * 2 * g.page_size + 2 * off) = n16;
        if (status && __hisinf(n16)) atomicOr(status, RQ_STATUS_NORM_OVERFLOW);
      }
    }
    if (!ok && lane == 0 && status) atomicOr(status, RQ_STATUS_TIMEOUT);
  } else if (warp < kCodeWarps + kLoadWarps) {
    // ================= X loads: tile i into buffer i % 2 =================
    const int lt = tid - kCodeThreads;
    auto issue = [&](int i) {
      const uint32_t xb = base + kX + (uint32_t)(i & 1) * 32768;
      const long long t0 = (long long)(sub + i * cpp) * kRows;
      for (int q = lt; q < kRows * 16; q += kLoadThreads) {
        const int r = q >> 4, c = q & 15;
        const long long t = t0 + r;
        const uint32_t d = xb + (c >> 3) * 16384 + tc::sw128(r, c & 7);
        if (t < n)
          cp_async16_tc(d, src + ((size_t)t * hkv + h) * kHeadDim + 8 * c);
        else
          *reinterpret_cast<uint4*>(sm + (d - base)) = make_uint4(0u, 0u, 0u, 0u);
      }
      asm volatile("cp.async.commit_group;" ::: "memory");
    };
    bool ok = true;
    issue(0);
    for (int i = 0; i < my_tiles && ok; ++i) {
      asm volatile("cp.async.wait_group 0;" ::: "memory");  // tile i has landed
      tc::fence_async_smem();
      tc::mbar_arrive(mb + kBarXFull + 8 * (i & 1));
      if (i + 1 < my_tiles) {  // the next tile, once tile i - 1 has left its buffer
        if (i >= 1)
          ok = __all_sync(0xffffffffu, tc::role_wait(mb + kBarXEmpty + 8 * ((i + 1) & 1), (uint32_t)(((i - 1) >> 1) & 1),
                                                     abort_flag));
        if (ok) issue(i + 1);
      }
    }
    if (!ok && lane == 0 && status) atomicOr(status, RQ_STATUS_TIMEOUT);
  } else if (lane == 0) {
    // ================= MMA issue (one thread) =================
    const uint32_t id = tc::idesc_f16(kRows, 128);
    bool ok = true;
    int issued = 0;
    for (int i = 0; i < my_tiles && ok; ++i) {
      const int b = i & 1;
      ok = tc::role_wait(mb + kBarXFull + 8 * b, (uint32_t)((i >> 1) & 1), abort_flag) &&
           (i < 2 || tc::role_wait(mb + kBarYEmpty + 8 * b, (uint32_t)(((i >> 1) - 1) & 1), abort_flag));
      if (!ok) break;
      tc::fence_after_sync();
      const uint32_t xb = base + kX + (uint32_t)b * 32768;
#pragma unroll
      for (int hl = 0; hl < 2; ++hl)
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          tc::umma_f16_ss(tmem + 128 * b, tc::sdesc(xb + (ks >> 2) * 16384 + (ks & 3) * 32),
                          tc::sdesc(base + kR + hl * 32768 + (ks >> 2) * 16384 + (ks & 3) * 32), id, hl > 0 || ks > 0);
      tc::umma_commit(mb + kBarYFull + 8 * b);
      ++issued;
    }
    if (issued > 0) {  // drain: nothing may be running when the tensor memory is freed
      tc::umma_commit(mb + kBarDrain);
      for (int i = 0; i < tc::kWaitLimit; ++i)
        if (tc::mbar_test(mb + kBarDrain, 0u)) break;
    }
    if (!ok && status) atomicOr(status, RQ_STATUS_TIMEOUT);
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == kCodeWarps + kLoadWarps) tc::tmem_dealloc(tmem, kTmemCols);
}

template <int BITS>
cudaError_t launch_append_bits(const Geometry& g, const __half* k, const __half* v, const int32_t* slots, int n,
                               uint8_t* pages, int32_t* status, cudaStream_t stream, int sms) {
  if (g.mode == RQ_DENSE) {
    // CTAs per (K or V, head): the SMs shared out, at most the head's tiles, at least one
    const int npairs = 2 * g.num_kv_heads;
    const long long nblk = ((long long)n + dtc::kRows - 1) / dtc::kRows;
    long long cpp = sms / npairs;
    if (cpp > nblk) cpp = nblk;
    if (cpp < 1) cpp = 1;
    if ((long long)npairs * cpp > 0x7fffffffLL) return cudaErrorInvalidValue;
    append_dense_tc_kernel<BITS><<<(unsigned)(npairs * cpp), dtc::kThreads, dtc::kSmem, stream>>>(g, k, v, slots, n, pages,
                                                                                                 status);
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
  cudaError_t e = cudaFuncSetAttribute(append_dense_tc_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, dtc::kSmem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(append_dense_tc_kernel<3>, cudaFuncAttributeMaxDynamicSharedMemorySize, dtc::kSmem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(append_dense_tc_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, dtc::kSmem);
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
