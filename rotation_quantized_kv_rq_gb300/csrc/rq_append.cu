// Fused quantize-pack-append ("SGLang 1-Bit Turbo" README, section "RotorQuant KV Cache
// Compression": norm, fixed data-oblivious rotation -- 2D Givens pairs or 4D quaternion
// blocks -- then Lloyd-Max scalar codes, bit-packed into the paged cache).
//
// Work item = one (token, kv head).  A warp takes items in a grid-stride loop: lanes 0-15
// encode the K vector and lanes 16-31 the V vector.  Lane j of a half owns dimensions
// 8j..8j+7 -- four whole Givens pairs or two whole quaternion blocks -- so the rotation is
// lane-local and only the squared norm is reduced (4 xor-shuffles within the half).  Each lane
// reads 16 bytes, and the next item's 16 bytes are in flight while the current one is coded.
// The kernel is bound by HBM: 512 bytes of fp16 in, 2 * (16 * bits + 2) bytes out per item.
#include <cuda_fp16.h>

#include "rq_internal.h"
#include "../../include/rq.h"

namespace rq {
namespace {

constexpr int kAppendThreads = 256;
constexpr int kAppendWarps = kAppendThreads / 32;

// Number of boundaries strictly below u (b ascending, in registers): a binary search written as
// a select tree, one compare per level and no indexed memory.
__device__ __forceinline__ int code_of(float u, const float (&b)[15], int bits) {
  if (bits == 3) {
    const bool s2 = u > b[3];
    const bool s1 = u > (s2 ? b[5] : b[1]);
    const bool s0 = u > (s2 ? (s1 ? b[6] : b[4]) : (s1 ? b[2] : b[0]));
    return (s2 ? 4 : 0) + (s1 ? 2 : 0) + (s0 ? 1 : 0);
  }
  const bool s3 = u > b[7];
  const bool s2 = u > (s3 ? b[11] : b[3]);
  const bool s1 = u > (s3 ? (s2 ? b[13] : b[9]) : (s2 ? b[5] : b[1]));
  const float m0 = s3 ? (s2 ? (s1 ? b[14] : b[12]) : (s1 ? b[10] : b[8]))
                      : (s2 ? (s1 ? b[6] : b[4]) : (s1 ? b[2] : b[0]));
  const bool s0 = u > m0;
  return (s3 ? 8 : 0) + (s2 ? 4 : 0) + (s1 ? 2 : 0) + (s0 ? 1 : 0);
}

struct Item {
  int t, h, slot;
  uint4 raw;  // 8 fp16 of this lane's half (K or V)
};

__device__ __forceinline__ void fetch(Item& it, long long item, const Geometry& g, const __half* src_k,
                                      const __half* src_v, const int32_t* slots, int half, int j) {
  it.t = (int)(item / g.num_kv_heads);
  it.h = (int)(item % g.num_kv_heads);
  it.slot = __ldg(slots + it.t);
  const __half* src = (half ? src_v : src_k) + ((size_t)it.t * g.num_kv_heads + it.h) * kHeadDim + 8 * j;
  it.raw = __ldg(reinterpret_cast<const uint4*>(src));
}

template <int BITS>
__global__ void __launch_bounds__(kAppendThreads)
append_kernel(Geometry g, const __half* __restrict__ k, const __half* __restrict__ v,
              const int32_t* __restrict__ slots, int n, uint8_t* __restrict__ pages,
              int32_t* __restrict__ status) {
  float bnd[15];
#pragma unroll
  for (int i = 0; i < 15; ++i) bnd[i] = i < (1 << BITS) - 1 ? __ldg(g.boundaries + i) : 0.f;

  const int lane = threadIdx.x & 31;
  const int half = lane >> 4;        // 0: K, 1: V
  const int j = lane & 15;           // dims 8j..8j+7
  const long long items = (long long)n * g.num_kv_heads;
  const long long stride = (long long)gridDim.x * kAppendWarps;
  const float* rot = half ? g.rot_v : g.rot_k;
  const int vb = BITS * 16;
  const long long pool_slots = (long long)g.num_pages * g.page_size;

  long long item = (long long)blockIdx.x * kAppendWarps + (threadIdx.x >> 5);
  if (item >= items) return;
  Item cur, nxt;
  fetch(cur, item, g, k, v, slots, half, j);
  for (; item < items; item += stride) {
    if (item + stride < items) fetch(nxt, item + stride, g, k, v, slots, half, j);

    const int slot = cur.slot;
    const bool bad = (long long)slot >= pool_slots;
    if (bad && lane == 0 && status) atomicOr(status, RQ_STATUS_BAD_SLOT);
    if (slot >= 0 && !bad) {  // uniform across the warp
      const float4 p0 = __ldg(reinterpret_cast<const float4*>(rot + (size_t)cur.h * kHeadDim + 8 * j));
      const float4 p1 = __ldg(reinterpret_cast<const float4*>(rot + (size_t)cur.h * kHeadDim + 8 * j + 4));
      const uint32_t w[4] = {cur.raw.x, cur.raw.y, cur.raw.z, cur.raw.w};
      float x[8];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[e]));
        x[2 * e] = f.x;
        x[2 * e + 1] = f.y;
      }
      float ss = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) ss += x[e] * x[e];
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      const float nrm = __fsqrt_rn(ss);

      float y[8];
      const float pr[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
      if (g.mode == RQ_PLANAR) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float c = pr[2 * q], s = pr[2 * q + 1];
          y[2 * q] = c * x[2 * q] - s * x[2 * q + 1];
          y[2 * q + 1] = s * x[2 * q] + c * x[2 * q + 1];
        }
      } else {  // Hamilton product (a,b,c,d) (x) (x0,x1,x2,x3)
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const float a = pr[4 * q], b = pr[4 * q + 1], c = pr[4 * q + 2], d = pr[4 * q + 3];
          const float* xb = x + 4 * q;
          y[4 * q + 0] = a * xb[0] - b * xb[1] - c * xb[2] - d * xb[3];
          y[4 * q + 1] = b * xb[0] + a * xb[1] - d * xb[2] + c * xb[3];
          y[4 * q + 2] = c * xb[0] + d * xb[1] + a * xb[2] - b * xb[3];
          y[4 * q + 3] = d * xb[0] - c * xb[1] + b * xb[2] + a * xb[3];
        }
      }
      // u = y / n as y * (1/n): within an ulp of the quotient, so a code can differ from the
      // quotient's only for u within ~1e-7 of a boundary.
      const float rcp = nrm > 0.f ? __frcp_rn(nrm) : 0.f;
      int code[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) code[e] = code_of(y[e] * rcp, bnd, BITS);

      const int page = slot / g.page_size, off = slot % g.page_size;
      uint8_t* chunk = pages + ((size_t)page * g.num_kv_heads + cur.h) * (size_t)g.page_bytes;
      uint8_t* dst = chunk + (size_t)half * g.page_size * vb + (size_t)off * vb;
      if (BITS == 4) {
        uint32_t word = 0;
#pragma unroll
        for (int e = 0; e < 8; ++e) word |= (uint32_t)code[e] << (4 * e);
        if (half == 0) {
          *reinterpret_cast<uint32_t*>(dst + 4 * j) = word;
        } else {
          // V: token pairs (2p, 2p+1) share 128 bytes; the 8-byte unit of 16-dim group c of
          // token 2p + h sits at 16 * (c ^ (2p mod 8)) + 8h.  Lane j holds half of unit j / 2.
          const int pair = off >> 1, hv = off & 1, c = j >> 1;
          uint8_t* vsec = chunk + (size_t)g.page_size * vb;
          *reinterpret_cast<uint32_t*>(vsec + pair * 128 + 16 * (c ^ ((2 * pair) & 7)) + 8 * hv + 4 * (j & 1)) = word;
        }
      } else {
        // Lane j covers dims 8m..8m+7 of 32-dim group w = j/4 (m = j%4).  Its low bits are
        // bytes 2m, 2m+1 of the group's W0|W1; its high bits fill half of bytes 2(m&1) and
        // 2(m&1)+1 of W2, shared with lane j^2 (same k, other h).
        const int w = j >> 2, m = j & 3, hh = m >> 1;
        uint32_t lo = 0, hib = 0;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          lo |= (uint32_t)(code[e] & 3) << (2 * e);
          const int r = e & 3, kk = e >> 2;  // dim 8m + e = 16hh + 4(2(m&1) + kk) + r
          const int off_r = (r < 2) ? 4 + r : r - 2;
          hib |= (uint32_t)(code[e] >> 2) << (8 * kk + 2 * hh + off_r);
        }
        const uint32_t partner = __shfl_xor_sync(0xffffffffu, hib, 2);
        *reinterpret_cast<uint16_t*>(dst + 12 * w + 2 * m) = (uint16_t)lo;
        if (hh == 0) *reinterpret_cast<uint16_t*>(dst + 12 * w + 8 + 2 * (m & 1)) = (uint16_t)(hib | partner);
      }
      if (j == 0) {
        const __half n16 = __float2half_rn(nrm);
        uint8_t* nb = chunk + (size_t)2 * g.page_size * vb + (size_t)half * 2 * g.page_size + 2 * off;
        *reinterpret_cast<__half*>(nb) = n16;
        if (status && __hisinf(n16)) atomicOr(status, RQ_STATUS_NORM_OVERFLOW);
      }
    }
    cur = nxt;
  }
}

}  // namespace

cudaError_t launch_append(const Geometry& g, const void* k, const void* v, const int32_t* slots, int n,
                          uint8_t* pages, int32_t* status, cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  static int max_blocks = 0;
  if (max_blocks == 0) {
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    max_blocks = (sms > 0 ? sms : 132) * (2048 / kAppendThreads);
  }
  const long long items = (long long)n * g.num_kv_heads;
  long long blocks = (items + kAppendWarps - 1) / kAppendWarps;
  if (blocks > max_blocks) blocks = max_blocks;
  if (g.bits == 4)
    append_kernel<4><<<(unsigned)blocks, kAppendThreads, 0, stream>>>(g, (const __half*)k, (const __half*)v,
                                                                     slots, n, pages, status);
  else
    append_kernel<3><<<(unsigned)blocks, kAppendThreads, 0, stream>>>(g, (const __half*)k, (const __half*)v,
                                                                     slots, n, pages, status);
  return cudaGetLastError();
}

}  // namespace rq
