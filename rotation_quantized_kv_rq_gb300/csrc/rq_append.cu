// Fused quantize-pack-append ("SGLang 1-Bit Turbo" README, section "RotorQuant KV Cache
// Compression": norm, fixed data-oblivious rotation -- 2D Givens pairs or 4D quaternion
// blocks -- then Lloyd-Max scalar codes, bit-packed into the paged cache).
//
// One warp encodes the K and the V vector of one (token, kv head).  Lane l owns dimensions
// 4l..4l+3, which hold two whole Givens pairs or one whole quaternion block, so the rotation
// needs no data from other lanes; only the squared norm is reduced across the warp.
// The kernel is bound by HBM: 512 bytes of fp16 in, 2 * (16 * bits + 2) bytes out per
// (token, head).
#include <cuda_fp16.h>

#include "rq_internal.h"
#include "../../include/rq.h"

namespace rq {
namespace {

constexpr int kAppendWarps = 8;

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Number of boundaries strictly below u: branchless binary search over the sorted table.
template <int BITS>
__device__ __forceinline__ int code_of(float u, const float* bnd) {
  int lo = 0;
#pragma unroll
  for (int step = (1 << BITS) / 2; step >= 1; step >>= 1)
    if (bnd[lo + step - 1] < u) lo += step;
  return lo;
}

template <int BITS>
__global__ void __launch_bounds__(kAppendWarps * 32)
append_kernel(Geometry g, const __half* __restrict__ k, const __half* __restrict__ v,
              const int32_t* __restrict__ slots, int n, uint8_t* __restrict__ pages,
              int32_t* __restrict__ status) {
  __shared__ float bnd[16];
  if (threadIdx.x < (1 << BITS) - 1) bnd[threadIdx.x] = g.boundaries[threadIdx.x];
  __syncthreads();

  const int lane = threadIdx.x & 31;
  const long long item = (long long)blockIdx.x * kAppendWarps + (threadIdx.x >> 5);
  if (item >= (long long)n * g.num_kv_heads) return;
  const int t = (int)(item / g.num_kv_heads);
  const int h = (int)(item % g.num_kv_heads);
  const int slot = slots[t];
  if (slot < 0) return;
  if ((long long)slot >= (long long)g.num_pages * g.page_size) {
    if (lane == 0 && status) atomicOr(status, RQ_STATUS_BAD_SLOT);
    return;
  }
  const int page = slot / g.page_size, off = slot % g.page_size;
  uint8_t* chunk = pages + ((size_t)page * g.num_kv_heads + h) * (size_t)g.page_bytes;
  const int vb = BITS * 16;

  // Issue both loads before any arithmetic.
  const size_t src = ((size_t)t * g.num_kv_heads + h) * kHeadDim + 4 * lane;
  uint2 raw[2];
  raw[0] = __ldg(reinterpret_cast<const uint2*>(k + src));
  raw[1] = __ldg(reinterpret_cast<const uint2*>(v + src));

#pragma unroll
  for (int which = 0; which < 2; ++which) {
    const float4 p = __ldg(reinterpret_cast<const float4*>((which ? g.rot_v : g.rot_k) + (size_t)h * kHeadDim) + lane);
    const float2 x01 = __half22float2(*reinterpret_cast<const __half2*>(&raw[which].x));
    const float2 x23 = __half22float2(*reinterpret_cast<const __half2*>(&raw[which].y));
    float x[4] = {x01.x, x01.y, x23.x, x23.y};
    float ss = x[0] * x[0] + x[1] * x[1] + x[2] * x[2] + x[3] * x[3];
    ss = warp_sum(ss);
    const float nrm = __fsqrt_rn(ss);

    float y[4];
    if (g.mode == RQ_PLANAR) {
      y[0] = p.x * x[0] - p.y * x[1];
      y[1] = p.y * x[0] + p.x * x[1];
      y[2] = p.z * x[2] - p.w * x[3];
      y[3] = p.w * x[2] + p.z * x[3];
    } else {  // Hamilton product (a,b,c,d) (x) (x0,x1,x2,x3)
      const float a = p.x, b = p.y, c = p.z, d = p.w;
      y[0] = a * x[0] - b * x[1] - c * x[2] - d * x[3];
      y[1] = b * x[0] + a * x[1] - d * x[2] + c * x[3];
      y[2] = c * x[0] + d * x[1] + a * x[2] - b * x[3];
      y[3] = d * x[0] - c * x[1] + b * x[2] + a * x[3];
    }
    int code[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const float u = nrm > 0.f ? __fdiv_rn(y[r], nrm) : 0.f;
      code[r] = code_of<BITS>(u, bnd);
    }

    uint8_t* dst = chunk + (size_t)which * g.page_size * vb + (size_t)off * vb;
    if (BITS == 4) {
      const uint16_t two = (uint16_t)(code[0] | (code[1] << 4) | (code[2] << 8) | (code[3] << 12));
      *reinterpret_cast<uint16_t*>(dst + 2 * lane) = two;
    } else {
      // Lane l covers dims 4j..4j+3 of 32-dim group w = l/8 (j = l%8).  Its low bits form
      // byte j of the group's W0|W1; its high bits go to byte j%4 of W2 at bits
      // 2*(j/4) + {4,5,0,1}[r], shared with lane j^4.
      const int w = lane >> 3, j = lane & 7, hh = j >> 2;
      const uint32_t lo = (code[0] & 3) | ((code[1] & 3) << 2) | ((code[2] & 3) << 4) | ((code[3] & 3) << 6);
      const uint32_t hib = ((code[0] >> 2) << (2 * hh + 4)) | ((code[1] >> 2) << (2 * hh + 5)) |
                           ((code[2] >> 2) << (2 * hh)) | ((code[3] >> 2) << (2 * hh + 1));
      const uint32_t partner = __shfl_down_sync(0xffffffffu, hib, 4);
      dst[12 * w + j] = (uint8_t)lo;
      if (hh == 0) dst[12 * w + 8 + j] = (uint8_t)(hib | partner);
    }
    if (lane == 0) {
      const __half n16 = __float2half_rn(nrm);
      uint8_t* nb = chunk + (size_t)2 * g.page_size * vb + (size_t)which * 2 * g.page_size + 2 * off;
      *reinterpret_cast<__half*>(nb) = n16;
      if (status && __hisinf(n16)) atomicOr(status, RQ_STATUS_NORM_OVERFLOW);
    }
  }
}

}  // namespace

cudaError_t launch_append(const Geometry& g, const void* k, const void* v, const int32_t* slots, int n,
                          uint8_t* pages, int32_t* status, cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  const long long items = (long long)n * g.num_kv_heads;
  const unsigned blocks = (unsigned)((items + kAppendWarps - 1) / kAppendWarps);
  if (g.bits == 4)
    append_kernel<4><<<blocks, kAppendWarps * 32, 0, stream>>>(g, (const __half*)k, (const __half*)v, slots, n,
                                                               pages, status);
  else
    append_kernel<3><<<blocks, kAppendWarps * 32, 0, stream>>>(g, (const __half*)k, (const __half*)v, slots, n,
                                                               pages, status);
  return cudaGetLastError();
}

}  // namespace rq
