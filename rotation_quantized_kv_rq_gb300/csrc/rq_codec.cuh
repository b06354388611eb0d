// Codec device code shared by the append kernels and the decode-step append inside the
// attention kernel: the code search over the fp32 bin boundaries, and the packing of a
// vector's codes into the storage contract of include/rq.h (section "RotorQuant KV Cache
// Compression" of the "SGLang 1-Bit Turbo" README for the method; the bit layout is this
// library's).  A vector is coded by a half-warp: lane j holds its dims 8j..8j+7.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

#include "../../include/rq.h"
#include "rq_internal.h"

namespace rq {
namespace codec {

// Number of boundaries strictly below u (b ascending, in registers): a binary search written as
// a select tree, one compare per level and no indexed memory.
template <int BITS>
__device__ __forceinline__ int code_of(float u, const float (&b)[15]) {
  if constexpr (BITS == 2) {
    const bool s1 = u > b[1];
    const bool s0 = u > (s1 ? b[2] : b[0]);
    return (s1 ? 2 : 0) + (s0 ? 1 : 0);
  } else if constexpr (BITS == 3) {
    const bool s2 = u > b[3];
    const bool s1 = u > (s2 ? b[5] : b[1]);
    const bool s0 = u > (s2 ? (s1 ? b[6] : b[4]) : (s1 ? b[2] : b[0]));
    return (s2 ? 4 : 0) + (s1 ? 2 : 0) + (s0 ? 1 : 0);
  } else {
    const bool s3 = u > b[7];
    const bool s2 = u > (s3 ? b[11] : b[3]);
    const bool s1 = u > (s3 ? (s2 ? b[13] : b[9]) : (s2 ? b[5] : b[1]));
    const float m0 = s3 ? (s2 ? (s1 ? b[14] : b[12]) : (s1 ? b[10] : b[8]))
                        : (s2 ? (s1 ? b[6] : b[4]) : (s1 ? b[2] : b[0]));
    const bool s0 = u > m0;
    return (s3 ? 8 : 0) + (s2 ? 4 : 0) + (s1 ? 2 : 0) + (s0 ? 1 : 0);
  }
}

// code_of that also returns the distance from u to the nearest boundary: the boundaries on
// either side of u are both among those the search compares against.
template <int BITS>
__device__ __forceinline__ int code_of_margin(float u, const float (&b)[15], float& dmin) {
  if constexpr (BITS == 2) {
    const bool s1 = u > b[1];
    const float m0 = s1 ? b[2] : b[0];
    dmin = fminf(fabsf(u - b[1]), fabsf(u - m0));
    return (s1 ? 2 : 0) + (u > m0 ? 1 : 0);
  } else if constexpr (BITS == 3) {
    const bool s2 = u > b[3];
    const float m1 = s2 ? b[5] : b[1];
    const bool s1 = u > m1;
    const float m0 = s2 ? (s1 ? b[6] : b[4]) : (s1 ? b[2] : b[0]);
    dmin = fminf(fminf(fabsf(u - b[3]), fabsf(u - m1)), fabsf(u - m0));
    return (s2 ? 4 : 0) + (s1 ? 2 : 0) + (u > m0 ? 1 : 0);
  } else {
    const bool s3 = u > b[7];
    const float m2 = s3 ? b[11] : b[3];
    const bool s2 = u > m2;
    const float m1 = s3 ? (s2 ? b[13] : b[9]) : (s2 ? b[5] : b[1]);
    const bool s1 = u > m1;
    const float m0 = s3 ? (s2 ? (s1 ? b[14] : b[12]) : (s1 ? b[10] : b[8]))
                        : (s2 ? (s1 ? b[6] : b[4]) : (s1 ? b[2] : b[0]));
    dmin = fminf(fminf(fabsf(u - b[7]), fabsf(u - m2)), fminf(fabsf(u - m1), fabsf(u - m0)));
    return (s3 ? 8 : 0) + (s2 ? 4 : 0) + (s1 ? 2 : 0) + (u > m0 ? 1 : 0);
  }
}

// A lane's share of one coded vector: its packed codes (see pack_codes) and the vector's fp16
// norm (bits).
struct Packed {
  uint32_t codes;
  uint32_t norm;
};

// Packs the codes of dims 8j..8j+7 (j = lane within its half-warp) of one vector: 4-bit, eight
// nibbles; 2-bit, 16 bits; 3-bit, the low bits (16) | the high-bit bytes (16) that lanes j and
// j ^ 2 share, exchanged here.  Every lane of the warp must call it.
template <int BITS>
__device__ __forceinline__ uint32_t pack_codes(const int (&code)[8], int j) {
  if constexpr (BITS == 4) {
    uint32_t word = 0;
#pragma unroll
    for (int e = 0; e < 8; ++e) word |= (uint32_t)code[e] << (4 * e);
    return word;
  } else if constexpr (BITS == 2) {
    uint32_t half_word = 0;
#pragma unroll
    for (int e = 0; e < 8; ++e) half_word |= (uint32_t)code[e] << (2 * e);
    return half_word;
  } else {
    // Lane j covers dims 8m..8m+7 of 32-dim group w = j/4 (m = j%4).  Its low bits are
    // bytes 2m, 2m+1 of the group's W0|W1; its high bits fill half of bytes 2(m&1) and
    // 2(m&1)+1 of W2, shared with lane j^2 (same k, other h).
    const int m = j & 3, hh = m >> 1;
    uint32_t lo = 0, hib = 0;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      lo |= (uint32_t)(code[e] & 3) << (2 * e);
      const int r = e & 3, kk = e >> 2;  // dim 8m + e = 16hh + 4(2(m&1) + kk) + r
      const int off_r = (r < 2) ? 4 + r : r - 2;
      hib |= (uint32_t)(code[e] >> 2) << (8 * kk + 2 * hh + off_r);
    }
    const uint32_t partner = __shfl_xor_sync(0xffffffffu, hib, 2);
    return lo | (hib | partner) << 16;
  }
}

// Writes a lane's packed codes and (lane j == 0) the norm to the vector's place in `chunk`
// (kind 0 = K, 1 = V; `off` = offset in page).  No shuffles: any subset of lanes may call it.
// A non-null status gets RQ_STATUS_NORM_OVERFLOW for an infinite norm.
template <int BITS>
__device__ __forceinline__ void store_packed(Packed pk, uint8_t* chunk, int page_size, int kind, int off, int j,
                                             int32_t* status) {
  constexpr int vb = BITS * 16;
  uint8_t* dst = chunk + (size_t)kind * page_size * vb + (size_t)off * vb;
  uint8_t* vsec = chunk + (size_t)page_size * vb;
  const int pair = off >> 1, hv = off & 1, c = j >> 1;  // V pair placement (2- and 4-bit)
  if constexpr (BITS == 4) {
    if (kind == 0) {
      *reinterpret_cast<uint32_t*>(dst + 4 * j) = pk.codes;
    } else {
      // V: token pairs (2p, 2p+1) share 128 bytes; the 8-byte unit of 16-dim group c of
      // token 2p + h sits at 16 * (c ^ (2p mod 8)) + 8h.  Lane j holds half of unit j / 2.
      *reinterpret_cast<uint32_t*>(vsec + pair * 128 + 16 * (c ^ ((2 * pair) & 7)) + 8 * hv + 4 * (j & 1)) = pk.codes;
    }
  } else if constexpr (BITS == 2) {
    if (kind == 0) {
      *reinterpret_cast<uint16_t*>(dst + 2 * j) = (uint16_t)pk.codes;
    } else {
      // V: token pairs share 64 bytes; the 4-byte unit of group c of token 2p + h sits at
      // 8 * (c ^ (4 * (p / 2 mod 2))) + 4h.  Lane j holds half of unit j / 2.
      *reinterpret_cast<uint16_t*>(vsec + pair * 64 + 8 * (c ^ (4 * ((pair >> 1) & 1))) + 4 * hv + 2 * (j & 1)) =
          (uint16_t)pk.codes;
    }
  } else {
    const int w = j >> 2, m = j & 3, hh = m >> 1;
    *reinterpret_cast<uint16_t*>(dst + 12 * w + 2 * m) = (uint16_t)pk.codes;
    if (hh == 0) *reinterpret_cast<uint16_t*>(dst + 12 * w + 8 + 2 * (m & 1)) = (uint16_t)(pk.codes >> 16);
  }
  if (j == 0) {
    const __half n16 = __ushort_as_half((unsigned short)pk.norm);
    uint8_t* nb = chunk + (size_t)2 * page_size * vb + (size_t)kind * 2 * page_size + 2 * off;
    *reinterpret_cast<__half*>(nb) = n16;
    if (status && __hisinf(n16)) atomicOr(status, RQ_STATUS_NORM_OVERFLOW);
  }
}

// pack_codes + store_packed: the vector's codes and fp16 norm to its place in `chunk`.  Every
// lane of the warp must call it; with `store` false nothing is written.
template <int BITS>
__device__ __forceinline__ void pack_store(const int (&code)[8], float nrm, uint8_t* chunk, int page_size, int kind,
                                           int off, int j, bool store, int32_t* status) {
  const Packed pk{pack_codes<BITS>(code, j), (uint32_t)__half_as_ushort(__float2half_rn(nrm))};
  if (store) store_packed<BITS>(pk, chunk, page_size, kind, off, j, status);
}

// 1 / n, so that u = y / n is formed as y * (1/n): within an ulp of the quotient, so a code can
// differ from the quotient's only for u within ~1e-7 of a boundary.  n = 0 gives u = 0.
__device__ __forceinline__ float inv_norm(float nrm) { return nrm > 0.f ? __frcp_rn(nrm) : 0.f; }

template <int BITS>
__device__ __forceinline__ void load_boundaries(float (&bnd)[15], const float* boundaries) {
#pragma unroll
  for (int i = 0; i < 15; ++i) bnd[i] = i < (1 << BITS) - 1 ? __ldg(boundaries + i) : 0.f;
}


// The structured rotation of the lane's 8 dims (dims 8j..8j+7: four Givens pairs or two
// quaternion blocks), p = the lane's 8 parameters.
__device__ __forceinline__ void rotate8(float (&y)[8], const float (&x)[8], const float (&p)[8], int mode) {
  if (mode == RQ_PLANAR) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float c = p[2 * q], s = p[2 * q + 1];
      y[2 * q] = c * x[2 * q] - s * x[2 * q + 1];
      y[2 * q + 1] = s * x[2 * q] + c * x[2 * q + 1];
    }
  } else {  // Hamilton product (a,b,c,d) (x) (x0,x1,x2,x3)
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const float a = p[4 * q], b = p[4 * q + 1], c = p[4 * q + 2], d = p[4 * q + 3];
      const float* xb = x + 4 * q;
      y[4 * q + 0] = a * xb[0] - b * xb[1] - c * xb[2] - d * xb[3];
      y[4 * q + 1] = b * xb[0] + a * xb[1] - d * xb[2] + c * xb[3];
      y[4 * q + 2] = c * xb[0] + d * xb[1] + a * xb[2] - b * xb[3];
      y[4 * q + 3] = d * xb[0] - c * xb[1] + b * xb[2] + a * xb[3];
    }
  }
}

// Codes one fp16 vector with a structured rotation: lane j of the half-warp passes its 16 bytes
// of x (dims 8j..8j+7) and its rotation parameters, and gets its share of the result.  Every
// lane of the warp must call it (shuffles).
template <int BITS>
__device__ __forceinline__ Packed encode_packed(uint4 raw, const float (&p)[8], int mode, const float (&bnd)[15],
                                                int j) {
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
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
  rotate8(y, x, p, mode);
  const float rcp = inv_norm(nrm);
  int code[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) code[e] = code_of<BITS>(y[e] * rcp, bnd);
  return Packed{pack_codes<BITS>(code, j), (uint32_t)__half_as_ushort(__float2half_rn(nrm))};
}

// y_i = sum_m x_m R[i][m] for one vector, summed exactly enough to be correctly rounded in all
// but pathological cases: error-free products (fma) and error-free sums (two-sum), the rounding
// errors carried in a second word.  Lane j of the half-warp holds x[8j..8j+7]; `row` is R's row
// i in global memory (rarely read: L2).  Every lane of the warp calls it (shuffles stay within
// each half).
__device__ __forceinline__ float dot_compensated(const float (&x)[8], const float* row, int j) {
  const float4 r0 = __ldg(reinterpret_cast<const float4*>(row + 8 * j));
  const float4 r1 = __ldg(reinterpret_cast<const float4*>(row + 8 * j + 4));
  const float rr[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
  float s = 0.f, c = 0.f;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const float p = x[e] * rr[e];
    const float pe = fmaf(x[e], rr[e], -p);  // x * r = p + pe exactly
    const float t = s + p;
    const float z = t - s;
    c += ((s - (t - z)) + (p - z)) + pe;     // s + p = t + (that) exactly
    s = t;
  }
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) {
    const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
    const float c2 = __shfl_xor_sync(0xffffffffu, c, o);
    const float t = s + s2;
    const float z = t - s;
    c += c2 + ((s - (t - z)) + (s2 - z));
    s = t;
  }
  return s + c;
}

// A dense rotation's y = R x is computed approximately (tensor cores, or an fp32 multiply-add
// chain) and trusted to decide a code when u is farther than this from every boundary.  The
// tensor-core error is the hi + lo split (|R - hi - lo| <= 6e-8 per entry, so <= 7e-7 in u by
// Cauchy-Schwarz) plus the accumulation of 16 fp32 MMA steps (a few fp32 ulps of n each); an fp32
// chain of 128 multiply-adds stays well inside it too.
constexpr float kFixBand = 1e-5f;

// code_of through the binned code table in shared memory (rq_internal.h): the bin is
// RNE(u * kCodeBinScale) (u times a power of two is exact, and adding 1.5 * 2^23 rounds it to an
// integer in the low mantissa bits), clamped to the out-of-range entry; near = u lies within
// kFixBand of a boundary.  The bin's one boundary is the only one within 2e-5 of it, so both
// equal what the select tree and code_of_margin decide, NaN included (code 0, not near).
__device__ __forceinline__ int code_of_table(float u, const uint2* tab, bool& near) {
  const float t = fmaf(u, (float)kCodeBinScale, 12582912.f);
  const uint32_t k = min(__float_as_uint(t) - (0x4B400000u - (uint32_t)kCodeBinHalf), (uint32_t)(kCodeBins - 1));
  const uint2 e = tab[k];
  const float b = __uint_as_float(e.y);
  near = fabsf(u - b) < kFixBand;
  return (int)e.x + (u > b ? 1 : 0);
}

// Codes of one vector under a dense rotation, a half-warp per vector (lane j: dims 8j..8j+7):
// raw = the lane's 16 bytes of x (fp16), y = its 8 coordinates of the approximate R x.  Each
// coordinate whose u lies within kFixBand of a boundary is recomputed with dot_compensated from
// the fp32 rows of R (r32, row-major), one at a time per half-warp (both halves walk their lists
// together), and re-coded; so the codes are those of the correctly rounded y, whichever
// approximation gave y.  Also returns the fp32 norm.  Every lane of the warp must call it.
template <int BITS>
__device__ __forceinline__ void dense_codes(int (&code)[8], float& nrm, uint4 raw, const float (&y)[8],
                                            const float (&bnd)[15], const float* r32, bool store, int lane) {
  const int half = lane >> 4, j = lane & 15;
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
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
  nrm = __fsqrt_rn(ss);
  const float rcp = inv_norm(nrm);
  uint32_t todo = 0;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    float dm;
    code[e] = code_of_margin<BITS>(y[e] * rcp, bnd, dm);
    if (dm < kFixBand && store) todo |= 1u << e;
  }
  while (__any_sync(0xffffffffu, todo != 0)) {
    const uint32_t want = __ballot_sync(0xffffffffu, todo != 0) & (half ? 0xffff0000u : 0x0000ffffu);
    const int leader = want ? __ffs(want) - 1 : (half << 4);  // no work: any lane, result unused
    const int e_lead = __shfl_sync(0xffffffffu, todo ? __ffs(todo) - 1 : 0, leader);
    const int i = 8 * (leader & 15) + e_lead;  // the coordinate (dim of y) being recomputed
    const float yi = dot_compensated(x, r32 + i * 128, j);
    if (lane == leader && want) {
      const int c = code_of<BITS>(yi * rcp, bnd);
#pragma unroll
      for (int e = 0; e < 8; ++e)
        if (e == e_lead) code[e] = c;
      todo &= ~(1u << e_lead);
    }
  }
}

// encode_packed, written to slot `off` of `chunk` (`store` false writes nothing).
template <int BITS>
__device__ __forceinline__ void encode_structured(uint4 raw, const float (&p)[8], int mode, const float (&bnd)[15],
                                                  uint8_t* chunk, int page_size, int kind, int off, int j, bool store,
                                                  int32_t* status) {
  const Packed pk = encode_packed<BITS>(raw, p, mode, bnd, j);
  if (store) store_packed<BITS>(pk, chunk, page_size, kind, off, j, status);
}

}  // namespace codec
}  // namespace rq
