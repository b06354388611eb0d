// Fused quantize-pack-append ("SGLang 1-Bit Turbo" README, section "RotorQuant KV Cache
// Compression": norm, fixed data-oblivious rotation -- 2D Givens pairs or 4D quaternion
// blocks -- then Lloyd-Max scalar codes, bit-packed into the paged cache; section "TurboQuant
// KV Cache Compression" for the dense random rotation).
//
// Structured rotations (planar / iso): work item = one (token, kv head).  A warp takes items
// in a grid-stride loop: lanes 0-15 encode the K vector and lanes 16-31 the V vector.  Lane j
// of a half owns dimensions 8j..8j+7 -- four whole Givens pairs or two whole quaternion
// blocks -- so the rotation is lane-local and only the squared norm is reduced (4
// xor-shuffles within the half).  Each lane reads 16 bytes, and the next item's 16 bytes are
// in flight while the current one is coded.  The kernel is bound by HBM: 512 bytes of fp16
// in, 2 * (16 * bits + 2) bytes out per item.
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
constexpr int kAppendWarps = kAppendThreads / 32;

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
struct Item {
  int t, h, slot;
  uint4 raw;  // 8 fp16 of this lane's half (K or V)
};

__device__ __forceinline__ void fetch(Item& it, int t, int h, const Geometry& g, const __half* src_k,
                                      const __half* src_v, const int32_t* slots, int half, int j) {
  it.t = t;
  it.h = h;
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
  load_boundaries<BITS>(bnd, g.boundaries);

  const int lane = threadIdx.x & 31;
  const int half = lane >> 4;        // 0: K, 1: V
  const int j = lane & 15;           // dims 8j..8j+7
  const long long items = (long long)n * g.num_kv_heads;
  const long long stride = (long long)gridDim.x * kAppendWarps;
  const float* rot = half ? g.rot_v : g.rot_k;
  const long long pool_slots = (long long)g.num_pages * g.page_size;
  const PageSplit split(g.page_size);

  long long item = (long long)blockIdx.x * kAppendWarps + (threadIdx.x >> 5);
  if (item >= items) return;
  // item = t * Hkv + h: divided once, then advanced by the stride without dividing (a 64-bit
  // division is a long instruction sequence, comparable to coding the vectors)
  const int hkv = g.num_kv_heads;
  int t = (int)(item / hkv), h = (int)(item % hkv);
  const int stride_t = (int)(stride / hkv), stride_h = (int)(stride % hkv);
  Item cur, nxt;
  fetch(cur, t, h, g, k, v, slots, half, j);
  for (; item < items; item += stride) {
    t += stride_t;
    h += stride_h;
    if (h >= hkv) {
      h -= hkv;
      ++t;
    }
    if (item + stride < items) fetch(nxt, t, h, g, k, v, slots, half, j);

    const int slot = cur.slot;
    const bool bad = (long long)slot >= pool_slots;
    if (bad && lane == 0 && status) atomicOr(status, RQ_STATUS_BAD_SLOT);
    if (slot >= 0 && !bad) {  // uniform across the warp
      const float4 p0 = __ldg(reinterpret_cast<const float4*>(rot + (size_t)cur.h * kHeadDim + 8 * j));
      const float4 p1 = __ldg(reinterpret_cast<const float4*>(rot + (size_t)cur.h * kHeadDim + 8 * j + 4));
      const float pr[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
      int page, off;
      split(slot, page, off);
      uint8_t* chunk = pages + ((size_t)page * g.num_kv_heads + cur.h) * (size_t)g.page_bytes;
      encode_structured<BITS>(cur.raw, pr, g.mode, bnd, chunk, g.page_size, half, off, j, true, status);
    }
    cur = nxt;
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
    long long blocks = (items + kAppendWarps - 1) / kAppendWarps;
    const long long max_blocks = (long long)sms * (2048 / kAppendThreads);
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
