// Extend (prefill) attention over the packed cache: T new query tokens per sequence, each
// attending causally to the cached prefix and to the new tokens up to itself ("SGLang 1-Bit
// Turbo" README, section "RotorQuant KV Cache Compression": queries are rotated once, values
// summed in the rotated space and the output rotated back once).  Query row j of sequence b
// sees positions 0 .. seq_lens[b] - T + j -- the definition of chain verify, here for T in the
// hundreds or thousands, where the split-K kernel (which re-reads the cache for every 8 query
// rows) stops paying.
//
// Design (sm_103a): a CTA of 4 warps takes 64 query rows of one (sequence, kv head) -- rows
// r = j * group + k -- and walks the cache in 32-token tiles up to the last position its rows
// can see.  Each thread owns the K and V 32-dim code groups of one (token, group) pair of a
// tile: it loads the next tile's code words and norms into registers while the current tile's
// MMAs run, then dequantizes them into fp16 shared memory (centroid values; the norms scale the
// scores and the probabilities), shared by all 64 rows: every warp computes S = Q~ K~^T for its
// 16 rows and O~ += P' V~ with mma.sync m16n8k16, reading K~ and V~ with ldmatrix (V~
// transposed).  Online softmax in base 2 as in the split-K kernel.
#include <cuda_fp16.h>
#include <math_constants.h>

#include "rq_internal.h"
#include "../../include/rq.h"

namespace rq {
namespace {

constexpr int kXWarps = 4;
constexpr int kXThreads = 32 * kXWarps;
constexpr int kXRows = 16 * kXWarps;  // query rows per CTA
constexpr int kXTok = 32;             // tokens per K/V tile
constexpr int kXOStride = 132;        // floats per staged output row
// shared memory: K~ and V~ tiles fp16 [32][128] (16-byte chunks XOR-swizzled by row), the
// tile's norms, the fp16 centroids, then the query staging (fp16 [64][128]) that the output
// staging (fp32 [64][132]) later reuses
constexpr int kXSmemK = 0;
constexpr int kXSmemV = kXSmemK + kXTok * 256;
constexpr int kXSmemNk = kXSmemV + kXTok * 256;
constexpr int kXSmemNv = kXSmemNk + kXTok * 4;
constexpr int kXSmemCb = kXSmemNv + kXTok * 4;
constexpr int kXSmemQ = kXSmemCb + 64;
constexpr int kXSmem = kXSmemQ + kXRows * kXOStride * 4;  // 50,496 bytes

__device__ __forceinline__ uint32_t xswz(int row, int chunk) { return (uint32_t)(row * 256 + ((chunk ^ (row & 7)) << 4)); }

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
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
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// One (token, 32-dim group) of a K or V vector as stored (include/rq.h): the code words and the
// token's fp16 norm, loaded from global memory ahead of use.
struct GroupRaw {
  uint32_t w[4];  // 4-bit: 4 words (8 codes each); 2-bit: 2 words (16 each); 3-bit: W0, W1, W2
  uint32_t norm;  // fp16 bits (group 0 only), 0 past the sequence
};

// Loads group g of token pos of kind (0 K, 1 V) of the (sequence, kv head) whose page table row
// is bt (npages valid entries); zeros past len.  Page ids outside the pool read page 0 and set
// RQ_STATUS_BAD_PAGE.
template <int BITS>
__device__ __forceinline__ void load_group(GroupRaw& r, const Geometry& g, const AttnArgs& a, const int32_t* bt,
                                           int h, int pos, int len, int kind, int grp) {
  constexpr int vb = 16 * BITS;
  r.w[0] = r.w[1] = r.w[2] = r.w[3] = 0u;
  r.norm = 0u;
  if (pos >= len) return;
  const int P = g.page_size;
  int page = __ldg(bt + pos / P);
  if (page < 0 || page >= g.num_pages) {
    if (a.status) atomicOr(a.status, RQ_STATUS_BAD_PAGE);
    page = 0;
  }
  const int off = pos % P;
  const uint8_t* chunk = a.pages + ((size_t)page * g.num_kv_heads + h) * g.page_bytes;
  const uint8_t* sec = chunk + (size_t)kind * P * vb;
  if constexpr (BITS == 4) {
    if (kind == 0) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(sec + off * vb + 16 * grp));
      r.w[0] = v.x, r.w[1] = v.y, r.w[2] = v.z, r.w[3] = v.w;
    } else {  // pair rows: unit u of token 2p + h at 16 (u ^ 2p mod 8) + 8h, units 2 grp, 2 grp + 1
      const int p = off >> 1;
      const uint8_t* row = sec + p * 128 + 8 * (off & 1);
      const uint2 u0 = __ldg(reinterpret_cast<const uint2*>(row + 16 * ((2 * grp) ^ ((2 * p) & 7))));
      const uint2 u1 = __ldg(reinterpret_cast<const uint2*>(row + 16 * ((2 * grp + 1) ^ ((2 * p) & 7))));
      r.w[0] = u0.x, r.w[1] = u0.y, r.w[2] = u1.x, r.w[3] = u1.y;
    }
  } else if constexpr (BITS == 2) {
    if (kind == 0) {
      const uint2 v = __ldg(reinterpret_cast<const uint2*>(sec + off * vb + 8 * grp));
      r.w[0] = v.x, r.w[1] = v.y;
    } else {  // pair rows: unit u of token 2p + h at 8 (u ^ 4 (p/2 mod 2)) + 4h
      const int p = off >> 1;
      const uint8_t* row = sec + p * 64 + 4 * (off & 1);
      r.w[0] = __ldg(reinterpret_cast<const uint32_t*>(row + 8 * ((2 * grp) ^ (4 * ((p >> 1) & 1)))));
      r.w[1] = __ldg(reinterpret_cast<const uint32_t*>(row + 8 * ((2 * grp + 1) ^ (4 * ((p >> 1) & 1)))));
    }
  } else {  // 12 bytes of group grp: W0, W1, W2
    const uint32_t* gw = reinterpret_cast<const uint32_t*>(sec + off * vb + 12 * grp);
    r.w[0] = __ldg(gw), r.w[1] = __ldg(gw + 1), r.w[2] = __ldg(gw + 2);
  }
  if (grp == 0)
    r.norm = __ldg(reinterpret_cast<const uint16_t*>(chunk + (size_t)2 * P * vb + kind * 2 * P + 2 * off));
}

// The code of dim i (0..31) of a loaded group.
template <int BITS>
__device__ __forceinline__ int group_code(const GroupRaw& r, int i) {
  if constexpr (BITS == 4) {
    return (int)((r.w[i >> 3] >> (4 * (i & 7))) & 15u);
  } else if constexpr (BITS == 2) {
    return (int)((r.w[i >> 4] >> (2 * (i & 15))) & 3u);
  } else {  // low bits: W0 (dims 0-15) / W1 (16-31); high bit of i = 16h + 4k + r at 8k + 2h + {4,5,0,1}[r]
    const int lo = (int)((r.w[i >> 4] >> (2 * (i & 15))) & 3u);
    const int hh = i >> 4, k = (i >> 2) & 3, rr = i & 3;
    const int bit = 8 * k + 2 * hh + (rr < 2 ? 4 + rr : rr - 2);
    return lo | (int)(((r.w[2] >> bit) & 1u) << 2);
  }
}

template <int BITS>
__global__ void __launch_bounds__(kXThreads)
extend_kernel(const Geometry g, const AttnArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t sbase = (uint32_t)__cvta_generic_to_shared(smem);
  float* nk = reinterpret_cast<float*>(smem + kXSmemNk);
  float* nv = reinterpret_cast<float*>(smem + kXSmemNv);
  __half* cb16 = reinterpret_cast<__half*>(smem + kXSmemCb);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gq = lane >> 2, tq = lane & 3;
  const int n_rb = (a.rows + kXRows - 1) / kXRows;
  const int rb = blockIdx.x % n_rb;
  const int h = (blockIdx.x / n_rb) % g.num_kv_heads;
  const int b = blockIdx.x / (n_rb * g.num_kv_heads);
  const int P = g.page_size;
  const int cap = a.max_pages * P;
  int len = a.seq_lens[b];
  if (len < 0 || len > cap || (len > 0 && len < a.T)) {
    if (rb == 0 && h == 0 && threadIdx.x == 0 && a.status) atomicOr(a.status, RQ_STATUS_BAD_LEN);
    len = len < 0 ? 0 : (len > cap ? cap : len);
  }
  if (threadIdx.x < (1 << BITS)) cb16[threadIdx.x] = __float2half_rn(g.centroids[threadIdx.x]);

  // ---- q~ = R_k q * sm_scale * log2(e) of the CTA's 64 rows, fp16, staged for ldmatrix ----
  const __half* qh = reinterpret_cast<const __half*>(a.q);
  for (int i = threadIdx.x; i < kXRows * 32; i += kXThreads) {
    const int rr = i >> 5, quad = i & 31;  // row, dims 4 quad .. 4 quad + 3
    const int r = rb * kXRows + rr;
    float y[4] = {0.f, 0.f, 0.f, 0.f};
    if (r < a.rows) {
      const int j = r / g.group, head = h * g.group + r % g.group;
      const uint2 raw = *reinterpret_cast<const uint2*>(qh + (((size_t)b * a.T + j) * g.num_q_heads + head) * kHeadDim + 4 * quad);
      const float2 x01 = __half22float2(*reinterpret_cast<const __half2*>(&raw.x));
      const float2 x23 = __half22float2(*reinterpret_cast<const __half2*>(&raw.y));
      const float4 p = __ldg(reinterpret_cast<const float4*>(g.rot_k + (size_t)h * kHeadDim) + quad);
      if (g.mode == RQ_PLANAR) {
        y[0] = p.x * x01.x - p.y * x01.y;
        y[1] = p.y * x01.x + p.x * x01.y;
        y[2] = p.z * x23.x - p.w * x23.y;
        y[3] = p.w * x23.x + p.z * x23.y;
      } else {  // Hamilton product (a,b,c,d) (x) x
        y[0] = p.x * x01.x - p.y * x01.y - p.z * x23.x - p.w * x23.y;
        y[1] = p.y * x01.x + p.x * x01.y - p.w * x23.x + p.z * x23.y;
        y[2] = p.z * x01.x + p.w * x01.y + p.x * x23.x - p.y * x23.y;
        y[3] = p.w * x01.x - p.z * x01.y + p.y * x23.x + p.x * x23.y;
      }
    }
    const uint2 v = make_uint2(pack_h2(y[0] * g.q_scale, y[1] * g.q_scale), pack_h2(y[2] * g.q_scale, y[3] * g.q_scale));
    *reinterpret_cast<uint2*>(smem + kXSmemQ + xswz(rr, quad >> 1) + 8 * (quad & 1)) = v;
  }
  __syncthreads();
  uint32_t qa[8][4];  // A fragments of the warp's 16 rows, k-steps of 16 dims
#pragma unroll
  for (int ks = 0; ks < 8; ++ks)
    ldsm_x4(qa[ks], sbase + kXSmemQ + xswz(16 * warp + (lane & 15), 2 * ks + (lane >> 4)));

  // rows g and g + 8 of the warp: their last visible position (-1: none, or not a row)
  int qpos[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int r = rb * kXRows + 16 * warp + gq + 8 * i;
    qpos[i] = r < a.rows ? len - a.T + r / g.group : -1;
  }
  const int r_last = min(a.rows, (rb + 1) * kXRows) - 1;
  const int kv_end = min(len, len - a.T + r_last / g.group + 1);  // positions any row here sees

  float m_run[2] = {-CUDART_INF_F, -CUDART_INF_F};
  float l_run[2] = {0.f, 0.f};
  float o[16][4];
#pragma unroll
  for (int nd = 0; nd < 16; ++nd) o[nd][0] = o[nd][1] = o[nd][2] = o[nd][3] = 0.f;
  // thread t owns (token t / 4, 32-dim group t % 4) of every tile, for K and for V
  const int32_t* bt = a.block_table + (size_t)b * a.max_pages;
  const int my_tok = threadIdx.x >> 2, my_grp = threadIdx.x & 3;
  GroupRaw cur[2], nxt[2];
  load_group<BITS>(cur[0], g, a, bt, h, my_tok, len, 0, my_grp);
  load_group<BITS>(cur[1], g, a, bt, h, my_tok, len, 1, my_grp);

  for (int t0 = 0; t0 < kv_end; t0 += kXTok) {
    __syncthreads();  // the previous tile's K~, V~ are consumed
    // ---- dequantize this thread's two groups into the fp16 tiles ----
#pragma unroll
    for (int kind = 0; kind < 2; ++kind) {
      uint8_t* tile = smem + (kind ? kXSmemV : kXSmemK);
#pragma unroll
      for (int q = 0; q < 4; ++q) {  // 8 dims = one 16-byte chunk of the row
        uint32_t wv[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const __half lo = cb16[group_code<BITS>(cur[kind], 8 * q + 2 * e)];
          const __half hi = cb16[group_code<BITS>(cur[kind], 8 * q + 2 * e + 1)];
          wv[e] = (uint32_t)__half_as_ushort(lo) | ((uint32_t)__half_as_ushort(hi) << 16);
        }
        *reinterpret_cast<uint4*>(tile + xswz(my_tok, 4 * my_grp + q)) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
      }
      if (my_grp == 0) (kind ? nv : nk)[my_tok] = __half2float(__ushort_as_half((unsigned short)cur[kind].norm));
    }
    __syncthreads();
    // ---- the next tile's groups are in flight while this one is multiplied ----
    if (t0 + kXTok < kv_end) {
      load_group<BITS>(nxt[0], g, a, bt, h, t0 + kXTok + my_tok, len, 0, my_grp);
      load_group<BITS>(nxt[1], g, a, bt, h, t0 + kXTok + my_tok, len, 1, my_grp);
    }

    // ---- S = q~ K~^T for the warp's 16 rows x 32 tokens ----
    float s[4][4];
#pragma unroll
    for (int nn = 0; nn < 4; ++nn) s[nn][0] = s[nn][1] = s[nn][2] = s[nn][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
#pragma unroll
      for (int np = 0; np < 2; ++np) {
        uint32_t kb[4];  // b0, b1 of token n-tile 2np, then of 2np + 1
        ldsm_x4(kb, sbase + kXSmemK + xswz(8 * (2 * np + (lane >> 4)) + (lane & 7), 2 * ks + ((lane >> 3) & 1)));
        mma16816(s[2 * np], qa[ks], kb[0], kb[1]);
        mma16816(s[2 * np + 1], qa[ks], kb[2], kb[3]);
      }
    }
    // scale by the key norms, mask, online softmax (rows g: elements 0,1; g + 8: elements 2,3)
    float tmax[2] = {-CUDART_INF_F, -CUDART_INF_F};
#pragma unroll
    for (int nn = 0; nn < 4; ++nn) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int tok = 8 * nn + 2 * tq + (e & 1);
        float v = s[nn][e] * nk[tok];
        if (t0 + tok > qpos[e >> 1]) v = -CUDART_INF_F;
        s[nn][e] = v;
        tmax[e >> 1] = fmaxf(tmax[e >> 1], v);
      }
    }
    float alpha[2], m_use[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      tmax[i] = fmaxf(tmax[i], __shfl_xor_sync(0xffffffffu, tmax[i], 1));
      tmax[i] = fmaxf(tmax[i], __shfl_xor_sync(0xffffffffu, tmax[i], 2));
      const float m_new = fmaxf(m_run[i], tmax[i]);
      m_use[i] = m_new == -CUDART_INF_F ? 0.f : m_new;
      alpha[i] = ex2(m_run[i] - m_use[i]);
      m_run[i] = m_new;
      l_run[i] *= alpha[i];
    }
#pragma unroll
    for (int nd = 0; nd < 16; ++nd) {
      o[nd][0] *= alpha[0];
      o[nd][1] *= alpha[0];
      o[nd][2] *= alpha[1];
      o[nd][3] *= alpha[1];
    }
    uint32_t pa[2][4];  // P' = p * n_v as A fragments of two 16-token k-steps
#pragma unroll
    for (int nn = 0; nn < 4; ++nn) {
      float pv[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float p = ex2(s[nn][e] - m_use[e >> 1]);  // masked: +0
        l_run[e >> 1] += p;
        pv[e] = p * nv[8 * nn + 2 * tq + (e & 1)];
      }
      pa[nn >> 1][2 * (nn & 1)] = pack_h2(pv[0], pv[1]);      // row g
      pa[nn >> 1][2 * (nn & 1) + 1] = pack_h2(pv[2], pv[3]);  // row g + 8
    }
    // ---- O~ += P' V~ ----
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
#pragma unroll
      for (int nd = 0; nd < 16; nd += 2) {
        uint32_t vb[4];  // b0, b1 of dim n-tile nd, then of nd + 1
        ldsm_x4_t(vb, sbase + kXSmemV + xswz(16 * kk + 8 * ((lane >> 3) & 1) + (lane & 7), nd + (lane >> 4)));
        mma16816(o[nd], pa[kk], vb[0], vb[1]);
        mma16816(o[nd + 1], pa[kk], vb[2], vb[3]);
      }
    }
    cur[0] = nxt[0];
    cur[1] = nxt[1];
  }

  // ---- normalise, stage, rotate back, store ----
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    l_run[i] += __shfl_xor_sync(0xffffffffu, l_run[i], 1);
    l_run[i] += __shfl_xor_sync(0xffffffffu, l_run[i], 2);
  }
  const float inv0 = l_run[0] > 0.f ? 1.f / l_run[0] : 0.f, inv1 = l_run[1] > 0.f ? 1.f / l_run[1] : 0.f;
  __syncthreads();  // everyone is done with the query staging, which the output staging reuses
  float* os = reinterpret_cast<float*>(smem + kXSmemQ);
#pragma unroll
  for (int nd = 0; nd < 16; ++nd) {
    const int d = 8 * nd + 2 * tq;
    *reinterpret_cast<float2*>(os + (16 * warp + gq) * kXOStride + d) = make_float2(o[nd][0] * inv0, o[nd][1] * inv0);
    *reinterpret_cast<float2*>(os + (16 * warp + gq + 8) * kXOStride + d) = make_float2(o[nd][2] * inv1, o[nd][3] * inv1);
  }
  __syncthreads();
  __half* out = reinterpret_cast<__half*>(a.out);
  for (int i = threadIdx.x; i < kXRows * 32; i += kXThreads) {
    const int rr = i >> 5, quad = i & 31;
    const int r = rb * kXRows + rr;
    if (r >= a.rows) continue;
    const float4 yv = *reinterpret_cast<const float4*>(os + rr * kXOStride + 4 * quad);
    const float4 p = __ldg(reinterpret_cast<const float4*>(g.rot_v + (size_t)h * kHeadDim) + quad);
    float x[4];
    if (g.mode == RQ_PLANAR) {
      x[0] = p.x * yv.x + p.y * yv.y;
      x[1] = -p.y * yv.x + p.x * yv.y;
      x[2] = p.z * yv.z + p.w * yv.w;
      x[3] = -p.w * yv.z + p.z * yv.w;
    } else {  // L(q)^T y
      x[0] = p.x * yv.x + p.y * yv.y + p.z * yv.z + p.w * yv.w;
      x[1] = -p.y * yv.x + p.x * yv.y + p.w * yv.z - p.z * yv.w;
      x[2] = -p.z * yv.x - p.w * yv.y + p.x * yv.z + p.y * yv.w;
      x[3] = -p.w * yv.x + p.z * yv.y - p.y * yv.z + p.x * yv.w;
    }
    const int j = r / g.group, head = h * g.group + r % g.group;
    *reinterpret_cast<uint2*>(out + (((size_t)b * a.T + j) * g.num_q_heads + head) * kHeadDim + 4 * quad) =
        make_uint2(pack_h2(x[0], x[1]), pack_h2(x[2], x[3]));
  }
}

}  // namespace

cudaError_t extend_prepare() {
  cudaError_t e = cudaFuncSetAttribute(extend_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, kXSmem);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(extend_kernel<3>, cudaFuncAttributeMaxDynamicSharedMemorySize, kXSmem);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(extend_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, kXSmem);
  return e;
}

cudaError_t launch_extend(const Geometry& g, const AttnArgs& a, cudaStream_t stream, cudaEvent_t ev_start,
                          cudaEvent_t ev_end) {
  if (a.B <= 0) return cudaSuccess;
  if (g.mode == RQ_DENSE) return cudaErrorInvalidValue;
  const long long ctas = (long long)a.B * g.num_kv_heads * ((a.rows + kXRows - 1) / kXRows);
  if (ctas > 0x7fffffffLL) return cudaErrorInvalidValue;
  if (ev_start) cudaEventRecord(ev_start, stream);
  if (g.bits == 4)
    extend_kernel<4><<<(unsigned)ctas, kXThreads, kXSmem, stream>>>(g, a);
  else if (g.bits == 3)
    extend_kernel<3><<<(unsigned)ctas, kXThreads, kXSmem, stream>>>(g, a);
  else
    extend_kernel<2><<<(unsigned)ctas, kXThreads, kXSmem, stream>>>(g, a);
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess && ev_end) cudaEventRecord(ev_end, stream);
  return e;
}

}  // namespace rq
