// Extend (prefill) attention over the packed cache: T new query tokens per sequence, each
// attending causally to the cached prefix and to the new tokens up to itself ("SGLang 1-Bit
// Turbo" README, section "RotorQuant KV Cache Compression": queries are rotated once, values
// summed in the rotated space and the output rotated back once).  Query row j of sequence b
// sees positions 0 .. seq_lens[b] - T + j -- the definition of chain verify, here for T in the
// hundreds or thousands, where the split-K kernel (which re-reads the cache for every 8 query
// rows) stops paying.
//
// Design (sm_103a, 5th-generation tensor cores): one CTA per SM takes 256 query rows of one
// (sequence, kv head) -- rows r = j * group + k, in two blocks of 128 -- and walks the cache in
// 64-token tiles up to the last position its rows can see, with warps specialised by role and
// coupled only through mbarriers:
//   dequant (4 warps): per tile, K~ (token-major, centroid, with the key norms beside it) and
//     V~^T (dim-major, centroid times value norm), two stages each, as fp16 in the K-major
//     128-byte-swizzled operand layout; code bytes index a lane-replicated table of centroid
//     pairs (rq_lut.cuh), one shared load per two values; code words load ahead;
//   MMA (one thread): all operands of the row side live in tensor memory -- q~_b (A of S),
//     S_b and, over S_b's first 32 columns once the softmax has read it, P_b (A of PV~) -- and
//     the cache side comes from shared memory.  When block b's P(t) is ready it issues
//     O~_b += P_b V~(t) (M 128 x N 128 x K 64) and right behind it S_b(t + 1) = q~_b K~(t + 1)^T
//     (M 128 x N 64 x K 128): the tensor core runs one block's MMAs while the other block's
//     softmax runs, and S_b reuses its columns only after the PV~ that read them (one thread's
//     MMAs run in order);
//   softmax (8 warps, one thread per row, block b = warps 4b .. 4b + 3): reads its row of S
//     (tcgen05.ld), scales it by the key norms (f32), masks it, runs the online softmax in base
//     2 with no cross-thread reduction and writes p as fp16 over the row's S (tcgen05.st); the
//     running max moves only past a margin, so O~ is rarely rescaled (S(t) complete means the
//     PV~ before it is too); at the end it normalises, rotates back and stores its row.
// Every wait is bounded: one that runs out sets RQ_STATUS_TIMEOUT and an abort flag every role
// polls; the MMA thread drains what it issued before the tensor memory is freed.
#include <cuda_fp16.h>
#include <math_constants.h>

#include "rq_internal.h"
#include "rq_lut.cuh"
#include "rq_tc.cuh"
#include "../../include/rq.h"

namespace rq {
namespace {

constexpr int kXSoftWarps = 8;   // warps 0-7: softmax, thread i = row i of the CTA's 256
constexpr int kXDeqWarps = 4;    // warps 8-11: K~ dequantisation, warps 12-15: V~^T dequantisation
constexpr int kXThreads = 32 * (kXSoftWarps + 2 * kXDeqWarps + 1);  // + warp 16: MMA issue
constexpr int kXSoftThreads = 32 * kXSoftWarps, kXDeqThreads = 32 * kXDeqWarps;
constexpr int kXStages = 2;      // K~ and V~^T rings
constexpr int kXBlock = 128;    // rows per block: M of every MMA
constexpr int kXRows = 2 * kXBlock;
constexpr int kXTok = 64;       // tokens per K/V tile: N of S, K of PV~
// Shared memory: the 64 KB code table at the first 64 KB-aligned address of the window, the
// buffers (1024-aligned) below it where they fit, else above it.  The shared-memory MMA operands
// (K~, V~^T) are K-major with
// the 128-byte swizzle: 128-byte rows (64 fp16 of K), 16-byte chunk c of row r stored at chunk
// c ^ (r % 8), 8-row groups 1024 bytes apart, a second 64-wide K atom after all rows of the first.
constexpr uint32_t kXKBytes = 16384;   // K~: 64 tokens x 128 dims, two atoms of 8 KB
constexpr uint32_t kXVBytes = 16384;   // V~^T: 128 dims x 64 tokens
constexpr uint32_t kXMiscBytes = 1024; // centroids f32[16], the mbarriers, the tensor-memory
                                       // address, the abort flag; K norms f32[2][64] at 512
constexpr int kXSmem = 232448;         // the whole opt-in window (one CTA per SM)
constexpr uint32_t kXTmemCols = 512;   // O~_b at [128 b, 128 b + 128); q~_b (fp16 pairs) at
constexpr uint32_t kXColQ = 256;       //   256 + 64 b; S_b at 384 + 64 b, P_b (fp16 pairs) over
constexpr uint32_t kXColS = 384;       //   its first 32 columns
constexpr float kLazyMax = 8.f;        // running-max slack of the online softmax (log2 units)

struct XPlan {
  uint32_t lut, k[2], v[2], misc, end;  // shared addresses
};
__device__ __forceinline__ XPlan x_plan(uint32_t raw) {
  XPlan pl;
  pl.lut = (raw + 0xFFFFu) & ~0xFFFFu;
  uint32_t lo = (raw + 1023u) & ~1023u, hi = pl.lut + (uint32_t)lut::kBytes;
  auto place = [&](uint32_t bytes) {
    uint32_t at;
    if (lo + bytes <= pl.lut) {
      at = lo;
      lo += bytes;
    } else {
      at = hi;
      hi += bytes;
    }
    return at;
  };
  pl.k[0] = place(kXKBytes);
  pl.k[1] = place(kXKBytes);
  pl.v[0] = place(kXVBytes);
  pl.v[1] = place(kXVBytes);
  pl.misc = place(kXMiscBytes);
  pl.end = hi;
  return pl;
}

// mbarriers in the misc area (arrival counts in brackets)
constexpr uint32_t kBarKFull = 64;     // [2] K~ stage filled (128 dequant threads)
constexpr uint32_t kBarKEmpty = 80;    // [2] K~ stage read by S (MMA commit); its norms are read
                                       // once both blocks have released the tile's S (kBarSEmpty)
constexpr uint32_t kBarVFull = 224;    // [2] V~^T stage filled (128 dequant threads)
constexpr uint32_t kBarVEmpty = 240;   // [2] V~^T stage read by PV~ (MMA commit)
constexpr uint32_t kBarSFull = 96;     // [block] S ready (MMA commit)
constexpr uint32_t kBarSEmpty = 128;   // [block][stage] S and the stage's key norms read (128 softmax threads)
constexpr uint32_t kBarPFull = 160;    // [block] P written to tensor memory, O~ rescaled (128 softmax threads)
constexpr uint32_t kBarODone = 176;    // [block] PV~ done (MMA commit)
constexpr uint32_t kBarDrain = 192;    // everything the MMA thread issued is done
constexpr uint32_t kTmemSlot = 200, kAbortFlag = 204, kKNorms = 512;

using namespace tc;
__device__ __forceinline__ uint32_t xswz(int row, int chunk) { return sw128(row, chunk); }

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}
template <uint32_t LUT3>
__device__ __forceinline__ uint32_t lop3(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, %4;" : "=r"(d) : "r"(a), "r"(b), "r"(c), "n"(LUT3));
  return d;
}
// (a & c) | (b & ~c)
__device__ __forceinline__ uint32_t bitsel(uint32_t a, uint32_t b, uint32_t c) { return lop3<0xE4>(a, b, c); }

// One (token, 32-dim group) of a K or V vector as stored (include/rq.h): the code words and the
// token's fp16 norm, loaded from global memory ahead of use.
struct GroupRaw {
  uint32_t w[4];  // 4-bit: 4 words (8 codes each); 2-bit: 2 words (16 each); 3-bit: W0, W1, W2
  uint32_t norm;  // the token's fp16 norm (bits), 0 past the sequence
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
  r.norm = __ldg(reinterpret_cast<const uint16_t*>(chunk + (size_t)2 * P * vb + kind * 2 * P + 2 * off));
}

// ---- K~ rows: one token's 32-dim group -> four 16-byte chunks of 8 fp16 ----
// Chunk q holds dims 8q .. 8q + 7 of the group, as the half2 of dim pairs.  4-bit: byte j of
// word q is the pair (8q + 2j, 8q + 2j + 1).  3-bit: X0 = W0.lo | W2.hi and X1 = W2.lo | W0.hi
// give pairs 2k (T1) and 2k + 1 (T2) from byte k, X2 = W1.lo | (W2 >> 2).hi and X3 =
// (W2 >> 2).lo | W1.hi pairs 8 + 2k and 9 + 2k.  2-bit: byte j of word q >> 1 carries dims
// 4j' .. 4j' + 3; U1 gives (4j', 4j' + 2) and U2 (4j' + 1, 4j' + 3), so within every 4-dim
// block the stored order is 0, 2, 1, 3 -- and q~ is stored in the same order.
template <int BITS>
__device__ __forceinline__ void k_chunks(uint4 (&ch)[4], const GroupRaw& r, uint32_t key1, uint32_t key2) {
  if constexpr (BITS == 4) {
#pragma unroll
    for (int q = 0; q < 4; ++q)
      ch[q] = make_uint4(lut::get(r.w[q], 0, key1), lut::get(r.w[q], 1, key1), lut::get(r.w[q], 2, key1),
                         lut::get(r.w[q], 3, key1));
  } else if constexpr (BITS == 2) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t w = r.w[q >> 1];
      const int j0 = 2 * (q & 1);
      lut::get2(w, j0, key1, ch[q].x, ch[q].y);  // (U1, U2) of one index byte: one 8-byte load
      lut::get2(w, j0 + 1, key1, ch[q].z, ch[q].w);
    }
  } else {
    const uint32_t w2s = r.w[2] >> 2;
    const uint32_t X0 = bitsel(r.w[0], r.w[2], 0x0F0F0F0Fu), X1 = bitsel(r.w[2], r.w[0], 0x0F0F0F0Fu);
    const uint32_t X2 = bitsel(r.w[1], w2s, 0x0F0F0F0Fu), X3 = bitsel(w2s, r.w[1], 0x0F0F0F0Fu);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t xe = q < 2 ? X0 : X2, xo = q < 2 ? X1 : X3;
      const int j0 = 2 * (q & 1);
      ch[q] = make_uint4(lut::get(xe, j0, key1), lut::get(xo, j0, key2), lut::get(xe, j0 + 1, key1),
                         lut::get(xo, j0 + 1, key2));
    }
  }
}

// ---- V~^T rows: 16 dims (half hh of a 32-dim group) of a token pair (A, B) -> 16 half2 ----
// out[i] = (c[A's code of dim 16 hh + i], c[B's]).  Index bytes interleave the two tokens' codes
// of one dim.  4-bit: XE = A | B << 4 per nibble pair gives dims 2k (T4), XO dims 2k + 1.
// 2-bit: XE byte k gives dims 4k (U1) and 4k + 1 (U2), XO dims 4k + 2, 4k + 3.  3-bit: with E / O
// the two tokens' low bits of even / odd dims and M / M2 their high bits, XE1 (T1), XO1 (T1), XE2
// (T2), XO2 (T2) byte k give dims 4k, 4k + 1, 4k + 2, 4k + 3.
template <int BITS>
__device__ __forceinline__ void v_pairs(uint32_t (&out)[16], const GroupRaw& A, const GroupRaw& B, int hh,
                                        uint32_t key1, uint32_t key2) {
  if constexpr (BITS == 4) {
#pragma unroll
    for (int u = 0; u < 2; ++u) {  // (selects, not a runtime index: the words stay in registers)
      const uint32_t a = hh ? A.w[2 + u] : A.w[u], b = hh ? B.w[2 + u] : B.w[u];
      const uint32_t XE = bitsel(a, b << 4, 0x0F0F0F0Fu), XO = bitsel(a >> 4, b, 0x0F0F0F0Fu);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        out[8 * u + 2 * k] = lut::get(XE, k, key1);
        out[8 * u + 2 * k + 1] = lut::get(XO, k, key1);
      }
    }
  } else if constexpr (BITS == 2) {
    const uint32_t a = hh ? A.w[1] : A.w[0], b = hh ? B.w[1] : B.w[0];
    const uint32_t XE = bitsel(a, b << 4, 0x0F0F0F0Fu), XO = bitsel(a >> 4, b, 0x0F0F0F0Fu);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      lut::get2(XE, k, key1, out[4 * k], out[4 * k + 1]);
      lut::get2(XO, k, key1, out[4 * k + 2], out[4 * k + 3]);
    }
  } else {
    const int sh = 2 * hh;
    const uint32_t a = hh ? A.w[1] : A.w[0], b = hh ? B.w[1] : B.w[0], a2 = A.w[2], b2 = B.w[2];
    const uint32_t E = bitsel(a, b << 2, 0x33333333u), O = bitsel(a >> 2, b, 0x33333333u);
    const uint32_t M = bitsel(a2, b2 << 1, 0x55555555u) >> sh, M2 = bitsel(a2 >> 1, b2, 0x55555555u) >> sh;
    const uint32_t XE1 = bitsel(E, M, 0x0F0F0F0Fu), XE2 = bitsel(M, E, 0x0F0F0F0Fu);
    const uint32_t XO1 = bitsel(O, M2, 0x0F0F0F0Fu), XO2 = bitsel(M2, O, 0x0F0F0F0Fu);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      out[4 * k] = lut::get(XE1, k, key1);
      out[4 * k + 1] = lut::get(XO1, k, key1);
      out[4 * k + 2] = lut::get(XE2, k, key2);
      out[4 * k + 3] = lut::get(XO2, k, key2);
    }
  }
}

// DENSE: a dense rotation (TurboQuant): the queries come pre-rotated in a.q_rot (fp32), and the
// output rotation R_v^T is a 128 x 128 matrix-vector product per row, done once every role is
// finished with R_v staged in the code table's 64 KB.
template <int BITS, bool DENSE>
__global__ void __launch_bounds__(kXThreads, 1)
extend_kernel(const Geometry g, const AttnArgs a, int smem_bytes) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = (uint32_t)__cvta_generic_to_shared(smem_raw);
  const XPlan pl = x_plan(raw);
  if (pl.end - raw > (uint32_t)smem_bytes) {  // unexpected reserved shared memory
    if (threadIdx.x == 0 && a.status) atomicOr(a.status, RQ_STATUS_TIMEOUT);
    return;
  }
  auto at = [&](uint32_t addr) { return smem_raw + (addr - raw); };
  float* const cb = reinterpret_cast<float*>(at(pl.misc));
  float* const knorm = reinterpret_cast<float*>(at(pl.misc + kKNorms));  // [stage][64]
  volatile int* const abort_flag = reinterpret_cast<volatile int*>(at(pl.misc + kAbortFlag));
  const uint32_t mb = pl.misc;  // barrier base
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_rb = (a.rows + kXRows - 1) / kXRows;
  const int rb = n_rb - 1 - (int)(blockIdx.x % n_rb);  // latest rows (longest reach) first
  const int h = (blockIdx.x / n_rb) % g.num_kv_heads;
  const int b = blockIdx.x / (n_rb * g.num_kv_heads);
  const int cap = a.max_pages * g.page_size;
  int len = a.seq_lens[b];
  if (len < 0 || len > cap || (len > 0 && len < a.T)) {
    if (rb == n_rb - 1 && h == 0 && tid == 0 && a.status) atomicOr(a.status, RQ_STATUS_BAD_LEN);
    len = len < 0 ? 0 : (len > cap ? cap : len);
  }
  if (tid < (1 << BITS)) cb[tid] = g.centroids[tid];
  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(mb + kBarKFull + 8 * i, kXDeqThreads);
      mbar_init(mb + kBarKEmpty + 8 * i, 1);
      mbar_init(mb + kBarPFull + 8 * i, kXBlock);
      mbar_init(mb + kBarODone + 8 * i, 1);
      mbar_init(mb + kBarSFull + 8 * i, 1);
      for (int j = 0; j < 2; ++j) mbar_init(mb + kBarSEmpty + 16 * i + 8 * j, kXBlock);
    }
    mbar_init(mb + kBarDrain, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(mb + kBarVFull + 8 * i, kXDeqThreads);
      mbar_init(mb + kBarVEmpty + 8 * i, 1);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncwarp();  // tcgen05.alloc is warp-collective
  if (warp == 0) {
    tmem_alloc(mb + kTmemSlot, kXTmemCols);
  }

  // row r sees positions <= qpos (-1: nothing, or not a row); the CTA's rows see < kv_end
  const int r_last = min(a.rows, (rb + 1) * kXRows) - 1;
  const int kv_end = min(len, len - a.T + r_last / g.group + 1);
  const int n_tiles = kv_end > 0 ? (kv_end + kXTok - 1) / kXTok : 0;
  const int32_t* bt = a.block_table + (size_t)b * a.max_pages;
  const int blk = (warp >> 2) & 1;                    // softmax: row block
  const int brow = 32 * (warp & 3) + lane;            // softmax: row within the block (= lane of tensor memory)
  const int r = rb * kXRows + kXBlock * blk + brow;   // softmax: query row

  __syncthreads();  // the centroids are staged, the barriers initialised
  lut::fill<BITS>(reinterpret_cast<uint32_t*>(at(pl.lut)), cb, tid, kXThreads);
  const uint32_t key1 = lut::key<BITS>(pl.lut, lane, 0), key2 = lut::key<BITS>(pl.lut, lane, 1);
  fence_async_smem();
  fence_before_sync();
  __syncthreads();  // the code table and the tensor-memory address are in place
  fence_after_sync();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(at(mb + kTmemSlot));

  // ---- q~ = R_k q * sm_scale * log2(e) of row r, fp16 pairs, into the A operand of its block
  // (tensor memory: the thread's lane, columns kXColQ + 64 blk + k / 2 for the operand's K order) ----
  if (warp < kXSoftWarps) {
    const bool valid = r < a.rows;
    const int j = valid ? r / g.group : 0, head = h * g.group + (valid ? r % g.group : 0);
    const uint4* qrow = reinterpret_cast<const uint4*>(reinterpret_cast<const __half*>(a.q) +
                                                       (((size_t)b * a.T + j) * g.num_q_heads + head) * kHeadDim);
    const float4* rk = reinterpret_cast<const float4*>(g.rot_k + (size_t)h * kHeadDim);
    const float4* qrot = DENSE ? reinterpret_cast<const float4*>(a.q_rot + (((size_t)b * a.T + j) * g.num_q_heads + head) *
                                                                              kHeadDim)
                               : nullptr;
    const uint32_t q_cols = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + kXColQ + 64 * blk;
#pragma unroll 1
    for (int cc = 0; cc < 4; ++cc) {  // dims 32 cc .. 32 cc + 31: 16 columns
      uint32_t qw[16];
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {  // dims 8c .. 8c + 7: two rotation blocks of 4
        const int c = 4 * cc + c4;
        uint32_t w[4] = {0u, 0u, 0u, 0u};
        if (DENSE && valid) {  // R_k q, formed before the launch
#pragma unroll
          for (int bk = 0; bk < 2; ++bk) {
            const float4 yv = __ldg(qrot + 2 * c + bk);
            const float y[4] = {yv.x, yv.y, yv.z, yv.w};
            const int s1 = BITS == 2 ? 2 : 1, s2 = BITS == 2 ? 1 : 2;  // the K~ order of a 4-dim block
            w[2 * bk] = pack_h2(y[0] * g.q_scale, y[s1] * g.q_scale);
            w[2 * bk + 1] = pack_h2(y[s2] * g.q_scale, y[3] * g.q_scale);
          }
        } else if (valid) {
          const uint4 raw8 = __ldg(qrow + c);
          const uint32_t hw[4] = {raw8.x, raw8.y, raw8.z, raw8.w};
#pragma unroll
          for (int bk = 0; bk < 2; ++bk) {
            const float2 x01 = __half22float2(*reinterpret_cast<const __half2*>(&hw[2 * bk]));
            const float2 x23 = __half22float2(*reinterpret_cast<const __half2*>(&hw[2 * bk + 1]));
            const float4 p = __ldg(rk + 2 * c + bk);
            float y[4];
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
            const int s1 = BITS == 2 ? 2 : 1, s2 = BITS == 2 ? 1 : 2;  // the K~ order of a 4-dim block
            w[2 * bk] = pack_h2(y[0] * g.q_scale, y[s1] * g.q_scale);
            w[2 * bk + 1] = pack_h2(y[s2] * g.q_scale, y[3] * g.q_scale);
          }
        }
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) qw[4 * c4 + jj] = w[jj];
      }
      tmem_st16u(q_cols + 16 * cc, qw);
    }
    tmem_wait_st();
  }
  fence_before_sync();
  __syncthreads();  // q~ is in tensor memory
  fence_after_sync();

  float soft_inv = 0.f;   // dense: the row's 1 / l, for the epilogue after every role is done
  bool soft_ok = false;
  if (warp < kXSoftWarps) {
    // ================= softmax: one thread per row of block blk =================
    const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
    const uint32_t tmem_o = tmem + lane_off + 128 * blk;
    const int qpos = r < a.rows ? len - a.T + r / g.group : -1;
    float m_run = -CUDART_INF_F, l_run = 0.f;
    bool ok = true;
    for (int t = 0; t < n_tiles && ok; ++t) {
      const int t0 = t * kXTok, i = t & 1;
      // S_b(t) complete: so is every MMA issued before it, PV~_b(t - 1) included
      ok = __all_sync(0xffffffffu, role_wait(mb + kBarSFull + 8 * blk, (uint32_t)(t & 1), abort_flag));
      if (!ok) break;
      fence_after_sync();
      const uint32_t s_cols = tmem + lane_off + kXColS + 64 * blk;
      float s[kXTok];
#pragma unroll
      for (int c = 0; c < kXTok / 16; ++c) {
        float v[16];
        tmem_ld16(s_cols + 16 * c, v);
#pragma unroll
        for (int k = 0; k < 16; ++k) s[16 * c + k] = v[k];
      }
      tmem_wait_ld();
      // t = s * n_k - m_use (base 2, one FMA a key), m_use the running max (0 before the first)
      const float m_use0 = m_run == -CUDART_INF_F ? 0.f : m_run;
      {  // key norms of the tile (stage t % 2)
        const float4* n4 = reinterpret_cast<const float4*>(knorm + 64 * (t % kXStages));
#pragma unroll
        for (int c = 0; c < kXTok / 4; ++c) {
          const float4 nn = n4[c];
          s[4 * c] = fmaf(s[4 * c], nn.x, -m_use0);
          s[4 * c + 1] = fmaf(s[4 * c + 1], nn.y, -m_use0);
          s[4 * c + 2] = fmaf(s[4 * c + 2], nn.z, -m_use0);
          s[4 * c + 3] = fmaf(s[4 * c + 3], nn.w, -m_use0);
        }
      }
      fence_before_sync();
      mbar_arrive(mb + kBarSEmpty + 16 * blk + 8 * i);  // the tile's key norms may be reused
      if (!(t0 + kXTok - 1 <= qpos)) {  // mask what the row may not see
#pragma unroll
        for (int jj = 0; jj < kXTok; ++jj)
          if (t0 + jj > qpos) s[jj] = -CUDART_INF_F;
      }
      float tm[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) tm[k] = s[k];
#pragma unroll
      for (int jj = 8; jj < kXTok; ++jj) tm[jj & 7] = fmaxf(tm[jj & 7], s[jj]);
      const float tmax = fmaxf(fmaxf(fmaxf(tm[0], tm[1]), fmaxf(tm[2], tm[3])), fmaxf(fmaxf(tm[4], tm[5]), fmaxf(tm[6], tm[7])));
      // The running max moves only when the tile's max passes it by more than kLazyMax (log2
      // units): p = 2^t then stays <= 2^kLazyMax, exact in fp16 and f32, and O~ is rescaled
      // rarely instead of on most tiles.  Before the first visible key any visible t moves it.
      float alpha = 1.f;
      if (tmax > (m_run == -CUDART_INF_F ? -CUDART_INF_F : kLazyMax)) {
        const float m_new = tmax + m_use0;
        alpha = ex2(m_run - m_new);  // 0 while nothing was seen yet
        m_run = m_new;
        const float shift = m_use0 - m_new;
#pragma unroll
        for (int jj = 0; jj < kXTok; ++jj) s[jj] += shift;
      }
      float ls[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) ls[k] = 0.f;
#pragma unroll
      for (int jj = 0; jj < kXTok; ++jj) {
        const float pr = ex2(s[jj]);  // masked: +0
        ls[jj & 7] += pr;
        s[jj] = pr;
      }
      l_run = l_run * alpha + (((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7])));
      // P_b(t) as fp16 pairs over the first 32 columns of S_b (already read)
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t pw[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) pw[k] = pack_h2(s[32 * c + 2 * k], s[32 * c + 2 * k + 1]);
        tmem_st16u(s_cols + 16 * c, pw);
      }
      if (t > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {  // O~ *= alpha (the warp's rows)
#pragma unroll 1
        for (int c = 0; c < kHeadDim / 16; ++c) {
          float v[16];
          tmem_ld16(tmem_o + 16 * c, v);
          tmem_wait_ld();
#pragma unroll
          for (int k = 0; k < 16; ++k) v[k] *= alpha;
          tmem_st16(tmem_o + 16 * c, v);
        }
      }
      tmem_wait_st();
      fence_before_sync();
      mbar_arrive(mb + kBarPFull + 8 * blk);
    }
    // ---- normalise, rotate back, store ----
    if (ok && n_tiles > 0) {
      ok = __all_sync(0xffffffffu, role_wait(mb + kBarODone + 8 * blk, (uint32_t)((n_tiles - 1) & 1), abort_flag));
      if (ok) fence_after_sync();
    }
    if (DENSE) {
      soft_ok = ok;
      soft_inv = l_run > 0.f ? g.out_scale / l_run : 0.f;
    } else if (ok) {
      const bool store = r < a.rows;
      const float inv = l_run > 0.f ? g.out_scale / l_run : 0.f;
      const int j = store ? r / g.group : 0, head = h * g.group + (store ? r % g.group : 0);
      uint4* orow = reinterpret_cast<uint4*>(reinterpret_cast<__half*>(a.out) +
                                             (((size_t)b * a.T + j) * g.num_q_heads + head) * kHeadDim);
      const float4* rv = reinterpret_cast<const float4*>(g.rot_v + (size_t)h * kHeadDim);
#pragma unroll 1
      for (int c = 0; c < kHeadDim / 16; ++c) {  // dims 16c .. 16c + 15
        float y[16];
        __syncwarp();       // the previous stores diverged by row
        if (n_tiles > 0) {  // uniform over the CTA
          tmem_ld16(tmem_o + 16 * c, y);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int k = 0; k < 16; ++k) y[k] = 0.f;
        }
        if (store) {
          uint32_t w[8];
#pragma unroll
          for (int bk = 0; bk < 4; ++bk) {
            const float4 p = __ldg(rv + 4 * c + bk);
            const float y0 = y[4 * bk] * inv, y1 = y[4 * bk + 1] * inv, y2 = y[4 * bk + 2] * inv, y3 = y[4 * bk + 3] * inv;
            float x[4];
            if (g.mode == RQ_PLANAR) {
              x[0] = p.x * y0 + p.y * y1;
              x[1] = -p.y * y0 + p.x * y1;
              x[2] = p.z * y2 + p.w * y3;
              x[3] = -p.w * y2 + p.z * y3;
            } else {  // L(q)^T y
              x[0] = p.x * y0 + p.y * y1 + p.z * y2 + p.w * y3;
              x[1] = -p.y * y0 + p.x * y1 + p.w * y2 - p.z * y3;
              x[2] = -p.z * y0 - p.w * y1 + p.x * y2 + p.y * y3;
              x[3] = -p.w * y0 + p.z * y1 - p.y * y2 + p.x * y3;
            }
            w[2 * bk] = pack_h2(x[0], x[1]);
            w[2 * bk + 1] = pack_h2(x[2], x[3]);
          }
          orow[2 * c] = make_uint4(w[0], w[1], w[2], w[3]);
          orow[2 * c + 1] = make_uint4(w[4], w[5], w[6], w[7]);
        }
      }
    }
    if (!ok && lane == 0 && a.status) atomicOr(a.status, RQ_STATUS_TIMEOUT);
  } else if (warp < kXSoftWarps + 2 * kXDeqWarps) {
    // ================= dequantisation: K~ (warps 8-11) and V~^T (warps 12-15) =================
    // K~: thread (token dt % 64, code groups dt / 64 and dt / 64 + 2) -> 4 chunks of a row each;
    // a stage is free once S(t - 2) is done.  V~^T: warp dw takes dims 32 dw .. 32 dw + 31 (code
    // group dw), lane p the token pair (2p, 2p + 1), one half2 per dim row -- a warp writes 128
    // consecutive bytes a row; a stage is free once PV~(t - 2) is done.  The two run
    // independently, each loading its next tile's code words while it works on this one.
    const bool k_role = warp < kXSoftWarps + kXDeqWarps;
    const int dt = tid - kXSoftThreads - (k_role ? 0 : kXDeqThreads), dw = dt >> 5;
    const int ktok = dt & 63, kg0 = dt >> 6;
    GroupRaw k0, k1, va, vb;
    auto load_k = [&](int t0) {
      load_group<BITS>(k0, g, a, bt, h, t0 + ktok, len, 0, kg0);
      load_group<BITS>(k1, g, a, bt, h, t0 + ktok, len, 0, kg0 + 2);
    };
    auto load_v = [&](int t0) {
      load_group<BITS>(va, g, a, bt, h, t0 + 2 * lane, len, 1, dw);
      load_group<BITS>(vb, g, a, bt, h, t0 + 2 * lane + 1, len, 1, dw);
    };
    auto produce_k = [&](int t) -> bool {  // K~(t) (centroids) into stage t % 2, its norms beside it
      const int st = t % kXStages;
      if (t >= kXStages) {  // S(t - 2) done, and both blocks have read its S and norms
        const uint32_t par = (uint32_t)((t / kXStages - 1) & 1);
        bool w = role_wait(mb + kBarKEmpty + 8 * st, par, abort_flag);
        w = w && role_wait(mb + kBarSEmpty + 8 * st, par, abort_flag);
        w = w && role_wait(mb + kBarSEmpty + 16 + 8 * st, par, abort_flag);
        if (!__all_sync(0xffffffffu, w)) return false;
      }
#pragma unroll
      for (int gi = 0; gi < 2; ++gi) {
        const int grp = kg0 + 2 * gi;
        uint4 ch[4];
        k_chunks<BITS>(ch, gi ? k1 : k0, key1, key2);
        uint8_t* const atom = at(st ? pl.k[1] : pl.k[0]) + (grp >> 1) * 8192;
#pragma unroll
        for (int q = 0; q < 4; ++q) *reinterpret_cast<uint4*>(atom + xswz(ktok, 4 * (grp & 1) + q)) = ch[q];
      }
      if (dt < 64) knorm[64 * st + ktok] = __half2float(__ushort_as_half((unsigned short)k0.norm));
      if (t + 1 < n_tiles) load_k((t + 1) * kXTok);
      fence_async_smem();
      mbar_arrive(mb + kBarKFull + 8 * st);
      return true;
    };
    auto produce_v = [&](int t) -> bool {  // V~(t)^T = n_v * centroid into stage t % 2
      const int st = t % kXStages;
      if (t >= kXStages &&  // PV~(t - 2) has read the stage
          !__all_sync(0xffffffffu, role_wait(mb + kBarVEmpty + 8 * st, (uint32_t)((t / kXStages - 1) & 1), abort_flag)))
        return false;
      const uint32_t nbits = (va.norm & 0xFFFFu) | (vb.norm << 16);
      const __half2 n2 = *reinterpret_cast<const __half2*>(&nbits);
      uint8_t* const vt = at(st ? pl.v[1] : pl.v[0]);
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        uint32_t pv[16];
        v_pairs<BITS>(pv, va, vb, hh, key1, key2);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int row = 32 * dw + 16 * hh + i;
          const __half2 x = __hmul2(*reinterpret_cast<const __half2*>(&pv[i]), n2);
          *reinterpret_cast<__half2*>(vt + row * 128 + (((lane >> 2) ^ (row & 7)) << 4) + 4 * (lane & 3)) = x;
        }
      }
      if (t + 1 < n_tiles) load_v((t + 1) * kXTok);
      fence_async_smem();
      mbar_arrive(mb + kBarVFull + 8 * st);
      return true;
    };
    bool ok = true;
    if (k_role) {
      if (n_tiles > 0) load_k(0);
      for (int t = 0; t < n_tiles && ok; ++t) ok = produce_k(t);
    } else {
      if (n_tiles > 0) load_v(0);
      for (int t = 0; t < n_tiles && ok; ++t) ok = produce_v(t);
    }
    if (!ok && lane == 0 && a.status) atomicOr(a.status, RQ_STATUS_TIMEOUT);
  } else if (lane == 0) {
    // ================= MMA issue (one thread) =================
    const uint32_t id_s = idesc_f16(kXBlock, kXTok), id_o = idesc_f16(kXBlock, kHeadDim);
    bool ok = true;
    int issued = 0;
    // S_b(t) = q~_b K~(t)^T: A from tensor memory (q~_b), B the K~ stage at kb; into S_b's columns
    auto s_mmas = [&](int bb, uint32_t kb) {
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        umma_f16_ts(tmem + kXColS + 64 * bb, tmem + kXColQ + 64 * bb + 8 * ks,
                    sdesc(kb + (ks >> 2) * 8192 + (ks & 3) * 32), id_s, ks > 0);
      umma_commit(mb + kBarSFull + 8 * bb);
      ++issued;
    };
    auto wait_k = [&](int t) {
      return role_wait(mb + kBarKFull + 8 * (t % kXStages), (uint32_t)((t / kXStages) & 1), abort_flag);
    };
    if (n_tiles > 0 && (ok = wait_k(0))) {
      fence_after_sync();
      s_mmas(0, pl.k[0]);
      s_mmas(1, pl.k[0]);
      umma_commit(mb + kBarKEmpty);  // stage 0's K~ has been read
    }
    for (int t = 0; t < n_tiles && ok; ++t) {
      const int vs = t % kXStages, ks1 = (t + 1) % kXStages;
      const bool next = t + 1 < n_tiles;
      if (!(ok = role_wait(mb + kBarVFull + 8 * vs, (uint32_t)((t / kXStages) & 1), abort_flag))) break;
      if (next && !(ok = wait_k(t + 1))) break;
      const uint32_t vb = vs ? pl.v[1] : pl.v[0], kb = ks1 ? pl.k[1] : pl.k[0];
#pragma unroll 1
      for (int bb = 0; bb < 2; ++bb) {
        if (!(ok = role_wait(mb + kBarPFull + 8 * bb, (uint32_t)(t & 1), abort_flag))) break;
        fence_after_sync();
        // O~_b += P_b(t) V~(t), P_b from the first 32 columns of S_b
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          umma_f16_ts(tmem + 128 * bb, tmem + kXColS + 64 * bb + 8 * ks, sdesc(vb + ks * 32), id_o, t > 0 || ks > 0);
        umma_commit(mb + kBarODone + 8 * bb);
        ++issued;
        if (next) s_mmas(bb, kb);  // S_b(t + 1) over the same columns, behind the PV~ that reads them
      }
      if (!ok) break;
      umma_commit(mb + kBarVEmpty + 8 * vs);                 // the V~^T stage has been read
      if (next) umma_commit(mb + kBarKEmpty + 8 * ks1);      // and the next tile's K~ stage
    }
    if (issued > 0) {  // drain: nothing may be running when the tensor memory is freed
      umma_commit(mb + kBarDrain);
      for (int i = 0; i < kWaitLimit; ++i)
        if (mbar_test(mb + kBarDrain, 0u)) break;
    }
    if (!ok && a.status) atomicOr(a.status, RQ_STATUS_TIMEOUT);
  }
  if constexpr (DENSE) {
    // ---- normalise, rotate back (out = R_v^T o~, a full matrix), store ----
    fence_before_sync();
    __syncthreads();  // every role is done: the code table is free and O~ is final
    fence_after_sync();
    float4* const rvs = reinterpret_cast<float4*>(at(pl.lut));  // R_v row-major: [m][i / 4]
    const float4* rsrc = reinterpret_cast<const float4*>(g.rot_v + (size_t)h * kHeadDim * kHeadDim);
    for (int c = tid; c < kHeadDim * kHeadDim / 4; c += kXThreads) rvs[c] = __ldg(rsrc + c);
    __syncthreads();
    if (warp < kXSoftWarps && soft_ok) {  // soft_ok is uniform over each warp
      const uint32_t tmem_o = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + 128 * blk;
      const bool store = r < a.rows;
      const int j = store ? r / g.group : 0, head = h * g.group + (store ? r % g.group : 0);
      uint4* orow = reinterpret_cast<uint4*>(reinterpret_cast<__half*>(a.out) +
                                             (((size_t)b * a.T + j) * g.num_q_heads + head) * kHeadDim);
#pragma unroll 1
      for (int ic = 0; ic < kHeadDim / 32; ++ic) {  // outputs 32 ic .. 32 ic + 31
        float acc[32];
#pragma unroll
        for (int k = 0; k < 32; ++k) acc[k] = 0.f;
#pragma unroll 1
        for (int mc = 0; mc < kHeadDim / 16; ++mc) {  // o~ dims 16 mc .. 16 mc + 15
          float v[16];
          if (n_tiles > 0) {  // uniform over the CTA
            tmem_ld16(tmem_o + 16 * mc, v);
            tmem_wait_ld();
          } else {
#pragma unroll
            for (int k = 0; k < 16; ++k) v[k] = 0.f;
          }
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const float om = v[k] * soft_inv;
            const float4* wrow = rvs + (16 * mc + k) * (kHeadDim / 4) + 8 * ic;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const float4 w = wrow[q];
              acc[4 * q] = fmaf(w.x, om, acc[4 * q]);
              acc[4 * q + 1] = fmaf(w.y, om, acc[4 * q + 1]);
              acc[4 * q + 2] = fmaf(w.z, om, acc[4 * q + 2]);
              acc[4 * q + 3] = fmaf(w.w, om, acc[4 * q + 3]);
            }
          }
        }
        if (store) {
#pragma unroll
          for (int q = 0; q < 4; ++q)
            orow[4 * ic + q] = make_uint4(pack_h2(acc[8 * q], acc[8 * q + 1]), pack_h2(acc[8 * q + 2], acc[8 * q + 3]),
                                          pack_h2(acc[8 * q + 4], acc[8 * q + 5]), pack_h2(acc[8 * q + 6], acc[8 * q + 7]));
        }
      }
    }
  }
  fence_before_sync();
  __syncthreads();
  if (warp == 0)
    tmem_dealloc(tmem, kXTmemCols);
}

}  // namespace

template <bool DENSE>
static cudaError_t extend_prepare_flag() {
  cudaError_t e = cudaFuncSetAttribute(extend_kernel<2, DENSE>, cudaFuncAttributeMaxDynamicSharedMemorySize, kXSmem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(extend_kernel<3, DENSE>, cudaFuncAttributeMaxDynamicSharedMemorySize, kXSmem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(extend_kernel<4, DENSE>, cudaFuncAttributeMaxDynamicSharedMemorySize, kXSmem);
  return e;
}

cudaError_t extend_prepare() {
  cudaError_t e = extend_prepare_flag<false>();
  if (e == cudaSuccess) e = extend_prepare_flag<true>();
  return e;
}

template <bool DENSE>
static void launch_extend_flag(const Geometry& g, const AttnArgs& a, unsigned ctas, cudaStream_t stream) {
  if (g.bits == 4)
    extend_kernel<4, DENSE><<<ctas, kXThreads, kXSmem, stream>>>(g, a, kXSmem);
  else if (g.bits == 3)
    extend_kernel<3, DENSE><<<ctas, kXThreads, kXSmem, stream>>>(g, a, kXSmem);
  else
    extend_kernel<2, DENSE><<<ctas, kXThreads, kXSmem, stream>>>(g, a, kXSmem);
}

cudaError_t launch_extend(const Geometry& g, const AttnArgs& a, cudaStream_t stream, cudaEvent_t ev_start,
                          cudaEvent_t ev_end) {
  if (a.B <= 0) return cudaSuccess;
  const bool dense = g.mode == RQ_DENSE;
  if (dense != (a.q_rot != nullptr)) return cudaErrorInvalidValue;
  const long long ctas = (long long)a.B * g.num_kv_heads * ((a.rows + kXRows - 1) / kXRows);
  if (ctas > 0x7fffffffLL) return cudaErrorInvalidValue;
  if (dense) {  // R_k q of every row first
    cudaError_t e = launch_dense_rotate_q(g, a, stream);
    if (e != cudaSuccess) return e;
  }
  if (ev_start) cudaEventRecord(ev_start, stream);
  if (dense)
    launch_extend_flag<true>(g, a, (unsigned)ctas, stream);
  else
    launch_extend_flag<false>(g, a, (unsigned)ctas, stream);
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess && ev_end) cudaEventRecord(ev_end, stream);
  return e;
}

}  // namespace rq
