// GQA decode / chain-verify attention that reads the packed cache directly, and the
// log-sum-exp combine that merges the split-K partials and rotates the output back.
//
// Method ("SGLang 1-Bit Turbo" README, section "RotorQuant KV Cache Compression"): keys and
// values are stored as norm * R^T c[code] with an orthogonal structured R.  Hence
//   <q, k>  = n_k * <R_k q, c[code_k]>          (rotate q once, never un-rotate a key)
//   sum p v = R_v^T sum p n_v c[code_v]          (sum in rotated space, rotate back once)
//
// Kernel design (sm_103a):
//   * One CTA of 16 warps per SM, stream-K partition: the work of all units (sequence, kv head,
//     query n-tile), in that order, counted in rounds -- 32 consecutive 16-token tiles, one
//     pair of tiles per warp -- plus a fixed cost per unit for opening a fragment on it, is cut
//     into gridDim.x equal contiguous ranges, so every SM gets about the same work whatever the
//     lengths.  The part of a unit that falls in one CTA's range is a fragment: the CTA stages
//     its page ids in shared memory, the warps take its tiles two at a time round-robin, and
//     their (m, l, O) are merged through shared memory into one partial per fragment.
//   * Per 16-token tile both contractions run on the tensor cores with mma.sync m16n8k16
//     (fp16 in, fp32 accumulate): S^T[16 tok x 8 q] = K~[16 x 128] q~^T and
//     O^T[128 x 8 q] += V~^T[128 x 16 tok] P^T.  The <= 8 query rows of a kv head (the GQA
//     group, or group x drafts for verify) are the N = 8 side, so no query padding to 16.
//   * Codes become fp16 centroids through a lane-replicated shared-memory table: one byte of
//     codes (two 4-bit codes, two 3-bit codes assembled from the 3-bit planes, or four 2-bit
//     codes read as two halves) indexes a half2 entry; each lane reads its own copy of the
//     entry, so lookups never conflict.
//   * A decode step can hand the kernel the step's new K/V token of every sequence: the warp
//     that stages a unit's last tile quantizes the token into the cache before it copies that
//     tile, so the step needs no separate append launch.
//   * Dense rotations (TurboQuant) change only the two ends: a small kernel forms R_k q for the
//     whole call first, and the CTA that finishes a unit applies the full R_v^T to its rows.
//   * P is moved from the S^T accumulator layout to the B-operand layout with movmatrix.
//   * Scores are kept in base 2 (sm_scale * log2 e folded into q~).
#include <cuda_fp16.h>
#include <math_constants.h>

#include <algorithm>

#include "rq_codec.cuh"
#include "rq_lut.cuh"
#include "rq_internal.h"
#include "../../include/rq.h"

namespace rq {
namespace {

constexpr int kLutBytes = lut::kBytes;
constexpr int kMaxSplitPages = 1024;          // page ids staged per item
constexpr int kWaitLimit = 1 << 22;           // bounded mbarrier polling (about a second)
// The running softmax max of the split-K kernel moves only when a score passes it by more than
// this (base 2): p = 2^(s - m) <= 2^8 in between, so most pairs need no warp reduction and no
// rescale.  Pairs holding a value norm >= 2^8 take the exact path (p <= 1) so that the fp16
// operand P' = p * n_v cannot overflow.
constexpr float kLazyMargin = 8.f;

// Staged tiles.  Each warp owns kSlots slots of SB bytes used as kSlots/2 stages of two
// consecutive tiles (32 tokens); one mbarrier per stage.  A stage holds its pair in one of two
// layouts, fixed by the page size:
//   * tile by tile (16-token pages, whose pair spans two pages, and pages of an odd number of
//     tiles): each slot is one tile as a 16-token page chunk is laid out, K codes [16][vb] |
//     V codes [16][vb] | K norms fp16 [16] | V norms fp16 [16];
//   * section by section (an even number of tiles per page, so a pair lies in one page):
//     K codes [32][vb] | V codes [32][vb] | K norms [32] | V norms [32], the four runs of the
//     page that the pair covers, so the pair is four bulk copies.
// The slots sit on both sides of the 64 KB-aligned lookup table (see smem_plan).
template <int BITS>
struct Ring {
  static constexpr int VB = BITS * 16;
  static constexpr int SB = 32 * VB + 64;     // slot bytes: 2112 (4-bit), 1600 (3-bit), 1088 (2-bit)
};
constexpr int kSlotsTotal = 64;               // staged tiles per CTA, whatever its warp count

// A unit of work covers NT n-tiles (8 query rows each) of one kv head: a warp then shares every
// dequantised K~ and V~ fragment between NT MMAs, so a verify of T drafts x G heads (e.g. 24
// rows) unpacks the cache once, not once per 8 rows.  Registers decide the warp count: 16 warps
// at 128 registers for NT = 1 (decode), 8 warps at up to 255 for NT = 2, 3, whose accumulators
// (NT x 32 floats of O, NT x 16 registers of queries) need them; the 64 staged tiles are then 4
// stages per warp instead of 2, so the bytes in flight per SM stay the same.
template <int NT>
struct Shape {
  static constexpr int kWarps = NT == 1 ? kAttnWarps : kAttnWarps / 2;
  static constexpr int kThreads = kWarps * 32;
  static constexpr int kSlots = kSlotsTotal / kWarps;  // per warp
  static constexpr int kStages = kSlots / 2;           // pairs of tiles in flight per warp
  static constexpr int kRoundTiles = 2 * kWarps;       // a round: one pair of 16-token tiles per warp
  // A CTA pays about 96 tiles' worth of work (3 rounds of 16 warps) for each extra fragment
  // (prologue, pipeline refill, the barriers and the merge), measured on 16 x 8K-token decode:
  // one whole unit per CTA on 128 of 152 SMs beat 13.5 rounds in two fragments per CTA on all 152.
  static constexpr int kFragmentRounds = 96 / kRoundTiles;
  static constexpr int kMergeHalfBytes = kWarps * 4 * kPartialStride * 4;  // 4 query columns of all warps
};

// Shared-memory plan for a CTA whose dynamic window starts at shared address `base`:
//   [base, lut)          low slots (as many whole pairs of slots as fit), or nothing
//   [lut, lut + 64 KB)   lookup table; lut = first 64 KB-aligned address >= base
//   [lut + 64 KB, ...)   the remaining slots, page ids int[1024], mbarriers u64[64 / 2],
//                        centroids float[16], the CTA's position in its tile range (Walk)
// Between items the two halves of the merge buffer (query columns 0-3 and 4-7) reuse slot
// space: the low region when it holds a half, else the high slots.
struct SmemPlan {
  uint32_t lut;        // shared address of the table
  int n_lo;            // slots below the table
  uint32_t hi;         // shared address of the first high slot
  uint32_t tail;       // shared address of the page-id array
  uint32_t merge_lo;   // shared address of merge half 0 (columns 0-3)
  uint32_t merge_hi;   // shared address of merge half 1 (columns 4-7)
  uint32_t obuf;       // dense rotation: 8 normalised output rows [8][128] f32 before R_v^T
  uint32_t end;        // one past the last byte used
};
constexpr int kObufBytes = 8 * 128 * 4;

// Rounds of one unit of a sequence of len tokens: ceil(tiles / kRoundTiles).
template <int NT>
__host__ __device__ __forceinline__ int unit_rounds(int len) {
  return ((len + 15) / 16 + Shape<NT>::kRoundTiles - 1) / Shape<NT>::kRoundTiles;
}

// Where a CTA stands in its range [x, x_end) of the partition's cost: sequence b, whose units'
// cost starts at cumb (a unit of rb rounds costs rb + the fragment overhead, see frag_at).  Kept in shared memory (thread 0 advances it between fragments) so that none of it
// occupies registers during the tile loop.
struct Walk {
  long long x, x_end, cumb;
  int b, len;  // len: sequence b's tokens, clamped to the block table (> 0 while x < x_end)
  // Units whose last-finished fragment was this CTA's (set by thread 0): at most the first and
  // the last fragment of a CTA's range are partial units, the ones between are whole.
  int n_fin;
  int fin[2];
};
constexpr int kWalkBytes = (int)((sizeof(Walk) + 15) / 16 * 16);
// The tail of the window: page ids, the warps' mbarriers (one per stage: kSlotsTotal / 2), the
// centroids and the walk.
constexpr int kTailBytes = kMaxSplitPages * 4 + (kSlotsTotal / 2) * 8 + 64 + kWalkBytes;

// The fragment at the walk's position: rounds [r0, r1) of the rb rounds of unit uib of
// sequence b (uib = kv head * units per head + unit of the head), i.e. its tiles [t0, t1) of tb.
// The partition splits cost, not rounds: unit u of a sequence covers [cumb + u C, cumb + (u + 1)
// C) with C = rb + kFragmentRounds, its first kFragmentRounds standing for the work of opening a
// fragment, the rest for its rounds, so a range that crosses many small units is shorter in
// rounds.  A range that ends inside a unit's opening part takes none of its rounds (r1 <= r0).
struct Frag {
  int tb, rb, uib, r0, r1, t0, t1;
};
template <int NT>
__device__ __forceinline__ Frag frag_at(const Walk& w) {
  constexpr int F = Shape<NT>::kFragmentRounds;
  Frag f;
  f.tb = (w.len + 15) / 16;
  f.rb = max(unit_rounds<NT>(w.len), 1);      // >= 1 whenever the walk has work left
  const int c = f.rb + F;
  const long long off = w.x - w.cumb;         // < the cost of one sequence's units
  f.uib = (int)(off / c);
  f.r0 = max((int)(off % c) - F, 0);
  f.r1 = (int)min((long long)f.rb, w.x_end - w.cumb - (long long)f.uib * c - F);
  f.t0 = f.r0 * Shape<NT>::kRoundTiles;
  f.t1 = min(f.tb, f.r1 * Shape<NT>::kRoundTiles);
  return f;
}

template <int BITS, int NT>
__host__ __device__ constexpr SmemPlan smem_plan(uint32_t base) {
  constexpr uint32_t merge_half = Shape<NT>::kMergeHalfBytes;
  SmemPlan p{};
  p.lut = (base + 0xFFFFu) & ~0xFFFFu;
  int n_lo = (int)((p.lut - base) / Ring<BITS>::SB) & ~1;  // whole pairs: a warp's slots 2s, 2s+1 adjoin
  if (n_lo > kSlotsTotal) n_lo = kSlotsTotal;
  p.n_lo = n_lo;
  p.hi = p.lut + kLutBytes;
  const uint32_t hi_bytes = (uint32_t)(kSlotsTotal - n_lo) * Ring<BITS>::SB;
  const bool lo_merge = (uint32_t)n_lo * Ring<BITS>::SB >= merge_half;
  p.merge_lo = lo_merge ? base : p.hi;
  p.merge_hi = lo_merge ? p.hi : p.hi + merge_half;
  const uint32_t hi_need = lo_merge ? merge_half : 2 * merge_half;
  p.tail = p.hi + (hi_bytes > hi_need ? hi_bytes : hi_need);
  p.obuf = p.tail + kTailBytes;
  p.end = p.obuf + kObufBytes;
  return p;
}

// ---------------------------------------------------------------------------------------
// PTX helpers
// ---------------------------------------------------------------------------------------
template <uint32_t LUT>
__device__ __forceinline__ uint32_t lop3(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, %4;" : "=r"(d) : "r"(a), "r"(b), "r"(c), "n"(LUT));
  return d;
}
// (a & c) | (b & ~c)
__device__ __forceinline__ uint32_t bitsel(uint32_t a, uint32_t b, uint32_t c) { return lop3<0xE4>(a, b, c); }

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// d = A B with a zero accumulator (C given as constant zeros, so no register needs clearing).
__device__ __forceinline__ void mma16816_z(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                           uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%10,%10,%10,%10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.f));
}

__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(x));
  return d;
}

__device__ __forceinline__ void mbar_init(uint32_t addr, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(addr), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t addr, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(addr), "r"(bytes) : "memory");
}
__device__ __forceinline__ uint32_t mbar_try_wait(uint32_t addr, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(addr), "r"(parity)
      : "memory");
  return ok;
}
// Polls an mbarrier phase at most kWaitLimit times; false if it never completed.
// (try_wait itself suspends the thread for a while, so the first poll nearly always succeeds.)
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t addr, uint32_t parity) {
  if (mbar_try_wait(addr, parity)) return true;
  for (int i = 1; i < kWaitLimit; ++i)
    if (mbar_try_wait(addr, parity)) return true;
  return false;
}
// 1-D bulk copy global -> this CTA's shared memory (TMA), completing on an mbarrier.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t mbar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(mbar)
               : "memory");
}
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
// True in one lane of the (converged) warp.
__device__ __forceinline__ bool elect_one() {
  uint32_t is_leader;
  asm volatile("{\n .reg .pred p;\n elect.sync _|p, 0xffffffff;\n selp.u32 %0, 1, 0, p;\n}" : "=r"(is_leader));
  return is_leader != 0;
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ float half_bits_to_float(uint32_t bits16) {
  return __half2float(__ushort_as_half((unsigned short)bits16));
}

// ---------------------------------------------------------------------------------------
// Code tables (rq_lut.cuh): T4 / T1 + T2 / U1 + U2 turn an index byte of two codes into the
// half2 of their centroids with one shared load.
// ---------------------------------------------------------------------------------------
// Half2 of the two codes in byte J of index word x (SECOND selects the second table); key1 /
// key2 are the lane's table keys (lut::key).
template <int J, int SECOND>
__device__ __forceinline__ uint32_t lut_at(uint32_t x, uint32_t key1, uint32_t key2) {
  return lut::get(x, J, SECOND ? key2 : key1);
}
template <int SECOND>
__device__ __forceinline__ uint32_t lut_dyn(uint32_t x, int j, uint32_t key1, uint32_t key2) {
  return lut::get(x, j, SECOND ? key2 : key1);
}

// 2^x on the SFU (x = -inf gives +0, which masked scores rely on).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---------------------------------------------------------------------------------------
// Raw tile data of one lane (lane = 4g + t), read from a staged tile in shared memory.
// The MMA rows of a tile map to its tokens through rho(r): the identity for 4- and 2-bit codes,
// whose V token pairs are stored swizzled, and r ^ ((r >> 1) & 1) for 3-bit codes, a permutation
// chosen so that the staged reads are conflict-free for K and at most 2-way for V:
//   K rows g and g+8 -> tokens rho(g), rho(g) + 8, the 32 dims 32t..32t+31 of each;
//   V k-slots 2t, 2t+1, 2t+8, 2t+9 -> tokens rho(2t), rho(2t+1), rho(2t) + 8, rho(2t+1) + 8,
//     the 16 dims 16g..16g+15 of each;
//   the K and V norms of tokens rho(g) and rho(g) + 8.
// Both contractions sum over tokens, so any permutation gives the same result as long as the
// score rows, the norms, the masks and the P^T operand use the same one.
// ---------------------------------------------------------------------------------------
template <int BITS>
__device__ __forceinline__ int rho(int r) {
  return BITS == 3 ? (r ^ ((r >> 1) & 1)) : r;
}

template <int BITS>
struct Raw;

template <>
struct Raw<4> {
  uint4 k[2];        // 16 bytes = 32 codes per K row
  uint2 v[4];        // 8 bytes = 16 codes per V token
  uint32_t nk, nv;   // fp16 norms of the two K rows' tokens (low, high)
};
template <>
struct Raw<2> {
  uint2 k[2];        // 8 bytes = 32 codes per K row
  uint2 v[2];        // V token pairs (2t, 2t+1) and (2t+8, 2t+9): 4 bytes = 16 codes per token
  uint32_t nk, nv;
};
template <>
struct Raw<3> {
  uint32_t k[2][3];  // W0, W1, W2 of group t
  uint32_t v[4][2];  // W(g&1) and W2 of group g/2
  uint32_t nk, nv;
};

// Tile data at: st its K code rows, vbp its V code rows, nkb / nvb its K / V norms.
template <int BITS>
__device__ __forceinline__ void load_stage(Raw<BITS>& r, const uint8_t* st, const uint8_t* vbp, const uint8_t* nkb,
                                           const uint8_t* nvb, int g, int t) {
  const int rk = rho<BITS>(g);
  if constexpr (BITS == 4) {
    r.k[0] = *reinterpret_cast<const uint4*>(st + rk * 64 + 16 * t);
    r.k[1] = *reinterpret_cast<const uint4*>(st + (rk + 8) * 64 + 16 * t);
    // V token pairs (2t, 2t+1) and (2t+8, 2t+9) are 128-byte pair rows t and t+4; the lane's
    // 16-dim group g of both tokens is one 16-byte unit, at 16 * (g ^ 2t mod 8) in either row.
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int pair = t + 4 * i;
      const uint4 u = *reinterpret_cast<const uint4*>(vbp + pair * 128 + 16 * (g ^ ((2 * pair) & 7)));
      r.v[2 * i] = make_uint2(u.x, u.y);
      r.v[2 * i + 1] = make_uint2(u.z, u.w);
    }
  } else if constexpr (BITS == 2) {
    r.k[0] = *reinterpret_cast<const uint2*>(st + rk * 32 + 8 * t);
    r.k[1] = *reinterpret_cast<const uint2*>(st + (rk + 8) * 32 + 8 * t);
    // 64-byte pair rows t and t+4; the 4-byte units of group g of both tokens are adjacent, at
    // 8 * (g ^ (4 * (pair / 2 mod 2))).
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int pair = t + 4 * i;
      r.v[i] = *reinterpret_cast<const uint2*>(vbp + pair * 64 + 8 * (g ^ (4 * ((pair >> 1) & 1))));
    }
  } else {
    const int va = rho<BITS>(2 * t), vbt = rho<BITS>(2 * t + 1);
    const int vt[4] = {va, vbt, va + 8, vbt + 8};
#pragma unroll
    for (int rr = 0; rr < 2; ++rr)
#pragma unroll
      for (int w = 0; w < 3; ++w)
        r.k[rr][w] = *reinterpret_cast<const uint32_t*>(st + (rk + 8 * rr) * 48 + 12 * t + 4 * w);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      r.v[i][0] = *reinterpret_cast<const uint32_t*>(vbp + vt[i] * 48 + 12 * (g >> 1) + 4 * (g & 1));
      r.v[i][1] = *reinterpret_cast<const uint32_t*>(vbp + vt[i] * 48 + 12 * (g >> 1) + 8);
    }
  }
  const uint16_t* nk16 = reinterpret_cast<const uint16_t*>(nkb);
  const uint16_t* nv16 = reinterpret_cast<const uint16_t*>(nvb);
  r.nk = (uint32_t)nk16[rk] | ((uint32_t)nk16[rk + 8] << 16);
  r.nv = (uint32_t)nv16[rk] | ((uint32_t)nv16[rk + 8] << 16);
}

// A operand of S^T = K~ q~^T for k-chunk kc: rows g / g+8 hold the two K rows, k-slots
// 2t,2t+1 hold dim pair 2kc and 2t+8,2t+9 dim pair 2kc+1 of the lane's 32 dims.
// 4-bit: pair j is byte j of the row's 16 bytes.
// 2-bit: byte kc of the row's 8 bytes carries dims 4kc..4kc+3; U1 gives (4kc, 4kc+2) for
//        k-slots 2t,2t+1 and U2 gives (4kc+1, 4kc+3) for 2t+8,2t+9, and q~ is packed to match.
// 3-bit: X0 = W0.lo | W2.hi (T1, pairs 2k), X1 = W2.lo | W0.hi (T2, pairs 2k+1),
//        X2 = W1.lo | (W2>>2).hi (T1, pairs 8+2k), X3 = (W2>>2).lo | W1.hi (T2, pairs 9+2k).
// With NT n-tiles, each A fragment feeds NT MMAs (one per n-tile's queries); with one, the even
// and odd k-chunks accumulate in two chains for the MMAs' latency.
template <int BITS, int NT>
__device__ __forceinline__ void qk_tile(float (&s)[NT][4], const Raw<BITS>& r, const uint32_t (&qf)[NT][8][2],
                                        uint32_t key1, uint32_t key2) {
  float s2[4];
  // (the first MMA of each chain starts from zero: kc 0 and 1 with one n-tile, kc 0 with more)
  auto mma_all = [&](int kc, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3) {
    if constexpr (NT == 1) {
      if (kc == 0) mma16816_z(s[0], a0, a1, a2, a3, qf[0][kc][0], qf[0][kc][1]);
      else if (kc == 1) mma16816_z(s2, a0, a1, a2, a3, qf[0][kc][0], qf[0][kc][1]);
      else if (kc & 1) mma16816(s2, a0, a1, a2, a3, qf[0][kc][0], qf[0][kc][1]);
      else mma16816(s[0], a0, a1, a2, a3, qf[0][kc][0], qf[0][kc][1]);
    } else {
#pragma unroll
      for (int i = 0; i < NT; ++i) {
        if (kc == 0) mma16816_z(s[i], a0, a1, a2, a3, qf[i][kc][0], qf[i][kc][1]);
        else mma16816(s[i], a0, a1, a2, a3, qf[i][kc][0], qf[i][kc][1]);
      }
    }
  };
  if constexpr (BITS == 4) {
    const uint32_t k0[4] = {r.k[0].x, r.k[0].y, r.k[0].z, r.k[0].w};
    const uint32_t k1[4] = {r.k[1].x, r.k[1].y, r.k[1].z, r.k[1].w};
#pragma unroll
    for (int kc = 0; kc < 8; ++kc) {
      const int w = kc >> 1, j0 = (2 * kc) & 3;
      uint32_t a0, a1, a2, a3;
      if (j0 == 0) {
        a0 = lut_at<0, 0>(k0[w], key1, key2);
        a1 = lut_at<0, 0>(k1[w], key1, key2);
        a2 = lut_at<1, 0>(k0[w], key1, key2);
        a3 = lut_at<1, 0>(k1[w], key1, key2);
      } else {
        a0 = lut_at<2, 0>(k0[w], key1, key2);
        a1 = lut_at<2, 0>(k1[w], key1, key2);
        a2 = lut_at<3, 0>(k0[w], key1, key2);
        a3 = lut_at<3, 0>(k1[w], key1, key2);
      }
      mma_all(kc, a0, a1, a2, a3);
    }
  } else if constexpr (BITS == 2) {
    const uint32_t k0[2] = {r.k[0].x, r.k[0].y};
    const uint32_t k1[2] = {r.k[1].x, r.k[1].y};
#pragma unroll
    for (int kc = 0; kc < 8; ++kc) {
      const int w = kc >> 2, byte = kc & 3;
      uint32_t a0, a1, a2, a3;
      lut::get2(k0[w], byte, key1, a0, a2);  // (U1, U2) of one index byte: one 8-byte load
      lut::get2(k1[w], byte, key1, a1, a3);
      mma_all(kc, a0, a1, a2, a3);
    }
  } else {
    uint32_t X[2][4];
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      const uint32_t w0 = r.k[rr][0], w1 = r.k[rr][1], w2 = r.k[rr][2], w2s = w2 >> 2;
      X[rr][0] = bitsel(w0, w2, 0x0F0F0F0Fu);
      X[rr][1] = bitsel(w2, w0, 0x0F0F0F0Fu);
      X[rr][2] = bitsel(w1, w2s, 0x0F0F0F0Fu);
      X[rr][3] = bitsel(w2s, w1, 0x0F0F0F0Fu);
    }
#pragma unroll
    for (int kc = 0; kc < 8; ++kc) {
      const int hi = kc >> 2, byte = kc & 3;
      const uint32_t a0 = lut_dyn<0>(X[0][2 * hi], byte, key1, key2);
      const uint32_t a1 = lut_dyn<0>(X[1][2 * hi], byte, key1, key2);
      const uint32_t a2 = lut_dyn<1>(X[0][2 * hi + 1], byte, key1, key2);
      const uint32_t a3 = lut_dyn<1>(X[1][2 * hi + 1], byte, key1, key2);
      mma_all(kc, a0, a1, a2, a3);
    }
  }
  if constexpr (NT == 1) {
#pragma unroll
    for (int i = 0; i < 4; ++i) s[0][i] += s2[i];
  }
}

// A operand of O^T += V~^T P^T for m-tile mt: rows g / g+8 hold dims 16g+2mt / 16g+2mt+1,
// k-slots 2t,2t+1 and 2t+8,2t+9 the lane's two V token pairs.  Index bytes carry one
// dim of two tokens, so the two tokens' code words are interleaved first.
// Each A fragment feeds NT MMAs, one per n-tile's P^T (pb[i] = its two B registers).
template <int BITS, int NT>
__device__ __forceinline__ void pv_tile(float (&o)[NT][8][4], const Raw<BITS>& r, const uint32_t (&pb)[NT][2],
                                        uint32_t key1, uint32_t key2, int g) {
  auto mma_all = [&](int mt, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3) {
#pragma unroll
    for (int i = 0; i < NT; ++i) mma16816(o[i][mt], a0, a1, a2, a3, pb[i][0], pb[i][1]);
  };
  if constexpr (BITS == 4) {
    uint32_t XE[2][2], XO[2][2];  // [token pair][word]
#pragma unroll
    for (int pr = 0; pr < 2; ++pr) {
      const uint2 A = r.v[2 * pr], B = r.v[2 * pr + 1];
      XE[pr][0] = bitsel(A.x, B.x << 4, 0x0F0F0F0Fu);
      XE[pr][1] = bitsel(A.y, B.y << 4, 0x0F0F0F0Fu);
      XO[pr][0] = bitsel(A.x >> 4, B.x, 0x0F0F0F0Fu);
      XO[pr][1] = bitsel(A.y >> 4, B.y, 0x0F0F0F0Fu);
    }
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      const int w = mt >> 2, j = mt & 3;
      const uint32_t a0 = lut_dyn<0>(XE[0][w], j, key1, key2);
      const uint32_t a1 = lut_dyn<0>(XO[0][w], j, key1, key2);
      const uint32_t a2 = lut_dyn<0>(XE[1][w], j, key1, key2);
      const uint32_t a3 = lut_dyn<0>(XO[1][w], j, key1, key2);
      mma_all(mt, a0, a1, a2, a3);
    }
  } else if constexpr (BITS == 2) {
    // Nibble-interleave each token pair: byte k of XE = (dims 4k, 4k+1 of the first token,
    // the same dims of the second); XO the same for dims 4k+2, 4k+3.  U1 of such a byte is
    // the k-slot pair of the lower dim, U2 that of the upper one.
    uint32_t XE[2], XO[2];
#pragma unroll
    for (int pr = 0; pr < 2; ++pr) {
      const uint32_t A = r.v[pr].x, B = r.v[pr].y;
      XE[pr] = bitsel(A, B << 4, 0x0F0F0F0Fu);
      XO[pr] = bitsel(A >> 4, B, 0x0F0F0F0Fu);
    }
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      const int j = mt >> 1;
      const uint32_t x0 = (mt & 1) ? XO[0] : XE[0], x1 = (mt & 1) ? XO[1] : XE[1];
      uint32_t a0, a1, a2, a3;
      lut::get2(x0, j, key1, a0, a1);
      lut::get2(x1, j, key1, a2, a3);
      mma_all(mt, a0, a1, a2, a3);
    }
  } else {
    const int sh = 2 * (g & 1);
    uint32_t XE1[2], XE2[2], XO1[2], XO2[2];
#pragma unroll
    for (int pr = 0; pr < 2; ++pr) {
      const uint32_t A = r.v[2 * pr][0], B = r.v[2 * pr + 1][0];
      const uint32_t A2 = r.v[2 * pr][1], B2 = r.v[2 * pr + 1][1];
      const uint32_t E = bitsel(A, B << 2, 0x33333333u);
      const uint32_t O = bitsel(A >> 2, B, 0x33333333u);
      const uint32_t M = bitsel(A2, B2 << 1, 0x55555555u) >> sh;
      const uint32_t M2 = bitsel(A2 >> 1, B2, 0x55555555u) >> sh;
      XE1[pr] = bitsel(E, M, 0x0F0F0F0Fu);
      XE2[pr] = bitsel(M, E, 0x0F0F0F0Fu);
      XO1[pr] = bitsel(O, M2, 0x0F0F0F0Fu);
      XO2[pr] = bitsel(M2, O, 0x0F0F0F0Fu);
    }
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      const int j = mt >> 1;
      uint32_t a0, a1, a2, a3;
      if ((mt & 1) == 0) {
        a0 = lut_dyn<0>(XE1[0], j, key1, key2);
        a1 = lut_dyn<0>(XO1[0], j, key1, key2);
        a2 = lut_dyn<0>(XE1[1], j, key1, key2);
        a3 = lut_dyn<0>(XO1[1], j, key1, key2);
      } else {
        a0 = lut_dyn<1>(XE2[0], j, key1, key2);
        a1 = lut_dyn<1>(XO2[0], j, key1, key2);
        a2 = lut_dyn<1>(XE2[1], j, key1, key2);
        a3 = lut_dyn<1>(XO2[1], j, key1, key2);
      }
      mma_all(mt, a0, a1, a2, a3);
    }
  }
}

// ---------------------------------------------------------------------------------------
// Log-sum-exp merge of one query row's split partials: o~ = sum_s 2^(m_s - M) O_s / L with
// M = max_s m_s and L = sum_s 2^(m_s - M) l_s, for the lane's dims 4 lane .. 4 lane + 3.  The
// lanes take the splits' (m, l) one split each, so M and L are warp reductions rather than
// chains of dependent loads, and the O sum issues its independent loads eight at a time.
// Zeros for an empty (or invalid) sequence.  All 32 lanes must call it.
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ float4 merge_splits(const Geometry& g, const AttnArgs& a, int b, int h, int row, int lane) {
  const int rows_u = 8 * a.nt;  // query rows per unit
  const int ug = row / rows_u, col = row - ug * rows_u;
  int len = a.seq_lens[b];
  const int cap = a.max_pages * g.page_size;
  len = len < 0 ? 0 : (len > cap ? cap : len);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (len == 0 || len < a.T) return acc;
  // the unit's fragments: CTAs first .. last, partials at slots unit + c
  const int unit = (b * g.num_kv_heads + h) * ((a.n_tiles_n + a.nt - 1) / a.nt) + ug;
  // written by other CTAs of this launch (or the previous kernel): read through L2
  const int first = __ldcg(a.frag + 2 * unit), last = __ldcg(a.frag + 2 * unit + 1);
  if (first < 0 || last < first || last >= a.grid) return acc;  // a launch that gave up early
  const int ns = last - first + 1;
  const size_t stride = (size_t)rows_u * kPartialStride;  // between consecutive slots
  const float* base = a.ws + (size_t)(unit + first) * stride + (size_t)col * kPartialStride;
  // (m, l) of the lane's slots, one load each; running max and rescaled sum, then warp-merged
  float M = -CUDART_INF_F, L = 0.f;
  for (int s = lane; s < ns; s += 32) {
    const float2 ml = __ldcg(reinterpret_cast<const float2*>(base + s * stride));
    if (ml.x == -CUDART_INF_F) continue;
    const float m_new = fmaxf(M, ml.x);
    L = L * exp2f(M - m_new) + ml.y * exp2f(ml.x - m_new);
    M = m_new;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float M2 = __shfl_xor_sync(0xffffffffu, M, o), L2 = __shfl_xor_sync(0xffffffffu, L, o);
    const float m_new = fmaxf(M, M2);
    if (m_new != -CUDART_INF_F) L = (M == -CUDART_INF_F ? 0.f : L * exp2f(M - m_new)) +
                                    (M2 == -CUDART_INF_F ? 0.f : L2 * exp2f(M2 - m_new));
    M = m_new;
  }
  if (M == -CUDART_INF_F) return acc;
#pragma unroll 8
  for (int s = 0; s < ns; ++s) {
    const float* ps = base + s * stride;
    const float w = exp2f(__ldcg(ps) - M);
    const float4 v = __ldcg(reinterpret_cast<const float4*>(ps + 4 + 4 * lane));
    acc.x += v.x * w;
    acc.y += v.y * w;
    acc.z += v.z * w;
    acc.w += v.w * w;
  }
  const float inv = L > 0.f ? g.out_scale / L : 0.f;
  return make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
}

// The four R_v entries of kv head h for dims d0 & ~3 .. (d0 & ~3) + 3: a Givens pair's (c, s)
// twice, or the block's quaternion.  Loaded ahead of the merge that needs them.
__device__ __forceinline__ float4 rot_v_block(const Geometry& g, int h, int d0) {
  return __ldg(reinterpret_cast<const float4*>(g.rot_v + (size_t)h * kHeadDim + (d0 & ~3)));
}

// out = R_v^T o~ for query row `row` of kv head h of sequence b (planar / iso: block-local),
// the lane's dims 4 lane .. 4 lane + 3, as fp16; p = rot_v_block(g, h, 4 lane).  All 32 lanes of
// the warp call it.
__device__ __forceinline__ void store_row(const Geometry& g, const AttnArgs& a, int b, int h, int row, int lane,
                                          float4 o, float4 p) {
  const float y[4] = {o.x, o.y, o.z, o.w};
  float x[4];
  if (g.mode == RQ_PLANAR) {
    x[0] = p.x * y[0] + p.y * y[1];
    x[1] = -p.y * y[0] + p.x * y[1];
    x[2] = p.z * y[2] + p.w * y[3];
    x[3] = -p.w * y[2] + p.z * y[3];
  } else {  // L(q)^T y
    const float qa = p.x, qb = p.y, qc = p.z, qd = p.w;
    x[0] = qa * y[0] + qb * y[1] + qc * y[2] + qd * y[3];
    x[1] = -qb * y[0] + qa * y[1] + qd * y[2] - qc * y[3];
    x[2] = -qc * y[0] - qd * y[1] + qa * y[2] + qb * y[3];
    x[3] = -qd * y[0] + qc * y[1] - qb * y[2] + qa * y[3];
  }
  const int j = row / g.group, head = h * g.group + row % g.group;
  __half2* out = reinterpret_cast<__half2*>(reinterpret_cast<__half*>(a.out) +
                                            (((size_t)b * a.T + j) * g.num_q_heads + head) * kHeadDim + 4 * lane);
  out[0] = __floats2half2_rn(x[0], x[1]);
  out[1] = __floats2half2_rn(x[2], x[3]);
}

// The same for the two dims d0, d0 + 1 (d0 even) of row `row`, held as (y0, y1) by this lane;
// with a quaternion rotation the block's other two dims are held by lane ^ 1 (d0 ^ 2).
// r = rot_v_block(g, h, d0).  All 32 lanes of the warp call it.
__device__ __forceinline__ void store_pair(const Geometry& g, const AttnArgs& a, int b, int h, int row, int d0,
                                           float y0, float y1, float4 r) {
  const float z0 = __shfl_xor_sync(0xffffffffu, y0, 1), z1 = __shfl_xor_sync(0xffffffffu, y1, 1);
  float x0, x1;
  if (g.mode == RQ_PLANAR) {  // the pair's (c, s): first or second half of the block
    const float c = (d0 & 2) ? r.z : r.x, sn = (d0 & 2) ? r.w : r.y;
    x0 = c * y0 + sn * y1;
    x1 = -sn * y0 + c * y1;
  } else {
    const float qa = r.x, qb = r.y, qc = r.z, qd = r.w;
    if ((d0 & 2) == 0) {  // own dims 0, 1 of the block; the partner's are 2, 3
      x0 = qa * y0 + qb * y1 + qc * z0 + qd * z1;
      x1 = -qb * y0 + qa * y1 + qd * z0 - qc * z1;
    } else {              // own dims 2, 3; the partner's are 0, 1
      x0 = -qc * z0 - qd * z1 + qa * y0 + qb * y1;
      x1 = -qd * z0 + qc * z1 - qb * y0 + qa * y1;
    }
  }
  const int j = row / g.group, head = h * g.group + row % g.group;
  *reinterpret_cast<__half2*>(reinterpret_cast<__half*>(a.out) +
                              (((size_t)b * a.T + j) * g.num_q_heads + head) * kHeadDim + d0) =
      __floats2half2_rn(x0, x1);
}

// ---------------------------------------------------------------------------------------
// The split-K kernel.
// ---------------------------------------------------------------------------------------
// The lane's 32 dims 32tq..32tq+31 of R_k q for query row `row` of kv head h (zeros past the
// rows): read from the call's pre-rotated buffer for a dense rotation (PRE), else the row's
// fp16 q turned here -- Givens pairs or quaternion blocks never leave the lane's dims.
template <bool PRE>
__device__ __forceinline__ void rotated_query(float (&y)[32], const Geometry& g, const AttnArgs& a, int b, int h,
                                              int row, int tq) {
  const int j = row / g.group, head = h * g.group + row % g.group;
  const size_t qoff = (((size_t)b * a.T + j) * g.num_q_heads + head) * kHeadDim + 32 * tq;
  if constexpr (PRE) {
    const float4* src = reinterpret_cast<const float4*>(a.q_rot + qoff);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const float4 f = row < a.rows ? src[c] : make_float4(0.f, 0.f, 0.f, 0.f);
      y[4 * c] = f.x;
      y[4 * c + 1] = f.y;
      y[4 * c + 2] = f.z;
      y[4 * c + 3] = f.w;
    }
  } else {
    float qv[32];
    if (row < a.rows) {
      const __half* src = reinterpret_cast<const __half*>(a.q) + qoff;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const uint4 raw = *reinterpret_cast<const uint4*>(src + 8 * c);
        const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[e]));
          qv[8 * c + 2 * e] = f.x;
          qv[8 * c + 2 * e + 1] = f.y;
        }
      }
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) qv[i] = 0.f;
    }
    const float4* rp = reinterpret_cast<const float4*>(g.rot_k + (size_t)h * kHeadDim + 32 * tq);
#pragma unroll
    for (int blk = 0; blk < 8; ++blk) {
      const float4 p = __ldg(rp + blk);
      const float* x = qv + 4 * blk;
      if (g.mode == RQ_PLANAR) {
        y[4 * blk + 0] = p.x * x[0] - p.y * x[1];
        y[4 * blk + 1] = p.y * x[0] + p.x * x[1];
        y[4 * blk + 2] = p.z * x[2] - p.w * x[3];
        y[4 * blk + 3] = p.w * x[2] + p.z * x[3];
      } else {
        y[4 * blk + 0] = p.x * x[0] - p.y * x[1] - p.z * x[2] - p.w * x[3];
        y[4 * blk + 1] = p.y * x[0] + p.x * x[1] - p.w * x[2] + p.z * x[3];
        y[4 * blk + 2] = p.z * x[0] + p.w * x[1] + p.x * x[2] - p.y * x[3];
        y[4 * blk + 3] = p.w * x[0] - p.z * x[1] + p.y * x[2] + p.x * x[3];
      }
    }
  }
}
// The stream-K partition: CTA `cta` of `grid` gets rounds [x0, x1) of `total`.  Parts =
// min(CTAs, rounds), so that every part is non-empty: the combine takes the CTAs between a
// unit's first and last fragment to all hold one.  CTAs past the parts idle.  When every unit
// has the same rounds and there are no more units than CTAs, one whole unit per part is the
// other candidate: a CTA's cost is its rounds plus frag_rounds per fragment, and equal parts
// that do not divide the units cost most CTAs two fragments.  I is uint32_t whenever
// total * grid fits it (every practical launch: the 64-bit division is a long software
// sequence), else long long.
template <typename I>
__device__ __forceinline__ void partition(I total, I n_units, I max_rounds, I grid, I cta, I frag_rounds,
                                          long long& x0, long long& x1) {
  // total: the cost of all units (rounds + frag_rounds each); whole units, one a CTA, when they
  // are all alike and that beats splitting the rounds over the grid
  const I rounds = total - n_units * frag_rounds;
  I parts = min(grid, rounds);
  if (n_units > 0 && n_units <= grid && rounds == n_units * max_rounds) {
    const I per_part = (rounds + parts - 1) / parts;
    const I cost_split = per_part + (max_rounds % per_part == 0 ? 1 : 2) * frag_rounds;
    if (max_rounds + frag_rounds <= cost_split) parts = n_units;
  }
  x0 = cta < parts ? (long long)(total * cta / parts) : 0;
  x1 = cta < parts ? (long long)(total * (cta + 1) / parts) : 0;
}

// Starts an L2 fill of line `line` (128 bytes) of [p, p + lines * 128), if it exists.
__device__ __forceinline__ void prefetch_line_l2(const void* p, uint32_t lines, uint32_t line) {
  if (line < lines) asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<const char*>(p) + (size_t)line * 128));
}

// Sequence b's tokens, clamped to what its block-table row can hold.
__device__ __forceinline__ int clamp_len(const AttnArgs& a, int b, int cap) {
  const int l = a.seq_lens[b];
  return l < 0 ? 0 : (l > cap ? cap : l);
}

// Moves a walk past the fragment f it stands on (thread 0, between fragments): to the next
// unit's cost when f finished its unit, else to the end of the range.
template <int NT>
__device__ __forceinline__ void walk_advance(Walk& w, const Frag& f, int upb, const AttnArgs& a, int cap) {
  const int c = f.rb + Shape<NT>::kFragmentRounds;
  w.x = f.r1 == f.rb ? w.cumb + (long long)(f.uib + 1) * c : w.x_end;
  if (w.x >= w.x_end) return;  // the range is done: no next sequence to look up
  if (f.uib == upb - 1) {  // sequence b is done: on to the next one with tiles
    w.cumb += (long long)c * upb;
    for (++w.b; w.x < w.x_end && w.b < a.B; ++w.b) {
      w.len = clamp_len(a, w.b, cap);
      if (w.len > 0) break;
    }
    if (w.b >= a.B) w.x = w.x_end;  // nothing left (cannot happen with a consistent prefix)
  }
}

// Decode step: quantizes the newest token (position len - 1) of sequence b, kv head h into its
// slot of the cache, one warp (lanes 0-15 K, 16-31 V, 8 dims each).  The caller is the warp that
// stages the unit's last tile, which holds the token, and issues that tile's copy only after
// this returns: the proxy fence and the warp barrier order the writes before it.  The units of
// one kv head (more than 3 n-tiles) may write the same token from several CTAs, with equal bytes.
template <int BITS>
__device__ __forceinline__ void append_token(const Geometry& g, const AttnArgs& a, int b, int h, int len) {
  const int lane = threadIdx.x & 31, half = lane >> 4, j = lane & 15;
  float bnd[15];
  codec::load_boundaries<BITS>(bnd, g.boundaries);
  const int pos = len - 1;
  const int page = a.block_table[(size_t)b * a.max_pages + pos / g.page_size];
  const bool ok = page >= 0 && page < g.num_pages;
  if (!ok && lane == 0 && a.status) atomicOr(a.status, RQ_STATUS_BAD_PAGE);
  const __half* src = (half ? a.v_new : a.k_new) + ((size_t)b * g.num_kv_heads + h) * kHeadDim + 8 * j;
  const float* rot = (half ? g.rot_v : g.rot_k) + (size_t)h * kHeadDim + 8 * j;
  const float4 p0 = __ldg(reinterpret_cast<const float4*>(rot));
  const float4 p1 = __ldg(reinterpret_cast<const float4*>(rot + 4));
  const float pr[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
  // the cache is the caller's writable pool; the attention arguments carry it read-only
  uint8_t* chunk = const_cast<uint8_t*>(a.pages) + ((size_t)(ok ? page : 0) * g.num_kv_heads + h) * g.page_bytes;
  codec::encode_structured<BITS>(*reinterpret_cast<const uint4*>(src), pr, g.mode, bnd, chunk, g.page_size, half,
                                 pos % g.page_size, j, ok, a.status);
  asm volatile("fence.proxy.async.global;" ::: "memory");
  __syncwarp();
}

// Dense rotation: out = R_v^T o~ for nrows (<= 8) query rows row0 .. of kv head h of sequence b,
// whose normalised o~ (already times out_scale / l) are in ob[r][128] (shared memory).  Every
// thread of the CTA calls it: thread (rp, i) of 128-thread groups rp owns output dim i of rows
// rp, rp + groups, ...; R_v is read from L2 (each entry once per group of 128 threads).
template <int THREADS>
__device__ __forceinline__ void dense_finish_rows(const Geometry& g, const AttnArgs& a, int b, int h, int row0,
                                                  int nrows, const float (*ob)[kHeadDim]) {
  constexpr int kGroups = THREADS / kHeadDim, kPer = 8 / kGroups;
  const int i = threadIdx.x % kHeadDim, rp = threadIdx.x / kHeadDim;
  float acc[kPer];
#pragma unroll
  for (int q = 0; q < kPer; ++q) acc[q] = 0.f;
  const float* rv = g.rot_v + (size_t)h * kHeadDim * kHeadDim + i;  // R_v[m][i], row-major
  // 32 independent loads in flight per round trip to L2 (the column is read once per thread)
#pragma unroll 1
  for (int m0 = 0; m0 < kHeadDim; m0 += 32) {
    float w[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) w[e] = __ldg(rv + (size_t)(m0 + e) * kHeadDim);
#pragma unroll
    for (int e = 0; e < 32; ++e)
#pragma unroll
      for (int q = 0; q < kPer; ++q) acc[q] = fmaf(w[e], ob[rp + kGroups * q][m0 + e], acc[q]);
  }
#pragma unroll
  for (int q = 0; q < kPer; ++q) {
    const int r = rp + kGroups * q;
    if (r < nrows) {
      const int row = row0 + r, j = row / g.group, head = h * g.group + row % g.group;
      reinterpret_cast<__half*>(a.out)[(((size_t)b * a.T + j) * g.num_q_heads + head) * kHeadDim + i] =
          __float2half_rn(acc[q]);
    }
  }
}

// PRE: the queries were rotated before the launch (dense rotation).  STEP: a decode step that
// quantizes each sequence's newest token first (a.k_new, a.v_new; structured rotations).
// NT: query n-tiles per unit (Shape), each warp carrying all NT of them through every tile.
template <int BITS, bool PRE, bool STEP, int NT>
__global__ void __launch_bounds__(Shape<NT>::kThreads, 1)
attn_splitk_kernel(const Geometry g, const AttnArgs a, int smem_bytes) {
  using R = Ring<BITS>;
  constexpr int kWarps = Shape<NT>::kWarps;
  constexpr int kThreads = Shape<NT>::kThreads;
  constexpr int kSlots = Shape<NT>::kSlots;
  constexpr int kStages = Shape<NT>::kStages;
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t dyn_base = (uint32_t)__cvta_generic_to_shared(smem);
  const SmemPlan plan = smem_plan<BITS, NT>(dyn_base);
  if (plan.end - dyn_base > (uint32_t)smem_bytes || a.nt != NT) {  // unexpected reserved shared memory
    if (threadIdx.x == 0 && a.status) atomicOr(a.status, RQ_STATUS_TIMEOUT);
    return;
  }
  auto at = [&](uint32_t addr) { return smem + (addr - dyn_base); };
  uint32_t* lut_words = reinterpret_cast<uint32_t*>(at(plan.lut));
  int* page_ids = reinterpret_cast<int*>(at(plan.tail));
  uint64_t* mbar = reinterpret_cast<uint64_t*>(page_ids + kMaxSplitPages);
  float* cb = reinterpret_cast<float*>(mbar + kSlotsTotal / 2);
  Walk* walk = reinterpret_cast<Walk*>(cb + 16);
  float* const merge_lo = reinterpret_cast<float*>(at(plan.merge_lo));
  float* const merge_hi = reinterpret_cast<float*>(at(plan.merge_hi));

  // The small inputs that CTAs read once their partition is known -- block table, queries,
  // rotation parameters, a decode step's new tokens -- start filling L2 now, a line per thread
  // of the grid, so those reads hit L2 instead of queueing behind the first bulk copies.
  {  // line counts stay far below 2^32 (sizes are bounded at creation)
    const uint32_t line = threadIdx.x * gridDim.x + blockIdx.x;
    prefetch_line_l2(a.block_table, (uint32_t)(((size_t)a.B * a.max_pages * 4 + 127) / 128), line);
    if constexpr (!PRE) {
      const uint32_t rot_lines = (uint32_t)g.num_kv_heads * kHeadDim * 4 / 128;
      prefetch_line_l2(a.q, (uint32_t)(((size_t)a.B * a.T * g.num_q_heads * kHeadDim * 2) / 128), line);
      prefetch_line_l2(g.rot_k, rot_lines, line);
      prefetch_line_l2(g.rot_v, rot_lines, line);
    }
    if constexpr (STEP) {
      const uint32_t new_lines = (uint32_t)a.B * g.num_kv_heads * kHeadDim * 2 / 128;
      prefetch_line_l2(a.k_new, new_lines, line);
      prefetch_line_l2(a.v_new, new_lines, line);
    }
  }
  // The centroids' load is in flight with the lengths' below; the table is filled once the
  // first fragment's copies are issued, in their shadow.
  const float cb_val = threadIdx.x < (1 << BITS) ? g.centroids[threadIdx.x] : 0.f;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gq = lane >> 2, tq = lane & 3;
  const uint32_t key1 = lut::key<BITS>(plan.lut, lane, 0);
  const uint32_t key2 = lut::key<BITS>(plan.lut, lane, 1);
  const int P = g.page_size;
  const int tiles_per_page = P / 16;
  // Stage layout (see Ring): section by section when a pair always lies in one page.
  const bool by_section = (tiles_per_page & 1) == 0;
  // Offsets in a stage of tile A's (first) and tile B's K rows, V rows, K norms and V norms.
  const uint32_t st_kB = by_section ? 16u * R::VB : (uint32_t)R::SB;
  const uint32_t st_vA = by_section ? 32u * R::VB : 16u * R::VB;
  const uint32_t st_vB = by_section ? 48u * R::VB : (uint32_t)R::SB + 16u * R::VB;
  const uint32_t st_nA = by_section ? 64u * R::VB : 32u * R::VB;
  const uint32_t st_nB = by_section ? 64u * R::VB + 32u : (uint32_t)R::SB + 32u * R::VB;
  const uint32_t st_nv = by_section ? 64u : 32u;  // V norms after K norms
  // Shared address of this warp's stage st: slots 2st (first tile) and 2st + 1 (second tile,
  // SB bytes after the first: the slot plan keeps a warp's pairs of slots on one side of the table).
  const int sl0 = warp * kSlots;
  const uint32_t slot0 = sl0 < plan.n_lo ? dyn_base + (uint32_t)(sl0 * R::SB) : plan.hi + (uint32_t)((sl0 - plan.n_lo) * R::SB);
  const uint32_t slot2 = sl0 + 2 < plan.n_lo ? dyn_base + (uint32_t)((sl0 + 2) * R::SB)
                                             : plan.hi + (uint32_t)((sl0 + 2 - plan.n_lo) * R::SB);
  auto stage_slot = [&](int st) -> uint32_t {
    if constexpr (kStages == 2) {
      return st ? slot2 : slot0;
    } else {
      const int sl = sl0 + 2 * st;
      return sl < plan.n_lo ? dyn_base + (uint32_t)(sl * R::SB) : plan.hi + (uint32_t)((sl - plan.n_lo) * R::SB);
    }
  };
  const uint32_t mbar_addr = (uint32_t)__cvta_generic_to_shared(mbar + warp * kStages);
  if (lane == 0) {
    for (int st = 0; st < kStages; ++st) mbar_init(mbar_addr + 8 * st, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  uint32_t phase = 0;   // bit st: parity of the next completion of stage st
  bool broken = false;  // a staged copy never completed: stop using the ring

  // ---- this CTA's range [x, x_end) of cost in the stream-K partition ----
  // cum[b] = cost of all units of sequences < b (frag_at) and lens[b] = sequence b's clamped tokens,
  // built with a block scan at the start of the window: slots and table, unused before the
  // first fragment (at most 8001 x 8 + 8000 x 4 bytes; the table and the 64 slots span more).
  const int n_ug = (a.n_tiles_n + NT - 1) / NT;  // units per kv head
  const int upb = g.num_kv_heads * n_ug;          // units per sequence
  const int cap = a.max_pages * P;
  {
    long long* cum = reinterpret_cast<long long*>(smem);
    int* lens = reinterpret_cast<int*>(cum + a.B + 1);
    long long* wsum = reinterpret_cast<long long*>(page_ids);  // [kWarps] scan scratch
    int* wunits = page_ids + 2 * kWarps;                       // [kWarps]: units with tokens
    int* wmax = wunits + kWarps;                                // [kWarps]: largest unit (rounds)
    long long total = 0;
    int n_units = 0, max_rounds = 0;
    for (int c0 = 0; c0 < a.B; c0 += kThreads) {
      const int bb = c0 + threadIdx.x;
      long long v = 0;
      if (bb < a.B) {
        int len = a.seq_lens[bb];
        if (len < 0 || len > cap || (len > 0 && len < a.T)) {
          if (blockIdx.x == 0 && a.status) atomicOr(a.status, RQ_STATUS_BAD_LEN);
          len = len < 0 ? 0 : (len > cap ? cap : len);
        }
        v = len > 0 ? (long long)(unit_rounds<NT>(len) + Shape<NT>::kFragmentRounds) * upb : 0;
        lens[bb] = len;
      }
      int nu = v > 0 ? upb : 0, mr = v > 0 ? (int)(v / upb) - Shape<NT>::kFragmentRounds : 0;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        nu += __shfl_xor_sync(0xffffffffu, nu, o);
        mr = max(mr, __shfl_xor_sync(0xffffffffu, mr, o));
      }
      if (lane == 0) {
        wunits[warp] = nu;
        wmax[warp] = mr;
      }
      long long inc = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const long long n = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += n;
      }
      if (lane == 31) wsum[warp] = inc;
      __syncthreads();
      if (warp == 0) {
        long long w = lane < kWarps ? wsum[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const long long n = __shfl_up_sync(0xffffffffu, w, o);
          if (lane >= o) w += n;
        }
        if (lane < kWarps) wsum[lane] = w;
      }
      __syncthreads();
      if (bb < a.B) cum[bb + 1] = total + (warp > 0 ? wsum[warp - 1] : 0) + inc;
      total += wsum[kWarps - 1];
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        n_units += wunits[w];
        max_rounds = max(max_rounds, wmax[w]);
      }
      __syncthreads();
    }
    if (threadIdx.x == 0) cum[0] = 0;
    __syncthreads();
    long long x0, x1;
    if (total * gridDim.x < (1LL << 32))
      partition<uint32_t>((uint32_t)total, n_units, max_rounds, gridDim.x, blockIdx.x, Shape<NT>::kFragmentRounds,
                          x0, x1);
    else
      partition<long long>(total, n_units, max_rounds, gridDim.x, blockIdx.x, Shape<NT>::kFragmentRounds, x0, x1);
    int lo = 0, hi = a.B;  // the last sequence b with cum[b] <= x0, which skips empty ones
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (cum[mid] <= x0) lo = mid;
      else hi = mid;
    }
    if (threadIdx.x == 0) *walk = Walk{x0, x1, cum[lo], lo, a.B > 0 ? lens[lo] : 0};
    {  // a sequence without tokens has no fragments: its rows are zeros
      for (int bb = blockIdx.x; bb < a.B; bb += gridDim.x) {
        if (cum[bb + 1] != cum[bb]) continue;
        const int n16 = a.T * g.num_q_heads * (kHeadDim / 8);
        uint4* o16 = reinterpret_cast<uint4*>(reinterpret_cast<__half*>(a.out) + (size_t)bb * a.T * g.num_q_heads * kHeadDim);
        for (int i = threadIdx.x; i < n16; i += kThreads) o16[i] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    if (threadIdx.x < (1 << BITS)) cb[threadIdx.x] = cb_val;
    __syncthreads();  // the scratch is slot and table space from here on
  }

  // Every fragment advances the walk by at least one unit of cost, so this bound (the range's
  // cost) is never reached; it only guarantees that the loop ends.
  const long long max_fragments = walk->x_end - walk->x;
  for (long long n_frag = 0; n_frag < max_fragments; ++n_frag) {
    if (walk->x >= walk->x_end) break;
    const int len = walk->len;
    const Frag fr = frag_at<NT>(*walk);
    if (fr.r1 <= fr.r0) break;  // the range ends inside a unit's opening cost: nothing left
    const int t1 = fr.t1;
    struct {
      int b, h, nt0;
    } it = {walk->b, fr.uib / n_ug, (fr.uib % n_ug) * NT};

    // q~ = R_k q * sm_scale * log2(e) for query column gq of each of the unit's n-tiles, the
    // lane's 32 dims, formed once the fragment's first copies are in flight (below).
    uint32_t qf[NT][8][2];
    int last_pos[NT][2];  // last position wholly visible to query columns 2tq, 2tq+1 of each n-tile

    float m_run[NT][2], l_run[NT][2];  // m_run: -inf before the column's first visible score
    float o[NT][8][4];
#pragma unroll
    for (int i = 0; i < NT; ++i) {
      m_run[i][0] = m_run[i][1] = -CUDART_INF_F;
      l_run[i][0] = l_run[i][1] = 0.f;
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) o[i][mt][0] = o[i][mt][1] = o[i][mt][2] = o[i][mt][3] = 0.f;
    }

    // The fragment in chunks of at most kMaxSplitPages pages (one chunk unless a CTA's range
    // is very long); the warps' states carry over from chunk to chunk.
    for (int tile0 = fr.t0; tile0 < t1;) {
    const int p0 = tile0 / tiles_per_page;
    const int tile1 = min(t1, (p0 + kMaxSplitPages) * tiles_per_page);
    const int p1 = (tile1 + tiles_per_page - 1) / tiles_per_page;
    __syncthreads();  // every warp is done with the previous chunk's page ids
    for (int i = threadIdx.x; i < p1 - p0; i += kThreads) {  // stage them, clamped into the pool
      int pg = a.block_table[(size_t)it.b * a.max_pages + p0 + i];
      if (pg < 0 || pg >= g.num_pages) {
        if (a.status) atomicOr(a.status, RQ_STATUS_BAD_PAGE);
        pg = 0;
      }
      page_ids[i] = pg;
    }
    __syncthreads();

    // The chunk's tiles, taken two at a time: pair q = tiles tile0 + 2q and tile0 + 2q + 1
    // (the second exists unless the chunk ends there); warp w takes pairs w + kWarps k.
    const int n_pairs = (tile1 - tile0 + 1) / 2;
    // A pair whose second tile lies past the chunk reads a stale slot for it: its positions,
    // all past pos_lim, are masked like positions past the sequence.
    const int pos_lim = tile1 * 16 - 1;
    const int n_w = (warp < n_pairs && !broken) ? (n_pairs - 1 - warp) / kWarps + 1 : 0;
    // The warp's k-th pair is tiles tA = tA0 + 2 kWarps k and tA + 1 (if it exists); all lanes
    // take part and one elected lane announces the stage's bytes and issues its bulk copies from
    // warp-uniform addresses.  A 16-token page is one copy per tile; a pair inside one page
    // (section by section) is four, one per run; other pairs are four per tile.  When the tiles
    // per page divide 2 kWarps (every power-of-two page size) the pair's position in its page is
    // the same for every k and its page-id entry moves by 2 kWarps / tiles_per_page per pair.
    const int tA0 = tile0 + 2 * warp;
    const bool cp_regular = (2 * kWarps) % tiles_per_page == 0;
    const int cp_step = cp_regular ? 2 * kWarps / tiles_per_page : 0;
    const int cp_pid0 = tA0 / tiles_per_page - p0;                  // page-id entry of pair 0
    const int cp_off0 = (tA0 - (cp_pid0 + p0) * tiles_per_page) * 16;  // its first token in the page
    // chunk (page, kv head) at page * Hkv * page_bytes + h * page_bytes: both products stay
    // below 2^31 per page (checked at creation), so a 32 x 32 -> 64-bit multiply-add forms it
    const uint32_t page_stride = (uint32_t)(g.num_kv_heads * g.page_bytes);
    const uint8_t* const head_base = a.pages + (size_t)it.h * g.page_bytes;
    auto chunk_of = [&](int pid) {  // the chunk of page-id entry pid (the same in every lane)
      const uint32_t page = (uint32_t)__shfl_sync(0xffffffffu, page_ids[pid], 0);
      return head_base + (uint64_t)page * page_stride;
    };
    auto issue = [&](int k) {
      const int st = k % kStages;
      const int tA = tA0 + 2 * kWarps * k;
      const bool two = tA + 1 < tile1;  // the pair's second tile exists
      const uint32_t mb = mbar_addr + 8 * st;
      const uint32_t dst = stage_slot(st);
      int pid = cp_pid0 + cp_step * k, off = cp_off0;
      if (!cp_regular) {
        const int pq = tA / tiles_per_page;
        pid = pq - p0;
        off = (tA - pq * tiles_per_page) * 16;
      }
      if (P == 16) {
        const uint8_t* cA = chunk_of(pid);
        const uint8_t* cB = chunk_of(two ? pid + 1 : pid);
        if (elect_one()) {
          mbar_expect_tx(mb, two ? 2 * R::SB : R::SB);
          bulk_g2s(dst, cA, R::SB, mb);
          if (two) bulk_g2s(dst + R::SB, cB, R::SB, mb);
        }
      } else if (by_section) {
        const uint8_t* c = chunk_of(pid);
        const uint32_t n = two ? 32u : 16u;
        if (elect_one()) {
          mbar_expect_tx(mb, two ? 2 * R::SB : R::SB);
          bulk_g2s(dst, c + off * R::VB, n * R::VB, mb);
          bulk_g2s(dst + 32u * R::VB, c + (P + off) * R::VB, n * R::VB, mb);
          bulk_g2s(dst + 64u * R::VB, c + 2 * P * R::VB + 2 * off, 2 * n, mb);
          bulk_g2s(dst + 64u * R::VB + 64u, c + 2 * P * R::VB + 2 * P + 2 * off, 2 * n, mb);
        }
      } else {  // an odd number of tiles per page: tile by tile, the second maybe in the next page
        const bool next = off + 16 == P;  // tile A ends its page
        const uint8_t* cA = chunk_of(pid);
        const uint8_t* cB = chunk_of(two && next ? pid + 1 : pid);
        const int offB = next ? 0 : off + 16;
        if (elect_one()) {
          mbar_expect_tx(mb, two ? 2 * R::SB : R::SB);
#pragma unroll 1
          for (int t = 0; t < (two ? 2 : 1); ++t) {
            const uint8_t* c = t ? cB : cA;
            const int o = t ? offB : off;
            const uint32_t d = dst + (t ? (uint32_t)R::SB : 0u);
            bulk_g2s(d, c + o * R::VB, 16u * R::VB, mb);
            bulk_g2s(d + 16u * R::VB, c + (P + o) * R::VB, 16u * R::VB, mb);
            bulk_g2s(d + 32u * R::VB, c + 2 * P * R::VB + 2 * o, 32u, mb);
            bulk_g2s(d + 32u * R::VB + 32u, c + 2 * P * R::VB + 2 * P + 2 * o, 32u, mb);
          }
        }
      }
    };
    // A decode step's token lies in the unit's last tile, which ends the chunk's last pair when
    // the chunk ends the unit: the warp that stages that pair (its last) writes the token first,
    // deferring the pair's copy when it is one of the first stages.
    const bool appends = STEP && tile1 == fr.tb && warp == (n_pairs - 1) % kWarps;
    const int n_first = min(kStages, n_w) - (appends && n_w <= kStages ? 1 : 0);
    if (n_first > 0) {
      fence_proxy_async();
      for (int k = 0; k < n_first; ++k) issue(k);
    }
    const bool first_chunk = n_frag == 0 && tile0 == fr.t0;  // uniform over the CTA
    if (first_chunk) lut::fill<BITS>(lut_words, cb, threadIdx.x, kThreads);
    if constexpr (STEP) {
      if (appends) {
        append_token<BITS>(g, a, it.b, it.h, len);
        if (n_w > 0 && n_w <= kStages) {
          fence_proxy_async();
          issue(n_w - 1);
        }
      }
    }
    if (tile0 == fr.t0) {  // the fragment's first chunk: its copies overlap the query's loads
      // k-slot order of the K operand: dims (4kc, 4kc+1 | 4kc+2, 4kc+3) of the lane's 32, or
      // (4kc, 4kc+2 | 4kc+1, 4kc+3) for 2-bit codes
      constexpr int s1 = BITS == 2 ? 2 : 1, s2 = BITS == 2 ? 1 : 2;
#pragma unroll
      for (int i = 0; i < NT; ++i) {
        float y[32];
        // query row of the kv head: draft j = row / group, head row % group
        rotated_query<PRE>(y, g, a, it.b, it.h, (it.nt0 + i) * 8 + gq, tq);
#pragma unroll
        for (int kc = 0; kc < 8; ++kc) {
          qf[i][kc][0] = pack_half2(y[4 * kc] * g.q_scale, y[4 * kc + s1] * g.q_scale);
          qf[i][kc][1] = pack_half2(y[4 * kc + s2] * g.q_scale, y[4 * kc + 3] * g.q_scale);
        }
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int rc = (it.nt0 + i) * 8 + 2 * tq + c;
          const int j = rc < a.rows ? rc / g.group : a.T - 1;
          // chain: row j sees positions <= len - T + j; tree: the prefix for sure (the drafts
          // by their mask bit), so only the prefix counts as wholly visible
          last_pos[i][c] = a.tree_mask ? len - a.T - 1 : len - a.T + j;
        }
      }
    }
    if (first_chunk) __syncthreads();  // the table is complete
    int consumed = 0;
    for (int k = 0; k < n_w; ++k) {
      const int st = k % kStages;
      const bool ok = mbar_wait_bounded(mbar_addr + 8 * st, (phase >> st) & 1u);
      if (!__all_sync(0xffffffffu, ok)) {
        broken = true;
        break;
      }
      phase ^= 1u << st;
      consumed = k + 1;
      const uint8_t* const sp = at(stage_slot(st));
      const int pos0 = (tile0 + 2 * (warp + k * kWarps)) * 16;  // first token of the pair

      // ---- shifted scores t = s - m_use (base 2) of the lane's four K rows (two per tile) for
      // columns 2tq, 2tq+1 of each n-tile, one FMA each from the dot product and the key norm.
      // The running max moves lazily: only when some t exceeds kLazyMargin (or the pair holds
      // a value norm that could overflow the fp16 P' = p * n_v, or the column has no max yet)
      // does the warp reduce the pair's exact max, rescale and re-shift; otherwise
      // p = 2^t <= 2^kLazyMargin and nothing is reduced or rescaled.
      // m_use: the max the exponents are taken against (m_run, or 0 while m_run is -inf); thr:
      // the t above which the pair takes the exact path (kLazyMargin, or -inf before a max).
      float m_use[NT][2], thr[NT][2];
#pragma unroll
      for (int i = 0; i < NT; ++i)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const bool none = m_run[i][c] == -CUDART_INF_F;
          m_use[i][c] = none ? 0.f : m_run[i][c];
          thr[i][c] = none ? -CUDART_INF_F : kLazyMargin;
        }
      float sc[NT][8];  // [n-tile][tile][row][col]: t, then p
      uint32_t nv_bits[2];
      {
        Raw<BITS> rk;
        float s[NT][4];
        load_stage<BITS>(rk, sp, sp + st_vA, sp + st_nA, sp + st_nA + st_nv, gq, tq);
        qk_tile<BITS, NT>(s, rk, qf, key1, key2);
        nv_bits[0] = rk.nv;
        const float nk0 = half_bits_to_float(rk.nk & 0xffffu), nk1 = half_bits_to_float(rk.nk >> 16);
#pragma unroll
        for (int i = 0; i < NT; ++i) {
          sc[i][0] = fmaf(s[i][0], nk0, -m_use[i][0]);
          sc[i][1] = fmaf(s[i][1], nk0, -m_use[i][1]);
          sc[i][2] = fmaf(s[i][2], nk1, -m_use[i][0]);
          sc[i][3] = fmaf(s[i][3], nk1, -m_use[i][1]);
        }
        load_stage<BITS>(rk, sp + st_kB, sp + st_vB, sp + st_nB, sp + st_nB + st_nv, gq, tq);
        qk_tile<BITS, NT>(s, rk, qf, key1, key2);
        nv_bits[1] = rk.nv;
        const float nk2 = half_bits_to_float(rk.nk & 0xffffu), nk3 = half_bits_to_float(rk.nk >> 16);
#pragma unroll
        for (int i = 0; i < NT; ++i) {
          sc[i][4] = fmaf(s[i][0], nk2, -m_use[i][0]);
          sc[i][5] = fmaf(s[i][1], nk2, -m_use[i][1]);
          sc[i][6] = fmaf(s[i][2], nk3, -m_use[i][0]);
          sc[i][7] = fmaf(s[i][3], nk3, -m_use[i][1]);
        }
      }
      // Pairs wholly inside every column's visible range skip the per-element mask.
      int vis_min = pos_lim;
#pragma unroll
      for (int i = 0; i < NT; ++i) vis_min = min(vis_min, min(last_pos[i][0], last_pos[i][1]));
      const bool interior = __all_sync(0xffffffffu, pos0 + 31 <= vis_min);
      if (!interior) {
#pragma unroll
        for (int i = 0; i < NT; ++i) {
          const int draft0 = last_pos[i][0] + 1;  // tree: the first draft follows the prefix
          uint64_t draft_mask[2] = {0ull, 0ull};  // tree: the columns' draft visibility bits (re-read here,
          if (a.tree_mask) {                      // not held in registers through the loop)
#pragma unroll
            for (int c = 0; c < 2; ++c) {
              const int rc = (it.nt0 + i) * 8 + 2 * tq + c;
              draft_mask[c] = a.tree_mask[(size_t)it.b * a.T + (rc < a.rows ? rc / g.group : a.T - 1)];
            }
          }
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int pos = pos0 + 16 * (e >> 2) + rho<BITS>(gq) + 8 * ((e >> 1) & 1);
            bool vis;
            if (a.tree_mask) {
              const int d = pos - draft0;
              vis = d < 0 || (d < a.T && ((draft_mask[e & 1] >> d) & 1ull));
            } else {
              vis = pos <= last_pos[i][e & 1];
            }
            if (!vis || pos > pos_lim) sc[i][e] = -CUDART_INF_F;
          }
        }
      }
      float cmax[NT][2];
      bool grow = false;
#pragma unroll
      for (int i = 0; i < NT; ++i) {
        cmax[i][0] = fmaxf(fmaxf(sc[i][0], sc[i][2]), fmaxf(sc[i][4], sc[i][6]));
        cmax[i][1] = fmaxf(fmaxf(sc[i][1], sc[i][3]), fmaxf(sc[i][5], sc[i][7]));
        grow = grow || cmax[i][0] > thr[i][0] || cmax[i][1] > thr[i][1];
      }
      // fp16 norms at or above 2^8 (bits >= 0x5C00; norms are >= 0, so a half has no sign bit
      // and adding 0x2400 to it carries into its bit 15 exactly then) take the exact path,
      // where p <= 1
      const bool nv_big = (((nv_bits[0] + 0x24002400u) | (nv_bits[1] + 0x24002400u)) & 0x80008000u) != 0u;
      if (__any_sync(0xffffffffu, grow || nv_big)) {
        float alpha[NT][2], shift[NT][2];
        bool moved = false;
#pragma unroll
        for (int i = 0; i < NT; ++i) {
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            float tmax = cmax[i][c];
            tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 4));
            tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 8));
            tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 16));
            // (a column with no visible score yet keeps m_run = -inf and m_use = 0: its masked
            // scores must give p = 2^(-inf) = 0)
            const float m_new = fmaxf(m_run[i][c], tmax + m_use[i][c]);
            const float mu = m_new == -CUDART_INF_F ? 0.f : m_new;
            alpha[i][c] = ex2(m_run[i][c] - mu);  // 0 when there was no max yet
            shift[i][c] = m_use[i][c] - mu;
            l_run[i][c] *= alpha[i][c];
            m_run[i][c] = m_new;
            moved = moved || alpha[i][c] != 1.f;
          }
#pragma unroll
          for (int e = 0; e < 8; ++e) sc[i][e] += shift[i][e & 1];
        }
        if (__any_sync(0xffffffffu, moved)) {
#pragma unroll
          for (int i = 0; i < NT; ++i)
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
              o[i][mt][0] *= alpha[i][0];
              o[i][mt][2] *= alpha[i][0];
              o[i][mt][1] *= alpha[i][1];
              o[i][mt][3] *= alpha[i][1];
            }
        }
      }
      // P' = p * n_v, zero for masked tokens whatever their stored norm; to the B layout.
      uint32_t pb[2][NT][2];  // [tile][n-tile]
#pragma unroll
      for (int i = 0; i < NT; ++i) {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          sc[i][e] = ex2(sc[i][e]);  // now p; masked entries give 0
          l_run[i][e & 1] += sc[i][e];
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const float nva = half_bits_to_float(nv_bits[h] & 0xffffu), nvb = half_bits_to_float(nv_bits[h] >> 16);
          float q0 = sc[i][4 * h + 0] * nva, q1 = sc[i][4 * h + 1] * nva;
          float q2 = sc[i][4 * h + 2] * nvb, q3 = sc[i][4 * h + 3] * nvb;
          if (!interior) {
            q0 = sc[i][4 * h + 0] == 0.f ? 0.f : q0;
            q1 = sc[i][4 * h + 1] == 0.f ? 0.f : q1;
            q2 = sc[i][4 * h + 2] == 0.f ? 0.f : q2;
            q3 = sc[i][4 * h + 3] == 0.f ? 0.f : q3;
          }
          pb[h][i][0] = movmatrix_t(pack_half2(q0, q1));
          pb[h][i][1] = movmatrix_t(pack_half2(q2, q3));
        }
      }
      // ---- values: read both tiles' V codes, hand the stage back, accumulate
      Raw<BITS> rvA, rvB;
      load_stage<BITS>(rvA, sp, sp + st_vA, sp + st_nA, sp + st_nA + st_nv, gq, tq);
      load_stage<BITS>(rvB, sp + st_kB, sp + st_vB, sp + st_nB, sp + st_nB + st_nv, gq, tq);
      __syncwarp();
      if (k + kStages < n_w) {  // refill this stage while the pair is accumulated
        fence_proxy_async();
        issue(k + kStages);
      }
      pv_tile<BITS, NT>(o, rvA, pb[0], key1, key2, gq);
      pv_tile<BITS, NT>(o, rvB, pb[1], key1, key2, gq);
    }
    if (broken) {
      // A copy never landed: flag it, wait (bounded) for the copies still in flight so none
      // lands in a reused buffer, and leave the ring alone from now on.
      if (lane == 0 && a.status) atomicOr(a.status, RQ_STATUS_TIMEOUT);
      for (int k = consumed; k < min(n_w, consumed + kStages); ++k)
        mbar_wait_bounded(mbar_addr + 8 * (k % kStages), (phase >> (k % kStages)) & 1u);
    }
    tile0 = tile1;
    }

    // ---- merge the warps' partial states of this fragment, one n-tile at a time ----
    // Warp w's O goes to row (w, mt & 3) of merge half mt / 4 as one float4 per lane: rows of
    // 132 floats, so the writes are contiguous and the column-wise reads hit distinct bank
    // groups.  m and l go to the page-id array, free until the next fragment.  Fragment
    // partials of unit u sit at slots u + c for its CTAs c (8 NT rows each): slots never
    // collide, because both the units and the CTAs' ranges follow the same order.  A fragment
    // that is its unit's whole range finishes the unit right here (a dense rotation through
    // the normalised rows staged in obuf and dense_finish_rows).
    const int unit = (it.b * g.num_kv_heads + it.h) * n_ug + it.nt0 / NT;
    const Frag f = frag_at<NT>(*walk);
    const bool whole = f.t0 == 0 && f.t1 == f.tb;  // uniform over the CTA
    float (*const obuf)[kHeadDim] = reinterpret_cast<float (*)[kHeadDim]>(at(plan.obuf));
    float* dst = a.ws + (size_t)(unit + blockIdx.x) * (8 * NT) * kPartialStride;
    if (threadIdx.x == 0 && !whole) {
      if (f.t0 == 0) a.frag[2 * unit] = blockIdx.x;         // the unit's first CTA
      if (f.t1 == f.tb) a.frag[2 * unit + 1] = blockIdx.x;  // and its last
    }
    float* const ml = reinterpret_cast<float*>(page_ids);  // [warp][column][m, l]
#pragma unroll
    for (int i = 0; i < NT; ++i) {
      __syncthreads();  // every warp is done with its slots (or the previous n-tile's merge)
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        float l = l_run[i][c];
        l += __shfl_xor_sync(0xffffffffu, l, 4);
        l += __shfl_xor_sync(0xffffffffu, l, 8);
        l += __shfl_xor_sync(0xffffffffu, l, 16);
        l_run[i][c] = l;
      }
      if (gq == 0) {
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          ml[(warp * 8 + 2 * tq + c) * 2] = m_run[i][c];
          ml[(warp * 8 + 2 * tq + c) * 2 + 1] = l_run[i][c];
        }
      }
#pragma unroll
      for (int mt = 0; mt < 8; ++mt)
        reinterpret_cast<float4*>((mt < 4 ? merge_lo : merge_hi) + (warp * 4 + (mt & 3)) * kPartialStride)[lane] =
            make_float4(o[i][mt][0], o[i][mt][1], o[i][mt][2], o[i][mt][3]);
      __syncthreads();
      const int nt = it.nt0 + i;
      const int cols = min(8, a.rows - nt * 8);
      // thread (c, gq', mt') merges dims 16 gq' + 2 mt' and +1 of column c: lane 4 gq' + c / 2
      // of every warp held them, as components (c & 1) and (c & 1) + 2 of its float4 mt'
#pragma unroll
      for (int idx0 = 0; idx0 < 512; idx0 += kThreads) {
        const int idx = idx0 + threadIdx.x;
        const int c = idx >> 6, gm = (idx >> 3) & 7, mm = idx & 7;
        // a whole unit's R_v entries, loaded while the partials are summed
        const float4 rv = (!PRE && whole && c < cols) ? rot_v_block(g, it.h, 16 * gm + 2 * mm)
                                                      : make_float4(0.f, 0.f, 0.f, 0.f);
        if (c < cols) {  // c is uniform over each warp
          float M = -CUDART_INF_F;
#pragma unroll 4
          for (int w = 0; w < kWarps; ++w) M = fmaxf(M, ml[(w * 8 + c) * 2]);
          float acc0 = 0.f, acc1 = 0.f, lsum = 0.f;
          if (M != -CUDART_INF_F) {
            const float* half_base = (mm < 4 ? merge_lo : merge_hi) + (mm & 3) * kPartialStride + 4 * (4 * gm + (c >> 1));
#pragma unroll 4
            for (int w = 0; w < kWarps; ++w) {
              const float scale = exp2f(ml[(w * 8 + c) * 2] - M);
              const float4 v = *reinterpret_cast<const float4*>(half_base + w * 4 * kPartialStride);
              acc0 += ((c & 1) ? v.y : v.x) * scale;
              acc1 += ((c & 1) ? v.w : v.z) * scale;
              lsum += ml[(w * 8 + c) * 2 + 1] * scale;
            }
          }
          if (whole) {
            const float inv = (lsum > 0.f && len >= a.T) ? g.out_scale / lsum : 0.f;
            if constexpr (PRE) {
              *reinterpret_cast<float2*>(&obuf[c][16 * gm + 2 * mm]) = make_float2(acc0 * inv, acc1 * inv);
            } else {
              store_pair(g, a, it.b, it.h, nt * 8 + c, 16 * gm + 2 * mm, acc0 * inv, acc1 * inv, rv);
            }
          } else {
            float* drow = dst + (i * 8 + c) * kPartialStride;
            *reinterpret_cast<float2*>(drow + 4 + 16 * gm + 2 * mm) = make_float2(acc0, acc1);
            if (gm == 0 && mm == 0) {
              drow[0] = M;
              drow[1] = lsum;
            }
          }
        }
      }
      if (PRE && whole) {  // uniform over the CTA
        __syncthreads();
        dense_finish_rows<kThreads>(g, a, it.b, it.h, nt * 8, cols, obuf);
      }
    }
    if (!whole) {
      // Publish the partial and count the unit's finished rounds: the barrier orders every
      // thread's partial before thread 0's fence and add.  The CTA whose rounds complete the
      // unit merges all its partials once its own range is done (no CTA waits for another)
      // and puts the counter back to zero for the next launch.
      __syncthreads();
      if (threadIdx.x == 0) {
        const int n = f.r1 - f.r0;
        __threadfence();
        if (atomicAdd(a.cnt + unit, n) + n >= f.rb) {
          a.cnt[unit] = 0;
          if (walk->n_fin < 2) walk->fin[walk->n_fin++] = unit;
          else if (a.status) atomicOr(a.status, RQ_STATUS_TIMEOUT);  // cannot happen (see Walk)
        }
      }
    }
    __syncthreads();  // the merge buffer reuses slot space
    if (threadIdx.x == 0) {
      Walk w = *walk;
      walk_advance<NT>(w, frag_at<NT>(w), upb, a, cap);
      *walk = w;
    }
    __syncthreads();
  }

  // Finish the units this CTA completed: a warp per query row of the unit (a dense rotation:
  // 8 rows at a time, staged in obuf for dense_finish_rows).
  if (threadIdx.x == 0 && walk->n_fin > 0) __threadfence();  // after the adds that saw them done
  __syncthreads();
  for (int k = 0; k < walk->n_fin; ++k) {
    const int unit = walk->fin[k];
    const int ug = unit % n_ug, h = (unit / n_ug) % g.num_kv_heads, b = unit / (n_ug * g.num_kv_heads);
    const int row0 = ug * 8 * NT, nrows = min(8 * NT, a.rows - row0);
    if constexpr (PRE) {
      float (*const obuf)[kHeadDim] = reinterpret_cast<float (*)[kHeadDim]>(at(plan.obuf));
      for (int r0 = 0; r0 < nrows; r0 += 8) {  // uniform over the CTA
        if (warp < min(8, nrows - r0)) {
          const float4 v = merge_splits(g, a, b, h, row0 + r0 + warp, lane);
          *reinterpret_cast<float4*>(&obuf[warp][4 * lane]) = v;
        }
        __syncthreads();
        dense_finish_rows<kThreads>(g, a, b, h, row0 + r0, min(8, nrows - r0), obuf);
        __syncthreads();
      }
    } else {
      const float4 rv = rot_v_block(g, h, 4 * lane);
      for (int r = warp; r < nrows; r += kWarps)
        store_row(g, a, b, h, row0 + r, lane, merge_splits(g, a, b, h, row0 + r, lane), rv);
    }
  }
}

// ---------------------------------------------------------------------------------------
// Dense rotation (TurboQuant): the queries' end of the call.  The query rows of one kv head --
// over every sequence and query token -- are numbered r = (b * T + j) * group + k, in groups of
// 16.  A warp forms y = R_k q for 16 rows and 32 output dims on the tensor cores: the fp16
// query times R_k's fp16 hi and lo halves (R_k = hi + lo to about 2^-22), both products into
// one fp32 accumulator (g.rotq holds the halves in the MMA's fragment order).  A decode step's
// new tokens take the fp32 path of the append instead (thread i owns output dim i: per step of
// the sum it reads four entries of the staged matrix and the 16 rows' four inputs as float4
// broadcasts from shared memory), whose decisions the stored codes must repeat.
// ---------------------------------------------------------------------------------------
constexpr int kDenseRows = 16;
constexpr int kRotqWords = 8 * 16 * 32 * 4;  // a kv head's fragments: [k-step][n-tile][lane][4] u32

constexpr int kDenseSmem = kHeadDim * kHeadDim * 4;  // the 128 x 128 fp32 matrix, staged

// Stages the 64 KB matrix w into shared memory ws: every thread's 32 16-byte copies are in
// flight at once (one memory round trip instead of one per step of the sum).
__device__ __forceinline__ void stage_matrix(float* ws, const float* __restrict__ w) {
  const uint32_t dst = (uint32_t)__cvta_generic_to_shared(ws);
  for (int c = threadIdx.x; c < kHeadDim * kHeadDim / 4; c += blockDim.x)
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst + 16 * c), "l"(w + 4 * c) : "memory");
  asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;" ::: "memory");
}

// out[r][i] = sum_m ws[m * 128 + i] * xs[r][m] for 16 rows (the calling thread's dim i).
template <int N>
__device__ __forceinline__ void dense_rows(float (&acc)[N], const float* ws, const float (*xs)[kHeadDim], int i) {
#pragma unroll
  for (int r = 0; r < N; ++r) acc[r] = 0.f;
#pragma unroll 2
  for (int m = 0; m < kHeadDim; m += 4) {
    const float w0 = ws[(m + 0) * kHeadDim + i], w1 = ws[(m + 1) * kHeadDim + i];
    const float w2 = ws[(m + 2) * kHeadDim + i], w3 = ws[(m + 3) * kHeadDim + i];
#pragma unroll
    for (int r = 0; r < N; ++r) {
      const float4 x = *reinterpret_cast<const float4*>(&xs[r][m]);
      acc[r] = fmaf(w0, x.x, fmaf(w1, x.y, fmaf(w2, x.z, fmaf(w3, x.w, acc[r]))));
    }
  }
}

// Query row r of kv head h -> its index in the [B][T][Hq] query / output arrays.
__device__ __forceinline__ size_t dense_row_index(const Geometry& g, int h, int r) {
  const int bj = r / g.group, k = r % g.group;
  return (size_t)bj * g.num_q_heads + h * g.group + k;
}

// y[16 rows][32 dims] = q R_k^T for rows r0 .. r0 + 15 of kv head h (rows >= rows read as zero and
// are not stored) and output dims 32 ds .. 32 ds + 31: four n-tiles, eight k-steps, two MMAs
// (hi, lo) each.  The MMA's k-slots of lane t (2t, 2t+1 | 2t+8, 2t+9) carry input dims 32t + 4ks
// + (0, 1 | 2, 3), an order g.rotq's words follow too, so each lane reads its row's inputs as
// 8-byte pieces of one 64-byte span.  frag: the head's fragments in shared memory.
__device__ __forceinline__ void rotate_rows_tc(const Geometry& g, const AttnArgs& a, const uint4* frag, int h,
                                               int r0, int rows, int ds, int lane) {
  const int gq = lane >> 2, tq = lane & 3;
  const __half* q = reinterpret_cast<const __half*>(a.q);
  const int ra = r0 + gq, rb = r0 + gq + 8;
  const uint2* pa = ra < rows ? reinterpret_cast<const uint2*>(q + dense_row_index(g, h, ra) * kHeadDim + 32 * tq) : nullptr;
  const uint2* pb = rb < rows ? reinterpret_cast<const uint2*>(q + dense_row_index(g, h, rb) * kHeadDim + 32 * tq) : nullptr;
  float acc[4][4];
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    const uint2 xa = pa ? pa[ks] : make_uint2(0u, 0u), xb = pb ? pb[ks] : make_uint2(0u, 0u);
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      const uint4 w = frag[(ks * 16 + 4 * ds + nt) * 32 + lane];  // hi b0, hi b1, lo b0, lo b1
      if (ks == 0)
        mma16816_z(acc[nt], xa.x, xb.x, xa.y, xb.y, w.x, w.y);
      else
        mma16816(acc[nt], xa.x, xb.x, xa.y, xb.y, w.x, w.y);
      mma16816(acc[nt], xa.x, xb.x, xa.y, xb.y, w.z, w.w);
    }
  }
#pragma unroll
  for (int nt = 0; nt < 4; ++nt) {
    const int col = 32 * ds + 8 * nt + 2 * tq;
    if (pa) *reinterpret_cast<float2*>(a.q_rot + dense_row_index(g, h, ra) * kHeadDim + col) = make_float2(acc[nt][0], acc[nt][1]);
    if (pb) *reinterpret_cast<float2*>(a.q_rot + dense_row_index(g, h, rb) * kHeadDim + col) = make_float2(acc[nt][2], acc[nt][3]);
  }
}

// The dense rotation's work before the split-K kernel, one launch of 512-thread CTAs:
//   * CTAs [0, q_ctas): q_rot[b][j][head] = R_k q[b][j][head] (fp32, unscaled).  Each kv head's
//     rows, in groups of 64, are shared out over q_ctas / Hkv CTAs, which stage the head's
//     fragments (64 KB) once; warp w takes rows 16 (w / 4) .. + 15 and dims 32 (w % 4) .. + 31
//     of each group (rotate_rows_tc).
//   * a decode step (a.k_new) adds 2 Hkv ceil(B / 16) CTAs, each coding 16 sequences' newest K
//     (R_k) or V (R_v) vector of one kv head and writing it at position seq_lens[b] - 1: R
//     staged transposed, four 128-thread slices forming y = R x for 4 vectors each (thread i
//     owns output dim i), then a half-warp per vector codes it.  The fp32 R x of dense_rows
//     decides every code farther than kFixBand from a boundary and the compensated dot product
//     the others -- the decisions rq_quantize_append makes, so the two write the same bytes.
constexpr int kDenseSlices = 4;
constexpr int kDenseThreads = kDenseSlices * kHeadDim;
template <int BITS>
__global__ void __launch_bounds__(kDenseThreads, 2)
dense_prologue_kernel(const Geometry g, const AttnArgs a, int q_ctas) {
  __shared__ __align__(16) float qs[kDenseSlices][kDenseRows][kHeadDim];
  extern __shared__ __align__(16) float wsm[];
  const int hkv = g.num_kv_heads;
  const int slice = threadIdx.x / kHeadDim, i = threadIdx.x % kHeadDim;
  if ((int)blockIdx.x < q_ctas) {
    const int h = blockIdx.x % hkv, per_head = q_ctas / hkv;
    stage_matrix(wsm, reinterpret_cast<const float*>(g.rotq) + (size_t)h * kRotqWords);  // 64 KB either way
    __syncthreads();
    const uint4* frag = reinterpret_cast<const uint4*>(wsm);
    const int rows = a.B * a.T * g.group;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int r0 = (blockIdx.x / hkv) * 64; r0 < rows; r0 += per_head * 64)
      rotate_rows_tc(g, a, frag, h, r0 + 16 * (warp >> 2), rows, warp & 3, lane);
    return;
  }
  // ---- the decode step's new tokens (every thread stages and reaches the barriers) ----
  const int c = blockIdx.x - q_ctas;
  const int h = c % hkv, kind = (c / hkv) & 1, b0 = (c / (2 * hkv)) * kDenseRows;
  // [m][i] = R[i][m]: R_k and R_v are both kept transposed for this
  stage_matrix(wsm, (kind ? g.rot_vt : g.rot_k) + (size_t)h * kHeadDim * kHeadDim);
  static_assert(kDenseRows == 4 * kDenseSlices && kDenseThreads / 32 >= kDenseRows / 2, "the step's shares");
  const __half* src = kind ? a.v_new : a.k_new;
  for (int e = threadIdx.x; e < kDenseRows * kHeadDim / 8; e += kDenseThreads) {  // 8 fp16 at a time
    const int r = e >> 4, ch = e & 15, b = b0 + r;
    float2 f[4] = {};
    if (b < a.B) {
      const uint4 raw = *reinterpret_cast<const uint4*>(src + ((size_t)b * hkv + h) * kHeadDim + 8 * ch);
      f[0] = __half22float2(*reinterpret_cast<const __half2*>(&raw.x));
      f[1] = __half22float2(*reinterpret_cast<const __half2*>(&raw.y));
      f[2] = __half22float2(*reinterpret_cast<const __half2*>(&raw.z));
      f[3] = __half22float2(*reinterpret_cast<const __half2*>(&raw.w));
    }
    reinterpret_cast<float4*>(&qs[0][r][8 * ch])[0] = make_float4(f[0].x, f[0].y, f[1].x, f[1].y);
    reinterpret_cast<float4*>(&qs[0][r][8 * ch])[1] = make_float4(f[2].x, f[2].y, f[3].x, f[3].y);
  }
  __syncthreads();
  {  // slice s forms rows 4s .. 4s + 3
    float acc[kDenseRows / kDenseSlices];
    dense_rows(acc, wsm, qs[0] + 4 * slice, i);
#pragma unroll
    for (int r = 0; r < kDenseRows / kDenseSlices; ++r) qs[1][4 * slice + r][i] = acc[r];  // y, beside x
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, half = lane >> 4, j = lane & 15;
  if (warp >= kDenseRows / 2) return;  // a half-warp per vector; no barrier follows
  float bnd[15];
  codec::load_boundaries<BITS>(bnd, g.boundaries);
  const float* r32 = g.dense32 + ((size_t)kind * hkv + h) * kHeadDim * kHeadDim;  // fp32 R rows
  const int cap = a.max_pages * g.page_size;
  {
    const int r = 2 * warp + half, b = b0 + r;
    bool store = false;
    int page = 0, off = 0;
    uint4 raw = make_uint4(0u, 0u, 0u, 0u);
    if (b < a.B) {
      const int len = a.seq_lens[b];  // an out-of-range length is flagged by the split-K kernel
      if (len >= 1 && len <= cap) {
        const int pos = len - 1;
        page = a.block_table[(size_t)b * a.max_pages + pos / g.page_size];
        off = pos % g.page_size;
        store = page >= 0 && page < g.num_pages;
        if (!store && j == 0 && a.status) atomicOr(a.status, RQ_STATUS_BAD_PAGE);
        if (!store) page = 0;
      }
      raw = *reinterpret_cast<const uint4*>(src + ((size_t)b * hkv + h) * kHeadDim + 8 * j);
    }
    float y[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) y[e] = qs[1][r][8 * j + e];
    int code[8];
    float nrm;
    codec::dense_codes<BITS>(code, nrm, raw, y, bnd, r32, store, lane);
    uint8_t* chunk = const_cast<uint8_t*>(a.pages) + ((size_t)page * hkv + h) * (size_t)g.page_bytes;
    codec::pack_store<BITS>(code, nrm, chunk, g.page_size, kind, off, j, store, a.status);
  }
}

}  // namespace

// Dynamic shared memory of a variant: its layout end for a window that starts right after the
// driver's reserved shared memory (the kernels declare no static shared memory).
template <int NT>
static int smem_bytes_nt(int bits) {
  int dev = 0, reserved = 0;
  cudaGetDevice(&dev);
  if (cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev) != cudaSuccess) reserved = 0;
  const uint32_t base = (uint32_t)reserved;
  const uint32_t end = bits == 4 ? smem_plan<4, NT>(base).end
                                 : (bits == 3 ? smem_plan<3, NT>(base).end : smem_plan<2, NT>(base).end);
  return (int)(end - base);
}
static int smem_bytes_for(int bits, int nt) {
  return nt == 1 ? smem_bytes_nt<1>(bits) : (nt == 2 ? smem_bytes_nt<2>(bits) : smem_bytes_nt<3>(bits));
}

size_t attention_smem_bytes() {
  size_t m = 0;
  for (int bits = 2; bits <= 4; ++bits)
    for (int nt = 1; nt <= 3; ++nt)
      if ((size_t)smem_bytes_for(bits, nt) > m) m = (size_t)smem_bytes_for(bits, nt);
  return m;
}

// The n-tiles a unit carries for a call whose kv heads have n_tiles n-tiles of 8 query rows:
// all of them up to 3.
int attention_unit_tiles(int n_tiles, bool) { return n_tiles < 3 ? n_tiles : 3; }

template <int BITS, bool PRE, bool STEP, int NT>
static cudaError_t set_smem_limit() {
  return cudaFuncSetAttribute(attn_splitk_kernel<BITS, PRE, STEP, NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              smem_bytes_for(BITS, NT));
}

template <int BITS>
static cudaError_t set_smem_limits() {
  cudaError_t e = set_smem_limit<BITS, false, false, 1>();
  if (e == cudaSuccess) e = set_smem_limit<BITS, false, false, 2>();
  if (e == cudaSuccess) e = set_smem_limit<BITS, false, false, 3>();
  if (e == cudaSuccess) e = set_smem_limit<BITS, true, false, 1>();
  if (e == cudaSuccess) e = set_smem_limit<BITS, true, false, 2>();
  if (e == cudaSuccess) e = set_smem_limit<BITS, true, false, 3>();
  if (e == cudaSuccess) e = set_smem_limit<BITS, false, true, 1>();
  if (e == cudaSuccess) e = set_smem_limit<BITS, false, true, 2>();
  if (e == cudaSuccess) e = set_smem_limit<BITS, false, true, 3>();
  return e;
}

cudaError_t attention_prepare() {
  cudaError_t e = set_smem_limits<2>();
  if (e == cudaSuccess) e = set_smem_limits<3>();
  if (e == cudaSuccess) e = set_smem_limits<4>();
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(dense_prologue_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, kDenseSmem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(dense_prologue_kernel<3>, cudaFuncAttributeMaxDynamicSharedMemorySize, kDenseSmem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(dense_prologue_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, kDenseSmem);

  return e;
}

template <int BITS, int NT>
static void launch_splitk_nt(const Geometry& g, const AttnArgs& a, cudaStream_t stream) {
  const int smem = smem_bytes_for(BITS, NT);
  constexpr int threads = Shape<NT>::kThreads;
  if (a.q_rot)
    attn_splitk_kernel<BITS, true, false, NT><<<a.grid, threads, smem, stream>>>(g, a, smem);
  else if (a.k_new)
    attn_splitk_kernel<BITS, false, true, NT><<<a.grid, threads, smem, stream>>>(g, a, smem);
  else
    attn_splitk_kernel<BITS, false, false, NT><<<a.grid, threads, smem, stream>>>(g, a, smem);
}

template <int BITS>
static void launch_splitk(const Geometry& g, const AttnArgs& a, cudaStream_t stream) {
  if (a.nt == 1)
    launch_splitk_nt<BITS, 1>(g, a, stream);
  else if (a.nt == 2)
    launch_splitk_nt<BITS, 2>(g, a, stream);
  else
    launch_splitk_nt<BITS, 3>(g, a, stream);
}

// The dense rotation's prologue launch: query rows, plus a decode step's new tokens.  A kv
// head's 64-row groups go to at most as many CTAs as make two per SM over all kv heads (each
// stages the head's 64 KB of fragments once).
static cudaError_t launch_dense_prologue(const Geometry& g, const AttnArgs& a, cudaStream_t stream) {
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const long long rows_per_head = (long long)a.B * a.T * g.group;
  const long long groups = (rows_per_head + 63) / 64;
  const long long cap = std::max(1LL, 2LL * sms / g.num_kv_heads);
  const long long q_ctas = (long long)g.num_kv_heads * std::min(groups, cap);
  const long long step_ctas = a.k_new ? 2LL * g.num_kv_heads * ((a.B + kDenseRows - 1) / kDenseRows) : 0;
  if (q_ctas + step_ctas > 0x7fffffffLL) return cudaErrorInvalidValue;
  const unsigned ctas = (unsigned)(q_ctas + step_ctas);
  if (g.bits == 4)
    dense_prologue_kernel<4><<<ctas, kDenseThreads, kDenseSmem, stream>>>(g, a, (int)q_ctas);
  else if (g.bits == 3)
    dense_prologue_kernel<3><<<ctas, kDenseThreads, kDenseSmem, stream>>>(g, a, (int)q_ctas);
  else
    dense_prologue_kernel<2><<<ctas, kDenseThreads, kDenseSmem, stream>>>(g, a, (int)q_ctas);
  return cudaGetLastError();
}

cudaError_t launch_dense_rotate_q(const Geometry& g, const AttnArgs& a, cudaStream_t stream) {
  if (a.B <= 0) return cudaSuccess;
  if (g.mode != RQ_DENSE || !a.q_rot || a.k_new) return cudaErrorInvalidValue;
  return launch_dense_prologue(g, a, stream);
}

cudaError_t launch_attention(const Geometry& g, const AttnArgs& a, cudaStream_t stream, cudaEvent_t ev_start,
                             cudaEvent_t ev_end) {
  if (a.B <= 0) return cudaSuccess;
  const bool dense = g.mode == RQ_DENSE;
  if (dense != (a.q_rot != nullptr)) return cudaErrorInvalidValue;
  if (a.k_new && (!a.v_new || !g.boundaries || a.T != 1 || (dense && !g.dense32))) return cudaErrorInvalidValue;
  if (a.nt != attention_unit_tiles(a.n_tiles_n, a.k_new != nullptr)) return cudaErrorInvalidValue;
  if (dense) {  // R_k q (and a decode step's new tokens) first; the split-K kernel reads them
    cudaError_t e = launch_dense_prologue(g, a, stream);
    if (e != cudaSuccess) return e;
  }
  if (a.grid > 0) {
    if (ev_start) cudaEventRecord(ev_start, stream);
    if (g.bits == 4)
      launch_splitk<4>(g, a, stream);
    else if (g.bits == 3)
      launch_splitk<3>(g, a, stream);
    else
      launch_splitk<2>(g, a, stream);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (ev_end) cudaEventRecord(ev_end, stream);
  }
  // the split-K kernel finishes every unit itself (normalise, R_v^T, store)
  return cudaGetLastError();
}

}  // namespace rq
