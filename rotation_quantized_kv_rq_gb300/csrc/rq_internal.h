// Internal interface between the host API (rq_api.cpp) and the sm_103a kernels (*.cu).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace rq {

constexpr int kHeadDim = 128;
constexpr int kAttnWarps = 16;      // warps per split-K attention CTA (one CTA per SM)
constexpr int kAttnPairTokens = 32; // tokens a warp takes per iteration (two 16-token tiles)

// Binned code table: u in [-kCodeBinHalf, kCodeBinHalf) / kCodeBinScale falls in bin
// k = RNE(u * kCodeBinScale) + kCodeBinHalf (bins 1 / kCodeBinScale wide); entry k = {the count
// of boundaries below the bin, the one boundary within 2e-5 of the bin or +inf}, so that the
// code is count + (u > boundary) and the boundary is the only one u can lie within 1e-5 of.
// Entry kCodeBins - 1 takes every u outside the range (none for a unit vector's coordinates)
// and NaN: code 0, as the boundary count gives.
constexpr int kCodeBinScale = 2048;
constexpr int kCodeBinHalf = 2304;
constexpr int kCodeBins = 2 * kCodeBinHalf + 1;

// Device-side copy of what every kernel needs to know about a context.
struct Geometry {
  int num_q_heads;
  int num_kv_heads;
  int group;           // Hq / Hkv
  int bits;            // 2, 3 or 4
  int mode;            // 0 planar, 1 iso, 2 dense
  int page_size;
  int num_pages;
  int vec_bytes;       // head_dim * bits / 8
  int page_bytes;      // page_size * (2 * vec_bytes + 4)
  // The attention kernels multiply fp16 centroids c' = c / out_scale (the table `centroids`),
  // out_scale chosen so that the codebook's fp16 images are as exact as possible; q_scale and
  // the final normalisation carry it back, so the results are those of c.
  float q_scale;       // sm_scale * log2(e) * out_scale: scores are kept in base 2
  float out_scale;     // multiplies every attention output row (with its 1 / sum of p)
  // planar / iso: device [Hkv][128] rotation parameters.
  // dense: rot_k = device [Hkv][128][128] R_k TRANSPOSED (query rotation reads it column-wise),
  //        rot_v = device [Hkv][128][128] R_v (output rotation R_v^T o reads it row-wise).
  const float* rot_k;
  const float* rot_v;
  // dense only: device fp16 [2 (K, V)][Hkv][2 (hi, lo)][128][128], R = hi + lo split for the
  // tensor-core append (hi = fp16(R), lo = fp16(R - hi)); null otherwise.
  const __half* dense16;
  // dense only: device fp32 [2 (K, V)][Hkv][128][128] row-major R (exact recompute in the append)
  const float* dense32;
  // dense only: device [Hkv][8 k-steps][16 n-tiles][32 lanes][4] u32, R_k's fp16 hi and lo as the
  // B operands of the query rotation's m16n8k16 MMAs (lane 4g + t: output dim 8 n-tile + g;
  // words hi(m, m+1), hi(m+2, m+3), lo(m, m+1), lo(m+2, m+3) with m = 32t + 4 k-step, the lower
  // dim in the low half); null otherwise.
  const uint32_t* rotq;
  // dense only: device fp32 [Hkv][128][128] R_v TRANSPOSED ([m][i] = R_v[i][m]: a decode step's
  // V coding stages it as it is); null otherwise.
  const float* rot_vt;
  // device u32 [kCodeBins][2] (count, boundary bits): the binned code table, or null when two
  // boundaries are too close for its bins (the select tree decides then)
  const uint32_t* code_table;
  const float* centroids;   // device [2^bits]: c / out_scale, the fp16 operands' source
  const float* boundaries;  // device [2^bits - 1]
};

// One attention launch (decode is T = 1).
struct AttnArgs {
  const void* q;             // fp16 [B][T][Hq][128]
  const uint8_t* pages;
  const int32_t* block_table;
  int max_pages;
  const int32_t* seq_lens;
  int B;
  int T;
  void* out;                 // fp16 [B][T][Hq][128]
  int32_t* status;           // nullable
  // A unit is (sequence, kv head, group of nt n-tiles): units = B * Hkv * ceil(n_tiles_n / nt).
  float* ws;                 // fragment partials: [units + grid][8 nt rows][kPartialStride] floats
  int* frag;                 // [units][2]: first and last CTA holding a fragment of each unit
  int* cnt;                  // [units]: rounds finished per unit; zero between launches
  int grid;                  // CTAs of the split-K launch (the stream-K partition's parts)
  int rows;                  // T * group: query rows per kv head
  int n_tiles_n;             // ceil(rows / 8)
  int nt;                    // n-tiles per unit: attention_unit_tiles(n_tiles_n, k_new != null)
  const uint64_t* tree_mask; // [B][T] draft visibility bits (tree verify), or null (causal chain)
  float* q_rot;              // dense: fp32 [B][T][Hq][128] scratch for R_k q; null otherwise
  // Decode step: fp16 [B][Hkv][128] K and V of each sequence's newest token, position
  // seq_lens[b] - 1, quantized into the cache by the split-K kernel itself (planar / iso) or by
  // the dense prologue kernel (dense); or null.
  const __half* k_new;
  const __half* v_new;
};

constexpr int kPartialStride = 132;   // floats per partial row: m, l, pad, pad, o[128]

cudaError_t launch_append(const Geometry& g, const void* k, const void* v, const int32_t* slots,
                          int n, uint8_t* pages, int32_t* status, cudaStream_t stream);
cudaError_t append_prepare();  // sets the dense append kernel's shared-memory limit

cudaError_t launch_attention(const Geometry& g, const AttnArgs& a, cudaStream_t stream,
                             cudaEvent_t ev_start = nullptr, cudaEvent_t ev_end = nullptr);

// The split-K kernel's prefix of tiles per sequence lives in its low slot region: at most this
// many sequences per call.
constexpr int kMaxBatch = 8000;

// Dense rotation: a.q_rot = R_k q for every query row of the call (fp32), one launch.
cudaError_t launch_dense_rotate_q(const Geometry& g, const AttnArgs& a, cudaStream_t stream);

// Extend (prefill) attention: T query tokens per sequence, causal; a dense rotation's queries
// come pre-rotated in a.q_rot (launch_dense_rotate_q), other rotations need no workspace.
cudaError_t launch_extend(const Geometry& g, const AttnArgs& a, cudaStream_t stream, cudaEvent_t ev_start = nullptr,
                          cudaEvent_t ev_end = nullptr);
cudaError_t extend_prepare();

// n-tiles of 8 query rows a split-K unit carries, for kv heads of n_tiles n-tiles: min(n_tiles,
// 3), for decode, verify and a decode step alike (`step` is kept for the workspace sizing).
int attention_unit_tiles(int n_tiles, bool step);

// Split-K workspace of a call with B sequences, Hkv kv heads, n_tiles n-tiles per kv head and
// `grid` CTAs: units, partial floats ((units + grid) slots of 8 nt rows).
inline void attention_workspace(long long B, int hkv, int n_tiles, bool step, int grid, long long* units,
                                long long* partial_floats) {
  const int nt = attention_unit_tiles(n_tiles, step);
  *units = B * hkv * ((n_tiles + nt - 1) / nt);
  *partial_floats = (*units + grid) * 8LL * nt * kPartialStride;
}

// Dynamic shared memory the attention kernel needs (set as the kernel's maximum once).
size_t attention_smem_bytes();
cudaError_t attention_prepare();

}  // namespace rq
