/*
 * rq.h -- C ABI of the rotation-quantized KV cache library (librq.so), GB300 / sm_103a.
 *
 * The method (the README "SGLang 1-Bit Turbo -- AMD ROCm Inference with PrismML Quantization +
 * Speculative Decoding Support", called "the README" below; its section "RotorQuant KV Cache
 * Compression", and
 * the TurboQuant section it is compared with): every K and V vector written to the cache
 * keeps its L2 norm, is turned by a fixed data-oblivious rotation -- 2D Givens pairs
 * (PlanarQuant), 4D unit-quaternion blocks (IsoQuant) or one dense orthogonal matrix
 * (TurboQuant) -- and each rotated coordinate is coded with a b-bit Lloyd-Max scalar
 * quantizer (rq3/rq4 x planar/iso, tq2/tq3/tq4 dense; every mode takes 2, 3 or 4 bits).  Attention
 * reads the packed cache directly: because the rotation is orthogonal, a query is rotated
 * once instead of un-rotating every key, values are summed in the rotated space and the
 * output is rotated back once.
 *
 * Conventions for every call:
 *   - Pointers marked "device" are CUDA device pointers owned by the caller; the library
 *     never frees them.  Pointers marked "host" are read during the call only.
 *   - fp16 means IEEE binary16 stored as 2-byte values.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls enqueue work and
 *     return without synchronising; the caller keeps inputs alive until the stream passes.
 *   - A context holds one split-K workspace: calls on the same context must not overlap on
 *     the GPU (issue them on one stream, or order the streams).
 *   - Return value: RQ_OK or an RQ_ERR_* code.  Argument errors are detected on the host
 *     before anything is enqueued.  Nothing throws across this boundary.
 *   - `d_status` (device int32, nullable): data-dependent range faults found by a kernel
 *     (a page id outside [0, num_pages), a slot outside the pool, a sequence longer than
 *     its block-table row) are OR-ed into *d_status as RQ_STATUS_* bits; the offending
 *     index is clamped so no access leaves its buffer, and the outputs of the affected
 *     sequence are unspecified.  The library never clears *d_status.
 *
 * Storage contract (the method's description fixes none of it; this library's choice):
 *   page pool   : device bytes [num_pages][num_kv_heads][page_bytes]; the chunk of
 *                 (page, kv head) is   K codes [P][vb] | V codes [P][vb] | K norms fp16 [P] |
 *                 V norms fp16 [P],  vb = head_dim * bits / 8, page_bytes = P * (2 vb + 4).
 *   4-bit codes : byte j = code[2j] | code[2j+1] << 4.  In the V-codes section of a chunk,
 *                 tokens are stored as pairs: pair p = tokens (2p, 2p+1) fills 128 bytes and the
 *                 8 bytes of 16-dim group c of token 2p + h sit at 16 * (c ^ (2p mod 8)) + 8h.
 *                 K codes, and 3-bit V codes, are stored token after token.
 *   2-bit codes : byte j = code[4j] | code[4j+1] << 2 | code[4j+2] << 4 | code[4j+3] << 6.  In
 *                 the V-codes section, pair p = tokens (2p, 2p+1) fills 64 bytes and the 4 bytes
 *                 of 16-dim group c of token 2p + h sit at 8 * (c ^ (4 * (p / 2 mod 2))) + 4h.
 *   3-bit codes : per 32-dim group w, 12 bytes at 12w = little-endian words W0, W1, W2:
 *                 W0 bits 2i.. = code[32w+i] & 3, W1 bits 2i.. = code[32w+16+i] & 3
 *                 (i = 0..15), W2 bit p(i) = code[32w+i] >> 2 with i = 16h + 4k + r and
 *                 p(i) = 8k + 2h + {4,5,0,1}[r].
 *   code        : number of bin boundaries strictly below u = (R x)_i / ||x||, where the
 *                 boundaries are midpoints of consecutive centroids; a vector of norm 0
 *                 codes every coordinate as 2^(bits-1) - 1.
 *   norm        : ||x|| rounded to fp16 (nearest even).
 *   slot        : page * P + offset in page; block_table[b][i] is the page holding tokens
 *                 i*P .. i*P+P-1 of sequence b.
 */
#ifndef RQ_H
#define RQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes */
#define RQ_OK 0
#define RQ_ERR_INVALID 1       /* a NULL pointer, a negative size, inconsistent geometry */
#define RQ_ERR_UNSUPPORTED 2   /* valid but not built: head_dim != 128, bits not 2/3/4, ... */
#define RQ_ERR_CUDA 3          /* a CUDA call failed (allocation, copy or launch) */
#define RQ_ERR_CAPACITY 4      /* batch, query tokens or block-table width above the context's limits */

/* Bits of *d_status */
#define RQ_STATUS_BAD_PAGE 1   /* block-table entry outside [0, num_pages) */
#define RQ_STATUS_BAD_SLOT 2   /* slot_mapping entry >= num_pages * page_size */
#define RQ_STATUS_BAD_LEN 4    /* seq_len < 0 or above max_pages * page_size, or below T */
#define RQ_STATUS_NORM_OVERFLOW 8 /* a vector norm above the fp16 range (stored as inf) */
#define RQ_STATUS_TIMEOUT 16   /* an attention kernel's staged page copy did not complete within
                                  its bounded wait (outputs of that call are unspecified) */

/* Rotation families.  Source: README, CLI Reference > KV Cache Compression Flags (--kv-cache-dtype
   rq{3,4}_{planar,iso}, tq{2,3,4}) and the two mode tables under Core Features (RotorQuant: 2D
   Givens or 4D quaternion; TurboQuant: dense random rotation). */
#define RQ_PLANAR 0            /* PlanarQuant: 2D Givens rotation per dimension pair */
#define RQ_ISO 1               /* IsoQuant: unit quaternion per 4-dimension block */
#define RQ_DENSE 2             /* TurboQuant: one dense orthogonal head_dim x head_dim matrix */

typedef struct rq_ctx rq_ctx;  /* opaque, owned by the library */

typedef struct {
  int head_dim;              /* must be 128 */
  int num_q_heads;           /* Hq, a multiple of num_kv_heads */
  int num_kv_heads;          /* Hkv >= 1 */
  int bits;                  /* 2, 3 or 4 */
  int mode;                  /* RQ_PLANAR, RQ_ISO or RQ_DENSE */
  int page_size;             /* P: a multiple of 16, at most 256 */
  int num_pages;             /* pages in the caller's pool */
  int max_batch;             /* largest B of an attention call */
  int max_query_tokens;      /* largest T of a verify call (>= 1) */
  int max_pages_per_seq;     /* largest block-table width (max_pages) of an attention call */
  /* host float32.  planar -> [Hkv][d/2][2] = (cos t, sin t) of the pair (2i, 2i+1),
     y_2i = c x_2i - s x_2i+1, y_2i+1 = s x_2i + c x_2i+1;
     iso -> [Hkv][d/4][4] = unit quaternion (a, b, c, d) of block 4i..4i+3, y = q (x) x
     (Hamilton product, q on the left);
     dense -> [Hkv][d][d] = row-major R, y_i = sum_j R[i][j] x_j.  R must be orthogonal (the
     library does not check; decoding multiplies by R^T).
     rot_k turns keys and queries, rot_v values. */
  const float *rot_k;
  const float *rot_v;
  /* host float32 [2^bits] ascending centroids, or NULL for the Lloyd-Max quantizer of
     N(0, 1/head_dim) (the levels of N(0,1) divided by sqrt(head_dim)). */
  const float *codebook;
  float sm_scale;            /* softmax scale; 0 selects 1/sqrt(head_dim) */
  int device;                /* CUDA device ordinal the context lives on; -1 = current */
} rq_config;

/* Source: this library (the constructor of the context that rq_free releases); the tables it holds
   are the rotations of README > Core Features > RotorQuant / TurboQuant KV Cache Compression and
   the Lloyd-Max codebook named in its Acknowledgments (TurboQuant entry). Validates cfg, copies the
   rotation tables and codebook to the device and allocates the split-K workspace on cfg->device.
   On success *out is a new context; on failure *out is NULL and nothing stays allocated.  Errors:
   RQ_ERR_INVALID, RQ_ERR_UNSUPPORTED, RQ_ERR_CUDA. */
int rq_create(rq_ctx **out, const rq_config *cfg);

/* Source: this library.  Releases everything rq_create allocated.  NULL-safe.  The caller must make
   sure no work of this context is still running (synchronise its stream first). */
void rq_free(rq_ctx *ctx);

/* Source: this library's storage contract (above).  Bytes of one (page, kv head) chunk: page_size *
   (2 * head_dim * bits / 8 + 4).  0 for NULL. */
size_t rq_page_bytes(const rq_ctx *ctx);

/* Source: README, Acknowledgments (TurboQuant entry: "Lloyd-Max scalar quantization"), read as the
   Lloyd-Max quantizer of the N(0, 1/head_dim) coordinates of a rotated unit vector. Host only (no
   GPU needed): the default codebook -- ascending centroids of the Lloyd-Max quantizer of N(0,1)
   with 2^bits levels, divided by sqrt(head_dim), rounded to float32 -- into centroids[2^bits].
   bits in 1..8, head_dim >= 1.  Returns RQ_OK or RQ_ERR_INVALID. */
int rq_lloyd_max_codebook(int bits, int head_dim, float *centroids);

/* Source: this library.  Host copies of the context's centroids [2^bits] and bin boundaries
   [2^bits - 1] (float32; boundary j = float((centroid_j + centroid_{j+1}) / 2) computed in
   double).  Either may be NULL. */
int rq_get_codebook(const rq_ctx *ctx, float *centroids, float *boundaries);

/*
 * Source: README > Core Features > RotorQuant KV Cache Compression (a fixed, data-oblivious 2D
 * Givens or 4D quaternion rotation, 3- or 4-bit codes) and > TurboQuant KV Cache Compression (a
 * dense random rotation, 2-4 bits), with Acknowledgments (rotation, then Lloyd-Max scalar
 * quantization).  The norm and the packing are this library's storage contract.
 * Quantize-on-append (one fused kernel): for token t < n and kv head h, encode
 * k[t][h][:] and v[t][h][:] (device fp16 [n][Hkv][head_dim]) into slot slot_mapping[t]
 * (device int32 [n]) of the page pool kv_pages (device, see the storage contract).  A slot
 * < 0 is skipped (padding); a slot >= num_pages * page_size sets RQ_STATUS_BAD_SLOT and is
 * skipped.  Slots within one call must be distinct.  n = 0 is a no-op.  k, v and kv_pages must be
 * 16-byte aligned (RQ_ERR_INVALID otherwise).
 */
int rq_quantize_append(rq_ctx *ctx, const void *k, const void *v, const int32_t *slot_mapping,
                       int n, void *kv_pages, int32_t *d_status, void *stream);

/*
 * Source: README > RDNA2 Crash Fixes, rows 6 and 10 (decode attention over a paged cache addressed
 * through kv_indices, the page table), read over the packed cache of Core
 * Features > RotorQuant KV Cache Compression: the query is rotated once, values are summed in
 * the rotated space and the output is rotated back once (the rotation is orthogonal).
 * GQA decode attention over the packed cache (split-K flash-decode + log-sum-exp combine).
 *   q           device fp16 [B][Hq][head_dim]
 *   kv_pages    device page pool
 *   block_table device int32 [B][max_pages]
 *   seq_lens    device int32 [B]: tokens of sequence b, all attended (0 gives zeros)
 *   out         device fp16 [B][Hq][head_dim]; head hq reads kv head hq / (Hq / Hkv)
 * out = softmax(sm_scale * q K^T) V over the dequantised cache.  B may be 0.  q, kv_pages and
 * out must be 16-byte aligned (this and every attention entry point below).
 * Errors: RQ_ERR_INVALID (also a misaligned q, kv_pages or out), RQ_ERR_CAPACITY (B > max_batch, max_pages > max_pages_per_seq),
 * RQ_ERR_CUDA.
 */
int rq_decode_attention(rq_ctx *ctx, const void *q, const void *kv_pages, const int32_t *block_table,
                        int max_pages, const int32_t *seq_lens, int B, void *out, int32_t *d_status,
                        void *stream);

/*
 * Source: README > RDNA2 Crash Fixes, row 5 (extend attention over partial tiles) and row 9a (the
 * extend path), over the packed cache of Core Features > RotorQuant KV Cache Compression.
 * Extend (prefill) attention: T new query tokens per sequence, already appended as the last T
 * tokens of the cache, each attending to the cached prefix and causally to the new tokens:
 * query row j (0 <= j < T) sees positions 0 .. seq_lens[b] - T + j -- the same result as
 * rq_verify_attention, computed by a kernel built for large T (256 query rows share every
 * dequantized tile of the cache; tensor-core QK^T and PV).  Planar and iso rotations use no
 * workspace: T is limited only by the q / out buffers, not by max_query_tokens.  A dense rotation
 * (RQ_DENSE) rotates the queries into the context's workspace first, so there T must not exceed
 * max_query_tokens (RQ_ERR_CAPACITY otherwise).
 *   q   device fp16 [B][T][Hq][head_dim],   out device fp16 [B][T][Hq][head_dim]
 * Other arguments as rq_verify_attention.  Errors as rq_verify_attention (except that T above
 * max_query_tokens is allowed for planar and iso rotations).
 */
int rq_extend_attention(rq_ctx *ctx, const void *q, int T, const void *kv_pages, const int32_t *block_table,
                        int max_pages, const int32_t *seq_lens, int B, void *out, int32_t *d_status,
                        void *stream);

/*
 * Source: this library -- rq_quantize_append of one token per sequence followed by
 * rq_decode_attention, in one launch.
 * One decode step in one kernel launch (planar, iso): quantize-append of every sequence's newest
 * K/V token, folded into rq_decode_attention's split-K kernel, then decode attention over the cache
 * including that token (the combine of split partials runs in the same kernel).
 *   k_new, v_new  device fp16 [B][Hkv][head_dim]: the token of sequence b, written to position
 *                 seq_lens[b] - 1 -- page block_table[b][(seq_lens[b] - 1) / P], offset
 *                 (seq_lens[b] - 1) % P -- exactly as rq_quantize_append would write it
 *   kv_pages      device page pool (written: the step's tokens; read: everything)
 *   other arguments as rq_decode_attention; seq_lens[b] counts the new token, and a sequence
 *   with seq_lens[b] = 0 appends nothing.
 * The result equals rq_quantize_append of the tokens followed by rq_decode_attention (the same
 * bytes written, the same output).  A dense rotation (RQ_DENSE) codes the new tokens in the
 * launch that rotates the queries, before the split-K kernel (which applies the output
 * rotation itself): two launches instead of four.  A page id out of range for the new token sets RQ_STATUS_BAD_PAGE
 * and skips its write.  Errors as rq_decode_attention, plus RQ_ERR_INVALID for a NULL or
 * non-16-byte-aligned k_new / v_new.
 */
int rq_decode_step(rq_ctx *ctx, const void *q, const void *k_new, const void *v_new, void *kv_pages,
                   const int32_t *block_table, int max_pages, const int32_t *seq_lens, int B, void *out,
                   int32_t *d_status, void *stream);

/*
 * Source: README > Core Features > EAGLE3 / P-EAGLE Speculative Decoding (the target model
 * verifies the draft tokens) and RDNA2 Crash Fixes rows 9b and 11 (verify extends seq_lens by the
 * drafts); a chain is a top-1 draft.
 * Speculative chain-verify attention: T query tokens per sequence, the last T cached tokens
 * being the drafts themselves (append them first).  Query row j (0 <= j < T) attends to
 * positions 0 .. seq_lens[b] - T + j (causal over the draft tail).
 *   q   device fp16 [B][T][Hq][head_dim],   out device fp16 [B][T][Hq][head_dim]
 * Other arguments as rq_decode_attention; T = 1 is decode.  0 < seq_lens[b] < T sets
 * RQ_STATUS_BAD_LEN.  Errors as rq_decode_attention, plus RQ_ERR_CAPACITY for
 * T > max_query_tokens.
 */
int rq_verify_attention(rq_ctx *ctx, const void *q, int T, const void *kv_pages,
                        const int32_t *block_table, int max_pages, const int32_t *seq_lens, int B,
                        void *out, int32_t *d_status, void *stream);

/*
 * Source: README > Core Features > EAGLE3 / P-EAGLE Speculative Decoding (probabilistic tree
 * sampling of drafts): verify over a draft tree.
 * Speculative tree-verify attention (a draft tree, e.g. top-k > 1 EAGLE trees): like
 * rq_verify_attention, except that query row j attends to the prefix, positions
 * 0 .. seq_lens[b] - T - 1, and to draft i (position seq_lens[b] - T + i) exactly when bit i of
 * tree_mask[b][j] is set -- usually draft j's ancestors and draft j itself.
 *   tree_mask  device uint64 [B][T], 1 <= T <= 64
 * A causal chain is tree_mask[b][j] = 2^(j+1) - 1 and gives rq_verify_attention's result.  A row
 * that sees nothing (empty prefix and mask 0) gives zeros.  Errors as rq_verify_attention, plus
 * RQ_ERR_INVALID for T > 64 or a NULL mask.
 */
int rq_tree_verify_attention(rq_ctx *ctx, const void *q, int T, const uint64_t *tree_mask, const void *kv_pages,
                             const int32_t *block_table, int max_pages, const int32_t *seq_lens, int B,
                             void *out, int32_t *d_status, void *stream);

/*
 * Decode attention that allocates nothing.  The pages have no counterpart to this entry point:
 * it exists for callers that cannot call cudaMalloc -- for example code running inside a
 * serving engine whose memory pool has already reserved the device's free memory (a raw
 * allocation would fail or fragment the pool), or a plugin whose host framework forbids
 * allocations outside its own allocator.  Such callers cannot create a context either, so
 * everything comes in as arguments:
 *   cfg         host; only head_dim, num_q_heads, num_kv_heads, bits, mode, page_size, num_pages
 *               and sm_scale are read (the max_* limits, host tables, codebook and device are
 *               ignored).  mode RQ_DENSE returns RQ_ERR_UNSUPPORTED (its query rotation needs
 *               a workspace).
 *   d_rot_k, d_rot_v   device float32 [Hkv][head_dim], laid out as rq_config.rot_k / rot_v
 *   d_centroids        device float32 [2^bits], ascending (e.g. from rq_lloyd_max_codebook)
 *   other arguments    as rq_decode_attention, on the CURRENT device
 * The result equals rq_decode_attention's on the same inputs.
 * Scratch: the split-K partials, the per-unit fragment bounds and round counters live in one
 * file-scope 16 MiB device array that every GPU which loads the library holds until the process
 * exits.  With n = ceil(group / 8) tiles of 8 query rows per kv head, m = min(n, 3) of them per
 * work unit and U = B * num_kv_heads * ceil(n / m) work units, a call with U > 8,192, or with
 * (U + the device's SM count) * m > 3,948 partial slots, returns RQ_ERR_CAPACITY; so do
 * B > 8,000 and a block table whose max_pages * page_size exceeds INT32_MAX.
 * The first call on a device sets up that device (resolves the array's address, reads the SM
 * count, sets the kernel's shared-memory limit); make that first call before any stream
 * capture.  The round counters start at zero (the array is zero-initialised when the library
 * loads) and every call leaves them at zero.  Every call shares the one array, so calls that
 * overlap on the GPU (different streams, or different host threads) race: serialise them.
 */
int rq_decode_attention_noalloc(const rq_config *cfg, const float *d_rot_k, const float *d_rot_v,
                                const float *d_centroids, const void *q, const void *kv_pages,
                                const int32_t *block_table, int max_pages, const int32_t *seq_lens,
                                int B, void *out, int32_t *d_status, void *stream);

/* Source: this library.  Diagnostics.  While set, every attention call records ev_start on its
   stream just before its split-K kernel and ev_end just after it (both cudaEvent_t created by the
   caller, who reads the elapsed time); NULL, NULL stops recording.  Costs nothing when unset. */
int rq_set_profile_events(rq_ctx *ctx, void *ev_start, void *ev_end);

/* Source: this library.  Static English text for a return code (never NULL). */
const char *rq_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* RQ_H */
