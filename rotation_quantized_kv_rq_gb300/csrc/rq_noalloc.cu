// rq_decode_attention_noalloc: the decode attention of rq_decode_attention for callers that
// cannot allocate device memory.  Its split-K scratch (the per-split partial states and the
// two work counters) lives in one file-scope __device__ array instead of a context's
// cudaMalloc'd workspace, and the tables come from the caller as device pointers, so the call
// allocates nothing.  The kernels are the library's own attention kernels.
#include <cuda_runtime.h>

#include <cmath>
#include <mutex>

#include "../../include/rq.h"
#include "rq_internal.h"

namespace {

// Scratch: the two work counters, then split partials of kPartialStride floats per row.
constexpr size_t kScratchBytes = (size_t)16 << 20;
constexpr size_t kCounterBytes = 256;
constexpr size_t kRowBytes = 8 * rq::kPartialStride * sizeof(float);  // one item: 8 query rows
constexpr size_t kScratchItems = (kScratchBytes - kCounterBytes) / kRowBytes;
constexpr int kMaxDevices = 64;
constexpr int kMaxSplits = 64;
constexpr int kMaxSplitPages = 1024;

// Every GPU that loads the library holds this array until the process exits.  Host code must
// not use its name as an address: the device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

struct DeviceSlot {
  bool ready = false;
  unsigned char* scratch = nullptr;
  int num_sms = 0;
};
DeviceSlot g_slots[kMaxDevices];
std::mutex g_setup_mutex;

// Once per device, with that device current: resolve the scratch address and the SM count and
// set the attention kernel's shared-memory limit.  Nothing here allocates.
cudaError_t setup_device(int dev, DeviceSlot** out) {
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  DeviceSlot& s = g_slots[dev];
  if (!s.ready) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&s.num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = rq::attention_prepare();
    if (e != cudaSuccess) return e;
    s.scratch = static_cast<unsigned char*>(p);
    s.ready = true;
  }
  *out = &s;
  return cudaSuccess;
}

}  // namespace

extern "C" int rq_decode_attention_noalloc(const rq_config* cfg, const float* d_rot_k, const float* d_rot_v,
                                           const float* d_centroids, const void* q, const void* kv_pages,
                                           const int32_t* block_table, int max_pages, const int32_t* seq_lens,
                                           int B, void* out, int32_t* d_status, void* stream) {
  if (!cfg || B < 0 || max_pages < 1) return RQ_ERR_INVALID;
  if (cfg->num_q_heads <= 0 || cfg->num_kv_heads <= 0 || cfg->page_size <= 0 || cfg->num_pages <= 0 ||
      cfg->num_q_heads % cfg->num_kv_heads != 0 ||
      (cfg->mode != RQ_PLANAR && cfg->mode != RQ_ISO && cfg->mode != RQ_DENSE) ||
      !(cfg->sm_scale >= 0.0f) || std::isinf(cfg->sm_scale))
    return RQ_ERR_INVALID;
  if (cfg->mode == RQ_DENSE) return RQ_ERR_UNSUPPORTED;  // its query rotation needs a workspace
  if (cfg->head_dim != rq::kHeadDim || cfg->bits < 2 || cfg->bits > 4 || cfg->page_size % 16 != 0 ||
      cfg->page_size > 256)
    return RQ_ERR_UNSUPPORTED;
  if (B == 0) return RQ_OK;
  if (!d_rot_k || !d_rot_v || !d_centroids || !q || !kv_pages || !block_table || !seq_lens || !out)
    return RQ_ERR_INVALID;

  const int hkv = cfg->num_kv_heads, group = cfg->num_q_heads / hkv;
  const long long units = (long long)B * hkv * ((group + 7) / 8);
  if (units > (long long)kScratchItems) return RQ_ERR_CAPACITY;  // not even one split fits
  if ((max_pages + kMaxSplitPages - 1) / kMaxSplitPages > kMaxSplits) return RQ_ERR_CAPACITY;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return RQ_ERR_CUDA;
  DeviceSlot* slot = nullptr;
  if (setup_device(dev, &slot) != cudaSuccess) return RQ_ERR_CUDA;

  rq::Geometry g;
  g.num_q_heads = cfg->num_q_heads;
  g.num_kv_heads = hkv;
  g.group = group;
  g.bits = cfg->bits;
  g.mode = cfg->mode;
  g.page_size = cfg->page_size;
  g.num_pages = cfg->num_pages;
  g.vec_bytes = rq::kHeadDim * cfg->bits / 8;
  g.page_bytes = cfg->page_size * (2 * g.vec_bytes + 4);
  const float scale = cfg->sm_scale > 0.f ? cfg->sm_scale : (float)(1.0 / std::sqrt((double)rq::kHeadDim));
  g.q_scale = (float)(scale * 1.44269504088896340736);
  g.rot_k = d_rot_k;
  g.rot_v = d_rot_v;
  g.dense16 = nullptr;
  g.dense32 = nullptr;
  g.centroids = d_centroids;
  g.boundaries = nullptr;  // decode never codes

  rq::AttnArgs a;
  a.q = q;
  a.pages = (const uint8_t*)kv_pages;
  a.block_table = block_table;
  a.max_pages = max_pages;
  a.seq_lens = seq_lens;
  a.B = B;
  a.T = 1;
  a.out = out;
  a.status = d_status;
  a.tree_mask = nullptr;
  a.q_rot = nullptr;
  a.rows = group;
  a.n_tiles_n = (group + 7) / 8;

  // Split choice as in the context path (whole 256-token rounds, fewest worst-case rounds),
  // restricted to what the scratch array holds.
  const int P = cfg->page_size;
  // one round = every warp of a CTA taking one 32-token pair
  const int round_tokens = rq::kAttnWarps * rq::kAttnPairTokens;
  const int quantum = round_tokens / P > 0 ? round_tokens / P : 1;
  long long best_pps = -1, best_cost = -1, best_ns = 0;
  for (int ns = 1; ns <= kMaxSplits; ++ns) {
    long long pps = (max_pages + ns - 1) / ns;
    pps = (pps + quantum - 1) / quantum * quantum;
    if (pps > kMaxSplitPages) continue;
    const long long nsplit = (max_pages + pps - 1) / pps;
    if (units * nsplit > (long long)kScratchItems) continue;
    const long long rounds = (units * nsplit + slot->num_sms - 1) / slot->num_sms;
    const long long cost = rounds * ((pps * P + round_tokens - 1) / round_tokens + 1);
    if (best_cost < 0 || cost < best_cost) best_cost = cost, best_pps = pps, best_ns = nsplit;
  }
  if (best_pps < 0) return RQ_ERR_CAPACITY;
  a.pages_per_split = (int)best_pps;
  a.max_splits = (int)best_ns;
  a.counters = reinterpret_cast<int*>(slot->scratch);
  a.ws = reinterpret_cast<float*>(slot->scratch + kCounterBytes);

  // The array keeps whatever the last call left: the counters must start every launch at 0.
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaMemsetAsync(slot->scratch, 0, 2 * sizeof(int), st) != cudaSuccess) return RQ_ERR_CUDA;
  return rq::launch_attention(g, a, slot->num_sms, st) == cudaSuccess ? RQ_OK : RQ_ERR_CUDA;
}
