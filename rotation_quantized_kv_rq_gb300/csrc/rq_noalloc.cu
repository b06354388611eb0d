// rq_decode_attention_noalloc: the decode attention of rq_decode_attention for callers that
// cannot allocate device memory.  Its split-K scratch (the fragment partials, the per-unit
// fragment bounds and round counters) lives in one file-scope __device__ array instead of a context's
// cudaMalloc'd workspace, and the tables come from the caller as device pointers, so the call
// allocates nothing.  The kernels are the library's own attention kernels.
#include <cuda_runtime.h>

#include <cmath>
#include <mutex>

#include "../../include/rq.h"
#include "rq_internal.h"

namespace {

// Scratch: fragment bounds (2 ints per unit), round counters (1 int per unit), then fragment
// partials of 8 query rows x kPartialStride floats per n-tile of a unit.  A call with U units
// and G CTAs uses 3U ints and (U + G) x (n-tiles per unit) 8-row slots.
constexpr size_t kScratchBytes = (size_t)16 << 20;
constexpr size_t kMaxUnits = 8192;
constexpr size_t kFragBytes = kMaxUnits * 2 * sizeof(int);              // 64 KiB
constexpr size_t kCntBytes = kMaxUnits * sizeof(int);                   // 32 KiB
constexpr size_t kSlotBytes = 8 * rq::kPartialStride * sizeof(float);   // 8 query rows of one fragment
constexpr size_t kScratchSlots = (kScratchBytes - kFragBytes - kCntBytes) / kSlotBytes;  // 3,948
constexpr int kMaxDevices = 64;

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
      cfg->page_size > 256 || (long long)cfg->num_kv_heads * cfg->page_size * (2 * 16 * cfg->bits + 4) > INT32_MAX)
    return RQ_ERR_UNSUPPORTED;
  if (B == 0) return RQ_OK;
  if (!d_rot_k || !d_rot_v || !d_centroids || !q || !kv_pages || !block_table || !seq_lens || !out)
    return RQ_ERR_INVALID;
  if ((uintptr_t)q % 16 != 0 || (uintptr_t)kv_pages % 16 != 0 || (uintptr_t)out % 16 != 0)
    return RQ_ERR_INVALID;  // bulk copies and vector I/O

  const int hkv = cfg->num_kv_heads, group = cfg->num_q_heads / hkv;
  const int n_tiles = (group + 7) / 8;
  long long units = 0, partial_floats = 0;
  rq::attention_workspace(B, hkv, n_tiles, false, 0, &units, &partial_floats);
  const int nt = rq::attention_unit_tiles(n_tiles, false);
  if (B > rq::kMaxBatch || units > (long long)kMaxUnits) return RQ_ERR_CAPACITY;
  if ((long long)max_pages * cfg->page_size > INT32_MAX) return RQ_ERR_CAPACITY;  // positions are int

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return RQ_ERR_CUDA;
  DeviceSlot* slot = nullptr;
  if (setup_device(dev, &slot) != cudaSuccess) return RQ_ERR_CUDA;
  if ((units + slot->num_sms) * nt > (long long)kScratchSlots) return RQ_ERR_CAPACITY;

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
  g.out_scale = 1.f;  // the caller's centroids, unscaled
  g.rot_k = d_rot_k;
  g.rot_v = d_rot_v;
  g.dense16 = nullptr;
  g.dense32 = nullptr;
  g.rotq = nullptr;
  g.rot_vt = nullptr;
  g.code_table = nullptr;
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
  a.k_new = a.v_new = nullptr;
  a.rows = group;
  a.n_tiles_n = n_tiles;
  a.nt = nt;

  a.frag = reinterpret_cast<int*>(slot->scratch);
  a.cnt = reinterpret_cast<int*>(slot->scratch + kFragBytes);
  a.ws = reinterpret_cast<float*>(slot->scratch + kFragBytes + kCntBytes);
  a.grid = slot->num_sms;
  // Only the round counters need a starting value: zero, as the array is zero-initialised when
  // the module loads, and every launch that runs to its end leaves them at zero again.  The
  // bounds and partials are written by each launch before they are read.
  return rq::launch_attention(g, a, (cudaStream_t)stream) == cudaSuccess ? RQ_OK : RQ_ERR_CUDA;
}
