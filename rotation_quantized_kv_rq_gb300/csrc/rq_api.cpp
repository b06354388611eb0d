// Host side of the C ABI declared in include/rq.h: argument validation, the context (device
// tables and split-K workspace), the default Lloyd-Max codebook and launch planning.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <new>
#include <vector>

#include "../../include/rq.h"
#include "rq_internal.h"

struct rq_ctx {
  rq_config cfg;          // host pointers cleared after creation
  rq::Geometry g;
  int device;
  int num_sms;
  float* d_tables;        // rot_k | rot_v | centroids | boundaries
  __half* d_dense16;      // dense: fp16 hi/lo split of R_k and R_v for the append GEMM
  float* d_dense32;       // dense: fp32 R_k and R_v, row-major, for the append's exact recompute; then R_v^T
  uint32_t* d_rotq;       // dense: R_k's fp16 hi / lo in the query rotation's MMA fragment order
  uint32_t* d_codetab;    // the binned code table (rq_internal.h), or null
  float* d_qrot;          // dense: fp32 R_k q of one attention call [max_batch][max_T][Hq][128]
  float* d_ws;            // fragment partials of the stream-K split
  int* d_frag;            // first / last CTA of each unit's fragments [2 U], then rounds done per unit [U]
  size_t ws_floats;
  size_t max_units;       // most split-K units of a call: max_batch * Hkv * ceil(max_query_tokens * group / 8)
  int max_n_tiles;        // ceil(max_query_tokens * group / 8)
  cudaEvent_t prof_start; // optional diagnostics events (caller-owned)
  cudaEvent_t prof_end;
  float centroids[256];
  float boundaries[255];
  double c_scale;         // the attention kernels' centroid scale (Geometry::out_scale)
};

namespace {

// Makes `dev` current for the scope and restores the previous device afterwards.
class DeviceScope {
 public:
  explicit DeviceScope(int dev) {
    ok_ = cudaGetDevice(&prev_) == cudaSuccess;
    if (ok_ && dev >= 0 && dev != prev_) {
      ok_ = cudaSetDevice(dev) == cudaSuccess;
      switched_ = ok_;
    }
  }
  ~DeviceScope() {
    if (switched_) cudaSetDevice(prev_);
  }
  bool ok() const { return ok_; }

 private:
  int prev_ = 0;
  bool ok_ = false, switched_ = false;
};

// Lloyd-Max levels of the standard normal with 2^bits levels.  The quantizer is symmetric,
// so only the positive half is iterated: cells [x_{k-1}, x_k) with x_0 = 0 and x_K = inf,
// levels y_k = E[X | cell k] = (phi(x_{k-1}) - phi(x_k)) / (Q(x_{k-1}) - Q(x_k)) with Q the
// upper tail, thresholds x_k = (y_k + y_{k+1}) / 2; repeated until the levels stop moving.
void lloyd_max_positive_half(int levels, double* out_ascending) {
  const int K = levels / 2;
  double y[128], x[129];
  for (int k = 0; k < K; ++k) y[k] = 4.0 * (k + 0.5) / K;
  auto pdf = [](double v) { return std::exp(-0.5 * v * v) * 0.39894228040143267794; };
  auto tail = [](double v) { return 0.5 * std::erfc(v * 0.70710678118654752440); };
  for (int iter = 0; iter < 4000000; ++iter) {
    x[0] = 0.0;
    for (int k = 1; k < K; ++k) x[k] = 0.5 * (y[k - 1] + y[k]);
    double change = 0.0;
    for (int k = 0; k < K; ++k) {
      const double a = x[k];
      const double num = pdf(a) - (k + 1 < K ? pdf(x[k + 1]) : 0.0);
      const double den = tail(a) - (k + 1 < K ? tail(x[k + 1]) : 0.0);
      const double ny = num / den;
      change = std::fmax(change, std::fabs(ny - y[k]));
      y[k] = ny;
    }
    if (change < 1e-15) break;
  }
  for (int k = 0; k < K; ++k) {
    out_ascending[K + k] = y[k];
    out_ascending[K - 1 - k] = -y[k];
  }
}

// The scale S in [1, 2) for which the fp16 images of c_j / S, times S, are closest to the
// centroids c_j (largest relative error over j, smallest over a grid of 2^16 candidates).  fp16
// keeps 11 significant bits; with 2 to 8 distinct magnitudes a common scale brings them much
// closer to exact than S = 1, which the attention kernels then undo in fp32 for free.
double centroid_scale(const float* c, int L) {
  double best_s = 1.0, best_err = 1e30;
  for (int k = 0; k < (1 << 16); ++k) {
    const double s = 1.0 + k / 65536.0;
    double err = 0.0;
    for (int j = 0; j < L && err < best_err; ++j) {
      if (c[j] == 0.f) continue;
      const double h = (double)__half2float(__float2half_rn((float)((double)c[j] / s)));
      err = std::fmax(err, std::fabs(h * s - (double)c[j]) / std::fabs((double)c[j]));
    }
    if (err < best_err) {
      best_err = err;
      best_s = s;
    }
  }
  return best_s;
}

int check_geometry(const rq_config* c) {
  if (c->head_dim <= 0 || c->num_q_heads <= 0 || c->num_kv_heads <= 0 || c->page_size <= 0 || c->num_pages <= 0 ||
      c->max_batch <= 0 || c->max_query_tokens <= 0 || c->max_pages_per_seq <= 0)
    return RQ_ERR_INVALID;
  if (c->num_q_heads % c->num_kv_heads != 0) return RQ_ERR_INVALID;
  if (c->mode != RQ_PLANAR && c->mode != RQ_ISO && c->mode != RQ_DENSE) return RQ_ERR_INVALID;
  if (!c->rot_k || !c->rot_v) return RQ_ERR_INVALID;
  if (c->head_dim != rq::kHeadDim) return RQ_ERR_UNSUPPORTED;
  if (c->bits < 2 || c->bits > 4) return RQ_ERR_UNSUPPORTED;
  if (c->page_size % 16 != 0 || c->page_size > 256) return RQ_ERR_UNSUPPORTED;
  if ((long long)c->num_pages * c->page_size > INT32_MAX) return RQ_ERR_UNSUPPORTED;
  if ((long long)c->max_pages_per_seq * c->page_size > INT32_MAX) return RQ_ERR_UNSUPPORTED;  // positions are int
  // one page's chunks of all kv heads stay below 2^31 bytes (32-bit page strides in the kernels)
  if ((long long)c->num_kv_heads * c->page_size * (2 * 16 * c->bits + 4) > INT32_MAX) return RQ_ERR_UNSUPPORTED;
  if (c->max_batch > rq::kMaxBatch) return RQ_ERR_UNSUPPORTED;
  if (!(c->sm_scale >= 0.0f) || std::isinf(c->sm_scale)) return RQ_ERR_INVALID;
  return RQ_OK;
}

int to_status(cudaError_t e) { return e == cudaSuccess ? RQ_OK : RQ_ERR_CUDA; }

}  // namespace

extern "C" {

const char* rq_status_string(int status) {
  switch (status) {
    case RQ_OK: return "ok";
    case RQ_ERR_INVALID: return "invalid argument";
    case RQ_ERR_UNSUPPORTED: return "unsupported configuration";
    case RQ_ERR_CUDA: return "CUDA error";
    case RQ_ERR_CAPACITY: return "above the context's capacity";
    default: return "unknown status";
  }
}

int rq_lloyd_max_codebook(int bits, int head_dim, float* centroids) {
  if (bits < 1 || bits > 8 || head_dim < 1 || !centroids) return RQ_ERR_INVALID;
  const int L = 1 << bits;
  double c[256];
  lloyd_max_positive_half(L, c);
  const double s = 1.0 / std::sqrt((double)head_dim);
  for (int j = 0; j < L; ++j) centroids[j] = (float)(c[j] * s);
  return RQ_OK;
}

// The binned code table of boundaries bnd[0 .. nb - 1] (ascending): bin n = k - kCodeBinHalf
// holds every u with RNE(u * kCodeBinScale) = n, i.e. u in [(n - 1/2) / scale, (n + 1/2) /
// scale]; widened by 2e-5 on each side it may hold one boundary at most, else there is no table.
static bool build_code_table(const float* bnd, int nb, uint32_t* tab) {
  const double ext = 2e-5;
  for (int k = 0; k + 1 < rq::kCodeBins; ++k) {
    const int n = k - rq::kCodeBinHalf;
    const double lo = (n - 0.5) / rq::kCodeBinScale - ext, hi = (n + 0.5) / rq::kCodeBinScale + ext;
    uint32_t below = 0;
    int inside = 0;
    float near = INFINITY;
    for (int j = 0; j < nb; ++j) {
      if ((double)bnd[j] < lo) {
        ++below;
      } else if ((double)bnd[j] <= hi) {
        ++inside;
        near = bnd[j];
      }
    }
    if (inside > 1) return false;
    tab[2 * k] = below;
    std::memcpy(&tab[2 * k + 1], &near, 4);
  }
  const float inf = INFINITY;
  tab[2 * (rq::kCodeBins - 1)] = 0u;
  std::memcpy(&tab[2 * (rq::kCodeBins - 1) + 1], &inf, 4);
  return true;
}

int rq_create(rq_ctx** out, const rq_config* cfg) {
  if (!out) return RQ_ERR_INVALID;
  *out = nullptr;
  if (!cfg) return RQ_ERR_INVALID;
  int st = check_geometry(cfg);
  if (st != RQ_OK) return st;

  rq_ctx* ctx = new (std::nothrow) rq_ctx();
  if (!ctx) return RQ_ERR_CUDA;
  ctx->cfg = *cfg;
  const int L = 1 << cfg->bits;
  if (cfg->codebook) {
    for (int j = 0; j < L; ++j) {
      if (!std::isfinite(cfg->codebook[j]) || (j > 0 && !(cfg->codebook[j] > cfg->codebook[j - 1]))) {
        delete ctx;
        return RQ_ERR_INVALID;
      }
      ctx->centroids[j] = cfg->codebook[j];
    }
  } else {
    rq_lloyd_max_codebook(cfg->bits, cfg->head_dim, ctx->centroids);
  }
  for (int j = 0; j + 1 < L; ++j)
    ctx->boundaries[j] = (float)(0.5 * ((double)ctx->centroids[j] + (double)ctx->centroids[j + 1]));
  ctx->cfg.rot_k = ctx->cfg.rot_v = ctx->cfg.codebook = nullptr;

  int dev = cfg->device;
  if (dev < 0 && cudaGetDevice(&dev) != cudaSuccess) {
    delete ctx;
    return RQ_ERR_CUDA;
  }
  ctx->device = dev;
  DeviceScope scope(dev);
  if (!scope.ok() || cudaDeviceGetAttribute(&ctx->num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    delete ctx;
    return RQ_ERR_CUDA;
  }

  const int hkv = cfg->num_kv_heads, d = cfg->head_dim;
  const bool dense = cfg->mode == RQ_DENSE;
  const size_t rot = (size_t)hkv * d * (dense ? d : 1);
  const size_t table_floats = 2 * rot + 256 + 256;
  const int group = cfg->num_q_heads / hkv;
  ctx->max_n_tiles = (cfg->max_query_tokens * group + 7) / 8;
  // one partial slot per fragment: at most units + CTAs of them (stream-K split); a unit covers
  // up to 3 n-tiles of a kv head, so the largest workspace is taken over every T the context
  // allows (and over the one-n-tile units of a decode step)
  ctx->max_units = 0;
  ctx->ws_floats = 0;
  for (int nt = 1; nt <= ctx->max_n_tiles; ++nt)
    for (int step = 0; step < 2; ++step) {
      long long units = 0, floats = 0;
      rq::attention_workspace(cfg->max_batch, hkv, nt, step != 0, ctx->num_sms, &units, &floats);
      if ((size_t)units > ctx->max_units) ctx->max_units = (size_t)units;
      if ((size_t)floats > ctx->ws_floats) ctx->ws_floats = (size_t)floats;
    }

  cudaError_t e = cudaMalloc(&ctx->d_tables, table_floats * sizeof(float));
  if (e == cudaSuccess) e = cudaMalloc(&ctx->d_ws, ctx->ws_floats * sizeof(float));
  if (e == cudaSuccess) e = cudaMalloc(&ctx->d_frag, 3 * ctx->max_units * sizeof(int));
  // the per-unit round counters start at zero; every launch leaves them at zero
  if (e == cudaSuccess) e = cudaMemset(ctx->d_frag, 0, 3 * ctx->max_units * sizeof(int));
  const size_t dense16_halves = dense ? 2 * rot * 2 : 0;  // [K, V][Hkv][hi, lo][d][d]
  if (e == cudaSuccess && dense) {
    e = cudaMalloc(&ctx->d_dense16, dense16_halves * sizeof(__half));
    if (e == cudaSuccess) e = cudaMalloc(&ctx->d_dense32, 3 * rot * sizeof(float));  // R_k, R_v, R_v^T
    if (e == cudaSuccess) e = cudaMalloc(&ctx->d_rotq, rot * sizeof(uint32_t));  // 4 words per 4 entries
    if (e == cudaSuccess) e = cudaMemcpy(ctx->d_dense32, cfg->rot_k, rot * sizeof(float), cudaMemcpyHostToDevice);
    if (e == cudaSuccess)
      e = cudaMemcpy(ctx->d_dense32 + rot, cfg->rot_v, rot * sizeof(float), cudaMemcpyHostToDevice);
    if (e == cudaSuccess) {
      std::vector<float> vt(rot);
      for (int h = 0; h < hkv; ++h)
        for (int i = 0; i < d; ++i)
          for (int m = 0; m < d; ++m) vt[((size_t)h * d + m) * d + i] = cfg->rot_v[((size_t)h * d + i) * d + m];
      e = cudaMemcpy(ctx->d_dense32 + 2 * rot, vt.data(), rot * sizeof(float), cudaMemcpyHostToDevice);
    }
    if (e == cudaSuccess)
      e = cudaMalloc(&ctx->d_qrot, (size_t)cfg->max_batch * cfg->max_query_tokens * cfg->num_q_heads * d * sizeof(float));
  }
  float* host = nullptr;
  __half* host16 = nullptr;
  if (e == cudaSuccess) {
    host = (float*)std::calloc(table_floats, sizeof(float));
    if (dense) host16 = (__half*)std::calloc(dense16_halves, sizeof(__half));
    if (!host || (dense && !host16)) e = cudaErrorMemoryAllocation;
  }
  if (e == cudaSuccess) {
    if (dense) {
      // rot_k is kept transposed (the query rotation walks it by columns), rot_v as given, and
      // both are split into fp16 hi + lo for the append's tensor-core GEMM.
      for (int h = 0; h < hkv; ++h)
        for (int i = 0; i < d; ++i)
          for (int m = 0; m < d; ++m) host[((size_t)h * d + m) * d + i] = cfg->rot_k[((size_t)h * d + i) * d + m];
      std::memcpy(host + rot, cfg->rot_v, rot * sizeof(float));
      for (int kind = 0; kind < 2; ++kind) {
        const float* R = kind ? cfg->rot_v : cfg->rot_k;
        for (int h = 0; h < hkv; ++h)
          for (size_t e2 = 0; e2 < (size_t)d * d; ++e2) {
            const double x = (double)R[(size_t)h * d * d + e2];
            const __half hi = __double2half(x);
            const __half lo = __double2half(x - (double)__half2float(hi));
            __half* dst = host16 + (((size_t)kind * hkv + h) * 2) * d * d;
            dst[e2] = hi;
            dst[(size_t)d * d + e2] = lo;
          }
      }
      e = cudaMemcpy(ctx->d_dense16, host16, dense16_halves * sizeof(__half), cudaMemcpyHostToDevice);
      // the same halves of R_k as the query rotation's MMA B operands: per kv head, k-step ks,
      // n-tile nt and lane 4g + t, output dim n = 8 nt + g and input dims m = 32t + 4ks .. m + 3
      std::vector<uint32_t> words(rot);
      auto half_bits = [&](int part, int h, int n, int m) {
        uint16_t b;
        std::memcpy(&b, host16 + (((size_t)h * 2 + part) * d + n) * d + m, 2);
        return (uint32_t)b;
      };
      for (int h = 0; h < hkv; ++h)
        for (int ks = 0; ks < 8; ++ks)
          for (int nt = 0; nt < 16; ++nt)
            for (int lane = 0; lane < 32; ++lane) {
              const int n = 8 * nt + lane / 4, m = 32 * (lane % 4) + 4 * ks;
              uint32_t* w = words.data() + ((((size_t)h * 8 + ks) * 16 + nt) * 32 + lane) * 4;
              for (int part = 0; part < 2; ++part) {
                w[2 * part] = half_bits(part, h, n, m) | half_bits(part, h, n, m + 1) << 16;
                w[2 * part + 1] = half_bits(part, h, n, m + 2) | half_bits(part, h, n, m + 3) << 16;
              }
            }
      if (e == cudaSuccess) e = cudaMemcpy(ctx->d_rotq, words.data(), rot * sizeof(uint32_t), cudaMemcpyHostToDevice);
    } else {
      std::memcpy(host, cfg->rot_k, rot * sizeof(float));
      std::memcpy(host + rot, cfg->rot_v, rot * sizeof(float));
    }
    ctx->c_scale = centroid_scale(ctx->centroids, L);
    for (int j = 0; j < L; ++j) host[2 * rot + j] = (float)((double)ctx->centroids[j] / ctx->c_scale);
    std::memcpy(host + 2 * rot + 256, ctx->boundaries, (L - 1) * sizeof(float));
    if (e == cudaSuccess) e = cudaMemcpy(ctx->d_tables, host, table_floats * sizeof(float), cudaMemcpyHostToDevice);
  }
  std::free(host);
  std::free(host16);
  if (e == cudaSuccess) {
    std::vector<uint32_t> tab(2 * rq::kCodeBins);
    if (build_code_table(ctx->boundaries, L - 1, tab.data())) {
      e = cudaMalloc(&ctx->d_codetab, tab.size() * sizeof(uint32_t));
      if (e == cudaSuccess)
        e = cudaMemcpy(ctx->d_codetab, tab.data(), tab.size() * sizeof(uint32_t), cudaMemcpyHostToDevice);
    }
  }
  if (e == cudaSuccess) e = rq::attention_prepare();
  if (e == cudaSuccess) e = rq::append_prepare();
  if (e == cudaSuccess) e = rq::extend_prepare();
  if (e != cudaSuccess) {
    cudaFree(ctx->d_tables);
    cudaFree(ctx->d_ws);
    cudaFree(ctx->d_frag);
    cudaFree(ctx->d_dense16);
    cudaFree(ctx->d_dense32);
    cudaFree(ctx->d_rotq);
    cudaFree(ctx->d_codetab);
    cudaFree(ctx->d_qrot);
    delete ctx;
    return RQ_ERR_CUDA;
  }

  rq::Geometry& g = ctx->g;
  g.num_q_heads = cfg->num_q_heads;
  g.num_kv_heads = hkv;
  g.group = group;
  g.bits = cfg->bits;
  g.mode = cfg->mode;
  g.page_size = cfg->page_size;
  g.num_pages = cfg->num_pages;
  g.vec_bytes = d * cfg->bits / 8;
  g.page_bytes = cfg->page_size * (2 * g.vec_bytes + 4);
  const float scale = cfg->sm_scale > 0.f ? cfg->sm_scale : (float)(1.0 / std::sqrt((double)d));
  g.q_scale = (float)(scale * 1.44269504088896340736 * ctx->c_scale);
  g.out_scale = (float)ctx->c_scale;
  g.rot_k = ctx->d_tables;
  g.rot_v = ctx->d_tables + rot;
  g.dense16 = ctx->d_dense16;
  g.dense32 = ctx->d_dense32;
  g.rotq = ctx->d_rotq;
  g.rot_vt = dense ? ctx->d_dense32 + 2 * rot : nullptr;
  g.code_table = ctx->d_codetab;
  g.centroids = ctx->d_tables + 2 * rot;  // c / c_scale
  g.boundaries = ctx->d_tables + 2 * rot + 256;
  *out = ctx;
  return RQ_OK;
}

void rq_free(rq_ctx* ctx) {
  if (!ctx) return;
  {
    DeviceScope scope(ctx->device);
    cudaFree(ctx->d_tables);
    cudaFree(ctx->d_ws);
    cudaFree(ctx->d_frag);
    cudaFree(ctx->d_dense16);
    cudaFree(ctx->d_dense32);
    cudaFree(ctx->d_rotq);
    cudaFree(ctx->d_codetab);
    cudaFree(ctx->d_qrot);
  }
  delete ctx;
}

int rq_set_profile_events(rq_ctx* ctx, void* ev_start, void* ev_end) {
  if (!ctx || (!ev_start) != (!ev_end)) return RQ_ERR_INVALID;
  ctx->prof_start = (cudaEvent_t)ev_start;
  ctx->prof_end = (cudaEvent_t)ev_end;
  return RQ_OK;
}

size_t rq_page_bytes(const rq_ctx* ctx) { return ctx ? (size_t)ctx->g.page_bytes : 0; }

int rq_get_codebook(const rq_ctx* ctx, float* centroids, float* boundaries) {
  if (!ctx) return RQ_ERR_INVALID;
  const int L = 1 << ctx->g.bits;
  if (centroids) std::memcpy(centroids, ctx->centroids, L * sizeof(float));
  if (boundaries) std::memcpy(boundaries, ctx->boundaries, (L - 1) * sizeof(float));
  return RQ_OK;
}

int rq_quantize_append(rq_ctx* ctx, const void* k, const void* v, const int32_t* slot_mapping, int n,
                       void* kv_pages, int32_t* d_status, void* stream) {
  if (!ctx || n < 0) return RQ_ERR_INVALID;
  if (n == 0) return RQ_OK;
  if (!k || !v || !slot_mapping || !kv_pages) return RQ_ERR_INVALID;
  if ((uintptr_t)k % 16 != 0 || (uintptr_t)v % 16 != 0 || (uintptr_t)kv_pages % 16 != 0)
    return RQ_ERR_INVALID;  // 16-byte vector loads and stores
  DeviceScope scope(ctx->device);
  if (!scope.ok()) return RQ_ERR_CUDA;
  return to_status(rq::launch_append(ctx->g, k, v, slot_mapping, n, (uint8_t*)kv_pages, d_status,
                                     (cudaStream_t)stream));
}

static bool misaligned16(const void* p) { return (uintptr_t)p % 16 != 0; }

static int attention_call(rq_ctx* ctx, const void* q, int T, const uint64_t* tree_mask, const void* kv_pages,
                          const int32_t* block_table, int max_pages, const int32_t* seq_lens, int B, void* out,
                          int32_t* d_status, void* stream, const void* k_new = nullptr, const void* v_new = nullptr) {
  if (!ctx || B < 0 || T < 1 || max_pages < 1) return RQ_ERR_INVALID;
  if (B == 0) return RQ_OK;
  if (!q || !kv_pages || !block_table || !seq_lens || !out) return RQ_ERR_INVALID;
  if (misaligned16(q) || misaligned16(kv_pages) || misaligned16(out)) return RQ_ERR_INVALID;  // bulk copies, vector I/O
  if (B > ctx->cfg.max_batch || T > ctx->cfg.max_query_tokens || max_pages > ctx->cfg.max_pages_per_seq)
    return RQ_ERR_CAPACITY;
  DeviceScope scope(ctx->device);
  if (!scope.ok()) return RQ_ERR_CUDA;

  rq::AttnArgs a;
  a.q = q;
  a.pages = (const uint8_t*)kv_pages;
  a.block_table = block_table;
  a.max_pages = max_pages;
  a.seq_lens = seq_lens;
  a.B = B;
  a.T = T;
  a.out = out;
  a.status = d_status;
  a.tree_mask = tree_mask;
  a.q_rot = ctx->d_qrot;  // null unless dense
  a.k_new = (const __half*)k_new;
  a.v_new = (const __half*)v_new;
  a.ws = ctx->d_ws;
  a.rows = T * ctx->g.group;
  a.n_tiles_n = (a.rows + 7) / 8;
  a.nt = rq::attention_unit_tiles(a.n_tiles_n, k_new != nullptr);
  a.frag = ctx->d_frag;
  a.cnt = ctx->d_frag + 2 * ctx->max_units;
  a.grid = ctx->num_sms;  // one CTA per SM, each an equal share of the tiles
  return to_status(rq::launch_attention(ctx->g, a, (cudaStream_t)stream, ctx->prof_start, ctx->prof_end));
}

int rq_verify_attention(rq_ctx* ctx, const void* q, int T, const void* kv_pages, const int32_t* block_table,
                        int max_pages, const int32_t* seq_lens, int B, void* out, int32_t* d_status, void* stream) {
  return attention_call(ctx, q, T, nullptr, kv_pages, block_table, max_pages, seq_lens, B, out, d_status, stream);
}

int rq_tree_verify_attention(rq_ctx* ctx, const void* q, int T, const uint64_t* tree_mask, const void* kv_pages,
                             const int32_t* block_table, int max_pages, const int32_t* seq_lens, int B, void* out,
                             int32_t* d_status, void* stream) {
  if (T > 64 || (B > 0 && !tree_mask)) return RQ_ERR_INVALID;
  return attention_call(ctx, q, T, tree_mask, kv_pages, block_table, max_pages, seq_lens, B, out, d_status, stream);
}

int rq_extend_attention(rq_ctx* ctx, const void* q, int T, const void* kv_pages, const int32_t* block_table,
                        int max_pages, const int32_t* seq_lens, int B, void* out, int32_t* d_status, void* stream) {
  if (!ctx || B < 0 || T < 1 || max_pages < 1) return RQ_ERR_INVALID;
  if (B == 0) return RQ_OK;
  if (!q || !kv_pages || !block_table || !seq_lens || !out) return RQ_ERR_INVALID;
  if (misaligned16(q) || misaligned16(kv_pages) || misaligned16(out)) return RQ_ERR_INVALID;  // vector loads, stores
  if (B > ctx->cfg.max_batch || max_pages > ctx->cfg.max_pages_per_seq) return RQ_ERR_CAPACITY;
  // a dense rotation's queries are rotated into the context's workspace first
  if (ctx->g.mode == RQ_DENSE && T > ctx->cfg.max_query_tokens) return RQ_ERR_CAPACITY;
  if ((long long)T * ctx->g.group > INT32_MAX / 2) return RQ_ERR_CAPACITY;
  DeviceScope scope(ctx->device);
  if (!scope.ok()) return RQ_ERR_CUDA;
  rq::AttnArgs a{};
  a.q = q;
  a.pages = (const uint8_t*)kv_pages;
  a.block_table = block_table;
  a.max_pages = max_pages;
  a.seq_lens = seq_lens;
  a.B = B;
  a.T = T;
  a.out = out;
  a.status = d_status;
  a.rows = T * ctx->g.group;
  a.q_rot = ctx->d_qrot;  // null unless dense
  return to_status(rq::launch_extend(ctx->g, a, (cudaStream_t)stream, ctx->prof_start, ctx->prof_end));
}

int rq_decode_step(rq_ctx* ctx, const void* q, const void* k_new, const void* v_new, void* kv_pages,
                   const int32_t* block_table, int max_pages, const int32_t* seq_lens, int B, void* out, int32_t* d_status,
                   void* stream) {
  if (!ctx) return RQ_ERR_INVALID;
  if (B > 0 && (!k_new || !v_new || (uintptr_t)k_new % 16 != 0 || (uintptr_t)v_new % 16 != 0)) return RQ_ERR_INVALID;
  return attention_call(ctx, q, 1, nullptr, kv_pages, block_table, max_pages, seq_lens, B, out, d_status, stream, k_new,
                        v_new);
}

int rq_decode_attention(rq_ctx* ctx, const void* q, const void* kv_pages, const int32_t* block_table, int max_pages,
                        const int32_t* seq_lens, int B, void* out, int32_t* d_status, void* stream) {
  return attention_call(ctx, q, 1, nullptr, kv_pages, block_table, max_pages, seq_lens, B, out, d_status, stream);
}

}  // extern "C"
