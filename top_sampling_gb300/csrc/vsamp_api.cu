// Host side of libvsamp.so: argument checks, per-device limits, launch geometry (cluster size, vectors
// per thread) and the extern "C" entry points declared in include/vsamp.h.
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "vsamp_host.h"
#include "vsamp_split.cuh"

namespace vsamp {

constexpr int kMaxDevices = 64;

static DeviceInfo g_dev[kMaxDevices];
static std::mutex g_mu;

int env_int(const char* name, int dflt) {
  const char* v = std::getenv(name);
  if (!v || !*v) return dflt;
  return std::atoi(v);
}

long long env_ll(const char* name, long long dflt) {
  const char* v = std::getenv(name);
  if (!v || !*v) return dflt;
  return std::strtoll(v, nullptr, 10);
}

int cached_max_clusters(const void* kern, int threads, int smem, int C) {
  struct Entry {
    int dev;
    const void* kern;
    int threads, smem, C, n;
  };
  static Entry cache[256];
  static int used = 0;
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  std::lock_guard<std::mutex> lk(mu);
  // the kernel's shared-memory limit only ever grows, so every launch seen so far stays valid
  int limit = 0;
  for (int i = 0; i < used; ++i)
    if (cache[i].dev == dev && cache[i].kern == kern && cache[i].smem > limit) limit = cache[i].smem;
  for (int i = 0; i < used; ++i) {
    const Entry& e = cache[i];
    if (e.dev == dev && e.kern == kern && e.threads == threads && e.smem == smem && e.C == C) return e.n;
  }
  if ((smem > limit && cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) ||
      (C > 8 && cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)) {
    cudaGetLastError();
    return 0;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3((unsigned)threads, 1, 1);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.gridDim = dim3((unsigned)C, 1, 1);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
    cudaGetLastError();
    n = 0;
  }
  if (used < 256) cache[used++] = Entry{dev, kern, threads, smem, C, n};
  return n;
}

vsamp_status device_info(int dev, DeviceInfo& out) {
  if (dev < 0 || dev >= kMaxDevices) return VSAMP_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.ready) {
    if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) {
      cudaGetLastError();
      return VSAMP_ERR_CUDA;
    }
    cudaDeviceGetAttribute(&d.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
    int cl = 0;
    cudaDeviceGetAttribute(&cl, cudaDevAttrClusterLaunch, dev);
    cudaGetLastError();
    d.max_cluster = cl ? 16 : 1;
    // a smaller opt-in can be simulated for tests of the capacity checks
    const int ov = env_int("VSAMP_SMEM_OPTIN_OVERRIDE", 0);
    if (ov > 0 && ov < d.optin) d.optin = ov;
    d.ready = 1;
  }
  out = d;
  return VSAMP_OK;
}

// Launch geometry. A row spans C CTAs (one cluster); each CTA holds NT * q 16-byte vectors of it in
// shared memory. The per-CTA budget keeps `per_sm` CTAs resident on an SM. Among the
// cluster sizes whose slices fit, the one with the least padding is taken (q odd when that costs at
// most an eighth: conflict-free 16-byte shared-memory loads); small batches spread rows over more CTAs.
vsamp_status choose_geometry(int64_t V, int esize, int64_t B, const DeviceInfo& d, Geometry& g) {
  const int NT = env_int("VSAMP_THREADS", 256) == 128 ? kThreadsSmall : kThreadsLarge;
  const int head = NT == kThreadsSmall ? slice_offset<kThreadsSmall>() : slice_offset<kThreadsLarge>();
  const int per_sm = env_int("VSAMP_CTAS_PER_SM", NT == kThreadsSmall ? 5 : 3);
  return choose_geometry_for(V, esize, B, d, NT, head, per_sm, g);
}

vsamp_status choose_geometry_for(int64_t V, int esize, int64_t B, const DeviceInfo& d, int NT, int head, int per_sm,
                                 Geometry& g, int max_nbuf, int max_spread) {
  const int64_t VE = 16 / esize;
  const int64_t nvec = (V + VE - 1) / VE;
  const int smem_sm = d.smem_per_sm > 0 ? d.smem_per_sm : d.optin;
  const int odd = env_int("VSAMP_ODD_Q", 1);
  const int forced = env_int("VSAMP_CLUSTER", 0);
  auto q_for = [&](int C) {
    int64_t q = (nvec + (int64_t)C * NT - 1) / ((int64_t)C * NT);
    if (q < 1) q = 1;
    if (odd && (q & 1) == 0 && (q + 1) * 8 <= q * 9) ++q;
    return q;
  };
  const int64_t cap1 = (int64_t)d.optin - head;                       // one buffer, one CTA per SM
  for (int nbuf = max_nbuf; nbuf >= 1; --nbuf) {
    int64_t budget = ((int64_t)smem_sm / (per_sm > 0 ? per_sm : 1) - 1024 - head) / nbuf;
    if (budget * nbuf > cap1) budget = cap1 / nbuf;
    int C = 0;
    if (forced > 0) {
      if (forced <= d.max_cluster && (int64_t)NT * q_for(forced) * 16 * nbuf <= cap1) C = forced;
    } else {
      int cmin = 0;
      for (int c = 1; c <= d.max_cluster; ++c)
        if ((int64_t)NT * q_for(c) * 16 <= budget) { cmin = c; break; }
      if (!cmin && nbuf == 1) {
        for (int c = 1; c <= d.max_cluster; ++c)
          if ((int64_t)NT * q_for(c) * 16 <= cap1) { cmin = c; break; }
      }
      if (cmin) {
        C = cmin;
        int64_t best = (int64_t)cmin * q_for(cmin);
        for (int c = cmin + 1; c <= cmin + 3 && c <= d.max_cluster; ++c)
          if ((int64_t)c * q_for(c) < best) { best = (int64_t)c * q_for(c); C = c; }
        // small batches: more CTAs per row while slices stay >= 8 KB
        while (C < d.max_cluster && C < max_spread && B * C < 2LL * d.sm_count &&
               (int64_t)NT * q_for(C + 1) * 16 >= 8192)
          ++C;
      }
    }
    if (!C) continue;
    // a second buffer only pays when clusters have more than one row to stream
    if (nbuf > 1 && forced <= 0 && B * C < 3LL * d.sm_count * (per_sm > 0 ? per_sm : 1) / 2) continue;
    g.NT = NT;
    g.C = C;
    g.q = (int)q_for(C);
    g.nbuf = nbuf;
    g.smem = head + nbuf * NT * g.q * 16;
    return VSAMP_OK;
  }
  return VSAMP_ERR_UNSUPPORTED;
}

template <int MODE>
static vsamp_status dispatch(Params p, vsamp_dtype dt, int64_t B, cudaStream_t s) {
  if (dt == VSAMP_F32) return launch<float, MODE>(p, B, 4, s);
  if (dt == VSAMP_BF16) return launch<__nv_bfloat16, MODE>(p, B, 2, s);
  return VSAMP_ERR_INVALID_ARG;
}

// Row statistics (MODE_LSE, MODE_LOGPROB): the streaming piece kernel, or the cluster row kernel for rows longer
// than it takes (VSAMP_STATS_ROW=1 forces the row kernel)
template <int MODE>
static vsamp_status dispatch_stats(Params p, vsamp_dtype dt, int64_t B, cudaStream_t s) {
  if (env_int("VSAMP_STATS_ROW", 0) == 0) {
    vsamp_status st = VSAMP_ERR_UNSUPPORTED;
    if (dt == VSAMP_F32) st = launch_stats<float, MODE>(p, B, 4, s);
    else if (dt == VSAMP_BF16) st = launch_stats<__nv_bfloat16, MODE>(p, B, 2, s);
    if (st != VSAMP_ERR_UNSUPPORTED) return st;
  }
  return dispatch<MODE>(p, dt, B, s);
}

static bool aligned16(const void* ptr, int64_t ld, int esize) {
  return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0 && ((ld * esize) & 15) == 0;
}

static vsamp_status check_common(const void* x, vsamp_dtype dt, int64_t B, int64_t V, int64_t ld) {
  if (!x) return VSAMP_ERR_INVALID_ARG;
  if (dt != VSAMP_F32 && dt != VSAMP_BF16) return VSAMP_ERR_INVALID_ARG;
  if (B <= 0 || V <= 0 || ld < V) return VSAMP_ERR_INVALID_ARG;
  if (V > 0x7FFFFFF0LL) return VSAMP_ERR_UNSUPPORTED;
  return VSAMP_OK;
}

static Params base_params(const void* x, vsamp_dtype dt, int64_t B, int64_t V, int64_t ld) {
  Params p;
  std::memset(&p, 0, sizeof(p));
  p.x = static_cast<const unsigned char*>(x);
  p.B = B;
  p.V = V;
  p.ld = ld;
  const int es = dt == VSAMP_F32 ? 4 : 2;
  p.tma = aligned16(x, ld, es) && env_int("VSAMP_NO_TMA", 0) == 0;
  return p;
}

// Log-probability from given statistics: one thread per row.
template <typename T>
__global__ void logprob_from_stats_kernel(const unsigned char* x, int64_t B, int64_t V, int64_t ld,
                                          const float* temperature, const int32_t* token, const float* row_max,
                                          const float* row_logsum, float* out, int32_t* row_status) {
  const int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= B) return;
  const int32_t tk = token[r];
  const float temp = temperature ? temperature[r] : 1.f;
  int st = VSAMP_OK;
  float lp = __int_as_float(0x7FC00000);
  if (tk < 0 || (int64_t)tk >= V || isnan(temp) || isinf(temp)) {
    st = VSAMP_ERR_INVALID_ARG;
  } else {
    const float Teff = temp > 0.f ? temp : 1.f;
    const float xt = Traits<T>::load_global(x, r * ld + tk);
    const float m = row_max[r], ls = row_logsum[r];
    if (!isfinite(xt) || !isfinite(m) || !isfinite(ls)) {
      st = VSAMP_ERR_NONFINITE;
    } else {
      const double s = (double)((xt - m) * (1.f / Teff));
      lp = (float)fmin(s - (double)ls, 0.0);
    }
  }
  out[r] = lp;
  if (row_status) row_status[r] = st;
}

// Top-N log-probability lists from a top-N select (indices in ascending order) and the row statistics: one
// CTA per row, grid-stride over rows. A token's place in the list is the number of listed tokens before it
// in the order (logit descending, index ascending); equal logits keep their ascending index order.
constexpr int kTopnThreads = 256;

template <typename T>
__global__ void __launch_bounds__(kTopnThreads) topn_rank_kernel(const unsigned char* x, int64_t B, int64_t V,
                                                                 int64_t ld, const float* temperature, int32_t N,
                                                                 const float* row_max, const float* row_logsum,
                                                                 int32_t* out_idx, float* out_lp) {
  extern __shared__ float topn_smem[];
  float* sv = topn_smem;                                        // [N] logits of the listed tokens
  int32_t* si = reinterpret_cast<int32_t*>(topn_smem + N);      // [N] their indices
  const int n = (int)(V < (int64_t)N ? V : (int64_t)N);
  const float qnan = __int_as_float(0x7FC00000);
  for (int64_t r = blockIdx.x; r < B; r += gridDim.x) {
    int32_t* oi = out_idx + r * N;
    float* ol = out_lp + r * N;
    const float m = row_max[r], ls = row_logsum[r];
    if (!(isfinite(m) && isfinite(ls))) {   // the statistics of an error row are NaN: an empty list
      for (int j = threadIdx.x; j < N; j += blockDim.x) {
        oi[j] = -1;
        ol[j] = qnan;
      }
      continue;
    }
    const float temp = temperature ? temperature[r] : 1.f;
    const float invT = 1.f / (temp > 0.f ? temp : 1.f);
    for (int j = threadIdx.x; j < n; j += blockDim.x) {
      const int32_t v = oi[j];
      si[j] = v;
      sv[j] = (v >= 0 && (int64_t)v < V) ? Traits<T>::load_global(x, r * ld + v) : -INFINITY;
    }
    __syncthreads();
    for (int j = threadIdx.x; j < n; j += blockDim.x) {
      const float xj = sv[j];
      int rank = 0;
      for (int i = 0; i < n; ++i) {
        const float xi = sv[i];
        rank += (xi > xj || (xi == xj && i < j)) ? 1 : 0;
      }
      oi[rank] = si[j];
      ol[rank] = (float)fmin((double)((xj - m) * invT) - (double)ls, 0.0);
    }
    for (int j = n + threadIdx.x; j < N; j += blockDim.x) {
      oi[j] = -1;
      ol[j] = qnan;
    }
    __syncthreads();   // the next row reuses the shared arrays
  }
}

}  // namespace vsamp

namespace vsamp {

// vsamp_sample_static's workspace: a fixed array in this module's device memory, so that call allocates
// nothing. Its address on each device is looked up once, with that device current.
static __device__ __align__(256) unsigned char g_static_scratch[VSAMP_STATIC_SCRATCH_BYTES];
static void* g_static_ptr[kMaxDevices];   // guarded by g_mu

static vsamp_status static_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return VSAMP_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return VSAMP_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_static_ptr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress((void**)&ptr, g_static_scratch) != cudaSuccess || !ptr) {
      cudaGetLastError();
      return VSAMP_ERR_CUDA;
    }
    g_static_ptr[dev] = ptr;
  }
  *out = g_static_ptr[dev];
  return VSAMP_OK;
}

}  // namespace vsamp

using namespace vsamp;

extern "C" {

vsamp_status vsamp_softmax_lse(const void* logits, vsamp_dtype dt, int64_t B, int64_t V, int64_t ld,
                               const float* temperature, float* row_max, float* row_logsum,
                               int32_t* row_status, void* stream) {
  vsamp_status st = check_common(logits, dt, B, V, ld);
  if (st != VSAMP_OK) return st;
  Params p = base_params(logits, dt, B, V, ld);
  p.temperature = temperature;
  p.row_max = row_max;
  p.row_logsum = row_logsum;
  p.row_status = row_status;
  return dispatch_stats<MODE_LSE>(p, dt, B, static_cast<cudaStream_t>(stream));
}

vsamp_status vsamp_topk_select(const void* scores, vsamp_dtype dt, int64_t B, int64_t max_len, int64_t ld,
                               const int32_t* lengths, const int32_t* k, int32_t k_max, int32_t* out_idx,
                               int32_t* row_status, void* stream) {
  vsamp_status st = check_common(scores, dt, B, max_len, ld);
  if (st != VSAMP_OK) return st;
  if (!out_idx || k_max <= 0) return VSAMP_ERR_INVALID_ARG;
  Params p = base_params(scores, dt, B, max_len, ld);
  p.lengths = lengths;
  p.k_sel = k;
  p.k_max = k_max;
  p.out_idx = out_idx;
  p.row_status = row_status;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // rows that a cluster cannot hold on chip (or VSAMP_SELECT_STREAM=1) take the uncached path
  if (env_int("VSAMP_SELECT_STREAM", 0) == 0) {
    st = dispatch<MODE_SELECT>(p, dt, B, s);
    if (st != VSAMP_ERR_UNSUPPORTED) return st;
  }
  if (dt == VSAMP_F32) return launch_select_stream<float>(p, B, s);
  return launch_select_stream<__nv_bfloat16>(p, B, s);
}

vsamp_status vsamp_topp_minp_mask(const void* logits, vsamp_dtype dt, int64_t B, int64_t V, int64_t ld,
                                  const float* temperature, const int32_t* top_k, const float* top_p,
                                  const float* min_p, vsamp_cut* cut, uint8_t* mask, int32_t* stats,
                                  void* stream) {
  vsamp_status st = check_common(logits, dt, B, V, ld);
  if (st != VSAMP_OK) return st;
  if (!cut) return VSAMP_ERR_INVALID_ARG;
  Params p = base_params(logits, dt, B, V, ld);
  p.temperature = temperature;
  p.top_k = top_k;
  p.top_p = top_p;
  p.min_p = min_p;
  p.cut = cut;
  p.mask = mask;
  p.stats = stats;
  if (mask) return dispatch<MODE_CUT | MODE_MASK>(p, dt, B, static_cast<cudaStream_t>(stream));
  return dispatch<MODE_CUT>(p, dt, B, static_cast<cudaStream_t>(stream));
}

vsamp_status vsamp_sample(const void* logits, vsamp_dtype dt, int64_t B, int64_t V, int64_t ld,
                          const float* temperature, const int32_t* top_k, const float* top_p, const float* min_p,
                          const uint64_t* seed, const uint64_t* step, const uint32_t* row_id, int32_t* token,
                          float* logprob, int32_t* row_status, int32_t* stats, void* stream) {
  vsamp_status st = check_common(logits, dt, B, V, ld);
  if (st != VSAMP_OK) return st;
  if (!token) return VSAMP_ERR_INVALID_ARG;
  Params p = base_params(logits, dt, B, V, ld);
  p.temperature = temperature;
  p.top_k = top_k;
  p.top_p = top_p;
  p.min_p = min_p;
  p.seed = seed;
  p.step = step;
  p.row_id = row_id;
  p.token = token;
  p.logprob = logprob;
  p.row_status = row_status;
  p.stats = stats;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (env_int("VSAMP_SAMPLE_STREAM", 0) != 0) {
    const vsamp_status ss = dt == VSAMP_F32 ? launch_sample_stream<float>(p, B, 4, s)
                                            : launch_sample_stream<__nv_bfloat16>(p, B, 2, s);
    if (ss != VSAMP_ERR_UNSUPPORTED) return ss;
  }
  if (dt == VSAMP_F32) return launch_sample<float>(p, B, 4, s);
  return launch_sample<__nv_bfloat16>(p, B, 2, s);
}

size_t vsamp_sample_workspace_size(vsamp_dtype dt, int64_t B, int64_t V) {
  if ((dt != VSAMP_F32 && dt != VSAMP_BF16) || B <= 0 || V <= 0) return 0;
  const int es = dt == VSAMP_F32 ? 4 : 2;
  return split_workspace_bytes(B, V, es);
}

vsamp_status vsamp_sample_ws(const void* logits, vsamp_dtype dt, int64_t B, int64_t V, int64_t ld,
                             const float* temperature, const int32_t* top_k, const float* top_p,
                             const float* min_p, const uint64_t* seed, const uint64_t* step,
                             const uint32_t* row_id, int32_t* token, float* logprob, int32_t* row_status,
                             int32_t* stats, void* workspace, size_t workspace_bytes, void* stream) {
  vsamp_status st = check_common(logits, dt, B, V, ld);
  if (st != VSAMP_OK) return st;
  if (!token || !workspace || (reinterpret_cast<uintptr_t>(workspace) & 15u) != 0) return VSAMP_ERR_INVALID_ARG;
  if (workspace_bytes < vsamp_sample_workspace_size(dt, B, V)) return VSAMP_ERR_INVALID_ARG;
  if (V > 0x7FFEFFFFLL) return VSAMP_ERR_UNSUPPORTED;   // 32-bit element indices, chunk ends included
  Params p = base_params(logits, dt, B, V, ld);
  p.temperature = temperature;
  p.top_k = top_k;
  p.top_p = top_p;
  p.min_p = min_p;
  p.seed = seed;
  p.step = step;
  p.row_id = row_id;
  p.token = token;
  p.logprob = logprob;
  p.row_status = row_status;
  p.stats = stats;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dt == VSAMP_F32) return launch_sample_split<float>(p, B, 4, workspace, s);
  return launch_sample_split<__nv_bfloat16>(p, B, 2, workspace, s);
}

vsamp_status vsamp_sample_static(const void* logits, vsamp_dtype dt, int64_t B, int64_t V, int64_t ld,
                                 const float* temperature, const int32_t* top_k, const float* top_p,
                                 const float* min_p, const uint64_t* seed, const uint64_t* step,
                                 const uint32_t* row_id, int32_t* token, float* logprob, int32_t* row_status,
                                 int32_t* stats, void* stream) {
  vsamp_status st = check_common(logits, dt, B, V, ld);
  if (st != VSAMP_OK) return st;
  if (!token) return VSAMP_ERR_INVALID_ARG;
  if (V > 0x7FFEFFFFLL) return VSAMP_ERR_UNSUPPORTED;
  const size_t need = vsamp_sample_workspace_size(dt, B, V);
  if (need > (size_t)VSAMP_STATIC_SCRATCH_BYTES) return VSAMP_ERR_SCRATCH_LIMIT;
  void* scratch = nullptr;
  st = static_scratch(&scratch);
  if (st != VSAMP_OK) return st;
  // no clear: the streaming kernels write every plan and piece statistic before reading it, and reset the
  // draw slot themselves, so the previous call's contents are never read
  return vsamp_sample_ws(logits, dt, B, V, ld, temperature, top_k, top_p, min_p, seed, step, row_id, token,
                         logprob, row_status, stats, scratch, (size_t)VSAMP_STATIC_SCRATCH_BYTES, stream);
}

static_assert(sizeof(vsamp_piece_rec) == sizeof(vsamp::PieceRec) && offsetof(vsamp_piece_rec, s) == 8 &&
                  offsetof(vsamp_piece_rec, mn) == 16,
              "vsamp_piece_rec mirrors the piece record the kernels write");

vsamp_status vsamp_sample_rejection(const void* logits, vsamp_dtype dt, int64_t B, int64_t V, int64_t ld,
                                    const float* temperature, const int32_t* top_k, const float* top_p,
                                    const float* min_p, const uint64_t* seed, const uint64_t* step,
                                    const uint32_t* row_id, int32_t* token, float* logprob, int32_t* row_status,
                                    int32_t* stats, void* stream) {
  vsamp_status st = check_common(logits, dt, B, V, ld);
  if (st != VSAMP_OK) return st;
  if (!token) return VSAMP_ERR_INVALID_ARG;
  Params p = base_params(logits, dt, B, V, ld);
  p.temperature = temperature;
  p.top_k = top_k;
  p.top_p = top_p;
  p.min_p = min_p;
  p.seed = seed;
  p.step = step;
  p.row_id = row_id;
  p.token = token;
  p.logprob = logprob;
  p.row_status = row_status;
  p.stats = stats;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dt == VSAMP_F32) return launch_reject<float>(p, B, s);
  return launch_reject<__nv_bfloat16>(p, B, s);
}

int64_t vsamp_shard_pieces(vsamp_dtype dt, int64_t V_shard) {
  if ((dt != VSAMP_F32 && dt != VSAMP_BF16) || V_shard <= 0) return 0;
  return split_nchunks(V_shard, dt == VSAMP_F32 ? 4 : 2);
}

size_t vsamp_shard_workspace_size(vsamp_dtype dt, int64_t B, int64_t V_shard) {
  if ((dt != VSAMP_F32 && dt != VSAMP_BF16) || B <= 0 || V_shard <= 0) return 0;
  return sizeof(StreamHeader) + (size_t)B * (size_t)split_nchunks(V_shard, dt == VSAMP_F32 ? 4 : 2) * 128u;
}

vsamp_status vsamp_shard_partial(const void* logits, vsamp_dtype dt, int64_t B, int64_t V_shard, int64_t ld,
                                 int64_t v0, int64_t NP, const float* temperature, const uint64_t* seed,
                                 const uint64_t* step, const uint32_t* row_id, const int32_t* target,
                                 vsamp_piece_rec* recs, vsamp_shard_win* win, void* workspace,
                                 size_t workspace_bytes, void* stream) {
  vsamp_status st = check_common(logits, dt, B, V_shard, ld);
  if (st != VSAMP_OK) return st;
  const int ve = dt == VSAMP_F32 ? 4 : 8;
  if (!recs || !win || !workspace || (reinterpret_cast<uintptr_t>(workspace) & 15u) != 0 ||
      (reinterpret_cast<uintptr_t>(recs) & 15u) != 0)
    return VSAMP_ERR_INVALID_ARG;
  if (v0 < 0 || v0 % ve != 0 || v0 + V_shard > 0x7FFEFFFFLL) return VSAMP_ERR_INVALID_ARG;
  if (NP < vsamp_shard_pieces(dt, V_shard)) return VSAMP_ERR_INVALID_ARG;
  if (workspace_bytes < vsamp_shard_workspace_size(dt, B, V_shard)) return VSAMP_ERR_INVALID_ARG;
  Params p = base_params(logits, dt, B, V_shard, ld);
  p.temperature = temperature;
  p.seed = seed;
  p.step = step;
  p.row_id = row_id;
  p.v0 = v0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dt == VSAMP_F32) return launch_shard_partial<float>(p, B, 4, NP, target, win, recs, workspace, s);
  return launch_shard_partial<__nv_bfloat16>(p, B, 2, NP, target, win, recs, workspace, s);
}

vsamp_status vsamp_shard_merge(const vsamp_piece_rec* recs, const vsamp_shard_win* wins, int32_t R, int64_t B,
                               int64_t NP, int64_t V, const float* temperature, const uint64_t* seed,
                               const uint64_t* step, const uint32_t* row_id, float* row_max, float* row_logsum,
                               int32_t* token, float* logprob, float* target_logprob, int32_t* row_status,
                               void* stream) {
  if (!recs || !wins || R <= 0 || B <= 0 || NP <= 0 || V <= 0 || V > 0x7FFEFFFFLL) return VSAMP_ERR_INVALID_ARG;
  return launch_shard_merge(recs, wins, R, B, NP, V, temperature, seed, step, row_id, row_max, row_logsum, token,
                            logprob, target_logprob, row_status, static_cast<cudaStream_t>(stream));
}

vsamp_status vsamp_logprob(const void* logits, vsamp_dtype dt, int64_t B, int64_t V, int64_t ld,
                           const float* temperature, const int32_t* token, const float* row_max,
                           const float* row_logsum, float* out, int32_t* row_status, void* stream) {
  vsamp_status st = check_common(logits, dt, B, V, ld);
  if (st != VSAMP_OK) return st;
  if (!token || !out) return VSAMP_ERR_INVALID_ARG;
  if ((row_max == nullptr) != (row_logsum == nullptr)) return VSAMP_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (row_max) {
    const int threads = 256;
    const unsigned blocks = (unsigned)((B + threads - 1) / threads);
    const unsigned char* x = static_cast<const unsigned char*>(logits);
    if (dt == VSAMP_F32)
      logprob_from_stats_kernel<float><<<blocks, threads, 0, s>>>(x, B, V, ld, temperature, token, row_max,
                                                                  row_logsum, out, row_status);
    else
      logprob_from_stats_kernel<__nv_bfloat16><<<blocks, threads, 0, s>>>(x, B, V, ld, temperature, token,
                                                                          row_max, row_logsum, out, row_status);
    if (cudaGetLastError() != cudaSuccess) return VSAMP_ERR_CUDA;
    return VSAMP_OK;
  }
  Params p = base_params(logits, dt, B, V, ld);
  p.temperature = temperature;
  p.token_in = token;
  p.logprob = out;
  p.row_status = row_status;
  return dispatch_stats<MODE_LOGPROB>(p, dt, B, s);
}

vsamp_status vsamp_topn_logprobs(const void* logits, vsamp_dtype dt, int64_t B, int64_t V, int64_t ld,
                                 const float* temperature, int32_t N, float* row_max, float* row_logsum,
                                 int32_t* out_idx, float* out_lp, int32_t* row_status, void* stream) {
  vsamp_status st = check_common(logits, dt, B, V, ld);
  if (st != VSAMP_OK) return st;
  if (N <= 0 || N > VSAMP_TOPN_MAX || !row_max || !row_logsum || !out_idx || !out_lp) return VSAMP_ERR_INVALID_ARG;
  if (V > 0x7FFFFFFFLL) return VSAMP_ERR_UNSUPPORTED;   // 32-bit token indices
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // 1. one pass over each row: the row statistics at the row's temperature, the row status, and the N best
  //    indices (the top-k cut with k = N) in ascending index order
  Params p = base_params(logits, dt, B, V, ld);
  p.temperature = temperature;
  p.row_max = row_max;
  p.row_logsum = row_logsum;
  p.row_status = row_status;
  p.k_max = N;
  p.out_idx = out_idx;
  st = dispatch<MODE_LSE | MODE_TOPN>(p, dt, B, s);
  if (st != VSAMP_OK) return st;
  // 2. order the list and attach the log-probabilities
  DeviceInfo d;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return VSAMP_ERR_CUDA;
  }
  st = device_info(dev, d);
  if (st != VSAMP_OK) return st;
  const int64_t cap = (int64_t)d.sm_count * 8;
  const unsigned blocks = (unsigned)(B < cap ? B : cap);
  const size_t smem = (size_t)N * (sizeof(float) + sizeof(int32_t));
  const unsigned char* x = static_cast<const unsigned char*>(logits);
  if (dt == VSAMP_F32)
    topn_rank_kernel<float><<<blocks, kTopnThreads, smem, s>>>(x, B, V, ld, temperature, N, row_max, row_logsum,
                                                               out_idx, out_lp);
  else
    topn_rank_kernel<__nv_bfloat16><<<blocks, kTopnThreads, smem, s>>>(x, B, V, ld, temperature, N, row_max,
                                                                       row_logsum, out_idx, out_lp);
  if (cudaGetLastError() != cudaSuccess) return VSAMP_ERR_CUDA;
  return VSAMP_OK;
}

vsamp_status vsamp_kept_logprob(const void* logits, vsamp_dtype dt, int64_t B, int64_t V, int64_t ld,
                                const float* temperature, const int32_t* top_k, const float* top_p,
                                const float* min_p, const int32_t* token, float* out, int32_t* row_status,
                                void* stream) {
  vsamp_status st = check_common(logits, dt, B, V, ld);
  if (st != VSAMP_OK) return st;
  if (!token || !out) return VSAMP_ERR_INVALID_ARG;
  Params p = base_params(logits, dt, B, V, ld);
  p.temperature = temperature;
  p.top_k = top_k;
  p.top_p = top_p;
  p.min_p = min_p;
  p.token_in = token;
  p.logprob = out;
  p.row_status = row_status;
  return dispatch<MODE_KEPT>(p, dt, B, static_cast<cudaStream_t>(stream));
}

const char* vsamp_status_string(vsamp_status s) {
  switch (s) {
    case VSAMP_OK: return "ok";
    case VSAMP_ERR_INVALID_ARG: return "invalid argument";
    case VSAMP_ERR_UNSUPPORTED: return "unsupported on this device (shared memory or cluster size)";
    case VSAMP_ERR_CUDA: return "CUDA runtime error";
    case VSAMP_ERR_NONFINITE: return "non-finite value in the row";
    case VSAMP_ERR_TIMEOUT: return "device-side wait timed out";
    case VSAMP_ERR_SCRATCH_LIMIT: return "batch needs more than the fixed scratch array of vsamp_sample_static";
  }
  return "unknown status";
}

vsamp_status vsamp_device_info(int device, vsamp_limits* out) {
  if (!out) return VSAMP_ERR_INVALID_ARG;
  DeviceInfo d;
  vsamp_status st = device_info(device, d);
  if (st != VSAMP_OK) return st;
  out->sm_count = d.sm_count;
  out->smem_optin_bytes = d.optin;
  out->max_cluster = d.max_cluster;
  const int64_t per_cta = ((int64_t)d.optin - slice_offset<kThreadsLarge>()) / 16 * 16;
  out->max_row_f32 = per_cta / 4 * d.max_cluster;
  out->max_row_bf16 = per_cta / 2 * d.max_cluster;
  return VSAMP_OK;
}

int32_t vsamp_version(void) { return (1 << 16) | 0; }

}  // extern "C"
