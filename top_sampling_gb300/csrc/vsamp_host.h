// Host-side pieces shared by the translation units of libvsamp.so: device limits, launch geometry and
// the kernel launcher.
#pragma once

#include <cstdint>
#include <cstdlib>

#include "vsamp.h"
#include "vsamp_row.cuh"

namespace vsamp {

constexpr int kThreadsSmall = 128;   // threads per CTA (two instantiations of every kernel)
constexpr int kThreadsLarge = 256;

struct DeviceInfo {
  int ready = 0;
  int sm_count = 0;
  int optin = 0;           // max shared memory per block (opt-in)
  int smem_per_sm = 0;     // shared memory per multiprocessor
  int max_cluster = 0;     // largest cluster size the kernels request
};

struct Geometry {
  int NT = 256;    // threads per CTA
  int C = 1;       // CTAs per row (cluster size)
  int q = 1;       // 16-byte vectors per thread
  int nbuf = 2;    // slice buffers per CTA
  int smem = 0;    // dynamic shared memory bytes
};

// Clusters of `kern` resident at once for a launch of cluster size C with `smem` bytes of dynamic shared
// memory on the current device; the kernel's shared-memory and cluster attributes are set on the first query
// of each (device, kernel, smem, C) and the answer is cached. 0 when the device cannot run the launch.
int cached_max_clusters(const void* kern, int threads, int smem, int C);

int env_int(const char* name, int dflt);
long long env_ll(const char* name, long long dflt);
vsamp_status device_info(int dev, DeviceInfo& out);
vsamp_status choose_geometry(int64_t V, int esize, int64_t B, const DeviceInfo& d, Geometry& g);
// NT data threads per CTA, head bytes of shared memory before the slice, per_sm CTAs resident per SM; small
// batches spread a row over more CTAs, up to max_spread per cluster
vsamp_status choose_geometry_for(int64_t V, int esize, int64_t B, const DeviceInfo& d, int NT, int head, int per_sm,
                                 Geometry& g, int max_nbuf = 1, int max_spread = 16);

// vsamp_sample's kernel (specialised warps), in its own translation units
template <typename T>
vsamp_status launch_sample(Params p, int64_t B, int esize, cudaStream_t stream);

// vsamp_sample_ws's kernels (split vocabulary, caller's workspace)
template <typename T>
vsamp_status launch_sample_split(Params p, int64_t B, int esize, void* workspace, cudaStream_t stream);

// vsamp_shard_partial's kernels (piece pass over a vocabulary shard, the shard's winners)
template <typename T>
vsamp_status launch_shard_partial(Params p, int64_t B, int esize, int64_t NP, const int32_t* target, void* win,
                                  void* recs, void* workspace, cudaStream_t stream);

// vsamp_sample_rejection's kernel (dual-pivot rejection rounds, one CTA per row)
template <typename T>
vsamp_status launch_reject(Params p, int64_t B, cudaStream_t stream);

// vsamp_topk_select's uncached path (rows longer than a cluster holds on chip)
template <typename T>
vsamp_status launch_select_stream(Params p, int64_t B, cudaStream_t stream);
// vsamp_stats.cuh: row statistics by streaming pieces (MODE_LSE or MODE_LOGPROB); VSAMP_ERR_UNSUPPORTED for rows
// longer than it takes
template <typename T, int MODE>
vsamp_status launch_stats(Params p, int64_t B, int esize, cudaStream_t stream);
// vsamp_sample_stream.cuh: the streaming sampler without a workspace; VSAMP_ERR_UNSUPPORTED for rows longer than
// it takes
template <typename T>
vsamp_status launch_sample_stream(Params p, int64_t B, int esize, cudaStream_t stream);

// vsamp_shard_merge's kernel (dtype-free)
vsamp_status launch_shard_merge(const void* recs, const void* wins, int R, int64_t B, int64_t NP, int64_t V,
                                const float* temperature, const uint64_t* seed, const uint64_t* step,
                                const uint32_t* row_id, float* row_max, float* row_logsum, int32_t* token,
                                float* logprob, float* target_logprob, int32_t* row_status, cudaStream_t stream);

template <typename T, int MODE>
vsamp_status launch(Params p, int64_t B, int esize, cudaStream_t stream);

}  // namespace vsamp
