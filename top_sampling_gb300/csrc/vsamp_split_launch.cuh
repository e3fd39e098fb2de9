// Launcher of the streaming sampling kernels (vsamp_sample_ws): chunk statistics, plans, the draw, the outputs.
#pragma once

#include <mutex>

#include "vsamp_host.h"
#include "vsamp_split.cuh"

namespace vsamp {

inline size_t split_workspace_bytes(int64_t B, int64_t V, int esize) {
  return sizeof(StreamHeader) + (size_t)B * sizeof(RowPlan) +
         (size_t)B * (size_t)split_nchunks(V, esize) * sizeof(ChunkStat);
}

// CTAs of `kern` resident per SM on `dev` (queried once per device and kernel)
template <typename K>
static int stream_blocks_per_sm(K kern, int dev, int (&cache)[64], std::mutex& mu) {
  if (dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lk(mu);
  if (!cache[dev]) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kStreamThreads, 0) != cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    cache[dev] = n;
  }
  return cache[dev];
}

template <typename T>
vsamp_status launch_sample_split(Params p, int64_t B, int esize, void* workspace, cudaStream_t stream) {
  static int occ_stats[64] = {0}, occ_draw[64] = {0};
  static std::mutex mu;
  const int64_t np = split_nchunks(p.V, esize);
  if (np > 0x7FFFFFFF) return VSAMP_ERR_UNSUPPORTED;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return VSAMP_ERR_CUDA; }
  DeviceInfo d;
  vsamp_status st = device_info(dev, d);
  if (st != VSAMP_OK) return st;
  const int ps = stream_blocks_per_sm(warp_stats_kernel<T>, dev, occ_stats, mu);
  const int pd = stream_blocks_per_sm(warp_draw_kernel<T>, dev, occ_draw, mu);
  if (ps < 1 || pd < 1) return VSAMP_ERR_UNSUPPORTED;
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  RowPlan* plans = reinterpret_cast<RowPlan*>(ws + sizeof(StreamHeader));
  ChunkStat* stats = reinterpret_cast<ChunkStat*>(ws + sizeof(StreamHeader) + (size_t)B * sizeof(RowPlan));
  const long long warps = (long long)B * np;   // one warp per item at most
  auto grid_of = [&](int per_sm) {
    long long g = (long long)per_sm * d.sm_count;
    const long long need = (warps + kStreamThreads / 32 - 1) / (kStreamThreads / 32);
    return g > need ? need : g;
  };
  p.row0 = 0;
  const unsigned rows = (unsigned)B;
  warp_stats_kernel<T><<<(unsigned)grid_of(ps), kStreamThreads, 0, stream>>>(p, stats, (int)np);
  if (cudaGetLastError() != cudaSuccess) return VSAMP_ERR_CUDA;
  stream_plan_kernel<T><<<rows, kSplitThreads, 0, stream>>>(p, plans, stats, (int)np);
  if (cudaGetLastError() != cudaSuccess) return VSAMP_ERR_CUDA;
  warp_draw_kernel<T><<<(unsigned)grid_of(pd), kStreamThreads, 0, stream>>>(p, plans, (int)np);
  if (cudaGetLastError() != cudaSuccess) return VSAMP_ERR_CUDA;
  stream_finish_kernel<T><<<rows, kSplitThreads, 0, stream>>>(p, plans);
  if (cudaGetLastError() != cudaSuccess) return VSAMP_ERR_CUDA;
  return VSAMP_OK;
}

}  // namespace vsamp
