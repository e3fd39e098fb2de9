// Kernel launcher: cluster launch of row_kernel over (C, B) blocks; rows beyond 65535 take more launches.
#pragma once

#include "vsamp_host.h"

namespace vsamp {

template <typename T, int NT, int MODE>
static vsamp_status launch_nt(Params p, int64_t B, const Geometry& g, cudaStream_t stream) {
  auto kern = row_kernel<T, NT, MODE>;
  // a byte per vector after the slice (each vector's largest value bin in a radix search's first round) and
  // four mask words per thread, where they cost no CTA per SM
  int smem = g.smem;
  p.vbytes = 0;
  if (g.q <= 64) {
    int dev = 0;
    DeviceInfo d;
    if (cudaGetDevice(&dev) == cudaSuccess && device_info(dev, d) == VSAMP_OK) {
      const int smem_sm = d.smem_per_sm > 0 ? d.smem_per_sm : d.optin;
      const int per_sm = NT <= 128 ? 6 : 3;   // the kernel's launch bound
      const int vb = (NT * g.q + 15) / 16 * 16 + NT * 16;   // the bytes, then four mask words per thread
      auto fit = [&](int s) { const int f = smem_sm / (s + 1024); return f < per_sm ? f : per_sm; };
      if (g.smem + vb <= d.optin && fit(g.smem + vb) >= fit(g.smem)) {
        smem = g.smem + vb;
        p.vbytes = 1;
      }
    } else {
      cudaGetLastError();
    }
  }
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(NT, 1, 1);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)g.C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // persistent clusters: as many as fit at once, then evened out so every cluster has the same number
  // of rows (+-1)
  cfg.gridDim = dim3((unsigned)g.C, 1, 1);
  const int nclusters = cached_max_clusters(reinterpret_cast<const void*>(kern), NT, smem, g.C);
  if (nclusters < 1) return VSAMP_ERR_UNSUPPORTED;
  const int fit = env_int("VSAMP_GRID_CLUSTERS", 0) > 0 ? env_int("VSAMP_GRID_CLUSTERS", 0) : nclusters;
  int64_t G = B < fit ? B : fit;
  const int64_t rounds = (B + G - 1) / G;
  G = (B + rounds - 1) / rounds;
  if (G > 65535) G = 65535;
  p.row0 = 0;
  cfg.gridDim = dim3((unsigned)g.C, (unsigned)G, 1);
  if (cudaLaunchKernelEx(&cfg, kern, p) != cudaSuccess) {
    cudaGetLastError();
    return VSAMP_ERR_CUDA;
  }
  return VSAMP_OK;
}

template <typename T, int MODE>
vsamp_status launch(Params p, int64_t B, int esize, cudaStream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return VSAMP_ERR_CUDA; }
  DeviceInfo d;
  vsamp_status st = device_info(dev, d);
  if (st != VSAMP_OK) return st;
  Geometry g;
  st = choose_geometry(p.V, esize, B, d, g);
  if (st != VSAMP_OK) return st;
  p.q = g.q;
  // bound of a load wait: ~2 s at the maximum SM clock unless VSAMP_WAIT_CYCLES sets another
  const long long wc = env_ll("VSAMP_WAIT_CYCLES", 0);
  p.wait_cycles = wc > 0 ? wc : 4000000000LL;
  p.drop_loads = env_int("VSAMP_TEST_DROP_LOADS", 0) != 0 ? 1 : 0;
  if (g.NT == kThreadsSmall) return launch_nt<T, kThreadsSmall, MODE>(p, B, g, stream);
  return launch_nt<T, kThreadsLarge, MODE>(p, B, g, stream);
}

}  // namespace vsamp

#define VSAMP_INSTANTIATE(T)                                                              \
  template vsamp_status launch<T, MODE_LSE>(Params, int64_t, int, cudaStream_t);          \
  template vsamp_status launch<T, MODE_SELECT>(Params, int64_t, int, cudaStream_t);       \
  template vsamp_status launch<T, MODE_CUT>(Params, int64_t, int, cudaStream_t);          \
  template vsamp_status launch<T, MODE_CUT | MODE_MASK>(Params, int64_t, int, cudaStream_t); \
  template vsamp_status launch<T, MODE_SAMPLE>(Params, int64_t, int, cudaStream_t);       \
  template vsamp_status launch<T, MODE_LOGPROB>(Params, int64_t, int, cudaStream_t);       \
  template vsamp_status launch<T, MODE_LSE | MODE_TOPN>(Params, int64_t, int, cudaStream_t);       \
  template vsamp_status launch<T, MODE_KEPT>(Params, int64_t, int, cudaStream_t);
