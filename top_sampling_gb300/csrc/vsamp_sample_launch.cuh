// Launcher of the specialised-warp sampling kernel: cluster launch over (C, G) blocks of kSampleThreads
// threads, persistent over rows.
#pragma once

#include "vsamp_host.h"
#include "vsamp_sample.cuh"

namespace vsamp {

template <typename T, int NDW, int PER_SM>
static vsamp_status launch_sample_cfg(Params p, int64_t B, int esize, const DeviceInfo& d, cudaStream_t stream) {
  constexpr int kDataThreads = NDW * 32;
  constexpr int kSampleThreads = kDataThreads + 32;
  Geometry g;
  // small batches: at most 6 CTAs per row. Every radix round and plan of the sampling kernel is a cluster
  // exchange through the control warps, whose cost grows with the cluster (B = 4 x V = 32,000 fp32: 106 us at
  // 16 CTAs per row, 55 us at 4-6, 68 us at 2).
  vsamp_status st = choose_geometry_for(p.V, esize, B, d, kDataThreads, sample_slice_offset(), PER_SM, g,
                                        env_int("VSAMP_NBUF", 1) == 2 ? 2 : 1, 6);
  if (st != VSAMP_OK) return st;
  p.q = g.q;
  p.nbuf = g.nbuf;
  const long long wc = env_ll("VSAMP_WAIT_CYCLES", 0);
  p.wait_cycles = wc > 0 ? wc : 4000000000LL;   // ~2 s at the maximum SM clock
  p.drop_loads = env_int("VSAMP_TEST_DROP_LOADS", 0) != 0 ? 1 : 0;
  auto kern = sample_kernel<T, NDW, PER_SM>;
  const int smem_sm = d.smem_per_sm > 0 ? d.smem_per_sm : d.optin;
  int per_sm = PER_SM;
  // a slice that leaves no room for a second CTA on an SM: the instantiation without a register cap (the
  // capped one spills its row state, and with the shared-memory carve-out at its largest the spills miss L1)
  if constexpr (NDW == 8 && PER_SM > 1) {
    if (2 * (g.smem + 1024) > smem_sm) {
      kern = sample_kernel<T, NDW, 1>;
      per_sm = 1;
    }
  }
  // a byte per vector after the slices (each vector's largest value bin in a radix search's first round) and
  // four mask words per thread, where they cost no CTA per SM
  int smem = g.smem;
  p.vbytes = 0;
  if (g.q <= 64) {
    const int vb = (kDataThreads * g.q + 15) / 16 * 16 + kDataThreads * 16;   // the bytes, then four mask words per thread
    auto fit = [&](int s) { const int f = smem_sm / (s + 1024); return f < per_sm ? f : per_sm; };
    if (g.smem + vb <= d.optin && fit(g.smem + vb) >= fit(g.smem)) {
      smem = g.smem + vb;
      p.vbytes = 1;
    }
  }
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kSampleThreads, 1, 1);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)g.C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3((unsigned)g.C, 1, 1);
  const int nclusters = cached_max_clusters(reinterpret_cast<const void*>(kern), kSampleThreads, smem, g.C);
  if (nclusters < 1) return VSAMP_ERR_UNSUPPORTED;
  const int fit = env_int("VSAMP_GRID_CLUSTERS", 0) > 0 ? env_int("VSAMP_GRID_CLUSTERS", 0) : nclusters;
  int64_t G = B < fit ? B : fit;
  const int64_t rounds = (B + G - 1) / G;   // every cluster gets the same number of rows (+-1)
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

template <typename T>
vsamp_status launch_sample(Params p, int64_t B, int esize, cudaStream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return VSAMP_ERR_CUDA; }
  DeviceInfo d;
  vsamp_status st = device_info(dev, d);
  if (st != VSAMP_OK) return st;
  switch (env_int("VSAMP_SAMPLE_CFG", 0)) {
    case 1: return launch_sample_cfg<T, 4, 6>(p, B, esize, d, stream);
    case 2: return launch_sample_cfg<T, 4, 5>(p, B, esize, d, stream);
    case 3: return launch_sample_cfg<T, 8, 4>(p, B, esize, d, stream);
    default: return launch_sample_cfg<T, 8, 3>(p, B, esize, d, stream);
  }
}

}  // namespace vsamp
