// Launchers of the split-vocabulary sampling kernels (vsamp_sample_ws).
#pragma once

#include "vsamp_host.h"
#include "vsamp_split.cuh"

namespace vsamp {

inline size_t split_workspace_bytes(int64_t B, int64_t V, int esize) {
  return (size_t)B * sizeof(RowPlan) + (size_t)B * (size_t)split_nchunks(V, esize) * sizeof(ChunkStat);
}

template <typename T>
vsamp_status launch_sample_split(Params p, int64_t B, int esize, void* workspace, cudaStream_t stream) {
  const int64_t nch = split_nchunks(p.V, esize);
  if (nch > 0x7FFFFFFF) return VSAMP_ERR_UNSUPPORTED;
  RowPlan* plans = static_cast<RowPlan*>(workspace);
  ChunkStat* stats = reinterpret_cast<ChunkStat*>(static_cast<unsigned char*>(workspace) + (size_t)B * sizeof(RowPlan));
  for (int64_t r0 = 0; r0 < B; r0 += 65535) {
    const int64_t nb = B - r0 < 65535 ? B - r0 : 65535;
    p.row0 = r0;
    const dim3 grid((unsigned)nch, (unsigned)nb, 1);
    split_stats_kernel<T><<<grid, kSplitThreads, 0, stream>>>(p, plans, stats, (int)nch);
    if (cudaGetLastError() != cudaSuccess) return VSAMP_ERR_CUDA;
    split_draw_kernel<T><<<grid, kSplitThreads, 0, stream>>>(p, plans, (int)nch);
    if (cudaGetLastError() != cudaSuccess) return VSAMP_ERR_CUDA;
  }
  return VSAMP_OK;
}

}  // namespace vsamp
