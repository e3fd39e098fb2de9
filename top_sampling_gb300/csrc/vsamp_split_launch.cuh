// Launcher of the fused streaming sampling kernel (vsamp_sample_ws, vsamp_sample_static).
#pragma once

#include <mutex>

#include "vsamp_host.h"
#include "vsamp_shard.cuh"

namespace vsamp {

template <typename T>
vsamp_status launch_sample_split(Params p, int64_t B, int esize, void* workspace, cudaStream_t stream) {
  static int occ[64] = {0};
  static std::mutex mu;
  const int64_t np = split_nchunks(p.V, esize);
  if (np > 0x7FFFFFFF) return VSAMP_ERR_UNSUPPORTED;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return VSAMP_ERR_CUDA; }
  if (dev < 0 || dev >= 64) return VSAMP_ERR_UNSUPPORTED;
  DeviceInfo d;
  vsamp_status st = device_info(dev, d);
  if (st != VSAMP_OK) return st;
  auto kern = piece_kernel<T>;
  const int smem = (int)sizeof(PieceSmem);
  int per_sm = 0;
  {
    std::lock_guard<std::mutex> lk(mu);
    if (!occ[dev]) {
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess ||
          cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ[dev], kern, kStreamThreads, smem) != cudaSuccess) {
        cudaGetLastError();
        occ[dev] = 0;
        return VSAMP_ERR_UNSUPPORTED;
      }
    }
    per_sm = occ[dev];
  }
  if (per_sm < 1) return VSAMP_ERR_UNSUPPORTED;
  unsigned char* w = static_cast<unsigned char*>(workspace);
  StreamWs ws;
  ws.recs = reinterpret_cast<PieceRec*>(w + sizeof(StreamHeader));
  ws.rec_ld = np;
  ws.codes = reinterpret_cast<uint32_t*>(w + sizeof(StreamHeader) + (size_t)B * (size_t)np * sizeof(PieceRec));
  const long long pieces = (long long)B * np;
  long long grid = (long long)per_sm * d.sm_count;
  const long long need = (pieces + kItemPieces - 1) / kItemPieces;
  if (grid > need) grid = need;
  p.row0 = 0;
  // bound of a load wait: ~2 s at the maximum SM clock unless VSAMP_WAIT_CYCLES sets another
  const long long wc = env_ll("VSAMP_WAIT_CYCLES", 0);
  p.wait_cycles = wc > 0 ? wc : 4000000000LL;
  p.drop_loads = env_int("VSAMP_TEST_DROP_LOADS", 0) != 0 ? 1 : 0;
  kern<<<(unsigned)grid, kStreamThreads, smem, stream>>>(p, ws, (int)np);
  if (cudaGetLastError() != cudaSuccess) return VSAMP_ERR_CUDA;
  const int64_t rows = B < 0x7FFFFFFF ? B : 0x7FFFFFFF;
  row_finish_kernel<T><<<(unsigned)rows, kStreamThreads, 0, stream>>>(p, ws, (int)np);
  if (cudaGetLastError() != cudaSuccess) return VSAMP_ERR_CUDA;
  return VSAMP_OK;
}

// vsamp_shard_partial: the piece pass over the shard, then the shard's winners. The codes live in the workspace.
template <typename T>
vsamp_status launch_shard_partial(Params p, int64_t B, int esize, int64_t NP, const int32_t* target, void* win,
                                  void* recs, void* workspace, cudaStream_t stream) {
  static int occ[64] = {0};
  static std::mutex mu;
  const int64_t np = split_nchunks(p.V, esize);
  if (np > NP || np >= (1LL << 31) / 32) return VSAMP_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return VSAMP_ERR_CUDA; }
  if (dev < 0 || dev >= 64) return VSAMP_ERR_UNSUPPORTED;
  DeviceInfo d;
  vsamp_status st = device_info(dev, d);
  if (st != VSAMP_OK) return st;
  auto kern = piece_kernel<T>;
  const int smem = (int)sizeof(PieceSmem);
  int per_sm = 0;
  {
    std::lock_guard<std::mutex> lk(mu);
    if (!occ[dev]) {
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess ||
          cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ[dev], kern, kStreamThreads, smem) != cudaSuccess) {
        cudaGetLastError();
        occ[dev] = 0;
        return VSAMP_ERR_UNSUPPORTED;
      }
    }
    per_sm = occ[dev];
  }
  if (per_sm < 1) return VSAMP_ERR_UNSUPPORTED;
  StreamWs ws;
  ws.recs = static_cast<PieceRec*>(recs);
  ws.rec_ld = NP;
  ws.codes = reinterpret_cast<uint32_t*>(static_cast<unsigned char*>(workspace) + sizeof(StreamHeader));
  const long long pieces = (long long)B * np;
  long long grid = (long long)per_sm * d.sm_count;
  const long long need = (pieces + kItemPieces - 1) / kItemPieces;
  if (grid > need) grid = need;
  const long long wc = env_ll("VSAMP_WAIT_CYCLES", 0);
  p.wait_cycles = wc > 0 ? wc : 4000000000LL;
  p.drop_loads = env_int("VSAMP_TEST_DROP_LOADS", 0) != 0 ? 1 : 0;
  kern<<<(unsigned)grid, kStreamThreads, smem, stream>>>(p, ws, (int)np);
  if (cudaGetLastError() != cudaSuccess) return VSAMP_ERR_CUDA;
  const int64_t rows = B < 0x7FFFFFFF ? B : 0x7FFFFFFF;
  shard_finish_kernel<T><<<(unsigned)rows, kStreamThreads, 0, stream>>>(p, ws, (int)np, target,
                                                                        static_cast<ShardWin*>(win));
  if (cudaGetLastError() != cudaSuccess) return VSAMP_ERR_CUDA;
  return VSAMP_OK;
}

}  // namespace vsamp
