// f32 instantiation of the split-vocabulary sampling kernels and their launchers; the shard merge (dtype-free).
#include "vsamp_reject.cuh"
#include "vsamp_select_stream.cuh"
#include "vsamp_split_launch.cuh"
#include "vsamp_sample_stream.cuh"
#include "vsamp_stats.cuh"

namespace vsamp {
template vsamp_status launch_sample_stream<float>(Params, int64_t, int, cudaStream_t);
template vsamp_status launch_stats<float, MODE_LSE>(Params, int64_t, int, cudaStream_t);
template vsamp_status launch_stats<float, MODE_LOGPROB>(Params, int64_t, int, cudaStream_t);
template vsamp_status launch_select_stream<float>(Params, int64_t, cudaStream_t);
template vsamp_status launch_reject<float>(Params, int64_t, cudaStream_t);
template vsamp_status launch_sample_split<float>(Params, int64_t, int, void*, cudaStream_t);
template vsamp_status launch_shard_partial<float>(Params, int64_t, int, int64_t, const int32_t*, void*, void*, void*,
                                                  cudaStream_t);

vsamp_status launch_shard_merge(const void* recs, const void* wins, int R, int64_t B, int64_t NP, int64_t V,
                                const float* temperature, const uint64_t* seed, const uint64_t* step,
                                const uint32_t* row_id, float* row_max, float* row_logsum, int32_t* token,
                                float* logprob, float* target_logprob, int32_t* row_status, cudaStream_t stream) {
  const int64_t rows = B < 0x7FFFFFFF ? B : 0x7FFFFFFF;
  shard_merge_kernel<0><<<(unsigned)rows, kStreamThreads, 0, stream>>>(
      static_cast<const PieceRec*>(recs), static_cast<const ShardWin*>(wins), R, B, NP, V, temperature, seed, step,
      row_id, row_max, row_logsum, token, logprob, target_logprob, row_status);
  if (cudaGetLastError() != cudaSuccess) return VSAMP_ERR_CUDA;
  return VSAMP_OK;
}
}  // namespace vsamp
