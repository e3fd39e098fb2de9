// bf16 instantiation of the split-vocabulary sampling kernels and their launchers.
#include "vsamp_reject.cuh"
#include "vsamp_select_stream.cuh"
#include "vsamp_split_launch.cuh"
#include "vsamp_sample_stream.cuh"
#include "vsamp_stats.cuh"

namespace vsamp {
template vsamp_status launch_sample_stream<__nv_bfloat16>(Params, int64_t, int, cudaStream_t);
template vsamp_status launch_stats<__nv_bfloat16, MODE_LSE>(Params, int64_t, int, cudaStream_t);
template vsamp_status launch_stats<__nv_bfloat16, MODE_LOGPROB>(Params, int64_t, int, cudaStream_t);
template vsamp_status launch_select_stream<__nv_bfloat16>(Params, int64_t, cudaStream_t);
template vsamp_status launch_reject<__nv_bfloat16>(Params, int64_t, cudaStream_t);
template vsamp_status launch_sample_split<__nv_bfloat16>(Params, int64_t, int, void*, cudaStream_t);
template vsamp_status launch_shard_partial<__nv_bfloat16>(Params, int64_t, int, int64_t, const int32_t*, void*, void*,
                                                          void*, cudaStream_t);
}  // namespace vsamp
