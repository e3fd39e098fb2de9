// bf16 instantiation of the specialised-warp sampling kernel and its launcher.
#include "vsamp_sample_launch.cuh"

namespace vsamp {
template vsamp_status launch_sample<__nv_bfloat16>(Params, int64_t, int, cudaStream_t);
}  // namespace vsamp
