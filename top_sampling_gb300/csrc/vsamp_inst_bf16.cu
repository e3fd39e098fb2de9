// bf16 instantiations of the row kernel and its launcher.
#include "vsamp_launch.cuh"

namespace vsamp {
VSAMP_INSTANTIATE(__nv_bfloat16)
}  // namespace vsamp
