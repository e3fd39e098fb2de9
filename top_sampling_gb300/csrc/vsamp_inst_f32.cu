// fp32 instantiations of the row kernel and its launcher.
#include "vsamp_launch.cuh"

namespace vsamp {
VSAMP_INSTANTIATE(float)
}  // namespace vsamp
