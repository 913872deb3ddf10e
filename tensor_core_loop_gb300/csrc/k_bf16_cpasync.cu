// Instantiates one group of GEMM kernel variants (see launch.cuh); kept in its
// own translation unit so that the groups compile in parallel.
#include "launch.cuh"

namespace tcl {

cudaError_t launch_group_bf16_cpasync(const LaunchArgs& a, bool* found) {
    *found = false;
    TCL_GROUP_BF16_CPASYNC(TCL_VARIANT_CASE)
    return cudaErrorNotSupported;
}

}  // namespace tcl
