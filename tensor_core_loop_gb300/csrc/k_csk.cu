// Instantiates the kernel that sums a tile's K ranges inside a cluster
// (gemm_kernel_csk.cuh) and launches it: one cluster of CL CTAs per tile.
#include "gemm_kernel_csk.cuh"
#include "launch.cuh"

namespace tcl {
namespace {

constexpr int kCskStages = 4;

template <OutKind OK, int CL>
cudaError_t launch_csk_t(const LaunchArgs& a) {
    using C = CskCfg<OK, CL, kCskStages>;
    static bool done[64] = {};
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (!(dev >= 0 && dev < 64 && done[dev])) {
        err = cudaFuncSetAttribute(gemm_csk_kernel<OK, CL, kCskStages>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   C::SMEM_BYTES);
        if (err != cudaSuccess) return err;
        if (dev >= 0 && dev < 64) done[dev] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    cfg.gridDim = dim3(a.grid);
    cfg.blockDim = dim3(C::THREADS);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = a.stream;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (a.pdl) {
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.numAttrs = 2;
    }
    return cudaLaunchKernelEx(&cfg, gemm_csk_kernel<OK, CL, kCskStages>, a.tmA, a.tmB, a.tmC, a.p);
}

}  // namespace

cudaError_t launch_csk(const LaunchArgs& a, bool* found) {
    *found = true;
    if (a.in == InKind::BF16 && a.bn == 64) {
        if (a.out == OutKind::F32 && a.csk == 2) return launch_csk_t<OutKind::F32, 2>(a);
        if (a.out == OutKind::F32 && a.csk == 4) return launch_csk_t<OutKind::F32, 4>(a);
        if (a.out == OutKind::BF16 && a.csk == 2) return launch_csk_t<OutKind::BF16, 2>(a);
        if (a.out == OutKind::BF16 && a.csk == 4) return launch_csk_t<OutKind::BF16, 4>(a);
    }
    *found = false;
    return cudaSuccess;
}

int csk_stages() { return kCskStages; }
int csk_smem_bytes(int cl) {
    return cl == 4 ? CskCfg<OutKind::F32, 4, kCskStages>::SMEM_BYTES : CskCfg<OutKind::F32, 2, kCskStages>::SMEM_BYTES;
}

}  // namespace tcl
