// Instantiates the 64×64-tile kernel for small grids (gemm_kernel_m64.cuh) and
// launches it, one CTA per tile.
#include "gemm_kernel_m64.cuh"
#include "launch.cuh"

namespace tcl {
namespace {

// stages of one k-block (16 KB) or of two (32 KB, A through a 3-D map)
constexpr int kM64Stages1 = 8;
constexpr int kM64Stages2 = 6;

template <OutKind OK, int STAGES, int KPS>
cudaError_t launch_m64_t(const LaunchArgs& a) {
    using C = M64Cfg<OK, STAGES, KPS>;
    static bool done[64] = {};
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (!(dev >= 0 && dev < 64 && done[dev])) {
        err = cudaFuncSetAttribute(gemm_m64_kernel<OK, STAGES, KPS, 0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   C::SMEM_BYTES);
        if (err != cudaSuccess) return err;
        if (dev >= 0 && dev < 64) done[dev] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3(a.grid);
    cfg.blockDim = dim3(C::THREADS);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = a.stream;
    cfg.attrs = attr;
    cfg.numAttrs = 0;
    if (a.pdl) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, gemm_m64_kernel<OK, STAGES, KPS, 0>, a.tmA, a.tmB, a.p);
}

}  // namespace

cudaError_t launch_m64(const LaunchArgs& a, bool* found) {
    *found = a.in == InKind::BF16 && a.bn == 64 && (a.out == OutKind::F32 || a.out == OutKind::BF16) &&
             (a.m64 == 1 || a.m64 == 2);
    if (!*found) return cudaSuccess;
    if (a.m64 == 2)
        return a.out == OutKind::F32 ? launch_m64_t<OutKind::F32, kM64Stages2, 2>(a)
                                     : launch_m64_t<OutKind::BF16, kM64Stages2, 2>(a);
    return a.out == OutKind::F32 ? launch_m64_t<OutKind::F32, kM64Stages1, 1>(a)
                                 : launch_m64_t<OutKind::BF16, kM64Stages1, 1>(a);
}

int m64_stages(int kps) { return kps == 2 ? kM64Stages2 : kM64Stages1; }
int m64_smem_bytes(int kps) {
    return kps == 2 ? M64Cfg<OutKind::F32, kM64Stages2, 2>::SMEM_BYTES : M64Cfg<OutKind::F32, kM64Stages1, 1>::SMEM_BYTES;
}

}  // namespace tcl
