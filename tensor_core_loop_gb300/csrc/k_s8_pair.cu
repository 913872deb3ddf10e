// Instantiates the two-SM int8 kernel that widens its operands in the kernel
// (gemm_kernel_s8.cuh) and launches it as clusters of one CTA pair.
#include "gemm_kernel_s8.cuh"
#include "launch.cuh"

namespace tcl {
namespace {

constexpr int kS8Stages = 4;   // fp16 stages the MMA reads
constexpr int kS8Raw = 4;      // raw int8 slots the TMA fills

cudaLaunchConfig_t s8_config(int grid, cudaStream_t stream, cudaLaunchAttribute* attr, bool pdl) {
    using C = S8PairCfg<kS8Stages, kS8Raw>;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(C::THREADS);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (pdl) {
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.numAttrs = 2;
    }
    return cfg;
}

cudaError_t prepare_s8() {
    static bool done[64] = {};
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev >= 0 && dev < 64 && done[dev]) return cudaSuccess;
    err = cudaFuncSetAttribute(gemm_s8_pair_kernel<kS8Stages, kS8Raw>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               S8PairCfg<kS8Stages, kS8Raw>::SMEM_BYTES);
    if (err == cudaSuccess && dev >= 0 && dev < 64) done[dev] = true;
    return err;
}

}  // namespace

int s8_pair_stages() { return kS8Stages; }
int s8_pair_smem_bytes() { return S8PairCfg<kS8Stages, kS8Raw>::SMEM_BYTES; }

cudaError_t launch_s8_pair(const LaunchArgs& a) {
    cudaError_t err = prepare_s8();
    if (err != cudaSuccess) return err;
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = s8_config(a.grid, a.stream, attr, a.pdl);
    return cudaLaunchKernelEx(&cfg, gemm_s8_pair_kernel<kS8Stages, kS8Raw>, a.tmA, a.tmB, a.tmC, a.p);
}

int s8_pair_max_clusters() {
    if (prepare_s8() != cudaSuccess) return 0;
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = s8_config(2, 0, attr, false);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, gemm_s8_pair_kernel<kS8Stages, kS8Raw>, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

}  // namespace tcl
