// Instantiates the two-SM (cta_group::2) GEMM variants and launches them as
// clusters of one CTA pair.
#include "launch.cuh"

namespace tcl {
namespace {

// attr must hold two entries; pdl adds programmatic stream serialisation
// (the kernel may start its set-up while the previous kernel in the stream
// finishes; it waits for that kernel before touching global memory).
template <InKind IK, OutKind OK, int BN, int STAGES, int SLOTS>
cudaLaunchConfig_t pair_config(int grid, cudaStream_t stream, cudaLaunchAttribute* attr, bool pdl = false) {
    using C = PairCfg<OK, BN, STAGES, SLOTS, IK>;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(C::THREADS);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = C::CL;
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

template <InKind IK, OutKind OK, int BN, int STAGES, int SLOTS>
cudaError_t prepare() {
    using C = PairCfg<OK, BN, STAGES, SLOTS, IK>;
    static bool done[64] = {};
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev >= 0 && dev < 64 && done[dev]) return cudaSuccess;
    err = cudaFuncSetAttribute(gemm_pair_kernel<OK, BN, STAGES, SLOTS, IK>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               C::SMEM_BYTES);
    if (err == cudaSuccess && dev >= 0 && dev < 64) done[dev] = true;
    return err;
}

template <InKind IK, OutKind OK, int BN, int STAGES, int SLOTS>
cudaError_t launch_pair(const LaunchArgs& a) {
    cudaError_t err = prepare<IK, OK, BN, STAGES, SLOTS>();
    if (err != cudaSuccess) return err;
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = pair_config<IK, OK, BN, STAGES, SLOTS>(a.grid, a.stream, attr, a.pdl);
    return cudaLaunchKernelEx(&cfg, gemm_pair_kernel<OK, BN, STAGES, SLOTS, IK>, a.tmA, a.tmB, a.tmC,
                              a.p);
}

template <InKind IK, OutKind OK, int BN, int STAGES, int SLOTS>
int max_clusters() {
    using C = PairCfg<OK, BN, STAGES, SLOTS, IK>;
    if (prepare<IK, OK, BN, STAGES, SLOTS>() != cudaSuccess) return 0;
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = pair_config<IK, OK, BN, STAGES, SLOTS>(C::CL, 0, attr);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, gemm_pair_kernel<OK, BN, STAGES, SLOTS, IK>, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

}  // namespace

#define TCL_PAIR_CASE(IK, OK, BN, ST, SL)                                                           \
    if (a.in == InKind::IK && a.out == OutKind::OK && a.bn == BN && a.stages == ST && a.slots == SL) { \
        *found = true;                                                                                \
        return launch_pair<InKind::IK, OutKind::OK, BN, ST, SL>(a);                                   \
    }

cudaError_t launch_group_pair(const LaunchArgs& a, bool* found) {
    *found = false;
    if (!a.pair || a.prod != PROD_TMA) return cudaErrorNotSupported;
    TCL_GROUP_PAIR(TCL_PAIR_CASE)
    return cudaErrorNotSupported;
}

#define TCL_PAIR_OCC(IK, OK, BN, ST, SL)                                                 \
    if (in == InKind::IK && out == OutKind::OK && bn == BN && stages == ST && slots == SL) \
        return max_clusters<InKind::IK, OutKind::OK, BN, ST, SL>();

int pair_max_clusters(InKind in, OutKind out, int bn, int stages, int slots) {
    TCL_GROUP_PAIR(TCL_PAIR_OCC)
    return 0;
}

}  // namespace tcl
