// Internal launch interface between the C-ABI (api.cu) and the translation
// units that instantiate the GEMM kernel (k_*.cu). Not installed, not public.
#pragma once

#include <cuda_runtime.h>

#include "gemm_kernel.cuh"

namespace tcl {

struct LaunchArgs {
    InKind in;
    OutKind out;
    int bn;
    int stages;
    CUtensorMap tmA, tmB, tmC;
    GemmParams p;
    int grid;
    cudaStream_t stream;
};

// Launches the instantiation matching (in, out, bn, stages). Sets *found to
// false (and launches nothing) when this unit does not hold that variant.
cudaError_t launch_group_bf16_f32_bn256(const LaunchArgs& a, bool* found);
cudaError_t launch_group_bf16_f32_bn128(const LaunchArgs& a, bool* found);
cudaError_t launch_group_bf16_misc(const LaunchArgs& a, bool* found);
cudaError_t launch_group_tf32(const LaunchArgs& a, bool* found);

// int8 -> bf16 widening (exact) into a packed row-major buffer with ld_dst
// columns per row; columns past `cols` are left untouched.
cudaError_t launch_s8_to_bf16(const int8_t* src, long long ld_src, void* dst, long long ld_dst,
                              int rows, int cols, int sms, cudaStream_t stream);

// dst (cols × rows) = transpose of src (rows × cols), fp32, bit for bit.
cudaError_t launch_transpose_f32(const float* src, long long ld_src, float* dst, long long ld_dst, int rows,
                                 int cols, int sms, cudaStream_t stream);

// One entry per instantiated variant, so the host can validate a requested
// configuration before it builds tensor maps.
struct VariantInfo {
    InKind in;
    OutKind out;
    int bn;
    int stages;
    int smem_bytes;
};
int variant_table(const VariantInfo** table);

template <InKind IK, OutKind OK, int BN, int STAGES>
cudaError_t launch_variant(const LaunchArgs& a) {
    using C = KCfg<IK, OK, BN, STAGES>;
    auto kern = gemm_tc_kernel<IK, OK, BN, STAGES>;
    // The shared-memory opt-in is per function and device: set it once per device.
    static bool attr_done[64] = {};
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= 64 || !attr_done[dev]) {
        err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
        if (err != cudaSuccess) return err;
        if (dev >= 0 && dev < 64) attr_done[dev] = true;
    }
    kern<<<a.grid, C::THREADS, C::SMEM_BYTES, a.stream>>>(a.tmA, a.tmB, a.tmC, a.p);
    return cudaGetLastError();
}

// The instantiated variants, grouped by translation unit (compiled in parallel).
#define TCL_GROUP_BF16_F32_BN256(X) \
    X(BF16, F32, 256, 1) X(BF16, F32, 256, 2) X(BF16, F32, 256, 3) X(BF16, F32, 256, 4)
#define TCL_GROUP_BF16_F32_BN128(X) \
    X(BF16, F32, 128, 1) X(BF16, F32, 128, 2) X(BF16, F32, 128, 4) X(BF16, F32, 128, 6)
#define TCL_GROUP_BF16_MISC(X) X(BF16, BF16, 256, 4) X(BF16, BF16, 128, 6) X(BF16, S32, 128, 6)
#define TCL_GROUP_TF32(X) X(TF32, F32, 256, 4) X(TF32, F32, 128, 6)

#define TCL_VARIANT_INFO(IK, OK, BN, ST) \
    {InKind::IK, OutKind::OK, BN, ST, KCfg<InKind::IK, OutKind::OK, BN, ST>::SMEM_BYTES},

#define TCL_VARIANT_CASE(IK, OK, BN, ST)                                                   \
    if (a.in == InKind::IK && a.out == OutKind::OK && a.bn == BN && a.stages == ST) {      \
        *found = true;                                                                     \
        return launch_variant<InKind::IK, OutKind::OK, BN, ST>(a);                         \
    }

}  // namespace tcl
