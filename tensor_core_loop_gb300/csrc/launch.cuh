// Internal launch interface between the C-ABI (api.cu) and the translation
// units that instantiate the GEMM kernel (k_*.cu). Not installed, not public.
#pragma once

#include <cuda_runtime.h>

#include "gemm_kernel.cuh"
#include "gemm_kernel_pair.cuh"

namespace tcl {

struct LaunchArgs {
    InKind in;
    OutKind out;
    int bn;
    int stages;
    int prod;   // PROD_TMA, PROD_SYNC or PROD_CPASYNC
    int pair;   // 1: two-SM kernel (one CTA pair per cluster); 0: one-SM kernel
    int slots;  // epilogue staging slabs per warp (two-SM kernel)
    int csk;    // > 1: K ranges of one tile summed in a cluster of this many CTAs (k_csk.cu)
    int m64;    // 1 or 2: 64×64 tiles with that many k-blocks per stage (k_m64.cu)
    bool pdl;   // programmatic dependent launch
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
cudaError_t launch_group_bf16_sync(const LaunchArgs& a, bool* found);
cudaError_t launch_group_bf16_cpasync(const LaunchArgs& a, bool* found);
cudaError_t launch_group_pair(const LaunchArgs& a, bool* found);
// Largest number of CTA-pair clusters of the given pair variant that can be
// resident at once on the current device (0 on error).
int pair_max_clusters(InKind in, OutKind out, int bn, int stages, int slots);
cudaError_t launch_group_tf32(const LaunchArgs& a, bool* found);
// Two-SM int8 kernel that widens its operands itself (k_s8_pair.cu): a.tmA and
// a.tmB map the int8 matrices (unswizzled boxes of 64 K × 128 rows and 128
// columns × 64 K), a.tmC the int32 output; s8_pair_stages() fp16 stages.
cudaError_t launch_s8_pair(const LaunchArgs& a);
// Cluster-summed K ranges (k_csk.cu): bf16 in, fp32 or bf16 C, 128×64 tiles,
// a.csk = 2 or 4 CTAs per tile; a.grid = tiles × a.csk.
cudaError_t launch_csk(const LaunchArgs& a, bool* found);
// 64×64 tiles, one CTA per tile (k_m64.cu): bf16 in, fp32 or bf16 C, a.bn = 64,
// a.m64 k-blocks per stage (1: a.tmA maps A in boxes of 64 K × 64 rows; 2: a
// 3-D map of A, boxes of 64 K × 64 rows × 2 k-blocks, and a.tmB boxes of 128
// K-rows); C is written from registers.
cudaError_t launch_m64(const LaunchArgs& a, bool* found);
int m64_stages(int kps);
int m64_smem_bytes(int kps);
int csk_stages();
int csk_smem_bytes(int cl);
int s8_pair_stages();
int s8_pair_smem_bytes();
int s8_pair_max_clusters();
// Die of each pair of SMs (k_diemap.cu): fills die_of_tpc[SM id / 2] with 0 or 1 and the
// pairs per die; false when the measurement shows no clear two groups.
bool calibrate_die_map(int sms, uint8_t* die_of_tpc, int max_tpc, int* n0, int* n1);

// int8 -> bf16 widening (exact) of two matrices in one launch: rows × cols of
// src (leading dimension ld_src) into a packed row-major buffer dst with ld_dst
// columns per row, the columns from `cols` up to the next multiple of 16 below
// ld_dst written as zeros; `vec` is set by the launcher.
struct S8Widen {
    const int8_t* src;
    long long ld_src;
    uint16_t* dst;
    long long ld_dst;
    int rows, cols, vec;
};
cudaError_t launch_s8_to_bf16(S8Widen a, S8Widen b, int sms, cudaStream_t stream);

// C (M×N, fp32 or bf16 rounded to nearest even) = sum over s = 0..splits-1, in
// that order, of the fp32 partial tiles W[s·rows_per_split + i][j] (leading dimension ldw).
cudaError_t launch_splitk_reduce(const float* W, long long ldw, long long rows_per_split, int splits, void* C,
                                 long long ldc, int M, int N, int out_bf16, int sms, cudaStream_t stream);

// dst[r][c] = src[r][c] (r < rows, c < cols), zeros elsewhere in rows_pad ×
// cols_pad; elements of 2 or 4 bytes, any alignment. With rows_pad = rows and
// cols_pad = cols it is a plain strided copy.
cudaError_t launch_repack(const void* src, long long ld_src, int rows, int cols, void* dst, long long ld_dst,
                          int rows_pad, int cols_pad, int elem_bytes, int sms, cudaStream_t stream);

// SIMT fp32 GEMM on the CUDA cores (k_simt.cu). vec: A, B, C bases 16-byte
// aligned and lda, ldb, ldc multiples of 4.
cudaError_t launch_sgemm_simt(const float* A, long long lda, const float* B, long long ldb, float* C, long long ldc,
                              int M, int N, int K, bool vec, cudaStream_t stream);


// One entry per instantiated variant, so the host can validate a requested
// configuration before it builds tensor maps.
struct VariantInfo {
    InKind in;
    OutKind out;
    int bn;
    int stages;
    int prod;
    int smem_bytes;
    int threads;
    int pair;
    int slots;
};
int variant_table(const VariantInfo** table);

template <InKind IK, OutKind OK, int BN, int STAGES, int PROD>
cudaError_t launch_variant(const LaunchArgs& a) {
    using C = KCfg<IK, OK, BN, STAGES, PROD>;
    auto kern = gemm_tc_kernel<IK, OK, BN, STAGES, PROD>;
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
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.grid);
    cfg.blockDim = dim3(C::THREADS);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = a.stream;
    cudaLaunchAttribute attr[1];
    if (a.pdl) {   // set-up may overlap the previous kernel in the stream (the kernel waits before any global access)
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, kern, a.tmA, a.tmB, a.tmC, a.p);
}

// The instantiated variants (input, output, BN, ring depth, producer),
// grouped by translation unit so that the groups compile in parallel.
#define TCL_GROUP_BF16_F32_BN256(X) \
    X(BF16, F32, 256, 1, 0) X(BF16, F32, 256, 2, 0) X(BF16, F32, 256, 3, 0) X(BF16, F32, 256, 4, 0)
#define TCL_GROUP_BF16_F32_BN128(X) \
    X(BF16, F32, 128, 1, 0) X(BF16, F32, 128, 2, 0) X(BF16, F32, 128, 4, 0) X(BF16, F32, 128, 6, 0) \
    X(BF16, F32, 64, 8, 0)
#define TCL_GROUP_BF16_MISC(X) \
    X(BF16, BF16, 256, 4, 0) X(BF16, BF16, 128, 6, 0) X(BF16, S32, 128, 6, 0) X(BF16, BF16, 64, 8, 0)
#define TCL_GROUP_BF16_SYNC(X) X(BF16, F32, 256, 1, 1) X(BF16, F32, 256, 2, 1) X(BF16, F32, 256, 4, 1)
#define TCL_GROUP_BF16_CPASYNC(X) \
    X(BF16, F32, 256, 1, 2) X(BF16, F32, 256, 2, 2) X(BF16, F32, 256, 3, 2) X(BF16, F32, 256, 4, 2)
#define TCL_GROUP_TF32(X) X(TF32, F32, 256, 4, 0) X(TF32, F32, 128, 6, 0)

#define TCL_VARIANT_INFO(IK, OK, BN, ST, PR)                                               \
    {InKind::IK, OutKind::OK, BN, ST, PR, KCfg<InKind::IK, OutKind::OK, BN, ST, PR>::SMEM_BYTES, \
     KCfg<InKind::IK, OutKind::OK, BN, ST, PR>::THREADS, 0, KCfg<InKind::IK, OutKind::OK, BN, ST, PR>::EPI_SLOTS},

// Two-SM variants (TMA producer, 256-row pair tiles): input, output, tile
// width, ring depth, epilogue staging slabs per warp.
#define TCL_GROUP_PAIR(X)                                                                                    \
    X(BF16, F32, 256, 6, 2) X(BF16, F32, 256, 4, 2) X(BF16, BF16, 256, 6, 2)                                 \
    X(BF16, F32, 224, 6, 2) X(BF16, F32, 224, 5, 4) X(BF16, BF16, 256, 5, 4)                                 \
    X(TF32, F32, 256, 6, 2) X(TF32, F32, 224, 6, 2) X(BF16, S32, 128, 8, 2)                                  \
    X(BF16, S32, 256, 6, 1)
#define TCL_PAIR_INFO(IK, OK, BN, ST, SL)                                                               \
    {InKind::IK, OutKind::OK, BN, ST, 0, PairCfg<OutKind::OK, BN, ST, SL, InKind::IK>::SMEM_BYTES,      \
     PairCfg<OutKind::OK, BN, ST, SL, InKind::IK>::THREADS, 1, SL},

#define TCL_VARIANT_CASE(IK, OK, BN, ST, PR)                                                           \
    if (!a.pair && a.in == InKind::IK && a.out == OutKind::OK && a.bn == BN && a.stages == ST && a.prod == PR) { \
        *found = true;                                                                                 \
        return launch_variant<InKind::IK, OutKind::OK, BN, ST, PR>(a);                                 \
    }

}  // namespace tcl
