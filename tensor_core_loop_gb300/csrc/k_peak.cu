// MMA-only peak probe: back-to-back tcgen05.mma on operands already in shared
// memory, no loads, no epilogue. It measures the tensor pipe's own rate per SM
// (cycles per MMA instruction, from %clock64 around the issue loop and the
// final commit), which is the denominator of the clock-corrected roofline.
#include <cuda_runtime.h>

#include "launch.cuh"
#include "tcl_gemm.h"

namespace tcl {
namespace {

// align slack, 4 stages of A (128 rows × 128 B) and B (256 rows × 128 B), barrier
constexpr int kPeakStages = 4;
constexpr int kPeakA = 16384, kPeakB = 32768;
constexpr int kPeakSmem = 1024 + kPeakStages * (kPeakA + kPeakB) + 256;
constexpr int kPeakRequest = 232448 - 1024;

// flags: bit 0 — chain every MMA into one accumulator (as a GEMM tile does)
//        instead of alternating two; bit 1 — walk the operand addresses like a
//        GEMM k-loop (4 k-slices × 4 stages) instead of reusing one k-slice;
//        bit 3 — per group of MMAs, what a GEMM k-block adds (a stage-barrier
//        wait, a fence and a commit); bit 4 — of that, the wait and fence only;
//        bit 5 — the commit only; bit 6 — groups of eight MMAs (two k-blocks)
//        instead of four.
template <int N, bool TF32, bool B_MN>
__global__ void __launch_bounds__(128, 1) mma_peak_kernel(int iters, int flags, unsigned long long timeout_ns,
                                                          unsigned long long* cycles, unsigned int* status) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    const uint32_t sa0 = ptx::smem_u32(smem);
    const uint32_t sb0 = sa0 + kPeakStages * kPeakA;
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kPeakStages * (kPeakA + kPeakB));
    uint32_t* holder = reinterpret_cast<uint32_t*>(bar + 3);   // bar[0]: completion, bar[1]: ready, bar[2]: commits
    // operands: a fixed pseudo-random bf16/fp32 pattern of moderate magnitude
    for (int i = threadIdx.x; i < kPeakStages * (kPeakA + kPeakB) / 4; i += blockDim.x) {
        const uint32_t h = (static_cast<uint32_t>(i) * 2654435761u) >> 9;
        reinterpret_cast<uint32_t*>(smem)[i] = TF32 ? (0x3F000000u | (h & 0x7FFFFFu)) : (0x3F003F00u | (h & 0x007F007Fu));
    }
    ptx::fence_proxy_async_smem();
    if (threadIdx.x == 0) {
        ptx::mbar_init(ptx::smem_u32(bar), 1);
        ptx::mbar_init(ptx::smem_u32(bar + 1), 1);
        ptx::mbar_init(ptx::smem_u32(bar + 2), 1);
        ptx::fence_mbar_init();
    }
    if (threadIdx.x < 32) {
        ptx::tmem_alloc(ptx::smem_u32(holder), 512);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *holder;
    if (threadIdx.x < 32) {
        // Warp 0 runs the issue loop converged; one elected lane issues every MMA
        // (four per k-slice group, as the GEMM kernels do), so the probe measures
        // the tensor pipe rather than a lone thread's loop.
        constexpr uint32_t fmt = TF32 ? 2u : 1u;
        // A K-major; B K-major (N rows of 128 B) or N-major (N/64 column groups of
        // 16 K-rows × 128 B, 2 KB apart), as in one k-slice of a GEMM tile
        constexpr uint32_t idesc = ptx::make_idesc(fmt, fmt, 0, B_MN ? 1u : 0u, 128, N);
        const bool chain = flags & 1, walk = flags & 2;
        // bit 2: N-major B laid out as a GEMM stage holds it, 64-column groups of
        // BK = 64 rows (8 KB apart) instead of 16 rows (2 KB apart)
        const uint32_t b_lbo = (flags & 4) ? 8192u : 2048u;
        const uint64_t t0 = ptx::clock64();
        const bool do_wait = flags & (8 | 16), do_commit = flags & (8 | 32);
        const int group = (flags & 64) ? 8 : 4;
        for (int i = 0; i < iters; i += 4) {
            // four MMAs on the four k-slices of one stage (or on one k-slice)
            const int st = walk ? ((i / 4) % kPeakStages) : 0;
            const uint32_t sa = sa0 + st * kPeakA, sb = sb0 + st * kPeakB;
            uint64_t ad[4], bd[4];
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                const int k = walk ? ks : 0;
                ad[ks] = ptx::sdesc_sw128(sa + k * 32, 16, 1024);
                bd[ks] = B_MN ? ptx::sdesc_sw128(sb + k * (TF32 ? 8 : 16) * 128, b_lbo, 1024)
                              : ptx::sdesc_sw128(sb + k * 32, 16, 1024);
            }
            const uint32_t d = tmem + ((!chain && ((i / 4) & 1)) ? N : 0);
            if (do_wait && i % group == 0) {
                // the rest of a GEMM issue loop: wait on a (completed) stage barrier, fence
                __all_sync(0xffffffffu, ptx::mbar_try_wait(ptx::smem_u32(bar + 1), 1));
                ptx::tc_fence_after();
            }
            const uint32_t acc = i >= (chain ? 4 : 8) ? 1u : 0u;
            if constexpr (TF32)
                ptx::mma_tf32_x4_elected(d, ad[0], bd[0], ad[1], bd[1], ad[2], bd[2], ad[3], bd[3], idesc, acc);
            else
                ptx::mma_f16_x4_elected(d, ad[0], bd[0], ad[1], bd[1], ad[2], bd[2], ad[3], bd[3], idesc, acc);
            if (do_commit && (i + 4) % group == 0) ptx::mma_commit_elected(ptx::smem_u32(bar + 2));   // ... and commit
        }
        ptx::mma_commit_elected(ptx::smem_u32(bar));
        bool done = false;
        if ((threadIdx.x & 31) == 0) {
            const uint64_t t_start = ptx::globaltimer_ns();
            while (!(done = ptx::mbar_try_wait(ptx::smem_u32(bar), 0))) {
                if (ptx::globaltimer_ns() - t_start > timeout_ns) break;
            }
            const uint64_t t1 = ptx::clock64();
            cycles[blockIdx.x] = done ? (t1 - t0) : 0ull;
            if (!done) atomicCAS(status, 0u, static_cast<unsigned int>(DEV_TIMEOUT_MMA_FULL));
        }
        __syncwarp();
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (threadIdx.x < 32) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 512);
    }
}

// Warp-level MMA (mma.sync), the instruction the pages' kernels are built on:
// 8 warps per CTA, each `iters` rounds of eight independent MMAs on register
// operands, no loads. S8: m16n8k32 int8 → int32, the only int8 tensor-core
// instruction sm_103a accepts (8192 ops each); else m16n8k16 bf16 → fp32 (4096
// flop each). cycles[blockIdx] = %clock64 from the first issue to the last.
constexpr int kWarpMmaWarps = 8, kWarpMmaChains = 8;
template <bool S8>
__global__ void __launch_bounds__(32 * kWarpMmaWarps, 1) warp_mma_peak_kernel(int iters, unsigned long long* cycles) {
    uint32_t a[4], b[2];
#pragma unroll
    for (int i = 0; i < 4; ++i) a[i] = ((threadIdx.x + 7u * i) * 2654435761u >> 8) & (S8 ? 0x3F3F3F3Fu : 0x007F007Fu);
#pragma unroll
    for (int i = 0; i < 2; ++i) b[i] = ((threadIdx.x + 5u * i) * 40503u >> 4) & (S8 ? 0x1F1F1F1Fu : 0x007F007Fu);
    if (!S8) {
#pragma unroll
        for (int i = 0; i < 4; ++i) a[i] |= 0x3F003F00u;   // bf16 values in [0.5, 1)
#pragma unroll
        for (int i = 0; i < 2; ++i) b[i] |= 0x3F003F00u;
    }
    uint32_t acc[kWarpMmaChains][4] = {};
    __syncthreads();
    const uint64_t t0 = ptx::clock64();
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int j = 0; j < kWarpMmaChains; ++j) {
            if constexpr (S8)
                asm volatile(
                    "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                    "{%0,%1,%2,%3};"
                    : "+r"(acc[j][0]), "+r"(acc[j][1]), "+r"(acc[j][2]), "+r"(acc[j][3])
                    : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
            else
                asm volatile(
                    "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                    "{%0,%1,%2,%3};"
                    : "+r"(acc[j][0]), "+r"(acc[j][1]), "+r"(acc[j][2]), "+r"(acc[j][3])
                    : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
        }
    }
    __syncthreads();
    const uint64_t t1 = ptx::clock64();
    if (threadIdx.x == 0) cycles[blockIdx.x] = t1 - t0;
    if (iters < 0) {   // never (iters >= 8): keeps the sums live for the compiler
        uint32_t x = 0;
#pragma unroll
        for (int j = 0; j < kWarpMmaChains; ++j) x ^= acc[j][0] ^ acc[j][1] ^ acc[j][2] ^ acc[j][3];
        cycles[blockIdx.x] = x;
    }
}

template <int N, bool TF32, bool B_MN>
cudaError_t launch_peak(int iters, int flags, int grid, unsigned long long* cycles, unsigned int* status,
                        cudaStream_t stream) {
    auto kern = mma_peak_kernel<N, TF32, B_MN>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kPeakRequest);
    if (err != cudaSuccess) return err;
    kern<<<grid, 128, kPeakRequest, stream>>>(iters, flags, 1000000000ull, cycles, status);
    return cudaGetLastError();
}

template <bool TF32, bool B_MN>
cudaError_t launch_peak_n(int n, int iters, int flags, int grid, unsigned long long* cycles, unsigned int* status,
                          cudaStream_t stream) {
    switch (n) {
        case 128: return launch_peak<128, TF32, B_MN>(iters, flags, grid, cycles, status, stream);
        case 192: return launch_peak<192, TF32, B_MN>(iters, flags, grid, cycles, status, stream);
        case 224: return launch_peak<224, TF32, B_MN>(iters, flags, grid, cycles, status, stream);
        default: return launch_peak<256, TF32, B_MN>(iters, flags, grid, cycles, status, stream);
    }
}

}  // namespace

int device_context(int* dev, int* sms, unsigned int** status);   // api.cu

}  // namespace tcl

using namespace tcl;

extern "C" TCL_API int tcl_mma_peak(int in_kind, int n, int b_mn, int flags, int iters, int grid,
                                    unsigned long long* cycles, cudaStream_t stream) {
    if (!cycles) return TCL_ERR_NULL;
    if (iters < 8 || iters % 4 || grid < 1 || (n != 128 && n != 192 && n != 224 && n != 256) ||
        (in_kind != 0 && in_kind != 1 && in_kind != 2) ||
        (b_mn != 0 && b_mn != 1) || (in_kind != 0 && b_mn))
        return TCL_ERR_DIMS;
    static_assert(kPeakSmem <= kPeakRequest, "probe fits its shared memory request");
    const bool warp_mma = in_kind == 2 || (flags & 128);
    if (flags < 0 || flags > 255 || ((flags & 64) && iters % 8) || (warp_mma && (flags & 127)) ||
        (in_kind == 1 && (flags & 128)))
        return TCL_ERR_CONFIG;
    int dev = 0, sms = 0;
    unsigned int* status = nullptr;
    int st = device_context(&dev, &sms, &status);
    if (st) return st;
    cudaError_t err;
    if (warp_mma) {
        if (in_kind == 2)
            warp_mma_peak_kernel<true><<<grid, 32 * kWarpMmaWarps, 0, stream>>>(iters, cycles);
        else
            warp_mma_peak_kernel<false><<<grid, 32 * kWarpMmaWarps, 0, stream>>>(iters, cycles);
        err = cudaGetLastError();
    } else if (in_kind == 1)
        err = launch_peak_n<true, false>(n, iters, flags, grid, cycles, status, stream);
    else if (b_mn)
        err = launch_peak_n<false, true>(n, iters, flags, grid, cycles, status, stream);
    else
        err = launch_peak_n<false, false>(n, iters, flags, grid, cycles, status, stream);
    if (err != cudaSuccess) {
        cudaGetLastError();
        return TCL_ERR_LAUNCH;
    }
    return TCL_OK;
}
