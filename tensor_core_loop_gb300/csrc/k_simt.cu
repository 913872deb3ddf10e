// SIMT fp32 GEMM on the CUDA cores (fused multiply-adds, no tensor cores): the
// architecture-level anchor that the pages set beside their tensor-core
// ladders ("4.1 CUDA GEMM 算子性能优化" §4–§9: thread-block tiling, register
// (thread) tiling, A transposed in shared memory so both operands are read as
// float4, conflict-free shared-memory layouts, double buffering through
// registers).
//
// One CTA of 256 threads (one per SM: the registers go to the 64
// accumulators and the next step's operands, and 1024 tiles of a 4096² C make
// 6.7 waves of 152 instead of 3.4 of 304) computes a 128×128 tile of C,
// walking K in steps of 16. Thread (tx, ty) of the 16×16 grid owns an 8×8 block of C made of the rows
// ty·4..ty·4+3 and 64+ty·4..64+ty·4+3 and the columns tx·4.. and 64+tx·4..:
// every shared-memory read is a float4, a warp's A reads hit two addresses and
// its B reads 256 contiguous bytes. The next K-step is loaded into registers
// while the current one is multiplied, then stored into the other shared
// buffer: one barrier per K-step.
//
// Accumulation: each output is a chain of fmaf in increasing k, starting from
// 0 — one rounding per step, so |C - C_exact| <= K·u/(1 - K·u) · Σ|a·b| with
// u = 2^-24.
#include <cuda_runtime.h>

#include <cstdint>

#include "launch.cuh"
#include "tcl_gemm.h"

namespace tcl {
namespace {

constexpr int SM_ = 128, SN_ = 128, SK_ = 16, ST_ = 256;

// VEC: every row of A, B and C starts 16-byte aligned (bases and leading
// dimensions), so in-range groups of four consecutive elements move as float4.
template <bool VEC>
__global__ void __launch_bounds__(ST_, 1) sgemm_simt_kernel(const float* __restrict__ A, long long lda,
                                                            const float* __restrict__ B, long long ldb,
                                                            float* __restrict__ C, long long ldc, int M, int N,
                                                            int K) {
    __shared__ __align__(16) float As[2][SK_][SM_];   // A transposed: As[k][m]
    __shared__ __align__(16) float Bs[2][SK_][SN_];   // Bs[k][n]
    const int tid = threadIdx.x;
    const int tx = tid & 15, ty = tid >> 4;
    const int m0 = blockIdx.y * SM_, n0 = blockIdx.x * SN_;
    // Global -> register assignment: A row am, k offsets ak..ak+7 (a warp takes 32
    // consecutive rows, so the transposed stores are conflict-free); B row bk,
    // columns bn..bn+3 and 64+bn..64+bn+3 (16 lanes store 256 contiguous bytes).
    const int am = tid & 127, ak = (tid >> 7) * 8;
    const int bk = tid >> 4, bn = (tid & 15) * 4;
    float ra[8], rb[8];

    auto load = [&](int k0) {
        const int gm = m0 + am, gka = k0 + ak;
        if (VEC && gm < M && gka + 8 <= K) {
            const float4* p = reinterpret_cast<const float4*>(A + gm * lda + gka);
            const float4 x = __ldg(p), y = __ldg(p + 1);
            ra[0] = x.x, ra[1] = x.y, ra[2] = x.z, ra[3] = x.w, ra[4] = y.x, ra[5] = y.y, ra[6] = y.z, ra[7] = y.w;
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) ra[j] = (gm < M && gka + j < K) ? __ldg(A + gm * lda + gka + j) : 0.0f;
        }
        const int gkb = k0 + bk;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int gn = n0 + h * 64 + bn;
            float* r = rb + 4 * h;
            if (VEC && gkb < K && gn + 4 <= N) {
                const float4 x = __ldg(reinterpret_cast<const float4*>(B + gkb * ldb + gn));
                r[0] = x.x, r[1] = x.y, r[2] = x.z, r[3] = x.w;
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j) r[j] = (gkb < K && gn + j < N) ? __ldg(B + gkb * ldb + gn + j) : 0.0f;
            }
        }
    };
    auto store = [&](int buf) {
#pragma unroll
        for (int j = 0; j < 8; ++j) As[buf][ak + j][am] = ra[j];
        *reinterpret_cast<float4*>(&Bs[buf][bk][bn]) = make_float4(rb[0], rb[1], rb[2], rb[3]);
        *reinterpret_cast<float4*>(&Bs[buf][bk][64 + bn]) = make_float4(rb[4], rb[5], rb[6], rb[7]);
    };

    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.0f;

    const int ksteps = (K + SK_ - 1) / SK_;
    load(0);
    store(0);
    __syncthreads();
    for (int ks = 0; ks < ksteps; ++ks) {
        const int cur = ks & 1;
        if (ks + 1 < ksteps) load((ks + 1) * SK_);   // in flight while this step's FMAs run
#pragma unroll
        for (int k = 0; k < SK_; ++k) {
            const float4 a0 = *reinterpret_cast<const float4*>(&As[cur][k][ty * 4]);
            const float4 a1 = *reinterpret_cast<const float4*>(&As[cur][k][64 + ty * 4]);
            const float4 b0 = *reinterpret_cast<const float4*>(&Bs[cur][k][tx * 4]);
            const float4 b1 = *reinterpret_cast<const float4*>(&Bs[cur][k][64 + tx * 4]);
            const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            const float b[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        if (ks + 1 < ksteps) store(cur ^ 1);   // the other buffer was last read before the previous barrier
        __syncthreads();
    }

#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int gm = m0 + (i < 4 ? ty * 4 + i : 64 + ty * 4 + i - 4);
        if (gm >= M) continue;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int gn = n0 + h * 64 + tx * 4;
            float* dst = C + gm * ldc + gn;
            const float* v = &acc[i][h * 4];
            if (VEC && gn + 4 <= N) {
                *reinterpret_cast<float4*>(dst) = make_float4(v[0], v[1], v[2], v[3]);
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (gn + j < N) dst[j] = v[j];
            }
        }
    }
}

}  // namespace

cudaError_t launch_sgemm_simt(const float* A, long long lda, const float* B, long long ldb, float* C, long long ldc,
                              int M, int N, int K, bool vec, cudaStream_t stream) {
    const dim3 grid((N + SN_ - 1) / SN_, (M + SM_ - 1) / SM_);
    if (vec)
        sgemm_simt_kernel<true><<<grid, ST_, 0, stream>>>(A, lda, B, ldb, C, ldc, M, N, K);
    else
        sgemm_simt_kernel<false><<<grid, ST_, 0, stream>>>(A, lda, B, ldb, C, ldc, M, N, K);
    return cudaGetLastError();
}

}  // namespace tcl
