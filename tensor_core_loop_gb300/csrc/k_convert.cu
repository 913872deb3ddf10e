// Passes that run before or after the GEMM kernel on some paths:
//   * exact int8 -> bf16 widening (integer GEMM);
//   * the fixed-order sum of split-K partial tiles;
//   * 2-D copies with zero fill, for operands or outputs whose base address or
//     leading dimension is off the 16-byte grid the tensor copies need.
//
// int8 -> bf16:
// Every int8 value (|x| <= 128) has at most 8 significant bits, so it is
// represented exactly by bf16; the bf16 pattern is the upper half of the
// binary32 encoding of the integer. Both operands are widened by one launch;
// a block takes one row at a time (rows of A, then rows of B) and its threads
// the row's 16-element chunks: one 16-byte load, two 16-byte stores. The
// destination rows are padded to a multiple of 8 elements (the padding is
// written as zeros). When the source base and leading dimension are 16-byte
// aligned (`vec`), full chunks use vector loads; otherwise, and at a ragged row
// tail, bytes are read one by one.
#include <cuda_bf16.h>

#include <cstdint>

#include "launch.cuh"

namespace tcl {

// The binary32 value of an integer |x| <= 128 without a conversion instruction:
// 1.5·2^23 + x is exact in [2^23, 2^24) (unit in the last place 1), so its bit
// pattern is that of 1.5·2^23 plus x, and subtracting 1.5·2^23 leaves x exactly.
__device__ __forceinline__ uint32_t s8_f32_bits(int x) {
    return __float_as_uint(__int_as_float(0x4B400000 + x) - 12582912.0f);
}

__device__ __forceinline__ uint32_t s8_pair_to_bf16x2(int lo, int hi) {
    return (s8_f32_bits(lo) >> 16) | (s8_f32_bits(hi) & 0xFFFF0000u);
}

// One block per row of A, then of B (the grid covers every row: on GB300 this
// ran ~4 µs faster at 8192 rows of 4096 than eight resident blocks per SM
// striding over the rows).
__global__ void __launch_bounds__(256) s8_to_bf16_kernel(S8Widen a, S8Widen b) {
    // the GEMM that reads these copies is launched programmatically behind this
    // pass: let it be scheduled now; it waits for this grid to complete (and its
    // writes to be visible) before it reads anything
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const long long total = static_cast<long long>(a.rows) + b.rows;
    for (long long rr = blockIdx.x; rr < total; rr += gridDim.x) {
        const bool in_a = rr < a.rows;
        const S8Widen& job = in_a ? a : b;
        const long long r = in_a ? rr : rr - a.rows;
        const int cols = job.cols;
        const int chunks_per_row = (cols + 15) / 16;
        for (int ch = threadIdx.x; ch < chunks_per_row; ch += blockDim.x) {
            const int c0 = ch * 16;
            const int8_t* s = job.src + r * job.ld_src + c0;
            uint16_t* d = job.dst + r * job.ld_dst + c0;
            if (c0 + 16 <= cols) {
                int4 raw;
                if (job.vec) {
                    raw = *reinterpret_cast<const int4*>(s);
                } else {
                    int8_t* rb = reinterpret_cast<int8_t*>(&raw);
#pragma unroll
                    for (int j = 0; j < 16; ++j) rb[j] = s[j];
                }
                const int8_t* v = reinterpret_cast<const int8_t*>(&raw);
                uint4 o0, o1;
                o0.x = s8_pair_to_bf16x2(v[0], v[1]);
                o0.y = s8_pair_to_bf16x2(v[2], v[3]);
                o0.z = s8_pair_to_bf16x2(v[4], v[5]);
                o0.w = s8_pair_to_bf16x2(v[6], v[7]);
                o1.x = s8_pair_to_bf16x2(v[8], v[9]);
                o1.y = s8_pair_to_bf16x2(v[10], v[11]);
                o1.z = s8_pair_to_bf16x2(v[12], v[13]);
                o1.w = s8_pair_to_bf16x2(v[14], v[15]);
                reinterpret_cast<uint4*>(d)[0] = o0;
                reinterpret_cast<uint4*>(d)[1] = o1;
            } else {
                // ragged row end: convert what is there and zero the padding up to ld_dst,
                // so that tensor loads that round the row end up to 16 bytes read zeros
                int j = 0;
                for (; c0 + j < cols; ++j) d[j] = static_cast<uint16_t>(s8_f32_bits(s[j]) >> 16);
                for (; c0 + j < job.ld_dst && j < 16; ++j) d[j] = 0;
            }
        }
    }
}

cudaError_t launch_s8_to_bf16(S8Widen a, S8Widen b, int sms, cudaStream_t stream) {
    a.vec = (reinterpret_cast<uintptr_t>(a.src) % 16 == 0 && a.ld_src % 16 == 0) ? 1 : 0;
    b.vec = (reinterpret_cast<uintptr_t>(b.src) % 16 == 0 && b.ld_src % 16 == 0) ? 1 : 0;
    const long long rows = static_cast<long long>(a.rows) + b.rows;
    long long blocks = rows;
    const long long cap = 1LL << 30;   // rows beyond the grid: row-stride
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    (void)sms;
    s8_to_bf16_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(a, b);
    return cudaGetLastError();
}

// dst[r][c] = src[r][c] for r < rows, c < cols, and 0 for the rest of the
// rows_pad × cols_pad block (elements of T; any source or destination
// alignment, so element by element, consecutive threads on consecutive columns).
template <class T>
__global__ void __launch_bounds__(256) repack_kernel(const T* __restrict__ src, long long ld_src, int rows,
                                                      int cols, T* __restrict__ dst, long long ld_dst, int rows_pad,
                                                      int cols_pad) {
    const long long total = static_cast<long long>(rows_pad) * cols_pad;
    for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; idx < total;
         idx += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int r = static_cast<int>(idx / cols_pad);
        const int c = static_cast<int>(idx - static_cast<long long>(r) * cols_pad);
        dst[r * ld_dst + c] = (r < rows && c < cols) ? src[r * ld_src + c] : T(0);
    }
}

cudaError_t launch_repack(const void* src, long long ld_src, int rows, int cols, void* dst, long long ld_dst,
                          int rows_pad, int cols_pad, int elem_bytes, int sms, cudaStream_t stream) {
    const long long total = static_cast<long long>(rows_pad) * cols_pad;
    long long blocks = (total + 255) / 256;
    const long long cap = static_cast<long long>(sms) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    if (elem_bytes == 2)
        repack_kernel<uint16_t><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
            static_cast<const uint16_t*>(src), ld_src, rows, cols, static_cast<uint16_t*>(dst), ld_dst, rows_pad,
            cols_pad);
    else if (elem_bytes == 4)
        repack_kernel<uint32_t><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
            static_cast<const uint32_t*>(src), ld_src, rows, cols, static_cast<uint32_t*>(dst), ld_dst, rows_pad,
            cols_pad);
    else
        return cudaErrorInvalidValue;
    return cudaGetLastError();
}

// Split-K reduction: each thread owns four consecutive columns of one row and
// adds the splits' fp32 partial tiles in order s = 0, 1, ..., splits-1 (the
// result does not depend on which CTA finished first), then writes fp32 or
// bf16 (round to nearest even). The workspace rows are padded to a multiple
// of 4 columns, so its loads are always 16-byte vectors; C gets vector stores
// where a whole chunk is inside the row and scalar stores at a ragged edge.
__global__ void __launch_bounds__(256) splitk_reduce_kernel(const float* __restrict__ W, long long ldw,
                                                             long long split_stride, int splits,
                                                             void* __restrict__ C, long long ldc, int M, int N,
                                                             int out_bf16) {
    const int chunks = (N + 3) / 4;
    const long long total = static_cast<long long>(M) * chunks;
    // launched programmatically behind the GEMM: wait for its partial tiles
    asm volatile("griddepcontrol.wait;" ::: "memory");
    for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; idx < total;
         idx += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int r = static_cast<int>(idx / chunks);
        const int c0 = static_cast<int>(idx - static_cast<long long>(r) * chunks) * 4;
        const float* w = W + r * ldw + c0;
        float4 acc = *reinterpret_cast<const float4*>(w);
        for (int sp = 1; sp < splits; ++sp) {
            const float4 v = *reinterpret_cast<const float4*>(w + sp * split_stride);
            acc.x += v.x;
            acc.y += v.y;
            acc.z += v.z;
            acc.w += v.w;
        }
        const float vals[4] = {acc.x, acc.y, acc.z, acc.w};
        const bool whole = c0 + 4 <= N;
        if (!out_bf16) {
            float* dst = static_cast<float*>(C) + r * ldc + c0;
            if (whole) {
                *reinterpret_cast<float4*>(dst) = acc;
            } else {
                for (int j = 0; c0 + j < N; ++j) dst[j] = vals[j];
            }
        } else {
            __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(C) + r * ldc + c0;
            if (whole) {
                __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
                __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
                uint2 packed;
                packed.x = *reinterpret_cast<uint32_t*>(&lo);
                packed.y = *reinterpret_cast<uint32_t*>(&hi);
                *reinterpret_cast<uint2*>(dst) = packed;
            } else {
                for (int j = 0; c0 + j < N; ++j) dst[j] = __float2bfloat16_rn(vals[j]);
            }
        }
    }
}

cudaError_t launch_splitk_reduce(const float* W, long long ldw, long long rows_per_split, int splits, void* C,
                                 long long ldc, int M, int N, int out_bf16, int sms, cudaStream_t stream) {
    const long long total = static_cast<long long>(M) * ((N + 3) / 4);
    long long blocks = (total + 255) / 256;
    const long long cap = static_cast<long long>(sms) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    // Programmatic launch: the blocks are scheduled while the GEMM finishes and
    // wait (griddepcontrol.wait) until it has completed and its partials are visible.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks));
    cfg.blockDim = dim3(256);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, splitk_reduce_kernel, W, ldw, rows_per_split * ldw, splits, C, ldc, M, N,
                              out_bf16);
}

}  // namespace tcl
