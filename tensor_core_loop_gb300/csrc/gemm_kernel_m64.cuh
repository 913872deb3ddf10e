// 64×64 output tiles for small grids: one CTA per tile, tcgen05.mma with M = 64.
//
// At M = N = 512 a grid of 128-row tiles leaves most SMs idle and each CTA's
// time is a chain of fixed latencies plus its operand stream: with 128×64
// tiles every k-block brings 16 KB of A and 8 KB of B into one SM. Tiles of 64
// rows halve A's share (8 KB + 8 KB per k-block) and double the CTAs (64 at
// 512²), so each SM's stream of operands is a third shorter.
//
// Pipeline as in the one-SM kernel (TMA ring of STAGES stages with full/empty
// mbarriers, one elected thread issuing four tcgen05.mma of 64×64×16 per
// 64-deep k-block, one TMEM accumulator of 64 columns). A stage holds KPS
// k-blocks brought by two tensor copies whatever KPS is (KPS = 2: A through a
// 3-D map whose third dimension steps from one 64-wide K block to the next, so
// one box is two 8 KB swizzle tiles; B in a box of 128 K-rows): on GB300 the
// stages of two 8 KB boxes landed ~445 cycles apart for 64 cycles of MMA work,
// and a tensor copy's cost barely depended on its size (a microbenchmark: the
// issuing thread busy ~150–190 cycles per copy from 4 to 32 KB). The M = 64 accumulator
// occupies 16 TMEM lanes of each 32-lane quarter (rows 16q..16q+15 in lanes
// 32q..32q+15; LAYOUT 1 would be rows 0..63 in lanes 0..63); each of the four
// epilogue warps reads its quarter and its first 16 lanes store their rows
// straight from registers (16-byte stores where the row is whole and aligned,
// element stores at a ragged edge), without a staging tile.
#pragma once

#include "gemm_kernel.cuh"

namespace tcl {

template <OutKind OK, int STAGES_, int KPS_ = 1, int LAYOUT_ = 0>
struct M64Cfg {
    static constexpr int STAGES = STAGES_;
    static constexpr int KPS = KPS_;                   // k-blocks per stage
    static constexpr int LAYOUT = LAYOUT_;
    static constexpr int BM = 64, BN = 64, BK = 64;   // bf16: BK is one 128-byte row
    static constexpr int A_KB_BYTES = BM * 128;        // one k-block of A: 8 KB, K-major, 128-byte swizzle
    static constexpr int B_KB_BYTES = BK * 128;        // one k-block of B: 64 columns × 64 K-rows, N-major
    static constexpr int A_BYTES = KPS * A_KB_BYTES;
    static constexpr int B_BYTES = KPS * B_KB_BYTES;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int TMEM_COLS = 64;
    static constexpr int NBARS = 2 * STAGES + 2;       // full[S], empty[S], acc_full, drain
    static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + 256;
    static constexpr int THREADS = 192;
    static constexpr uint32_t IDESC = ptx::make_idesc(InTraits<InKind::BF16>::FMT, InTraits<InKind::BF16>::FMT,
                                                      /*A K-major*/ 0, /*B N-major*/ 1, BM, BN);
    static_assert(OK == OutKind::F32 || OK == OutKind::BF16, "fp32 or bf16 C");
    static_assert(KPS == 1 || KPS == 2, "one or two k-blocks per stage");
    static_assert(NBARS * 8 + 8 <= 256, "barrier area");
    static_assert(SMEM_BYTES <= 232448, "exceeds the 227 KB per-block shared memory limit");
};

template <OutKind OK, int STAGES, int KPS, int LAYOUT>
__global__ void __launch_bounds__(M64Cfg<OK, STAGES, KPS, LAYOUT>::THREADS, 1)
    gemm_m64_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const GemmParams p) {
    using C = M64Cfg<OK, STAGES, KPS, LAYOUT>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = ptx::smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
    uint8_t* stage_base = smem;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * C::STAGE_BYTES);
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + C::NBARS);
    volatile uint32_t* abort_flag = tmem_holder + 1;

    const uint32_t full0 = ptx::smem_u32(bars);
    const uint32_t empty0 = ptx::smem_u32(bars + STAGES);
    const uint32_t accf = ptx::smem_u32(bars + 2 * STAGES);
    const uint32_t drain_bar = ptx::smem_u32(bars + 2 * STAGES + 1);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(full0 + 8 * s, 1);
            ptx::mbar_init(empty0 + 8 * s, 1);
        }
        ptx::mbar_init(accf, 1);
        ptx::mbar_init(drain_bar, 1);
        *abort_flag = 0u;
        ptx::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tensormap(&tmA);
        ptx::prefetch_tensormap(&tmB);
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_u32(tmem_holder), C::TMEM_COLS);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    ptx::griddep_wait();   // global memory only after the previous kernel in the stream
    ptx::griddep_launch_dependents();

    int mb, nb;
    tile_coords(static_cast<int>(blockIdx.x), p, mb, nb);
    const int nkb = p.num_kb;
    const int nst = (nkb + KPS - 1) / KPS;   // stage loads (a last odd k-block's partner is read as zeros)
    const bool tracing = (p.trace != nullptr) && (blockIdx.x == 0);
    if (tracing && threadIdx.x == 0) {
        p.trace[4 * p.trace_cap + 1] = ptx::globaltimer_ns();
        p.trace[4 * p.trace_cap + 0] = ptx::clock64();
    }

    if (warp == 0) {
        // ------------------------------------------------ producer (TMA)
        uint32_t it = 0;
        bool ok = true;
        for (int st = 0; st < nst; ++st, ++it) {
            const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
            if (!wait_warp(empty0 + 8 * s, ph ^ 1u, abort_flag, p.timeout_ns, p.status, DEV_TIMEOUT_PRODUCER)) {
                ok = false;
                break;
            }
            if (tracing && lane == 0) {
                const uint64_t now = ptx::clock64();
                if (it >= STAGES && it - STAGES < (uint32_t)p.trace_cap) p.trace[4 * (it - STAGES) + 3] = now;
                if (it < (uint32_t)p.trace_cap) p.trace[4 * it + 0] = now;
            }
            const uint32_t full = full0 + 8 * s;
            const uint32_t sa = ptx::smem_u32(stage_base + s * C::STAGE_BYTES);
            if (blockIdx.x == 0 && static_cast<int>(it) == p.debug_skip_kb) continue;
            ptx::mbar_arrive_expect_tx_elected(full, C::STAGE_BYTES);
            if constexpr (KPS == 2)   // A: 64 K × 64 rows × 2 k-blocks through the 3-D map
                ptx::tma_load_3d_elected(sa, &tmA, full, 0, mb * C::BM, st * KPS);
            else
                ptx::tma_load_2d_elected(sa, &tmA, full, st * C::BK, mb * C::BM);
            ptx::tma_load_2d_elected(sa + C::A_BYTES, &tmB, full, nb * C::BN, st * KPS * C::BK);
        }
        if (!ok && lane == 0) {   // let the loads in flight land before the CTA can exit
            const uint32_t first = it > (uint32_t)STAGES ? it - STAGES : 0u;
            for (uint32_t j = first; j < it; ++j) wait_drain(full0 + 8 * (j % STAGES), (j / STAGES) & 1u, p.timeout_ns);
        }
        if (ok && tracing && lane == 0) {   // "MMAs done" of the k-blocks whose stages were not reused
            const uint32_t first = it > (uint32_t)STAGES ? it - STAGES : 0u;
            for (uint32_t j = first; j < it && j < (uint32_t)p.trace_cap && !*abort_flag; ++j) {
                wait_drain(empty0 + 8 * (j % STAGES), (j / STAGES) & 1u, p.timeout_ns);
                p.trace[4 * j + 3] = ptx::clock64();
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        const uint32_t stage0 = ptx::smem_u32(stage_base);
        const uint64_t adesc0 = ptx::sdesc_sw128(stage0, 16, 1024);
        const uint64_t bdesc0 = ptx::sdesc(stage0 + C::A_BYTES, C::B_KB_BYTES, InTraits<InKind::BF16>::B_SBO,
                                           InTraits<InKind::BF16>::B_LAYOUT);
        constexpr uint64_t A_STEP = 16 * 2 / 16;     // a k-slice: 16 bf16 along the row
        constexpr uint64_t B_STEP = 16 * 128 / 16;   // a k-slice: 16 K-rows of 128 B
        constexpr uint64_t S_STEP = C::STAGE_BYTES / 16;
        constexpr uint64_t KB_STEP = C::A_KB_BYTES / 16;   // next k-block of the stage (A and B alike)
        static_assert(C::A_KB_BYTES == C::B_KB_BYTES, "k-blocks of A and B step alike");
        uint32_t it = 0;
        bool ok = true;
        for (int st = 0; st < nst; ++st, ++it) {
            const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
            if (!wait_warp(full0 + 8 * s, ph, abort_flag, p.timeout_ns, p.status, DEV_TIMEOUT_MMA_FULL)) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            if (tracing && lane == 0 && it < (uint32_t)p.trace_cap) p.trace[4 * it + 1] = ptx::clock64();
#pragma unroll
            for (int j = 0; j < KPS; ++j) {
                if (st * KPS + j >= nkb) break;
                const uint64_t ad = adesc0 + s * S_STEP + j * KB_STEP;
                const uint64_t bd = bdesc0 + s * S_STEP + j * KB_STEP;
                ptx::mma_f16_x4_elected(tmem_base, ad, bd, ad + A_STEP, bd + B_STEP, ad + 2 * A_STEP,
                                        bd + 2 * B_STEP, ad + 3 * A_STEP, bd + 3 * B_STEP, C::IDESC,
                                        st * KPS + j > 0 ? 1u : 0u);
            }
            ptx::mma_commit_elected(empty0 + 8 * s);
            if (tracing && lane == 0 && it < (uint32_t)p.trace_cap) p.trace[4 * it + 2] = ptx::clock64();
        }
        if (ok) {
            ptx::mma_commit_elected(accf);
        } else {
            ptx::mma_commit_elected(drain_bar);   // no MMA in flight when TMEM is freed
            if (lane == 0) wait_drain(drain_bar, 0, p.timeout_ns);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ epilogue: TMEM -> registers -> C
        const int q = warp & 3;   // TMEM lane quarter this warp may read
        int got = 1;
        if (lane == 0) got = wait_bounded(accf, 0, abort_flag, p.timeout_ns, p.status, DEV_TIMEOUT_EPILOGUE) ? 1 : 0;
        if (__shfl_sync(0xffffffffu, got, 0)) {
            ptx::tc_fence_after();
            const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
            uint32_t v[64];
            __syncwarp();   // tcgen05.ld is warp-collective
            ptx::tmem_ld_32x32b_x32(tb, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
            ptx::tmem_ld_32x32b_x32(tb + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
            ptx::tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(&v[0]));
            ptx::tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(&v[32]));
            // this lane's row of the tile, if it holds one
            const int r = LAYOUT == 0 ? (lane < 16 ? q * 16 + lane : -1) : (q < 2 ? q * 32 + lane : -1);
            const int row = mb * C::BM + r;
            const int col0 = nb * C::BN;
            if (r >= 0 && row < p.M) {
                const int n = min(C::BN, p.N - col0);   // columns of this row inside C
                if constexpr (OK == OutKind::F32) {
                    float* dst = static_cast<float*>(p.C) + static_cast<long long>(row) * p.ldc + col0;
                    if (n == C::BN && (reinterpret_cast<uintptr_t>(dst) & 15u) == 0) {
#pragma unroll
                        for (int c = 0; c < 16; ++c)
                            *reinterpret_cast<uint4*>(dst + 4 * c) =
                                make_uint4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
                    } else {
#pragma unroll
                        for (int i = 0; i < C::BN; ++i)
                            if (i < n) dst[i] = __uint_as_float(v[i]);
                    }
                } else {
                    uint32_t w[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        __nv_bfloat162 t = __floats2bfloat162_rn(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
                        w[i] = *reinterpret_cast<uint32_t*>(&t);
                    }
                    uint16_t* dst = static_cast<uint16_t*>(p.C) + static_cast<long long>(row) * p.ldc + col0;
                    if (n == C::BN && (reinterpret_cast<uintptr_t>(dst) & 15u) == 0) {
#pragma unroll
                        for (int c = 0; c < 8; ++c)
                            *reinterpret_cast<uint4*>(dst + 8 * c) = make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
                    } else {
#pragma unroll
                        for (int i = 0; i < C::BN; ++i)
                            if (i < n) dst[i] = static_cast<uint16_t>((i & 1) ? (w[i >> 1] >> 16) : (w[i >> 1] & 0xFFFFu));
                    }
                }
            }
        }
    }

    // ------------------------------------------------ teardown
    ptx::tc_fence_before();
    __syncthreads();
    if (tracing && threadIdx.x == 0) {
        p.trace[4 * p.trace_cap + 2] = ptx::clock64();
        p.trace[4 * p.trace_cap + 3] = ptx::globaltimer_ns();
    }
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

}  // namespace tcl
