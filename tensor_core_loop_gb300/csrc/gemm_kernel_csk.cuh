// K ranges of one output tile summed inside a thread-block cluster.
//
// For grids that a tile per SM would leave mostly idle (a few dozen 128×64
// tiles, e.g. 512² outputs), the CL CTAs of a cluster compute one tile
// together ("4.1 CUDA GEMM 算子性能优化" §2.3: too few blocks for the SMs is the
// tail effect at its worst; split-K in the K-sweep of "cp.async / ldmatrix
// 消融实验"). CTA r of the cluster runs the k-blocks [r·nkb/CL, (r+1)·nkb/CL)
// through the pipeline of the one-SM kernel: TMA loads into a ring of STAGES
// stages, tcgen05.mma issued by one thread into a TMEM accumulator. Then the
// CTAs r > 0 move their fp32 partial tile from TMEM into their own shared
// memory (over the ring, which the MMAs have finished reading) and push it with
// one bulk copy into receive slot r-1 of the first CTA's shared memory, the
// copy completing on the first CTA's receive barrier; the first CTA adds the
// slots to its own partial in the fixed order r = 1, 2, ..., CL-1 and stores C
// with tensor stores. One launch, no workspace in global memory, and the same
// bits on every run.
//
// Measured on GB300 (512², CUDA graphs of back-to-back calls) it is slower than
// one CTA per 64-wide tile below K = 2048 and than split-K with a reduction
// launch above, so the planner uses it on request only. %globaltimer stamps at
// 512²×256 with four CTAs per tile: the peers' bulk copies of 3 × 32 KB took
// ~2.1 µs to land in the first CTA, its sum and stores ~2.5 µs, the closing
// cluster barrier ~0.5 µs, against ~0.7 µs from the last MMA to the end for one
// CTA per tile. (Reading the partials with 16-byte loads over distributed
// shared memory after a cluster barrier instead was no faster.)
//
// Partial tile layout: chunk c (columns 4c..4c+3) of row R at (c·128 + R)·16
// bytes, so that a warp's access to one chunk of its 32 rows is 512 contiguous
// bytes (no bank conflict).
//
// Roles: warp 0 loads, warp 1 allocates TMEM and issues the MMAs, warps 2-5
// drain TMEM lane quarters (warp w reads lanes 32·(w mod 4)..+31). Waits on
// mbarriers are bounded as in the other kernels. A cluster barrier after the
// barrier set-up (before the previous kernel's end, under a programmatic
// launch) lets the peers signal the first CTA's barrier; one at the end keeps
// every CTA, and the first CTA's receive slots, alive until all copies have
// landed. Every CTA reaches both whatever happened in between.
#pragma once

#include "gemm_kernel.cuh"

namespace tcl {

template <OutKind OK, int CL_, int STAGES_>
struct CskCfg {
    static constexpr int CL = CL_;
    static constexpr int STAGES = STAGES_;
    static constexpr int BM = 128, BN = 64, BK = 64;   // bf16 operands: BK is one 128-byte row
    static constexpr int A_BYTES = BM * 128;            // 16 KB, K-major, 128-byte swizzle
    static constexpr int B_BYTES = BK * 128;            // one N-major box: 64 columns × 64 K-rows
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int PART_BYTES = BM * BN * 4;      // the fp32 partial tile
    static constexpr int OUT_ES = OK == OutKind::BF16 ? 2 : 4;
    static constexpr int SLAB_BYTES = 32 * 128;
    static constexpr int EPI_SLOTS = 2;
    static constexpr int STAGING_BYTES = 4 * EPI_SLOTS * SLAB_BYTES;
    static constexpr int RECV_BYTES = (CL - 1) * PART_BYTES;   // the first CTA's receive slots
    static constexpr int TMEM_COLS = 64;
    static constexpr int NBARS = 2 * STAGES + 3;        // full[S], empty[S], acc_full, drain, receive
    static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + RECV_BYTES + STAGING_BYTES + 256;
    static constexpr int THREADS = 192;
    static constexpr int EPI_WARP0 = 2;
    static constexpr uint32_t IDESC = ptx::make_idesc(InTraits<InKind::BF16>::FMT, InTraits<InKind::BF16>::FMT,
                                                      /*A K-major*/ 0, /*B N-major*/ 1, BM, BN);
    static_assert(OK == OutKind::F32 || OK == OutKind::BF16, "fp32 or bf16 C");
    static_assert(CL >= 2 && CL <= 8, "portable cluster size");
    static_assert(STAGES * STAGE_BYTES >= PART_BYTES, "the partial tile reuses the ring");
    static_assert(NBARS * 8 + 8 <= 256, "barrier area");
    static_assert(SMEM_BYTES <= 232448, "exceeds the 227 KB per-block shared memory limit");
};

template <OutKind OK, int CL, int STAGES>
__global__ void __launch_bounds__(CskCfg<OK, CL, STAGES>::THREADS, 1)
    gemm_csk_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmC, const GemmParams p) {
    using C = CskCfg<OK, CL, STAGES>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = ptx::smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
    uint8_t* stage_base = smem;
    uint8_t* recv_base = smem + STAGES * C::STAGE_BYTES;
    uint8_t* staging = recv_base + C::RECV_BYTES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(staging + C::STAGING_BYTES);
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + C::NBARS);
    volatile uint32_t* abort_flag = tmem_holder + 1;

    const uint32_t full0 = ptx::smem_u32(bars);
    const uint32_t empty0 = ptx::smem_u32(bars + STAGES);
    const uint32_t accf = ptx::smem_u32(bars + 2 * STAGES);
    const uint32_t drain_bar = ptx::smem_u32(bars + 2 * STAGES + 1);
    const uint32_t recv_bar = ptx::smem_u32(bars + 2 * STAGES + 2);   // the first CTA's: partials landed

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t r = ptx::cluster_ctarank();   // this CTA's K range of the tile

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(full0 + 8 * s, 1);
            ptx::mbar_init(empty0 + 8 * s, 1);
        }
        ptx::mbar_init(accf, 1);
        ptx::mbar_init(drain_bar, 1);
        ptx::mbar_init(recv_bar, 1);   // the first CTA's expect_tx; the peers' copies bring the bytes
        *abort_flag = 0u;
        ptx::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tensormap(&tmA);
        ptx::prefetch_tensormap(&tmB);
        ptx::prefetch_tensormap(&tmC);
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_u32(tmem_holder), C::TMEM_COLS);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    ptx::cluster_sync();   // every CTA's barriers initialised before any peer signals one
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    if (r == 0 && threadIdx.x == 0) ptx::mbar_arrive_expect_tx(recv_bar, C::RECV_BYTES);
    ptx::griddep_wait();   // global memory only after the previous kernel in the stream
    ptx::griddep_launch_dependents();

    const int kb_lo = static_cast<int>(r) * p.num_kb / CL;
    const int kb_hi = (static_cast<int>(r) + 1) * p.num_kb / CL;
    int mb, nb;
    tile_coords(static_cast<int>(blockIdx.x) / CL, p, mb, nb);
    const bool tracing = (p.trace != nullptr) && (blockIdx.x == 0);
    if (tracing && threadIdx.x == 0) {
        p.trace[4 * p.trace_cap + 1] = ptx::globaltimer_ns();
        p.trace[4 * p.trace_cap + 0] = ptx::clock64();
    }
    bool epi_ok = false;   // epilogue warps: this CTA's accumulator is complete

    if (warp == 0) {
        // ------------------------------------------------ producer (TMA)
        uint32_t it = 0;
        bool ok = true;
        for (int kb = kb_lo; kb < kb_hi; ++kb, ++it) {
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
            ptx::tma_load_2d_elected(sa, &tmA, full, kb * C::BK, mb * C::BM);
            ptx::tma_load_2d_elected(sa + C::A_BYTES, &tmB, full, nb * C::BN, kb * C::BK);
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
        const uint64_t bdesc0 = ptx::sdesc(stage0 + C::A_BYTES, C::B_BYTES, InTraits<InKind::BF16>::B_SBO,
                                           InTraits<InKind::BF16>::B_LAYOUT);
        constexpr uint64_t A_STEP = 16 * 2 / 16;     // a k-slice: 16 bf16 along the row
        constexpr uint64_t B_STEP = 16 * 128 / 16;   // a k-slice: 16 K-rows of 128 B
        constexpr uint64_t S_STEP = C::STAGE_BYTES / 16;
        uint32_t it = 0;
        bool ok = true;
        for (int kb = kb_lo; kb < kb_hi; ++kb, ++it) {
            const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
            if (!wait_warp(full0 + 8 * s, ph, abort_flag, p.timeout_ns, p.status, DEV_TIMEOUT_MMA_FULL)) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            if (tracing && lane == 0 && it < (uint32_t)p.trace_cap) p.trace[4 * it + 1] = ptx::clock64();
            const uint64_t ad = adesc0 + s * S_STEP;
            const uint64_t bd = bdesc0 + s * S_STEP;
            ptx::mma_f16_x4_elected(tmem_base, ad, bd, ad + A_STEP, bd + B_STEP, ad + 2 * A_STEP, bd + 2 * B_STEP,
                                    ad + 3 * A_STEP, bd + 3 * B_STEP, C::IDESC, kb > kb_lo ? 1u : 0u);
            ptx::mma_commit_elected(empty0 + 8 * s);
            if (tracing && lane == 0 && it < (uint32_t)p.trace_cap) p.trace[4 * it + 2] = ptx::clock64();
        }
        if (ok) {
            ptx::mma_commit_elected(accf);   // the partial tile is complete
        } else {
            ptx::mma_commit_elected(drain_bar);   // no MMA in flight when TMEM is freed
            if (lane == 0) wait_drain(drain_bar, 0, p.timeout_ns);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ epilogue: CTAs r > 0 publish their partial tile
        const int q = warp & 3;
        const int row = q * 32 + lane;   // row of the tile this thread drains
        int got = 1;
        if (lane == 0) got = wait_bounded(accf, 0, abort_flag, p.timeout_ns, p.status, DEV_TIMEOUT_EPILOGUE) ? 1 : 0;
        epi_ok = __shfl_sync(0xffffffffu, got, 0) != 0;
        if (epi_ok && r > 0) {
            ptx::tc_fence_after();
            const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
            uint32_t v[64];
            if (kb_hi > kb_lo) {
                __syncwarp();   // tcgen05.ld is warp-collective
                ptx::tmem_ld_32x32b_x32(tb, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
                ptx::tmem_ld_32x32b_x32(tb + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
                ptx::tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(&v[0]));
                ptx::tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(&v[32]));
            } else {   // an empty K range (fewer k-blocks than CTAs) adds nothing
#pragma unroll
                for (int i = 0; i < 64; ++i) v[i] = 0u;
            }
            const uint32_t base = ptx::smem_u32(stage_base) + row * 16;
#pragma unroll
            for (int c = 0; c < 16; ++c)
                st_shared_v4(base + c * (C::BM * 16), v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
            ptx::fence_proxy_async_smem();   // these stores, then the bulk copy's reads
        }
        if (r > 0) {
            // once the four epilogue warps have stored their rows (and none gave up: a wait
            // that runs out raises the abort flag), one thread pushes the partial tile into
            // the first CTA's receive slot r-1
            ptx::named_bar_sync(1, 4 * 32);
            if (warp == C::EPI_WARP0 && lane == 0 && !*abort_flag) {
                const uint32_t dst = ptx::mapa_shared(ptx::smem_u32(recv_base) + (r - 1) * C::PART_BYTES, 0u);
                ptx::bulk_copy_to_cluster(dst, ptx::smem_u32(stage_base), C::PART_BYTES,
                                          ptx::mapa_shared(recv_bar, 0u));
            }
        }
    }

    if (r == 0 && warp >= C::EPI_WARP0) {
        // ------------------------------------------------ first CTA: sum in range order, store C
        const int q = warp & 3;
        const int row = q * 32 + lane;
        const bool have = epi_ok && !*abort_flag;
        uint32_t v[64];
        if (have && kb_hi > kb_lo) {   // its own partial first, while the peers' copies land
            ptx::tc_fence_after();
            const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
            __syncwarp();
            ptx::tmem_ld_32x32b_x32(tb, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
            ptx::tmem_ld_32x32b_x32(tb + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
            ptx::tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(&v[0]));
            ptx::tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(&v[32]));
        } else {
#pragma unroll
            for (int i = 0; i < 64; ++i) v[i] = 0u;
        }
        // The receive slots are waited for after a failure too (bounded): no copy may
        // still be writing this CTA's shared memory when it exits.
        int got = 0;
        if (lane == 0) {
            got = (have && wait_bounded(recv_bar, 0, abort_flag, p.timeout_ns, p.status, DEV_TIMEOUT_EPILOGUE)) ? 1 : 0;
            if (!got) wait_drain(recv_bar, 0, p.timeout_ns);
        }
        if (__shfl_sync(0xffffffffu, got, 0)) {
            const uint32_t slots = ptx::smem_u32(recv_base) + row * 16;
#pragma unroll 1
            for (int rr = 1; rr < CL; ++rr) {
                const uint32_t slot = slots + (rr - 1) * C::PART_BYTES;
                uint4 x[16];
#pragma unroll
                for (int c = 0; c < 16; ++c) x[c] = ld_shared_v4(slot + c * (C::BM * 16));
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    v[4 * c + 0] = __float_as_uint(__uint_as_float(v[4 * c + 0]) + __uint_as_float(x[c].x));
                    v[4 * c + 1] = __float_as_uint(__uint_as_float(v[4 * c + 1]) + __uint_as_float(x[c].y));
                    v[4 * c + 2] = __float_as_uint(__uint_as_float(v[4 * c + 2]) + __uint_as_float(x[c].z));
                    v[4 * c + 3] = __float_as_uint(__uint_as_float(v[4 * c + 3]) + __uint_as_float(x[c].w));
                }
            }
            uint8_t* slab_pair = staging + (warp - C::EPI_WARP0) * C::EPI_SLOTS * C::SLAB_BYTES;
            int store_count = 0;
            const int row0 = mb * C::BM + q * 32;
            if constexpr (OK == OutKind::BF16) {
                uint32_t w[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    __nv_bfloat162 t =
                        __floats2bfloat162_rn(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
                    w[i] = *reinterpret_cast<uint32_t*>(&t);
                }
                store_slab<C::SLAB_BYTES, 2, C::EPI_SLOTS>(&tmC, slab_pair, store_count, w, lane, nb * C::BN, row0, p);
            } else {
#pragma unroll
                for (int c = 0; c < 2; ++c)
                    store_slab<C::SLAB_BYTES, 4, C::EPI_SLOTS>(&tmC, slab_pair, store_count,
                                                               *reinterpret_cast<const uint32_t(*)[32]>(&v[32 * c]),
                                                               lane, nb * C::BN + 32 * c, row0, p);
            }
            if (lane == 0) ptx::bulk_wait<0>();
            __syncwarp();
        }
    }
    // the peers keep their shared memory until their copies have landed in the first CTA
    ptx::tc_fence_before();
    ptx::cluster_sync();
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
