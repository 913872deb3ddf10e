// Exact int8 GEMM on two SMs per 256×256 tile, with the int8 operands widened
// inside the kernel instead of by a separate pass over HBM.
//
// The arithmetic is that of the exact-integer mode of the other kernels: int8
// values are exact in fp16 (|x| <= 128 < 2^11), every product is an exact
// integer of magnitude at most 2^14, and fp32 holds every integer up to 2^24,
// so a TMEM accumulation unit of at most 1024 K values is exact; each unit is
// converted and added into int32 registers.
//
// What differs is how the operands reach shared memory. A producer warp
// copies this CTA's share of the raw int8 operands for each k-block (its 128
// rows of A × 64 K and 64 K-rows × its 128 columns of B, 16 KB) with TMA into
// a ring of RAW slots (no swizzle; out-of-range rows and columns read as
// zeros). Four converter warps per CTA then read a slot with 16-byte shared
// loads, widen each byte to fp16 with byte permutes and one packed subtraction,
// and store the fp16 values into a stage of the MMA ring in the
// 128-byte-swizzled layout the tensor core reads (A K-major, B N-major in boxes
// of 64 columns). After a proxy fence, one lane per converter warp frees the
// raw slot and arrives on the leader CTA's full barrier, which completes once
// the eight converter warps of the pair have filled the stage. (The converters
// load nothing from global memory themselves: an arrive with release
// semantics would wait for such loads, which put a full memory latency into
// every k-block of a first version.) The leader's MMA warp, the stage ring,
// the two accumulators, the stream-K tail and the eight int32 epilogue warps
// are those of the two-SM kernel.
//
// Warp roles by warpgroup, with the registers split between them at the start
// (setmaxnreg; launch: 512 threads × 128 registers = 65,536):
//   warps 0-3   converters                       REGS_CONV
//   warps 4-7   MMA issuer, raw producer, idle   REGS_MMA
//   warps 8-15  epilogue (128 int32 sums/thread) REGS_EPI
//   128·REGS_CONV + 128·REGS_MMA + 256·REGS_EPI = 65,536.
//
// This trades a widening pass over HBM at 4096³ (read 32 MB, write 64 MB, then
// read the 64 MB of fp16 copies) for 48 KB of shared-memory traffic per k-block
// (16 KB read, 32 KB written) and about 200 integer/fp16 instructions per
// converter thread per k-block.
#pragma once

#include "gemm_kernel_pair.cuh"

namespace tcl {

template <int STAGES_, int RAW_>
struct S8PairCfg {
    static constexpr int STAGES = STAGES_;           // fp16 stages the MMA reads
    static constexpr int RAW = RAW_;                 // raw int8 slots the TMA fills
    static constexpr int BM = 256;                   // rows per pair tile (128 per SM)
    static constexpr int BN = 256;                   // columns per pair tile
    static constexpr int ROWS = 128;                 // rows of A and C per CTA
    static constexpr int COLS = BN / 2;              // columns of B this CTA supplies
    static constexpr int BK = 64;                    // K per k-block: one 128-byte row of fp16
    static constexpr int A_BYTES = ROWS * 128;       // 16 KB, K-major, 128-byte swizzle
    static constexpr int B_BOX_N = 64;               // N-major B in boxes of 64 columns × BK rows
    static constexpr int B_BOXES = COLS / B_BOX_N;
    static constexpr int B_BOX_BYTES = BK * 128;
    static constexpr int STAGE_BYTES = A_BYTES + B_BOXES * B_BOX_BYTES;   // 32 KB
    static constexpr int RAW_A_BYTES = ROWS * BK;    // 128 rows × 64 int8
    static constexpr int RAW_BYTES = RAW_A_BYTES + BK * COLS;            // 16 KB
    static constexpr int CONV_WARPS = 4;             // warpgroup 0
    static constexpr int MMA_WARP = 4;               // warpgroup 1
    static constexpr int RAW_WARP = 5;               //   (warps 6, 7 idle)
    static constexpr int EPI_WARP0 = 8;              // warpgroups 2-3
    static constexpr int EPI_WARPS = 8;
    static constexpr int THREADS = 512;
    static constexpr int REGS_CONV = 88, REGS_MMA = 72, REGS_EPI = 176;
    static constexpr int CW = BN / 2;                // int32 columns per epilogue warp (two warps per lane quarter)
    static constexpr int SLAB_BYTES = 32 * 128;
    static constexpr int EPI_SLOTS = 1;
    static constexpr int STAGING_BYTES = EPI_WARPS * EPI_SLOTS * SLAB_BYTES;
    static constexpr int ACC_STRIDE = 256;
    static constexpr int TMEM_COLS = 512;
    static constexpr int NBARS = 3 * STAGES + 5 + 2 * RAW;
    static constexpr int TOKEN_BYTES = 16;           // per stage: what the peer's forwarder copies
    static constexpr int SMEM_BYTES =
        1024 + STAGES * STAGE_BYTES + RAW * RAW_BYTES + STAGING_BYTES + STAGES * TOKEN_BYTES + 256;
    static constexpr int FORWARD_WARP = 6;           // the peer's: hands its converted stages to the leader
    static constexpr int CONV_THREADS = 32 * CONV_WARPS;
    static constexpr int A_PER = ROWS * BK / 16 / CONV_THREADS;   // 16-byte int8 chunks per thread: 4
    static constexpr int B_PER = BK * COLS / 16 / CONV_THREADS;   // 4
    // f16 × f16 -> f32, A K-major, B N-major, M = 256 (pair), N = 256
    static constexpr uint32_t IDESC = ptx::make_idesc(0, 0, 0, 1, BM, BN);

    static_assert(A_PER * CONV_THREADS * 16 == ROWS * BK && B_PER * CONV_THREADS * 16 == BK * COLS, "chunks");
    static_assert(SMEM_BYTES <= 232448, "exceeds the 227 KB per-block shared memory limit");
    static_assert(NBARS * 8 + 12 <= 256, "barrier area");
    static_assert(128 * REGS_CONV + 128 * REGS_MMA + 256 * REGS_EPI <= THREADS * 128, "register split");
};

// Warp-uniform bounded wait, as wait_warp_pair, on a barrier whose arrivals
// come from threads of both CTAs (acquire at cluster scope).
__device__ __forceinline__ bool wait_warp_pair_cluster(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag,
                                                       AbortNet peer_abort, unsigned long long timeout_ns,
                                                       unsigned int* status, unsigned int code) {
    if (__all_sync(0xffffffffu, ptx::mbar_try_wait_cluster(bar, parity))) return true;
    int ok = 1;
    if ((threadIdx.x & 31) == 0) {
        const uint64_t t0 = ptx::globaltimer_ns();
        while (!ptx::mbar_try_wait_cluster(bar, parity)) {
            if (*abort_flag) {
                ok = 0;
                break;
            }
            if (ptx::globaltimer_ns() - t0 > timeout_ns) {
                *abort_flag = 1u;
                peer_abort.raise();
                atomicCAS(status, 0u, code);
                ok = 0;
                break;
            }
        }
    }
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// Two of the four biased bytes of u (b + 128 each, chosen by the byte-permute
// selector) as two fp16 values b: 0x6400 | (b + 128) is the fp16 pattern of
// 1024 + b + 128, exactly, and subtracting 1152 in both halves is exact (every
// integer below 2048 is an fp16 value).
__device__ __forceinline__ uint32_t s8x2_to_f16x2(uint32_t u, uint32_t sel) {
    const uint32_t x = __byte_perm(u, 0x64u, sel);
    uint32_t r;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(x), "r"(0x64806480u));
    return r;
}

// 16 int8 values (in memory order) -> 16 fp16 values, h[0..3] the first 8, h[4..7] the last 8.
__device__ __forceinline__ void s8x16_to_f16(const uint4& v, uint32_t (&h)[8]) {
    const uint32_t w[4] = {v.x ^ 0x80808080u, v.y ^ 0x80808080u, v.z ^ 0x80808080u, v.w ^ 0x80808080u};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        h[2 * i] = s8x2_to_f16x2(w[i], 0x4140u);       // bytes 0, 1
        h[2 * i + 1] = s8x2_to_f16x2(w[i], 0x4342u);   // bytes 2, 3
    }
}

template <int STAGES, int RAW>
__global__ void __launch_bounds__(S8PairCfg<STAGES, RAW>::THREADS, 1)
    gemm_s8_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmC, const GemmParams p) {
    using C = S8PairCfg<STAGES, RAW>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = ptx::smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
    uint8_t* stage_base = smem;
    uint8_t* raw_base = smem + STAGES * C::STAGE_BYTES;
    uint8_t* staging = raw_base + RAW * C::RAW_BYTES;
    uint8_t* tokens = staging + C::STAGING_BYTES;   // STAGES × 16 B, 16-byte aligned
    uint64_t* bars = reinterpret_cast<uint64_t*>(tokens + STAGES * C::TOKEN_BYTES);
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + C::NBARS);
    volatile uint32_t* abort_flag = tmem_holder + 1;

    const uint32_t full0 = ptx::smem_u32(bars);
    const uint32_t empty0 = ptx::smem_u32(bars + STAGES);
    const uint32_t accf0 = ptx::smem_u32(bars + 2 * STAGES);
    const uint32_t acce0 = ptx::smem_u32(bars + 2 * STAGES + 2);
    const uint32_t drain_bar = ptx::smem_u32(bars + 2 * STAGES + 4);
    const uint32_t rfull0 = ptx::smem_u32(bars + 2 * STAGES + 5);
    const uint32_t rempty0 = ptx::smem_u32(bars + 2 * STAGES + 5 + RAW);
    const uint32_t cfull0 = ptx::smem_u32(bars + 2 * STAGES + 5 + 2 * RAW);   // this CTA's stage converted

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = ptx::cluster_ctarank() & 1u;   // 0: leader (issues the pair MMAs), 1: peer
    const bool leader = rank == 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(full0 + 8 * s, 1);                 // leader's: its MMA warp's expect_tx, completed
                                                              // by the bytes of the peer forwarder's token copy
            ptx::mbar_init(empty0 + 8 * s, 1);                // the leader's multicast commit
            ptx::mbar_init(cfull0 + 8 * s, C::CONV_WARPS);    // this CTA's converter warps
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(accf0 + 8 * b, 1);
            ptx::mbar_init(acce0 + 8 * b, 2 * C::EPI_WARPS);
        }
        ptx::mbar_init(drain_bar, 1);
        for (int r = 0; r < RAW; ++r) {
            ptx::mbar_init(rfull0 + 8 * r, 1);                 // the producer's arrival + the copy's bytes
            ptx::mbar_init(rempty0 + 8 * r, C::CONV_WARPS);    // this CTA's converter warps
        }
        *abort_flag = 0u;
        ptx::fence_mbar_init();
    }
    if (warp == C::MMA_WARP) {   // one warp in each CTA of the pair allocates, collectively
        ptx::tmem_alloc_pair(ptx::smem_u32(tmem_holder), C::TMEM_COLS);
        ptx::tmem_relinquish_pair();
    }
    if (warp == C::RAW_WARP && lane == 0) {
        ptx::prefetch_tensormap(&tmA);
        ptx::prefetch_tensormap(&tmB);
        ptx::prefetch_tensormap(&tmC);
    }
    __syncwarp();
    ptx::tc_fence_before();
    ptx::cluster_sync();
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    ptx::griddep_wait();   // global memory only after the previous kernel in the stream
    ptx::griddep_launch_dependents();

    const uint32_t full_leader0 = ptx::mapa_shared(full0, 0u);
    const uint32_t tokens0 = ptx::smem_u32(tokens);
    const uint32_t tokens_leader0 = ptx::mapa_shared(tokens0, 0u);
    const uint32_t acce_leader0 = ptx::mapa_shared(acce0, 0u);
    const AbortNet peer_abort{ptx::smem_u32(const_cast<uint32_t*>(abort_flag)), 2};
    const Sched S = make_sched(p, blockIdx.x / 2, gridDim.x / 2);   // the whole grid (no die split here)
    const int units = pair_units(p, S);
    // per-k-block %clock64 stamps of CTA 0 (raw copy issued by the producer; raw slot
    // landed, stage converted and fenced, stage handed over — seen by the first
    // converter thread)
    const bool tracing = (p.trace != nullptr) && (blockIdx.x == 0);

    if (warp < C::CONV_WARPS) {
        // ------------------------------------------------ converters (warpgroup 0, both CTAs)
        ptx::setmaxnreg_dec<C::REGS_CONV>();
        const int tid = threadIdx.x;   // 0..127: chunks tid + 128·i of a raw slot
        uint32_t it = 0;
        bool ok = true;
        for (int u = 0; ok && u < units; ++u) {
            const PairUnit U = pair_unit(p, S, u);
            for (int kb = U.kb_lo; kb < U.kb_hi; ++kb, ++it) {
                const uint32_t r = it % RAW, rph = (it / RAW) & 1u;
                const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
                // the raw slot has landed, and the stage is free
                if (!wait_warp_pair(rfull0 + 8 * r, rph, abort_flag, peer_abort, p.timeout_ns, p.status,
                                    DEV_TIMEOUT_PRODUCER)) {
                    ok = false;
                    break;
                }
                if (tracing && tid == 0 && it < (uint32_t)p.trace_cap) p.trace[4 * it + 1] = ptx::clock64();
                if (!wait_warp_pair(empty0 + 8 * s, ph ^ 1u, abort_flag, peer_abort, p.timeout_ns, p.status,
                                    DEV_TIMEOUT_PRODUCER)) {
                    ok = false;
                    break;
                }
                const uint32_t src = ptx::smem_u32(raw_base + r * C::RAW_BYTES) + tid * 16;
                const uint32_t sa = ptx::smem_u32(stage_base + s * C::STAGE_BYTES);
                const uint32_t sb = sa + C::A_BYTES;
                // all of this thread's raw chunks first (their latencies overlap), then widen and store
                uint4 raw[C::A_PER + C::B_PER];
#pragma unroll
                for (int i = 0; i < C::A_PER; ++i) raw[i] = ld_shared_v4(src + C::CONV_THREADS * 16 * i);
#pragma unroll
                for (int i = 0; i < C::B_PER; ++i)
                    raw[C::A_PER + i] = ld_shared_v4(src + C::RAW_A_BYTES + C::CONV_THREADS * 16 * i);
#pragma unroll
                for (int i = 0; i < C::A_PER; ++i) {   // A chunk ch: row ch / 4, K (ch % 4)·16
                    const int ch = tid + C::CONV_THREADS * i;
                    const int row = ch >> 2, j0 = 2 * (ch & 3), sw = row & 7;
                    uint32_t v[8];
                    s8x16_to_f16(raw[i], v);
                    const uint32_t base = sa + row * 128;
                    st_shared_v4(base + ((j0 ^ sw) << 4), v[0], v[1], v[2], v[3]);
                    st_shared_v4(base + (((j0 + 1) ^ sw) << 4), v[4], v[5], v[6], v[7]);
                }
#pragma unroll
                for (int i = 0; i < C::B_PER; ++i) {   // B chunk ch: K-row ch / 8, N (ch % 8)·16
                    const int ch = tid + C::CONV_THREADS * i;
                    const int k = ch >> 3, qq = ch & 7, j0 = 2 * (qq & 3), sw = k & 7;
                    uint32_t v[8];
                    s8x16_to_f16(raw[C::A_PER + i], v);
                    const uint32_t base = sb + (qq >> 2) * C::B_BOX_BYTES + k * 128;
                    st_shared_v4(base + ((j0 ^ sw) << 4), v[0], v[1], v[2], v[3]);
                    st_shared_v4(base + (((j0 + 1) ^ sw) << 4), v[4], v[5], v[6], v[7]);
                }
                ptx::fence_proxy_async_smem();   // generic-proxy stores -> visible to the tensor core
                __syncwarp();
                if (tracing && tid == 0 && it < (uint32_t)p.trace_cap) p.trace[4 * it + 2] = ptx::clock64();
                if (lane == 0) {
                    ptx::mbar_arrive(rempty0 + 8 * r);   // the raw slot may be refilled
                    // (test hook: CTA 0 never hands this k-block over, so the MMA warp's wait runs out)
                    if (!(blockIdx.x == 0 && static_cast<int>(it) == p.debug_skip_kb)) ptx::mbar_arrive(cfull0 + 8 * s);
                    if (tracing && tid == 0 && it < (uint32_t)p.trace_cap) p.trace[4 * it + 3] = ptx::clock64();
                }
            }
        }
        __syncwarp();
    } else if (warp < C::EPI_WARP0) {
        ptx::setmaxnreg_dec<C::REGS_MMA>();
        if (warp == C::RAW_WARP) {
            // -------------------------------------------- raw int8 producer (TMA), both CTAs
            uint32_t it = 0;
            bool ok = true;
            for (int u = 0; ok && u < units; ++u) {
                const PairUnit U = pair_unit(p, S, u);
                int mb, nb;
                sched_tile_coords(U.tile, p, S, mb, nb);
                const int row = mb * C::BM + static_cast<int>(rank) * C::ROWS;
                const int col = nb * C::BN + static_cast<int>(rank) * C::COLS;
                for (int kb = U.kb_lo; kb < U.kb_hi; ++kb, ++it) {
                    const uint32_t r = it % RAW, rph = (it / RAW) & 1u;
                    if (!wait_warp_pair(rempty0 + 8 * r, rph ^ 1u, abort_flag, peer_abort, p.timeout_ns, p.status,
                                        DEV_TIMEOUT_PRODUCER)) {
                        ok = false;
                        break;
                    }
                    const int kc = load_kblock(p, u, kb, U.kb_lo, U.kb_hi);
                    const uint32_t dst = ptx::smem_u32(raw_base + r * C::RAW_BYTES);
                    if (tracing && lane == 0 && it < (uint32_t)p.trace_cap) p.trace[4 * it + 0] = ptx::clock64();
                    ptx::mbar_arrive_expect_tx_elected(rfull0 + 8 * r, C::RAW_BYTES);
                    ptx::tma_load_2d_elected(dst, &tmA, rfull0 + 8 * r, kc * C::BK, row);
                    ptx::tma_load_2d_elected(dst + C::RAW_A_BYTES, &tmB, rfull0 + 8 * r, col, kc * C::BK);
                }
            }
            if (!ok && lane == 0) {   // let copies issued before the abort land before the CTA exits
                const uint32_t first = it > static_cast<uint32_t>(RAW) ? it - RAW : 0u;
                for (uint32_t j = first; j < it; ++j) wait_drain(rfull0 + 8 * (j % RAW), (j / RAW) & 1u, p.timeout_ns);
            }
        } else if (warp == C::FORWARD_WARP && !leader) {
            // -------------------------------------------- forwarder (peer CTA): each stage this CTA's
            // converters filled is announced to the leader's MMA warp, in ring order
            uint32_t it = 0;
            bool ok = true;
            for (int u = 0; ok && u < units; ++u) {
                const PairUnit U = pair_unit(p, S, u);
                for (int kb = U.kb_lo; kb < U.kb_hi; ++kb, ++it) {
                    const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
                    if (!wait_warp_pair(cfull0 + 8 * s, ph, abort_flag, peer_abort, p.timeout_ns, p.status,
                                        DEV_TIMEOUT_PRODUCER)) {
                        ok = false;
                        break;
                    }
                    // a 16-byte copy into the leader's shared memory, completed on its full[s]: an
                    // asynchronous signal (a release arrive at cluster scope would stall this warp
                    // for ~850 cycles per stage, measured on GB300)
                    if (lane == 0)
                        ptx::bulk_copy_to_cluster(tokens_leader0 + s * C::TOKEN_BYTES, tokens0 + s * C::TOKEN_BYTES,
                                                  C::TOKEN_BYTES, full_leader0 + 8 * s);
                    __syncwarp();
                }
            }
            // after an abort the leader stops waiting for tokens: let the copies issued so far
            // land (within microseconds) before the pair can exit
            if (!ok && lane == 0) spin_ns(200000);
        } else if (warp == C::MMA_WARP && leader) {
            // -------------------------------------------- MMA issuer (leader CTA only)
            const uint32_t stage0 = ptx::smem_u32(stage_base);
            const uint64_t adesc0 = ptx::sdesc_sw128(stage0, 16, 1024);
            const uint64_t bdesc0 = ptx::sdesc_sw128(stage0 + C::A_BYTES, C::B_BOX_BYTES, 1024);
            constexpr uint64_t A_STEP = 16 * 2 / 16;     // a k-slice: 16 fp16 along the row
            constexpr uint64_t B_STEP = 16 * 128 / 16;   // a k-slice: 16 rows of 128 B
            constexpr uint64_t S_STEP = C::STAGE_BYTES / 16;
            uint32_t unit = 0, s = 0, ph = 0, mit = 0;
            bool ok = true;
            for (int u = 0; ok && u < units; ++u) {
                const PairUnit U = pair_unit(p, S, u);
                for (int kb0 = U.kb_lo; ok && kb0 < U.kb_hi; kb0 += p.kb_per_unit, ++unit) {
                    const int kb1 = min(kb0 + p.kb_per_unit, U.kb_hi);
                    const uint32_t buf = unit & 1u;
                    const uint32_t uph = (unit >> 1) & 1u;
                    if (!wait_warp_pair(acce0 + 8 * buf, uph ^ 1u, abort_flag, peer_abort, p.timeout_ns, p.status,
                                        DEV_TIMEOUT_MMA_ACC)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t d_tmem = tmem_base + buf * C::ACC_STRIDE;
                    for (int kb = kb0; kb < kb1; ++kb, ++mit) {
                        // the stage was written by threads of both CTAs: this CTA's converters
                        // (cfull), and the peer's, whose forwarder's token copy completes full
                        ptx::mbar_arrive_expect_tx_elected(full0 + 8 * s, C::TOKEN_BYTES);
                        if (!wait_warp_pair(cfull0 + 8 * s, ph, abort_flag, peer_abort, p.timeout_ns, p.status,
                                            DEV_TIMEOUT_MMA_FULL) ||
                            !wait_warp_pair_cluster(full0 + 8 * s, ph, abort_flag, peer_abort, p.timeout_ns,
                                                    p.status, DEV_TIMEOUT_MMA_FULL)) {
                            ok = false;
                            break;
                        }
                        ptx::tc_fence_after();
                        const uint64_t ad = adesc0 + s * S_STEP;
                        const uint64_t bd = bdesc0 + s * S_STEP;
                        ptx::mma_f16_pair_x4_elected(d_tmem, ad, bd, ad + A_STEP, bd + B_STEP, ad + 2 * A_STEP,
                                                     bd + 2 * B_STEP, ad + 3 * A_STEP, bd + 3 * B_STEP, C::IDESC,
                                                     kb > kb0 ? 1u : 0u);
                        ptx::mma_commit_pair_multicast_elected(empty0 + 8 * s, 0x3);
                        const uint32_t wrap = (s + 1 == static_cast<uint32_t>(STAGES)) ? 1u : 0u;
                        s = wrap ? 0u : s + 1;
                        ph ^= wrap;
                    }
                    if (!ok) break;
                    ptx::mma_commit_pair_multicast_elected(accf0 + 8 * buf, 0x3);
                }
            }
            if (!ok) {
                ptx::mma_commit_pair_multicast_elected(drain_bar, 0x1);
                if (lane == 0) wait_drain(drain_bar, 0, p.timeout_ns);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ epilogue (warpgroups 2-3, both CTAs)
        ptx::setmaxnreg_inc<C::REGS_EPI>();
        const int ew = warp - C::EPI_WARP0;   // 0..7
        const int q = warp & 3;               // TMEM lane quarter this warp may read
        const int h = ew >> 2;                // which half of the tile's columns its int32 sums cover
        uint8_t* slab = staging + ew * C::SLAB_BYTES;
        int store_count = 0;
        uint32_t unit = 0;
        bool ok = true;
        for (int u = 0; ok && u < units; ++u) {
            const PairUnit U = pair_unit(p, S, u);
            int mb, nb;
            sched_tile_coords(U.tile, p, S, mb, nb);
            const int row0 = mb * C::BM + static_cast<int>(rank) * C::ROWS + q * 32;
            uint32_t* flag =
                U.sk_index >= 0 ? p.sk_flags + (U.sk_index * 2 + rank) * C::EPI_WARPS + ew : nullptr;
            int32_t iacc[C::CW];
#pragma unroll
            for (int i = 0; i < C::CW; ++i) iacc[i] = 0;
            for (int kb0 = U.kb_lo; kb0 < U.kb_hi; kb0 += p.kb_per_unit, ++unit) {
                const uint32_t buf = unit & 1u;
                const uint32_t uph = (unit >> 1) & 1u;
                int got = 1;
                if (lane == 0)
                    got = wait_bounded_pair(accf0 + 8 * buf, uph, abort_flag, peer_abort, p.timeout_ns, p.status,
                                            DEV_TIMEOUT_EPILOGUE)
                              ? 1
                              : 0;
                if (!__shfl_sync(0xffffffffu, got, 0)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t tb =
                    tmem_base + (static_cast<uint32_t>(q * 32) << 16) + buf * C::ACC_STRIDE + h * C::CW;
#pragma unroll
                for (int c = 0; c < C::CW / 16; ++c) {
                    __syncwarp();   // tcgen05.ld is warp-collective
                    uint32_t r[16];
                    ptx::tmem_ld_32x32b_x16(tb + c * 16, r);
                    ptx::tmem_ld_wait(r);
#pragma unroll
                    for (int i = 0; i < 16; ++i) iacc[c * 16 + i] += __float2int_rn(__uint_as_float(r[i]));
                }
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive_cluster_relaxed(acce_leader0 + 8 * buf);
            }
            if (!ok) break;
            // the tile's (or piece's) int32 sums; a stream-K piece after the first adds its
            // sums once the previous piece has handed the rows over
            if (flag && U.piece > 0) {
                if (!wait_sk_flag(flag, (p.sk_gen << 3) | static_cast<uint32_t>(U.piece), abort_flag, peer_abort,
                                  p.timeout_ns, p.status)) {
                    ok = false;
                    break;
                }
                if (U.piece + 1 == p.sk_pieces) {   // the flag's last reader leaves it at 0 (graph replays)
                    __syncwarp();
                    if (lane == 0) *reinterpret_cast<volatile uint32_t*>(flag) = 0u;
                }
            }
#pragma unroll
            for (int c = 0; c < C::CW / 32; ++c) {
                const uint32_t(&v)[32] = *reinterpret_cast<const uint32_t(*)[32]>(&iacc[c * 32]);
                store_slab<C::SLAB_BYTES, 4, C::EPI_SLOTS, true>(&tmC, slab, store_count, v, lane,
                                                                  nb * C::BN + h * C::CW + c * 32, row0, p,
                                                                  U.piece > 0);
            }
            if (flag && U.piece + 1 < p.sk_pieces) {
                __threadfence();   // the ragged-edge chunk's element writes, from every lane
                __syncwarp();
                const bool held = p.debug_sk_stall && U.sk_index == 0 && U.piece == 0;
                if (lane == 0) {
                    ptx::bulk_wait<0>();                // this warp's stores/reductions completed
                    ptx::fence_proxy_async_global();    // ... and ordered before the release
                    if (!held) ptx::st_release_gpu(flag, (p.sk_gen << 3) | static_cast<uint32_t>(U.piece + 1));
                }
                __syncwarp();
            }
        }
        if (lane == 0) ptx::bulk_wait<0>();
        __syncwarp();
    }

    // ------------------------------------------------ teardown
    ptx::tc_fence_before();
    __syncthreads();
    ptx::cluster_sync();   // no CTA frees TMEM or exits while its peer may still signal it
    if (warp == C::MMA_WARP) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
    }
}

}  // namespace tcl
