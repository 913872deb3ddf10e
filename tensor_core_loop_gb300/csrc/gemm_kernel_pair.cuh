// Two-SM variant of the pipelined GEMM: a cluster of two CTAs on two SMs
// computes one 256×256 output tile with tcgen05.mma.cta_group::2.
//
// Same pipeline as gemm_kernel.cuh (TMA producer → S-deep mbarrier ring →
// single-thread MMA issue → TMEM → TMA-store epilogue, persistent grouped
// raster), with the work of one tile split over the pair:
//   * each CTA loads only its own 128 rows of A and its own half (128
//     columns) of the B tile, so each SM moves 32 KB per 64-deep k-block
//     instead of 48 KB for the same 128×256 share of the MMA work;
//   * both CTAs' loads count their bytes on the even (leader) CTA's full[s]
//     barrier, whose producer announces the pair's total;
//   * the leader's MMA warp issues the pair MMA (M=256: each SM's tensor core
//     produces its own 128 rows into its own TMEM, reading B from both SMs)
//     and commits empty[s] and acc_full[b] to both CTAs at once (multicast);
//   * both CTAs' epilogues drain their own TMEM and release the accumulator
//     on the leader's acc_empty[b] (8 arrivals: 4 warps × 2 CTAs).
// Every TMA load brings a box into the issuing CTA's own shared memory; only
// the MMA completions (tcgen05.commit) are signalled to both CTAs at once.
// TF32 inputs (IK = TF32) take B N-major too, in boxes of 32 columns × 32 K
// rows swizzled in 32-byte units (the form the tensor core reads 4-byte
// N-major operands in).
// Exact integers (OK = S32, int8 widened to bf16) accumulate units of 1024 K
// values per TMEM buffer and add each unit, converted, into int32 registers:
// 128 columns per thread, so a 256-wide tile has eight epilogue warps.
// A stream-K tail cuts the last partial wave of tiles into K pieces run by the
// otherwise idle pairs; piece i > 0 adds its sums after piece i-1 (per-warp
// flags): into C for fp32 and int32, through an fp32 workspace for bf16, whose
// last piece rounds once.
// Waits are bounded as in the one-SM kernel; a role that gives up raises the
// abort flag of every CTA of the cluster.
#pragma once

#include "gemm_kernel.cuh"

namespace tcl {

template <OutKind OK, int BN_, int STAGES_, int SLOTS_, InKind IK = InKind::BF16>
struct PairCfg {
    static constexpr int CL = 2;                     // CTAs per cluster: one pair
    static constexpr uint16_t ALL = 0x3;             // commit mask: both CTAs of the pair
    static constexpr int STAGES = STAGES_;
    static constexpr int BM = 256;                   // rows per pair tile (128 per SM)
    static constexpr int BN = BN_;                   // columns per pair tile (each SM supplies BN/2 of B)
    static constexpr int ROWS = 128;                 // rows of A and C per CTA
    static constexpr int ES = InTraits<IK>::ES;
    static constexpr int BK = 128 / ES;              // one 128-byte swizzle row of K (64 bf16, 32 TF32)
    static constexpr int UMMA_K = InTraits<IK>::UMMA_K;
    static constexpr int KSUB = BK / UMMA_K;
    static constexpr int A_BYTES = ROWS * 128;       // 16 KB
    // this CTA's half of B, N-major: whole boxes of one 128-byte row of N (64
    // bf16 or 32 TF32 columns) × BK rows (at BN=224 the last box also brings 16
    // columns the MMA does not read)
    static constexpr int B_BOX_N = 128 / ES;
    static constexpr int B_BOXES = (BN / 2 + B_BOX_N - 1) / B_BOX_N;
    static constexpr int B_BOX_BYTES = BK * 128;
    static constexpr int B_BYTES = B_BOXES * B_BOX_BYTES;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;   // 32 KB per CTA
    // the ring holds the A slots of all stages first, then their B slots, so that
    // consecutive slots of each operand are contiguous (one copy may fill two). Measured on
    // GB300 (CUDA graphs, round robin in one process) this is also faster than keeping each
    // slot's A and B together, with one k-block per copy as with two: 4096³ 115 against 127
    // and 94 against 102 µs, 256×224 tiles at 4096²×1024 39.8 against 43.5 µs
    static constexpr int A_RING_BYTES = STAGES * A_BYTES;
    static constexpr int PAIR_TX = 2 * STAGE_BYTES;         // bytes the leader's full[s] expects
    static constexpr int OUT_ES = (OK == OutKind::BF16) ? 2 : 4;
    static constexpr int EPI_COLS = 128 / OUT_ES;
    static constexpr int EPI_CHUNKS = BN / EPI_COLS;
    static constexpr int SLAB_BYTES = 32 * 128;
    static constexpr int EPI_SLOTS = SLOTS_;          // staging slabs per epilogue warp (stores in flight)
    // Epilogue warps: four (one per TMEM lane quarter, each over all BN columns),
    // or, for exact integers wider than 128 columns, eight: two per lane quarter,
    // each keeping the int32 sums of its rows over half of the columns.
    static constexpr int EPI_WARPS = (OK == OutKind::S32 && BN > 128) ? 8 : 4;
    static constexpr int EPI_COLS_PER_WARP = BN / (EPI_WARPS / 4);
    static constexpr int STAGING_BYTES = EPI_WARPS * EPI_SLOTS * SLAB_BYTES;
    static constexpr int ACC_STRIDE = 256;           // accumulator b starts at TMEM column b·256
    static constexpr int TMEM_COLS = 512;
    static constexpr int BAR_BYTES = 256;
    static constexpr int SMEM_USED = 1024 + STAGES * STAGE_BYTES + STAGING_BYTES + BAR_BYTES;
    static constexpr int SMEM_BYTES = SMEM_USED > 122880 ? SMEM_USED : 122880;
    static constexpr uint32_t IDESC =
        ptx::make_idesc(InTraits<IK>::FMT, InTraits<IK>::FMT, /*A K-major*/ 0, /*B N-major*/ 1, BM, BN);
    static constexpr int THREADS = 64 + 32 * EPI_WARPS;   // producer, MMA issuer, epilogue warps
    // ring slots released per commit, as in the one-SM kernel: each SM's share of a
    // pair k-block (128 rows × BN columns) keeps its tensor pipe as long as a
    // one-SM k-block of width BN
    static constexpr int REL = (BN <= 128 && STAGES >= 4 && STAGES % 2 == 0) ? 2 : 1;

    static_assert(OK != OutKind::S32 || (EPI_COLS_PER_WARP <= 128 && IK == InKind::BF16),
                  "exact integer mode: int32 sums of at most 128 columns per thread in registers");
    static_assert(BN % 32 == 0 && BN <= 256 && BN % EPI_COLS == 0, "pair tile width");
    static_assert(SMEM_BYTES <= 232448, "exceeds the 227 KB per-block shared memory limit");
    static_assert(2 * STAGES + 5 <= 28, "barrier area");
    static_assert(KSUB == 4, "four MMAs per k-block");
};

// Raises the abort flag of both CTAs of the pair (addr: this CTA's flag).
struct AbortNet {
    uint32_t addr;
    int cl;
    __device__ __forceinline__ void raise() const {
        for (int r = 0; r < cl; ++r) ptx::st_cluster_u32(ptx::mapa_shared(addr, static_cast<uint32_t>(r)), 1u);
    }
};

// Bounded wait that, on giving up, raises the abort flag of this CTA and of its peer.
__device__ __forceinline__ bool wait_bounded_pair(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag,
                                                  AbortNet peer_abort, unsigned long long timeout_ns,
                                                  unsigned int* status, unsigned int code) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer_ns();
    while (true) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (ptx::globaltimer_ns() - t0 > timeout_ns) {
            *abort_flag = 1u;
            peer_abort.raise();
            atomicCAS(status, 0u, code);
            return false;
        }
    }
}

__device__ __forceinline__ bool wait_warp_pair(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag,
                                               AbortNet peer_abort, unsigned long long timeout_ns,
                                               unsigned int* status, unsigned int code) {
    if (__all_sync(0xffffffffu, ptx::mbar_try_wait(bar, parity))) return true;
    int ok = 1;
    if ((threadIdx.x & 31) == 0)
        ok = wait_bounded_pair(bar, parity, abort_flag, peer_abort, timeout_ns, status, code) ? 1 : 0;
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// The pair of SMs `cluster` (of `clusters`) walks its work units in this
// order. Split tiles are the last sk_tiles of the raster order; piece i of
// split tile d covers k-blocks [i·num_kb/sk_pieces, (i+1)·num_kb/sk_pieces)
// and belongs to pair d·sk_pieces + i. Whole tiles cluster, cluster +
// clusters, … (below the split ones) follow a pair's piece if that piece is
// not the last of its tile, and precede it if it is: piece i > 0 has to wait
// for piece i-1, and the last pieces, run last, find their predecessors done.
// Producer, MMA warp and epilogue enumerate the same sequence.
struct PairUnit {
    int tile, kb_lo, kb_hi, piece, sk_index;   // sk_index: split-tile number, -1 for a whole tile
};

// The tiles a pair walks: the whole grid (in groups of group_m tile rows), or under the
// die split its die's sub-grid (row by row: rs rows of a columns from s, then rows of b
// columns from u). cluster / clusters: the pair's index among the sub-grid's pairs and
// their number; split tiles are numbered from sk_off.
struct Sched {
    int cluster, clusters, num_tiles, sk_tiles, sk_pieces, sk_off;
    int split, rs, a, s, b, u;
};

__device__ __forceinline__ Sched make_sched(const GemmParams& p, int slot, int pairs) {
    Sched S;
    S.split = p.die_split;
    if (!p.die_split) {
        S.cluster = slot;
        S.clusters = pairs;
        S.num_tiles = p.num_tiles;
        S.sk_tiles = p.sk_tiles;
        S.sk_pieces = p.sk_pieces;
        S.sk_off = 0;
        S.rs = S.a = S.s = S.b = S.u = 0;
        return S;
    }
    const int h = slot < p.sub_n[0] ? 0 : 1;
    S.cluster = slot - (h ? p.sub_n[0] : 0);
    S.clusters = p.sub_n[h];
    S.rs = p.sub_rs;
    S.a = p.sub_a[h];
    S.s = p.sub_s[h];
    S.b = p.sub_b[h];
    S.u = p.sub_u[h];
    S.num_tiles = S.rs * S.a + (p.tiles_m - S.rs) * S.b;
    S.sk_tiles = p.sub_sk_tiles[h];
    S.sk_pieces = p.sub_sk_pieces[h];
    S.sk_off = h ? p.sub_sk_tiles[0] : 0;
    return S;
}

// Tile t of the walk: the grouped raster order over the whole grid, or the sub-grid's
// tiles row by row.
__device__ __forceinline__ void sched_tile_coords(int t, const GemmParams& p, const Sched& S, int& mb, int& nb) {
    if (!S.split) {
        tile_coords(t, p, mb, nb);
        return;
    }
    const int head = S.rs * S.a;   // tiles in the rows below rs
    if (t < head) {
        mb = t / S.a;
        nb = S.s + t % S.a;
    } else {
        const int r = t - head;
        mb = S.rs + r / S.b;
        nb = S.u + r % S.b;
    }
}

// Balanced stream-K: pair c's share of the region's k-blocks, [lo, hi) in the
// tile-major order of the region, as (tile, k-block) positions.
struct SkRange {
    int t_lo, k_lo, t_hi, k_hi;
};

__device__ __forceinline__ SkRange sk_range(const GemmParams& p, int c, int clusters) {
    const long long total = static_cast<long long>(p.sk_region) * p.num_kb;
    const long long lo = total * c / clusters, hi = total * (c + 1) / clusters;
    return {static_cast<int>(lo / p.num_kb), static_cast<int>(lo % p.num_kb), static_cast<int>(hi / p.num_kb),
            static_cast<int>(hi % p.num_kb)};
}

// A pair's units under balanced stream-K, in the order it runs them: the head
// piece that ends its range (the first piece of that tile: stored early), the
// whole tiles before the region (c, c + clusters, ...), the whole region tiles
// inside its range, and last the tail piece that begins its range (added after
// the head that the previous pair ran first).
__device__ __forceinline__ int pair_units_balanced(const GemmParams& p, int cluster, int clusters) {
    const SkRange r = sk_range(p, cluster, clusters);
    const int waves = p.sk_first / clusters;
    const int first_whole = r.k_lo > 0 ? r.t_lo + 1 : r.t_lo;
    return (r.k_hi > 0 ? 1 : 0) + waves + (r.t_hi - first_whole) + (r.k_lo > 0 ? 1 : 0);
}

__device__ __forceinline__ PairUnit pair_unit_balanced(const GemmParams& p, int cluster, int clusters, int u) {
    const SkRange r = sk_range(p, cluster, clusters);
    const int waves = p.sk_first / clusters;
    const int head = r.k_hi > 0 ? 1 : 0;
    const int first_whole = r.k_lo > 0 ? r.t_lo + 1 : r.t_lo;
    PairUnit U;
    U.sk_index = -1;
    U.piece = 0;
    U.kb_lo = 0;
    U.kb_hi = p.num_kb;
    if (u < head) {   // head of tile t_hi: the first piece of the tile cut by boundary `cluster`
        U.tile = p.sk_first + r.t_hi;
        U.kb_hi = r.k_hi;
        U.sk_index = cluster;
        return U;
    }
    u -= head;
    if (u < waves) {
        U.tile = cluster + u * clusters;
        return U;
    }
    u -= waves;
    if (u < r.t_hi - first_whole) {
        U.tile = p.sk_first + first_whole + u;
        return U;
    }
    // tail of tile t_lo: the last piece of the tile cut by boundary cluster - 1
    U.tile = p.sk_first + r.t_lo;
    U.kb_lo = r.k_lo;
    U.piece = 1;
    U.sk_index = cluster - 1;
    return U;
}

__device__ __forceinline__ int pair_units(const GemmParams& p, const Sched& S) {
    if (S.cluster < 0) return 0;   // die split without a rank (reported): no work
    if (p.sk_balanced) return pair_units_balanced(p, S.cluster, S.clusters);
    const int whole = S.num_tiles - S.sk_tiles;
    const int n = S.cluster < whole ? (whole - 1 - S.cluster) / S.clusters + 1 : 0;
    return n + (S.cluster < S.sk_tiles * S.sk_pieces ? 1 : 0);
}

// (tile numbers are the sub-grid's; sk_index is global)
__device__ __forceinline__ PairUnit pair_unit(const GemmParams& p, const Sched& S, int u) {
    if (p.sk_balanced) return pair_unit_balanced(p, S.cluster, S.clusters, u);
    PairUnit r;
    const int cluster = S.cluster;
    const bool has_piece = cluster < S.sk_tiles * S.sk_pieces;
    const int piece = has_piece ? cluster % S.sk_pieces : 0;
    const bool piece_first = has_piece && piece + 1 < S.sk_pieces;
    const int piece_at = piece_first ? 0 : pair_units(p, S) - 1;   // the piece's position
    if (has_piece && u == piece_at) {
        const int d = cluster / S.sk_pieces;
        r.sk_index = S.sk_off + d;
        r.piece = piece;
        r.tile = S.num_tiles - S.sk_tiles + d;
        r.kb_lo = r.piece * p.num_kb / S.sk_pieces;
        r.kb_hi = (r.piece + 1) * p.num_kb / S.sk_pieces;
    } else {
        r.sk_index = -1;
        r.piece = 0;
        r.tile = cluster + (u - (piece_first ? 1 : 0)) * S.clusters;
        r.kb_lo = 0;
        r.kb_hi = p.num_kb;
    }
    return r;
}

// Epilogue warp of a stream-K piece i > 0: wait until the warp with the same
// rows in piece i-1 has finished writing them (its flag reads gen·8 + i).
// Every lane performs an acquire of the flag before touching C.
__device__ __forceinline__ bool wait_sk_flag(const uint32_t* flag, uint32_t want, volatile uint32_t* abort_flag,
                                             AbortNet peer_abort, unsigned long long timeout_ns,
                                             unsigned int* status) {
    int ok = 1;
    if ((threadIdx.x & 31) == 0 && ptx::ld_acquire_gpu(flag) != want) {
        const uint64_t t0 = ptx::globaltimer_ns();
        while (ptx::ld_acquire_gpu(flag) != want) {
            if (*abort_flag) {
                ok = 0;
                break;
            }
            if (ptx::globaltimer_ns() - t0 > timeout_ns) {
                *abort_flag = 1u;
                peer_abort.raise();
                atomicCAS(status, 0u, static_cast<unsigned int>(DEV_TIMEOUT_SK_ORDER));
                ok = 0;
                break;
            }
        }
    }
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (ok) {
        (void)ptx::ld_acquire_gpu(flag);   // this lane's own acquire of the earlier piece's writes
        ptx::fence_proxy_async_global();  // ... ordered before this warp's TMA reductions
    }
    return ok != 0;
}

// Die split: this pair's rank (its slot among all pairs, sub-grid 0's first). One
// atomic on the counter of the pair's own die; when all of that die's ranks are taken
// (more pairs landed there than the map counted), one on the other die's. The counters
// start each launch at zero and every pair takes one rank, so the ranks are a
// permutation of the slots; -1 (reported) only if a counter was not zeroed.
__device__ __forceinline__ int claim_rank(const GemmParams& p) {
    const uint32_t tpc = ptx::smid() >> 1;
    uint32_t d = tpc < 128u ? p.die_of_tpc[tpc] : 255u;
    if (d > 1u) d = 0u;   // a pair the map does not place: either die (only locality depends on it)
    unsigned long long r = atomicAdd(p.sched_ctr + d, 1ull);
    if (r < static_cast<unsigned long long>(p.sub_n[d])) return (d ? p.sub_n[0] : 0) + static_cast<int>(r);
    const uint32_t e = d ^ 1u;
    r = atomicAdd(p.sched_ctr + e, 1ull);
    if (r < static_cast<unsigned long long>(p.sub_n[e])) return (e ? p.sub_n[0] : 0) + static_cast<int>(r);
    atomicCAS(p.status, 0u, DEV_SCHED_RANK);
    return -1;
}

__device__ __forceinline__ void spin_ns(unsigned long long ns) {
    const uint64_t t0 = ptx::globaltimer_ns();
    while (ptx::globaltimer_ns() - t0 < ns) {
    }
}

template <OutKind OK, int BN, int STAGES, int SLOTS, InKind IK>
__global__ void __launch_bounds__(PairCfg<OK, BN, STAGES, SLOTS, IK>::THREADS, 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmC, const GemmParams p) {
    using C = PairCfg<OK, BN, STAGES, SLOTS, IK>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = ptx::smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
    uint8_t* stage_base = smem;
    uint8_t* staging = smem + STAGES * C::STAGE_BYTES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(staging + C::STAGING_BYTES);
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 5);
    volatile uint32_t* abort_flag = tmem_holder + 1;
    volatile uint32_t* progress = tmem_holder + 2;   // k-blocks whose loads this CTA's producer has issued
    volatile int* slot_word = reinterpret_cast<volatile int*>(tmem_holder + 3);   // die split: the pair's rank

    const uint32_t full0 = ptx::smem_u32(bars);
    const uint32_t empty0 = ptx::smem_u32(bars + STAGES);
    const uint32_t accf0 = ptx::smem_u32(bars + 2 * STAGES);
    const uint32_t acce0 = ptx::smem_u32(bars + 2 * STAGES + 2);
    const uint32_t drain_bar = ptx::smem_u32(bars + 2 * STAGES + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t crank = ptx::cluster_ctarank();
    const uint32_t rank = crank & 1u;    // in the pair: 0 leader (issues the pair MMAs), 1 peer
    const bool leader = rank == 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(full0 + 8 * s, 1);    // leader's: its producer's arrival + both CTAs' bytes
            ptx::mbar_init(empty0 + 8 * s, 1);   // the leader's multicast commit
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(accf0 + 8 * b, 1);    // the leader's multicast commit
            ptx::mbar_init(acce0 + 8 * b, 2 * C::EPI_WARPS);   // leader's: every epilogue warp of both CTAs
        }
        ptx::mbar_init(drain_bar, 1);
        *abort_flag = 0u;
        *progress = 0u;
        ptx::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tensormap(&tmA);
        ptx::prefetch_tensormap(&tmB);
        ptx::prefetch_tensormap(&tmC);
    }
    if (warp == 1) {   // one warp in each CTA of the pair allocates, collectively
        ptx::tmem_alloc_pair(ptx::smem_u32(tmem_holder), C::TMEM_COLS);
        ptx::tmem_relinquish_pair();
    }
    __syncwarp();
    ptx::tc_fence_before();
    ptx::cluster_sync();   // barriers initialised and TMEM allocated in both CTAs
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    // Everything above touches only this CTA's own resources, so under a
    // programmatic launch it overlaps the previous kernel's tail; nothing
    // below reads or writes global memory before that kernel has finished.
    ptx::griddep_wait();
    ptx::griddep_launch_dependents();

    const uint32_t full_leader0 = ptx::mapa_shared(full0, 0u);
    const uint32_t acce_leader0 = ptx::mapa_shared(acce0, 0u);
    const AbortNet peer_abort{ptx::smem_u32(const_cast<uint32_t*>(abort_flag)), C::CL};
    const bool kps2 = p.kps2 != 0;
    const bool rel2 = C::REL == 2 || kps2;   // ring slots released in pairs (commits on odd slots)
    auto rel_slot = [rel2](uint32_t s) { return rel2 ? (s | 1u) : s; };
    const int pairs = gridDim.x / C::CL;
    int slot = blockIdx.x / C::CL;
    if (p.die_split) {
        // the leader takes the pair's rank and writes it into both CTAs; the cluster
        // barrier makes it visible to every thread of the pair
        if (leader && threadIdx.x == 0) {
            const int r = claim_rank(p);
            *slot_word = r;
            ptx::st_cluster_u32(ptx::mapa_shared(ptx::smem_u32(const_cast<int*>(slot_word)), 1u),
                                static_cast<uint32_t>(r));
        }
        ptx::cluster_sync();
        slot = *slot_word;
    }
    const Sched S = make_sched(p, slot, pairs);
    const bool tracing = (p.trace != nullptr) && (blockIdx.x == 0);
    if (tracing && threadIdx.x == 0) {   // SM clock and wall clock at the start of CTA 0's work
        p.trace[4 * p.trace_cap + 0] = ptx::clock64();
        p.trace[4 * p.trace_cap + 1] = ptx::globaltimer_ns();
    }

    if (warp == 0) {
        // ------------------------------------------------ producer (TMA), both CTAs
        // All 32 lanes run the loop; the arrival and the copies come from one
        // elected lane.
        uint32_t it = 0;
        bool ok = true;
        const bool hints = p.l2_hints != 0;
        const int units = pair_units(p, S);
        for (int u = 0; ok && u < units; ++u) {
            const PairUnit U = pair_unit(p, S, u);
            int mb, nb;
            sched_tile_coords(U.tile, p, S, mb, nb);
            const int row = mb * C::BM + static_cast<int>(rank) * C::ROWS;
            const int col = nb * C::BN + static_cast<int>(rank) * (C::BN / 2);
            for (int kb = U.kb_lo; kb < U.kb_hi; ++kb, ++it) {
                const uint32_t s = it % STAGES;
                const uint32_t ph = (it / STAGES) & 1u;
                if (kps2 && (s & 1u)) {   // loaded with the slot before it
                    if (lane == 0) *progress = it + 1;
                    continue;
                }
                const int kc = load_kblock(p, u, kb, U.kb_lo, U.kb_hi);
                if (!wait_warp_pair(empty0 + 8 * rel_slot(s), ph ^ 1u, abort_flag, peer_abort, p.timeout_ns,
                                    p.status, DEV_TIMEOUT_PRODUCER)) {
                    ok = false;
                    break;
                }
                if (tracing && lane == 0) {
                    const uint64_t now = ptx::clock64();
                    for (uint32_t j = it; j < it + (kps2 ? 2u : 1u); ++j) {   // (a pair of slots: both)
                        if (j >= STAGES && j - STAGES < (uint32_t)p.trace_cap) p.trace[4 * (j - STAGES) + 3] = now;
                        if (j < (uint32_t)p.trace_cap) p.trace[4 * j + 0] = now;
                    }
                }
                // a pair of slots: the copies bring this k-block and the next one of the walk (if
                // the tile has one; else the block after it in K, or zeros past the end of K),
                // the lower K coordinate first
                const bool two = kps2 && kb + 1 < U.kb_hi;
                if (leader) ptx::mbar_arrive_expect_tx_elected(full0 + 8 * s, kps2 ? 2 * C::PAIR_TX : C::PAIR_TX);
                const uint32_t sa = ptx::smem_u32(stage_base + s * C::A_BYTES);
                const uint32_t sb = ptx::smem_u32(stage_base + C::A_RING_BYTES + s * C::B_BYTES);
                const uint32_t fb = full_leader0 + 8 * s;
                const uint32_t done = it + (two ? 2u : 1u);
                // test hook: CTA 0 announces the stage's bytes but never loads its share
                if (blockIdx.x == 0 && (kps2 ? (it | 1u) == (static_cast<uint32_t>(p.debug_skip_kb) | 1u)
                                             : static_cast<int>(it) == p.debug_skip_kb)) {
                    if (lane == 0) *progress = done;
                    continue;
                }
                if (kps2) {
                    const int k0 = two ? min(kc, load_kblock(p, u, kb + 1, U.kb_lo, U.kb_hi)) : kc;
                    if (hints) {
                        ptx::tma_load_3d_pair_hint(sa, &tmA, fb, 0, row, k0, ptx::policy_evict_first());
                        ptx::tma_load_4d_pair_hint(sb, &tmB, fb, 0, 0, col / C::B_BOX_N, k0, ptx::policy_evict_last());
                    } else {
                        ptx::tma_load_3d_pair_elected(sa, &tmA, fb, 0, row, k0);
                        ptx::tma_load_4d_pair_elected(sb, &tmB, fb, 0, 0, col / C::B_BOX_N, k0);
                    }
                } else {
                    if (hints)
                        ptx::tma_load_2d_pair_hint(sa, &tmA, fb, kc * C::BK, row, ptx::policy_evict_first());
                    else
                        ptx::tma_load_2d_pair_elected(sa, &tmA, fb, kc * C::BK, row);
                    if (p.b_3d && hints) {
                        ptx::tma_load_3d_pair_hint(sb, &tmB, fb, 0, kc * C::BK, col / C::B_BOX_N,
                                                   ptx::policy_evict_last());
                    } else if (p.b_3d) {   // this CTA's B_BOXES boxes in one copy (boxes B_BOX_BYTES apart, as below)
                        ptx::tma_load_3d_pair_elected(sb, &tmB, fb, 0, kc * C::BK, col / C::B_BOX_N);
                    } else {
#pragma unroll
                        for (int b = 0; b < C::B_BOXES; ++b)
                            ptx::tma_load_2d_pair_elected(sb + b * C::B_BOX_BYTES, &tmB, fb, col + b * C::B_BOX_N,
                                                          kc * C::BK);
                    }
                }
                if (lane == 0) *progress = done;
            }
            if (ok && kps2 && (it & 1u)) {   // the next tile starts on an even slot
                ++it;
                if (lane == 0) *progress = it;
            }
        }
        if (!ok && lane == 0) spin_ns(200000);   // copies issued before the abort land within microseconds
        if (ok && tracing && lane == 0) {
            // stamp "MMAs done" for the last STAGES k-blocks, whose stages are never reused
            // (the same empty-barrier phases a reuse would have waited for; bounded)
            const uint32_t first = it > (uint32_t)STAGES ? it - STAGES : 0u;
            for (uint32_t j = first; j < it && j < (uint32_t)p.trace_cap && !*abort_flag; ++j) {
                wait_drain(empty0 + 8 * rel_slot(j % STAGES), (j / STAGES) & 1u, p.timeout_ns);
                p.trace[4 * j + 3] = ptx::clock64();
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer (leader CTA only)
        // All 32 lanes of the leader's MMA warp run the loop; the MMAs and
        // commits come from one elected lane through predicates.
        if (leader) {
            // Stage-0 descriptors; stages and k-slices are constant offsets of the
            // start-address field (16-byte units).
            const uint32_t stage0 = ptx::smem_u32(stage_base);
            const uint64_t adesc0 = ptx::sdesc_sw128(stage0, 16, 1024);
            // B N-major: boxes B_BOX_BYTES apart (leading offset), core groups of K-rows
            // B_SBO apart, a k-slice steps UMMA_K rows of 128 B
            const uint64_t bdesc0 = ptx::sdesc(stage0 + C::A_RING_BYTES, C::B_BOX_BYTES, InTraits<IK>::B_SBO,
                                               InTraits<IK>::B_LAYOUT);
            constexpr uint64_t A_STEP = C::UMMA_K * C::ES / 16;
            constexpr uint64_t B_STEP = C::UMMA_K * 128 / 16;
            constexpr uint64_t SA_STEP = C::A_BYTES / 16;
            constexpr uint64_t SB_STEP = C::B_BYTES / 16;
            static_assert(C::KSUB == 4, "four MMAs per k-block");
            uint32_t it = 0, unit = 0, s = 0, ph = 0;
            bool ok = true;
            const int units = pair_units(p, S);
            for (int u = 0; ok && u < units; ++u) {
                const PairUnit U = pair_unit(p, S, u);
                const bool desc = p.k_serpentine && (u & 1);   // this tile's loads walk K downwards
                // accumulation units of kb_per_unit k-blocks (exact-integer mode: 1024 K
                // values, drained into int32 sums; otherwise the whole range)
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
                    for (int kb = kb0; kb < kb1; ++kb, ++it) {
                        // (a pair of slots completes on the first one's barrier)
                        if (!wait_warp_pair(full0 + 8 * (kps2 ? (s & ~1u) : s), ph, abort_flag, peer_abort,
                                            p.timeout_ns, p.status, DEV_TIMEOUT_MMA_FULL)) {
                            ok = false;
                            break;
                        }
                        ptx::tc_fence_after();
                        if (tracing && lane == 0 && it < (uint32_t)p.trace_cap) p.trace[4 * it + 1] = ptx::clock64();
                        // a pair of slots holds the lower K block first: a tile walking K
                        // downwards takes the second slot first (the summation order of one
                        // k-block per copy)
                        const uint32_t ds = (kps2 && desc && ((s & 1u) || kb + 1 < U.kb_hi)) ? (s ^ 1u) : s;
                        const uint64_t ad = adesc0 + ds * SA_STEP;
                        const uint64_t bd = bdesc0 + ds * SB_STEP;
                        if constexpr (IK == InKind::TF32)
                            ptx::mma_tf32_pair_x4_elected(d_tmem, ad, bd, ad + A_STEP, bd + B_STEP, ad + 2 * A_STEP,
                                                          bd + 2 * B_STEP, ad + 3 * A_STEP, bd + 3 * B_STEP, C::IDESC,
                                                          kb > kb0 ? 1u : 0u);
                        else
                            ptx::mma_f16_pair_x4_elected(d_tmem, ad, bd, ad + A_STEP, bd + B_STEP, ad + 2 * A_STEP,
                                                         bd + 2 * B_STEP, ad + 3 * A_STEP, bd + 3 * B_STEP, C::IDESC,
                                                         kb > kb0 ? 1u : 0u);
                        // stage s (with s - 1, released in pairs) free in both CTAs once these MMAs are done
                        if (!rel2 || (s & 1u)) ptx::mma_commit_pair_multicast_elected(empty0 + 8 * s, C::ALL);
                        if (tracing && lane == 0 && it < (uint32_t)p.trace_cap) p.trace[4 * it + 2] = ptx::clock64();
                        const uint32_t wrap = (s + 1 == static_cast<uint32_t>(STAGES)) ? 1u : 0u;
                        s = wrap ? 0u : s + 1;
                        ph ^= wrap;
                    }
                    if (!ok) break;
                    ptx::mma_commit_pair_multicast_elected(accf0 + 8 * buf, C::ALL);
                }
                if (ok && kps2 && (s & 1u)) {
                    // the tile ended on the first slot of a pair: release the pair, skip the
                    // second slot (the next tile starts on an even slot)
                    ptx::mma_commit_pair_multicast_elected(empty0 + 8 * s, C::ALL);
                    const uint32_t wrap = (s + 1 == static_cast<uint32_t>(STAGES)) ? 1u : 0u;
                    s = wrap ? 0u : s + 1;
                    ph ^= wrap;
                    ++it;
                }
            }
            if (ok && tracing && C::REL == 2 && it > 0) {
                // slots released in pairs: release a last k-block left alone in an even slot,
                // so that the producer's trace sees its MMAs finish
                const uint32_t last = (s + STAGES - 1) % STAGES;
                if (!(last & 1u)) ptx::mma_commit_pair_multicast_elected(empty0 + 8 * (last | 1u), C::ALL);
            }
            if (!ok) {
                ptx::mma_commit_pair_multicast_elected(drain_bar, 0x1);
                if (lane == 0) wait_drain(drain_bar, 0, p.timeout_ns);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ epilogue (warps 2.., both CTAs)
        const int q = warp & 3;                                // TMEM lane quarter this warp may read
        [[maybe_unused]] const int h = (warp - 2) / 4;         // column part (exact integers, 8 warps)
        constexpr int CW = C::EPI_COLS_PER_WARP;
        uint8_t* slab_pair = staging + (warp - 2) * C::EPI_SLOTS * C::SLAB_BYTES;
        int store_count = 0;
        uint32_t unit = 0;
        uint32_t it_next = 0;   // the ring iteration at which the unit after this one starts
        bool ok = true;
        // stream-K: this warp's rows of split tile d, flags[d][rank][epilogue warp]
        auto sk_flag = [&](const PairUnit& U) -> uint32_t* {
            return U.sk_index >= 0 ? p.sk_flags + (U.sk_index * 2 + rank) * C::EPI_WARPS + (warp - 2) : nullptr;
        };
        // piece > 0: wait until the previous piece's sums are in C (or in the workspace)
        auto wait_turn = [&](uint32_t* flag, const PairUnit& U) {
            if (!wait_sk_flag(flag, (p.sk_gen << 3) | static_cast<uint32_t>(U.piece), abort_flag, peer_abort,
                              p.timeout_ns, p.status))
                return false;
            if (U.piece + 1 == S.sk_pieces) {
                // the flag's last reader leaves it as this launch found it (0), so that a
                // replay of the same launch (a CUDA graph: same generation) waits again
                __syncwarp();   // every lane has made its acquire of the flag
                if (lane == 0) *reinterpret_cast<volatile uint32_t*>(flag) = 0u;
            }
            return true;
        };
        auto hand_over = [&](uint32_t* flag, const PairUnit& U) {
            // hand these rows to the next piece once every write to them has landed
            __threadfence();   // the ragged-edge chunk's element writes, from every lane
            __syncwarp();
            // (test hook: the first piece of split tile 0 never hands over)
            const bool held = p.debug_sk_stall && U.sk_index == 0 && U.piece == 0;
            if (lane == 0) {
                ptx::bulk_wait<0>();               // this warp's stores/reductions completed
                ptx::fence_proxy_async_global();   // ... and ordered before the release
                if (!held) ptx::st_release_gpu(flag, (p.sk_gen << 3) | static_cast<uint32_t>(U.piece + 1));
            }
            __syncwarp();
        };
        const int units = pair_units(p, S);
        for (int u = 0; ok && u < units; ++u) {
            const PairUnit U = pair_unit(p, S, u);
            it_next += static_cast<uint32_t>(kps2 ? (U.kb_hi - U.kb_lo + 1) & ~1 : U.kb_hi - U.kb_lo);
            int mb, nb;
            sched_tile_coords(U.tile, p, S, mb, nb);
            const int row0 = mb * C::BM + static_cast<int>(rank) * C::ROWS + q * 32;
            // bf16 C, split tile: this warp's block of the fp32 workspace (32 rows × BN)
            [[maybe_unused]] float* blk = nullptr;
            if constexpr (OK == OutKind::BF16) {
                if (U.sk_index >= 0) {
                    const int wrow0 = (U.sk_index * 2 + static_cast<int>(rank)) * C::ROWS + q * 32;
                    blk = p.sk_ws + static_cast<long long>(wrow0) * C::BN;
                    // a later piece reads the block after its mainloop: have it in L2 by then
                    // (written near the start of the launch, it may have left L2 since)
                    if (U.piece > 0 && lane == 0) ptx::prefetch_l2_bulk(blk, 32 * C::BN * 4);
                }
            }
            [[maybe_unused]] int32_t iacc[(OK == OutKind::S32) ? CW : 1];
            if constexpr (OK == OutKind::S32) {
#pragma unroll
                for (int i = 0; i < CW; ++i) iacc[i] = 0;
            }
            for (int kb0 = U.kb_lo; ok && kb0 < U.kb_hi; kb0 += p.kb_per_unit, ++unit) {
                const uint32_t buf = unit & 1u;
                const uint32_t uph = (unit >> 1) & 1u;
                bool got = true;
                if (lane == 0)
                    got = wait_bounded_pair(accf0 + 8 * buf, uph, abort_flag, peer_abort, p.timeout_ns, p.status,
                                            DEV_TIMEOUT_EPILOGUE);
                if (__shfl_sync(0xffffffffu, got ? 1 : 0, 0) == 0) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                if constexpr (OK == OutKind::S32) {
                    // exact integers: this unit's fp32 sums (each an integer below 2^24 in
                    // magnitude) converted and added into int32 registers; the tile's int32
                    // result is stored after its last unit
                    const uint32_t tb =
                        tmem_base + (static_cast<uint32_t>(q * 32) << 16) + buf * C::ACC_STRIDE + h * CW;
                    // (16 columns at a time: the 128 sums already hold most of a thread's registers)
#pragma unroll
                    for (int c = 0; c < CW / 16; ++c) {
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
                    if (kb0 + p.kb_per_unit >= U.kb_hi) {
                        // a stream-K piece after the first adds its sums into C (integer reduction)
                        uint32_t* flag = sk_flag(U);
                        if (flag && U.piece > 0 && !wait_turn(flag, U)) {
                            ok = false;
                            break;
                        }
#pragma unroll
                        for (int c = 0; c < CW / 32; ++c) {
                            const uint32_t(&v)[32] = *reinterpret_cast<const uint32_t(*)[32]>(&iacc[c * 32]);
                            store_slab<C::SLAB_BYTES, 4, C::EPI_SLOTS, true>(
                                &tmC, slab_pair, store_count, v, lane, nb * C::BN + h * CW + c * 32, row0, p,
                                U.piece > 0);
                        }
                        if (flag && U.piece + 1 < S.sk_pieces) hand_over(flag, U);
                    }
                    continue;
                }
                uint32_t* flag = sk_flag(U);
                if (flag && U.piece > 0 && !wait_turn(flag, U)) {
                    ok = false;
                    break;
                }
                const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + buf * C::ACC_STRIDE;
                auto release = [&]() {
                    ptx::tc_fence_before();
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive_cluster_relaxed(acce_leader0 + 8 * buf);
                };
                if constexpr (OK == OutKind::BF16) {
                    if (flag) {
                        // bf16 C, split tile: the pieces' fp32 sums meet in this warp's
                        // workspace block (stored by piece 0, added by the next ones in piece
                        // order); the last piece adds the block and rounds once into C
                        if (U.piece + 1 < S.sk_pieces) {
                            drain_to_workspace<C::BN / 32>(tbase, lane, blk, release, U.piece > 0);
                            hand_over(flag, U);
                        } else {
                            drain_accumulator<OK, C::EPI_CHUNKS, C::SLAB_BYTES, C::EPI_SLOTS>(
                                &tmC, slab_pair, store_count, tbase, lane, nb * C::BN, row0, p, release, false,
                                NoPace(), blk);
                        }
                        continue;
                    }
                }
                drain_accumulator<OK, C::EPI_CHUNKS, C::SLAB_BYTES, C::EPI_SLOTS>(
                    &tmC, slab_pair, store_count, tbase, lane, nb * C::BN, row0, p, release,
                    /*add=*/U.piece > 0, [&](int c) {
                        // Spread this tile's stores over the next unit's mainloop: chunk c waits
                        // until the producer is c/EPI_CHUNKS of the way through that unit (a
                        // burst of TMA stores slows the tensor pipe's operand reads). The
                        // CTA's last unit, and a stream-K piece (the next piece waits for
                        // it), store at once.
                        if (u + 1 >= units || c == 0 || U.sk_index >= 0) return;
                        const PairUnit V = pair_unit(p, S, u + 1);
                        const uint32_t n = static_cast<uint32_t>(V.kb_hi - V.kb_lo);
                        // (the producer issues all n k-blocks of the next unit, so the target is reached)
                        const uint32_t target = it_next + min(n, STAGES + c * n / C::EPI_CHUNKS);
                        if (lane == 0 && *progress < target) {
                            const uint64_t t0 = ptx::globaltimer_ns();
                            while (*progress < target && !*abort_flag && ptx::globaltimer_ns() - t0 < p.timeout_ns) {
                            }
                        }
                        __syncwarp();
                    });
                if (flag && U.piece + 1 < S.sk_pieces) hand_over(flag, U);
            }
        }
        if (lane == 0) ptx::bulk_wait<0>();
        __syncwarp();
    }

    // ------------------------------------------------ teardown
    ptx::tc_fence_before();
    __syncthreads();
    if (tracing && threadIdx.x == 0) {   // ... and at its end: their ratio is the SM clock in the kernel
        p.trace[4 * p.trace_cap + 2] = ptx::clock64();
        p.trace[4 * p.trace_cap + 3] = ptx::globaltimer_ns();
    }
    ptx::cluster_sync();   // no CTA frees TMEM or exits while its peer may still signal it
    if (p.die_split && leader && threadIdx.x == 0) {
        // the last pair to finish zeroes the rank counters for the next launch (every
        // pair took its rank before it got here)
        __threadfence();
        const unsigned long long done = atomicAdd(p.sched_ctr + 2, 1ull);
        if (done + 1 == static_cast<unsigned long long>(pairs)) {
            __threadfence();
            atomicExch(p.sched_ctr + 0, 0ull);
            atomicExch(p.sched_ctr + 1, 0ull);
            atomicExch(p.sched_ctr + 2, 0ull);
        }
    }
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
    }
}

}  // namespace tcl
