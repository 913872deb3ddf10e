// Persistent, warp-specialised tensor-core GEMM for sm_103a:
//   C[M×N] = A[M×K] · B[K×N], A and B row-major, fp32 accumulation in TMEM.
//
// The K-loop is the software pipeline the pages describe ("流水化 GPU 内核",
// steps 3-4: prologue / steady state / drain with the load of tile k+1
// overlapping the MMA on tile k; "4.1 CUDA GEMM 算子性能优化" §9.3-§10.4:
// global→shared double buffering generalised to a multi-stage ring), rebuilt
// for Blackwell:
//   * warp 0 (producer): TMA 2-D tiled loads of the A tile (BM×BK, K-major)
//     and the B tile (BK×BN, N-major, straight from the row-major K×N
//     matrix) into stage s of a STAGES-deep ring, 128-byte swizzled (for
//     TF32's 4-byte B, in 32-byte units); completion tracked by the full[s]
//     mbarrier as transaction bytes. It waits on empty[s] before reusing a
//     stage.
//   * warp 1 (MMA issuer): one thread issues tcgen05.mma (kind::f16 or
//     kind::tf32) per UMMA_K slice into a TMEM accumulator, and commits
//     empty[s] when the stage's MMAs are done; at the end of a unit it
//     commits acc_full[b]. Two accumulators let the epilogue of one tile run
//     under the mainloop of the next.
//   * warps 2-5 (epilogue): tcgen05.ld 32 lanes × 32 columns per warp, convert
//     (fp32 pass-through, fp32→bf16 round-to-nearest-even, or exact
//     integer drain), write a 128-byte-swizzled staging slab and TMA-store
//     it to C; then release acc_empty[b].
//   * tiles are walked persistently (tile = blockIdx.x + i·gridDim.x) in a
//     grouped raster order ("4.1 CUDA GEMM 算子性能优化" §2.3: the order in
//     which blocks are scheduled decides the L2 hit rate).
//
// Exact integer mode (OutKind::S32): the operands are integers stored as
// bf16 (exact for |x| ≤ 256), every product is an exact integer, and fp32
// holds every integer of magnitude ≤ 2^24. The MMA warp therefore closes an
// accumulation unit every `kb_per_unit` k-blocks, chosen on the host so that
// the sum of |products| inside one unit stays ≤ 2^24, and the epilogue adds
// each unit, converted to int32, into per-thread int32 registers.
//
// Every wait on an mbarrier is bounded: after `timeout_ns` of %globaltimer it
// records an error code in the device status word, raises a shared abort
// flag that the other roles poll, lets its own in-flight copies and MMAs
// finish, and the kernel returns normally (TMEM freed). No trap, no assert.
#pragma once

#include <cuda_bf16.h>

#include "ptx.cuh"

namespace tcl {

enum class InKind : int { BF16 = 0, TF32 = 1 };
enum class OutKind : int { F32 = 0, BF16 = 1, S32 = 2 };

// Device status codes (first failure wins).
enum : unsigned int {
    DEV_OK = 0,
    DEV_TIMEOUT_PRODUCER = 1,   // producer waited too long for a free stage
    DEV_TIMEOUT_MMA_FULL = 2,   // MMA warp waited too long for a stage's data
    DEV_TIMEOUT_MMA_ACC = 3,    // MMA warp waited too long for a free accumulator
    DEV_TIMEOUT_EPILOGUE = 4,   // epilogue waited too long for a finished accumulator
    DEV_TIMEOUT_SK_ORDER = 5,   // epilogue waited too long for the previous piece of a split tile
    DEV_SCHED_RANK = 6,         // die split: a pair found no rank free (counters not zeroed)
};

template <InKind IK>
struct InTraits;
template <>
struct InTraits<InKind::BF16> {
    static constexpr int ES = 2;        // bytes per element
    static constexpr int UMMA_K = 16;   // K per tcgen05.mma
    static constexpr uint32_t FMT = 1;  // bf16
    // N-major B: descriptor layout (128-byte swizzle) and the byte distance
    // between the descriptor's core groups along K (8 rows of 128 bytes)
    static constexpr uint32_t B_LAYOUT = 2;
    static constexpr uint32_t B_SBO = 1024;
};
template <>
struct InTraits<InKind::TF32> {
    static constexpr int ES = 4;
    static constexpr int UMMA_K = 8;
    static constexpr uint32_t FMT = 2;  // tf32
    // N-major B of 4-byte elements: 128-byte swizzle in 32-byte units (the tensor
    // copy's SWIZZLE_128B_ATOM_32B), core groups of 4 rows of 128 bytes
    static constexpr uint32_t B_LAYOUT = 1;
    static constexpr uint32_t B_SBO = 512;
};

struct GemmParams {
    int M, N, K;
    int tiles_m, tiles_n, num_tiles;
    int num_kb;        // k-blocks per tile, ceil(K / BK)
    int kb_per_unit;   // k-blocks per TMEM accumulation unit (num_kb unless S32)
    int group_m;       // raster group height in tiles
    unsigned long long timeout_ns;
    unsigned int* status;        // device status word
    unsigned long long* trace;   // optional per-k-block timeline of CTA 0 (nullptr: off)
    int trace_cap;               // k-blocks the trace buffer holds
    void* C;                     // output base, for the ragged right edge only
    long long ldc;               // output leading dimension in elements
    const void* A;               // operand bases, read directly by the synchronous producer
    long long lda;
    const void* B;
    long long ldb;
    int debug_skip_kb;           // test hook: CTA 0's TMA producer never loads this k-block (-1: off)
    int splits;                  // K split into this many ranges (1: no split); work items = tiles × splits
    int kb_per_split;            // k-blocks per split (the last may have fewer)
    int split_rows;              // output rows between consecutive splits' partial results
    int out_rows;                // rows of the output tensor (M, or splits × split_rows)
    // Stream-K tail (two-SM kernel, fp32 C): the last sk_tiles tiles are each
    // cut into sk_pieces K ranges, one per pair of SMs; piece 0 stores its
    // result, piece i > 0 adds its own once piece i-1 has finished (flags).
    int sk_tiles;                // 0: every tile is whole
    int sk_pieces;               // K ranges per split tile (>= 2 when sk_tiles > 0)
    // Balanced stream-K (sk_balanced = 1): the tiles from sk_first on (sk_region of
    // them) are not dealt out whole; their k-blocks, in tile order, are cut into one
    // equal range per pair, so a pair's range may begin inside one tile and end inside
    // another. A tile cut by the boundary between pairs b and b+1 has two pieces: the
    // head [0, k) run by pair b (stored), the rest run by pair b+1 (added after the
    // head); the boundary's number b indexes its flags and workspace. sk_pieces is 2.
    int sk_balanced;
    int sk_first;
    int sk_region;
    unsigned int* sk_flags;      // [sk_tiles][2 CTAs][epilogue warp] progress flags
    unsigned int sk_gen;         // this launch's flag generation (flags hold gen·8 + pieces done)
    int debug_sk_stall;          // test hook: piece 0 of split tile 0 never publishes its flag
    // bf16 C with a stream-K tail: the pieces before the last add their fp32 sums in a
    // workspace of sk_ws_rows / 32 blocks, one per epilogue warp's 32 rows of a split
    // tile, each BN/4 groups × 32 lanes × 4 fp32 (a warp's 16-byte accesses to one
    // column group are 512 contiguous bytes); the last piece adds its block to its own
    // sums and rounds once into C
    float* sk_ws;
    int sk_ws_rows;
    // 1: the units at odd positions of each CTA's walk load their k-blocks in
    // descending order (the MMAs and the accumulation units follow the loads), so
    // that a wave starts on the operand rows the previous wave read last, which
    // are the ones still in L2
    int k_serpentine;
    // 1: tmB is a 3-D map (a box's columns, K, column blocks) and one tensor copy brings all
    // of a stage's B boxes (TMA producer, N a whole number of boxes)
    int b_3d;
    // 1 (two-SM kernel): two k-blocks per tensor copy. tmA is a 3-D map (K of a block, rows,
    // k-blocks) and tmB a 4-D one (a box's columns, K of a block, column blocks, k-blocks);
    // the copies at an even ring slot fill that slot and the next, the odd slot loads nothing,
    // slots are released in pairs, and each tile's walk starts on an even slot
    int kps2;
    // Die split (two-SM kernel): the tile columns are cut into two sub-grids, one per die
    // of the GPU, each walked by the pairs of SMs on that die (so that each die's half of
    // the L2 holds its own sub-grid's operands). A pair's leader takes a rank on its die
    // (sched_ctr[die], one atomic; when that die's ranks are all taken, a rank on the other
    // die), so every rank is taken exactly once whatever the placement; the last pair to
    // finish zeroes the counters (sched_ctr[2] counts finished pairs). Each sub-grid has
    // its own stream-K tail; its split tiles are numbered after those of the sub-grids
    // before it.
    // 1 (two-SM kernel): A's loads carry an L2 evict-first policy and B's evict-last, so
    // that each die's half of the L2 keeps the B columns its waves share while the rows
    // of A stream through
    int l2_hints;
    int die_split;
    int sub_n[2];            // pairs of each sub-grid (sub_n[0] + sub_n[1] = gridDim.x / 2)
    // Sub-grid h holds, in tile rows below sub_rs, the sub_a[h] tile columns from sub_s[h],
    // and in the other rows the sub_b[h] columns from sub_u[h]: a block of whole columns
    // plus part of one column, so that each sub-grid's tile count follows its pairs to the
    // tile. Walked row by row.
    int sub_rs;
    int sub_a[2], sub_s[2], sub_b[2], sub_u[2];
    int sub_sk_tiles[2];     // stream-K split tiles of each sub-grid
    int sub_sk_pieces[2];
    unsigned long long* sched_ctr;
    uint8_t die_of_tpc[128];   // die (0, 1; 255 unknown) of the pair of SMs (SM id / 2)
};

// K coordinate (in k-blocks) that the load at position kb of the range
// [kb_lo, kb_hi) fetches, for the unit at position `pos` of a CTA's walk.
__device__ __forceinline__ int load_kblock(const GemmParams& p, int pos, int kb, int kb_lo, int kb_hi) {
    return (p.k_serpentine && (pos & 1)) ? kb_lo + kb_hi - 1 - kb : kb;
}

// Work item w → output tile (mb, nb), its k-block range [kb_lo, kb_hi) and
// the row where its result starts in the output tensor. Splits of one tile
// are num_tiles work items apart, so a wave covers many tiles at once.
struct Work {
    int mb, nb, kb_lo, kb_hi, row_base;
};

__device__ __forceinline__ void tile_coords(int t, const GemmParams& p, int& mb, int& nb);

__device__ __forceinline__ Work work_item(int w, const GemmParams& p) {
    Work r;
    const int split = w / p.num_tiles;
    tile_coords(w - split * p.num_tiles, p, r.mb, r.nb);
    r.kb_lo = split * p.kb_per_split;
    r.kb_hi = min(p.num_kb, r.kb_lo + p.kb_per_split);
    r.row_base = split * p.split_rows;
    return r;
}

// Producer kinds: TMA bulk-tensor copies issued by one elected lane; the
// synchronous variant (four warps: ld.global into registers, st.shared into
// the same swizzled layout, then an mbarrier arrive); the cp.async variant
// (four warps issue 16-byte asynchronous copies straight into the swizzled
// layout, each thread's arrival fires when its copies land). The last two are
// the rungs below TMA in the ablation.
enum : int { PROD_TMA = 0, PROD_SYNC = 1, PROD_CPASYNC = 2 };

constexpr int pow2_at_least(int x, int lo) {
    int p = lo;
    while (p < x) p <<= 1;
    return p;
}

template <InKind IK, OutKind OK, int BN_, int STAGES_, int PROD_ = PROD_TMA>
struct KCfg {
    static constexpr int PROD = PROD_;
    static constexpr int P_WARPS = PROD == PROD_TMA ? 1 : 4;    // producer warps
    static constexpr int MMA_WARP = P_WARPS;                    // then the MMA warp
    static constexpr int EPI_WARP0 = P_WARPS + 1;               // then four epilogue warps
    static constexpr int FULL_ARRIVALS = PROD == PROD_TMA ? 1 : 32 * P_WARPS;
    static constexpr int BM = 128;
    static constexpr int BN = BN_;
    static constexpr int STAGES = STAGES_;
    static constexpr int ES = InTraits<IK>::ES;
    static constexpr int BK = 128 / ES;               // one 128-byte swizzle row of K
    static constexpr int UMMA_K = InTraits<IK>::UMMA_K;
    static constexpr int KSUB = BK / UMMA_K;          // MMAs per k-block
    static constexpr int A_BYTES = BM * 128;          // BM rows × 128 B
    // B as stored in global memory, N-major (row-major K×N), read as boxes of
    // one 128-byte row of N (64 bf16 or 32 TF32 columns) × BK rows.
    static constexpr int B_BOX_N = 128 / ES;   // N columns per box
    static constexpr int B_BOXES = BN / B_BOX_N;
    static constexpr int B_BOX_BYTES = BK * 128;
    static constexpr int B_BYTES = B_BOXES * B_BOX_BYTES;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int OUT_ES = (OK == OutKind::BF16) ? 2 : 4;
    static constexpr int EPI_COLS = 128 / OUT_ES;     // output columns per 128-byte staging row
    static constexpr int EPI_CHUNKS = BN / EPI_COLS;
    static constexpr int SLAB_BYTES = 32 * 128;       // one warp's 32 rows × 128 B
    static constexpr int EPI_SLOTS = 2;               // staging slabs per epilogue warp
    static constexpr int STAGING_BYTES = 4 * EPI_SLOTS * SLAB_BYTES;
    static constexpr int TMEM_COLS = pow2_at_least(2 * BN, 32);
    static constexpr int BAR_BYTES = 256;
    static constexpr int SMEM_USED = 1024 + STAGES * STAGE_BYTES + STAGING_BYTES + BAR_BYTES;
    // Request more than half of the SM's 228 KB so that exactly one CTA is
    // resident per SM: its TMEM allocation is then never contended and every
    // ring depth is measured under the same occupancy.
    static constexpr int SMEM_BYTES = SMEM_USED > 122880 ? SMEM_USED : 122880;
    static constexpr uint32_t IDESC =
        ptx::make_idesc(InTraits<IK>::FMT, InTraits<IK>::FMT, /*A K-major*/ 0, /*B N-major*/ 1, BM, BN);
    static constexpr int THREADS = 32 * (P_WARPS + 5);
    // Ring slots released per commit. A tcgen05.commit costs the tensor pipe
    // about 67 cycles when the MMAs between commits take less time than the
    // issue loop around them (N = 128: 4 MMAs of 64 cycles per k-block;
    // measured on GB300 with the tensor-pipe probe); from N = 192 on it is
    // hidden. With N <= 128 and an even ring of at least 4 slots, the MMA warp
    // commits only after the second slot of each pair (2j, 2j+1), and the
    // producer refills either slot once that commit has landed.
    static constexpr int REL = (BN <= 128 && STAGES >= 4 && STAGES % 2 == 0) ? 2 : 1;
    static __device__ __forceinline__ uint32_t rel_slot(uint32_t s) { return REL == 2 ? (s | 1u) : s; }

    static_assert(BN % B_BOX_N == 0, "BN must be a whole number of swizzle boxes");
    static_assert(BN % EPI_COLS == 0, "BN must be a whole number of epilogue chunks");
    static_assert(BN >= 16 && BN <= 256 && BN % 16 == 0, "UMMA N for M=128 is 16..256 step 16");
    static_assert(2 * BN <= 512, "two accumulators must fit the 512 TMEM columns");
    static_assert(STAGES >= 1 && 2 * STAGES + 5 <= 28, "barrier area");
    static_assert(SMEM_BYTES <= 232448, "exceeds the 227 KB per-block shared memory limit");
    static_assert(OK != OutKind::S32 || BN <= 128, "exact integer drain keeps BN int32 sums in registers");
    static_assert(PROD == PROD_TMA || PROD == PROD_SYNC || PROD == PROD_CPASYNC, "producer kind");
    static_assert(PROD == PROD_TMA || IK == InKind::BF16, "thread-copy producers: bf16 only");
};

__device__ __forceinline__ void tile_coords(int t, const GemmParams& p, int& mb, int& nb) {
    const int per_group = p.group_m * p.tiles_n;
    const int g = t / per_group;
    const int first_m = g * p.group_m;
    const int rows = min(p.tiles_m - first_m, p.group_m);
    const int r = t - g * per_group;
    mb = first_m + r % rows;
    nb = r / rows;
}

// Bounded wait on an mbarrier phase. Returns false (and raises the abort flag,
// recording `code` if it is the first failure) once `timeout_ns` has passed,
// or as soon as another role has raised the abort flag.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity,
                                             volatile uint32_t* abort_flag,
                                             unsigned long long timeout_ns, unsigned int* status,
                                             unsigned int code) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer_ns();
    while (true) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (ptx::globaltimer_ns() - t0 > timeout_ns) {
            *abort_flag = 1u;
            atomicCAS(status, 0u, code);
            return false;
        }
    }
}

// Bounded wait used only while draining after an abort: ignores the flag.
__device__ __forceinline__ void wait_drain(uint32_t bar, uint32_t parity,
                                           unsigned long long timeout_ns) {
    const uint64_t t0 = ptx::globaltimer_ns();
    while (!ptx::mbar_try_wait(bar, parity)) {
        if (ptx::globaltimer_ns() - t0 > timeout_ns) return;
    }
}

// Warp-uniform bounded wait for a warp whose 32 lanes run the same loop: all
// lanes poll once; unless the phase is complete for every lane, lane 0 takes
// the bounded slow path and broadcasts the outcome, so the warp never diverges.
__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag,
                                          unsigned long long timeout_ns, unsigned int* status, unsigned int code) {
    if (__all_sync(0xffffffffu, ptx::mbar_try_wait(bar, parity))) return true;
    int ok = 1;
    if ((threadIdx.x & 31) == 0) ok = wait_bounded(bar, parity, abort_flag, timeout_ns, status, code) ? 1 : 0;
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr)
                 : "memory");
    return v;
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

// One warp writes 32 rows × 128 bytes (row = lane) into a staging slab in the
// 128-byte swizzled layout the C tensor map expects (16-byte chunk j of row r
// lands at chunk j ^ (r mod 8)), then lane 0 TMA-stores the slab.
// Always commits one bulk group per call so that "at most SLOTS-1 groups
// pending" means "the slab used SLOTS calls ago is free".
//
// The tensor store writes whole 16-byte pieces of a row, so a chunk that
// crosses a right edge N not on a 16-byte boundary would also write the
// columns after N. That chunk is stored element by element from registers
// instead (rows past M skipped), leaving every byte outside C untouched.
// INT: the 4-byte values are int32 (an add is an integer add).
template <int SLAB_BYTES, int OUT_ES, int SLOTS, bool INT = false>
__device__ __forceinline__ void store_slab(const CUtensorMap* tmC, uint8_t* slab_pair, int& count,
                                           const uint32_t (&v)[32], int lane, int col0, int row0,
                                           const GemmParams& p, bool add = false) {
    constexpr int COLS = 128 / OUT_ES;
    const bool in_bounds = row0 < p.out_rows && col0 < p.N;
    if (in_bounds && col0 + COLS > p.N && (p.N * OUT_ES) % 16 != 0) {
        const int row = row0 + lane;
        if (row < p.out_rows) {
            const int n = p.N - col0;
            if constexpr (OUT_ES == 4) {
                uint32_t* dst = static_cast<uint32_t*>(p.C) + row * p.ldc + col0;
                if (add) {   // C += v, this warp being the only writer of these rows now
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (i < n)
                            dst[i] = INT ? dst[i] + v[i]
                                         : __float_as_uint(__uint_as_float(dst[i]) + __uint_as_float(v[i]));
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (i < n) dst[i] = v[i];
                }
            } else {
                uint16_t* dst = static_cast<uint16_t*>(p.C) + row * p.ldc + col0;
#pragma unroll
                for (int i = 0; i < 64; ++i)
                    if (i < n) dst[i] = static_cast<uint16_t>((i & 1) ? (v[i >> 1] >> 16) : (v[i >> 1] & 0xFFFFu));
            }
        }
        __syncwarp();
        if (lane == 0) ptx::bulk_commit();
        ++count;
        return;
    }
    uint8_t* slab = slab_pair + (count % SLOTS) * SLAB_BYTES;
    if (lane == 0) ptx::bulk_wait_read<SLOTS - 1>();
    __syncwarp();
    const uint32_t row_addr = ptx::smem_u32(slab) + lane * 128;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        st_shared_v4(row_addr + ((j ^ (lane & 7)) << 4), v[4 * j], v[4 * j + 1], v[4 * j + 2],
                     v[4 * j + 3]);
    }
    ptx::fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
        if (in_bounds) {
            if (add)
                ptx::tma_reduce_add_2d(tmC, ptx::smem_u32(slab), col0, row0);
            else
                ptx::tma_store_2d(tmC, ptx::smem_u32(slab), col0, row0);
        }
        ptx::bulk_commit();
    }
    ++count;
}

// Synchronous producer (the ablation's rung below TMA): the four producer
// warps copy each stage through registers — all 16-byte global loads of the
// stage first, then the stores into the same 128-byte-swizzled layout the TMA
// would have written — then make their shared-memory writes visible to the
// tensor core's (async) proxy and arrive on full[s]. Out-of-range rows,
// columns and K are written as zeros, as the TMA's fill would.
template <class C>
__device__ __forceinline__ void sync_producer(const GemmParams& p, uint8_t* stage_base, uint32_t full0,
                                              uint32_t empty0, volatile uint32_t* abort_flag, bool tracing) {
    constexpr int PT = 32 * C::P_WARPS;
    constexpr int A_PER = C::BM * 8 / PT;                  // 16-byte chunks per thread, A tile
    constexpr int B_PER = C::B_BOXES * C::BK * 8 / PT;     // and B tile
    static_assert(A_PER * PT == C::BM * 8 && B_PER * PT == C::B_BOXES * C::BK * 8, "chunk split");
    const int pt = threadIdx.x;
    const int lane = pt & 31;
    const uint16_t* Ag = static_cast<const uint16_t*>(p.A);
    const uint16_t* Bg = static_cast<const uint16_t*>(p.B);
    uint32_t it = 0;
    const int num_work = p.num_tiles * p.splits;
    for (int w = blockIdx.x; w < num_work; w += gridDim.x) {
        const Work wk = work_item(w, p);
        const int mb = wk.mb, nb = wk.nb;
        for (int kb = wk.kb_lo; kb < wk.kb_hi; ++kb, ++it) {
            const uint32_t s = it % C::STAGES;
            const uint32_t ph = (it / C::STAGES) & 1u;
            bool got = true;
            if (lane == 0)
                got = wait_bounded(empty0 + 8 * C::rel_slot(s), ph ^ 1u, abort_flag, p.timeout_ns, p.status,
                                   DEV_TIMEOUT_PRODUCER);
            if (__shfl_sync(0xffffffffu, got ? 1 : 0, 0) == 0) return;
            if (tracing && pt == 0) {
                const uint64_t now = ptx::clock64();
                if (it >= C::STAGES && it - C::STAGES < (uint32_t)p.trace_cap)
                    p.trace[4 * (it - C::STAGES) + 3] = now;
                if (it < (uint32_t)p.trace_cap) p.trace[4 * it + 0] = now;
            }
            const uint32_t sa = ptx::smem_u32(stage_base + s * C::STAGE_BYTES);
            const uint32_t sb = sa + C::A_BYTES;
            uint4 ra[A_PER], rb[B_PER];
#pragma unroll
            for (int i = 0; i < A_PER; ++i) {
                const int c = pt + i * PT, row = c >> 3, j = c & 7;
                const int gm = mb * C::BM + row, gk = kb * C::BK + j * 8;
                ra[i] = (gm < p.M && gk < p.K)
                            ? __ldg(reinterpret_cast<const uint4*>(Ag + static_cast<long long>(gm) * p.lda + gk))
                            : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int i = 0; i < B_PER; ++i) {
                const int c = pt + i * PT, box = c / (C::BK * 8), r = c % (C::BK * 8);
                const int k = r >> 3, j = r & 7;
                const int gk = kb * C::BK + k, gn = nb * C::BN + box * C::B_BOX_N + j * 8;
                const uint16_t* src = Bg + static_cast<long long>(gk) * p.ldb + gn;
                if (gk < p.K && gn + 8 <= p.N) {
                    rb[i] = __ldg(reinterpret_cast<const uint4*>(src));
                } else if (gk < p.K && gn < p.N) {
                    uint32_t w[4];
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        const uint32_t lo = gn + 2 * t < p.N ? src[2 * t] : 0u;
                        const uint32_t hi = gn + 2 * t + 1 < p.N ? src[2 * t + 1] : 0u;
                        w[t] = lo | (hi << 16);
                    }
                    rb[i] = make_uint4(w[0], w[1], w[2], w[3]);
                } else {
                    rb[i] = make_uint4(0, 0, 0, 0);
                }
            }
#pragma unroll
            for (int i = 0; i < A_PER; ++i) {
                const int c = pt + i * PT, row = c >> 3, j = c & 7;
                st_shared_v4(sa + row * 128 + ((j ^ (row & 7)) << 4), ra[i].x, ra[i].y, ra[i].z, ra[i].w);
            }
#pragma unroll
            for (int i = 0; i < B_PER; ++i) {
                const int c = pt + i * PT, box = c / (C::BK * 8), r = c % (C::BK * 8);
                const int k = r >> 3, j = r & 7;
                st_shared_v4(sb + box * C::B_BOX_BYTES + k * 128 + ((j ^ (k & 7)) << 4), rb[i].x, rb[i].y,
                             rb[i].z, rb[i].w);
            }
            ptx::fence_proxy_async_smem();   // generic-proxy writes -> visible to the tensor core
            ptx::mbar_arrive(full0 + 8 * s);
        }
    }
}

// Asynchronous-copy producer (the ablation's middle rung): the four producer
// warps issue one 16-byte cp.async per chunk of the stage, straight into the
// 128-byte-swizzled layout (no register staging), then each thread arms an
// arrival on full[s] that fires once all of its copies have landed, and moves
// on to the next stage without waiting. Out-of-range chunks copy zero bytes
// (zero fill); a chunk that straddles the right edge of B copies only its
// in-range columns. cp.async writes through the generic proxy, so the MMA warp
// fences toward the async proxy after it has seen full[s] complete.
template <class C>
__device__ __forceinline__ void cpasync_producer(const GemmParams& p, uint8_t* stage_base, uint32_t full0,
                                                 uint32_t empty0, volatile uint32_t* abort_flag, bool tracing) {
    constexpr int PT = 32 * C::P_WARPS;
    constexpr int A_PER = C::BM * 8 / PT;
    constexpr int B_PER = C::B_BOXES * C::BK * 8 / PT;
    static_assert(A_PER * PT == C::BM * 8 && B_PER * PT == C::B_BOXES * C::BK * 8, "chunk split");
    const int pt = threadIdx.x;
    const int lane = pt & 31;
    const uint16_t* Ag = static_cast<const uint16_t*>(p.A);
    const uint16_t* Bg = static_cast<const uint16_t*>(p.B);
    uint32_t it = 0;
    const int num_work = p.num_tiles * p.splits;
    for (int w = blockIdx.x; w < num_work; w += gridDim.x) {
        const Work wk = work_item(w, p);
        const int mb = wk.mb, nb = wk.nb;
        for (int kb = wk.kb_lo; kb < wk.kb_hi; ++kb, ++it) {
            const uint32_t s = it % C::STAGES;
            const uint32_t ph = (it / C::STAGES) & 1u;
            bool got = true;
            if (lane == 0)
                got = wait_bounded(empty0 + 8 * C::rel_slot(s), ph ^ 1u, abort_flag, p.timeout_ns, p.status,
                                   DEV_TIMEOUT_PRODUCER);
            if (__shfl_sync(0xffffffffu, got ? 1 : 0, 0) == 0) {
                ptx::cp_async_wait_all();   // nothing may still be writing when the CTA exits
                return;
            }
            if (tracing && pt == 0) {
                const uint64_t now = ptx::clock64();
                if (it >= C::STAGES && it - C::STAGES < (uint32_t)p.trace_cap)
                    p.trace[4 * (it - C::STAGES) + 3] = now;
                if (it < (uint32_t)p.trace_cap) p.trace[4 * it + 0] = now;
            }
            const uint32_t sa = ptx::smem_u32(stage_base + s * C::STAGE_BYTES);
            const uint32_t sb = sa + C::A_BYTES;
#pragma unroll
            for (int i = 0; i < A_PER; ++i) {
                const int c = pt + i * PT, row = c >> 3, j = c & 7;
                const int gm = mb * C::BM + row, gk = kb * C::BK + j * 8;
                const bool in = gm < p.M && gk < p.K;
                const uint16_t* src = in ? Ag + static_cast<long long>(gm) * p.lda + gk : Ag;
                ptx::cp_async_16(sa + row * 128 + ((j ^ (row & 7)) << 4), src, in ? 16u : 0u);
            }
#pragma unroll
            for (int i = 0; i < B_PER; ++i) {
                const int c = pt + i * PT, box = c / (C::BK * 8), r = c % (C::BK * 8);
                const int k = r >> 3, j = r & 7;
                const int gk = kb * C::BK + k, gn = nb * C::BN + box * C::B_BOX_N + j * 8;
                const bool in = gk < p.K && gn < p.N;
                const uint32_t bytes = in ? 2u * static_cast<uint32_t>(min(8, p.N - gn)) : 0u;
                const uint16_t* src = in ? Bg + static_cast<long long>(gk) * p.ldb + gn : Bg;
                ptx::cp_async_16(sb + box * C::B_BOX_BYTES + k * 128 + ((j ^ (k & 7)) << 4), src, bytes);
            }
            ptx::cp_async_arrive_noinc(full0 + 8 * s);
        }
    }
    ptx::cp_async_wait_all();
}

struct NoPace {
    __device__ __forceinline__ void operator()(int) const {}
};

// Drains one TMEM accumulator (this warp's 32 lanes × EPI_CHUNKS chunks) to C:
// F32 chunks are 32 fp32 columns, BF16 chunks 64 fp32 columns rounded to 64
// bf16. The TMEM load of chunk c+1 is issued before chunk c is staged and
// stored, so its latency hides under the shared-memory writes and the store
// issue. `release()` runs once every TMEM read of the accumulator is complete;
// `pace(c)` runs before chunk c is staged and stored (the two-SM kernel uses
// it to spread a tile's stores over the next tile's mainloop). `add`: reduce
// into C instead of storing (fp32). `pre`, if not null, is this warp's block of
// a stream-K workspace (column group g of lane l at pre[(g·32 + l)·4 ..]),
// added to the accumulator before the conversion.
template <OutKind OK, int EPI_CHUNKS, int SLAB_BYTES, int SLOTS, class Release, class Pace = NoPace>
__device__ __forceinline__ void drain_accumulator(const CUtensorMap* tmC, uint8_t* slab_pair, int& store_count,
                                                  uint32_t tbase, int lane, int col_base, int row0,
                                                  const GemmParams& p, Release release, bool add = false,
                                                  Pace pace = Pace(), const float* pre = nullptr) {
    constexpr int COLS = OK == OutKind::BF16 ? 64 : 32;   // TMEM columns per chunk
    constexpr int OUT_ES = OK == OutKind::BF16 ? 2 : 4;
    uint32_t buf[2][COLS];
    __syncwarp();   // tcgen05.ld is warp-collective
    ptx::tmem_ld_32x32b_x32(tbase, *reinterpret_cast<uint32_t(*)[32]>(&buf[0][0]));
    if constexpr (COLS == 64) ptx::tmem_ld_32x32b_x32(tbase + 32, *reinterpret_cast<uint32_t(*)[32]>(&buf[0][32]));
#pragma unroll
    for (int c = 0; c < EPI_CHUNKS; ++c) {
        uint32_t(&cur)[COLS] = buf[c & 1];
        ptx::tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(&cur[0]));
        if constexpr (COLS == 64) ptx::tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(&cur[32]));
        if (c + 1 < EPI_CHUNKS) {
            uint32_t(&nxt)[COLS] = buf[(c + 1) & 1];
            __syncwarp();
            ptx::tmem_ld_32x32b_x32(tbase + (c + 1) * COLS, *reinterpret_cast<uint32_t(*)[32]>(&nxt[0]));
            if constexpr (COLS == 64)
                ptx::tmem_ld_32x32b_x32(tbase + (c + 1) * COLS + 32, *reinterpret_cast<uint32_t(*)[32]>(&nxt[32]));
        } else {
            release();
        }
        if (pre) {
            // (read at L2: another SM wrote the block in this launch)
            const float4* src = reinterpret_cast<const float4*>(pre) + c * (COLS / 4) * 32 + lane;
#pragma unroll
            for (int j = 0; j < COLS / 4; ++j) {
                const float4 w = __ldcg(src + j * 32);
                cur[4 * j + 0] = __float_as_uint(__uint_as_float(cur[4 * j + 0]) + w.x);
                cur[4 * j + 1] = __float_as_uint(__uint_as_float(cur[4 * j + 1]) + w.y);
                cur[4 * j + 2] = __float_as_uint(__uint_as_float(cur[4 * j + 2]) + w.z);
                cur[4 * j + 3] = __float_as_uint(__uint_as_float(cur[4 * j + 3]) + w.w);
            }
        }
        uint32_t v[32];
        if constexpr (OK == OutKind::BF16) {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                __nv_bfloat162 t = __floats2bfloat162_rn(__uint_as_float(cur[2 * i]), __uint_as_float(cur[2 * i + 1]));
                v[i] = *reinterpret_cast<uint32_t*>(&t);
            }
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = cur[i];
        }
        pace(c);
        store_slab<SLAB_BYTES, OUT_ES, SLOTS>(tmC, slab_pair, store_count, v, lane, col_base + c * (128 / OUT_ES),
                                              row0, p, add);
    }
}

// Drains one TMEM accumulator (this warp's 32 lanes × 32·EPI_CHUNKS fp32 columns)
// into its block of a stream-K workspace (the layout `pre` of drain_accumulator
// reads), with plain 16-byte stores straight from registers: each store of the
// warp covers 512 contiguous bytes. `add`: add the block's values first (an
// earlier piece wrote them). `release()` as in drain_accumulator.
template <int EPI_CHUNKS, class Release>
__device__ __forceinline__ void drain_to_workspace(uint32_t tbase, int lane, float* blk, Release release,
                                                   bool add) {
    uint32_t buf[2][32];
    __syncwarp();   // tcgen05.ld is warp-collective
    ptx::tmem_ld_32x32b_x32(tbase, buf[0]);
#pragma unroll
    for (int c = 0; c < EPI_CHUNKS; ++c) {
        uint32_t(&cur)[32] = buf[c & 1];
        ptx::tmem_ld_wait(cur);
        if (c + 1 < EPI_CHUNKS) {
            __syncwarp();
            ptx::tmem_ld_32x32b_x32(tbase + (c + 1) * 32, buf[(c + 1) & 1]);
        } else {
            release();
        }
        float4* dst = reinterpret_cast<float4*>(blk) + c * 8 * 32 + lane;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            float4 v = make_float4(__uint_as_float(cur[4 * j]), __uint_as_float(cur[4 * j + 1]),
                                   __uint_as_float(cur[4 * j + 2]), __uint_as_float(cur[4 * j + 3]));
            if (add) {
                const float4 w = __ldcg(dst + j * 32);
                v.x += w.x;
                v.y += w.y;
                v.z += w.z;
                v.w += w.w;
            }
            __stcg(dst + j * 32, v);
        }
    }
}

template <InKind IK, OutKind OK, int BN, int STAGES, int PROD>
__global__ void __launch_bounds__(KCfg<IK, OK, BN, STAGES, PROD>::THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC, const GemmParams p) {
    using C = KCfg<IK, OK, BN, STAGES, PROD>;
    extern __shared__ uint8_t smem_raw[];
    // 128-byte swizzle atoms must sit on 1024-byte boundaries of the shared window.
    const uint32_t raw_addr = ptx::smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
    uint8_t* stage_base = smem;
    uint8_t* staging = smem + STAGES * C::STAGE_BYTES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(staging + C::STAGING_BYTES);
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 5);
    volatile uint32_t* abort_flag = tmem_holder + 1;

    const uint32_t full0 = ptx::smem_u32(bars);
    const uint32_t empty0 = ptx::smem_u32(bars + STAGES);
    const uint32_t accf0 = ptx::smem_u32(bars + 2 * STAGES);
    const uint32_t acce0 = ptx::smem_u32(bars + 2 * STAGES + 2);
    const uint32_t drain_bar = ptx::smem_u32(bars + 2 * STAGES + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(full0 + 8 * s, C::FULL_ARRIVALS);
            ptx::mbar_init(empty0 + 8 * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(accf0 + 8 * b, 1);
            ptx::mbar_init(acce0 + 8 * b, 4);
        }
        ptx::mbar_init(drain_bar, 1);
        *abort_flag = 0u;
        ptx::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tensormap(&tmA);
        ptx::prefetch_tensormap(&tmB);
        ptx::prefetch_tensormap(&tmC);
    }
    if (warp == C::MMA_WARP) {
        ptx::tmem_alloc(ptx::smem_u32(tmem_holder), C::TMEM_COLS);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    // Set-up above touches only this CTA's own resources: under a programmatic
    // launch it overlaps the previous kernel's tail; global memory only from here.
    ptx::griddep_wait();
    ptx::griddep_launch_dependents();
    const bool tracing = (p.trace != nullptr) && (blockIdx.x == 0);
    if (tracing && threadIdx.x == 0) {   // SM clock and wall clock at the start of CTA 0's work
        p.trace[4 * p.trace_cap + 0] = ptx::clock64();
        p.trace[4 * p.trace_cap + 1] = ptx::globaltimer_ns();
    }

    if (warp < C::P_WARPS && PROD == PROD_SYNC) {
        // ------------------------------------------------ producer (synchronous, ablation)
        sync_producer<C>(p, stage_base, full0, empty0, abort_flag, tracing);
    } else if (warp < C::P_WARPS && PROD == PROD_CPASYNC) {
        // ------------------------------------------------ producer (cp.async, ablation)
        cpasync_producer<C>(p, stage_base, full0, empty0, abort_flag, tracing);
    } else if (warp == 0) {
        // ------------------------------------------------ producer (TMA)
        // All 32 lanes run the loop; the arrival and the copies come from one
        // elected lane.
        uint32_t it = 0;
        bool ok = true;
        const int num_work = p.num_tiles * p.splits;
        for (int w = blockIdx.x, pos = 0; ok && w < num_work; w += gridDim.x, ++pos) {
            const Work wk = work_item(w, p);
            const int mb = wk.mb, nb = wk.nb;
            for (int kb = wk.kb_lo; kb < wk.kb_hi; ++kb, ++it) {
                const uint32_t s = it % STAGES;
                const uint32_t ph = (it / STAGES) & 1u;
                const int kc = load_kblock(p, pos, kb, wk.kb_lo, wk.kb_hi);
                if (!wait_warp(empty0 + 8 * C::rel_slot(s), ph ^ 1u, abort_flag, p.timeout_ns, p.status,
                               DEV_TIMEOUT_PRODUCER)) {
                    ok = false;
                    break;
                }
                if (tracing && lane == 0) {
                    const uint64_t now = ptx::clock64();
                    if (it >= STAGES && it - STAGES < (uint32_t)p.trace_cap)
                        p.trace[4 * (it - STAGES) + 3] = now;   // MMA of block it-STAGES done
                    if (it < (uint32_t)p.trace_cap) p.trace[4 * it + 0] = now;   // load issued
                }
                const uint32_t full = full0 + 8 * s;
                const uint32_t sa = ptx::smem_u32(stage_base + s * C::STAGE_BYTES);
                if (blockIdx.x == 0 && static_cast<int>(it) == p.debug_skip_kb) continue;
                ptx::mbar_arrive_expect_tx_elected(full, C::STAGE_BYTES);
                ptx::tma_load_2d_elected(sa, &tmA, full, kc * C::BK, mb * C::BM);
                if (p.b_3d) {   // all B_BOXES boxes in one copy (B_BOX_BYTES apart, as below)
                    ptx::tma_load_3d_elected(sa + C::A_BYTES, &tmB, full, 0, kc * C::BK, nb * BN / C::B_BOX_N);
                } else {
#pragma unroll
                    for (int b = 0; b < C::B_BOXES; ++b) {
                        ptx::tma_load_2d_elected(sa + C::A_BYTES + b * C::B_BOX_BYTES, &tmB, full,
                                                 nb * BN + b * C::B_BOX_N, kc * C::BK);
                    }
                }
            }
        }
        if (!ok && lane == 0) {
            // Let every load still in flight land before the CTA can exit.
            const uint32_t first = it > (uint32_t)STAGES ? it - STAGES : 0u;
            for (uint32_t j = first; j < it; ++j)
                wait_drain(full0 + 8 * (j % STAGES), (j / STAGES) & 1u, p.timeout_ns);
        }
        if (ok && tracing && lane == 0) {
            // The last STAGES k-blocks' stages are never reused, so the loop above never
            // saw their MMAs finish: wait (bounded) for the same empty-barrier phases a
            // reuse would have waited for, and stamp them.
            const uint32_t first = it > (uint32_t)STAGES ? it - STAGES : 0u;
            for (uint32_t j = first; j < it && j < (uint32_t)p.trace_cap && !*abort_flag; ++j) {
                wait_drain(empty0 + 8 * C::rel_slot(j % STAGES), (j / STAGES) & 1u, p.timeout_ns);
                p.trace[4 * j + 3] = ptx::clock64();
            }
        }
        __syncwarp();
    } else if (warp == C::MMA_WARP) {
        // ------------------------------------------------ MMA issuer
        // All 32 lanes run this loop (uniform control flow, no parked lanes);
        // each k-block's four MMAs and its commit come from one elected lane
        // through predicates. The issuing thread's loop, not the tensor pipe,
        // would otherwise set the pace.
        static_assert(C::KSUB == 4, "four MMAs per k-block");
        // Descriptors of stage 0; a stage and a k-slice are fixed offsets (in
        // 16-byte units) in the start-address field.
        const uint32_t stage0 = ptx::smem_u32(stage_base);
        const uint64_t adesc0 = ptx::sdesc_sw128(stage0, 16, 1024);
        // B N-major: boxes B_BOX_BYTES apart (the leading offset), core groups of K-rows
        // B_SBO apart; a k-slice steps UMMA_K rows of 128 B
        const uint64_t bdesc0 = ptx::sdesc(stage0 + C::A_BYTES, C::B_BOX_BYTES, InTraits<IK>::B_SBO,
                                           InTraits<IK>::B_LAYOUT);
        constexpr uint64_t A_STEP = C::UMMA_K * C::ES / 16;
        constexpr uint64_t B_STEP = C::UMMA_K * 128 / 16;
        constexpr uint64_t S_STEP = C::STAGE_BYTES / 16;
        uint32_t it = 0, unit = 0, s = 0, ph = 0;   // (s, ph): ring slot and phase of k-block `it`
        bool ok = true;
        const int num_work = p.num_tiles * p.splits;
        for (int w = blockIdx.x; ok && w < num_work; w += gridDim.x) {
            const Work wk = work_item(w, p);
            for (int kb0 = wk.kb_lo; kb0 < wk.kb_hi; kb0 += p.kb_per_unit, ++unit) {
                const uint32_t buf = unit & 1u;
                const uint32_t uph = (unit >> 1) & 1u;
                if (!wait_warp(acce0 + 8 * buf, uph ^ 1u, abort_flag, p.timeout_ns, p.status, DEV_TIMEOUT_MMA_ACC)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t d_tmem = tmem_base + buf * BN;
                const int kb1 = min(kb0 + p.kb_per_unit, wk.kb_hi);
                for (int kb = kb0; kb < kb1; ++kb, ++it) {
                    if (!wait_warp(full0 + 8 * s, ph, abort_flag, p.timeout_ns, p.status, DEV_TIMEOUT_MMA_FULL)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    // cp.async data arrived through the generic proxy: order it before the MMA's reads
                    if constexpr (PROD == PROD_CPASYNC) ptx::fence_proxy_async_smem();
                    if (tracing && lane == 0 && it < (uint32_t)p.trace_cap) p.trace[4 * it + 1] = ptx::clock64();
                    // A: K-major rows of 128 B, a k-slice steps UMMA_K elements along the row.
                    // B N-major: a k-slice steps UMMA_K rows of 128 B (boxes B_BOX_BYTES apart,
                    // the descriptor's leading offset).
                    const uint64_t ad = adesc0 + s * S_STEP;
                    const uint64_t bd = bdesc0 + s * S_STEP;
                    const uint32_t acc = kb > kb0 ? 1u : 0u;
                    if constexpr (IK == InKind::TF32)
                        ptx::mma_tf32_x4_elected(d_tmem, ad, bd, ad + A_STEP, bd + B_STEP, ad + 2 * A_STEP,
                                                 bd + 2 * B_STEP, ad + 3 * A_STEP, bd + 3 * B_STEP, C::IDESC, acc);
                    else
                        ptx::mma_f16_x4_elected(d_tmem, ad, bd, ad + A_STEP, bd + B_STEP, ad + 2 * A_STEP,
                                                bd + 2 * B_STEP, ad + 3 * A_STEP, bd + 3 * B_STEP, C::IDESC, acc);
                    // stage s (and, released in pairs, s - 1) free once these MMAs finish
                    if (C::REL == 1 || (s & 1u)) ptx::mma_commit_elected(empty0 + 8 * s);
                    if (tracing && lane == 0 && it < (uint32_t)p.trace_cap) p.trace[4 * it + 2] = ptx::clock64();
                    const uint32_t wrap = (s + 1 == static_cast<uint32_t>(STAGES)) ? 1u : 0u;
                    s = wrap ? 0u : s + 1;
                    ph ^= wrap;
                }
                if (!ok) break;
                ptx::mma_commit_elected(accf0 + 8 * buf);      // accumulator ready for the epilogue
            }
        }
        if (ok && tracing && C::REL == 2 && it > 0) {
            // slots are released in pairs: if the last k-block sat in an even slot, no commit
            // releases it; one more lets the producer's trace see its MMAs finish
            const uint32_t last = (s + STAGES - 1) % STAGES;
            if (!(last & 1u)) ptx::mma_commit_elected(empty0 + 8 * (last | 1u));
        }
        if (!ok) {
            ptx::mma_commit_elected(drain_bar);
            if (lane == 0) wait_drain(drain_bar, 0, p.timeout_ns);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ epilogue (four warps)
        const int q = warp & 3;   // TMEM lane quarter this warp may read
        uint8_t* slab_pair = staging + (warp - C::EPI_WARP0) * C::EPI_SLOTS * C::SLAB_BYTES;
        int store_count = 0;
        uint32_t unit = 0;
        bool ok = true;
        const int num_work = p.num_tiles * p.splits;
        for (int w = blockIdx.x; ok && w < num_work; w += gridDim.x) {
            const Work wk = work_item(w, p);
            const int nb = wk.nb;
            const int row0 = wk.row_base + wk.mb * C::BM + q * 32;
            [[maybe_unused]] int32_t iacc[(OK == OutKind::S32) ? BN : 1];
            if constexpr (OK == OutKind::S32) {
#pragma unroll
                for (int i = 0; i < BN; ++i) iacc[i] = 0;
            }
            for (int kb0 = wk.kb_lo; kb0 < wk.kb_hi; kb0 += p.kb_per_unit, ++unit) {
                const uint32_t buf = unit & 1u;
                const uint32_t uph = (unit >> 1) & 1u;
                bool got = true;
                if (lane == 0)
                    got = wait_bounded(accf0 + 8 * buf, uph, abort_flag, p.timeout_ns, p.status,
                                       DEV_TIMEOUT_EPILOGUE);
                got = __shfl_sync(0xffffffffu, got ? 1 : 0, 0) != 0;
                if (!got) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + buf * BN;
                if constexpr (OK == OutKind::S32) {
#pragma unroll
                    for (int c = 0; c < BN / 32; ++c) {
                        __syncwarp();   // tcgen05.ld is warp-collective
                        uint32_t r[32];
                        ptx::tmem_ld_32x32b_x32(tbase + c * 32, r);
                        ptx::tmem_ld_wait(r);
#pragma unroll
                        for (int i = 0; i < 32; ++i) iacc[c * 32 + i] += __float2int_rn(__uint_as_float(r[i]));
                    }
                    ptx::tc_fence_before();
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive_relaxed(acce0 + 8 * buf);
                    if (kb0 + p.kb_per_unit >= wk.kb_hi) {
#pragma unroll
                        for (int c = 0; c < BN / 32; ++c) {
                            const uint32_t(&v)[32] =
                                *reinterpret_cast<const uint32_t(*)[32]>(&iacc[c * 32]);
                            const int col0 = nb * BN + c * 32;
                            store_slab<C::SLAB_BYTES, C::OUT_ES, C::EPI_SLOTS>(&tmC, slab_pair, store_count, v, lane,
                                                                 col0, row0, p);
                        }
                    }
                } else {
                    drain_accumulator<OK, C::EPI_CHUNKS, C::SLAB_BYTES, C::EPI_SLOTS>(
                        &tmC, slab_pair, store_count, tbase, lane, nb * BN, row0, p, [&]() {
                            // all of this unit's TMEM columns are in registers: free the accumulator
                            ptx::tc_fence_before();
                            __syncwarp();
                            if (lane == 0) ptx::mbar_arrive_relaxed(acce0 + 8 * buf);
                        });
                }
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
    if (warp == C::MMA_WARP) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

}  // namespace tcl
