// Inline-PTX building blocks for sm_103a: mbarriers, TMA bulk-tensor copies,
// tcgen05 MMA / TMEM, async-proxy fences and timers.
//
// Each wrapper is one PTX instruction (or a tiny fixed sequence) written from
// the PTX ISA's description of that instruction. Nothing here knows about GEMM
// tiling; the kernel in gemm_kernel.cuh composes them.
#pragma once

#include <cstdint>
#include <cuda.h>

namespace tcl {
namespace ptx {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Index of the SM this thread runs on (two consecutive ids are the two SMs of a pair).
__device__ __forceinline__ uint32_t smid() {
    uint32_t s;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(s));
    return s;
}

__device__ __forceinline__ uint64_t clock64() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%clock64;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Makes the initialised barriers visible to the async proxy (TMA, tcgen05).
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// True once the phase with the given parity has completed.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// The same with acquire semantics at cluster scope: for a barrier on which
// threads of the other CTA of the pair arrive with release semantics.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// ---------------------------------------------------------------- TMA
// 2-D tiled load of one box into shared memory; completion is signalled on
// `bar` as transaction bytes. c0 is the innermost (contiguous) coordinate.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int32_t c0, int32_t c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1)
        : "memory");
}

// 2-D tiled store of one box from shared memory (bulk-group completion).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int32_t c0,
                                             int32_t c1) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(src), "r"(c0), "r"(c1)
                 : "memory");
}

// 2-D tiled reduction shared -> global: adds the shared-memory tile (fp32 for
// an fp32 tensor map) element by element into the global tile, in the L2.
// Completion and read-out are tracked by bulk groups like a store.
__device__ __forceinline__ void tma_reduce_add_2d(const CUtensorMap* map, uint32_t src, int32_t c0, int32_t c1) {
    asm volatile("cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(src), "r"(c0), "r"(c1)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Wait until at most N committed bulk groups still read their shared source.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Wait until at most N committed bulk groups are still in flight.
template <int N>
__device__ __forceinline__ void bulk_wait() {
    asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// Non-bulk asynchronous copy of 16 bytes global -> shared, bypassing L1. Only
// the first `src_bytes` (0..16) are read; the rest of the 16 bytes are written
// as zeros. Both addresses must be 16-byte aligned.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
                 : "memory");
}

// Arrive on the mbarrier once every cp.async this thread issued so far has
// landed. `noinc`: the arrival counts against the barrier's expected count.
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// A hint to the copy engine: bring `bytes` (a multiple of 16) of global memory
// starting at the 16-byte aligned `p` into L2. It moves no data anywhere else
// and orders nothing.
__device__ __forceinline__ void prefetch_l2_bulk(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(p)), "r"(bytes)
                 : "memory");
}

// Programmatic dependent launch. wait: block until the grids this one depends
// on in the stream have completed and their memory is visible (a no-op when
// the launch did not ask for programmatic serialisation). launch_dependents:
// let the next grid in the stream be scheduled (it still waits for this one
// before it reads anything).
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Orders this thread's view of global memory between the generic proxy and
// the async proxy (TMA stores/reductions), in both directions.
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

// GPU-scope acquire load and release store of a 32-bit flag in global memory.
__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release_gpu(uint32_t* p, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Orders generic-proxy shared-memory writes before later async-proxy reads
// (a TMA store or an MMA reading what threads wrote with st.shared).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Named barrier over `count` threads (count a multiple of 32).
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// ---------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem desc] · B[smem desc], bf16/f16 operands, one thread issues.
__device__ __forceinline__ void mma_f16_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                           uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Same with TF32 operands (fp32 storage, 10 explicit mantissa bits consumed).
__device__ __forceinline__ void mma_tf32_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                            uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on `bar` when every tcgen05 operation this thread issued so far is done.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}

// Each thread of the warp reads 32 consecutive 32-bit columns of its own TMEM lane.
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

// Each thread of the warp reads 16 consecutive 32-bit columns of its own TMEM lane.
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait(uint32_t (&r)[16]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                   "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                   "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
                 :
                 : "memory");
}

// Completes the thread's outstanding tcgen05.ld. The registers are threaded
// through as read-write operands so that no use of them can be scheduled
// before the wait.
__device__ __forceinline__ void tmem_ld_wait(uint32_t (&r)[32]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                   "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                   "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]),
                   "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
                   "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
                   "+r"(r[30]), "+r"(r[31])
                 :
                 : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ---------------------------------------------------------------- converged single-lane issue
// The MMA warp runs its loop on all 32 lanes (no divergence, uniform branches);
// these issue from one elected lane through a predicate instead of a branch.

// One k-block: four MMAs on consecutive k-slices (descriptors a0..a3 / b0..b3)
// into the same accumulator; the first takes `acc` (0 = overwrite), the rest
// accumulate. Issued by the warp's elected lane only.
__device__ __forceinline__ void mma_f16_x4_elected(uint32_t d, uint64_t a0, uint64_t b0, uint64_t a1, uint64_t b1,
                                                   uint64_t a2, uint64_t b2, uint64_t a3, uint64_t b3,
                                                   uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred el, p0, pt;\n\t.reg .b32 lane_sel;\n\t"
        "elect.sync lane_sel|el, 0xffffffff;\n\t"
        "setp.ne.b32 p0, %10, 0;\n\t"
        "setp.eq.b32 pt, 0, 0;\n\t"
        "@el tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %9, p0;\n\t"
        "@el tcgen05.mma.cta_group::1.kind::f16 [%0], %3, %4, %9, pt;\n\t"
        "@el tcgen05.mma.cta_group::1.kind::f16 [%0], %5, %6, %9, pt;\n\t"
        "@el tcgen05.mma.cta_group::1.kind::f16 [%0], %7, %8, %9, pt;\n\t}" ::"r"(d),
        "l"(a0), "l"(b0), "l"(a1), "l"(b1), "l"(a2), "l"(b2), "l"(a3), "l"(b3), "r"(idesc), "r"(acc)
        : "memory");
}

__device__ __forceinline__ void mma_tf32_x4_elected(uint32_t d, uint64_t a0, uint64_t b0, uint64_t a1, uint64_t b1,
                                                    uint64_t a2, uint64_t b2, uint64_t a3, uint64_t b3,
                                                    uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred el, p0, pt;\n\t.reg .b32 lane_sel;\n\t"
        "elect.sync lane_sel|el, 0xffffffff;\n\t"
        "setp.ne.b32 p0, %10, 0;\n\t"
        "setp.eq.b32 pt, 0, 0;\n\t"
        "@el tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %9, p0;\n\t"
        "@el tcgen05.mma.cta_group::1.kind::tf32 [%0], %3, %4, %9, pt;\n\t"
        "@el tcgen05.mma.cta_group::1.kind::tf32 [%0], %5, %6, %9, pt;\n\t"
        "@el tcgen05.mma.cta_group::1.kind::tf32 [%0], %7, %8, %9, pt;\n\t}" ::"r"(d),
        "l"(a0), "l"(b0), "l"(a1), "l"(b1), "l"(a2), "l"(b2), "l"(a3), "l"(b3), "r"(idesc), "r"(acc)
        : "memory");
}

__device__ __forceinline__ void mma_f16_pair_x4_elected(uint32_t d, uint64_t a0, uint64_t b0, uint64_t a1,
                                                        uint64_t b1, uint64_t a2, uint64_t b2, uint64_t a3,
                                                        uint64_t b3, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred el, p0, pt;\n\t.reg .b32 lane_sel;\n\t"
        "elect.sync lane_sel|el, 0xffffffff;\n\t"
        "setp.ne.b32 p0, %10, 0;\n\t"
        "setp.eq.b32 pt, 0, 0;\n\t"
        "@el tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %9, p0;\n\t"
        "@el tcgen05.mma.cta_group::2.kind::f16 [%0], %3, %4, %9, pt;\n\t"
        "@el tcgen05.mma.cta_group::2.kind::f16 [%0], %5, %6, %9, pt;\n\t"
        "@el tcgen05.mma.cta_group::2.kind::f16 [%0], %7, %8, %9, pt;\n\t}" ::"r"(d),
        "l"(a0), "l"(b0), "l"(a1), "l"(b1), "l"(a2), "l"(b2), "l"(a3), "l"(b3), "r"(idesc), "r"(acc)
        : "memory");
}

__device__ __forceinline__ void mma_tf32_pair_x4_elected(uint32_t d, uint64_t a0, uint64_t b0, uint64_t a1,
                                                         uint64_t b1, uint64_t a2, uint64_t b2, uint64_t a3,
                                                         uint64_t b3, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred el, p0, pt;\n\t.reg .b32 lane_sel;\n\t"
        "elect.sync lane_sel|el, 0xffffffff;\n\t"
        "setp.ne.b32 p0, %10, 0;\n\t"
        "setp.eq.b32 pt, 0, 0;\n\t"
        "@el tcgen05.mma.cta_group::2.kind::tf32 [%0], %1, %2, %9, p0;\n\t"
        "@el tcgen05.mma.cta_group::2.kind::tf32 [%0], %3, %4, %9, pt;\n\t"
        "@el tcgen05.mma.cta_group::2.kind::tf32 [%0], %5, %6, %9, pt;\n\t"
        "@el tcgen05.mma.cta_group::2.kind::tf32 [%0], %7, %8, %9, pt;\n\t}" ::"r"(d),
        "l"(a0), "l"(b0), "l"(a1), "l"(b1), "l"(a2), "l"(b2), "l"(a3), "l"(b3), "r"(idesc), "r"(acc)
        : "memory");
}

// tcgen05.commit from the elected lane (the same lane that issued the MMAs).
__device__ __forceinline__ void mma_commit_elected(uint32_t bar) {
    asm volatile(
        "{\n\t.reg .pred el;\n\t.reg .b32 lane_sel;\n\t"
        "elect.sync lane_sel|el, 0xffffffff;\n\t"
        "@el tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar)
        : "memory");
}

__device__ __forceinline__ void mma_commit_pair_multicast_elected(uint32_t bar, uint16_t mask) {
    asm volatile(
        "{\n\t.reg .pred el;\n\t.reg .b32 lane_sel;\n\t"
        "elect.sync lane_sel|el, 0xffffffff;\n\t"
        "@el tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;\n\t}" ::"r"(
            bar),
        "h"(mask)
        : "memory");
}

// Elected-lane forms of the producer's operations (one arrival, one copy per warp).
__device__ __forceinline__ void mbar_arrive_expect_tx_elected(uint32_t bar, uint32_t bytes) {
    asm volatile(
        "{\n\t.reg .pred el;\n\t.reg .b32 lane_sel;\n\t"
        "elect.sync lane_sel|el, 0xffffffff;\n\t"
        "@el mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n\t}" ::"r"(bar),
        "r"(bytes)
        : "memory");
}

__device__ __forceinline__ void tma_load_2d_elected(uint32_t dst, const CUtensorMap* map, uint32_t bar, int32_t c0,
                                                    int32_t c1) {
    asm volatile(
        "{\n\t.reg .pred el;\n\t.reg .b32 lane_sel;\n\t"
        "elect.sync lane_sel|el, 0xffffffff;\n\t"
        "@el cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];\n\t}" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1)
        : "memory");
}

// 3-D tiled load (coordinates innermost first), issued by one elected lane.
__device__ __forceinline__ void tma_load_3d_elected(uint32_t dst, const CUtensorMap* map, uint32_t bar, int32_t c0,
                                                    int32_t c1, int32_t c2) {
    asm volatile(
        "{\n\t.reg .pred el;\n\t.reg .b32 lane_sel;\n\t"
        "elect.sync lane_sel|el, 0xffffffff;\n\t"
        "@el cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];\n\t}" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

__device__ __forceinline__ void tma_load_2d_pair_elected(uint32_t dst, const CUtensorMap* map, uint32_t bar_cluster,
                                                         int32_t c0, int32_t c1) {
    asm volatile(
        "{\n\t.reg .pred el;\n\t.reg .b32 lane_sel;\n\t"
        "elect.sync lane_sel|el, 0xffffffff;\n\t"
        "@el cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];\n\t}" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(c0), "r"(c1)
        : "memory");
}

// 3-D form of the same (coordinates innermost first).
__device__ __forceinline__ void tma_load_3d_pair_elected(uint32_t dst, const CUtensorMap* map, uint32_t bar_cluster,
                                                         int32_t c0, int32_t c1, int32_t c2) {
    asm volatile(
        "{\n\t.reg .pred el;\n\t.reg .b32 lane_sel;\n\t"
        "elect.sync lane_sel|el, 0xffffffff;\n\t"
        "@el cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];\n\t}" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

// L2 eviction-priority policies (for whole lines) that tensor loads can carry
__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// The pair loads above with an L2 eviction-priority policy.
__device__ __forceinline__ void tma_load_2d_pair_hint(uint32_t dst, const CUtensorMap* map, uint32_t bar_cluster,
                                                      int32_t c0, int32_t c1, uint64_t pol) {
    asm volatile(
        "{\n\t.reg .pred el;\n\t.reg .b32 lane_sel;\n\t"
        "elect.sync lane_sel|el, 0xffffffff;\n\t"
        "@el cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4}], [%2], %5;\n\t}" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(c0), "r"(c1), "l"(pol)
        : "memory");
}
__device__ __forceinline__ void tma_load_3d_pair_hint(uint32_t dst, const CUtensorMap* map, uint32_t bar_cluster,
                                                      int32_t c0, int32_t c1, int32_t c2, uint64_t pol) {
    asm volatile(
        "{\n\t.reg .pred el;\n\t.reg .b32 lane_sel;\n\t"
        "elect.sync lane_sel|el, 0xffffffff;\n\t"
        "@el cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4, %5}], [%2], %6;\n\t}" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(c0), "r"(c1), "r"(c2), "l"(pol)
        : "memory");
}
__device__ __forceinline__ void tma_load_4d_pair_hint(uint32_t dst, const CUtensorMap* map, uint32_t bar_cluster,
                                                      int32_t c0, int32_t c1, int32_t c2, int32_t c3, uint64_t pol) {
    asm volatile(
        "{\n\t.reg .pred el;\n\t.reg .b32 lane_sel;\n\t"
        "elect.sync lane_sel|el, 0xffffffff;\n\t"
        "@el cp.async.bulk.tensor.4d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4, %5, %6}], [%2], %7;\n\t}" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "l"(pol)
        : "memory");
}

// 4-D form of the same (coordinates innermost first).
__device__ __forceinline__ void tma_load_4d_pair_elected(uint32_t dst, const CUtensorMap* map, uint32_t bar_cluster,
                                                         int32_t c0, int32_t c1, int32_t c2, int32_t c3) {
    asm volatile(
        "{\n\t.reg .pred el;\n\t.reg .b32 lane_sel;\n\t"
        "elect.sync lane_sel|el, 0xffffffff;\n\t"
        "@el cp.async.bulk.tensor.4d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6}], [%2];\n\t}" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
        : "memory");
}

// Per-warp register budget changes (all warps of a warpgroup execute the same
// one): dec releases registers down to N per thread, inc waits until N per
// thread can be granted from what the block's warps released.
template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_dec() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_inc() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

// Bulk copy of `bytes` (a multiple of 16) from this CTA's shared memory to the
// shared memory of a CTA of the cluster (shared::cluster addresses for the
// destination and its mbarrier), completed there as transaction bytes on that
// mbarrier. Asynchronous: the issuing thread does not wait.
__device__ __forceinline__ void bulk_copy_to_cluster(uint32_t dst_cluster, uint32_t src, uint32_t bytes,
                                                     uint32_t bar_cluster) {
    asm volatile(
        "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            dst_cluster),
        "r"(src), "r"(bytes), "r"(bar_cluster)
        : "memory");
}

// ---------------------------------------------------------------- clusters / CTA pairs
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// shared::cluster address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

// Every thread of every CTA in the cluster arrives and waits (release/acquire).
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Arrive once on an mbarrier given by its shared::cluster address (may be another CTA's).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// Arrivals that order nothing but what precedes them in this thread's program:
// an accumulator release, whose TMEM reads are complete at tcgen05.wait::ld.
// (The default release arrive would also wait until the thread's earlier global
// and local stores are performed: measured on GB300 at about 1,500 cycles per
// arrival in an epilogue that had spilled registers to local memory.)
__device__ __forceinline__ void mbar_arrive_relaxed(uint32_t bar) {
    asm volatile("mbarrier.arrive.relaxed.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_cluster_relaxed(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// 16-byte load from another CTA's shared memory (shared::cluster address).
__device__ __forceinline__ uint4 ld_cluster_v4(uint32_t cluster_addr) {
    uint4 v;
    asm volatile("ld.shared::cluster.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(cluster_addr)
                 : "memory");
    return v;
}

__device__ __forceinline__ void st_cluster_u32(uint32_t cluster_addr, uint32_t v) {
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}

// 2-D tiled load into this CTA's shared memory whose completion is counted on
// an mbarrier that may live in the peer CTA of the pair (shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar_cluster,
                                                 int32_t c0, int32_t c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(c0), "r"(c1)
        : "memory");
}

// Pair-wide TMEM management: one warp in each CTA of the pair executes these.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

// Pair MMA (issued by the even CTA only): D (M=256 split over the two SMs'
// TMEM) (+)= A (each SM's own 128 rows) · B (each SM's half of N).
__device__ __forceinline__ void mma_f16_ss_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                                uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on the mbarrier at this shared offset in every CTA of `mask`
// when the pair MMAs issued so far by this thread are done.
__device__ __forceinline__ void mma_commit_pair_multicast(uint32_t bar, uint16_t mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            bar),
        "h"(mask)
        : "memory");
}

// ---------------------------------------------------------------- descriptors
// Shared-memory matrix descriptor (tcgen05 format): start address, leading-
// and stride-dimension byte offsets (all in 16-byte units), the fixed version
// field 0b001 at bits 46-48, base offset 0 (atoms are 1024-byte aligned) and
// the layout type at bits 61-63: 2 = 128-byte swizzle (16-byte units permuted
// within each 128-byte row, pattern repeating every 8 rows), 1 = 128-byte
// swizzle with 32-byte atoms (32-byte units permuted, the form the tensor core
// reads 32-bit MN-major operands in: measured on GB300, a TF32 B stored N-major
// is read correctly only in this form, with core groups of 4 K-rows).
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes, uint32_t layout) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(layout & 7u) << 61;
    return d;
}

__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
    return sdesc(saddr, lbo_bytes, sbo_bytes, 2u);
}

// Instruction descriptor for kind::f16 / kind::tf32 (dense):
//   bits 4-5 D format (1 = f32), 7-9 A format, 10-12 B format
//   (f16 = 0, bf16 = 1, tf32 = 2), bit 15 A major (0 = K), bit 16 B major
//   (1 = MN), bits 17-22 N/8, bits 24-28 M/16.
__host__ __device__ constexpr uint32_t make_idesc(uint32_t afmt, uint32_t bfmt, uint32_t a_mn,
                                                  uint32_t b_mn, uint32_t M, uint32_t N) {
    return (1u << 4) | (afmt << 7) | (bfmt << 10) | (a_mn << 15) | (b_mn << 16) |
           ((N >> 3) << 17) | ((M >> 4) << 24);
}

}  // namespace ptx
}  // namespace tcl
