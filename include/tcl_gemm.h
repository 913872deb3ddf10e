/*
 * tcl_gemm.h — C ABI of the GB300 (sm_103a) pipelined tensor-core GEMM.
 *
 * Operation (every entry point): C = A · B, overwriting C.
 *   A is M×K, B is K×N, C is M×N, all row-major with leading dimensions
 *   lda, ldb, ldc counted in elements: A[i*lda + k], B[k*ldb + j],
 *   C[i*ldc + j]. There is no alpha/beta and no accumulation into C.
 *   Definition: "4.1 CUDA GEMM 算子性能优化", §1.1 (GEMM 的定义: C = A×B,
 *   A M×K, B K×N, 2·M·N·K flops) and the one-thread-per-element reference
 *   kernel of §3.1 (C[i][j] = sum_k A[i][k]·B[k][j], row-major A and B).
 *   How it is computed: the K-loop is tiled and software-pipelined so that
 *   the load of the next K-tile overlaps the tensor-core MMA on the current
 *   one ("流水化 GPU 内核", steps 3-4; "4.1 CUDA GEMM 算子性能优化", §9-§10);
 *   here with TMA loads into a multi-stage shared-memory ring, tcgen05.mma
 *   accumulating in fp32 in tensor memory, and a TMA-store epilogue.
 *
 * Memory and ownership: A, B and C are device pointers owned by the caller
 *   (allocated, kept alive until the stream has run the call, and freed by
 *   the caller). The library keeps a per-device cache of TMA descriptors and,
 *   per stream, a scratch buffer (the widened operands of gemm_s8, copies of
 *   operands or outputs off the 16-byte grid, split-K partial
 *   tiles for small grids, the fp32 partial sums of a bf16 C's stream-K
 *   tail) that it grows on demand (cudaMalloc, at least
 *   doubling; an outgrown buffer is kept, since enqueued or graph-captured
 *   work may still use it) and a small array of stream-K progress flags
 *   (8 KB, allocated and zeroed at the stream's first call). Calls on
 *   different streams therefore never share scratch or flags and may overlap
 *   on the GPU. (The pieces of a stream-K tile wait for one another, and the
 *   persistent grid is sized so that all of its CTAs fit on the GPU at once;
 *   a launch that another kernel keeps partly off the SMs for longer than
 *   timeout_ns reports device code 5 instead of waiting on.) The legacy and
 *   per-thread default streams share one set; a
 *   call captured into a graph on a stream that has not run a call outside
 *   capture before takes that default set too (and so do the graph's
 *   replays), so such a replay must not overlap work on the default streams.
 *   tcl_stream_release() frees one stream's set, tcl_shutdown() all of them.
 *
 * Streams: every call is asynchronous on `stream` (0 = legacy default
 *   stream) and returns once the work is enqueued. Calls on one stream run in
 *   order. The library is not thread-safe: serialise calls from several host
 *   threads.
 *
 * CUDA graphs: the device-pointer entry points may be captured into a graph
 *   and replayed. A captured call bakes in its TMA descriptors and scratch
 *   addresses, so the caller keeps A, B and C where they were; scratch is
 *   never freed before tcl_shutdown(), and a call that would have to grow it
 *   during capture returns TCL_ERR_CAPTURE (run the call once before
 *   capturing). Stream-K progress flags are left at zero by each launch that
 *   completes, so a replay (same flag generation) orders its pieces again; a
 *   replay after a launch that reported TCL_ERR_DEVICE_TIMEOUT is not safe.
 *
 * Alignment. Pointers must be aligned to their element size (bf16: 2
 *   bytes; fp32, int32: 4 bytes; int8: none), else TCL_ERR_ALIGN. The fast
 *   path also wants what the tensor copies (TMA) need — base addresses
 *   16-byte aligned and row strides a multiple of 16 bytes ("cp.async /
 *   ldmatrix 消融实验", §1.4 item 2 states the same 16-byte rule for
 *   cp.async) — and whole 16-byte pieces of K in a row of A (a tensor load
 *   rounds a row end up to 16 bytes):
 *   gemm_bf16: A, B, C 16-byte aligned; lda, ldb and K multiples of 8;
 *              ldc a multiple of 4 (fp32 C) or 8 (bf16 C).
 *   gemm_tf32: A, B, C 16-byte aligned; lda, ldb, K and ldc multiples of 4.
 *   gemm_s8:   C 16-byte aligned, ldc a multiple of 4 (A and B are always
 *              repacked).
 *   An operand that misses these is first copied into the library scratch
 *   with an aligned pitch and K zero-padded (to 8 for bf16, 4 for TF32), and
 *   a C that misses them is computed into scratch and then copied out: same
 *   result, one extra pass over that matrix. M and N are free (>= 1): edge
 *   tiles are zero-filled on load, rows past M are never written, and a
 *   right edge N that is not on a 16-byte boundary is written element by
 *   element, so nothing outside the M×N block of C changes.
 *
 * Errors: each entry point returns a tcl_status. Argument checks happen on
 *   the host before anything is enqueued; a nonzero status means nothing was
 *   launched. The library never prints, traps or aborts. Kernel-side waits
 *   are bounded; a wait that runs out records a code in a per-device status
 *   word that tcl_last_device_error() reads.
 */
#ifndef TCL_GEMM_H
#define TCL_GEMM_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define TCL_API __attribute__((visibility("default")))
#else
#define TCL_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    TCL_OK = 0,
    TCL_ERR_NULL = 1,            /* a required pointer is NULL */
    TCL_ERR_DIMS = 2,            /* M, N or K < 1 */
    TCL_ERR_LD = 3,              /* lda < K, ldb < N or ldc < N */
    TCL_ERR_ALIGN = 4,           /* a pointer is not aligned to its element size (gemm_s8_static:
                                    the stricter rule given there) */
    TCL_ERR_K_TOO_LARGE = 5,     /* gemm_s8: K > 131071, the int32 result could overflow */
    TCL_ERR_LAUNCH = 6,          /* a CUDA call or kernel launch failed */
    TCL_ERR_DEVICE_TIMEOUT = 7,  /* a bounded in-kernel wait ran out (see tcl_last_device_error) */
    TCL_ERR_CONFIG = 8,          /* tcl_config_t asks for a variant that is not built */
    TCL_ERR_NO_MEMORY = 9,       /* scratch allocation failed */
    TCL_ERR_DEVICE = 10,         /* current device is not an sm_103 GPU */
    TCL_ERR_STATIC_LIMIT = 11,   /* gemm_s8_static: the problem needs more scratch than the fixed
                                    TCL_S8_STATIC_SCRATCH_BYTES buffer holds */
    TCL_ERR_CAPTURE = 12         /* the call needs more library scratch than is allocated while its
                                    stream is being captured into a CUDA graph: run it (or a larger
                                    one) once outside capture first */
} tcl_status;

typedef enum { TCL_OUT_F32 = 0, TCL_OUT_BF16 = 1 } tcl_out_t;

/* Optional knobs for the *_ex entry points (ablation, tracing, tests).
 * Zero-initialise and set only what you need; zero means "automatic". */
typedef struct {
    int bn;                        /* N tile: 128 or 256; also 64 (one SM per tile, bf16 in, float
                                      out) and 224 (two SMs per tile) (0: chosen from M, N and the
                                      SM count) */
    int stages;                    /* shared-memory ring depth (0: the deepest that fits) */
    int one_cta_per_tile;          /* 0 (default): persistent, one CTA per SM walking the tiles;
                                      1: one CTA per output tile (no persistence) */
    int group_m;                   /* raster group height in tiles (0: automatic — 1 on the two-SM
                                      kernel when a row of A holds at least 16 KB (bf16 K >= 8192,
                                      TF32 K >= 4096), else 8) */
    int max_ctas;                  /* cap on resident CTAs for the persistent grid (0: all SMs) */
    unsigned long long timeout_ns; /* bound on every in-kernel wait (0: 1 s) */
    unsigned long long* trace;     /* device buffer of 4*trace_cap + 4 uint64, or NULL: %clock64
                                      stamps per k-block of CTA 0 (load issued, data landed,
                                      MMAs issued, MMAs done; int8 widened in the kernel: raw copy
                                      issued, raw slot landed, stage converted, stage handed over),
                                      then CTA 0's %clock64 and %globaltimer (ns) at its start and
                                      at its end (not written by the in-kernel int8 widening) */
    int trace_cap;                 /* k-blocks the trace buffer holds */
    int producer;                  /* 0 (default): TMA bulk-tensor loads issued by one thread;
                                      1: synchronous copy by four warps (ld.global -> registers ->
                                      st.shared), the ablation's lowest rung; 2: asynchronous copy
                                      by four warps (16-byte cp.async into shared memory, each
                                      thread's mbarrier arrival fires when its copies land), the
                                      middle rung. 1 and 2: bf16 only, one SM per tile, no
                                      debug_skip_kblock */
    int split_k;                   /* 0: automatic (when the output tiles alone would leave most SMs
                                      idle, K is cut into ranges whose fp32 partial tiles a second
                                      kernel adds in a fixed order); 1: never; s > 1: s ranges.
                                      One-SM kernel and floating-point output only */
    int cta_pair;                  /* 0: automatic; 1: one SM per tile (tcgen05 cta_group::1);
                                      2: two SMs per 256×256 tile (cta_group::2; bf16 in,
                                      fp32/bf16 out, TMA producer) */
    int epi_slots;                 /* epilogue staging slabs per warp, i.e. output stores in flight
                                      (0: automatic; two-SM kernel: 2 or 4, one-SM kernel: 2) */
    int debug_skip_kblock;         /* test hook, 0 = off. k > 0: CTA 0's TMA producer never loads
                                      the (k-1)-th k-block of its walk (two-SM kernel: CTA 0 skips
                                      its share while announcing the stage's bytes), so the MMA
                                      warp's bounded wait must run out; the call then reports
                                      TCL_ERR_DEVICE_TIMEOUT through tcl_last_device_error() and
                                      the outputs of that CTA are undefined */
    int stream_k;                  /* two-SM kernel, fp32 C: 0 automatic (when the last wave of
                                      tiles would leave pairs of SMs idle and the planner's cycle
                                      model favours it, each of those tiles is cut into 2..4 K
                                      ranges given to different pairs; range 0 stores, range i
                                      adds its result with a TMA reduction after range i-1 has
                                      finished, so the sum order is fixed); 1 never; s in 2..4
                                      exactly s ranges per tail tile of 256-wide tiles
                                      (TCL_ERR_CONFIG if they do not fit); 5 balanced: all waves of
                                      whole tiles but the last full one as usual, then the k-blocks of
                                      the remaining tiles cut into one equal range per pair, ranges
                                      crossing tile boundaries (a cut tile has two pieces; on request
                                      only: it was measured slower than equal pieces on GB300).
                                      Calls with a stream-K tail share progress flags on
                                      the device and must not run concurrently with one another */
    int serial_launch;             /* 0 (default): the GEMM kernels are launched with programmatic
                                      stream serialisation, so their set-up (barriers, TMEM, cluster
                                      handshake) overlaps the end of the previous kernel in the
                                      stream; they read and write global memory only after that
                                      kernel has completed. 1: plain stream order */
    int debug_stream_k_stall;      /* test hook, 0 = off. 1: the first stream-K piece of the first
                                      split tile never hands its tile over, so the next piece's
                                      bounded wait must run out (device status code 5) */
    int k_order;                   /* order in which a persistent CTA's successive tiles walk K:
                                      0 automatic (alternating where group_m's automatic value is 1,
                                      else ascending); 1 always ascending; 2
                                      alternating — every second tile of a CTA's walk loads its
                                      k-blocks in descending order, so that a wave of tiles starts
                                      on the operand blocks the previous wave read last (still in
                                      L2). The order changes the fp32 summation order of those
                                      tiles (not the exact int32 result). TMA producer only */
    int s8_path;                   /* gemm_s8 only: 0 automatic (= 1); 1 widening pass (int8 -> bf16
                                      copies of A and B in library scratch, then the GEMM); 2 widening
                                      inside the two-SM kernel (TMA copies the raw int8 tiles into
                                      shared memory, converter warps store them as fp16 into the MMA's
                                      stages; no scratch; needs 256-wide two-SM tiles and A, B 16-byte
                                      aligned with lda, ldb multiples of 16, else TCL_ERR_CONFIG /
                                      TCL_ERR_ALIGN). 2 is exact like 1 but slower on GB300 */
    int cluster_k;                 /* bf16 in, fp32 or bf16 C, one SM per tile: 0 or 1 one CTA per
                                      tile (the automatic choice: the cluster form was measured
                                      slower on GB300 at every 512² shape of the K sweep);
                                      2 or 4: each 128×64 tile is computed by a cluster of that many
                                      CTAs, CTA r summing the k-blocks [r·nkb/n, (r+1)·nkb/n), and
                                      the first CTA adds the others' partial tiles in rank order
                                      through distributed shared memory (one launch, no
                                      workspace). Not with split_k > 1, one_cta_per_tile, stages,
                                      producer != 0, or a bn other than 0 or 64 (TCL_ERR_CONFIG) */
    int tile_m;                    /* rows per output tile of the one-SM kernels: 0 automatic (64
                                      for grids of 128×128 tiles that fill at most a quarter of
                                      the SMs with fewer than 24 k-blocks, else 128), 128,
                                      or 64 (bf16 in, fp32 or bf16 C: 64×64 tiles, one CTA per tile,
                                      tcgen05.mma with M = 64, C stored from registers; not with
                                      split_k > 1, cluster_k > 1, cta_pair 2, stages, producer != 0,
                                      or a bn other than 0 or 64: TCL_ERR_CONFIG) */
    int kblocks_per_stage;         /* two-SM 256-wide tiles: k-blocks (64 bf16 or 32 TF32 values of
                                      K) that one tensor copy of A and one of B bring into the
                                      ring: 0 automatic (2 where allowed), 1, or 2 (needs K a
                                      multiple of the k-block, N of 64 bf16 / 32 TF32 columns, an
                                      even ring depth and the widening pass for int8, else
                                      TCL_ERR_CONFIG). Two halve the copies per k-block, which
                                      pace the stages on GB300 more than their bytes do; the
                                      result is the same either way (same summation order) */
    int b_copy;                    /* TMA producer, one k-block per copy: 0 automatic (a CTA's B
                                      boxes of a k-block in one 3-D tensor copy when N is a
                                      multiple of 64 bf16 / 32 TF32 columns and the tile has
                                      several boxes: 128- and 256-wide one-SM tiles, 256-wide
                                      two-SM tiles); 1 one copy per box. Same result */
    int die_split;                 /* two-SM kernel: 0 automatic (on for grids of at most 16 tile
                                      columns, at least 3 tiles per pair of SMs and at least 48
                                      k-blocks, 6 KB of K per operand row, when the die of every
                                      pair of SMs is known and no raster group is asked for),
                                      1 off, 2 on where possible (TCL_ERR_CONFIG otherwise). On:
                                      the tiles are cut into one block of columns per die of the
                                      GPU (whole columns and part of one, in proportion to the
                                      die's pairs of SMs), walked row by row by the pairs on that
                                      die, each block with its own stream-K tail, so that each
                                      die's half of the L2 holds its own block's operands. The die of each pair of SMs is
                                      measured once per device at the first call outside stream
                                      capture (a few tens of microseconds, synchronous). Each pair
                                      takes its place with one atomic on per-stream counters that
                                      the launch leaves zeroed (so calls sharing a set of counters,
                                      as graph-captured calls on different streams do, must not
                                      run concurrently); whole tiles give the same result either
                                      way */
    int l2_hints;                  /* two-SM kernel: 0 automatic (on with the die split for rows of
                                      A of at least 16 KB), 1 off, 2 on. On: the loads of A carry
                                      an L2 evict-first policy and those of B evict-last, so that
                                      each die's L2 keeps the B columns its waves share. Same
                                      result */
} tcl_config_t;

/* bf16 A, B (raw 16-bit patterns); fp32 accumulation; C fp32 (out = TCL_OUT_F32)
 * or bf16 rounded to nearest even (out = TCL_OUT_BF16). */
TCL_API int gemm_bf16(int M, int N, int K, const void* A, int lda, const void* B, int ldb, void* C, int ldc,
              int out, cudaStream_t stream);

/* fp32 A, B consumed by the tensor cores as TF32 (the low 13 mantissa bits of
 * each input are not used); fp32 accumulation; fp32 C. Both operands are read
 * in place: A K-major, B N-major (its rows as they lie in memory). */
TCL_API int gemm_tf32(int M, int N, int K, const float* A, int lda, const float* B, int ldb, float* C,
              int ldc, cudaStream_t stream);

/* int8 A, B; exact int32 C (bit-exact integer result for K <= 131071).
 * The operands are widened exactly to 16-bit floats (every int8 value is one):
 * by default a widening pass writes bf16 copies of A and B into library
 * scratch (tcl_config_t.s8_path selects the in-kernel widening instead), the
 * tensor cores accumulate in fp32 in units of at most 1024 K values (every
 * partial sum is an integer of magnitude at most 2^24, hence exact in fp32),
 * and each unit is added into int32 registers. */
TCL_API int gemm_s8(int M, int N, int K, const int8_t* A, int lda, const int8_t* B, int ldb, int32_t* C,
            int ldc, cudaStream_t stream);

/* gemm_bf16 on matrices in HOST memory (the end-to-end form of the call; the
 * pages have no counterpart): A, B and C are host pointers with the same
 * shapes, leading dimensions, element types and result as gemm_bf16 (no
 * 16-byte rule: the device copies are laid out by the library). B is uploaded
 * whole; A and C move in up to eight row chunks on the library's own streams, so
 * that the upload of a chunk, the GEMM of the previous one and the download of
 * the one before overlap. The pipeline starts after the work already queued
 * on `stream`, and `stream` waits for its end: C is complete once `stream` is
 * synchronised. Host buffers should be page-locked (cudaHostAlloc /
 * cudaHostRegister) for the copies to run asynchronously and overlap. Device
 * memory: the library scratch (grown on demand) holds A, B and C. */
TCL_API int gemm_bf16_host(int M, int N, int K, const void* A, int lda, const void* B, int ldb, void* C, int ldc,
                           int out, cudaStream_t stream);

/* SIMT fp32 GEMM: C = A·B with fp32 inputs, fp32 fused multiply-adds on the
 * CUDA cores (no tensor cores) and fp32 C — the architecture-level anchor the
 * pages set beside their tensor-core kernels ("4.1 CUDA GEMM 算子性能优化"
 * §4–§9: block and thread tiling, A transposed in shared memory, float4
 * accesses, double buffering). Each output is accumulated in increasing k
 * from 0, one rounding per step: |C - C_exact| <= K·u/(1-K·u)·Σ_k|a_ik·b_kj|,
 * u = 2^-24. Any leading dimensions and bases aligned to 4 bytes (16-byte
 * aligned rows take vector accesses); M up to 8,388,480. Allocates nothing. */
TCL_API int gemm_f32_simt(int M, int N, int K, const float* A, int lda, const float* B, int ldb, float* C, int ldc,
                          cudaStream_t stream);

/* Allocation-free int8 GEMM. (The pages have no counterpart: this is a
 * library service, not part of the method.)
 *
 * Same operation, arguments and exact int32 result as gemm_s8, but the
 * library allocates nothing (and so cannot repack off-grid C: A, B and C
 * must be 16-byte aligned, lda and ldb multiples of 16, ldc of 4, else
 * TCL_ERR_ALIGN): the bf16 copies of A and B are
 * written into a fixed buffer that is part of the library's device image, a
 * file-scope array of TCL_S8_STATIC_SCRATCH_BYTES (64 MiB). Every GPU on which
 * the library's code is loaded holds that buffer until the process exits.
 *
 * Who needs it: callers that cannot call cudaMalloc at the point of use —
 * a process whose device memory is already reserved by another allocator
 * (a framework's caching pool that holds the free memory, so a fresh
 * cudaMalloc fails or fragments it), and callers that must not have the
 * library allocate at the point of use (gemm_s8 grows its scratch with
 * cudaMalloc, which also cannot run while the stream is being captured).
 *
 * Limit: the packed copies need 2·(M·⌈K⌉₈ + K·⌈N⌉₈) bytes, each block rounded
 * up to 256 bytes; a larger problem returns TCL_ERR_STATIC_LIMIT before
 * anything is enqueued (4096×4096×4096 fits exactly).
 *
 * Set-up: the first call on a device (with that device current) looks up the
 * buffer's device address with cudaGetSymbolAddress and keeps it; make that
 * first call before any stream capture. Later calls do no set-up.
 *
 * Sharing: every call on a device uses the same buffer, which keeps the last
 * call's contents. Each call rewrites every byte the GEMM reads from it
 * (including the zero padding of ragged rows), so stale contents never leak
 * into a result. Calls whose GPU work overlaps (different streams without
 * ordering between them) race on the buffer; calls on one stream are ordered
 * and safe. Not thread-safe across host threads, like the rest of the API. */
#define TCL_S8_STATIC_SCRATCH_BYTES (64ull << 20)
TCL_API int gemm_s8_static(int M, int N, int K, const int8_t* A, int lda, const int8_t* B, int ldb,
                           int32_t* C, int ldc, cudaStream_t stream);

/* Same operations with explicit knobs; cfg may be NULL (= all automatic). */
TCL_API int gemm_bf16_ex(int M, int N, int K, const void* A, int lda, const void* B, int ldb, void* C,
                 int ldc, int out, const tcl_config_t* cfg, cudaStream_t stream);
TCL_API int gemm_tf32_ex(int M, int N, int K, const float* A, int lda, const float* B, int ldb, float* C,
                 int ldc, const tcl_config_t* cfg, cudaStream_t stream);
TCL_API int gemm_s8_ex(int M, int N, int K, const int8_t* A, int lda, const int8_t* B, int ldb, int32_t* C,
               int ldc, const tcl_config_t* cfg, cudaStream_t stream);

/* What the library would launch for a problem (see tcl_plan). */
typedef struct {
    int bn;                         /* output tile width (columns) */
    int stages;                     /* shared-memory ring depth */
    int grid;                       /* CTAs launched */
    int num_tiles;                  /* output tiles (of 128 or, for cta_pair 2, 256 rows) */
    int smem_bytes;                 /* dynamic shared memory per CTA */
    int cta_pair;                   /* 1: one SM per tile; 2: two SMs per tile */
    int splits;                     /* K ranges (1: no split-K) */
    int producer;                   /* 0: TMA, 1: synchronous copy, 2: cp.async */
    unsigned long long workspace_bytes;   /* library scratch for split-K partial tiles */
    int sk_tiles;                   /* tail tiles computed stream-K (0: none) */
    int sk_pieces;                  /* K ranges per stream-K tile */
    int sk_balanced;                /* 1: balanced stream-K (sk_tiles = tiles cut by range boundaries) */
    int group_m;                    /* raster group height in tiles */
    int k_serpentine;               /* 1: alternating K order (see tcl_config_t.k_order) */
    int s8_in_kernel;               /* int8: 1 if the kernel widens the operands itself
                                       (tcl_config_t.s8_path = 2), 0 for the widening pass */
    int cluster_k;                  /* CTAs per tile whose K ranges are summed in a cluster
                                       (1: one CTA per tile; see tcl_config_t.cluster_k) */
    int tile_m;                     /* rows per output tile (64, 128, or 256 for two SMs per tile) */
    int kblocks_per_stage;          /* k-blocks that one tensor copy of each operand brings (1 or 2) */
    int die_split;                  /* 1: the tile columns in one block per die (tcl_config_t.die_split) */
    int die_tiles0;                 /* with die_split: tiles of the first die's block */
    int l2_hints;                   /* 1: A's loads evict-first, B's evict-last (tcl_config_t.l2_hints) */
} tcl_plan_t;

/* Fills *plan (if not NULL) with the launch the library would make for this
 * problem, without launching: in_kind 0 = bf16, 1 = tf32, 2 = int8. With
 * cfg->max_ctas > 0 no device is queried (max_ctas stands for the SM count).
 * Returns a tcl_status (argument checks as above; no pointers needed). */
TCL_API int tcl_plan(int in_kind, int out, int M, int N, int K, const tcl_config_t* cfg, tcl_plan_t* plan);

/* Tensor-pipe rate probe (measurement, not part of the GEMM): `grid` CTAs
 * (one per SM) each issue `iters` (a multiple of 4, at least 8) back-to-back
 * tcgen05.mma, four at a time from one elected lane of a converged warp, of shape
 * M=128 × N=n (128, 192, 224 or 256) × K=16 (bf16, in_kind 0) or K=8 (TF32,
 * in_kind 1) on operands
 * already in shared memory (B K-major, or N-major if b_mn = 1; bf16 only),
 * and write the %clock64 cycles from the first issue to the completion of the
 * last into cycles[blockIdx] (device buffer of `grid` entries; 0 if the
 * bounded wait ran out). flop/clk/SM = 2·128·n·K·iters / cycles.
 * flags bit 0: chain every MMA into one accumulator, as the MMAs of one GEMM
 * tile are (default: alternate two independent accumulators); bit 1: walk
 * the operand addresses like a GEMM k-loop (4 k-slices × 4 ring stages);
 * bit 2: N-major B with 64-column groups of 64 K-rows (8 KB apart, as a GEMM
 * stage holds it) instead of 16 K-rows (2 KB apart); bit 3: per group of
 * MMAs, the rest of a GEMM issue loop (an mbarrier wait, a tcgen05 fence, a
 * commit); bit 4: of those, the wait and fence only; bit 5: the commit only;
 * bit 6: groups of 8 MMAs instead of 4 (iters then a multiple of 8).
 * Warp-level MMA instead (in_kind 2: int8 m16n8k32 → int32, the only int8
 * tensor-core instruction sm_103a has; in_kind 0 with flags = 128: bf16
 * m16n8k16 → fp32; n and b_mn are then ignored but must be valid, b_mn 0):
 * 8 warps per CTA, each `iters` rounds of 8 independent mma.sync on register
 * operands; cycles[blockIdx] = %clock64 over the loop, and
 * ops/clk/SM = 64·iters·(8192 for int8, 4096 for bf16) / cycles. */
TCL_API int tcl_mma_peak(int in_kind, int n, int b_mn, int flags, int iters, int grid,
                         unsigned long long* cycles, cudaStream_t stream);

/* Human-readable text for a tcl_status; never NULL. */
TCL_API const char* tcl_status_string(int status);

/* Synchronises `stream`, then reads and clears the current device's status
 * word. Returns TCL_OK, or TCL_ERR_DEVICE_TIMEOUT if any kernel since the
 * last read recorded a timed-out wait (*detail, if not NULL, receives the raw
 * code: 1 producer, 2 MMA waiting for data, 3 MMA waiting for an accumulator,
 * 4 epilogue, 5 stream-K piece waiting for the previous piece; 6, not a wait:
 * under the die split a pair of SMs found no place free because the counters
 * were not zero at the launch's start, its tiles then not computed), or
 * TCL_ERR_LAUNCH if synchronising failed. */
TCL_API int tcl_last_device_error(cudaStream_t stream, int* detail);

/* Streaming multiprocessors of the current device (0 on error). */
TCL_API int tcl_num_sms(void);

/* Pairs of SMs on each of the two dies of the current device, as measured for
 * the die split (tcl_config_t.die_split): *n0 + *n1 pairs, or 0 and 0 when the
 * measurement found no two clear groups (or has not run: it runs here, or at
 * the first call outside stream capture). Returns a tcl_status. */
TCL_API int tcl_die_pairs(int* n0, int* n1);

/* Frees the scratch buffer and stream-K flags that calls on `stream` (of the
 * current device) have used, after synchronising the stream: for a stream the
 * caller is about to destroy. Graphs that captured calls on that stream must
 * not be replayed afterwards. A stream the library holds nothing for, and the
 * default streams, are no-ops. TCL_OK, or TCL_ERR_LAUNCH if synchronising
 * failed. No counterpart in the source pages: library housekeeping. */
TCL_API int tcl_stream_release(cudaStream_t stream);

/* Frees the scratch buffers of every device and stream, the outgrown ones
 * included (after synchronising each device), the streams' stream-K flags,
 * and the host-buffer entry point's streams. */
TCL_API void tcl_shutdown(void);

/* Library version string, e.g. "tcl-gb300 0.1.0 sm_103a". */
TCL_API const char* tcl_version(void);

#ifdef __cplusplus
}
#endif

#endif /* TCL_GEMM_H */
