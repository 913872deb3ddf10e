// C ABI of the library (declared in include/tcl_gemm.h): argument checks,
// launch planning, TMA descriptor construction and caching, the int8 scratch,
// the device status word, and dispatch to the instantiated kernels.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <unordered_map>
#include <vector>

#include "launch.cuh"
#include "tcl_gemm.h"

namespace tcl {
namespace {

// Per-device status word written by kernels whose bounded waits ran out.
__device__ unsigned int g_status_word;

// Stream-K progress flags of the two-SM kernel: [split tile][CTA of the pair][epilogue warp].
// They only ever hold gen·8 + pieces done, gen being a per-device launch counter,
// so they never need clearing between launches.
constexpr int kMaxSkTiles = 128;
__device__ unsigned int g_sk_flags[kMaxSkTiles * 2 * 8];
// The die split's rank counters and finished-pair count (zero between launches).
__device__ unsigned long long g_sched_ctr[4];

constexpr int kMaxDevices = 64;
constexpr unsigned long long kDefaultTimeoutNs = 1000000000ull;   // 1 s
constexpr int kBM = 128;
// K values per exact fp32 unit: every partial sum of a unit, of any subset of its
// products, is an integer of magnitude at most 1024·2^14 = 2^24, and every such
// integer is an fp32 value (below 2^24 the unit in the last place is at most 1), so
// the fp32 accumulation and its conversion are exact.
// (Measured on GB300: 512-K units beat 256-K units converted with a cheaper add,
// 103 vs 108 us at int8 4096^3: the unit turnover costs more than the conversion.)
constexpr int kS32UnitK = 1024;

constexpr size_t kSkFlagBytes = sizeof(unsigned int) * kMaxSkTiles * 2 * 8;
constexpr size_t kStreamFlagBytes = kSkFlagBytes + 4 * sizeof(unsigned long long);   // + die split counters

// Scratch and stream-K progress flags of the calls on one stream. Calls on
// different streams may run on the GPU at the same time, so each stream has a
// set of its own, made at its first call.
struct StreamRes {
    void* scratch = nullptr;
    size_t scratch_bytes = 0;
    unsigned int* sk_flags = nullptr;   // kMaxSkTiles · 2 · 8 words
    unsigned long long* sched_ctr = nullptr;   // die split counters (after the flags in an own set)
    unsigned int sk_gen = 0;            // last stream-K flag generation used with these flags
    bool own_flags = false;             // allocated for this stream (the default set's are a static array)
};

struct DevState {
    bool probed = false;
    bool supported = false;
    int sms = 0;
    // which die each pair of SMs is on (calibrated once, outside stream capture)
    int die_state = 0;             // 0 not yet, 1 known, -1 unknown (no die split)
    int die_pairs[2] = {0, 0};
    uint8_t die_of_tpc[128] = {};
    int pair_clusters[16] = {};  // resident clusters per pair variant (0: not yet queried)
    unsigned int* status = nullptr;
    // the set of the legacy and per-thread default streams, also taken by a call
    // captured on a stream that has no set of its own yet
    StreamRes base;
    std::unordered_map<cudaStream_t, StreamRes> per_stream;
    std::vector<void*> retired;   // outgrown scratch buffers, freed by tcl_shutdown
    // host-buffer entry points: uploads, GEMMs and downloads on their own streams
    cudaStream_t up = nullptr, comp = nullptr, down = nullptr;
};

DevState g_dev[kMaxDevices];
std::mutex g_mu;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

const VariantInfo kVariants[] = {
    TCL_GROUP_BF16_F32_BN256(TCL_VARIANT_INFO) TCL_GROUP_BF16_F32_BN128(TCL_VARIANT_INFO)
        TCL_GROUP_BF16_MISC(TCL_VARIANT_INFO) TCL_GROUP_BF16_SYNC(TCL_VARIANT_INFO)
            TCL_GROUP_BF16_CPASYNC(TCL_VARIANT_INFO)
            TCL_GROUP_TF32(TCL_VARIANT_INFO) TCL_GROUP_PAIR(TCL_PAIR_INFO)};

struct MapKey {
    int dev;
    const void* ptr;
    int dtype;
    uint64_t d0, d1, stride;
    uint32_t b0, b1;
    int swizzle;
    uint64_t d2 = 0, stride2 = 0;   // a 3-D map's third dimension (0: 2-D)
    uint32_t b2 = 0;
    uint64_t d3 = 0, stride3 = 0;   // a 4-D map's fourth dimension (0: fewer)
    uint32_t b3 = 0;
    bool operator==(const MapKey& o) const {
        return dev == o.dev && ptr == o.ptr && dtype == o.dtype && d0 == o.d0 && d1 == o.d1 &&
               stride == o.stride && b0 == o.b0 && b1 == o.b1 && swizzle == o.swizzle && d2 == o.d2 &&
               stride2 == o.stride2 && b2 == o.b2 && d3 == o.d3 && stride3 == o.stride3 && b3 == o.b3;
    }
};
struct MapKeyHash {
    size_t operator()(const MapKey& k) const {
        uint64_t h = 1469598103934665603ull;
        auto mix = [&h](uint64_t v) {
            h ^= v;
            h *= 1099511628211ull;
        };
        mix(static_cast<uint64_t>(k.dev));
        mix(reinterpret_cast<uint64_t>(k.ptr));
        mix(static_cast<uint64_t>(k.dtype));
        mix(k.d0);
        mix(k.d1);
        mix(k.stride);
        mix((static_cast<uint64_t>(k.b0) << 32) | k.b1);
        mix(static_cast<uint64_t>(k.swizzle));
        mix(k.d2);
        mix(k.stride2);
        mix(k.b2);
        mix(k.d3);
        mix(k.stride3);
        mix(k.b3);
        return static_cast<size_t>(h);
    }
};
std::unordered_map<MapKey, CUtensorMap, MapKeyHash> g_maps;

int in_bytes(InKind k) { return k == InKind::TF32 ? 4 : 2; }
int out_bytes(OutKind k) { return k == OutKind::BF16 ? 2 : 4; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned_to(const void* p, uintptr_t n) { return (reinterpret_cast<uintptr_t>(p) % n) == 0; }
long long round_up(long long x, long long m) { return (x + m - 1) / m * m; }

bool is_capturing(cudaStream_t stream, int* st) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) {
        cudaGetLastError();
        *st = TCL_ERR_LAUNCH;
        return false;
    }
    *st = TCL_OK;
    return cs != cudaStreamCaptureStatusNone;
}

// The scratch and flag set of `stream` on this device. A stream gets its own set
// at its first call outside capture (its flags allocated and zeroed on the
// stream, ahead of the call's kernels); a call captured on a stream without a
// set takes the default streams' set, as will every replay of the graph.
int stream_res(DevState* ds, cudaStream_t stream, StreamRes** out) {
    if (stream == nullptr || stream == cudaStreamLegacy || stream == cudaStreamPerThread) {
        *out = &ds->base;
        return TCL_OK;
    }
    auto it = ds->per_stream.find(stream);
    if (it != ds->per_stream.end()) {
        *out = &it->second;
        return TCL_OK;
    }
    int st;
    const bool capturing = is_capturing(stream, &st);
    if (st) return st;
    if (capturing) {
        *out = &ds->base;
        return TCL_OK;
    }
    void* p = nullptr;
    if (cudaMalloc(&p, kStreamFlagBytes) != cudaSuccess) {
        cudaGetLastError();
        return TCL_ERR_NO_MEMORY;
    }
    if (cudaMemsetAsync(p, 0, kStreamFlagBytes, stream) != cudaSuccess) {
        cudaGetLastError();
        cudaFree(p);
        return TCL_ERR_LAUNCH;
    }
    StreamRes r;
    r.sk_flags = static_cast<unsigned int*>(p);
    r.sched_ctr = reinterpret_cast<unsigned long long*>(static_cast<char*>(p) + kSkFlagBytes);
    r.own_flags = true;
    *out = &ds->per_stream.emplace(stream, r).first->second;   // (map nodes never move)
    return TCL_OK;
}

// Grows a stream's scratch to at least `need` bytes (at least doubling it).
// The outgrown buffer is kept until tcl_shutdown: work already enqueued, or
// captured into a CUDA graph, may still use it. No allocation while `stream`
// is being captured (TCL_ERR_CAPTURE): a captured call must find its scratch
// already allocated by an earlier call outside capture.
int ensure_scratch(DevState* ds, StreamRes* sr, size_t need, cudaStream_t stream) {
    if (sr->scratch_bytes >= need) return TCL_OK;
    int st;
    const bool capturing = is_capturing(stream, &st);
    if (st) return st;
    if (capturing) return TCL_ERR_CAPTURE;
    const size_t want = std::max(need, 2 * sr->scratch_bytes);
    void* p = nullptr;
    if (cudaMalloc(&p, want) != cudaSuccess) {
        cudaGetLastError();
        return TCL_ERR_NO_MEMORY;
    }
    if (sr->scratch) ds->retired.push_back(sr->scratch);
    sr->scratch = p;
    sr->scratch_bytes = want;
    return TCL_OK;
}

// Host-side argument checks shared by every entry point; no CUDA call.
int check_common(int M, int N, int K, const void* A, int lda, const void* B, int ldb, const void* C,
                 int ldc) {
    if (!A || !B || !C) return TCL_ERR_NULL;
    if (M < 1 || N < 1 || K < 1) return TCL_ERR_DIMS;
    if (lda < K || ldb < N || ldc < N) return TCL_ERR_LD;
    return TCL_OK;
}

// Current device: probe capability, SM count and status-word address once.
int current_device(int* dev_out, DevState** st_out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return TCL_ERR_LAUNCH;
    }
    DevState& d = g_dev[dev];
    if (!d.probed) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return TCL_ERR_LAUNCH;
        }
        d.supported = (major == 10 && minor == 3);
        d.sms = sms;
        if (d.supported) {
            void* p = nullptr;
            if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) {
                cudaGetLastError();
                return TCL_ERR_LAUNCH;
            }
            d.status = static_cast<unsigned int*>(p);
            if (cudaGetSymbolAddress(&p, g_sk_flags) != cudaSuccess) {
                cudaGetLastError();
                return TCL_ERR_LAUNCH;
            }
            d.base.sk_flags = static_cast<unsigned int*>(p);
            if (cudaGetSymbolAddress(&p, g_sched_ctr) != cudaSuccess) {
                cudaGetLastError();
                return TCL_ERR_LAUNCH;
            }
            d.base.sched_ctr = static_cast<unsigned long long*>(p);
        }
        d.probed = true;
    }
    if (!d.supported) return TCL_ERR_DEVICE;
    *dev_out = dev;
    *st_out = &d;
    return TCL_OK;
}

int encode_fn() {
    if (g_encode) return TCL_OK;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr) {
        cudaGetLastError();
        return TCL_ERR_LAUNCH;
    }
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    return TCL_OK;
}

// 2-D row-major tensor map: inner extent d0 (contiguous), outer d1, row
// stride in bytes, box b0 × b1, 128-byte swizzle (in 16-byte units, or for
// swz = CU_TENSOR_MAP_SWIZZLE_128B_ATOM_32B in 32-byte units), zero fill out
// of bounds.
int tensor_map(int dev, const void* ptr, CUtensorMapDataType dtype, uint64_t d0, uint64_t d1,
               uint64_t stride_bytes, uint32_t b0, uint32_t b1, CUtensorMap* out,
               CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B) {
    const MapKey key{dev, ptr, static_cast<int>(dtype), d0, d1, stride_bytes, b0, b1, static_cast<int>(swz)};
    auto it = g_maps.find(key);
    if (it != g_maps.end()) {
        *out = it->second;
        return TCL_OK;
    }
    int st = encode_fn();
    if (st) return st;
    CUtensorMap m;
    const cuuint64_t dims[2] = {d0, d1};
    const cuuint64_t strides[1] = {stride_bytes};
    const cuuint32_t box[2] = {b0, b1};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(&m, dtype, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return TCL_ERR_LAUNCH;
    if (g_maps.size() > 4096) g_maps.clear();
    g_maps.emplace(key, m);
    *out = m;
    return TCL_OK;
}

// 3-D or 4-D map (d3 = 0: 3-D): dims innermost first, byte strides of
// dimensions 1.., box per dimension.
int tensor_map_nd(int dev, const void* ptr, CUtensorMapDataType dtype, uint64_t d0, uint64_t d1, uint64_t d2,
                  uint64_t d3, uint64_t stride1, uint64_t stride2, uint64_t stride3, uint32_t b0, uint32_t b1,
                  uint32_t b2, uint32_t b3, CUtensorMap* out, CUtensorMapSwizzle swz) {
    MapKey key{dev, ptr, static_cast<int>(dtype), d0, d1, stride1, b0, b1, static_cast<int>(swz)};
    key.d2 = d2;
    key.stride2 = stride2;
    key.b2 = b2;
    key.d3 = d3;
    key.stride3 = stride3;
    key.b3 = b3;
    auto it = g_maps.find(key);
    if (it != g_maps.end()) {
        *out = it->second;
        return TCL_OK;
    }
    int st = encode_fn();
    if (st) return st;
    CUtensorMap m;
    const cuuint32_t rank = d3 ? 4 : 3;
    const cuuint64_t dims[4] = {d0, d1, d2, d3};
    const cuuint64_t strides[3] = {stride1, stride2, stride3};
    const cuuint32_t box[4] = {b0, b1, b2, b3};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = g_encode(&m, dtype, rank, const_cast<void*>(ptr), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return TCL_ERR_LAUNCH;
    if (g_maps.size() > 4096) g_maps.clear();
    g_maps.emplace(key, m);
    *out = m;
    return TCL_OK;
}

int tensor_map_3d(int dev, const void* ptr, CUtensorMapDataType dtype, uint64_t d0, uint64_t d1, uint64_t d2,
                  uint64_t stride1, uint64_t stride2, uint32_t b0, uint32_t b1, uint32_t b2, CUtensorMap* out,
                  CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B) {
    return tensor_map_nd(dev, ptr, dtype, d0, d1, d2, 0, stride1, stride2, 0, b0, b1, b2, 0, out, swz);
}

struct Plan {
    int bn, stages, prod, pair, slots, grid, tiles_m, tiles_n, num_tiles, num_kb, kb_per_unit, group_m, smem;
    int sk_ws_rows;   // bf16 C with a stream-K tail: fp32 workspace rows (split tiles × 256), else 0
    int splits, kb_per_split;   // split-K: K cut into `splits` ranges of kb_per_split k-blocks
    int sk_tiles, sk_pieces;    // stream-K tail of the two-SM kernel (0 tiles: none)
    int sk_balanced, sk_first, sk_region;   // balanced stream-K (see GemmParams)
    int k_serpentine;           // odd units of a CTA's walk load K in descending order
    int s8_in_kernel;           // int8: the two-SM kernel that widens the operands itself
    int csk;                    // > 1: CTAs per tile summing its K ranges in a cluster (gemm_kernel_csk.cuh)
    int m64;                    // 1 or 2: 64×64 tiles, one CTA per tile, k-blocks per stage (gemm_kernel_m64.cuh)
    int kps;                    // two-SM kernel: k-blocks per tensor copy (1 or 2)
    // two-SM kernel: the tile columns in one sub-grid per die (see GemmParams)
    int l2_hints;               // two-SM kernel: A's loads evict-first, B's evict-last in L2
    int die_split, sub_n[2], sub_rs, sub_a[2], sub_s[2], sub_b[2], sub_u[2], sub_tiles[2], sub_sk_tiles[2],
        sub_sk_pieces[2];
};

// Split-K pays only when the k-blocks saved per CTA outweigh the partial-tile
// traffic and the extra reduction launch (measured on GB300 at M=N=512: a
// loss at K ≤ 1024, a gain from K = 4096 on).
constexpr int kMinKbPerSplit = 8;    // k-blocks each range keeps
constexpr int kMinKbForPair = 16;    // k-blocks a tile needs before two SMs per tile pay off
constexpr int kMinKbToSplit = 24;    // k-blocks a tile needs before splitting is considered
constexpr long long kMinKBytesForRowRaster = 16384;   // two-SM kernel: K bytes per operand row from which
                                                      // group 1 and alternating K order are the default

// Two-SM kernel: model cycles per k-block of a pair tile (64 bf16 or 32 TF32 deep) and
// the fixed part of a launch. The tensor pipe takes 512 cycles per 256-wide k-block
// and runs 224-wide tiles ~9.6 % below its rate (in-kernel timeline); the constants
// below are instead fitted to the planner's choices: CUDA graphs of back-to-back
// calls on GB300 at 42 shapes of bf16, TF32 and int8 between 768 and 8192 on a side
// and K from 512 to 8192, each timed on two-SM 224- and 256-wide and one-SM tiles in
// one process, round robin. With two k-blocks per tensor copy the 256-wide tiles pull
// ahead as K grows (a lower cost per k-block, a higher fixed part), and int8, whose
// one-SM tiles are 128 wide with an integer drain, keeps its own fixed part. Over
// those shapes the picks lose 0.5 % of time against the best choice (the earlier
// constants: 4 %; worst case now 8 % at 8192×2048×1024 with a bf16 C).
constexpr long long kPairKbCycles256 = 420;
constexpr long long kPairKbCycles224 = 520;
// Stream-K tail: at most this many pieces per split tile (each waits for the
// previous one before adding its result) and at least this many k-blocks each.
constexpr int kMaxSkPieces = 4;
constexpr int kSkBalanced = 5;   // tcl_config_t.stream_k value asking for balanced stream-K
constexpr int kMinKbPerPiece = 8;
// ... and only for tiles of at least this many k-blocks: below it the tile's
// epilogue is a large share of its time and the extra piece's epilogue eats
// the gain (measured on GB300 at 4096²: 224-wide whole tiles 8 % faster at
// K = 1024, even at 1536, stream-K ahead from 2048).
constexpr int kMinKbForSk = 32;
constexpr int kMaxDieSplitCols = 16;   // automatic die split up to this many tile columns (two blocks)
constexpr int kMinDieSplitPairs = 32;  // and only on a whole GPU's pairs
constexpr int kMinDieSplitWaves = 3;   // and at least this many tiles per pair
// and at least this many k-blocks (128-byte rows of K) per tile: measured on GB300 (CUDA
// graphs, round robin), the split against the whole grid is 2.6–5.1 % slower below 4 KB
// of K per operand row (bf16 K ≤ 1536, TF32 K = 768), about level at 4 KB (bf16 K = 2048,
// TF32 K = 1024: −1.0 to +1.3 % over five shapes), 0.4 % faster at 5 KB and 1.7–2.3 % at
// 6–8 KB (bf16 K = 3072, TF32 K = 2048)
constexpr int kMinDieSplitKb = 48;
constexpr long long kSkLinkCycles = 4096;   // one piece's epilogue, exposed when pieces are all a pair does

// Stream-K split of the last (partial) wave of pair tiles: with `tiles` tiles
// on `pairs` pairs of SMs, the tiles past the last full wave are each cut into
// `pieces` K ranges so that the otherwise idle pairs share them.
// want: 0 automatic, 1 never, s >= 2 exactly s pieces (TCL_ERR_CONFIG if that
// does not fit). Fills *sk_tiles = 0 when there is no stream-K tail.
int stream_k_split(long long tiles, int pairs, int num_kb, int want, int* sk_tiles, int* sk_pieces) {
    *sk_tiles = 0;
    *sk_pieces = 1;
    const long long rem = tiles % pairs;
    if (want == 1 || rem == 0) return TCL_OK;
    if (want >= 2) {
        if (want > kMaxSkPieces || rem * want > pairs || want > num_kb || rem > kMaxSkTiles) return TCL_ERR_CONFIG;
        *sk_tiles = static_cast<int>(rem);
        *sk_pieces = want;
        return TCL_OK;
    }
    const int s = static_cast<int>(std::min<long long>({kMaxSkPieces, pairs / rem, num_kb / kMinKbPerPiece}));
    if (s >= 2 && rem <= kMaxSkTiles && num_kb >= kMinKbForSk) {
        *sk_tiles = static_cast<int>(rem);
        *sk_pieces = s;
    }
    return TCL_OK;
}

// One SM per tile (bf16 operands): SM cycles per 64-deep k-block of a wave of
// 128×128 and 128×256 tiles, and the fixed cycles of a launch (first loads,
// last epilogue), fitted on GB300 (CUDA graphs of back-to-back calls at
// 1024×4096 and 2048² with K = 1024 and 4096: 128 wide ~0.23 µs per k-block
// and wave, 256 wide ~0.335; the launch's fixed part ~5 and ~6.3 µs).
constexpr long long kOneKbCycles128 = 440;
constexpr long long kOneKbCycles256 = 640;
constexpr long long kOneFixedCycles128 = 9500;
constexpr long long kOneFixedCycles256 = 12000;
constexpr long long kPairFixedCycles = 30500;
constexpr long long kPairFixedCyclesS32 = 13000;

// Busiest pair's k-block cycles for pair tiles of width w: ceil(tiles / pairs)
// whole tiles, or the full waves plus the largest stream-K piece.
long long pair_cost(long long tiles, int pairs, int num_kb, long long kb_cycles, int sk_tiles, int sk_pieces) {
    if (sk_tiles == 0) return (tiles + pairs - 1) / pairs * num_kb * kb_cycles;
    const long long waves = tiles / pairs;
    return (waves * num_kb + (num_kb + sk_pieces - 1) / sk_pieces) * kb_cycles +
           (waves == 0 ? (sk_pieces - 1) * kSkLinkCycles : 0);
}

// Cycles of a one-SM launch of 128-wide or 256-wide tiles (w = 0: the cheaper).
long long one_sm_cost(int M, int N, int num_kb, int sms, int w) {
    auto cost = [&](int bw, long long kb_cycles, long long fixed) {
        const long long tiles = static_cast<long long>((M + kBM - 1) / kBM) * ((N + bw - 1) / bw);
        return (tiles + sms - 1) / sms * num_kb * kb_cycles + fixed;
    };
    const long long c128 = cost(128, kOneKbCycles128, kOneFixedCycles128);
    const long long c256 = cost(256, kOneKbCycles256, kOneFixedCycles256);
    return w == 128 ? c128 : w == 256 ? c256 : std::min(c128, c256);
}

// Balanced stream-K over `pairs` pairs: the whole tiles of all waves but the
// last full one are dealt out as usual, and the k-blocks of the remaining
// tiles (between one and two waves of them) are cut into one equal range per
// pair. *split counts the tiles a range boundary cuts (two pieces each).
struct Balanced {
    int first, region, split;
    long long busiest_kb;   // k-blocks of the busiest pair
};

Balanced balanced_split(long long tiles, int pairs, int num_kb) {
    Balanced b{0, 0, 0, 0};
    if (tiles < pairs || pairs < 2) return b;
    const long long waves = tiles / pairs - 1;
    b.first = static_cast<int>(waves * pairs);
    b.region = static_cast<int>(tiles - b.first);
    const long long total = static_cast<long long>(b.region) * num_kb;
    for (int c = 0; c + 1 < pairs; ++c)
        if ((total * (c + 1) / pairs) % num_kb) ++b.split;
    b.busiest_kb = waves * num_kb + (total + pairs - 1) / pairs;
    return b;
}

// slots = 0 matches any staging depth (the first listed, i.e. two slabs per warp)
const VariantInfo* find_variant(InKind ik, OutKind ok, int bn, int stages, int prod, int pair, int slots = 0) {
    for (const auto& v : kVariants)
        if (v.in == ik && v.out == ok && v.bn == bn && v.stages == stages && v.prod == prod && v.pair == pair &&
            (slots == 0 || v.slots == slots))
            return &v;
    return nullptr;
}

int deepest_stages(InKind ik, OutKind ok, int bn, int prod, int pair, int slots = 0) {
    int best = 0;
    for (const auto& v : kVariants)
        if (v.in == ik && v.out == ok && v.bn == bn && v.prod == prod && v.pair == pair &&
            (slots == 0 || v.slots == slots) && v.stages > best)
            best = v.stages;
    return best;
}


// Chooses the tile shape, ring depth, one- or two-SM kernel and grid.
// `sms` is the SM count; `pair_clusters(v)` returns how many two-CTA clusters
// of pair variant v fit on the device at once.
// die_pairs[d]: pairs of SMs on each die of the device (0, 0: not known).
template <class PairClusters>
int make_plan(InKind ik, OutKind ok, int M, int N, int K, const tcl_config_t* cfg, int sms,
              PairClusters pair_clusters, const int* die_pairs, Plan* pl) {
    const int bk = 128 / in_bytes(ik);
    const int prod = cfg ? cfg->producer : PROD_TMA;
    if (prod != PROD_TMA && prod != PROD_SYNC && prod != PROD_CPASYNC) return TCL_ERR_CONFIG;
    const int want_pair = cfg ? cfg->cta_pair : 0;
    if (want_pair < 0 || want_pair > 2) return TCL_ERR_CONFIG;
    int bn = cfg ? cfg->bn : 0;
    // K ranges summed in a cluster: bf16 in, fp32 or bf16 C, one SM per 128×64 tile
    const int want_ck = cfg ? cfg->cluster_k : 0;
    if (want_ck < 0 || want_ck > 4 || want_ck == 3) return TCL_ERR_CONFIG;
    const bool ck_capable = ik == InKind::BF16 && (ok == OutKind::F32 || ok == OutKind::BF16) &&
                            prod == PROD_TMA && want_pair != 2 && !(cfg && cfg->one_cta_per_tile) &&
                            !(cfg && cfg->split_k > 1) && !(cfg && cfg->stages) && (bn == 0 || bn == 64);
    if (want_ck >= 2) {
        if (!ck_capable) return TCL_ERR_CONFIG;
        bn = 64;
    }
    // 64-row tiles: bf16 in, fp32 or bf16 C, one SM per 64×64 tile
    const int want_tm = cfg ? cfg->tile_m : 0;
    if (want_tm != 0 && want_tm != 64 && want_tm != 128) return TCL_ERR_CONFIG;
    bool use_m64 = want_tm == 64;
    if (want_tm == 64) {
        if (!(ik == InKind::BF16 && (ok == OutKind::F32 || ok == OutKind::BF16) && prod == PROD_TMA &&
              want_pair != 2 && !(cfg && cfg->one_cta_per_tile) && !(cfg && cfg->split_k > 1) && want_ck < 2 &&
              !(cfg && cfg->stages) && (bn == 0 || bn == 64)))
            return TCL_ERR_CONFIG;
        bn = 64;
    }
    int pair = 0;
    // the two-SM kernel: bf16 or TF32 in, float out (256 or 224 wide), or the
    // exact-integer mode (256 wide with eight epilogue warps, or 128 wide with
    // four: a thread keeps the int32 sums of one row over 128 columns)
    const bool pair_capable = prod == PROD_TMA && (ok != OutKind::S32 || ik == InKind::BF16);
    const int pair_bn = 256;
    if (want_pair == 2) {
        if (!pair_capable) return TCL_ERR_CONFIG;
        if (ok == OutKind::S32 ? (bn != 0 && bn != 128 && bn != 256) : (bn != 0 && bn != 256 && bn != 224))
            return TCL_ERR_CONFIG;
        pair = 1;
    } else if (want_pair == 0 && pair_capable && bn == 0 && !(cfg && cfg->stages) && want_ck < 2 && want_tm != 64) {
        // Two SMs per 256-row tile halve each SM's bytes per flop, but pay a longer
        // hand-off per tile. Take them when the cheaper of the best two-SM tiling
        // (256 or 224 wide, with the stream-K tail the launch would get; exact
        // integers: 256 wide) beats the best one-SM tiling (exact integers: 128 wide)
        // by the cost model above, and a tile has enough k-blocks for its mainloop to
        // outlast its epilogue (at 4096²×512 one SM per tile is faster, 22.0 against
        // 27.1 µs). A TF32 k-block (32 deep) takes the tensor pipe as long as a bf16
        // one (64 deep) and moves as many bytes, so the same constants serve both.
        // Measured on GB300: 1024×4096×4096 on two-SM 224-wide tiles 25.3 µs against
        // 36.0 on the 128-wide tiles an SM-count threshold chose (TF32 47.0 against
        // 73.6, int8 on two-SM 256-wide tiles 36.9 against 44.7); 3072²×1024 one SM,
        // 256 wide, 19.0 against 20.1 on two SMs.
        const int kblocks = (K + bk - 1) / bk;
        const int cap = cfg && cfg->max_ctas > 0 ? cfg->max_ctas : sms;
        const int pairs = std::max(1, cap / 2);
        const int want_sk = cfg ? cfg->stream_k : 0;
        long long best_pair = -1;
        for (int w : {256, 224}) {
            if (w == 224 && !(ok == OutKind::F32 && want_sk <= 1)) continue;
            const long long t = static_cast<long long>((M + 255) / 256) * ((N + w - 1) / w);
            // (the grid never has more pairs than tiles, so fewer tiles than pairs get no tail)
            const int pe = static_cast<int>(std::min<long long>(pairs, t));
            int skt = 0, skp = 1;
            if (stream_k_split(t, pe, kblocks, want_sk, &skt, &skp)) skt = 0, skp = 1;
            const long long c =
                pair_cost(t, pe, kblocks, w == 256 ? kPairKbCycles256 : kPairKbCycles224, skt, skp) +
                (ok == OutKind::S32 ? kPairFixedCyclesS32 : kPairFixedCycles);
            if (best_pair < 0 || c < best_pair) best_pair = c;
        }
        pair = (kblocks >= kMinKbForPair &&
                best_pair < one_sm_cost(M, N, kblocks, cap, ok == OutKind::S32 ? 128 : 0))
                   ? 1
                   : 0;
    }
    const int want_sk = cfg ? cfg->stream_k : 0;
    // stream-K pieces add into C (fp32, int32) or, for a bf16 C (which must be rounded
    // once), into an fp32 workspace that the last piece adds before rounding
    const bool sk_capable = ok == OutKind::F32 || ok == OutKind::S32 || ok == OutKind::BF16;
    if (want_sk < 0 || want_sk > kSkBalanced || (want_sk > 1 && (!pair || !sk_capable))) return TCL_ERR_CONFIG;
    if (pair) {
        if (bn == 0) {
            // Pair tile width: the fewest SM cycles on the busiest pair of SMs,
            // whole tiles only or with a stream-K tail (fp32 C can also use 224).
            bn = pair_bn;
            if (ok == OutKind::F32 && want_sk <= 1) {   // a requested stream-K split keeps 256
                const int pairs = std::max(1, (cfg && cfg->max_ctas > 0 ? cfg->max_ctas : sms) / 2);
                const int kb = (K + bk - 1) / bk;
                auto cost = [&](int w, long long kb_cycles) {
                    const long long t = static_cast<long long>((M + 255) / 256) * ((N + w - 1) / w);
                    int skt = 0, skp = 1;
                    if (stream_k_split(t, pairs, kb, want_sk, &skt, &skp)) skt = 0;
                    return pair_cost(t, pairs, kb, kb_cycles, skt, skp);
                };
                const int want_st = cfg && cfg->stages ? cfg->stages : deepest_stages(ik, ok, 224, prod, 1);
                if (find_variant(ik, ok, 224, want_st, prod, 1) &&
                    cost(224, kPairKbCycles224) < cost(256, kPairKbCycles256))
                    bn = 224;
            }
        }
    } else if (bn == 0) {
        if (ok == OutKind::S32) {
            bn = 128;
        } else {
            // Wide tiles halve the B traffic per flop; fall back to narrow tiles
            // when wide ones would leave SMs idle, or when a tile is at most 4
            // k-blocks deep: its time is then the latency of its loads, and
            // narrow tiles keep 6 of them in flight instead of 4 (measured on
            // GB300 at 4096²×256: 16.7 against 17.5 µs; at ×512 wide tiles win).
            // A bf16 C halves the stores that follow, and there the wide tiles
            // win at 4 k-blocks too (4096²×256: 12.5 against 12.9 µs).
            const long long tiles256 = static_cast<long long>((M + kBM - 1) / kBM) * ((N + 255) / 256);
            const int kblocks = (K + bk - 1) / bk;
            bn = (tiles256 >= sms && (kblocks > 4 || ok == OutKind::BF16)) ? 256 : 128;
            if (kblocks > 4) {   // beyond 4 k-blocks: by the cost model
                const int cap = cfg && cfg->max_ctas > 0 ? cfg->max_ctas : sms;
                bn = one_sm_cost(M, N, kblocks, cap, 256) <= one_sm_cost(M, N, kblocks, cap, 128) ? 256 : 128;
            }
            // Small grids (128-wide tiles filling at most a quarter of the SMs) too shallow
            // for split-K: 64-wide tiles give twice the CTAs, each with half the B bytes
            // and half the C stores (measured on GB300, CUDA graphs of back-to-back calls
            // at 512²: K = 256 4.37 against 4.98 µs, 512 5.21 against 5.92, 1024 6.74
            // against 7.76), and bf16 operands take 64 rows as well: 64×64 tiles, four
            // times the CTAs of 128×128 ones, half the A bytes per k-block (K = 256 3.90
            // against 4.41 µs for 128×64 tiles, 512 4.75 against 5.26, 1024 6.25
            // against 6.82; from 24 k-blocks split-K stays ahead).
            const long long tiles128 = static_cast<long long>((M + kBM - 1) / kBM) * ((N + 127) / 128);
            const bool split_asked = cfg && cfg->split_k > 1;
            if (bn == 128 && tiles128 * 4 <= sms && kblocks < kMinKbToSplit && !split_asked &&
                !(cfg && cfg->stages) && deepest_stages(ik, ok, 64, prod, 0) > 0) {
                bn = 64;
                if (want_tm == 0 && ik == InKind::BF16 && (ok == OutKind::F32 || ok == OutKind::BF16) &&
                    prod == PROD_TMA && want_ck < 2 && !(cfg && cfg->one_cta_per_tile))
                    use_m64 = true;
            }
        }
    }
    if (bn != 128 && bn != 256 && !(pair && bn == 224) && !(!pair && bn == 64)) return TCL_ERR_CONFIG;
    const int slots = cfg ? cfg->epi_slots : 0;
    if (slots < 0 || (slots && !pair && slots != 2)) return TCL_ERR_CONFIG;
    const int pv = pair ? 1 : 0;   // the variant table's kernel kind (1: two-SM kernel)
    int stages = cfg && cfg->stages ? cfg->stages : deepest_stages(ik, ok, bn, prod, pv, slots);
    const VariantInfo* v = find_variant(ik, ok, bn, stages, prod, pv, slots);
    if (!v) return TCL_ERR_CONFIG;
    pl->slots = v->slots;
    pl->bn = bn;
    pl->stages = stages;
    pl->prod = prod;
    pl->pair = pv;
    pl->smem = v->smem_bytes;
    // 64×64 tiles take two k-blocks per stage (one 3-D tensor copy of A, one of B)
    // when K is whole 64-wide blocks, so that no copy reads past a row's end
    pl->m64 = (use_m64 && !pair) ? (K % 64 == 0 ? 2 : 1) : 0;
    const int bm = pair ? 2 * kBM : pl->m64 ? 64 : kBM;
    pl->tiles_m = (M + bm - 1) / bm;
    pl->tiles_n = (N + bn - 1) / bn;
    const long long tiles = static_cast<long long>(pl->tiles_m) * pl->tiles_n;
    if (tiles > 0x3FFFFFFFll) return TCL_ERR_DIMS;
    pl->num_tiles = static_cast<int>(tiles);
    pl->num_kb = (K + bk - 1) / bk;
    pl->kb_per_unit = ok == OutKind::S32 ? kS32UnitK / bk : pl->num_kb;
    // A tile's K ranges on a cluster of 2 or 4 CTAs, summed through distributed shared
    // memory: on request only. Measured on GB300 at 512² (CUDA graphs of back-to-back
    // calls, round robin), it loses to one CTA per 64-wide tile below K = 2048 (K = 256:
    // 6.4 / 8.1 µs for clusters of 2 / 4 against 4.4) and to split-K with its reduction
    // launch above (K = 4096: 12.2 against 10.5): moving the 32 KB partial tiles between
    // the SMs of a cluster takes ~1 µs each, and a cluster barrier ~0.5 µs.
    if (pl->m64) {   // its own ring (16 KB stages of one k-block, 32 KB of two)
        pl->stages = m64_stages(pl->m64);
        pl->smem = m64_smem_bytes(pl->m64);
    }
    pl->csk = 0;
    if (ck_capable && !pair && bn == 64 && want_ck >= 2) {
        pl->csk = want_ck;
        pl->stages = csk_stages();
        pl->smem = csk_smem_bytes(want_ck);
    }
    // Raster group and K order for deep two-SM tiles (rows of A at least 16 KB
    // long): a wave of tiles then streams more operand bytes than one die's share
    // of L2 keeps, and each wave re-reads what the one before evicted. One row of
    // tiles at a time (group 1: a wave shares all of B and a few rows of A), with
    // every second tile of a CTA's walk taking K in descending order (so that a
    // wave starts on the blocks the previous wave read last, which are still in
    // L2), cut the DRAM reads of bf16 4096²×8192 from 340 to 272 MB and of TF32
    // 4096³ from 339 to 274 MB (ncu, cold L2). Timed round robin under the power
    // cap, the orders stay within 2 % of each other at every deep shape; with
    // shorter rows groups of 8 rows and ascending K are kept.
    const bool deep = pair && static_cast<long long>(pl->num_kb) * bk * in_bytes(ik) >= kMinKBytesForRowRaster;
    pl->group_m = cfg && cfg->group_m > 0 ? cfg->group_m : (deep ? 1 : 8);
    const int want_ko = cfg ? cfg->k_order : 0;
    if (want_ko < 0 || want_ko > 2 || (want_ko == 2 && prod != PROD_TMA)) return TCL_ERR_CONFIG;
    pl->k_serpentine = want_ko == 2 ? 1 : want_ko == 1 ? 0 : (deep ? 1 : 0);
    // int8 on 256-wide pair tiles can widen its operands inside the kernel (no pass
    // over HBM), on request only: measured on GB300 it is slower than the widening
    // pass followed by the bf16-input kernel (4096³: 142 against 95 µs, CUDA graphs
    // of back-to-back calls), its stages being bound by the converter warps'
    // shared-memory traffic and instruction latency
    const int want_s8 = cfg ? cfg->s8_path : 0;
    if (want_s8 < 0 || want_s8 > 2 || (want_s8 && ok != OutKind::S32)) return TCL_ERR_CONFIG;
    pl->s8_in_kernel = (ok == OutKind::S32 && pair && bn == 256 && want_s8 == 2 && !(cfg && cfg->stages) &&
                        !(cfg && cfg->epi_slots > 1))
                           ? 1
                           : 0;
    if (want_s8 == 2 && !pl->s8_in_kernel) return TCL_ERR_CONFIG;
    if (pl->s8_in_kernel) {   // its own ring (fp16 stages fed from raw int8 slots)
        pl->stages = s8_pair_stages();
        pl->smem = s8_pair_smem_bytes();
    }
    // Two-SM 256-wide tiles: one copy of A and one of B bring two k-blocks into two ring slots,
    // halving the tensor copies and byte announcements per k-block (what paces a stage, more
    // than its bytes). The maps cut K and N into whole blocks, so K must be a whole number of
    // k-blocks and N of B boxes (no box may read past a row's end), and the ring even, at
    // least 4. (The same in the one-SM kernel, with its B boxes in one 3-D copy or not, was
    // measured no faster on GB300 at 128×256 and 128×128 tiles.)
    const int want_kps = cfg ? cfg->kblocks_per_stage : 0;
    if (want_kps < 0 || want_kps > 2 || (cfg && (cfg->b_copy < 0 || cfg->b_copy > 1))) return TCL_ERR_CONFIG;
    if (cfg && (cfg->die_split < 0 || cfg->die_split > 2 || (cfg->die_split == 2 && !pair))) return TCL_ERR_CONFIG;
    if (cfg && (cfg->l2_hints < 0 || cfg->l2_hints > 2 || (cfg->l2_hints == 2 && !pair))) return TCL_ERR_CONFIG;
    const bool kps2_ok = pair && !pl->s8_in_kernel && bn == 256 && prod == PROD_TMA && K % bk == 0 &&
                         N % (128 / in_bytes(ik)) == 0 && pl->stages >= 4 && pl->stages % 2 == 0;
    if (want_kps == 2 && !kps2_ok) return TCL_ERR_CONFIG;
    pl->kps = kps2_ok && want_kps != 1 ? 2 : 1;
    // Split-K (one-SM kernel, floating-point output): when the output tiles
    // alone would leave most SMs idle, cut K into ranges computed by different
    // CTAs; a second kernel adds the partial tiles in a fixed order.
    pl->splits = 1;
    pl->kb_per_split = pl->num_kb;
    const int want_split = cfg ? cfg->split_k : 0;
    if (want_split < 0) return TCL_ERR_CONFIG;
    if (want_split > 1 && (pair || ok == OutKind::S32)) return TCL_ERR_CONFIG;
    if (!pair && ok != OutKind::S32 && want_split != 1 && !pl->csk && !pl->m64) {
        int sp = want_split;
        if (sp == 0) {
            const int cap = cfg && cfg->max_ctas > 0 ? cfg->max_ctas : sms;
            sp = (pl->num_tiles < cap / 2 && pl->num_kb >= kMinKbToSplit)
                     ? std::min(cap / pl->num_tiles, pl->num_kb / kMinKbPerSplit)
                     : 1;
        }
        sp = std::max(1, std::min(sp, pl->num_kb));
        pl->kb_per_split = (pl->num_kb + sp - 1) / sp;
        pl->splits = (pl->num_kb + pl->kb_per_split - 1) / pl->kb_per_split;
        if (pl->splits > 1) {
            // the partial tiles are fp32: the kernel runs in its fp32-output form
            const VariantInfo* v32 = find_variant(ik, OutKind::F32, bn, stages, prod, pv);
            if (!v32) return TCL_ERR_CONFIG;
            pl->smem = v32->smem_bytes;
        }
    }
    const long long work = static_cast<long long>(pl->num_tiles) * pl->splits;
    pl->sk_tiles = 0;
    pl->sk_pieces = 1;
    pl->sk_ws_rows = 0;
    pl->sk_balanced = pl->sk_first = pl->sk_region = 0;
    pl->die_split = 0;
    pl->l2_hints = 0;
    pl->sub_rs = 0;
    for (int h = 0; h < 2; ++h)
        pl->sub_n[h] = pl->sub_a[h] = pl->sub_s[h] = pl->sub_b[h] = pl->sub_u[h] = pl->sub_tiles[h] =
            pl->sub_sk_tiles[h] = 0;
    for (int h = 0; h < 2; ++h) pl->sub_sk_pieces[h] = 1;
    if (pair) {
        const int cl = 2;   // CTAs per cluster: one pair
        int clusters = cfg && cfg->max_ctas > 0 ? cfg->max_ctas / cl : pair_clusters(v);
        if (clusters < 1) return cfg && cfg->max_ctas > 0 ? TCL_ERR_CONFIG : TCL_ERR_LAUNCH;
        if (cfg && cfg->one_cta_per_tile) clusters = pl->num_tiles;
        pl->grid = cl * (pl->num_tiles < clusters ? pl->num_tiles : clusters);
        // Stream-K pieces wait on one another, so every pair of the grid must be
        // resident at once: the grid never exceeds the resident clusters here.
        if (sk_capable && !(cfg && cfg->one_cta_per_tile)) {
            // (a bf16 C adds its workspace round trip, yet the same threshold holds: measured
            // on GB300 at 4096², the tail against none at K = 2048 42.2 vs 42.2 µs, at 3072
            // 58.3 vs 59.7, at 4096 75.7 vs 78.1)
            const int pairs = pl->grid / cl;
            const int st = want_sk == kSkBalanced ? TCL_OK
                                                  : stream_k_split(pl->num_tiles, pairs, pl->num_kb, want_sk,
                                                                   &pl->sk_tiles, &pl->sk_pieces);
            if (st) return st;
            // Balanced stream-K (on request): every pair gets the same number of k-blocks,
            // ranges crossing tile boundaries. It shortens the busiest pair's walk at 4096³
            // (216 against 224 k-blocks) but was measured slower on GB300 (CUDA graphs,
            // round robin: 91.3 against 83.1 µs for an fp32 C, 87.6 against 83.1 for a bf16
            // C, 174.8 against 167.1 at 4096²×8192, 50.5 against 45.0 at 4096²×2048): the
            // 72 cut tiles' extra stores and reductions land together at the end of the
            // launch, where the equal-piece tail has 28.
            const Balanced bs = balanced_split(pl->num_tiles, pairs, pl->num_kb);
            if (want_sk == kSkBalanced) {
                if (!bs.region || pairs - 1 > kMaxSkTiles) {   // flags and workspace per range boundary
                    if (want_sk == kSkBalanced) return TCL_ERR_CONFIG;
                } else {
                    pl->sk_balanced = 1;
                    pl->sk_first = bs.first;
                    pl->sk_region = bs.region;
                    pl->sk_tiles = bs.split;
                    pl->sk_pieces = 2;
                }
            }
            if (pl->sk_tiles > kMaxSkTiles) {   // the progress flags hold kMaxSkTiles tiles
                if (want_sk > 1) return TCL_ERR_CONFIG;
                pl->sk_tiles = 0;
                pl->sk_pieces = 1;
                pl->sk_balanced = 0;
            }
            const int resident = cfg && cfg->max_ctas > 0 ? pair_clusters(v) : pl->grid / cl;   // 0: no device
            if ((pl->sk_tiles || pl->sk_balanced) && resident > 0 && pl->grid / cl > resident) {
                if (want_sk > 1) return TCL_ERR_CONFIG;
                pl->sk_tiles = 0;
                pl->sk_pieces = 1;
                pl->sk_balanced = 0;
            }
        }
        // Die split: each die's pairs walk their own block of tile columns, row by row, with
        // its own stream-K tail, so that each die's half of the L2 holds the operands of its
        // own tiles: each die's L2 keeps what its SMs read, so a wave whose pairs span all
        // of B holds B twice. The block is whole columns plus part of one (cut at a tile
        // row), so that each die's tile count follows its pairs to the tile (the dies of a
        // GB300 need not have equal pairs). Automatic where each die's block is at most about
        // 8 tile columns wide (a wave then covers whole rows of it) and holds at least 3 waves
        // of tiles. Measured on GB300 (CUDA graphs, on and off alternating in one process):
        // dies of 36 and 40 pairs, bf16 4096³ 81.4 against 83.3 µs, bf16 C 83.1 against 84.5,
        // int8 98.4 against 99.5, TF32 4096³ and 4096²×8192 within 0.5 and 0.9 % with 5–7 %
        // less HBM traffic; dies of 38 and 38, 6144×4096×4096 124.5 against 130.4, 4096²×3072
        // 66.1 against 68.0, 8192×4096×4096 164.2 against 166.8. Wider blocks (8192³ 3 %
        // slower) and shorter grids (128–144 tiles: up to 4.5 % slower) keep the whole grid.
        const int want_ds = cfg ? cfg->die_split : 0;
        if (want_ds < 0 || want_ds > 2) return TCL_ERR_CONFIG;
        const int pairs_all = pl->grid / cl;
        const bool ds_ok = die_pairs && die_pairs[0] > 0 && die_pairs[1] > 0 &&
                           die_pairs[0] + die_pairs[1] == pairs_all && pairs_all >= kMinDieSplitPairs &&
                           !pl->sk_balanced && !pl->s8_in_kernel &&
                           pl->tiles_n >= 2 && !(cfg && cfg->one_cta_per_tile);
        if (want_ds == 2 && !ds_ok) return TCL_ERR_CONFIG;
        // (a requested raster group keeps the whole grid unless the split is asked for too:
        // the blocks are walked row by row)
        const bool ds_auto = want_ds == 0 && pl->tiles_n <= kMaxDieSplitCols &&
                             pl->num_tiles >= kMinDieSplitWaves * pairs_all && pl->num_kb >= kMinDieSplitKb &&
                             !(cfg && cfg->group_m > 0);
        if (ds_ok && (want_ds == 2 || ds_auto)) {
            const int n0 = die_pairs[0], n1 = die_pairs[1];
            const long long all = static_cast<long long>(pl->tiles_m) * pl->tiles_n;
            long long t0 = (all * n0 + (n0 + n1) / 2) / (n0 + n1);
            t0 = std::max(1ll, std::min(t0, all - 1));
            const int c0 = static_cast<int>(t0 / pl->tiles_m);   // whole columns of die 0
            pl->die_split = 1;
            pl->sub_n[0] = n0;
            pl->sub_n[1] = n1;
            pl->sub_rs = static_cast<int>(t0 % pl->tiles_m);        // rows of column c0 that are die 0's
            pl->sub_a[0] = c0 + 1, pl->sub_s[0] = 0, pl->sub_b[0] = c0, pl->sub_u[0] = 0;
            pl->sub_a[1] = pl->tiles_n - c0 - 1, pl->sub_s[1] = c0 + 1, pl->sub_b[1] = pl->tiles_n - c0,
            pl->sub_u[1] = c0;
            int total_sk = 0;
            for (int h = 0; h < 2; ++h) {
                const long long t = static_cast<long long>(pl->sub_rs) * pl->sub_a[h] +
                                    static_cast<long long>(pl->tiles_m - pl->sub_rs) * pl->sub_b[h];
                pl->sub_tiles[h] = static_cast<int>(t);
                int skt = 0, skp = 1;
                if (sk_capable && want_sk != 1 &&
                    stream_k_split(t, static_cast<int>(std::min<long long>(pl->sub_n[h], t)), pl->num_kb,
                                   want_sk, &skt, &skp))
                    skt = 0, skp = 1;
                pl->sub_sk_tiles[h] = skt;
                pl->sub_sk_pieces[h] = skp;
                total_sk += skt;
            }
            if (total_sk > kMaxSkTiles) {
                for (int h = 0; h < 2; ++h) pl->sub_sk_tiles[h] = 0, pl->sub_sk_pieces[h] = 1;
                total_sk = 0;
            }
            pl->sk_tiles = total_sk;
            pl->sk_pieces = std::max(pl->sub_sk_pieces[0], pl->sub_sk_pieces[1]);
            pl->group_m = 1;   // the sub-grids are walked row by row
        }
        // L2 eviction priorities on the operand loads: under the die split, every wave of a
        // die's pairs shares that die's B columns while its rows of A are new, so A's loads
        // are marked evict-first and B's evict-last. For deep tiles (rows of A of at least
        // 16 KB) on GB300: bf16 4096²×8192 HBM traffic 1.51 → 1.31× the algorithmic bytes
        // and 172.0 → 169.6 µs, TF32 4096³ 1.51 → 1.35× and 170.4 → 168.2 µs; shorter rows
        // (4096³: 88.8 → 90.9 µs) and the whole grid (8192³: 5 % slower) keep plain loads.
        const int want_h = cfg ? cfg->l2_hints : 0;
        if (want_h == 2 && pl->s8_in_kernel) return TCL_ERR_CONFIG;
        pl->l2_hints = !pl->s8_in_kernel && (want_h == 2 || (want_h == 0 && pl->die_split && deep)) ? 1 : 0;
        // a bf16 C's fp32 workspace: one block per split tile (per range boundary when balanced)
        if (ok == OutKind::BF16 && (pl->sk_tiles || pl->sk_balanced))
            pl->sk_ws_rows = (pl->sk_balanced ? pl->grid / cl : pl->sk_tiles) * 2 * kBM;
    } else if (want_sk > 1) {
        return TCL_ERR_CONFIG;
    } else if (cfg && cfg->one_cta_per_tile) {
        pl->grid = static_cast<int>(std::min<long long>(work, 0x7FFFFFFF));
    } else if (pl->m64) {
        pl->grid = pl->num_tiles;   // one CTA per tile
    } else if (pl->csk) {
        const long long ctas = static_cast<long long>(pl->num_tiles) * pl->csk;   // one cluster per tile
        if (ctas > 0x7FFFFFFFll) return TCL_ERR_DIMS;
        pl->grid = static_cast<int>(ctas);
    } else {
        int cap = cfg && cfg->max_ctas > 0 ? cfg->max_ctas : sms;
        if (cap < 1) cap = 1;
        pl->grid = static_cast<int>(std::min<long long>(work, cap));
    }
    return TCL_OK;
}

// Split-K workspace: `splits` fp32 slabs of round_up(M, 128) rows × round_up(N, 4) columns;
// or, for a bf16 C with a stream-K tail, sk_ws_rows × bn fp32 (blocks of 32 rows,
// each laid out for one epilogue warp's coalesced 16-byte accesses).
struct Workspace {
    long long ld, rows_per_split;
    size_t bytes;
};

Workspace split_workspace(const Plan& pl, int M, int N) {
    Workspace w{0, 0, 0};
    if (pl.splits > 1) {
        w.ld = round_up(N, 4);
        w.rows_per_split = round_up(M, kBM);
        w.bytes = static_cast<size_t>(round_up(w.ld * w.rows_per_split * 4 * pl.splits, 256));
    } else if (pl.sk_ws_rows) {
        w.bytes = static_cast<size_t>(round_up(static_cast<long long>(pl.sk_ws_rows) * pl.bn * 4, 256));
    }
    return w;
}

// Resident pair clusters for a pair variant on the current device, queried once.
int device_pair_clusters(DevState* ds, const VariantInfo* v) {
    int idx = 0;
    for (const auto& w : kVariants) {
        if (&w == v) break;
        if (w.pair) ++idx;
    }
    if (idx >= 16) return 0;
    if (ds->pair_clusters[idx] == 0)
        ds->pair_clusters[idx] = pair_max_clusters(v->in, v->out, v->bn, v->stages, v->slots);
    return ds->pair_clusters[idx];
}

// Which die each pair of SMs is on (k_diemap.cu), measured at the first call that is
// not being captured (the measurement allocates and synchronises); up to three tries.
void ensure_die_map(DevState* ds, cudaStream_t stream) {
    if (ds->die_state > 0 || ds->die_state <= -3) return;
    int st = TCL_OK;
    if (is_capturing(stream, &st) || st) return;
    int n0 = 0, n1 = 0;
    if (calibrate_die_map(ds->sms, ds->die_of_tpc, 128, &n0, &n1)) {
        ds->die_pairs[0] = n0;
        ds->die_pairs[1] = n1;
        ds->die_state = 1;
    } else {
        ds->die_pairs[0] = ds->die_pairs[1] = 0;
        --ds->die_state;
    }
}

int plan_on_device(InKind ik, OutKind ok, int M, int N, int K, const tcl_config_t* cfg, DevState* ds, Plan* pl) {
    const int pairs[2] = {ds->die_pairs[0], ds->die_pairs[1]};
    return make_plan(ik, ok, M, N, K, cfg, ds->sms,
                     [ds](const VariantInfo* v) { return device_pair_clusters(ds, v); }, pairs, pl);
}

// Builds tensor maps and launches one GEMM over device operands (and, for a
// split-K plan, the reduction of the partial tiles from `workspace` into C).
int run_gemm(const Plan& pl, InKind ik, OutKind ok, int M, int N, int K, const void* A, long long lda,
             const void* B, long long ldb, void* C, long long ldc, void* workspace, const tcl_config_t* cfg,
             int dev, DevState* ds, StreamRes* sr, cudaStream_t stream) {
    int st;
    const Workspace ws = split_workspace(pl, M, N);
    const bool split = pl.splits > 1;
    const OutKind kernel_out = split ? OutKind::F32 : ok;
    const int ies = in_bytes(ik), oes = out_bytes(kernel_out);
    const int bk = 128 / ies;
    const CUtensorMapDataType in_t =
        ik == InKind::TF32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const CUtensorMapDataType out_t = kernel_out == OutKind::F32    ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                      : kernel_out == OutKind::BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                                    : CU_TENSOR_MAP_DATA_TYPE_INT32;
    LaunchArgs a;
    a.in = ik;
    a.out = kernel_out;
    a.bn = pl.bn;
    a.stages = pl.stages;
    a.prod = pl.prod;
    a.pair = pl.pair;
    a.slots = pl.slots;
    a.csk = pl.csk;
    a.m64 = pl.m64;
    a.pdl = !(cfg && cfg->serial_launch);
    a.grid = pl.grid;
    a.stream = stream;
    // A CTA's B boxes of a k-block (the whole tile's, or a two-SM CTA's half) come in one
    // tensor copy (a 3-D map) when N is a whole number of boxes, so that no box reads past a
    // row's end: a stage's copies, not its bytes, pace the stages (measured on GB300)
    // (a two-SM CTA's half starts at a multiple of 128 columns only in 256-wide tiles; the
    // third coordinate of the map counts whole boxes)
    const int b_boxes = (pl.pair ? pl.bn / 2 : pl.bn) / (128 / ies);   // per CTA and k-block
    const bool b3d = pl.kps == 1 && !pl.s8_in_kernel && !pl.m64 && !pl.csk && pl.prod == PROD_TMA && b_boxes > 1 &&
                     (!pl.pair || pl.bn == 256) && N % (128 / ies) == 0 && !(cfg && cfg->b_copy == 1);
    if (pl.s8_in_kernel) {
        // raw int8 operands, unswizzled: A in boxes of 64 K × 128 rows, B of 128 columns × 64 K
        if ((st = tensor_map(dev, A, CU_TENSOR_MAP_DATA_TYPE_UINT8, K, M, lda, 64, kBM, &a.tmA,
                             CU_TENSOR_MAP_SWIZZLE_NONE)) ||
            (st = tensor_map(dev, B, CU_TENSOR_MAP_DATA_TYPE_UINT8, N, K, ldb, 128, 64, &a.tmB,
                             CU_TENSOR_MAP_SWIZZLE_NONE)))
            return st;
    } else {
        const CUtensorMapSwizzle bswz =
            ik == InKind::TF32 ? CU_TENSOR_MAP_SWIZZLE_128B_ATOM_32B : CU_TENSOR_MAP_SWIZZLE_128B;
        if (pl.kps == 2) {
            // A as (K of a block, rows, k-blocks) in boxes of 128 rows × 2 blocks; B as (a box's
            // columns, K of a block, column blocks, k-blocks) in boxes of a CTA's half × 2 blocks
            const uint32_t bw = 128 / ies;
            if ((st = tensor_map_3d(dev, A, in_t, bk, M, K / bk, lda * ies, 128, bk, kBM, 2, &a.tmA)) ||
                (st = tensor_map_nd(dev, B, in_t, bw, bk, N / bw, K / bk, ldb * ies, 128,
                                    static_cast<uint64_t>(bk) * ldb * ies, bw, bk, static_cast<uint32_t>(b_boxes), 2,
                                    &a.tmB, bswz)))
                return st;
        } else if (pl.m64 == 2) {
            // A as (64 K, M rows, K/64 k-blocks): one box brings two k-blocks' swizzle tiles;
            // B in boxes of 128 K-rows
            if ((st = tensor_map_3d(dev, A, in_t, bk, M, K / bk, lda * ies, 128, bk, 64, 2, &a.tmA)) ||
                (st = tensor_map(dev, B, in_t, N, K, ldb * ies, 128 / ies, 2 * bk, &a.tmB)))
                return st;
        } else {
            if ((st = tensor_map(dev, A, in_t, K, M, lda * ies, bk, pl.m64 ? 64 : kBM, &a.tmA))) return st;
            // B N-major (K rows of N) in boxes of one 128-byte row of N × bk rows; TF32's
            // 4-byte elements are swizzled in 32-byte units (bswz), the form the tensor core
            // reads an N-major 32-bit operand in
            if (b3d) {
                // (columns of a box, K, column blocks): one box holds all of a CTA's B boxes
                const uint32_t bw = 128 / ies;
                if ((st = tensor_map_3d(dev, B, in_t, bw, K, N / bw, ldb * ies, 128, bw, bk,
                                        static_cast<uint32_t>(b_boxes), &a.tmB, bswz)))
                    return st;
            } else if ((st = tensor_map(dev, B, in_t, N, K, ldb * ies, 128 / ies, bk, &a.tmB, bswz))) {
                return st;
            }
        }
    }
    void* out_ptr = split ? workspace : C;
    const long long out_ld = split ? ws.ld : ldc;
    const long long out_rows = split ? ws.rows_per_split * pl.splits : M;
    if ((st = tensor_map(dev, out_ptr, out_t, N, static_cast<uint64_t>(out_rows), out_ld * oes, 128 / oes, 32,
                         &a.tmC)))
        return st;
    GemmParams& p = a.p;
    p.M = M;
    p.N = N;
    p.K = K;
    p.tiles_m = pl.tiles_m;
    p.tiles_n = pl.tiles_n;
    p.num_tiles = pl.num_tiles;
    p.num_kb = pl.num_kb;
    p.kb_per_unit = pl.kb_per_unit;
    p.group_m = pl.group_m;
    p.timeout_ns = cfg && cfg->timeout_ns ? cfg->timeout_ns : kDefaultTimeoutNs;
    p.status = ds->status;
    p.trace = cfg ? cfg->trace : nullptr;
    p.trace_cap = cfg && cfg->trace ? cfg->trace_cap : 0;
    p.C = out_ptr;
    p.ldc = out_ld;
    p.splits = pl.splits;
    p.kb_per_split = pl.kb_per_split;
    p.split_rows = split ? static_cast<int>(ws.rows_per_split) : 0;
    p.out_rows = static_cast<int>(out_rows);
    p.A = A;
    p.lda = lda;
    p.B = B;
    p.ldb = ldb;
    p.debug_skip_kb = cfg && cfg->debug_skip_kblock > 0 ? cfg->debug_skip_kblock - 1 : -1;
    p.sk_tiles = pl.sk_tiles;
    p.sk_pieces = pl.sk_pieces;
    p.sk_balanced = pl.sk_balanced;
    p.sk_first = pl.sk_first;
    p.sk_region = pl.sk_region;
    p.debug_sk_stall = cfg && cfg->debug_stream_k_stall ? 1 : 0;
    p.sk_flags = sr->sk_flags;
    p.sk_gen = 0;
    p.sk_ws = nullptr;
    p.sk_ws_rows = 0;
    p.k_serpentine = pl.k_serpentine;
    p.b_3d = b3d ? 1 : 0;
    p.kps2 = pl.kps == 2 ? 1 : 0;
    p.die_split = pl.die_split;
    p.l2_hints = pl.l2_hints;
    p.sub_rs = pl.sub_rs;
    for (int h = 0; h < 2; ++h) {
        p.sub_n[h] = pl.sub_n[h];
        p.sub_a[h] = pl.sub_a[h];
        p.sub_s[h] = pl.sub_s[h];
        p.sub_b[h] = pl.sub_b[h];
        p.sub_u[h] = pl.sub_u[h];
        p.sub_sk_tiles[h] = pl.sub_sk_tiles[h];
        p.sub_sk_pieces[h] = pl.sub_sk_pieces[h];
    }
    p.sched_ctr = sr->sched_ctr;
    std::memcpy(p.die_of_tpc, ds->die_of_tpc, sizeof p.die_of_tpc);
    if (pl.sk_ws_rows) {   // (16-byte accesses: the workspace starts on a 256-byte boundary)
        p.sk_ws = static_cast<float*>(workspace);
        p.sk_ws_rows = pl.sk_ws_rows;
    }
    if (pl.sk_tiles || pl.sk_balanced) {
        sr->sk_gen = (sr->sk_gen + 1) & 0x1FFFFFFFu;   // flags hold gen·8 + pieces done in 32 bits
        if (sr->sk_gen == 0) sr->sk_gen = 1;           // 0 is what the flags start as
        p.sk_gen = sr->sk_gen;
    }

    bool found = false;
    cudaError_t err = cudaSuccess;
    if (pl.s8_in_kernel) {
        found = true;
        err = launch_s8_pair(a);
    } else if (pl.csk) {
        err = launch_csk(a, &found);
    } else if (pl.m64) {
        err = launch_m64(a, &found);
    } else if (pl.pair) {
        err = launch_group_pair(a, &found);
    } else if (ik == InKind::TF32) {
        err = launch_group_tf32(a, &found);
    } else {
        err = launch_group_bf16_f32_bn256(a, &found);
        if (!found) err = launch_group_bf16_f32_bn128(a, &found);
        if (!found) err = launch_group_bf16_misc(a, &found);
        if (!found) err = launch_group_bf16_sync(a, &found);
        if (!found) err = launch_group_bf16_cpasync(a, &found);
    }
    if (!found) return TCL_ERR_CONFIG;
    if (err != cudaSuccess) {
        cudaGetLastError();
        return TCL_ERR_LAUNCH;
    }
    if (split && launch_splitk_reduce(static_cast<const float*>(workspace), ws.ld, ws.rows_per_split, pl.splits, C,
                                      ldc, M, N, ok == OutKind::BF16 ? 1 : 0, ds->sms, stream) != cudaSuccess) {
        cudaGetLastError();
        return TCL_ERR_LAUNCH;
    }
    return TCL_OK;
}

// Scratch layout of one call: packed copies of the operands and output that
// are off the 16-byte grid (each 256-byte aligned), then the split-K
// workspace. Sized before anything is enqueued: growing the scratch frees the
// old buffer.
struct Carve {
    uint8_t* base;
    size_t used;
    void* take(size_t bytes) {
        if (!bytes) return nullptr;
        void* p = base + used;
        used += static_cast<size_t>(round_up(static_cast<long long>(bytes), 256));
        return p;
    }
};

int gemm_bf16_impl(int M, int N, int K, const void* A, int lda, const void* B, int ldb, void* C,
                   int ldc, int out, const tcl_config_t* cfg, cudaStream_t stream) {
    int st = check_common(M, N, K, A, lda, B, ldb, C, ldc);
    if (st) return st;
    if (out != TCL_OUT_F32 && out != TCL_OUT_BF16) return TCL_ERR_CONFIG;
    const int oes = out == TCL_OUT_BF16 ? 2 : 4;
    if (!aligned_to(A, 2) || !aligned_to(B, 2) || !aligned_to(C, oes)) return TCL_ERR_ALIGN;
    // Tensor copies need 16-byte aligned bases and row pitches, and whole
    // 16-byte pieces of K in a row of A: operands that miss any of these are
    // repacked (K zero-padded to a multiple of 8), an output that misses them is
    // computed into scratch and copied out.
    const bool pack_a = !aligned16(A) || lda % 8 || K % 8;
    const bool pack_b = !aligned16(B) || ldb % 8 || K % 8;
    const bool pack_c = !aligned16(C) || ldc % (16 / oes);
    const int K2 = static_cast<int>(round_up(K, 8));
    const long long lda2 = K2, ldb2 = round_up(N, 8), ldc2 = round_up(N, 16 / oes);
    std::lock_guard<std::mutex> lock(g_mu);
    int dev;
    DevState* ds;
    if ((st = current_device(&dev, &ds))) return st;
    const OutKind ok = out == TCL_OUT_BF16 ? OutKind::BF16 : OutKind::F32;
    StreamRes* sr;
    if ((st = stream_res(ds, stream, &sr))) return st;
    Plan pl;
    ensure_die_map(ds, stream);
    if ((st = plan_on_device(InKind::BF16, ok, M, N, K2, cfg, ds, &pl))) return st;
    const size_t a_bytes = pack_a ? static_cast<size_t>(M) * lda2 * 2 : 0;
    const size_t b_bytes = pack_b ? static_cast<size_t>(K2) * ldb2 * 2 : 0;
    const size_t c_bytes = pack_c ? static_cast<size_t>(M) * ldc2 * oes : 0;
    const Workspace ws = split_workspace(pl, M, N);
    const size_t need = static_cast<size_t>(round_up(a_bytes, 256) + round_up(b_bytes, 256) +
                                            round_up(c_bytes, 256)) + ws.bytes;
    if (need && (st = ensure_scratch(ds, sr, need, stream))) return st;
    Carve cv{static_cast<uint8_t*>(sr->scratch), 0};
    void* a2 = cv.take(a_bytes);
    void* b2 = cv.take(b_bytes);
    void* c2 = cv.take(c_bytes);
    void* wsp = cv.take(ws.bytes);
    if ((pack_a && launch_repack(A, lda, M, K, a2, lda2, M, K2, 2, ds->sms, stream) != cudaSuccess) ||
        (pack_b && launch_repack(B, ldb, K, N, b2, ldb2, K2, N, 2, ds->sms, stream) != cudaSuccess)) {
        cudaGetLastError();
        return TCL_ERR_LAUNCH;
    }
    st = run_gemm(pl, InKind::BF16, ok, M, N, K2, pack_a ? a2 : A, pack_a ? lda2 : lda, pack_b ? b2 : B,
                  pack_b ? ldb2 : ldb, pack_c ? c2 : C, pack_c ? ldc2 : ldc, wsp, cfg, dev, ds, sr, stream);
    if (st) return st;
    if (pack_c && launch_repack(c2, ldc2, M, N, C, ldc, M, N, oes, ds->sms, stream) != cudaSuccess) {
        cudaGetLastError();
        return TCL_ERR_LAUNCH;
    }
    return TCL_OK;
}

int gemm_tf32_impl(int M, int N, int K, const float* A, int lda, const float* B, int ldb, float* C,
                   int ldc, const tcl_config_t* cfg, cudaStream_t stream) {
    int st = check_common(M, N, K, A, lda, B, ldb, C, ldc);
    if (st) return st;
    if (!aligned_to(A, 4) || !aligned_to(B, 4) || !aligned_to(C, 4)) return TCL_ERR_ALIGN;
    // As for bf16: operands off the tensor copies' 16-byte grid are repacked (K
    // zero-padded to a multiple of 4, in A's columns and B's rows), an off-grid
    // output goes through scratch. Both operands are read in place otherwise:
    // A K-major, B N-major straight from the row-major K×N matrix.
    const bool pack_a = !aligned16(A) || lda % 4 || K % 4;
    const bool pack_b = !aligned16(B) || ldb % 4 || K % 4;
    const bool pack_c = !aligned16(C) || ldc % 4;
    const int K4 = static_cast<int>(round_up(K, 4));
    const long long ldb2 = round_up(N, 4), ldc2 = round_up(N, 4);
    std::lock_guard<std::mutex> lock(g_mu);
    int dev;
    DevState* ds;
    if ((st = current_device(&dev, &ds))) return st;
    StreamRes* sr;
    if ((st = stream_res(ds, stream, &sr))) return st;
    Plan pl;
    ensure_die_map(ds, stream);
    if ((st = plan_on_device(InKind::TF32, OutKind::F32, M, N, K4, cfg, ds, &pl))) return st;
    const size_t a_bytes = pack_a ? static_cast<size_t>(M) * K4 * 4 : 0;
    const size_t b_bytes = pack_b ? static_cast<size_t>(K4) * ldb2 * 4 : 0;
    const size_t c_bytes = pack_c ? static_cast<size_t>(M) * ldc2 * 4 : 0;
    const Workspace ws = split_workspace(pl, M, N);
    const size_t need = static_cast<size_t>(round_up(a_bytes, 256) + round_up(b_bytes, 256) +
                                            round_up(c_bytes, 256)) + ws.bytes;
    if (need && (st = ensure_scratch(ds, sr, need, stream))) return st;
    Carve cv{static_cast<uint8_t*>(sr->scratch), 0};
    void* a2 = cv.take(a_bytes);
    void* b2 = cv.take(b_bytes);
    void* c2 = cv.take(c_bytes);
    void* wsp = cv.take(ws.bytes);
    if ((pack_a && launch_repack(A, lda, M, K, a2, K4, M, K4, 4, ds->sms, stream) != cudaSuccess) ||
        (pack_b && launch_repack(B, ldb, K, N, b2, ldb2, K4, N, 4, ds->sms, stream) != cudaSuccess)) {
        cudaGetLastError();
        return TCL_ERR_LAUNCH;
    }
    st = run_gemm(pl, InKind::TF32, OutKind::F32, M, N, K4, pack_a ? a2 : A, pack_a ? K4 : lda, pack_b ? b2 : B,
                  pack_b ? ldb2 : ldb, pack_c ? c2 : C, pack_c ? ldc2 : ldc, wsp, cfg, dev, ds, sr, stream);
    if (st) return st;
    if (pack_c && launch_repack(c2, ldc2, M, N, C, ldc, M, N, 4, ds->sms, stream) != cudaSuccess) {
        cudaGetLastError();
        return TCL_ERR_LAUNCH;
    }
    return TCL_OK;
}


int gemm_s8_impl(int M, int N, int K, const int8_t* A, int lda, const int8_t* B, int ldb, int32_t* C,
                 int ldc, const tcl_config_t* cfg, cudaStream_t stream) {
    int st = check_common(M, N, K, A, lda, B, ldb, C, ldc);
    if (st) return st;
    if (!aligned_to(C, 4)) return TCL_ERR_ALIGN;   // int8 operands: any alignment (repacked when needed)
    if (K > 131071) return TCL_ERR_K_TOO_LARGE;
    const bool pack_c = !aligned16(C) || ldc % 4;
    const long long ldc2 = round_up(N, 4);
    std::lock_guard<std::mutex> lock(g_mu);
    int dev;
    DevState* ds;
    if ((st = current_device(&dev, &ds))) return st;
    StreamRes* sr;
    if ((st = stream_res(ds, stream, &sr))) return st;
    Plan pl;
    ensure_die_map(ds, stream);
    if ((st = plan_on_device(InKind::BF16, OutKind::S32, M, N, K, cfg, ds, &pl))) return st;
    // The in-kernel widening copies the int8 rows with tensor copies: 16-byte rows only.
    if (pl.s8_in_kernel && !(aligned16(A) && aligned16(B) && lda % 16 == 0 && ldb % 16 == 0)) return TCL_ERR_ALIGN;
    const long long c_bytes = pack_c ? round_up(static_cast<long long>(M) * ldc2 * 4, 256) : 0;
    int32_t* c2 = nullptr;
    if (pl.s8_in_kernel) {
        if (c_bytes && (st = ensure_scratch(ds, sr, static_cast<size_t>(c_bytes), stream))) return st;
        if (pack_c) c2 = static_cast<int32_t*>(sr->scratch);
        st = run_gemm(pl, InKind::BF16, OutKind::S32, M, N, K, A, lda, B, ldb, pack_c ? c2 : C, pack_c ? ldc2 : ldc,
                      nullptr, cfg, dev, ds, sr, stream);
    } else {
        // Packed bf16 copies of A (M × lda2) and B (K × ldb2), each 256-byte aligned.
        const long long lda2 = round_up(K, 8), ldb2 = round_up(N, 8);
        const long long a_bytes = round_up(static_cast<long long>(M) * lda2 * 2, 256);
        const long long b_bytes = round_up(static_cast<long long>(K) * ldb2 * 2, 256);
        if ((st = ensure_scratch(ds, sr, static_cast<size_t>(a_bytes + b_bytes + c_bytes), stream))) return st;
        uint8_t* a2 = static_cast<uint8_t*>(sr->scratch);
        uint8_t* b2 = a2 + a_bytes;
        if (pack_c) c2 = reinterpret_cast<int32_t*>(b2 + b_bytes);
        if (launch_s8_to_bf16({A, lda, reinterpret_cast<uint16_t*>(a2), lda2, M, K, 0},
                              {B, ldb, reinterpret_cast<uint16_t*>(b2), ldb2, K, N, 0}, ds->sms,
                              stream) != cudaSuccess) {
            cudaGetLastError();
            return TCL_ERR_LAUNCH;
        }
        st = run_gemm(pl, InKind::BF16, OutKind::S32, M, N, K, a2, lda2, b2, ldb2, pack_c ? c2 : C,
                      pack_c ? ldc2 : ldc, nullptr, cfg, dev, ds, sr, stream);
    }
    if (st) return st;
    if (pack_c && launch_repack(c2, ldc2, M, N, C, ldc, M, N, 4, ds->sms, stream) != cudaSuccess) {
        cudaGetLastError();
        return TCL_ERR_LAUNCH;
    }
    return TCL_OK;
}

// Streams of the host-buffer entry points, created once per device.
int ensure_host_streams(DevState* ds) {
    if (ds->up) return TCL_OK;
    cudaStream_t s[3] = {nullptr, nullptr, nullptr};
    for (auto& x : s) {
        if (cudaStreamCreateWithFlags(&x, cudaStreamNonBlocking) != cudaSuccess) {
            cudaGetLastError();
            for (auto& y : s)
                if (y) cudaStreamDestroy(y);
            return TCL_ERR_LAUNCH;
        }
    }
    ds->up = s[0];
    ds->comp = s[1];
    ds->down = s[2];
    return TCL_OK;
}

// C = A·B with A, B and C in host memory (bf16 in, fp32 or bf16 out). B is
// uploaded whole; A and C move in row chunks on separate streams so that the
// upload of chunk i+1, the GEMM of chunk i and the download of chunk i-1
// overlap. The whole pipeline is ordered after earlier work on `stream` and
// `stream` waits for its end, so the call behaves like the device-pointer
// entry points on that stream.
int gemm_bf16_host_impl(int M, int N, int K, const void* A, int lda, const void* B, int ldb, void* C, int ldc,
                        int out, const tcl_config_t* cfg, cudaStream_t stream) {
    int st = check_common(M, N, K, A, lda, B, ldb, C, ldc);
    if (st) return st;
    if (out != TCL_OUT_F32 && out != TCL_OUT_BF16) return TCL_ERR_CONFIG;
    const int oes = out == TCL_OUT_BF16 ? 2 : 4;
    if (!aligned_to(A, 2) || !aligned_to(B, 2) || !aligned_to(C, oes)) return TCL_ERR_ALIGN;
    const OutKind ok = out == TCL_OUT_BF16 ? OutKind::BF16 : OutKind::F32;
    std::lock_guard<std::mutex> lock(g_mu);
    int dev;
    DevState* ds;
    if ((st = current_device(&dev, &ds))) return st;
    if ((st = ensure_host_streams(ds))) return st;
    // all of this path's work runs on the library's own streams: its scratch and
    // flags are those of its GEMM stream
    StreamRes* sr;
    if ((st = stream_res(ds, ds->comp, &sr))) return st;
    // device copies with tensor-copy pitches, K zero-padded to a multiple of 8
    const int K2 = static_cast<int>(round_up(K, 8));
    const long long lda2 = K2, ldb2 = round_up(N, 8), ldc2 = round_up(N, 16 / oes);
    // up to eight row chunks of at least 512 rows (whole 256-row tiles): the first
    // download starts after one chunk's upload and GEMM
    int chunks = std::max(1, std::min(8, M / 512));
    const int rows = static_cast<int>(round_up((M + chunks - 1) / chunks, 256));
    chunks = (M + rows - 1) / rows;
    const int last_rows = M - (chunks - 1) * rows;
    Plan pf, plast;
    ensure_die_map(ds, ds->comp);
    if ((st = plan_on_device(InKind::BF16, ok, rows < M ? rows : M, N, K2, cfg, ds, &pf))) return st;
    if ((st = plan_on_device(InKind::BF16, ok, last_rows, N, K2, cfg, ds, &plast))) return st;
    const size_t ws_bytes = std::max(split_workspace(pf, rows < M ? rows : M, N).bytes,
                                     split_workspace(plast, last_rows, N).bytes);
    const size_t a_bytes = static_cast<size_t>(M) * lda2 * 2, b_bytes = static_cast<size_t>(K2) * ldb2 * 2;
    const size_t c_bytes = static_cast<size_t>(M) * ldc2 * oes;
    const size_t need = static_cast<size_t>(round_up(a_bytes, 256) + round_up(b_bytes, 256) +
                                            round_up(c_bytes, 256)) + ws_bytes;
    if ((st = ensure_scratch(ds, sr, need, stream))) return st;
    Carve cv{static_cast<uint8_t*>(sr->scratch), 0};
    uint8_t* a2 = static_cast<uint8_t*>(cv.take(a_bytes));
    uint8_t* b2 = static_cast<uint8_t*>(cv.take(b_bytes));
    uint8_t* c2 = static_cast<uint8_t*>(cv.take(c_bytes));
    void* wsp = cv.take(ws_bytes);

    constexpr int kMaxChunks = 8;
    cudaEvent_t ev[3 + 2 * kMaxChunks] = {};
    const int nev = 3 + 2 * chunks;
    auto fail = [&](int code) {
        cudaGetLastError();
        for (int i = 0; i < nev; ++i)
            if (ev[i]) cudaEventDestroy(ev[i]);
        return code;
    };
    for (int i = 0; i < nev; ++i)
        if (cudaEventCreateWithFlags(&ev[i], cudaEventDisableTiming) != cudaSuccess) return fail(TCL_ERR_LAUNCH);
    cudaEvent_t entry = ev[0], b_in = ev[1], done = ev[2];
    cudaEvent_t* a_in = ev + 3;
    cudaEvent_t* c_out = ev + 3 + chunks;
    const char* Ah = static_cast<const char*>(A);
    char* Ch = static_cast<char*>(C);
    bool okq = cudaEventRecord(entry, stream) == cudaSuccess && cudaStreamWaitEvent(ds->up, entry, 0) == cudaSuccess &&
               cudaStreamWaitEvent(ds->comp, entry, 0) == cudaSuccess &&
               cudaStreamWaitEvent(ds->down, entry, 0) == cudaSuccess;
    if (okq && K2 != K) {   // zero the K padding of both operands
        okq = cudaMemsetAsync(a2, 0, a_bytes, ds->up) == cudaSuccess &&
              cudaMemsetAsync(b2 + static_cast<size_t>(K) * ldb2 * 2, 0, static_cast<size_t>(K2 - K) * ldb2 * 2,
                              ds->up) == cudaSuccess;
    }
    okq = okq &&
          cudaMemcpy2DAsync(b2, ldb2 * 2, B, static_cast<size_t>(ldb) * 2, static_cast<size_t>(N) * 2, K,
                            cudaMemcpyHostToDevice, ds->up) == cudaSuccess &&
          cudaEventRecord(b_in, ds->up) == cudaSuccess;
    for (int i = 0; okq && i < chunks; ++i) {
        const int r = i + 1 < chunks ? rows : last_rows;
        okq = cudaMemcpy2DAsync(a2 + static_cast<size_t>(i) * rows * lda2 * 2, lda2 * 2,
                                Ah + static_cast<size_t>(i) * rows * lda * 2, static_cast<size_t>(lda) * 2,
                                static_cast<size_t>(K) * 2, r, cudaMemcpyHostToDevice, ds->up) == cudaSuccess &&
              cudaEventRecord(a_in[i], ds->up) == cudaSuccess;
    }
    okq = okq && cudaStreamWaitEvent(ds->comp, b_in, 0) == cudaSuccess;
    for (int i = 0; okq && i < chunks; ++i) {
        const int r = i + 1 < chunks ? rows : last_rows;
        okq = cudaStreamWaitEvent(ds->comp, a_in[i], 0) == cudaSuccess;
        if (!okq) break;
        st = run_gemm(i + 1 < chunks ? pf : plast, InKind::BF16, ok, r, N, K2,
                      a2 + static_cast<size_t>(i) * rows * lda2 * 2, lda2, b2, ldb2,
                      c2 + static_cast<size_t>(i) * rows * ldc2 * oes, ldc2, wsp, cfg, dev, ds, sr, ds->comp);
        if (st) return fail(st);
        okq = cudaEventRecord(c_out[i], ds->comp) == cudaSuccess &&
              cudaStreamWaitEvent(ds->down, c_out[i], 0) == cudaSuccess &&
              cudaMemcpy2DAsync(Ch + static_cast<size_t>(i) * rows * ldc * oes, static_cast<size_t>(ldc) * oes,
                                c2 + static_cast<size_t>(i) * rows * ldc2 * oes, ldc2 * oes,
                                static_cast<size_t>(N) * oes, r, cudaMemcpyDeviceToHost, ds->down) == cudaSuccess;
    }
    okq = okq && cudaEventRecord(done, ds->down) == cudaSuccess && cudaStreamWaitEvent(stream, done, 0) == cudaSuccess;
    if (!okq) return fail(TCL_ERR_LAUNCH);
    for (int i = 0; i < nev; ++i) cudaEventDestroy(ev[i]);   // released once their work has completed
    return TCL_OK;
}

}  // namespace

// Internal services for other translation units of the library.
int device_context(int* dev, int* sms, unsigned int** status) {
    std::lock_guard<std::mutex> lock(g_mu);
    DevState* ds = nullptr;
    int st = current_device(dev, &ds);
    if (st) return st;
    *sms = ds->sms;
    *status = ds->status;
    return TCL_OK;
}

int tensor_map_uncached(const void* ptr, CUtensorMapDataType dtype, uint64_t d0, uint64_t d1,
                        uint64_t stride_bytes, uint32_t b0, uint32_t b1, CUtensorMap* out) {
    std::lock_guard<std::mutex> lock(g_mu);
    int st = encode_fn();
    if (st) return st;
    const cuuint64_t dims[2] = {d0, d1};
    const cuuint64_t strides[1] = {stride_bytes};
    const cuuint32_t box[2] = {b0, b1};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(out, dtype, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? TCL_OK : TCL_ERR_LAUNCH;
}

}  // namespace tcl

using namespace tcl;

extern "C" {

int gemm_bf16(int M, int N, int K, const void* A, int lda, const void* B, int ldb, void* C, int ldc,
              int out, cudaStream_t stream) {
    return gemm_bf16_impl(M, N, K, A, lda, B, ldb, C, ldc, out, nullptr, stream);
}

int gemm_bf16_ex(int M, int N, int K, const void* A, int lda, const void* B, int ldb, void* C,
                 int ldc, int out, const tcl_config_t* cfg, cudaStream_t stream) {
    return gemm_bf16_impl(M, N, K, A, lda, B, ldb, C, ldc, out, cfg, stream);
}

int gemm_bf16_host(int M, int N, int K, const void* A, int lda, const void* B, int ldb, void* C, int ldc, int out,
                   cudaStream_t stream) {
    return gemm_bf16_host_impl(M, N, K, A, lda, B, ldb, C, ldc, out, nullptr, stream);
}

int gemm_tf32(int M, int N, int K, const float* A, int lda, const float* B, int ldb, float* C,
              int ldc, cudaStream_t stream) {
    return gemm_tf32_impl(M, N, K, A, lda, B, ldb, C, ldc, nullptr, stream);
}

int gemm_tf32_ex(int M, int N, int K, const float* A, int lda, const float* B, int ldb, float* C,
                 int ldc, const tcl_config_t* cfg, cudaStream_t stream) {
    return gemm_tf32_impl(M, N, K, A, lda, B, ldb, C, ldc, cfg, stream);
}

int gemm_s8(int M, int N, int K, const int8_t* A, int lda, const int8_t* B, int ldb, int32_t* C,
            int ldc, cudaStream_t stream) {
    return gemm_s8_impl(M, N, K, A, lda, B, ldb, C, ldc, nullptr, stream);
}

int gemm_s8_ex(int M, int N, int K, const int8_t* A, int lda, const int8_t* B, int ldb, int32_t* C,
               int ldc, const tcl_config_t* cfg, cudaStream_t stream) {
    return gemm_s8_impl(M, N, K, A, lda, B, ldb, C, ldc, cfg, stream);
}

int gemm_f32_simt(int M, int N, int K, const float* A, int lda, const float* B, int ldb, float* C, int ldc,
                  cudaStream_t stream) {
    int st = check_common(M, N, K, A, lda, B, ldb, C, ldc);
    if (st) return st;
    if (!aligned_to(A, 4) || !aligned_to(B, 4) || !aligned_to(C, 4)) return TCL_ERR_ALIGN;
    if ((M + 127) / 128 > 65535) return TCL_ERR_DIMS;   // grid rows
    int dev;
    DevState* ds;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        if ((st = current_device(&dev, &ds))) return st;
    }
    const bool vec = aligned16(A) && aligned16(B) && aligned16(C) && lda % 4 == 0 && ldb % 4 == 0 && ldc % 4 == 0;
    if (launch_sgemm_simt(A, lda, B, ldb, C, ldc, M, N, K, vec, stream) != cudaSuccess) {
        cudaGetLastError();
        return TCL_ERR_LAUNCH;
    }
    return TCL_OK;
}

int tcl_plan(int in_kind, int out, int M, int N, int K, const tcl_config_t* cfg, tcl_plan_t* plan) {
    if (M < 1 || N < 1 || K < 1) return TCL_ERR_DIMS;
    InKind ik;
    OutKind ok;
    if (in_kind == 0) {
        ik = InKind::BF16;
        if (out == TCL_OUT_F32) ok = OutKind::F32;
        else if (out == TCL_OUT_BF16) ok = OutKind::BF16;
        else return TCL_ERR_CONFIG;
    } else if (in_kind == 1) {
        ik = InKind::TF32;
        ok = OutKind::F32;
    } else if (in_kind == 2) {
        ik = InKind::BF16;
        ok = OutKind::S32;
    } else {
        return TCL_ERR_CONFIG;
    }
    Plan pl;
    int st;
    if (cfg && cfg->max_ctas > 0) {
        // planning without a device: max_ctas stands for the SM count (pairs: max_ctas / 2,
        // half of them on each die)
        const int pairs[2] = {cfg->max_ctas / 4, cfg->max_ctas / 2 - cfg->max_ctas / 4};
        st = make_plan(ik, ok, M, N, K, cfg, cfg->max_ctas, [](const VariantInfo*) { return 0; }, pairs, &pl);
    } else {
        std::lock_guard<std::mutex> lock(g_mu);
        int dev;
        DevState* ds;
        st = current_device(&dev, &ds);
        if (st) return st;
        ensure_die_map(ds, cudaStreamLegacy);
        st = plan_on_device(ik, ok, M, N, K, cfg, ds, &pl);
    }
    if (st) return st;
    if (plan) {
        plan->bn = pl.bn;
        plan->stages = pl.stages;
        plan->grid = pl.grid;
        plan->num_tiles = pl.num_tiles;
        plan->smem_bytes = pl.smem;
        plan->cta_pair = pl.pair ? 2 : 1;
        plan->splits = pl.splits;
        plan->producer = pl.prod;
        plan->workspace_bytes = static_cast<unsigned long long>(split_workspace(pl, M, N).bytes);
        plan->sk_tiles = pl.sk_tiles;
        plan->sk_pieces = pl.sk_pieces;
        plan->sk_balanced = pl.sk_balanced;
        plan->group_m = pl.group_m;
        plan->k_serpentine = pl.k_serpentine;
        plan->s8_in_kernel = pl.s8_in_kernel;
        plan->cluster_k = pl.csk ? pl.csk : 1;
        plan->tile_m = pl.pair ? 256 : pl.m64 ? 64 : 128;
        plan->kblocks_per_stage = pl.m64 ? pl.m64 : pl.kps;
        plan->die_split = pl.die_split;
        plan->l2_hints = pl.l2_hints;
        plan->die_tiles0 = pl.die_split ? pl.sub_tiles[0] : 0;
    }
    return TCL_OK;
}

const char* tcl_status_string(int status) {
    switch (status) {
        case TCL_OK: return "ok";
        case TCL_ERR_NULL: return "null pointer argument";
        case TCL_ERR_DIMS: return "M, N and K must be at least 1";
        case TCL_ERR_LD: return "leading dimension smaller than the row width";
        case TCL_ERR_ALIGN: return "base address or leading dimension not 16-byte aligned";
        case TCL_ERR_K_TOO_LARGE: return "K too large for an exact int32 result";
        case TCL_ERR_LAUNCH: return "CUDA call or kernel launch failed";
        case TCL_ERR_DEVICE_TIMEOUT: return "a bounded in-kernel wait timed out";
        case TCL_ERR_CONFIG: return "requested configuration is not built";
        case TCL_ERR_NO_MEMORY: return "scratch allocation failed";
        case TCL_ERR_DEVICE: return "current device is not an sm_103 GPU";
        case TCL_ERR_STATIC_LIMIT: return "problem needs more scratch than the fixed static buffer holds";
        case TCL_ERR_CAPTURE: return "scratch would have to grow while the stream is being captured";
        default: return "unknown status";
    }
}

int tcl_last_device_error(cudaStream_t stream, int* detail) {
    if (detail) *detail = 0;
    std::lock_guard<std::mutex> lock(g_mu);
    int dev;
    DevState* ds;
    int st = current_device(&dev, &ds);
    if (st) return st;
    if (cudaStreamSynchronize(stream) != cudaSuccess) {
        cudaGetLastError();
        return TCL_ERR_LAUNCH;
    }
    unsigned int word = 0;
    const unsigned int zero = 0;
    if (cudaMemcpy(&word, ds->status, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemcpy(ds->status, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess) {
        cudaGetLastError();
        return TCL_ERR_LAUNCH;
    }
    if (detail) *detail = static_cast<int>(word);
    return word ? TCL_ERR_DEVICE_TIMEOUT : TCL_OK;
}

int tcl_num_sms(void) {
    std::lock_guard<std::mutex> lock(g_mu);
    int dev;
    DevState* ds;
    if (current_device(&dev, &ds)) return 0;
    return ds->sms;
}

int tcl_die_pairs(int* n0, int* n1) {
    if (n0) *n0 = 0;
    if (n1) *n1 = 0;
    std::lock_guard<std::mutex> lock(g_mu);
    int dev;
    DevState* ds;
    int st = current_device(&dev, &ds);
    if (st) return st;
    ensure_die_map(ds, cudaStreamLegacy);
    if (n0) *n0 = ds->die_pairs[0];
    if (n1) *n1 = ds->die_pairs[1];
    return TCL_OK;
}

int tcl_stream_release(cudaStream_t stream) {
    if (stream == nullptr || stream == cudaStreamLegacy || stream == cudaStreamPerThread) return TCL_OK;
    std::lock_guard<std::mutex> lock(g_mu);
    int dev;
    DevState* ds;
    int st = current_device(&dev, &ds);
    if (st) return st;
    auto it = ds->per_stream.find(stream);
    if (it == ds->per_stream.end()) return TCL_OK;
    if (cudaStreamSynchronize(stream) != cudaSuccess) {
        cudaGetLastError();
        return TCL_ERR_LAUNCH;
    }
    cudaFree(it->second.scratch);
    if (it->second.own_flags) cudaFree(it->second.sk_flags);
    ds->per_stream.erase(it);
    return TCL_OK;
}

void tcl_shutdown(void) {
    std::lock_guard<std::mutex> lock(g_mu);
    int prev = 0;
    if (cudaGetDevice(&prev) != cudaSuccess) {
        cudaGetLastError();
        return;
    }
    for (int d = 0; d < kMaxDevices; ++d) {
        if (g_dev[d].up) {
            if (cudaSetDevice(d) == cudaSuccess) {
                cudaDeviceSynchronize();
                cudaStreamDestroy(g_dev[d].up);
                cudaStreamDestroy(g_dev[d].comp);
                cudaStreamDestroy(g_dev[d].down);
            }
            g_dev[d].up = g_dev[d].comp = g_dev[d].down = nullptr;
        }
        DevState& ds = g_dev[d];
        if (ds.base.scratch || !ds.per_stream.empty() || !ds.retired.empty()) {
            if (cudaSetDevice(d) == cudaSuccess) {
                cudaDeviceSynchronize();
                cudaFree(ds.base.scratch);
                for (auto& kv : ds.per_stream) {
                    cudaFree(kv.second.scratch);
                    if (kv.second.own_flags) cudaFree(kv.second.sk_flags);
                }
                for (void* r : ds.retired) cudaFree(r);
            }
            ds.base.scratch = nullptr;
            ds.base.scratch_bytes = 0;
            ds.per_stream.clear();
            ds.retired.clear();
        }
    }
    cudaSetDevice(prev);
    cudaGetLastError();
    g_maps.clear();
}

const char* tcl_version(void) { return "tcl-gb300 0.1.0 sm_103a"; }

}  // extern "C"
