// gemm_s8_static: the int8 GEMM with its operand scratch in a fixed,
// file-scope device array instead of memory the library allocates, for
// callers that cannot have the library call cudaMalloc (see tcl_gemm.h).
//
// The path is the same as gemm_s8: widen A and B exactly to bf16 (zero-padded
// rows), then run the bf16 tensor-core kernel in exact-integer mode. Only
// where the packed copies live differs.
#include <cuda.h>

#include <cstdint>
#include <mutex>

#include "launch.cuh"
#include "tcl_gemm.h"

namespace tcl {

int device_context(int* dev, int* sms, unsigned int** status);   // api.cu
int tensor_map_uncached(const void* ptr, CUtensorMapDataType dtype, uint64_t d0, uint64_t d1,
                        uint64_t stride_bytes, uint32_t b0, uint32_t b1, CUtensorMap* out);   // api.cu

namespace {

// The fixed scratch. In host code this name is only a stand-in for the
// symbol; the device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_s8_static_scratch[TCL_S8_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {};   // device address of the array, per device
std::mutex g_static_mu;

long long round_up(long long x, long long m) { return (x + m - 1) / m * m; }

}  // namespace
}  // namespace tcl

using namespace tcl;

extern "C" TCL_API int gemm_s8_static(int M, int N, int K, const int8_t* A, int lda, const int8_t* B,
                                      int ldb, int32_t* C, int ldc, cudaStream_t stream) {
    // Argument checks, as gemm_s8, before any CUDA call.
    if (!A || !B || !C) return TCL_ERR_NULL;
    if (M < 1 || N < 1 || K < 1) return TCL_ERR_DIMS;
    if (lda < K || ldb < N || ldc < N) return TCL_ERR_LD;
    auto aligned16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    if (!aligned16(A) || !aligned16(B) || !aligned16(C) || lda % 16 || ldb % 16 || ldc % 4)
        return TCL_ERR_ALIGN;
    if (K > 131071) return TCL_ERR_K_TOO_LARGE;
    const long long lda2 = round_up(K, 8), ldb2 = round_up(N, 8);
    const long long a_bytes = round_up(static_cast<long long>(M) * lda2 * 2, 256);
    const long long b_bytes = round_up(static_cast<long long>(K) * ldb2 * 2, 256);
    if (static_cast<unsigned long long>(a_bytes + b_bytes) > TCL_S8_STATIC_SCRATCH_BYTES)
        return TCL_ERR_STATIC_LIMIT;

    std::lock_guard<std::mutex> lock(g_static_mu);
    int dev = 0, sms = 0;
    unsigned int* status = nullptr;
    int st = device_context(&dev, &sms, &status);
    if (st) return st;
    if (dev < 0 || dev >= kMaxDevices) return TCL_ERR_LAUNCH;
    if (!g_scratch_addr[dev]) {   // once per device, with that device current
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_s8_static_scratch) != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return TCL_ERR_LAUNCH;
        }
        g_scratch_addr[dev] = p;
    }
    uint8_t* a2 = static_cast<uint8_t*>(g_scratch_addr[dev]);
    uint8_t* b2 = a2 + a_bytes;

    // This path launches the one-SM exact-integer kernel only (no stream-K flags,
    // no workspace), so the plan is asked for exactly that. The planner returns a
    // plan only for a kernel variant that is built, so once it succeeds the launch
    // below finds its variant, and nothing is enqueued before this point.
    tcl_config_t cfg = {};
    cfg.max_ctas = sms;   // plan for this device without another device query
    cfg.cta_pair = 1;
    tcl_plan_t plan;
    if ((st = tcl_plan(2, TCL_OUT_F32, M, N, K, &cfg, &plan))) return st;
    const int bn = plan.bn, stages = plan.stages, grid = plan.grid;
    const int tiles_m = (M + 127) / 128, tiles_n = (N + bn - 1) / bn;
    if (plan.cta_pair != 1 || plan.splits != 1 || plan.sk_tiles != 0 || plan.num_tiles != tiles_m * tiles_n)
        return TCL_ERR_CONFIG;

    LaunchArgs a;
    a.in = InKind::BF16;
    a.out = OutKind::S32;
    a.bn = bn;
    a.stages = stages;
    a.prod = PROD_TMA;
    a.pair = 0;
    a.slots = 2;
    a.csk = 0;
    a.m64 = 0;
    a.pdl = false;
    a.grid = grid;
    a.stream = stream;
    if ((st = tensor_map_uncached(a2, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, K, M, lda2 * 2, 64, 128, &a.tmA)))
        return st;
    if ((st = tensor_map_uncached(b2, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, N, K, ldb2 * 2, 64, 64, &a.tmB)))
        return st;
    if ((st = tensor_map_uncached(C, CU_TENSOR_MAP_DATA_TYPE_INT32, N, M, static_cast<uint64_t>(ldc) * 4, 32, 32,
                                  &a.tmC)))
        return st;
    GemmParams& p = a.p;
    p.M = M;
    p.N = N;
    p.K = K;
    p.tiles_m = tiles_m;
    p.tiles_n = tiles_n;
    p.num_tiles = plan.num_tiles;
    p.num_kb = (K + 63) / 64;
    p.kb_per_unit = 1024 / 64;   // exact fp32 units of 1024 K values, as gemm_s8
    p.group_m = plan.group_m;
    p.timeout_ns = 1000000000ull;
    p.status = status;
    p.trace = nullptr;
    p.trace_cap = 0;
    p.C = C;
    p.ldc = ldc;
    p.A = a2;
    p.lda = lda2;
    p.B = b2;
    p.ldb = ldb2;
    p.debug_skip_kb = -1;
    p.splits = 1;
    p.kb_per_split = p.num_kb;
    p.split_rows = 0;
    p.out_rows = M;
    p.sk_tiles = 0;
    p.sk_pieces = 1;
    p.sk_balanced = 0;
    p.sk_first = 0;
    p.sk_region = 0;
    p.sk_flags = nullptr;
    p.sk_gen = 0;
    p.debug_sk_stall = 0;
    p.sk_ws = nullptr;
    p.sk_ws_rows = 0;
    p.k_serpentine = plan.k_serpentine;
    p.b_3d = 0;
    p.kps2 = 0;
    p.die_split = 0;
    p.l2_hints = 0;

    if (launch_s8_to_bf16({A, lda, reinterpret_cast<uint16_t*>(a2), lda2, M, K, 0},
                          {B, ldb, reinterpret_cast<uint16_t*>(b2), ldb2, K, N, 0}, sms, stream) != cudaSuccess) {
        cudaGetLastError();
        return TCL_ERR_LAUNCH;
    }
    bool found = false;
    cudaError_t err = launch_group_bf16_misc(a, &found);
    if (!found) return TCL_ERR_CONFIG;
    if (err != cudaSuccess) {
        cudaGetLastError();
        return TCL_ERR_LAUNCH;
    }
    return TCL_OK;
}
