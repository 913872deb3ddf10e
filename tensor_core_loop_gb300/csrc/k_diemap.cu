// Which SMs share a half of the L2: GB300 is two dies, and each die's L2 keeps
// the lines its own SMs read (an SM finds a line that an SM of its own die
// brought in at ~300 cycles, one that an SM of the other die brought in at
// ~475, one from HBM at ~820; measured with pointer chases on GB300). One CTA
// reads a small buffer into its die's L2; then every SM times a chase through
// its own slice of that buffer. The SMs that hit fast share the reader's die.
// Run once per device; the two-SM kernel uses the map to give each die's
// pairs their own block of tiles (gemm_kernel_pair.cuh, die split).
#include "launch.cuh"

namespace tcl {
namespace {

constexpr int kChainLines = 512;  // 128-byte lines of each SM's slice
constexpr int kHops = 24;         // steps of 37 or 38 lines: 24 distinct lines whatever the words hold

__device__ __forceinline__ uint32_t sm_id() {
    uint32_t s;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(s));
    return s;
}

__device__ __forceinline__ uint32_t ld_cg(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.global.cg.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Drops every line of the buffer from the L2 (its contents become undefined;
// nothing reads them as data).
__global__ void diemap_discard(uint8_t* buf, long long lines) {
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < lines;
         i += static_cast<long long>(gridDim.x) * blockDim.x)
        asm volatile("discard.global.L2 [%0], 128;" ::"l"(buf + i * 128) : "memory");
}

// One CTA: brings every line into the L2 of its own die.
__global__ void diemap_load(const uint8_t* buf, long long lines, uint32_t* out) {
    uint32_t acc = 0;
    for (long long i = threadIdx.x; i < lines; i += blockDim.x) acc += ld_cg(reinterpret_cast<const uint32_t*>(buf + i * 128));
    if (threadIdx.x == 0) out[0] = sm_id();
    if (acc == 0x9e3779b9u) out[1] = acc;   // keeps the loads
}

// One CTA per SM (the dynamic shared memory keeps two off one SM): thread 0 chases
// through its own slice; the next line depends on the loaded word (so the loads are
// serial), stays inside the slice and is never one visited before, whatever the word
// holds (a second visit would hit in this SM's own die).
__global__ void diemap_chase(const uint8_t* buf, uint32_t* smid, uint32_t* cycles) {
    extern __shared__ uint8_t pad[];
    if (threadIdx.x != 0) return;
    const uint8_t* base = buf + static_cast<long long>(blockIdx.x) * kChainLines * 128;
    uint32_t line = 0;
    const uint64_t t0 = clock64();
    for (int h = 0; h < kHops; ++h) {
        const uint32_t v = ld_cg(reinterpret_cast<const uint32_t*>(base + line * 128));
        line = (line + 37u + (v & 1u)) & (kChainLines - 1);
    }
    const uint64_t t1 = clock64();
    pad[0] = static_cast<uint8_t>(line);
    smid[blockIdx.x] = sm_id();
    cycles[blockIdx.x] = static_cast<uint32_t>((t1 - t0) / kHops);
}

}  // namespace

// Fills die_of_tpc[t] (t = SM id / 2, the pair of SMs a CTA pair runs on) with 0 or 1
// for the two dies, 255 for pairs not seen; returns the number of pairs found on each
// die in n0/n1, or false when the timings do not split into two clear groups (the map
// is then not used). Synchronous; a few tens of microseconds; not while capturing.
bool calibrate_die_map(int sms, uint8_t* die_of_tpc, int max_tpc, int* n0, int* n1) {
    for (int i = 0; i < max_tpc; ++i) die_of_tpc[i] = 255;
    *n0 = *n1 = 0;
    if (sms <= 0 || sms > 1024) return false;
    const long long lines = static_cast<long long>(sms) * kChainLines;
    uint8_t* buf = nullptr;
    uint32_t* dev = nullptr;   // [0..1] loader, [2, 2 + sms) SM ids, [2 + sms, 2 + 2·sms) cycles
    if (cudaMalloc(&buf, lines * 128) != cudaSuccess || cudaMalloc(&dev, (2 + 2 * sms) * sizeof(uint32_t)) != cudaSuccess) {
        cudaGetLastError();
        cudaFree(buf);
        return false;
    }
    const int smem = 160 * 1024;
    bool ok = cudaFuncSetAttribute(diemap_chase, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) == cudaSuccess;
    if (ok) {
        diemap_discard<<<64, 256>>>(buf, lines);
        diemap_load<<<1, 256>>>(buf, lines, dev);
        diemap_chase<<<sms, 32, smem>>>(buf, dev + 2, dev + 2 + sms);
        ok = cudaDeviceSynchronize() == cudaSuccess;
    }
    uint32_t* host = new uint32_t[2 + 2 * sms];
    if (ok) ok = cudaMemcpy(host, dev, (2 + 2 * sms) * sizeof(uint32_t), cudaMemcpyDeviceToHost) == cudaSuccess;
    cudaGetLastError();
    cudaFree(buf);
    cudaFree(dev);
    if (!ok) {
        delete[] host;
        return false;
    }
    const uint32_t* smid = host + 2;
    const uint32_t* cyc = host + 2 + sms;
    uint32_t lo = 0xffffffffu, hi = 0;
    for (int b = 0; b < sms; ++b) {
        lo = cyc[b] < lo ? cyc[b] : lo;
        hi = cyc[b] > hi ? cyc[b] : hi;
    }
    // two clear groups: the far hits at least 25 % slower than the near ones
    bool valid = hi * 4 >= lo * 5;
    const uint32_t mid = (lo + hi) / 2;
    const int loader_die = 0;   // the dies are numbered from the loader's
    for (int b = 0; b < sms && valid; ++b) {
        if (smid[b] / 2 >= static_cast<uint32_t>(max_tpc)) {
            valid = false;
            break;
        }
        const uint8_t d = static_cast<uint8_t>(cyc[b] <= mid ? loader_die : 1 - loader_die);
        uint8_t& slot = die_of_tpc[smid[b] / 2];
        if (slot != 255 && slot != d) valid = false;   // both SMs of a pair on one die
        slot = d;
        // no timing between the groups' ranges
        if (cyc[b] > lo + (hi - lo) / 3 && cyc[b] < hi - (hi - lo) / 3) valid = false;
    }
    delete[] host;
    int c0 = 0, c1 = 0;
    for (int t = 0; t < max_tpc; ++t) {
        if (die_of_tpc[t] == 0) ++c0;
        if (die_of_tpc[t] == 1) ++c1;
    }
    if (!valid || c0 == 0 || c1 == 0) {
        for (int i = 0; i < max_tpc; ++i) die_of_tpc[i] = 255;
        return false;
    }
    *n0 = c0;
    *n1 = c1;
    return true;
}

}  // namespace tcl
