// gq_host.cuh -- host-side launch helpers shared by the library's translation units: device
// geometry, occupancy-sized grids, launch status, the block runs of the segmented kernels, and
// the per-(gradient type, scheme) quantise launchers that live in their own translation units
// (compiled in parallel).
#pragma once
#include "gq.h"
#include "gq_kernels.cuh"

#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

namespace gqh {

using gq::kThreads;


constexpr int64_t kMaxD = int64_t(1) << 34;  // Philox counter word 0 holds j / 8 in 31 bits
constexpr int kMaxDevices = 64;

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline int sm_count() {
    static int cache[kMaxDevices] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 152;
    if (cache[dev] == 0) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
            v = 152;
        cache[dev] = v;
    }
    return cache[dev];
}

// Resident blocks per SM for a kernel with `smem` bytes of dynamic shared memory, cached per
// (kernel, device).  The first query for a kernel on a device also raises that kernel's
// dynamic shared-memory limit to `smem`.
template <typename K>
int blocks_per_sm(K kernel, int smem = 0, int threads = kThreads) {
    struct Entry {
        const void* fn;
        int dev;
        int nb;
    };
    static Entry table[512];
    static int used = 0;
    static std::mutex mu;
    const void* fn = reinterpret_cast<const void*>(kernel);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) dev = 0;
    std::lock_guard<std::mutex> lock(mu);
    for (int e = 0; e < used; ++e)
        if (table[e].fn == fn && table[e].dev == dev) return table[e].nb;
    if (smem > 0)  // dynamic + static shared memory may pass the default 48 KB
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    int nb = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, kernel, threads, smem) != cudaSuccess ||
        nb <= 0)
        nb = 1;
    if (used < 512) table[used++] = Entry{fn, dev, nb};
    return nb;
}

// Grid for a grid-stride kernel over `work` thread-items: one full wave of resident blocks
// (a multiple of the SM count), fewer when the work is smaller.
template <typename K>
unsigned grid_for(K kernel, int64_t work, int64_t cap = INT32_MAX, int smem = 0) {
    const int64_t full = static_cast<int64_t>(blocks_per_sm(kernel, smem)) * sm_count();
    int64_t need = (work + kThreads - 1) / kThreads;
    int64_t g = need < full ? need : full;
    if (g > cap) g = cap;
    if (g < 1) g = 1;
    return static_cast<unsigned>(g);
}

inline gq_status launch_status() {
    return cudaGetLastError() == cudaSuccess ? GQ_OK : GQ_ERR_CUDA;
}


// Runs of blocks for a chunk of segments: each gets a share of `target` blocks in proportion to
// its elements, at least one and at most one per 256 column groups of `cols` columns.
inline void plan_runs(gq::SegLaunch& L, const int64_t* d, int64_t n, int cols, int64_t target) {
    double total = 0.0;
    for (int k = 0; k < L.nseg; ++k) total += static_cast<double>(d[k]);
    int32_t b = 0;
    for (int k = 0; k < L.nseg; ++k) {
        const int64_t groups = (d[k] + cols - 1) / cols;
        const int64_t most = (groups + kThreads - 1) / kThreads;
        int64_t nb = static_cast<int64_t>(static_cast<double>(d[k]) / total * static_cast<double>(target));
        if (nb > most) nb = most;
        if (nb < 1) nb = 1;
        L.seg[k].d = d[k];
        L.seg[k].b0 = b;
        L.seg[k].nb = static_cast<int32_t>(nb);
        b += static_cast<int32_t>(nb);
    }
    (void)n;
}

inline int32_t total_blocks(const gq::SegLaunch& L) {
    return L.seg[L.nseg - 1].b0 + L.seg[L.nseg - 1].nb;
}


// The single-launch form of the fused call: blocks of gpb column groups, at most one per SM,
// each holding its n x (8 gpb) slice in shared memory; false when a slice would not fit.
inline bool resident_plan(int64_t n, int64_t d, int elt, int64_t* gpb, unsigned* nblk,
                          size_t* smem) {
    const int64_t groups = (d + gq::kQCols - 1) / gq::kQCols;
    const int64_t nsm = sm_count();
    const int64_t g = (groups + nsm - 1) / nsm;
    if (nsm > 255) return false;  // the grid barrier counts arrivals in 8 bits
    if (n > gq::kResTileBytes / (g * gq::kQCols * elt)) return false;
    *gpb = g;
    *nblk = static_cast<unsigned>((groups + g - 1) / g);
    *smem = static_cast<size_t>(n * g * gq::kQCols * elt);
    return true;
}

// Quantise launchers, one translation unit per (gradient type, scheme).  out: dequantise into
// outp (else only codes); trusted: the norm was computed from these gradients; status
// (nullable): the workspace status word, which lets large aligned problems take the bulk-copy
// kernel.
#define GQH_QUANT_LAUNCHERS(NAME)                                                                 \
    gq_status quant_##NAME(const void* grads, const gq::QuantArgs& a, int bits, bool out,          \
                           bool trusted, void* codes, void* outp, cudaStream_t st,                 \
                           unsigned int* status);                                                  \
    gq_status quant_segments_##NAME(gq::SegLaunch& L, const int64_t* d, int64_t n,                \
                                    const gq::QuantArgs& base, unsigned char* ws, cudaStream_t st); \
    gq_status resident_##NAME(const void* grads, const gq::QuantArgs& a, int mode, void* out,       \
                              float* norm_user, unsigned char* ws, cudaStream_t st, bool* taken);  \
    unsigned int debug_word_##NAME();
GQH_QUANT_LAUNCHERS(f32_l)
GQH_QUANT_LAUNCHERS(f32_e)
GQH_QUANT_LAUNCHERS(bf16_l)
GQH_QUANT_LAUNCHERS(bf16_e)
#undef GQH_QUANT_LAUNCHERS

}  // namespace gqh
