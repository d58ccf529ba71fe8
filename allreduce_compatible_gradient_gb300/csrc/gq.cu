// gq.cu -- C ABI (include/gq.h) over the sm_103a kernels in gq_kernels.cuh (the quantise
// launchers are in gq_quant_<type>_<scheme>.cu).
//
// Host side only: argument checks (returned synchronously, before anything is enqueued),
// launch geometry (grid = resident blocks per SM x SM count, capped by the work), and kernel
// dispatch on (dtype, scheme, code width, norm order).  No memory is allocated here.
#include "gq.h"
#include "gq_host.cuh"
#include "gq_kernels.cuh"

#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>

using namespace gqh;

namespace {

// The grid of a scheme argument (GQ_ROUND_U16 may be added to select the rounding mode).
inline int grid_of(int scheme) { return scheme & ~GQ_ROUND_U16; }
inline int u16_of(int scheme) { return (scheme & GQ_ROUND_U16) ? 1 : 0; }

gq_status check_grads(const void* grads, int dtype, int64_t n, int64_t d) {
    if (!grads || !aligned16(grads)) return GQ_ERR_INVALID;
    if (dtype != GQ_F32 && dtype != GQ_BF16) return GQ_ERR_INVALID;
    if (n < 1 || n >= (int64_t(1) << 31) || d < 1 || d >= kMaxD) return GQ_ERR_INVALID;
    return GQ_OK;
}

// The sum of n workers' codes fits int8: n s <= 127 (L) or n 2^(s-1) <= 127 (E).
bool fits_i8(int scheme, int s, int64_t n) {
    const int64_t unit = grid_of(scheme) == GQ_LINEAR ? s : (int64_t(1) << (s - 1));
    return n * unit <= 127;
}

gq_status check_scheme(int scheme, int s, int64_t n) {
    scheme = grid_of(scheme);
    if (scheme != GQ_LINEAR && scheme != GQ_EXP) return GQ_ERR_INVALID;
    if (scheme == GQ_LINEAR) {
        if (s < 1 || s > 127) return GQ_ERR_UNSUPPORTED;
        if (n * static_cast<int64_t>(s) >= (int64_t(1) << 24)) return GQ_ERR_OVERFLOW;
    } else {
        if (s < 1 || s > 24) return GQ_ERR_UNSUPPORTED;
        if (n * (int64_t(1) << (s - 1)) >= (int64_t(1) << 24)) return GQ_ERR_OVERFLOW;
    }
    return GQ_OK;
}

gq_status check_ws(const void* ws, size_t ws_bytes, int64_t n, int64_t d) {
    if (!ws || !aligned16(ws)) return GQ_ERR_WORKSPACE;
    if (ws_bytes < gq_workspace_bytes(n, d)) return GQ_ERR_WORKSPACE;
    return GQ_OK;
}

int norm_mode(int q, int p) {
    if (q == GQ_NORM_INF && p == GQ_NORM_INF) return gq::kMaxMax;
    if (q == GQ_NORM_L2 && p == GQ_NORM_L2) return gq::kL2L2;
    if (q == GQ_NORM_L2 && p == GQ_NORM_INF) return gq::kL2Max;
    if (q == GQ_NORM_INF && p == GQ_NORM_L2) return gq::kMaxL2;
    return -1;
}

// ---- norm ---------------------------------------------------------------------------------
// Blocks of the norm step for an n x d problem (the flat kernel for the (inf,inf) and (2,2)
// forms, whose threads take sixteen or eight 16-byte vectors per iteration; the per-column
// kernel else).
template <typename T, int MODE>
unsigned norm_grid(int64_t n, int64_t d) {
    constexpr int C = gq::Elem<T>::kCols;
    constexpr int U = MODE == gq::kMaxMax ? 16 : 8;
    if constexpr (MODE == gq::kMaxMax || MODE == gq::kL2L2)
        return grid_for(gq::norm_flat_kernel<T, MODE>, (n * d / C + U - 1) / U, gq::kMaxPartials);
    else
        return grid_for(gq::norm_kernel<T, MODE>, (d + C - 1) / C, gq::kMaxPartials);
}

template <typename T, int MODE>
gq_status run_norm(const T* x, int64_t n, int64_t d, float* norm_user, double* part_user,
                   unsigned char* ws, cudaStream_t st) {
    constexpr int C = gq::Elem<T>::kCols;
    const unsigned grid = norm_grid<T, MODE>(n, d);
    if constexpr (MODE == gq::kMaxMax || MODE == gq::kL2L2) {
        gq::norm_flat_kernel<T, MODE><<<grid, kThreads, 0, st>>>(x, n * d, norm_user, part_user, ws);
    } else {
        const int64_t groups = (d + C - 1) / C;
        const bool vec_rows = (d % C) == 0;
        gq::norm_kernel<T, MODE><<<grid, kThreads, 0, st>>>(x, n, d, groups, vec_rows, norm_user,
                                                            part_user, ws);
    }
    return launch_status();
}

template <typename T>
gq_status dispatch_norm(const void* grads, int mode, int64_t n, int64_t d, float* norm_user,
                        double* part_user, unsigned char* ws, cudaStream_t st) {
    const T* x = static_cast<const T*>(grads);
    switch (mode) {
        case gq::kMaxMax: return run_norm<T, gq::kMaxMax>(x, n, d, norm_user, part_user, ws, st);
        case gq::kL2L2: return run_norm<T, gq::kL2L2>(x, n, d, norm_user, part_user, ws, st);
        case gq::kL2Max: return run_norm<T, gq::kL2Max>(x, n, d, norm_user, part_user, ws, st);
        default: return run_norm<T, gq::kMaxL2>(x, n, d, norm_user, part_user, ws, st);
    }
}

gq_status norm_any(const void* grads, int dtype, int mode, int64_t n, int64_t d, float* norm_user,
                   void* ws, cudaStream_t st, double* part_user = nullptr) {
    unsigned char* w = static_cast<unsigned char*>(ws);
    return dtype == GQ_F32 ? dispatch_norm<float>(grads, mode, n, d, norm_user, part_user, w, st)
                           : dispatch_norm<uint16_t>(grads, mode, n, d, norm_user, part_user, w, st);
}

// ---- quantize (+ sum + dequantize): one launcher per (gradient type, scheme) --------------
// status (nullable): the workspace status word, for the bounded waits of the bulk-copy kernel
template <bool OUT, bool TRUSTED>
gq_status quant_any(const void* grads, int dtype, const gq::QuantArgs& a, int scheme, int bits,
                    void* codes, void* out, cudaStream_t st, unsigned int* status = nullptr) {
    scheme = grid_of(scheme);  // the rounding mode travels in a.u16
    if (dtype == GQ_F32)
        return scheme == GQ_LINEAR
                   ? quant_f32_l(grads, a, bits, OUT, TRUSTED, codes, out, st, status)
                   : quant_f32_e(grads, a, bits, OUT, TRUSTED, codes, out, st, status);
    return scheme == GQ_LINEAR ? quant_bf16_l(grads, a, bits, OUT, TRUSTED, codes, out, st, status)
                               : quant_bf16_e(grads, a, bits, OUT, TRUSTED, codes, out, st, status);
}

gq::QuantArgs make_args(const float* norm_ptr, int dtype, int64_t n, int64_t d, int s,
                        uint64_t seed, uint64_t step, int scheme) {
    gq::QuantArgs a;
    a.u16 = u16_of(scheme);
    a.norm_ptr = norm_ptr;
    a.s = static_cast<uint32_t>(s);
    a.key0 = static_cast<uint32_t>(seed);
    a.key1 = static_cast<uint32_t>(seed >> 32);
    for (int r = 0; r < 10; ++r) {  // Philox round keys: the key advanced by r Weyl steps
        a.rk[2 * r] = a.key0 + static_cast<uint32_t>(r) * 0x9E3779B9u;
        a.rk[2 * r + 1] = a.key1 + static_cast<uint32_t>(r) * 0xBB67AE85u;
    }
    a.step_lo = static_cast<uint32_t>(step);
    a.step_hi = static_cast<uint32_t>(step >> 32);
    a.n = n;
    a.d = d;
    a.pitch = gq_code_pitch(d);
    a.vec_rows = (d % (dtype == GQ_F32 ? 4 : 8)) == 0;
    a.row0 = 0;
    a.sums = nullptr;
    a.sums_i8 = 0;
    a.out_dtype = gq::kOutF32;
    a.compact = 0;
    a.pdl = 0;
    return a;
}

}  // namespace

extern "C" {

int gq_abi_version(void) { return 1; }

size_t gq_workspace_bytes(int64_t n, int64_t d) {
    (void)n;
    (void)d;
    return static_cast<size_t>(gq::kWorkspaceBytes);
}

int gq_fused_launches(int dtype, int64_t n, int64_t d, int with_codes) {
    if ((dtype != GQ_F32 && dtype != GQ_BF16) || n < 1 || n >= (int64_t(1) << 31) || d < 1 ||
        d >= kMaxD)
        return 0;
    const int elt = dtype == GQ_F32 ? 4 : 2;
    int64_t gpb = 0;
    unsigned nblk = 0;
    size_t smem = 0;
    if (!with_codes && d % (16 / elt) == 0 && resident_plan(n, d, elt, &gpb, &nblk, &smem))
        return 1;
    return 2;
}

gq_status gq_workspace_init(void* ws, size_t ws_bytes, void* stream) {
    if (!ws || !aligned16(ws) || ws_bytes < gq_workspace_bytes(1, 1))
        return GQ_ERR_WORKSPACE;
    if (cudaMemsetAsync(ws, 0, gq_workspace_bytes(1, 1), static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return GQ_ERR_CUDA;
    return GQ_OK;
}

int gq_code_bits(int scheme, int s) {
    scheme = grid_of(scheme);
    if (scheme != GQ_LINEAR && scheme != GQ_EXP) return 0;
    if (s < 1 || s > (scheme == GQ_LINEAR ? 127 : 24)) return 0;
    return s <= 7 ? 4 : 8;
}

int64_t gq_code_pitch(int64_t d) { return d < 1 ? 0 : (d + 31) / 32 * 32; }

size_t gq_code_bytes(int scheme, int s, int64_t n, int64_t d) {
    const int bits = gq_code_bits(scheme, s);
    if (!bits || n < 1 || d < 1) return 0;
    return static_cast<size_t>(n) * static_cast<size_t>(gq_code_pitch(d)) * bits / 8;
}

gq_status gq_global_norm(const void* grads, int dtype, int64_t n, int64_t d, int q, int p,
                         float* norm_dev, void* ws, size_t ws_bytes, void* stream) {
    gq_status st = check_grads(grads, dtype, n, d);
    if (st != GQ_OK) return st;
    const int mode = norm_mode(q, p);
    if (mode < 0 || !norm_dev) return GQ_ERR_INVALID;
    if ((st = check_ws(ws, ws_bytes, n, d)) != GQ_OK) return st;
    return norm_any(grads, dtype, mode, n, d, norm_dev, ws, static_cast<cudaStream_t>(stream));
}

gq_status gq_quantize_ws(const void* grads, int dtype, int64_t n, int64_t d,
                         const float* norm_dev, int scheme, int s, uint64_t seed, uint64_t step,
                         void* codes, void* ws, size_t ws_bytes, void* stream) {
    gq_status st = check_grads(grads, dtype, n, d);
    if (st != GQ_OK) return st;
    if ((st = check_scheme(scheme, s, n)) != GQ_OK) return st;
    if (!norm_dev || !codes || !aligned16(codes)) return GQ_ERR_INVALID;
    if (ws && (st = check_ws(ws, ws_bytes, n, d)) != GQ_OK) return st;
    const gq::QuantArgs a = make_args(norm_dev, dtype, n, d, s, seed, step, scheme);
    unsigned int* status = ws ? &reinterpret_cast<gq::WsHeader*>(ws)->status : nullptr;
    return quant_any<false, false>(grads, dtype, a, grid_of(scheme), gq_code_bits(scheme, s),
                                   codes, nullptr, static_cast<cudaStream_t>(stream), status);
}

gq_status gq_quantize(const void* grads, int dtype, int64_t n, int64_t d, const float* norm_dev,
                      int scheme, int s, uint64_t seed, uint64_t step, void* codes,
                      void* stream) {
    return gq_quantize_ws(grads, dtype, n, d, norm_dev, scheme, s, seed, step, codes, nullptr, 0,
                          stream);
}

gq_status gq_reduce_codes(const void* codes, int scheme, int s, int64_t n, int64_t d,
                          int32_t* sum_dev, void* stream) {
    if (!codes || !sum_dev || !aligned16(codes) || !aligned16(sum_dev)) return GQ_ERR_INVALID;
    if (n < 1 || n >= (int64_t(1) << 31) || d < 1 || d >= kMaxD) return GQ_ERR_INVALID;
    gq_status st = check_scheme(scheme, s, n);
    if (st != GQ_OK) return st;
    const int bits = gq_code_bits(scheme, s);
    const int64_t row_bytes = gq_code_pitch(d) * bits / 8;
    const int64_t chunks = row_bytes / 16;
    scheme = grid_of(scheme);  // the sum does not depend on the rounding mode
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    const unsigned char* c = static_cast<const unsigned char*>(codes);
#define GQ_REDUCE(BITS, SCH)                                                     \
    do {                                                                         \
        auto k = gq::reduce_codes_kernel<BITS, SCH>;                             \
        k<<<grid_for(k, chunks), kThreads, 0, cs>>>(c, n, d, row_bytes, chunks, sum_dev); \
    } while (0)
    if (bits == 8) {
        if (scheme == GQ_LINEAR) GQ_REDUCE(8, gq::kLinear); else GQ_REDUCE(8, gq::kExp);
    } else {
        if (scheme == GQ_LINEAR) GQ_REDUCE(4, gq::kLinear); else GQ_REDUCE(4, gq::kExp);
    }
#undef GQ_REDUCE
    return launch_status();
}

gq_status gq_dequantize_sums(const void* sum_dev, int sum_type, const float* norm_dev, int scheme,
                             int s, int64_t n, int64_t d, void* out_dev, int out_dtype,
                             void* stream) {
    if (!sum_dev || !norm_dev || !out_dev || !aligned16(sum_dev) || !aligned16(out_dev))
        return GQ_ERR_INVALID;
    if (out_dtype != GQ_F32 && out_dtype != GQ_BF16 && out_dtype != GQ_F16) return GQ_ERR_INVALID;
    if (sum_type != GQ_SUM_I32 && sum_type != GQ_SUM_I8) return GQ_ERR_INVALID;
    if (n < 1 || n >= (int64_t(1) << 31) || d < 1 || d >= kMaxD) return GQ_ERR_INVALID;
    gq_status st = check_scheme(scheme, s, n);
    if (st != GQ_OK) return st;
    scheme = grid_of(scheme);  // dequantisation does not depend on the rounding mode
    if (sum_type == GQ_SUM_I8 && !fits_i8(scheme, s, n)) return GQ_ERR_OVERFLOW;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    const int64_t quads = (d + 3) / 4;
    const uint32_t su = static_cast<uint32_t>(s);
    const bool i8 = sum_type == GQ_SUM_I8;
    if (scheme == GQ_LINEAR) {
        auto k = i8 ? gq::dequantize_kernel<gq::kLinear, true> : gq::dequantize_kernel<gq::kLinear, false>;
        k<<<grid_for(k, quads), kThreads, 0, cs>>>(sum_dev, norm_dev, n, su, d, out_dev, out_dtype);
    } else {
        auto k = i8 ? gq::dequantize_kernel<gq::kExp, true> : gq::dequantize_kernel<gq::kExp, false>;
        k<<<grid_for(k, quads), kThreads, 0, cs>>>(sum_dev, norm_dev, n, su, d, out_dev, out_dtype);
    }
    return launch_status();
}

gq_status gq_dequantize_to(const int32_t* sum_dev, const float* norm_dev, int scheme, int s,
                           int64_t n, int64_t d, void* out_dev, int out_dtype, void* stream) {
    return gq_dequantize_sums(sum_dev, GQ_SUM_I32, norm_dev, scheme, s, n, d, out_dev, out_dtype,
                              stream);
}

gq_status gq_dequantize(const int32_t* sum_dev, const float* norm_dev, int scheme, int s,
                        int64_t n, int64_t d, float* out_dev, void* stream) {
    return gq_dequantize_to(sum_dev, norm_dev, scheme, s, n, d, out_dev, GQ_F32, stream);
}

gq_status gq_allreduce_mean_to(const void* grads, int dtype, int64_t n, int64_t d, int q, int p,
                               int scheme, int s, uint64_t seed, uint64_t step, void* out_dev,
                               int out_dtype, float* norm_dev, void* codes, void* ws,
                               size_t ws_bytes, void* stream) {
    gq_status st = check_grads(grads, dtype, n, d);
    if (st != GQ_OK) return st;
    const int mode = norm_mode(q, p);
    if (mode < 0) return GQ_ERR_INVALID;
    if (out_dtype != GQ_F32 && out_dtype != GQ_BF16 && out_dtype != GQ_F16) return GQ_ERR_INVALID;
    if ((st = check_scheme(scheme, s, n)) != GQ_OK) return st;
    if (!out_dev || !aligned16(out_dev) || (codes && !aligned16(codes))) return GQ_ERR_INVALID;
    if ((st = check_ws(ws, ws_bytes, n, d)) != GQ_OK) return st;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    const float* ws_norm = &reinterpret_cast<const gq::WsHeader*>(ws)->norm;
    gq::QuantArgs a = make_args(ws_norm, dtype, n, d, s, seed, step, scheme);
    a.out_dtype = out_dtype;
    // under the l2 norm over the coordinates ((2,2), (inf,2)) most |x| / N lie far below the
    // first level: the quantise pass defers the few uncertain row-groups (compacting consumer)
    a.compact = mode == gq::kL2L2 || mode == gq::kMaxL2;
    if (!codes) {  // small problems: one launch, the matrix read once
        unsigned char* w = static_cast<unsigned char*>(ws);
        bool taken = false;
        if (dtype == GQ_F32)
            st = grid_of(scheme) == GQ_LINEAR
                     ? resident_f32_l(grads, a, mode, out_dev, norm_dev, w, cs, &taken)
                     : resident_f32_e(grads, a, mode, out_dev, norm_dev, w, cs, &taken);
        else
            st = grid_of(scheme) == GQ_LINEAR
                     ? resident_bf16_l(grads, a, mode, out_dev, norm_dev, w, cs, &taken)
                     : resident_bf16_e(grads, a, mode, out_dev, norm_dev, w, cs, &taken);
        if (taken) return st;
    }
    if ((st = norm_any(grads, dtype, mode, n, d, norm_dev, ws, cs)) != GQ_OK) return st;
    unsigned int* status = &reinterpret_cast<gq::WsHeader*>(ws)->status;
    a.pdl = 1;  // the quantise pass's launch overlaps the norm pass's tail
    return quant_any<true, true>(grads, dtype, a, scheme, gq_code_bits(scheme, s), codes, out_dev,
                                 cs, status);
}

gq_status gq_allreduce_mean(const void* grads, int dtype, int64_t n, int64_t d, int q, int p,
                            int scheme, int s, uint64_t seed, uint64_t step, float* out_dev,
                            float* norm_dev, void* codes, void* ws, size_t ws_bytes,
                            void* stream) {
    return gq_allreduce_mean_to(grads, dtype, n, d, q, p, scheme, s, seed, step, out_dev, GQ_F32,
                                norm_dev, codes, ws, ws_bytes, stream);
}

gq_status gq_allreduce_mean_with_norm_ws(const void* grads, int dtype, int64_t n, int64_t d,
                                         const float* norm_dev, int scheme, int s, uint64_t seed,
                                         uint64_t step, float* out_dev, void* codes, void* ws,
                                         size_t ws_bytes, void* stream) {
    gq_status st = check_grads(grads, dtype, n, d);
    if (st != GQ_OK) return st;
    if ((st = check_scheme(scheme, s, n)) != GQ_OK) return st;
    if (!norm_dev || !out_dev || !aligned16(out_dev) || (codes && !aligned16(codes)))
        return GQ_ERR_INVALID;
    if (ws && (st = check_ws(ws, ws_bytes, n, d)) != GQ_OK) return st;
    const gq::QuantArgs a = make_args(norm_dev, dtype, n, d, s, seed, step, scheme);
    unsigned int* status = ws ? &reinterpret_cast<gq::WsHeader*>(ws)->status : nullptr;
    return quant_any<true, false>(grads, dtype, a, scheme, gq_code_bits(scheme, s), codes,
                                  out_dev, static_cast<cudaStream_t>(stream), status);
}

gq_status gq_allreduce_mean_with_norm(const void* grads, int dtype, int64_t n, int64_t d,
                                      const float* norm_dev, int scheme, int s, uint64_t seed,
                                      uint64_t step, float* out_dev, void* codes, void* stream) {
    return gq_allreduce_mean_with_norm_ws(grads, dtype, n, d, norm_dev, scheme, s, seed, step,
                                          out_dev, codes, nullptr, 0, stream);
}

gq_status gq_philox4x32_10(const uint32_t* ctr_key_dev, uint32_t* out_dev, int64_t count,
                           void* stream) {
    if (!ctr_key_dev || !out_dev || count < 0 || count > (int64_t(1) << 40)) return GQ_ERR_INVALID;
    if (count == 0) return GQ_OK;
    const int64_t blocks = (count + kThreads - 1) / kThreads;
    if (blocks > INT32_MAX) return GQ_ERR_INVALID;
    gq::philox_kernel<<<static_cast<unsigned>(blocks), kThreads, 0,
                        static_cast<cudaStream_t>(stream)>>>(ctr_key_dev, out_dev, count);
    return launch_status();
}

gq_status gq_get_status(void* ws, void* stream) {
    if (!ws) return GQ_ERR_WORKSPACE;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(cs) != cudaSuccess) return GQ_ERR_CUDA;
    unsigned int v = 0;
    gq::WsHeader* hdr = static_cast<gq::WsHeader*>(ws);
    if (cudaMemcpy(&v, &hdr->status, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess)
        return GQ_ERR_CUDA;
    if (v != 0) {
        const unsigned int zero = 0;
        if (cudaMemcpy(&hdr->status, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess)
            return GQ_ERR_CUDA;
        // a wait that gave up may have left a completion ticket or the grid barrier's arrival
        // counts short of a full set: start them again from zero
        if (v == GQ_ERR_TIMEOUT &&
            (cudaMemcpy(&hdr->ticket, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess ||
             cudaMemcpy(&hdr->bar, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess))
            return GQ_ERR_CUDA;
    }
    return static_cast<gq_status>(v);
}

int gq_debug_status(void) {
#ifdef GQ_DEBUG
    if (cudaDeviceSynchronize() != cudaSuccess) return -2;
    const unsigned int words[5] = {gq::debug_word_take(), debug_word_f32_l(), debug_word_f32_e(),
                                   debug_word_bf16_l(), debug_word_bf16_e()};
    for (unsigned int w : words)
        if (w != 0u) return w == 0xFFFFFFFFu ? -2 : static_cast<int>(w);
    return 0;
#else
    return -1;
#endif
}

const char* gq_status_string(int status) {
    switch (status) {
        case GQ_OK: return "ok";
        case GQ_ERR_INVALID: return "invalid argument";
        case GQ_ERR_UNSUPPORTED: return "unsupported number of levels";
        case GQ_ERR_OVERFLOW: return "code sum would overflow the exact fp32 range";
        case GQ_ERR_NONFINITE: return "non-finite norm";
        case GQ_ERR_TIMEOUT: return "device wait timed out";
        case GQ_ERR_CUDA: return "CUDA error";
        case GQ_ERR_WORKSPACE: return "workspace null, too small or misaligned";
        default: return "unknown status";
    }
}

}  // extern "C"

// ---- allocation-free variant of gq_allreduce_mean ------------------------------------------
// Some callers cannot allocate device memory at the point where they need the allreduce: code
// that runs inside a framework's caching allocator or communication hook (where re-entering
// the allocator is not allowed), or a process whose device memory is fully planned ahead.
// This entry point takes the norm step's scratch (status word, completion ticket, norm and the
// per-block partials) from a fixed array in the library's own device memory instead of a
// caller-provided workspace.
namespace {

constexpr int kNoAllocPartials = 1024;  // block partials the fixed scratch holds
constexpr size_t kNoAllocScratchBytes =
    static_cast<size_t>(gq::kHeaderBytes) + sizeof(uint64_t) * kNoAllocPartials;  // 8,448 B

// Every GPU that loads the library holds this array until the process exits.  In host code the
// name is only a host-side stand-in: its device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the fixed scratch on the current device, looked up once per device.
gq_status noalloc_scratch(unsigned char** out) {
    static void* addr[kMaxDevices] = {nullptr};
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GQ_ERR_CUDA;
    std::lock_guard<std::mutex> lock(mu);
    if (addr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
            return GQ_ERR_CUDA;
        addr[dev] = p;
    }
    *out = static_cast<unsigned char*>(addr[dev]);
    return GQ_OK;
}

// Blocks the norm step launches for this problem (the same rule as gq_global_norm).
int64_t norm_blocks_any(int dtype, int mode, int64_t n, int64_t d) {
    if (dtype == GQ_F32) {
        switch (mode) {
            case gq::kMaxMax: return norm_grid<float, gq::kMaxMax>(n, d);
            case gq::kL2L2: return norm_grid<float, gq::kL2L2>(n, d);
            case gq::kL2Max: return norm_grid<float, gq::kL2Max>(n, d);
            default: return norm_grid<float, gq::kMaxL2>(n, d);
        }
    }
    switch (mode) {
        case gq::kMaxMax: return norm_grid<uint16_t, gq::kMaxMax>(n, d);
        case gq::kL2L2: return norm_grid<uint16_t, gq::kL2L2>(n, d);
        case gq::kL2Max: return norm_grid<uint16_t, gq::kL2Max>(n, d);
        default: return norm_grid<uint16_t, gq::kMaxL2>(n, d);
    }
}

}  // namespace

extern "C" int64_t gq_norm_blocks(int dtype, int64_t n, int64_t d, int q, int p) {
    if ((dtype != GQ_F32 && dtype != GQ_BF16) || n < 1 || n >= (int64_t(1) << 31) || d < 1 ||
        d >= kMaxD)
        return 0;
    const int mode = norm_mode(q, p);
    return mode < 0 ? 0 : norm_blocks_any(dtype, mode, n, d);
}

extern "C" int64_t gq_noalloc_max_blocks(void) { return kNoAllocPartials; }

extern "C" gq_status gq_allreduce_mean_noalloc(const void* grads, int dtype, int64_t n, int64_t d,
                                               int q, int p, int scheme, int s, uint64_t seed,
                                               uint64_t step, float* out_dev, float* norm_dev,
                                               void* codes, void* stream) {
    gq_status st = check_grads(grads, dtype, n, d);
    if (st != GQ_OK) return st;
    const int mode = norm_mode(q, p);
    if (mode < 0) return GQ_ERR_INVALID;
    if ((st = check_scheme(scheme, s, n)) != GQ_OK) return st;
    if (!out_dev || !aligned16(out_dev) || (codes && !aligned16(codes))) return GQ_ERR_INVALID;
    // the fixed scratch holds kNoAllocPartials block partials: refuse a launch that needs more
    if (norm_blocks_any(dtype, mode, n, d) > kNoAllocPartials) return GQ_ERR_WORKSPACE;
    unsigned char* ws = nullptr;
    if ((st = noalloc_scratch(&ws)) != GQ_OK) return st;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    // the array keeps the previous call's contents: the status word, the completion ticket and
    // the single launch's barrier word must start at zero
    if (cudaMemsetAsync(ws, 0, gq::kHeaderBytes, cs) != cudaSuccess) return GQ_ERR_CUDA;
    const float* ws_norm = &reinterpret_cast<const gq::WsHeader*>(ws)->norm;
    gq::QuantArgs a = make_args(ws_norm, dtype, n, d, s, seed, step, scheme);
    a.compact = mode == gq::kL2L2 || mode == gq::kMaxL2;  // as gq_allreduce_mean chooses
    if (!codes) {  // small problems: the single launch (its partials fit the scratch too)
        bool taken = false;
        if (dtype == GQ_F32)
            st = grid_of(scheme) == GQ_LINEAR ? resident_f32_l(grads, a, mode, out_dev, norm_dev, ws, cs, &taken)
                                     : resident_f32_e(grads, a, mode, out_dev, norm_dev, ws, cs, &taken);
        else
            st = grid_of(scheme) == GQ_LINEAR ? resident_bf16_l(grads, a, mode, out_dev, norm_dev, ws, cs, &taken)
                                     : resident_bf16_e(grads, a, mode, out_dev, norm_dev, ws, cs, &taken);
        if (taken) return st;
    }
    if ((st = norm_any(grads, dtype, mode, n, d, norm_dev, ws, cs)) != GQ_OK) return st;
    // the scratch's status word lets large aligned problems take the bulk-copy kernel, as
    // gq_allreduce_mean does (its bounded waits record a timeout there; nothing reads it back)
    unsigned int* status = &reinterpret_cast<gq::WsHeader*>(ws)->status;
    a.pdl = 1;
    return quant_any<true, true>(grads, dtype, a, scheme, gq_code_bits(scheme, s), codes, out_dev,
                                 cs, status);
}

// ---- Global-E allreduce with re-rounding at every hop --------------------------------------
namespace {

gq::ExpArgs make_exp_args(uint64_t seed, uint64_t step) {
    gq::ExpArgs ea;
    const uint32_t k0 = static_cast<uint32_t>(seed), k1 = static_cast<uint32_t>(seed >> 32);
    for (int r = 0; r < 10; ++r) {  // Philox round keys: the key advanced by r Weyl steps
        ea.rk[2 * r] = k0 + static_cast<uint32_t>(r) * 0x9E3779B9u;
        ea.rk[2 * r + 1] = k1 + static_cast<uint32_t>(r) * 0xBB67AE85u;
    }
    ea.step_lo = static_cast<uint32_t>(step);
    ea.step_hi = static_cast<uint32_t>(step >> 32);
    return ea;
}

}  // namespace

extern "C" uint32_t gq_exp_tree_stream(int level, int64_t m) {
    return 0x80000000u + (static_cast<uint32_t>(level) << 24) + static_cast<uint32_t>(m);
}

extern "C" uint32_t gq_exp_ring_stream(int64_t h, int64_t c) {
    return 0xC0000000u + (static_cast<uint32_t>(h) << 12) + static_cast<uint32_t>(c);
}

extern "C" gq_status gq_exp_combine(const int8_t* a, const int8_t* b, int64_t d, int64_t j0,
                                    uint64_t seed, uint64_t step, uint32_t stream_id, int8_t* out,
                                    void* stream) {
    if (!a || !b || !out || !aligned16(a) || !aligned16(b) || !aligned16(out)) return GQ_ERR_INVALID;
    if (d < 1 || j0 < 0 || j0 % 8 != 0 || j0 + d >= kMaxD) return GQ_ERR_INVALID;
    auto k = gq::exp_combine_kernel;
    const int64_t chunks = (d + 15) / 16;
    k<<<grid_for(k, chunks), kThreads, 0, static_cast<cudaStream_t>(stream)>>>(
        a, b, d, j0, stream_id, make_exp_args(seed, step), out);
    return launch_status();
}

extern "C" gq_status gq_exp_allreduce(const void* codes, int s, int64_t n, int64_t d, int order,
                                      const float* norm_dev, uint64_t seed, uint64_t step,
                                      float* out_dev, int8_t* root_codes, void* stream) {
    if (!codes || !norm_dev || !out_dev || !aligned16(codes) || !aligned16(out_dev))
        return GQ_ERR_INVALID;
    if (n < 1 || n > gq::kExpMaxWorkers || d < 1 || d >= kMaxD) return GQ_ERR_INVALID;
    if (order != GQ_ORDER_TREE && order != GQ_ORDER_RING) return GQ_ERR_INVALID;
    gq_status st = check_scheme(GQ_EXP, s, n);
    if (st != GQ_OK) return st;
    const int bits = gq_code_bits(GQ_EXP, s);
    const int64_t pitch = gq_code_pitch(d);
    const gq::ExpArgs ea = make_exp_args(seed, step);
    const unsigned char* c = static_cast<const unsigned char*>(codes);
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    const uint32_t su = static_cast<uint32_t>(s);
#define GQ_EXP_ALLREDUCE(ORD, BITS)                                                            \
    do {                                                                                       \
        auto k = gq::exp_allreduce_kernel<ORD, BITS>;                                          \
        k<<<grid_for(k, d), kThreads, 0, cs>>>(c, n, d, pitch, ea, norm_dev, su, out_dev,      \
                                               root_codes);                                    \
    } while (0)
    if (order == GQ_ORDER_TREE) {
        if (bits == 4) GQ_EXP_ALLREDUCE(0, 4); else GQ_EXP_ALLREDUCE(0, 8);
    } else {
        if (bits == 4) GQ_EXP_ALLREDUCE(1, 4); else GQ_EXP_ALLREDUCE(1, 8);
    }
#undef GQ_EXP_ALLREDUCE
    return launch_status();
}

extern "C" gq_status gq_exp_dequantize(const int8_t* codes, int64_t d, const float* norm_dev,
                                       int s, int64_t n, void* out_dev, int out_dtype,
                                       void* stream) {
    if (!codes || !norm_dev || !out_dev || !aligned16(codes) || !aligned16(out_dev))
        return GQ_ERR_INVALID;
    if (out_dtype != GQ_F32 && out_dtype != GQ_BF16 && out_dtype != GQ_F16) return GQ_ERR_INVALID;
    if (d < 1 || d >= kMaxD || n < 1 || n >= (int64_t(1) << 31)) return GQ_ERR_INVALID;
    if (s < 1 || s > 24) return GQ_ERR_UNSUPPORTED;
    auto k = gq::exp_dequantize_kernel;
    k<<<grid_for(k, (d + 15) / 16), kThreads, 0, static_cast<cudaStream_t>(stream)>>>(
        codes, d, norm_dev, static_cast<uint32_t>(s), n, out_dev, out_dtype);
    return launch_status();
}

// ---- one rank's share of a multi-GPU allreduce ---------------------------------------------
extern "C" gq_status gq_norm_partial(const void* grads, int dtype, int64_t m, int64_t d, int q,
                                     int p, double* part_dev, void* ws, size_t ws_bytes,
                                     void* stream) {
    gq_status st = check_grads(grads, dtype, m, d);
    if (st != GQ_OK) return st;
    const int mode = norm_mode(q, p);
    if (mode < 0 || !part_dev) return GQ_ERR_INVALID;
    if (mode != gq::kMaxMax && mode != gq::kL2L2) return GQ_ERR_UNSUPPORTED;
    if ((st = check_ws(ws, ws_bytes, m, d)) != GQ_OK) return st;
    return norm_any(grads, dtype, mode, m, d, nullptr, ws, static_cast<cudaStream_t>(stream),
                    part_dev);
}

extern "C" gq_status gq_norm_finish(const double* part_dev, int q, int p, float* norm_dev,
                                    void* stream) {
    const int mode = norm_mode(q, p);
    if (mode < 0 || !part_dev || !norm_dev) return GQ_ERR_INVALID;
    if (mode != gq::kMaxMax && mode != gq::kL2L2) return GQ_ERR_UNSUPPORTED;
    gq::norm_finish_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
        part_dev, mode == gq::kL2L2, norm_dev);
    return launch_status();
}

extern "C" gq_status gq_quantize_sum(const void* grads, int dtype, int64_t m, int64_t d,
                                     int64_t worker0, const float* norm_dev, int scheme, int s,
                                     uint64_t seed, uint64_t step, void* sum_dev, int sum_type,
                                     void* ws, size_t ws_bytes, void* stream) {
    gq_status st = check_grads(grads, dtype, m, d);
    if (st != GQ_OK) return st;
    if ((st = check_scheme(scheme, s, m)) != GQ_OK) return st;
    if (!norm_dev || !sum_dev || !aligned16(sum_dev)) return GQ_ERR_INVALID;
    if (sum_type != GQ_SUM_I32 && sum_type != GQ_SUM_I8) return GQ_ERR_INVALID;
    if (worker0 < 0 || worker0 + m > (int64_t(1) << 31)) return GQ_ERR_INVALID;
    if (sum_type == GQ_SUM_I8 && !fits_i8(scheme, s, m)) return GQ_ERR_OVERFLOW;
    if (ws && (st = check_ws(ws, ws_bytes, m, d)) != GQ_OK) return st;
    gq::QuantArgs a = make_args(norm_dev, dtype, m, d, s, seed, step, scheme);
    a.row0 = static_cast<uint32_t>(worker0);
    a.sums = sum_dev;
    a.sums_i8 = sum_type == GQ_SUM_I8;
    unsigned int* status = ws ? &reinterpret_cast<gq::WsHeader*>(ws)->status : nullptr;
    return quant_any<true, false>(grads, dtype, a, scheme, gq_code_bits(scheme, s), nullptr,
                                  nullptr, static_cast<cudaStream_t>(stream), status);
}

// ---- segmented form: many n x d_l problems in two launches per kSegChunk segments -----------
namespace {

template <typename T, int MODE>
gq_status run_norm_segments(gq::SegLaunch& L, const int64_t* d, int64_t n, int scheme, int s,
                            float* norms_user, unsigned char* ws, cudaStream_t st) {
    constexpr int C = gq::Elem<T>::kCols;
    auto k = gq::norm_segments_kernel<T, MODE>;
    const int64_t full = static_cast<int64_t>(blocks_per_sm(k)) * sm_count();
    int64_t target = 2 * full;
    if (target > gq::kMaxPartials - L.nseg) target = gq::kMaxPartials - L.nseg;
    plan_runs(L, d, n, C, target);
    k<<<total_blocks(L), kThreads, 0, st>>>(L, n, scheme, static_cast<uint32_t>(s), norms_user,
                                            ws);
    return launch_status();
}

template <typename T>
gq_status norm_segments_any(int mode, gq::SegLaunch& L, const int64_t* d, int64_t n, int scheme,
                            int s, float* norms_user, unsigned char* ws, cudaStream_t st) {
    switch (mode) {
        case gq::kMaxMax:
            return run_norm_segments<T, gq::kMaxMax>(L, d, n, scheme, s, norms_user, ws, st);
        case gq::kL2L2:
            return run_norm_segments<T, gq::kL2L2>(L, d, n, scheme, s, norms_user, ws, st);
        case gq::kL2Max:
            return run_norm_segments<T, gq::kL2Max>(L, d, n, scheme, s, norms_user, ws, st);
        default:
            return run_norm_segments<T, gq::kMaxL2>(L, d, n, scheme, s, norms_user, ws, st);
    }
}

}  // namespace

extern "C" gq_status gq_allreduce_mean_segments(int64_t nseg, const void* const* grads,
                                                const int64_t* d, int dtype, int64_t n, int q,
                                                int p, int scheme, int s, uint64_t seed,
                                                uint64_t step, void* const* out, int out_dtype,
                                                float* norms_dev, void* ws, size_t ws_bytes,
                                                void* stream) {
    if (nseg < 1 || nseg > 65536 || !grads || !d || !out) return GQ_ERR_INVALID;
    if (out_dtype != GQ_F32 && out_dtype != GQ_BF16 && out_dtype != GQ_F16) return GQ_ERR_INVALID;
    if (step >= (uint64_t(1) << 48)) return GQ_ERR_INVALID;
    gq_status st;
    for (int64_t l = 0; l < nseg; ++l) {
        if ((st = check_grads(grads[l], dtype, n, d[l])) != GQ_OK) return st;
        if (!out[l] || !aligned16(out[l])) return GQ_ERR_INVALID;
    }
    const int mode = norm_mode(q, p);
    if (mode < 0) return GQ_ERR_INVALID;
    if ((st = check_scheme(scheme, s, n)) != GQ_OK) return st;
    if ((st = check_ws(ws, ws_bytes, n, 1)) != GQ_OK) return st;
    unsigned char* w = static_cast<unsigned char*>(ws);
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    gq::QuantArgs base = make_args(nullptr, dtype, n, 1, s, seed, step << 16, scheme);
    base.out_dtype = out_dtype;
    gq::SegLaunch L;  // ~8 KB of kernel parameters per launch
    for (int64_t c0 = 0; c0 < nseg; c0 += gq::kSegChunk) {
        const int64_t m = nseg - c0 < gq::kSegChunk ? nseg - c0 : gq::kSegChunk;
        std::memset(&L, 0, sizeof(L));
        L.nseg = static_cast<int32_t>(m);
        L.seg0 = static_cast<int32_t>(c0);
        for (int64_t k = 0; k < m; ++k) {
            L.seg[k].x = grads[c0 + k];
            L.seg[k].out = out[c0 + k];
        }
        st = dtype == GQ_F32
                 ? norm_segments_any<float>(mode, L, d + c0, n, grid_of(scheme), s, norms_dev, w, cs)
                 : norm_segments_any<uint16_t>(mode, L, d + c0, n, grid_of(scheme), s, norms_dev, w, cs);
        if (st != GQ_OK) return st;
        if (dtype == GQ_F32)
            st = grid_of(scheme) == GQ_LINEAR ? quant_segments_f32_l(L, d + c0, n, base, w, cs)
                                     : quant_segments_f32_e(L, d + c0, n, base, w, cs);
        else
            st = grid_of(scheme) == GQ_LINEAR ? quant_segments_bf16_l(L, d + c0, n, base, w, cs)
                                     : quant_segments_bf16_e(L, d + c0, n, base, w, cs);
        if (st != GQ_OK) return st;
    }
    return GQ_OK;
}

// ---- self-test of the bounded waits ---------------------------------------------------------
extern "C" gq_status gq_selftest_wait_timeout(void* ws, size_t ws_bytes, uint64_t limit_ns,
                                              unsigned long long* elapsed_dev, void* stream) {
    gq_status st = check_ws(ws, ws_bytes, 1, 1);
    if (st != GQ_OK) return st;
    if (!elapsed_dev || limit_ns < 1000 || limit_ns > 4000000000ull) return GQ_ERR_INVALID;
    unsigned int* status = &static_cast<gq::WsHeader*>(ws)->status;
    gq::wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(status, limit_ns,
                                                                              elapsed_dev);
    return launch_status();
}

extern "C" gq_status gq_quantize_codes(const void* grads, int dtype, int64_t m, int64_t d,
                                       int64_t worker0, const float* norm_dev, int scheme, int s,
                                       uint64_t seed, uint64_t step, void* codes, int code_bits,
                                       void* ws, size_t ws_bytes, void* stream) {
    gq_status st = check_grads(grads, dtype, m, d);
    if (st != GQ_OK) return st;
    if ((st = check_scheme(scheme, s, m)) != GQ_OK) return st;
    if (!norm_dev || !codes || !aligned16(codes)) return GQ_ERR_INVALID;
    if (code_bits != 8 && !(code_bits == 4 && s <= 7)) return GQ_ERR_INVALID;
    if (worker0 < 0 || worker0 + m > (int64_t(1) << 31)) return GQ_ERR_INVALID;
    if (ws && (st = check_ws(ws, ws_bytes, m, d)) != GQ_OK) return st;
    gq::QuantArgs a = make_args(norm_dev, dtype, m, d, s, seed, step, scheme);
    a.row0 = static_cast<uint32_t>(worker0);
    unsigned int* status = ws ? &reinterpret_cast<gq::WsHeader*>(ws)->status : nullptr;
    return quant_any<false, false>(grads, dtype, a, scheme, code_bits, codes, nullptr,
                                   static_cast<cudaStream_t>(stream), status);
}
