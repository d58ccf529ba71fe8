// gq_quant.cuh -- quantise launch templates, instantiated once per (gradient type, scheme) by
// gq_quant_<type>_<scheme>.cu.
#pragma once
#include "gq_host.cuh"

namespace gqh {

// A kernel launch, programmatically dependent on the previous kernel on the stream when pdl
// (the quantise pass after the norm pass of the fused call: its launch overlaps the norm pass's
// tail, and the kernel waits for the norm in griddepcontrol.wait).
template <typename... P, typename... A>
gq_status launch(void (*kernel)(P...), unsigned grid, unsigned block, size_t smem,
                 cudaStream_t st, bool pdl, A... args) {
    if (!pdl) {
        kernel<<<grid, block, smem, st>>>(args...);
        return launch_status();
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...) == cudaSuccess ? GQ_OK : GQ_ERR_CUDA;
}

// ---- quantize (+ sum + dequantize) ----------------------------------------------------------
// TRUSTED: the norm comes from norm_kernel on the same gradients (fused path), so a finite norm
// rules out NaN and infinite elements.
// Problems with at least one 3840-column chunk per SM of 16-byte aligned rows take the kernel
// fed by bulk copies (it needs a status word for its bounded waits); the rest the direct one.
template <typename T, int SCHEME, int BITS, bool OUT, bool TRUSTED>
gq_status run_quant(const void* grads, const gq::QuantArgs& a, void* codes, void* out,
                    cudaStream_t st, unsigned int* status = nullptr) {
    const int64_t groups = BITS ? a.pitch / gq::kQCols : (a.d + gq::kQCols - 1) / gq::kQCols;
    const int64_t chunks = (a.d / gq::kQCols) / gq::kTmaConsumers;
    if (status && a.vec_rows && chunks >= sm_count()) {
        auto kt = gq::quantize_tma_kernel<T, SCHEME, BITS, OUT, TRUSTED, 2, true>;
        int tsmem = gq::TmaCfg<T>::kSmemBytes;
        // One or two workers (one rank's share of a multi-GPU call; small fused calls): ring
        // stages of one or two rows, as many as the ring holds, so that as many bytes stay in
        // flight as with four-row stages.
        if constexpr ((BITS == 0 && OUT) || (BITS != 0 && !OUT && !TRUSTED)) {
            if (a.n == 1)
                kt = gq::quantize_tma_kernel<T, SCHEME, BITS, OUT, TRUSTED, 1, true, false, 1>;
        }
        if constexpr (BITS == 0 && OUT && TRUSTED) {
            if (a.n == 2)
                kt = gq::quantize_tma_kernel<T, SCHEME, BITS, OUT, TRUSTED, 2, true, false, 2>;
            // under an l2 norm over all coordinates most elements round down: the compacting
            // consumer
            if (a.compact) {
                kt = a.n == 1   ? gq::quantize_tma_kernel<T, SCHEME, BITS, OUT, TRUSTED, 2, false,
                                                          true, 1>
                     : a.n == 2 ? gq::quantize_tma_kernel<T, SCHEME, BITS, OUT, TRUSTED, 2, false,
                                                          true, 2>
                                : gq::quantize_tma_kernel<T, SCHEME, BITS, OUT, TRUSTED, 2, false,
                                                          true>;
                tsmem = gq::CompactCfg<T>::kSmemBytes;
            }
        }
        if (blocks_per_sm(kt, tsmem, gq::kTmaBlock) < 1) return GQ_ERR_CUDA;
        const unsigned grid = static_cast<unsigned>(sm_count());
        return launch(kt, grid, gq::kTmaBlock, tsmem, st, a.pdl != 0, static_cast<const T*>(grads),
                      a, groups, static_cast<unsigned char*>(codes), out, status);
    }
    auto k = gq::quantize_kernel<T, SCHEME, BITS, OUT, TRUSTED>;
    constexpr int smem = gq::Staging<T>::kBytes;
    const unsigned grid = grid_for(k, groups, INT32_MAX, smem);
    return launch(k, grid, kThreads, smem, st, a.pdl != 0, static_cast<const T*>(grads), a, groups,
                  static_cast<unsigned char*>(codes), out);
}

template <typename T, int SCHEME, bool OUT, bool TRUSTED>
gq_status quant_bits(const void* grads, const gq::QuantArgs& a, int bits, void* codes, void* out,
                     cudaStream_t st, unsigned int* status) {
    if (!codes) return run_quant<T, SCHEME, 0, OUT, TRUSTED>(grads, a, nullptr, out, st, status);
    if (bits == 4) return run_quant<T, SCHEME, 4, OUT, TRUSTED>(grads, a, codes, out, st, status);
    return run_quant<T, SCHEME, 8, OUT, TRUSTED>(grads, a, codes, out, st, status);
}


template <typename T, int SCHEME>
gq_status run_quant_segments(gq::SegLaunch& L, const int64_t* d, int64_t n,
                             const gq::QuantArgs& base, unsigned char* ws, cudaStream_t st) {
    // Chunks of 3840 columns for every segment whose rows are 16-byte aligned; with at least one
    // chunk per SM they all go through the bulk-copy ring (runs b0 / nb now count chunks).
    // The groups outside the chunks (a ragged last group, or all groups of a segment without
    // chunks) are numbered across the launch: segment k's start at t0.
    constexpr int vec = 16 / static_cast<int>(sizeof(T));
    int32_t chunks = 0;
    int64_t tails = 0;
    for (int k = 0; k < L.nseg; ++k) {
        const int64_t full = d[k] % vec == 0 ? d[k] / gq::kQCols : 0;
        const int64_t nc = (full + gq::kTmaConsumers - 1) / gq::kTmaConsumers;
        L.seg[k].d = d[k];
        L.seg[k].b0 = chunks;
        L.seg[k].nb = static_cast<int32_t>(nc);
        L.seg[k].t0 = tails;
        chunks += static_cast<int32_t>(nc);
        tails += (d[k] + gq::kQCols - 1) / gq::kQCols - (nc > 0 ? full : 0);
    }
    L.ntail = tails;
    if (chunks >= sm_count()) {
        auto kt = gq::quantize_seg_tma_kernel<T, SCHEME>;
        constexpr int tsmem = gq::TmaCfg<T>::kSmemBytes;
        if (blocks_per_sm(kt, tsmem, gq::kTmaBlock) < 1) return GQ_ERR_CUDA;
        kt<<<static_cast<unsigned>(sm_count()), gq::kTmaBlock, tsmem, st>>>(L, base, chunks, ws);
        return launch_status();
    }
    auto k = gq::quantize_segments_kernel<T, SCHEME>;
    constexpr int smem = gq::Staging<T>::kBytes;
    const int64_t full = static_cast<int64_t>(blocks_per_sm(k, smem)) * sm_count();
    plan_runs(L, d, n, gq::kQCols, full);
    k<<<total_blocks(L), kThreads, smem, st>>>(L, base, ws);
    return launch_status();
}


// ---- single launch for problems that fit in shared memory ------------------------------------
template <typename T, int SCHEME, int MODE>
gq_status launch_resident(const T* x, const gq::QuantArgs& a, int64_t gpb, unsigned nblk,
                          size_t smem, void* out, float* norm_user, unsigned char* ws,
                          cudaStream_t st) {
    auto k = gq::resident_kernel<T, SCHEME, MODE>;
    if (blocks_per_sm(k, gq::kResTileBytes, gq::kResThreads) < 1) return GQ_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(nblk);
    cfg.blockDim = dim3(gq::kResThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;  // all blocks resident: they wait on each other
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k, x, a, gpb, out, norm_user, ws) == cudaSuccess ? GQ_OK
                                                                                     : GQ_ERR_CUDA;
}

// The fused call in one launch when the problem fits (aligned rows, no codes requested):
// *taken tells whether it ran.  A cooperative launch the device refuses (too many blocks for
// what is free of it) is not taken, and the two-pass form runs instead.
template <typename T, int SCHEME>
gq_status run_resident(const void* grads, const gq::QuantArgs& a, int mode, void* out,
                       float* norm_user, unsigned char* ws, cudaStream_t st, bool* taken) {
    int64_t gpb = 0;
    unsigned nblk = 0;
    size_t smem = 0;
    *taken = false;
    if (!a.vec_rows || !resident_plan(a.n, a.d, static_cast<int>(sizeof(T)), &gpb, &nblk, &smem))
        return GQ_OK;
    const T* x = static_cast<const T*>(grads);
    gq_status st_launch;
    switch (mode) {
        case gq::kMaxMax:
            st_launch = launch_resident<T, SCHEME, gq::kMaxMax>(x, a, gpb, nblk, smem, out, norm_user, ws, st);
            break;
        case gq::kL2L2:
            st_launch = launch_resident<T, SCHEME, gq::kL2L2>(x, a, gpb, nblk, smem, out, norm_user, ws, st);
            break;
        case gq::kL2Max:
            st_launch = launch_resident<T, SCHEME, gq::kL2Max>(x, a, gpb, nblk, smem, out, norm_user, ws, st);
            break;
        default:
            st_launch = launch_resident<T, SCHEME, gq::kMaxL2>(x, a, gpb, nblk, smem, out, norm_user, ws, st);
    }
    if (st_launch != GQ_OK) {
        cudaGetLastError();  // a refused launch leaves no lasting error
        return GQ_OK;
    }
    *taken = true;
    return GQ_OK;
}

template <typename T, int SCHEME>
gq_status quant_entry(const void* grads, const gq::QuantArgs& a, int bits, bool out, bool trusted,
                      void* codes, void* outp, cudaStream_t st, unsigned int* status) {
    if (!out) return quant_bits<T, SCHEME, false, false>(grads, a, bits, codes, outp, st, status);
    if (trusted) return quant_bits<T, SCHEME, true, true>(grads, a, bits, codes, outp, st, status);
    return quant_bits<T, SCHEME, true, false>(grads, a, bits, codes, outp, st, status);
}

}  // namespace gqh

// The two launchers of one (gradient type, scheme) pair.
#define GQH_DEFINE_QUANT(NAME, T, SCHEME)                                                         \
    gq_status gqh::quant_##NAME(const void* grads, const gq::QuantArgs& a, int bits, bool out,     \
                                bool trusted, void* codes, void* outp, cudaStream_t st,            \
                                unsigned int* status) {                                            \
        return quant_entry<T, SCHEME>(grads, a, bits, out, trusted, codes, outp, st, status);      \
    }                                                                                              \
    gq_status gqh::quant_segments_##NAME(gq::SegLaunch& L, const int64_t* d, int64_t n,           \
                                         const gq::QuantArgs& base, unsigned char* ws,             \
                                         cudaStream_t st) {                                        \
        return run_quant_segments<T, SCHEME>(L, d, n, base, ws, st);                               \
    }                                                                                              \
    gq_status gqh::resident_##NAME(const void* grads, const gq::QuantArgs& a, int mode, void* out, \
                                   float* norm_user, unsigned char* ws, cudaStream_t st,           \
                                   bool* taken) {                                                  \
        return run_resident<T, SCHEME>(grads, a, mode, out, norm_user, ws, st, taken);             \
    }                                                                                              \
    unsigned int gqh::debug_word_##NAME() { return gq::debug_word_take(); }
