// gq_kernels.cuh -- sm_103a kernels of the Global-QSGD compress / aggregate / decompress path.
//
// Method: "Global-QSGD: Practical Floatless Quantization for Distributed Learning with
// Theoretical Guarantees" (arXiv 2305.18627), cited as "Global-QSGD".  All kernels are
// HBM-bandwidth kernels (nothing here is a dense contraction): each thread owns a column group
// (8 coordinates in the quantise kernels) and walks the n worker rows of that group, so a warp
// reads contiguous bytes of one row per load; the (inf, inf) and (2, 2) norms read the matrix
// flat.  Grids are grid-stride loops sized to the resident capacity of the GPU (a multiple of
// its SM count); the bulk-copy quantise kernels and the single-launch form run one block per
// SM.  Every wait on another thread's progress (mbarrier, grid barrier) is bounded in time.
//
// Built with -fmad=false: every fp32 operation is a separately rounded IEEE operation, and the
// normalisation is the correctly rounded quotient (__fdiv_rn).
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace gq {

// Debug builds (-DGQ_DEBUG; compute-sanitizer stands in for nothing here): logical bounds checks
// at the kernels' stores and bulk copies.  A failed check records its source line in this
// translation unit's debug word and the kernel goes on (no trap); gq_debug_status reads and
// clears the words of all translation units.  Without GQ_DEBUG the checks compile to nothing.
#ifdef GQ_DEBUG
static __device__ unsigned int g_debug_word;
#define GQ_BOUND(cond)                                                                      \
    do {                                                                                    \
        if (!(cond)) atomicCAS(&::gq::g_debug_word, 0u, static_cast<unsigned int>(__LINE__)); \
    } while (0)
#else
#define GQ_BOUND(cond) \
    do {               \
    } while (0)
#endif

// This translation unit's debug word, read and cleared: 0 when no check failed (always 0 in a
// build without GQ_DEBUG), 0xFFFFFFFF if it could not be read.
static inline unsigned int debug_word_take() {
#ifdef GQ_DEBUG
    unsigned int v = 0u;
    const unsigned int zero = 0u;
    if (cudaMemcpyFromSymbol(&v, g_debug_word, sizeof v) != cudaSuccess) return 0xFFFFFFFFu;
    if (v != 0u && cudaMemcpyToSymbol(g_debug_word, &zero, sizeof zero) != cudaSuccess)
        return 0xFFFFFFFFu;
    return v;
#else
    return 0u;
#endif
}

constexpr int kThreads = 256;        // threads per block for every kernel
// output element types of the dequantised mean (the values of gq_dtype)
constexpr int kOutF32 = 0, kOutBF16 = 1, kOutF16 = 2;
constexpr int kMaxPartials = 4096;   // upper bound on norm-kernel blocks (workspace size)
constexpr int kHeaderBytes = 256;    // workspace header, then kMaxPartials 8-byte partials
constexpr int kSegChunk = 256;       // segments per launch of the segmented kernels
// after the partials: kSegChunk completion tickets, kSegChunk fp32 norms and kSegChunk fp32
// dequantisation scales (one each per segment of a segmented launch)
constexpr int kSegTicketsOff = kHeaderBytes + 8 * kMaxPartials;
constexpr int kSegNormsOff = kSegTicketsOff + 4 * kSegChunk;
constexpr int kSegScalesOff = kSegNormsOff + 4 * kSegChunk;  // fp32 dequantisation scales
constexpr int kWorkspaceBytes = kSegScalesOff + 4 * kSegChunk;

// Workspace header (device memory owned by the caller).
struct WsHeader {
    unsigned int status;  // sticky device-detected status (0 = ok)
    unsigned int ticket;  // blocks of the running norm kernel that have finished; 0 between calls
    float norm;           // fp32 norm written by the last norm kernel
    unsigned int bar;     // grid barrier of the single-launch kernel: generation << 8 | arrivals
    unsigned int pad[60];
};
static_assert(sizeof(WsHeader) == kHeaderBytes, "workspace header is 256 bytes");

enum NormMode { kMaxMax = 0, kL2L2 = 1, kL2Max = 2, kMaxL2 = 3 };  // (q, p) pairs
enum Scheme { kLinear = 0, kExp = 1 };

// The fp32 dequantisation scale from the fp32 norm, computed in fp64: N / (n s) for Global-L_s,
// N 2^-(s-1) / n for Global-E_s; 0 when the norm is 0 or not finite.
__device__ __forceinline__ float dequant_scale(int scheme, float nrm, int64_t n, uint32_t s) {
    if (!(nrm > 0.0f && nrm < __uint_as_float(0x7F800000u))) return 0.0f;
    const double num = static_cast<double>(nrm);
    return scheme == kLinear
               ? static_cast<float>(num / (static_cast<double>(n) * static_cast<double>(s)))
               : static_cast<float>(ldexp(num, -static_cast<int>(s - 1)) / static_cast<double>(n));
}

// Programmatic dependent launch between the two passes of the fused call: the norm kernel lets
// the launch of the kernel after it on the stream (the quantise pass) begin at once, and the
// quantise kernel waits, before reading anything, until the norm kernel has completed and its
// writes are visible.  Launched without the attribute, the wait returns at once.  Every norm
// kernel's grid is one wave of resident blocks, so the dependent blocks, which can only be
// placed where the norm blocks leave room, never hold back a norm block.
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ------------------------------------------------------------------------------------------
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11): ten rounds of the Philox-4x32 bijection.
// Each round multiplies counter words 0 and 2 by the round multipliers (full 64-bit products),
// xors the high halves into words 1 and 3 with the round key, and swaps; the key advances by
// the two Weyl constants between rounds.
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
    const uint32_t kMul0 = 0xD2511F53u, kMul1 = 0xCD9E8D57u;
    const uint32_t kWeyl0 = 0x9E3779B9u, kWeyl1 = 0xBB67AE85u;
#pragma unroll
    for (int round = 0; round < 10; ++round) {
        const uint32_t hi0 = __umulhi(kMul0, c.x), lo0 = kMul0 * c.x;
        const uint32_t hi1 = __umulhi(kMul1, c.z), lo1 = kMul1 * c.z;
        c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
        k0 += kWeyl0;
        k1 += kWeyl1;
    }
    return c;
}

// The same bijection with the ten round keys precomputed (rk[2r], rk[2r+1] = key words of
// round r); used by the quantise kernels, whose key is fixed for the whole launch.
__device__ __forceinline__ uint4 philox4x32_10_rk(uint4 c, const uint32_t (&rk)[20]) {
    const uint32_t kMul0 = 0xD2511F53u, kMul1 = 0xCD9E8D57u;
#pragma unroll
    for (int round = 0; round < 10; ++round) {
        const uint32_t hi0 = __umulhi(kMul0, c.x), lo0 = kMul0 * c.x;
        const uint32_t hi1 = __umulhi(kMul1, c.z), lo1 = kMul1 * c.z;
        c = make_uint4(hi1 ^ c.y ^ rk[2 * round], lo1, hi0 ^ c.w ^ rk[2 * round + 1], lo0);
    }
    return c;
}

// The same call for counter (g, row, step_lo, step_hi) split into the part that depends on the
// column group g only (computed once per group) and the rest (computed per row).  Rounds 1-3
// partly depend on g or on row alone: round 1's products are M0 g and M1 step_lo; round 2's are
// M0 (f(row)) and M1 (f(g)); round 3's first is M0 (f(g)).  Same outputs as philox4x32_10_rk.
struct PhiloxGroup {
    uint32_t lo0_1;   // round 1: low half of M0 g          (counter word 3 after round 1)
    uint32_t y2;      // round 2: low half of M1 z1         (counter word 1 after round 2)
    uint32_t z3k;     // round 3: high half of M0 x2, xor round-3 key word 1
    uint32_t lo0_3;   // round 3: low half of M0 x2         (counter word 3 after round 3)
};

__device__ __forceinline__ void mulhilo(uint32_t m, uint32_t a, uint32_t& hi, uint32_t& lo) {
    const uint64_t p = static_cast<uint64_t>(m) * a;
    hi = static_cast<uint32_t>(p >> 32);
    lo = static_cast<uint32_t>(p);
}

__device__ __forceinline__ PhiloxGroup philox_group(uint32_t g, uint32_t step_lo, uint32_t step_hi,
                                                    const uint32_t (&rk)[20]) {
    const uint32_t kMul0 = 0xD2511F53u, kMul1 = 0xCD9E8D57u;
    PhiloxGroup pg;
    uint32_t hi0, hi1s, lo1s, h, l;
    mulhilo(kMul0, g, hi0, pg.lo0_1);           // round 1, word 0 = g
    mulhilo(kMul1, step_lo, hi1s, lo1s);        // round 1, word 2 = step_lo
    const uint32_t z1 = hi0 ^ step_hi ^ rk[1];  // round 1 output word 2
    mulhilo(kMul1, z1, h, l);                   // round 2, word 2
    pg.y2 = l;
    const uint32_t x2 = h ^ lo1s ^ rk[2];       // round 2 output word 0 (round 1 word 1 = lo1s)
    mulhilo(kMul0, x2, h, l);                   // round 3, word 0
    pg.z3k = h ^ rk[5];
    pg.lo0_3 = l;
    return pg;
}

__device__ __forceinline__ uint4 philox_row(const PhiloxGroup& pg, uint32_t row, uint32_t step_lo,
                                            const uint32_t (&rk)[20]) {
    const uint32_t kMul0 = 0xD2511F53u, kMul1 = 0xCD9E8D57u;
    uint32_t hi1s, lo1s;
    mulhilo(kMul1, step_lo, hi1s, lo1s);        // round 1, word 2 (loop-invariant)
    const uint32_t x1 = hi1s ^ row ^ rk[0];     // round 1 output word 0
    uint32_t hi0, lo0;
    mulhilo(kMul0, x1, hi0, lo0);               // round 2, word 0
    const uint32_t z2 = hi0 ^ pg.lo0_1 ^ rk[3]; // round 2 output word 2 (round 1 word 3)
    uint32_t hi1, lo1;
    mulhilo(kMul1, z2, hi1, lo1);               // round 3, word 2
    uint4 c = make_uint4(hi1 ^ pg.y2 ^ rk[4], lo1, pg.z3k ^ lo0, pg.lo0_3);  // round 3 output
#pragma unroll
    for (int round = 3; round < 10; ++round) {
        mulhilo(kMul0, c.x, hi0, lo0);
        mulhilo(kMul1, c.z, hi1, lo1);
        c = make_uint4(hi1 ^ c.y ^ rk[2 * round], lo1, hi0 ^ c.w ^ rk[2 * round + 1], lo0);
    }
    return c;
}

// ------------------------------------------------------------------------------------------
// Element access: a 16-byte column group of one row, widened to fp32.
// ------------------------------------------------------------------------------------------
template <typename T> struct Elem;
template <> struct Elem<float> {
    static constexpr int kCols = 4;
    __device__ __forceinline__ static void load_vec(const float* p, float (&v)[4]) {
        const float4 t = __ldg(reinterpret_cast<const float4*>(p));
        v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
    }
    __device__ __forceinline__ static float load_one(const float* p) { return __ldg(p); }
};
// bf16 is the high half of a binary32 word: widening is a 16-bit shift of the bits.
template <> struct Elem<uint16_t> {
    static constexpr int kCols = 8;
    __device__ __forceinline__ static void load_vec(const uint16_t* p, float (&v)[8]) {
        const uint4 t = __ldg(reinterpret_cast<const uint4*>(p));
        const uint32_t w[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            v[2 * k] = __uint_as_float(w[k] << 16);
            v[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
        }
    }
    __device__ __forceinline__ static float load_one(const uint16_t* p) {
        return __uint_as_float(static_cast<uint32_t>(__ldg(p)) << 16);
    }
};

// Raw 16-byte column group g of row i (vector rows only; no bounds check) and its widening.
__device__ __forceinline__ uint4 load_raw16(const void* __restrict__ x, int64_t i, int64_t g,
                                            int64_t row_bytes) {
    return __ldg(reinterpret_cast<const uint4*>(static_cast<const unsigned char*>(x) +
                                                i * row_bytes) + g);
}
template <typename T>
__device__ __forceinline__ void widen16(const uint4& t, float (&v)[Elem<T>::kCols]) {
    if (sizeof(T) == 4) {
        v[0] = __uint_as_float(t.x); v[1] = __uint_as_float(t.y);
        v[2] = __uint_as_float(t.z); v[3] = __uint_as_float(t.w);
    } else {
        const uint32_t w[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            v[2 * k] = __uint_as_float(w[k] << 16);
            v[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
        }
    }
}

// Row i, column group g (columns g*C .. g*C+C-1) of the n x d matrix x, zero past column d.
template <typename T>
__device__ __forceinline__ void load_group(const T* __restrict__ x, int64_t i, int64_t g,
                                           int64_t d, bool vec_rows,
                                           float (&v)[Elem<T>::kCols]) {
    constexpr int C = Elem<T>::kCols;
    const int64_t j0 = g * C;
    const T* row = x + i * d;
    if (vec_rows && j0 + C <= d) {
        Elem<T>::load_vec(row + j0, v);
    } else {
#pragma unroll
        for (int c = 0; c < C; ++c) v[c] = (j0 + c < d) ? Elem<T>::load_one(row + j0 + c) : 0.0f;
    }
}

// 2^k as fp32 for k in [-149, 127] (exact: normal or subnormal power of two).
__device__ __forceinline__ float exp2i(int k) {
    return k >= -126 ? __int_as_float((k + 127) << 23) : __int_as_float(1 << (k + 149));
}

constexpr uint32_t kInfBits = 0x7F800000u;

// ------------------------------------------------------------------------------------------
// Sum of squares with a power-of-two scale (for the l2 norms).  Values are multiplied by
// f = 2^-E before squaring, where 2^(E+1) bounds every magnitude seen so far, so squares
// neither overflow nor vanish anywhere in the fp32 range; the squares are summed with Kahan
// compensation.  When a larger magnitude arrives the running sum is rescaled (rare).  NaN and
// infinite values flow through the arithmetic and leave the sum non-finite.
// ------------------------------------------------------------------------------------------
struct ScaledSumSq {
    float acc, comp;  // Kahan sum of (x * f)^2 and its running compensation
    float f;          // 2^-E
    float lim;        // 2^(E+1): magnitudes >= lim need a rescale first
    int e;            // E

    __device__ __forceinline__ void init() {
        acc = 0.0f; comp = 0.0f; e = -150; f = 1.0f; lim = exp2i(-149);  // any non-zero rescales
    }
    // Make 2^(E+1) bound the finite magnitude m >= lim.
    __device__ __forceinline__ void rescale(float m) {
        if (!(m < __uint_as_float(kInfBits))) return;  // Inf / NaN: left to the arithmetic
        const uint32_t eb = __float_as_uint(m) >> 23;
        const int ne = eb ? static_cast<int>(eb) - 127 : -127;  // m < 2^(ne+1)
        if (ne <= e) return;
        const int half = e - ne;  // the sum scales by 2^(2 half), half < 0
        if (half < -100) {
            acc = 0.0f;  // the old sum is below 2^-200 of one new square: negligible
            comp = 0.0f;
        } else {
            const float h = exp2i(half);
            acc = (acc * h) * h;
            comp = (comp * h) * h;
        }
        e = ne;
        f = exp2i(-ne);
        lim = (ne + 1 >= 128) ? __uint_as_float(kInfBits) : exp2i(ne + 1);
    }
    __device__ __forceinline__ void kahan_add(float y) {
        const float yy = y - comp;
        const float t = acc + yy;
        comp = (t - acc) - yy;
        acc = t;
    }
    // Add the squares of C values.
    template <int C>
    __device__ __forceinline__ void add(const float (&v)[C]) {
        float m = fabsf(v[0]);
#pragma unroll
        for (int c = 1; c < C; ++c) m = fmaxf(m, fabsf(v[c]));
        if (m >= lim) rescale(m);
        float sq[C];
#pragma unroll
        for (int c = 0; c < C; ++c) { const float t = v[c] * f; sq[c] = t * t; }
#pragma unroll
        for (int w = 1; w < C; w *= 2)
#pragma unroll
            for (int c = 0; c + w < C; c += 2 * w) sq[c] = sq[c] + sq[c + w];
        kahan_add(sq[0]);
    }
    __device__ __forceinline__ float sum() const { return acc - comp; }
    // The sum as fp64, scale removed: times 2^(2E), |2E| <= 300, an exact power of two in fp64.
    __device__ __forceinline__ double value() const {
        const double p2 = __longlong_as_double(static_cast<long long>(2 * e + 1023) << 52);
        return (static_cast<double>(acc) - static_cast<double>(comp)) * p2;
    }
};

// Order-preserving 64-bit key of c * 4^E for a normal positive fp32 c (maxima of scaled column
// norms without fp64 arithmetic per column): the exponent field extended past 8 bits.
__device__ __forceinline__ int64_t scaled_key(float c, int e) {
    return static_cast<int64_t>(__float_as_uint(c)) + (static_cast<int64_t>(2 * e) << 23);
}
// The fp64 value of a key (exact).
__device__ __forceinline__ double key_value(int64_t key) {
    const int64_t ex = (key >> 23) - 127;  // unbiased exponent of c * 4^E
    const uint64_t frac = static_cast<uint64_t>(key & 0x7FFFFF);
    const uint64_t bits = (static_cast<uint64_t>(ex + 1023) << 52) | (frac << 29);
    return __longlong_as_double(static_cast<long long>(bits));
}

// ------------------------------------------------------------------------------------------
// Block reductions (fixed order: deterministic for a given grid and block size).
// ------------------------------------------------------------------------------------------
// NT: threads of the block; sh holds NT / 32 values.
template <int NT = kThreads>
__device__ __forceinline__ double block_sum(double v, double* sh) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_down_sync(0xFFFFFFFFu, v, o);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) sh[warp] = v;
    __syncthreads();
    double r = 0.0;
    if (threadIdx.x == 0)
        for (int w = 0; w < NT / 32; ++w) r += sh[w];
    __syncthreads();
    return r;  // valid in thread 0
}
// Max over non-negative fp64 values by their bit patterns: NaN (sign clear) orders above +Inf,
// so a NaN anywhere wins.
template <int NT = kThreads>
__device__ __forceinline__ uint64_t block_max_bits(uint64_t v, uint64_t* sh) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const uint64_t t = __shfl_down_sync(0xFFFFFFFFu, v, o);
        v = t > v ? t : v;
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) sh[warp] = v;
    __syncthreads();
    uint64_t r = 0;
    if (threadIdx.x == 0)
        for (int w = 0; w < NT / 32; ++w) r = sh[w] > r ? sh[w] : r;
    __syncthreads();
    return r;
}

// ------------------------------------------------------------------------------------------
// Step 1: global norm ||x||_{q,p} (Global-QSGD, notation paragraph): the q-norm over the
// workers of every coordinate, then the p-norm over the coordinates.  One pass over x; each
// block writes one partial; the last block to finish (completion ticket, no waiting) combines
// the partials in index order and writes the fp32 norm.
// ------------------------------------------------------------------------------------------
// Where one norm's blocks leave their partials and the result.
struct NormSlots {
    uint64_t* partials;     // one per block of this norm
    unsigned int* ticket;   // completion count, zero between calls
    unsigned int* status;   // device status word
    float* norm;            // the fp32 norm (workspace copy)
    float* norm_user;       // nullable: the caller's copy
    double* part_user;      // nullable: the combinable value before the square root
    float* scale = nullptr; // nullable: the dequantisation scale of (scheme, s, n) below
    int scheme = 0;
    uint32_t s = 1;
    int64_t n = 1;
};

// The block's partial of a norm: a max or a sum, as a non-negative fp64 stored by its bits
// (valid in thread 0).  NT: threads of the block.
template <int MODE, int NT = kThreads>
__device__ __forceinline__ uint64_t block_partial(uint32_t maxbits, const ScaledSumSq& ssq,
                                                  int64_t best_key, uint32_t bad_col,
                                                  double* sh_d, uint64_t* sh_u) {
    if (MODE == kMaxMax) {
        const double m = static_cast<double>(__uint_as_float(maxbits));
        return block_max_bits<NT>(static_cast<uint64_t>(__double_as_longlong(m)), sh_u);
    } else if (MODE == kL2Max) {
        double m = best_key == INT64_MIN ? 0.0 : key_value(best_key);
        if (bad_col) m = static_cast<double>(__uint_as_float(bad_col));
        return block_max_bits<NT>(static_cast<uint64_t>(__double_as_longlong(m)), sh_u);
    } else {
        return static_cast<uint64_t>(__double_as_longlong(block_sum<NT>(ssq.value(), sh_d)));
    }
}

// The fixed-order combine of nb block partials (valid in thread 0): their max or their sum.
template <int MODE, int NT = kThreads>
__device__ __forceinline__ double combine_partials(const uint64_t* partials, int nb, double* sh_d,
                                                   uint64_t* sh_u) {
    if (MODE == kMaxMax || MODE == kL2Max) {
        uint64_t m = 0;
        for (int b = threadIdx.x; b < nb; b += NT) {
            const uint64_t v = __ldcg(reinterpret_cast<const unsigned long long*>(partials + b));
            m = v > m ? v : m;
        }
        m = block_max_bits<NT>(m, sh_u);
        return __longlong_as_double(static_cast<long long>(m));
    } else {
        double s = 0.0;
        for (int b = threadIdx.x; b < nb; b += NT)
            s += __longlong_as_double(static_cast<long long>(
                __ldcg(reinterpret_cast<const unsigned long long*>(partials + b))));
        return block_sum<NT>(s, sh_d);
    }
}

// The fp32 norm from the combined value: the max itself for (inf,inf), else the square root of
// a sum ((2,2), (inf,2)) or of a max of column sums ((2,inf)).
template <int MODE>
__device__ __forceinline__ float norm_from_combined(double v) {
    return static_cast<float>(MODE == kMaxMax ? v : sqrt(v));
}

// The block's partial, then, in the last of the nblk blocks of this norm to finish (completion
// ticket, no waiting), the fixed-order combine of the partials and the fp32 norm.
template <int MODE>
__device__ __forceinline__ void norm_finalize(uint32_t maxbits, const ScaledSumSq& ssq,
                                              int64_t best_key, uint32_t bad_col, int64_t vb,
                                              int64_t nblk, const NormSlots& out) {
    uint64_t* partials = out.partials;
    __shared__ double sh_d[kThreads / 32];
    __shared__ uint64_t sh_u[kThreads / 32];
    __shared__ bool is_last;

    const uint64_t part_bits = block_partial<MODE>(maxbits, ssq, best_key, bad_col, sh_d, sh_u);
    if (threadIdx.x == 0) {
        GQ_BOUND(vb >= 0 && vb < nblk && nblk <= kMaxPartials);
        partials[vb] = part_bits;
        __threadfence();
        const unsigned int t = atomicAdd(out.ticket, 1u);
        is_last = (t == nblk - 1);
    }
    __syncthreads();
    if (!is_last) return;
    __threadfence();

    // Last block: combine the nblk partials in a fixed order.
    const double result = combine_partials<MODE>(partials, static_cast<int>(nblk), sh_d, sh_u);
    if (threadIdx.x == 0) {
        if (out.part_user) *out.part_user = result;  // combinable across ranks: a sum or a max
        const float n32 = norm_from_combined<MODE>(result);
        *out.norm = n32;
        if (out.norm_user) *out.norm_user = n32;
        if (out.scale) *out.scale = dequant_scale(out.scheme, n32, out.n, out.s);
        if (!(fabsf(n32) < __uint_as_float(kInfBits))) atomicCAS(out.status, 0u, 4u);
        *out.ticket = 0;  // ready for the next call on this workspace
        __threadfence();
    }
}


// One norm computed by `nblk` blocks, this one being block `vb` of them.
template <typename T, int MODE>
__device__ __forceinline__ void norm_body(const T* __restrict__ x, int64_t n, int64_t d,
                                          int64_t groups, bool vec_rows, int64_t vb, int64_t nblk,
                                          const NormSlots& out) {
    constexpr int C = Elem<T>::kCols;
    const int64_t stride = nblk * kThreads;
    uint32_t maxbits = 0;       // kMaxMax: max |x| bit pattern
    ScaledSumSq ssq;            // kL2L2, kMaxL2
    ssq.init();
    int64_t best_key = INT64_MIN;  // kL2Max
    uint32_t bad_col = 0;          // kL2Max: a non-finite column norm was seen

    // rows in flight per thread: 8 raw 16-byte loads (widened when used); fewer for the
    // (2, inf) form, whose per-column scaled sums take C x 5 registers
    constexpr int U = (MODE == kL2Max) ? (C == 8 ? 2 : 4) : 8;
    const int64_t row_bytes = d * static_cast<int64_t>(sizeof(T));
    if constexpr (MODE == kL2Max) {
        // Plain fp32 column sums of squares (exact squares by FMA into NA interleaved
        // accumulators: relative error below (n/NA + 1) u <= 17 u, so below 1e-6 on the norm)
        // when n <= 16 NA; a column whose sum is not a normal number of at least 2^-100 (a NaN,
        // an overflow, or tiny values whose squares lose bits) is summed again with the scaled
        // form below.
        constexpr int NA = C == 8 ? 2 : 4;
        constexpr int UF = 8;  // rows in flight
        if (n <= 16 * NA) {
            for (int64_t g = vb * kThreads + threadIdx.x; g < groups; g += stride) {
                float acc[NA][C];
#pragma unroll
                for (int a = 0; a < NA; ++a)
#pragma unroll
                    for (int c = 0; c < C; ++c) acc[a][c] = 0.0f;
                const bool vec = vec_rows && (g + 1) * C <= d;
                for (int64_t i0 = 0; i0 < n; i0 += UF) {
                    uint4 raw[UF];
                    if (vec) {
#pragma unroll
                        for (int u = 0; u < UF; ++u)
                            raw[u] = (i0 + u < n) ? load_raw16(x, i0 + u, g, row_bytes)
                                                  : make_uint4(0u, 0u, 0u, 0u);
                    }
#pragma unroll
                    for (int u = 0; u < UF; ++u) {
                        float v[C];
                        if (vec) {
                            widen16<T>(raw[u], v);
                        } else if (i0 + u < n) {
                            load_group<T>(x, i0 + u, g, d, false, v);
                        } else {
#pragma unroll
                            for (int c = 0; c < C; ++c) v[c] = 0.0f;
                        }
#pragma unroll
                        for (int c = 0; c < C; ++c)
                            acc[u % NA][c] = __fmaf_rn(v[c], v[c], acc[u % NA][c]);
                    }
                }
#pragma unroll
                for (int c = 0; c < C; ++c) {
                    float sum = acc[0][c];
#pragma unroll
                    for (int a = 1; a < NA; ++a) sum = sum + acc[a][c];
                    if (sum >= 0x1p-100f && sum < __uint_as_float(kInfBits)) {
                        const int64_t key = scaled_key(sum, 0);
                        best_key = key > best_key ? key : best_key;
                        continue;
                    }
                    if (sum == 0.0f) continue;  // an all-zero column adds nothing
                    // rare: the scaled form for this column
                    ScaledSumSq cs;
                    cs.init();
                    for (int64_t i = 0; i < n; ++i) {
                        const int64_t j = g * C + c;
                        const float one[1] = {j < d ? Elem<T>::load_one(x + i * d + j) : 0.0f};
                        cs.add<1>(one);
                    }
                    const float ssum = cs.sum();
                    if (!(ssum < __uint_as_float(kInfBits))) {  // NaN or Inf column
                        const uint32_t b = __float_as_uint(ssum) & 0x7FFFFFFFu;
                        bad_col = b > bad_col ? b : bad_col;
                    } else if (ssum > 0.0f) {
                        const int64_t key = scaled_key(ssum, cs.e);
                        best_key = key > best_key ? key : best_key;
                    }
                }
            }
            norm_finalize<MODE>(maxbits, ssq, best_key, bad_col, vb, nblk, out);
            return;
        }
    }
    for (int64_t g = vb * kThreads + threadIdx.x; g < groups; g += stride) {
        uint32_t colmax[C];   // kMaxL2
        ScaledSumSq col[C];   // kL2Max
#pragma unroll
        for (int c = 0; c < C; ++c) { colmax[c] = 0; col[c].init(); }
        const bool vec = vec_rows && (g + 1) * C <= d;
        for (int64_t i0 = 0; i0 < n; i0 += U) {
            uint4 raw[U];
            if (vec) {
#pragma unroll
                for (int u = 0; u < U; ++u)
                    raw[u] = (i0 + u < n) ? load_raw16(x, i0 + u, g, row_bytes)
                                          : make_uint4(0u, 0u, 0u, 0u);  // zero rows add nothing
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                float v[C];
                if (vec) {
                    widen16<T>(raw[u], v);
                } else if (i0 + u < n) {
                    load_group<T>(x, i0 + u, g, d, false, v);
                } else {
#pragma unroll
                    for (int c = 0; c < C; ++c) v[c] = 0.0f;
                }
                if (MODE == kMaxMax) {
#pragma unroll
                    for (int c = 0; c < C; ++c) {
                        const uint32_t b = __float_as_uint(v[c]) & 0x7FFFFFFFu;
                        maxbits = b > maxbits ? b : maxbits;
                    }
                } else if (MODE == kL2L2) {
                    ssq.add<C>(v);
                } else if (MODE == kMaxL2) {
#pragma unroll
                    for (int c = 0; c < C; ++c) {
                        const uint32_t b = __float_as_uint(v[c]) & 0x7FFFFFFFu;
                        colmax[c] = b > colmax[c] ? b : colmax[c];
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < C; ++c) {
                        const float one[1] = {v[c]};
                        col[c].add<1>(one);
                    }
                }
            }
        }
        if (MODE == kMaxL2) {
            float m[C];
#pragma unroll
            for (int c = 0; c < C; ++c) m[c] = __uint_as_float(colmax[c]);
            ssq.add<C>(m);
        } else if (MODE == kL2Max) {
#pragma unroll
            for (int c = 0; c < C; ++c) {
                const float sum = col[c].sum();
                if (!(sum < __uint_as_float(kInfBits))) {  // NaN or Inf column
                    const uint32_t b = __float_as_uint(sum) & 0x7FFFFFFFu;
                    bad_col = b > bad_col ? b : bad_col;
                } else if (sum > 0.0f) {
                    const int64_t key = scaled_key(sum, col[c].e);
                    best_key = key > best_key ? key : best_key;
                }
            }
        }
    }

    norm_finalize<MODE>(maxbits, ssq, best_key, bad_col, vb, nblk, out);
}

// The mixed forms keep per-column state (more registers): two blocks per SM for (2, inf), three
// for (inf, 2), else four.
template <typename T, int MODE>
__global__ void __launch_bounds__(kThreads, MODE == kL2Max ? 2 : (MODE == kMaxL2 ? 3 : 4))
norm_kernel(const T* __restrict__ x, int64_t n, int64_t d, int64_t groups, bool vec_rows,
            float* __restrict__ norm_user, double* __restrict__ part_user,
            unsigned char* __restrict__ ws) {
    pdl_launch_dependents();
    WsHeader* hdr = reinterpret_cast<WsHeader*>(ws);
    const NormSlots slots{reinterpret_cast<uint64_t*>(ws + kHeaderBytes), &hdr->ticket,
                          &hdr->status, &hdr->norm, norm_user, part_user};
    norm_body<T, MODE>(x, n, d, groups, vec_rows, blockIdx.x, gridDim.x, slots);
}

// The (inf, inf) and (2, 2) norms do not depend on which coordinate an element belongs to: they
// are the max |x| and the sum of squares over all n d elements, read here as one flat array
// (sixteen 16-byte loads in flight per thread for (inf, inf), eight for (2, 2), whatever n is).
template <typename T, int MODE>
__global__ void __launch_bounds__(kThreads, 4)
norm_flat_kernel(const T* __restrict__ x, int64_t total, float* __restrict__ norm_user,
                 double* __restrict__ part_user, unsigned char* __restrict__ ws) {
    static_assert(MODE == kMaxMax || MODE == kL2L2, "flat norms: (inf, inf) and (2, 2)");
    constexpr int C = Elem<T>::kCols;
    constexpr int U = MODE == kMaxMax ? 16 : 8;  // 16-byte loads in flight per thread
    pdl_launch_dependents();
    WsHeader* hdr = reinterpret_cast<WsHeader*>(ws);
    const NormSlots slots{reinterpret_cast<uint64_t*>(ws + kHeaderBytes), &hdr->ticket,
                          &hdr->status, &hdr->norm, norm_user, part_user};
    const uint4* xv = reinterpret_cast<const uint4*>(x);
    const int64_t nvec = total / C;
    uint32_t maxbits = 0;
    ScaledSumSq ssq;
    ssq.init();
    const int64_t step = static_cast<int64_t>(gridDim.x) * kThreads * U;
    for (int64_t v0 = static_cast<int64_t>(blockIdx.x) * kThreads * U + threadIdx.x; v0 < nvec;
         v0 += step) {
        uint4 raw[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t v = v0 + static_cast<int64_t>(u) * kThreads;
            raw[u] = v < nvec ? __ldg(xv + v) : make_uint4(0u, 0u, 0u, 0u);  // zeros add nothing
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            float vals[C];
            widen16<T>(raw[u], vals);
            if (MODE == kMaxMax) {
#pragma unroll
                for (int c = 0; c < C; ++c) {
                    const uint32_t b = __float_as_uint(vals[c]) & 0x7FFFFFFFu;
                    maxbits = b > maxbits ? b : maxbits;
                }
            } else {
                ssq.add<C>(vals);
            }
        }
    }
    const int64_t tail = total - nvec * C;  // fewer than C elements past the last 16 bytes
    if (blockIdx.x == 0 && threadIdx.x < tail) {
        const float v[1] = {Elem<T>::load_one(x + nvec * C + threadIdx.x)};
        if (MODE == kMaxMax) {
            const uint32_t b = __float_as_uint(v[0]) & 0x7FFFFFFFu;
            maxbits = b > maxbits ? b : maxbits;
        } else {
            ssq.add<1>(v);
        }
    }
    norm_finalize<MODE>(maxbits, ssq, INT64_MIN, 0u, blockIdx.x, gridDim.x, slots);
}

// The norm from the combined partials of several ranks (a sum of squares for (2,2), a maximum
// magnitude for (inf,inf)), rounded to fp32 as norm_kernel rounds it.
static __global__ void norm_finish_kernel(const double* __restrict__ part, bool take_sqrt,
                                   float* __restrict__ norm) {
    if (threadIdx.x == 0 && blockIdx.x == 0) {
        const double v = *part;
        *norm = static_cast<float>(take_sqrt ? sqrt(v) : v);
    }
}

// ------------------------------------------------------------------------------------------
// Steps 2-4: stochastic rounding onto the level grid (Global-QSGD, Global-Q operator; grids of
// Global-L_s and Global-E_s), the integer sum over the workers and the dequantisation.
//
// Definitions (shared with the CPU oracle by specification only):
//   v = fp32(|x| / N) clamped to [0, 1] (NaN -> 0);
//   P(v) = position on the grid in level-index units: v s (L), or for E the level index of the
//          binade below v plus the fraction of the way to the next level;
//   T = floor(frac(P) 2^32); k = floor(P) + [r < T] = floor(P + rho), rho = (2^32 - 1 - r) / 2^32;
//   r = (half (j mod 8) of Philox(j/8, i, step)) << 16 | half (j mod 8) of Philox(2^31 + j/8, i,
//       step), key = seed.
//
// Fast path (per element, no division, no variable shift): an approximation P_c of P in 16.16
// fixed point, read off the bits of one fp32 result:
//   L: fp32(fp32(|x| RN(s/N)) + 128) has unit 2^-16 in [128, 256), so its bits minus those of 128
//      are P_c 2^16 (P <= s <= 127);
//   E: v_c = fp32(|x| RN(1/N)); for v_c >= 2^-(s-1) the bits of v_c shifted right by 7 are
//      (biased exponent, 16 fraction bits), i.e. (P_c + 127 - s) 2^16; below 2^-(s-1),
//      P = v 2^(s-1) is read off fp32(fp32(|x| 2^(s-1) RN(1/N)) + 128) as for L.
// |P_c 2^16 - P 2^16| < 2 in all cases (relative error below 3.0001 u of the products, u = 2^-24,
// times P <= 127, plus the 2^-16 rounding or truncation).  With H the high half of r,
// Y = P_c 2^16 + (0xFFFF - H) - 2 and the true P 2^16 + rho 2^16 in [Y, Y + 5), k = Y >> 16 is
// certain when (Y & 0xFFFF) <= 0xFFFB.  Otherwise (probability about 5/65536 per element) the
// eight elements of the row-group take the exact path: __fdiv_rn, integer grid position, and the
// second Philox call for the low half of r.  The fast path does not clamp v to 1 for Global-L: a
// level index above s (only when |x| exceeds the norm) sends the batch to the exact path too.
//
// The integer sum over the workers is accumulated in fp32: every partial sum is an integer of
// magnitude below 2^24 (the library rejects larger n s and n 2^(s-1)), so it is exact.
// ------------------------------------------------------------------------------------------

constexpr int kQCols = 8;  // coordinates per thread per row in the quantise kernels

// 64-bit right shift with the PTX rule that shift amounts above 64 give 0.
__device__ __forceinline__ uint64_t shr64(uint64_t v, uint32_t n) {
    uint64_t r;
    asm("shr.b64 %0, %1, %2;" : "=l"(r) : "l"(v), "r"(n));
    return r;
}

// Eight coordinates 8g..8g+7 of row i, widened to fp32; zero past column d.
template <typename T>
__device__ __forceinline__ void load8(const T* __restrict__ x, int64_t i, int64_t g, int64_t d,
                                      bool vec_rows, float (&v)[kQCols]) {
    const int64_t j0 = g * kQCols;
    const T* row = x + i * d + j0;
    if (vec_rows && j0 + kQCols <= d) {
        if (sizeof(T) == 4) {
            float a[4], b[4];
            Elem<float>::load_vec(reinterpret_cast<const float*>(row), a);
            Elem<float>::load_vec(reinterpret_cast<const float*>(row) + 4, b);
#pragma unroll
            for (int c = 0; c < 4; ++c) { v[c] = a[c]; v[c + 4] = b[c]; }
        } else {
            Elem<uint16_t>::load_vec(reinterpret_cast<const uint16_t*>(row), v);
        }
    } else {
#pragma unroll
        for (int c = 0; c < kQCols; ++c) v[c] = (j0 + c < d) ? Elem<T>::load_one(row + c) : 0.0f;
    }
}

// U = floor(P(v) 2^32) as (hi, lo) = (lower level index, T), for the bits vb of 0 <= v <= 1.
// Exact.  (A subnormal v is given the implicit bit; its U is below 1 either way, so 0.)
template <int SCHEME>
__device__ __forceinline__ void grid_position(uint32_t vb, uint32_t s, uint32_t& hi,
                                              uint32_t& lo) {
    const uint32_t eb = vb >> 23;  // biased exponent, 0..127
    const uint32_t mant = (vb & 0x7FFFFFu) | 0x800000u;  // v = mant 2^(eb - 150)
    if (SCHEME == kLinear) {
        // v s = (mant s) 2^(eb - 150): mant s < 2^31, so U = (mant s) 2^32 >> (150 - eb)
        const uint64_t w = shr64(static_cast<uint64_t>(mant * s) << 32, 150u - eb);
        hi = static_cast<uint32_t>(w >> 32);
        lo = static_cast<uint32_t>(w);
    } else if (eb + s >= 128u) {
        // v in [2^e, 2^(e+1)), e = eb - 127 >= -(s-1): level s + e, fraction = mantissa bits
        hi = eb + s - 127u;
        lo = vb << 9;
    } else {
        // v < 2^-(s-1): between level 0 and 2^-(s-1); U = v 2^(s-1) 2^32 = mant 2^(eb+s-119)
        hi = 0u;
        lo = static_cast<uint32_t>(shr64(static_cast<uint64_t>(mant) << 32, 151u - eb - s));
    }
}

// 16-bit half c of a Philox output (low half of word c/2 for even c).
__device__ __forceinline__ uint32_t half16(const uint32_t (&w)[4], int c) {
    return (c & 1) ? (w[c >> 1] >> 16) : (w[c >> 1] & 0xFFFFu);
}

struct QuantArgs {
    const float* norm_ptr;   // fp32 norm in device memory
    uint32_t s;
    uint32_t key0, key1;     // Philox key = seed
    uint32_t rk[20];         // Philox round keys of that key
    uint32_t step_lo, step_hi;
    int64_t n, d;
    int64_t pitch;           // code row pitch in elements
    bool vec_rows;
    uint32_t row0;           // worker index of local row 0 (keys the random words)
    void* sums;              // when set, the kernel writes the integer sums here instead of out
    int sums_i8;             // 1: the sums as int8 (they fit: |sum| <= 127), 0: as int32
    int out_dtype;           // kOutF32, kOutBF16 or kOutF16
    int compact;             // host hint: most elements round down (an l2 norm over coordinates):
                             // the compacting consumer
    int u16;                 // 1: the 16-bit-uniform rounding mode (decide H < F, no exact path)
    int pdl;                 // host: launch the quantise pass dependent on the norm pass
};

// Per-block fp32 dequantisation scale from the fp32 norm, computed in fp64 by one thread:
// N / (n s) for Global-L_s, N 2^-(s-1) / n for Global-E_s.  0 when the norm is 0 or non-finite.
template <int SCHEME>
__device__ __forceinline__ float block_scale(float nrm, int64_t n, uint32_t s, float* sh) {
    if (threadIdx.x == 0) *sh = dequant_scale(SCHEME, nrm, n, s);
    __syncthreads();
    return *sh;
}

// Store eight codes of one row (int8 bytes or int4 nibbles) for column group g.
template <int CODE_BITS>
__device__ __forceinline__ void store_codes(unsigned char* __restrict__ codes, int64_t i,
                                            int64_t g, int64_t pitch,
                                            const int32_t (&c)[kQCols]) {
    GQ_BOUND(i >= 0 && g >= 0 && (g + 1) * kQCols <= pitch);
    if (CODE_BITS == 8) {
        uint32_t w0 = 0, w1 = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            w0 |= (static_cast<uint32_t>(c[k]) & 0xFFu) << (8 * k);
            w1 |= (static_cast<uint32_t>(c[k + 4]) & 0xFFu) << (8 * k);
        }
        *reinterpret_cast<uint2*>(codes + i * pitch + g * kQCols) = make_uint2(w0, w1);
    } else {
        uint32_t w = 0;
#pragma unroll
        for (int k = 0; k < kQCols; ++k) w |= (static_cast<uint32_t>(c[k]) & 0xFu) << (4 * k);
        *reinterpret_cast<uint32_t*>(codes + i * (pitch / 2) + g * (kQCols / 2)) = w;
    }
}

// Per-kernel constants of the rounding decision.
// Exact mode: the addend c0 = 128 + 0xFFFD 2^-16 (so y = bits - H holds P_c + 0xFFFD - H), the
// decision is certain when y's low half is at most 0xFFFB.  16-bit-uniform mode: c0 = 128 +
// 0xFFFF 2^-16, so that y's high half is the level index plus [H < F]: every decision is final.
struct Decide {
    float nrm;        // N
    float rcp;        // RN(1 / N)
    float c1;         // L: RN(s / N); E: 2^(s-1) RN(1 / N)
    float c0;         // the addend that places P in 16.16 fixed point (see above)
    bool fast;        // 2^-100 <= N <= 2^100: the fast path's products stay normal and finite
    uint32_t bigmin;  // E: bits of 2^-(s-1)
    uint32_t cbig;    // E: ((s - 127) << 16) + bits of c0
    uint32_t bigpb;   // bits of c0 + 2^16 units: P_c >= 1 from here on
    uint32_t win;     // largest certain low half of y: 0xFFFB (exact), 0xFFFF (16-bit mode)
    uint32_t lsub;    // (bits of fp32(P_c + c0)) - lsub = the compacting test's bound on F
};

template <int SCHEME>
__device__ __forceinline__ Decide make_decide(float nrm, uint32_t s, int u16) {
    Decide dc;
    const uint32_t c0b = u16 ? 0x4300FFFFu : 0x4300FFFDu;
    dc.nrm = nrm;
    dc.rcp = __frcp_rn(nrm);
    dc.fast = nrm >= 0x1p-100f && nrm <= 0x1p100f;
    dc.c0 = __uint_as_float(c0b);
    dc.bigpb = c0b + 0x10000u;
    dc.win = u16 ? 0xFFFFu : 0xFFFBu;
    // exact mode: certain down when min H >= P_c + 3, i.e. bits - (c0 bits - 3) <= min H;
    // 16-bit mode: down when min H >= F = bits - c0 bits
    dc.lsub = u16 ? c0b : c0b - 3u;
    if (SCHEME == kLinear) {
        dc.c1 = __fdiv_rn(static_cast<float>(s), nrm);
        dc.bigmin = 0u;
        dc.cbig = 0u;
    } else {
        dc.c1 = dc.rcp * exp2i(static_cast<int>(s) - 1);
        dc.bigmin = (128u - s) << 23;
        dc.cbig = ((s - 127u) << 16) + c0b;
    }
    return dc;
}

// Level indices k of the eight elements of R row-groups (rows row0 .. row0+R-1), given the
// high-half Philox words aw of those rows, returned as y with k = y >> 16 (the low half is
// scratch).  The rare exact path runs for a row only if one of its elements needs it, and then
// only for those elements (one extra Philox call for the row).
template <int SCHEME, bool TRUSTED, int R>
__device__ __forceinline__ void decide_rows(const float (&xv)[R][kQCols], const Decide& dc,
                                            const QuantArgs& a, uint32_t g32, uint32_t row0,
                                            const uint32_t (&aw)[R][4],
                                            uint32_t (&yk)[R][kQCols]) {
    // y = bits(fp32(|x| c1) + c0) - H = 0x43000000 + P_c 2^16 + (0xFFFF - H) - 2: its low half
    // is that of Y = P_c 2^16 + (0xFFFF - H) - 2 and its high half k + 0x4300.  (c0 is a multiple
    // of the 2^-16 unit of [128, 256), so adding it inside the rounding moves the result by
    // exactly 0xFFFD units; P <= s <= 127 keeps the sum below 256.)
    constexpr uint32_t kOff = 0x4300u;
    // per-row, per-half maxima: the low half of worst[u] tracks the largest (Y & 0xFFFF) of
    // row u, the high half its largest level index Y >> 16
    uint32_t worst[R];
    bool anybig = false;
    uint32_t pbs[R][kQCols];
    // rows sent to the exact path whatever their estimates: all of them for a norm outside the
    // fast path's range, and rows holding a NaN (in both rounding modes)
    uint32_t force = dc.fast ? 0u : (1u << R) - 1u;
#pragma unroll
    for (int u = 0; u < R; ++u) {
        worst[u] = 0u;
#pragma unroll
        for (int c = 0; c < kQCols; ++c) {
            const float ax = fabsf(xv[u][c]);
            uint32_t pb;
            if (SCHEME == kLinear) {
                // no clamp to P <= s here: a level index above s (|x| above the norm) sends
                // the element to the exact path
                pb = __float_as_uint(__fmaf_rn(ax, dc.c1, dc.c0));
            } else {
                // below 2^-(s-1) (P < 1, the common case under l2 norms): P read as for L;
                // at or above it the binade form is computed for the row (see below)
                pb = __float_as_uint(__fmaf_rn(ax, dc.c1, dc.c0));
                anybig |= pb >= dc.bigpb;  // P_c >= 1
            }
            if (!TRUSTED && !(ax == ax)) force |= 1u << u;  // NaN: decided on the exact path
            pbs[u][c] = pb;
        }
    }
    if (SCHEME == kExp && anybig) {
        // v_c >= 2^-(s-1): (bits of v_c) >> 7 is (biased exponent, 16 fraction bits)
#pragma unroll
        for (int u = 0; u < R; ++u)
#pragma unroll
            for (int c = 0; c < kQCols; ++c) {
                const uint32_t vb = min(__float_as_uint(fabsf(xv[u][c]) * dc.rcp), 0x3F800000u);
                if (vb >= dc.bigmin) pbs[u][c] = (vb >> 7) + dc.cbig;
            }
    }
#pragma unroll
    for (int u = 0; u < R; ++u) {
#pragma unroll
        for (int c = 0; c < kQCols; ++c) {
            const uint32_t y = pbs[u][c] - half16(aw[u], c);
            yk[u][c] = y;
            worst[u] = __vmaxu2(worst[u], y);
        }
    }
    // exact path (the correctly rounded quotient and the full word) for an uncertain element,
    // a Global-L level index above s, a NaN, or every element when the norm is out of the fast
    // path's range; one test for all R rows first (almost always none needs it)
    uint32_t wall = worst[0];
#pragma unroll
    for (int u = 1; u < R; ++u) wall = __vmaxu2(wall, worst[u]);
    if (force == 0u && (wall & 0xFFFFu) <= dc.win &&
        !(SCHEME == kLinear && (wall >> 16) > a.s + kOff))
        return;
#pragma unroll
    for (int u = 0; u < R; ++u) {
        const bool over = SCHEME == kLinear && (worst[u] >> 16) > a.s + kOff;
        if ((worst[u] & 0xFFFFu) > dc.win || over || ((force >> u) & 1u)) {
            const uint4 rb = philox4x32_10_rk(
                make_uint4(g32 | 0x80000000u, row0 + u, a.step_lo, a.step_hi), a.rk);
            const uint32_t bw[4] = {rb.x, rb.y, rb.z, rb.w};
#pragma unroll
            for (int c = 0; c < kQCols; ++c) {
                const uint32_t y = yk[u][c];
                const bool need = !dc.fast || (y & 0xFFFFu) > dc.win ||
                                  (SCHEME == kLinear && (y >> 16) > a.s + kOff) ||
                                  (!TRUSTED && !(xv[u][c] == xv[u][c]));
                if (!need) continue;
                uint32_t vb = __float_as_uint(__fdiv_rn(fabsf(xv[u][c]), dc.nrm));
                vb = (vb > kInfBits) ? 0u : min(vb, 0x3F800000u);
                uint32_t hi, lo;
                grid_position<SCHEME>(vb, a.s, hi, lo);
                const uint32_t r = (half16(aw[u], c) << 16) | half16(bw, c);
                const uint32_t k = hi + (r < lo ? 1u : 0u);
                yk[u][c] = (k + kOff) << 16;
            }
        }
    }
}

// Packed fp32 pairs for the paired arithmetic of sm_100-class GPUs (add.f32x2, fma.f32x2: two
// IEEE operations, round to nearest even, in one instruction).
__device__ __forceinline__ unsigned long long pk2(float a, float b) {
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ void up2(unsigned long long r, float& a, float& b) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ unsigned long long add2(unsigned long long a, unsigned long long b) {
    unsigned long long d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ unsigned long long fma2(unsigned long long a, unsigned long long b,
                                                   unsigned long long c) {
    unsigned long long d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
// Paired add rounded toward zero (add.rz.f32x2).
__device__ __forceinline__ unsigned long long add2rz(unsigned long long a, unsigned long long b) {
    unsigned long long d;
    asm("add.rz.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
// Accumulate one row-group's codes (k = (yk >> 16) - 0x4300) into the sums (fp32, exact:
// integers below 2^24) and return the signed codes.  The level value is read off bit patterns:
// L: yk read as a float is 128 + k + f, f = (low half) 2^-16 < 1 (at most 0xFFFB on the exact
// mode's fast path, 0xFFFF in the 16-bit mode, 0 from the exact path), so adding 2^23 - 128
// with rounding toward zero gives exactly
// 2^23 + k (floating-point adds, off the integer pipe); E: the float with exponent field k + 126
// is 2^(k-1), and (v + 2^23) - 2^23 turns k = 0 (0.5) into 0 (the tie rounds to the even 2^23).
// The subtractions and the signed accumulation run on column pairs.
template <int SCHEME>
__device__ __forceinline__ void accumulate_row(const float (&xv)[kQCols],
                                               const uint32_t (&yk)[kQCols], float (&S)[kQCols],
                                               int32_t (&code)[kQCols]) {
#pragma unroll
    for (int c = 0; c < kQCols; c += 2) {
        float sg[2], raw[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint32_t xb = __float_as_uint(xv[c + h]);
            sg[h] = __uint_as_float((xb & 0x80000000u) | 0x3F800000u);
            if (SCHEME == kLinear)
                raw[h] = __uint_as_float(yk[c + h]);  // 128 + k + (low half) 2^-16
            else
                raw[h] = __uint_as_float(((yk[c + h] >> 16) << 23) + ((126u - 0x4300u) << 23));
            const int32_t k = static_cast<int32_t>(yk[c + h] >> 16) - 0x4300;
            const int32_t sgi = static_cast<int32_t>(xb) >> 31;
            code[c + h] = (k ^ sgi) - sgi;
        }
        unsigned long long units;
        if (SCHEME == kLinear) {
            // 128 + k + f (0 <= f < 1) plus 2^23 - 128, rounded toward zero, is 2^23 + k
            units = add2(add2rz(pk2(raw[0], raw[1]), pk2(8388480.0f, 8388480.0f)),
                         pk2(-8388608.0f, -8388608.0f));
        } else {
            units = add2(add2(pk2(raw[0], raw[1]), pk2(8388608.0f, 8388608.0f)),
                         pk2(-8388608.0f, -8388608.0f));
        }
        const unsigned long long s2 = fma2(pk2(sg[0], sg[1]), units, pk2(S[c], S[c + 1]));
        up2(s2, S[c], S[c + 1]);
    }
}

// Quantise column group g of all n rows with direct loads; accumulate the sums; optionally
// store codes.  Four rows are loaded at a time; each row is decided on its own.
template <typename T, int SCHEME, int CODE_BITS, bool TRUSTED>
__device__ __forceinline__ void quantize_group(const T* __restrict__ x, const QuantArgs& a,
                                               const Decide& dc, int64_t g,
                                               unsigned char* __restrict__ codes,
                                               float (&S)[kQCols]) {
    constexpr int U = 4;  // rows loaded per batch
#pragma unroll
    for (int c = 0; c < kQCols; ++c) S[c] = 0.0f;
    const uint32_t g32 = static_cast<uint32_t>(g);
    const PhiloxGroup pg = philox_group(g32, a.step_lo, a.step_hi, a.rk);
    for (int64_t i0 = 0; i0 < a.n; i0 += U) {
        float v[U][1][kQCols];
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (i0 + u < a.n) load8<T>(x, i0 + u, g, a.d, a.vec_rows, v[u][0]);
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (i0 + u >= a.n) break;
            const uint32_t row = static_cast<uint32_t>(i0 + u);
            const uint32_t worker = row + a.row0;
            const uint4 ra = philox_row(pg, worker, a.step_lo, a.rk);
            const uint32_t aw[1][4] = {{ra.x, ra.y, ra.z, ra.w}};
            uint32_t k[1][kQCols];
            decide_rows<SCHEME, TRUSTED, 1>(v[u], dc, a, g32, worker, aw, k);
            int32_t code[kQCols];
            accumulate_row<SCHEME>(v[u][0], k[0], S, code);
            if (CODE_BITS) store_codes<CODE_BITS>(codes, row, g, a.pitch, code);
        }
    }
}

// ------------------------------------------------------------------------------------------
// Asynchronous staging of the gradient rows.  Each thread copies its own 16-byte pieces of the
// next rows into its own shared-memory slots (cp.async, L1 bypassed) and reads them back when
// they are needed, so loads stay in flight without holding registers.  A thread only ever
// reads what it copied itself, so the only synchronisation is cp.async.wait_group (a hardware
// wait on the thread's own copies).
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
    const uint32_t sa = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sa), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <typename T>
struct Staging {
    // Measured on the quantise pass: staging pays for bf16 (twice the elements per byte, so a
    // thread spends longer per loaded byte) and not for fp32, where the direct loads of two
    // rows per batch already keep enough bytes in flight.
    static constexpr bool kEnabled = sizeof(T) == 2;
    static constexpr int kPieces = sizeof(T) == 4 ? 2 : 1;  // 16-byte pieces per row-group
    static constexpr int kRows = 2;                         // rows per batch
    static constexpr int kStages = 4;                       // batches in the ring
    static constexpr int kBytes = kEnabled ? kStages * kRows * kPieces * kThreads * 16 : 0;
};

// Widen one staged row-group (kPieces x 16 bytes) to eight fp32 values.
template <typename T>
__device__ __forceinline__ void unstage(const uint4* piece0, const uint4* piece1,
                                        float (&v)[kQCols]) {
    if (sizeof(T) == 4) {
        const uint4 p = *piece0, q = *piece1;
        v[0] = __uint_as_float(p.x); v[1] = __uint_as_float(p.y);
        v[2] = __uint_as_float(p.z); v[3] = __uint_as_float(p.w);
        v[4] = __uint_as_float(q.x); v[5] = __uint_as_float(q.y);
        v[6] = __uint_as_float(q.z); v[7] = __uint_as_float(q.w);
    } else {
        const uint4 p = *piece0;
        const uint32_t w[4] = {p.x, p.y, p.z, p.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            v[2 * k] = __uint_as_float(w[k] << 16);
            v[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
        }
    }
}

// Round-to-nearest-even conversions of the fp32 outputs to the 16-bit output types.
__device__ __forceinline__ uint32_t pack16(int dt, float lo, float hi) {
    if (dt == kOutBF16) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<const uint32_t*>(&h);
    }
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ void store1(void* out, int dt, int64_t j, float v) {
    if (dt == kOutF32) {
        static_cast<float*>(out)[j] = v;
    } else if (dt == kOutBF16) {
        static_cast<__nv_bfloat16*>(out)[j] = __float2bfloat16_rn(v);
    } else {
        static_cast<__half*>(out)[j] = __float2half_rn(v);
    }
}

// Output of one finished column group: dequantise the sums into out (fp32, bf16 or fp16), or,
// when `sums` is set, write the integer sums themselves as int32 or int8 (exact: every partial
// sum is an integer below 2^24, and below 128 in magnitude when int8 is asked for).
__device__ __forceinline__ void store_out(void* __restrict__ out, void* __restrict__ sums,
                                          int sums_i8, int dt, int64_t g, int64_t d, float scale,
                                          const float (&S)[kQCols]) {
    const int64_t j0 = g * kQCols;
    // callers pass every group of the code pitch (padding groups past d store nothing)
    GQ_BOUND(g >= 0 && j0 < (d + 31) / 32 * 32);
    if (sums) {
        if (sums_i8) {
            int8_t* q = static_cast<int8_t*>(sums);
            if (j0 + kQCols <= d) {
                uint32_t w[2] = {0u, 0u};
#pragma unroll
                for (int c = 0; c < kQCols; ++c)
                    w[c >> 2] |= (static_cast<uint32_t>(static_cast<int32_t>(S[c])) & 0xFFu)
                                 << (8 * (c & 3));
                *reinterpret_cast<uint2*>(q + j0) = make_uint2(w[0], w[1]);
            } else {
#pragma unroll
                for (int c = 0; c < kQCols; ++c)
                    if (j0 + c < d) q[j0 + c] = static_cast<int8_t>(static_cast<int32_t>(S[c]));
            }
            return;
        }
        int32_t* q = static_cast<int32_t*>(sums);
        if (j0 + kQCols <= d) {
#pragma unroll
            for (int h = 0; h < kQCols / 4; ++h)
                reinterpret_cast<int4*>(q + j0)[h] =
                    make_int4(static_cast<int32_t>(S[4 * h]), static_cast<int32_t>(S[4 * h + 1]),
                              static_cast<int32_t>(S[4 * h + 2]), static_cast<int32_t>(S[4 * h + 3]));
        } else {
#pragma unroll
            for (int c = 0; c < kQCols; ++c)
                if (j0 + c < d) q[j0 + c] = static_cast<int32_t>(S[c]);
        }
        return;
    }
    if (j0 + kQCols <= d) {
        if (dt == kOutF32) {
            float* o = static_cast<float*>(out);
#pragma unroll
            for (int h = 0; h < kQCols / 4; ++h)
                reinterpret_cast<float4*>(o + j0)[h] =
                    make_float4(scale * S[4 * h], scale * S[4 * h + 1], scale * S[4 * h + 2],
                                scale * S[4 * h + 3]);
        } else {  // eight 16-bit values: one 16-byte store
            *reinterpret_cast<uint4*>(static_cast<uint16_t*>(out) + j0) =
                make_uint4(pack16(dt, scale * S[0], scale * S[1]), pack16(dt, scale * S[2], scale * S[3]),
                           pack16(dt, scale * S[4], scale * S[5]), pack16(dt, scale * S[6], scale * S[7]));
        }
    } else {
#pragma unroll
        for (int c = 0; c < kQCols; ++c)
            if (j0 + c < d) store1(out, dt, j0 + c, scale * S[c]);
    }
}

// The column groups 0 .. full-1 (every row of them vector-aligned and inside d), visited from
// the last to the first in grid-stride order, with the rows staged through shared memory.
template <typename T, int SCHEME, int CODE_BITS, bool WRITE_OUT, bool TRUSTED>
__device__ __forceinline__ void staged_groups(const T* __restrict__ x, const QuantArgs& a,
                                              const Decide& dc, int64_t full, float scale,
                                              unsigned char* __restrict__ codes,
                                              void* __restrict__ out, uint4* stage, int64_t vb,
                                              int64_t nblk) {
    using St = Staging<T>;
    constexpr int R = St::kRows, P = St::kPieces, NS = St::kStages;
    const int64_t stride = nblk * kThreads;
    const int64_t it0 = vb * kThreads + threadIdx.x;
    const int64_t ngroups = it0 < full ? (full - 1 - it0) / stride + 1 : 0;
    const int64_t nb = (a.n + R - 1) / R;  // batches per group
    const int64_t total = ngroups * nb;
    auto slot = [&](int st, int u, int p) -> uint4* {
        return stage + ((st * R + u) * P + p) * kThreads + threadIdx.x;
    };
    // issue cursor: batch ib = (group iq, batch ir)
    int64_t ib = 0, iq = 0, ir = 0;
    auto issue = [&]() {
        if (ib < total) {
            const int64_t g = full - 1 - (it0 + iq * stride);
            const int st = static_cast<int>(ib % NS);
#pragma unroll
            for (int u = 0; u < R; ++u) {
                const int64_t row = ir * R + u;
                if (row < a.n) {
                    const T* src = x + row * a.d + g * kQCols;
#pragma unroll
                    for (int p = 0; p < P; ++p) cp_async16(slot(st, u, p), src + p * (16 / sizeof(T)));
                }
            }
            if (++ir == nb) { ir = 0; ++iq; }
        }
        ++ib;
        cp_async_commit();
    };
#pragma unroll
    for (int k = 0; k < NS - 1; ++k) issue();
    float S[kQCols];
    int64_t q = 0, r = 0;
    for (int64_t b = 0; b < total; ++b) {
        issue();
        cp_async_wait<NS - 1>();
        const int st = static_cast<int>(b % NS);
        const int64_t g = full - 1 - (it0 + q * stride);
        const uint32_t g32 = static_cast<uint32_t>(g);
        if (r == 0) {
#pragma unroll
            for (int c = 0; c < kQCols; ++c) S[c] = 0.0f;
        }
        float v[R][kQCols];
#pragma unroll
        for (int u = 0; u < R; ++u) {
            if (r * R + u < a.n) {
                unstage<T>(slot(st, u, 0), slot(st, u, P - 1), v[u]);
            } else {
#pragma unroll
                for (int c = 0; c < kQCols; ++c) v[u][c] = 0.0f;
            }
        }
        uint32_t aw[R][4];
        {
            const PhiloxGroup pg = philox_group(g32, a.step_lo, a.step_hi, a.rk);
#pragma unroll
            for (int u = 0; u < R; ++u) {
                const uint4 ra = philox_row(pg, static_cast<uint32_t>(r * R + u) + a.row0,
                                            a.step_lo, a.rk);
                aw[u][0] = ra.x; aw[u][1] = ra.y; aw[u][2] = ra.z; aw[u][3] = ra.w;
            }
        }
        uint32_t k[R][kQCols];
        decide_rows<SCHEME, TRUSTED, R>(v, dc, a, g32, static_cast<uint32_t>(r * R) + a.row0, aw,
                                        k);
#pragma unroll
        for (int u = 0; u < R; ++u) {
            const int64_t row64 = r * R + u;
            if (row64 >= a.n) break;
            int32_t code[kQCols];
            accumulate_row<SCHEME>(v[u], k[u], S, code);
            if (CODE_BITS) store_codes<CODE_BITS>(codes, row64, g, a.pitch, code);
        }
        if (++r == nb) {
            r = 0;
            ++q;
            if (WRITE_OUT) store_out(out, a.sums, a.sums_i8, a.out_dtype, g, a.d, scale, S);
        }
    }
    cp_async_wait<0>();
}

// Quantise (+ sum + dequantise).  CODE_BITS: 0 (no codes), 4 or 8.  WRITE_OUT: dequantise the
// sums into out.  TRUSTED: the norm was computed from these gradients by norm_kernel, so a
// finite norm means no element is NaN or infinite.  Groups of 8 columns run over ceil(d/8), or
// pitch/8 when codes are written (padding columns get zero codes), from the last group to the
// first: the fused path's norm pass ends on the last columns, which are still in L2.
template <typename T, int SCHEME, int CODE_BITS, bool WRITE_OUT, bool TRUSTED>
__device__ __forceinline__ void quantize_body(const T* __restrict__ x, const QuantArgs& a,
                                              int64_t groups, unsigned char* __restrict__ codes,
                                              void* __restrict__ out, uint4* stage, int64_t vb,
                                              int64_t nblk) {
    __shared__ float sh_scale;
    const float nrm = __ldg(a.norm_ptr);
    const float scale = block_scale<SCHEME>(nrm, a.n, a.s, &sh_scale);
    const bool live = nrm > 0.0f && nrm < __uint_as_float(kInfBits);
    const Decide dc = make_decide<SCHEME>(nrm, a.s, a.u16);
    // groups [0, full) are staged through shared memory; the rest (the ragged last group, code
    // padding, or everything when rows are not 16-byte aligned) use direct loads
    int64_t full = 0;
    if constexpr (Staging<T>::kEnabled) {
        full = (live && a.vec_rows) ? a.d / kQCols : 0;
        if (full > 0)
            staged_groups<T, SCHEME, CODE_BITS, WRITE_OUT, TRUSTED>(x, a, dc, full, scale, codes,
                                                                    out, stage, vb, nblk);
    }
    const int64_t stride = nblk * kThreads;
    const int64_t rest = groups - full;
    for (int64_t it = vb * kThreads + threadIdx.x; it < rest; it += stride) {
        const int64_t g = groups - 1 - it;
        float S[kQCols];
        if (live) {
            quantize_group<T, SCHEME, CODE_BITS, TRUSTED>(x, a, dc, g, codes, S);
        } else {
#pragma unroll
            for (int c = 0; c < kQCols; ++c) S[c] = 0.0f;
            if (CODE_BITS) {
                const int32_t zero[kQCols] = {0, 0, 0, 0, 0, 0, 0, 0};
                for (int64_t i = 0; i < a.n; ++i) store_codes<CODE_BITS>(codes, i, g, a.pitch, zero);
            }
        }
        if (WRITE_OUT) store_out(out, a.sums, a.sums_i8, a.out_dtype, g, a.d, scale, S);
    }
}

template <typename T, int SCHEME, int CODE_BITS, bool WRITE_OUT, bool TRUSTED>
__global__ void __launch_bounds__(kThreads, 2)
quantize_kernel(const T* __restrict__ x, QuantArgs a, int64_t groups,
                unsigned char* __restrict__ codes, void* __restrict__ out) {
    extern __shared__ uint4 stage[];
    pdl_wait();  // the norm of the fused call's first pass
    quantize_body<T, SCHEME, CODE_BITS, WRITE_OUT, TRUSTED>(x, a, groups, codes, out, stage,
                                                            blockIdx.x, gridDim.x);
}

// ------------------------------------------------------------------------------------------
// Segmented form: many independent problems (layers or gradient buckets), each its own n x d_l
// matrix with its own norm, in two launches for up to kSegChunk of them.  Every segment gets a
// run of consecutive blocks sized to its share of the elements; a block finds its segment by
// binary search over the run starts and then runs the same body as the single-problem kernels
// on a virtual grid of its segment's blocks.
// ------------------------------------------------------------------------------------------
struct SegDesc {
    const void* x;   // the segment's n x d rows
    void* out;       // its d outputs
    int64_t d;
    int32_t b0;      // first block of its run
    int32_t nb;      // blocks in its run
    int64_t t0;      // bulk-copy pass: index of its first direct-load group among the launch's
};
struct SegLaunch {
    SegDesc seg[kSegChunk];
    int32_t nseg;
    int32_t seg0;    // index of seg[0] among all segments of the call
    int64_t ntail;   // bulk-copy pass: groups outside the chunks, all segments
};

__device__ __forceinline__ int find_segment(const SegLaunch& L, int32_t b) {
    int lo = 0, hi = L.nseg - 1;  // the last segment whose run starts at or before b
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (L.seg[mid].b0 <= b) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// The segment of direct-load group `t` (numbered across the launch): the last whose first such
// group is at or before t.
__device__ __forceinline__ int find_tail_segment(const SegLaunch& L, int64_t t) {
    int lo = 0, hi = L.nseg - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (L.seg[mid].t0 <= t) lo = mid; else hi = mid - 1;
    }
    return lo;
}

template <typename T, int MODE>
__global__ void __launch_bounds__(kThreads, MODE == kL2Max ? 2 : (MODE == kMaxL2 ? 3 : 4))
norm_segments_kernel(const __grid_constant__ SegLaunch L, int64_t n, int scheme, uint32_t s,
                     float* __restrict__ norms_user, unsigned char* __restrict__ ws) {
    constexpr int C = Elem<T>::kCols;
    const int k = find_segment(L, static_cast<int32_t>(blockIdx.x));
    const SegDesc& sd = L.seg[k];
    WsHeader* hdr = reinterpret_cast<WsHeader*>(ws);
    uint64_t* partials = reinterpret_cast<uint64_t*>(ws + kHeaderBytes);
    NormSlots slots{partials + sd.b0,
                    reinterpret_cast<unsigned int*>(ws + kSegTicketsOff) + k, &hdr->status,
                    reinterpret_cast<float*>(ws + kSegNormsOff) + k,
                    norms_user ? norms_user + L.seg0 + k : nullptr, nullptr};
    slots.scale = reinterpret_cast<float*>(ws + kSegScalesOff) + k;
    slots.scheme = scheme;
    slots.s = s;
    slots.n = n;
    norm_body<T, MODE>(static_cast<const T*>(sd.x), n, sd.d, (sd.d + C - 1) / C, sd.d % C == 0,
                       static_cast<int64_t>(blockIdx.x) - sd.b0, sd.nb, slots);
}

// `base` holds the arguments common to every segment, with step_lo the call's step shifted left
// by 16 bits: segment l draws its random words with step (step << 16) | l.
template <typename T, int SCHEME>
__global__ void __launch_bounds__(kThreads, 2)
quantize_segments_kernel(const __grid_constant__ SegLaunch L, QuantArgs base,
                         unsigned char* __restrict__ ws) {
    extern __shared__ uint4 stage[];
    const int k = find_segment(L, static_cast<int32_t>(blockIdx.x));
    const SegDesc& sd = L.seg[k];
    QuantArgs a = base;
    a.norm_ptr = reinterpret_cast<const float*>(ws + kSegNormsOff) + k;
    a.d = sd.d;
    a.pitch = (sd.d + 31) / 32 * 32;
    a.vec_rows = sd.d % (16 / sizeof(T)) == 0;
    a.step_lo = base.step_lo | static_cast<uint32_t>(L.seg0 + k);
    quantize_body<T, SCHEME, 0, true, true>(static_cast<const T*>(sd.x), a,
                                            (sd.d + kQCols - 1) / kQCols, nullptr, sd.out, stage,
                                            static_cast<int64_t>(blockIdx.x) - sd.b0, sd.nb);
}

// ------------------------------------------------------------------------------------------
// Quantise pass fed by the bulk-copy engine.  One block per SM: 15 consumer warps, each thread
// owning one 8-column group of a 3840-column chunk, and a producer warp whose lane 0 keeps a
// ring of shared-memory stages (kRows rows x 3840 columns each) in flight with
// cp.async.bulk, completion counted on an mbarrier per stage.  The loads in flight no longer
// depend on the consumers' registers.  Same arithmetic, random words and outputs as
// quantize_kernel.  Every wait is bounded (about one second of global time): a wait that gives
// up records GQ_ERR_TIMEOUT (5) in the status word, stops the block's work, and the producer
// waits (bounded) for its own copies in flight before the block exits.
// ------------------------------------------------------------------------------------------
constexpr int kTmaWarps = 15;                       // consumer warps (16 warps in all)
constexpr int kTmaConsumers = kTmaWarps * 32;       // 480
constexpr int kTmaBlock = kTmaConsumers + 32;       // + the producer warp
constexpr int kTmaCols = kTmaConsumers * kQCols;    // 3840 columns per chunk
constexpr uint64_t kWaitLimitNs = 1000000000ull;    // one second
constexpr unsigned int kStatusTimeout = 5u;

template <typename T>
struct TmaCfg {
    static constexpr int kRows = 4;                           // rows per stage
    static constexpr int kStages = sizeof(T) == 4 ? 3 : 6;    // stages in the ring
    static constexpr int kRowBytes = kTmaCols * static_cast<int>(sizeof(T));
    static constexpr int kStageBytes = kRows * kRowBytes;     // 60 KB (fp32), 30 KB (bf16)
    static constexpr int kSmemBytes = kStages * kStageBytes;  // 180 KB
};

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}
// Wait for the completion of the phase with parity `parity`; false after limit_ns.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                          uint64_t limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (;;) {
#pragma unroll 1
        for (int k = 0; k < 64; ++k)
            if (mbar_try_wait(bar, parity)) return true;
        if (global_ns() - t0 > limit_ns) return false;
    }
}

// Self-test of the bounded wait: one thread waits on an mbarrier that nothing arrives on, gives
// up after limit_ns and records GQ_ERR_TIMEOUT in the status word, as the quantise kernels do;
// *elapsed_ns receives the time it waited.
static __global__ void wait_timeout_kernel(unsigned int* __restrict__ status, uint64_t limit_ns,
                                           unsigned long long* __restrict__ elapsed_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0) return;
    mbar_init(smem_u32(&bar), 1u);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    const uint64_t t0 = global_ns();
    const bool done = mbar_wait(smem_u32(&bar), 0u, limit_ns);
    *elapsed_ns = global_ns() - t0;
    if (!done) atomicCAS(status, 0u, kStatusTimeout);
}
// Bulk copy of `bytes` (a multiple of 16, both addresses 16-byte aligned) into shared memory,
// counted on the mbarrier `bar`.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// SUB: rows decided together (2; 1 for a single worker, whose stages hold one row).
// One stage of RB rows (rows b*RB ..) of one chunk, for consumer thread tid (group g of its
// problem): rows into registers SUB at a time, the stage released once its last rows are read,
// then random words, decisions and sums.  a: the problem's arguments (d, n, step, row0, s, rk).
// ZSKIP: while `probe` is set (from the start of a chunk, warp-uniform), every row pair is first
// tested for being +-0 across the warp and skipped if so; the first pair with a non-zero element
// clears `probe` for the rest of the chunk (zero blocks of sparse layers span whole columns, so a
// chunk is either zero in every row or dense).
template <typename T, int SCHEME, int CODE_BITS, bool TRUSTED, int SUB, bool ZSKIP = false>
__device__ __forceinline__ void tma_consume_stage(const unsigned char* stage, int lane, bool active,
                                                  int64_t b, int64_t g, const PhiloxGroup& pg,
                                                  const QuantArgs& a, const Decide& dc,
                                                  uint32_t empty_bar, float (&S)[kQCols],
                                                  unsigned char* __restrict__ codes,
                                                  bool* probe = nullptr) {
    using Cfg = TmaCfg<T>;
    constexpr int RB = Cfg::kRows;
    const uint32_t g32 = static_cast<uint32_t>(g);
#pragma unroll
    for (int u0 = 0; u0 < RB; u0 += SUB) {
        const int64_t r0 = b * RB + u0;
        float v[SUB][kQCols];
#pragma unroll
        for (int u = 0; u < SUB; ++u) {
            const uint4* p = reinterpret_cast<const uint4*>(stage + (u0 + u) * Cfg::kRowBytes);
            if (active && r0 + u < a.n) {
                unstage<T>(p, p + 1, v[u]);
            } else {
#pragma unroll
                for (int c = 0; c < kQCols; ++c) v[u][c] = 0.0f;
            }
        }
        if (u0 + SUB >= RB) {  // every row of the stage is in registers: release it
            __syncwarp();
            if (lane == 0) mbar_arrive(empty_bar);
        }
        if (ZSKIP && *probe) {
            // a zero element has code 0 whatever its random word: rows that are +-0 for every
            // lane of the warp need no random words or decisions
            uint32_t o = 0u;
            if (active && r0 < a.n) {
#pragma unroll
                for (int u = 0; u < SUB; ++u)
#pragma unroll
                    for (int c = 0; c < kQCols; ++c) o |= __float_as_uint(v[u][c]);
            }
            if (!__any_sync(0xFFFFFFFFu, (o & 0x7FFFFFFFu) != 0u)) {
                if (CODE_BITS && active) {
                    const int32_t zero[kQCols] = {0, 0, 0, 0, 0, 0, 0, 0};
#pragma unroll
                    for (int u = 0; u < SUB; ++u)
                        if (r0 + u < a.n) store_codes<CODE_BITS>(codes, r0 + u, g, a.pitch, zero);
                }
                continue;
            }
            *probe = false;
        }
        if (!active || r0 >= a.n) continue;  // past the last worker: nothing to do
        uint32_t aw[SUB][4];
#pragma unroll
        for (int u = 0; u < SUB; ++u) {
            const uint4 ra = philox_row(pg, static_cast<uint32_t>(r0 + u) + a.row0, a.step_lo,
                                        a.rk);
            aw[u][0] = ra.x; aw[u][1] = ra.y; aw[u][2] = ra.z; aw[u][3] = ra.w;
        }
        uint32_t yk[SUB][kQCols];
        decide_rows<SCHEME, TRUSTED, SUB>(v, dc, a, g32, static_cast<uint32_t>(r0) + a.row0, aw, yk);
#pragma unroll
        for (int u = 0; u < SUB; ++u) {
            if (r0 + u >= a.n) break;
            int32_t code[kQCols];
            accumulate_row<SCHEME>(v[u], yk[u], S, code);
            if (CODE_BITS) store_codes<CODE_BITS>(codes, r0 + u, g, a.pitch, code);
        }
    }
}

// ---- deferred decisions (the compacting consumer) -------------------------------------------
// Under an l2 norm of many elements most |x| / N are far below the first level, and most
// row-groups (eight elements of one row) round every element down: when the smallest high half
// H of their eight random words is at least the fast estimate P_c of the largest element's grid
// position plus 3 units of 2^-16 (P_c is within 2 units of the exact position, so every T < r),
// all eight codes are 0 and nothing is added.  That check costs one Philox call and a dozen
// instructions per row-group.  The row-groups that fail it are queued per warp in shared memory
// (raw values, random words, group and worker) and decided 32 at a time, one per lane, with the
// full decision; their code values go into per-warp integer sums in shared memory (exact:
// integers below 2^24), which each group's owner lane reads when its chunk's sums are complete.
// So the rare full decisions run on full warps instead of one lane at a time.  With two sum
// buffers (bf16, whose ring is small enough to leave room for them) a chunk's queue is not
// decided at its end: the next chunk adds to the other buffer, and one flush completes both, so
// flushes run on fuller queues and less often.  A queued item carries its buffer in bit 31 of
// its group index (group indices stay below 2^31).
constexpr int kQueue = 32;  // queued row-groups per warp

template <typename T>
struct CompactCfg {
    static constexpr int kXVec = sizeof(T) == 4 ? 2 : 1;  // 16-byte pieces of a row-group
    static constexpr int kSumBufs = sizeof(T) == 2 ? 2 : 1;
    static constexpr int kStages = sizeof(T) == 2 ? 5 : TmaCfg<T>::kStages;  // ring stages
    // per warp: raw values, random words, (group, worker), then the 8 x 32 integer sums per
    // buffer
    static constexpr int kWarpBytes = kQueue * (16 * kXVec + 16 + 8) + kSumBufs * kQCols * 32 * 4;
    static constexpr int kBytes = kTmaWarps * kWarpBytes;
    static constexpr int kSmemBytes = kStages * TmaCfg<T>::kStageBytes + kBytes;  // ring + queues
};

template <typename T>
struct WarpQueue {
    uint4* qx;     // [kQueue][kXVec]
    uint4* qw;     // [kQueue]
    uint2* qm;     // [kQueue]: group (bit 31: sum buffer), worker
    int32_t* sum;  // [kSumBufs][2][32][4]: column c of the group owned by lane l at
                   // (c / 4) * 128 + l * 4 + c % 4 (a lane's four columns in 16 bytes)
};

template <typename T>
__device__ __forceinline__ WarpQueue<T> warp_queue(unsigned char* base, int warp) {
    using C = CompactCfg<T>;
    unsigned char* p = base + warp * C::kWarpBytes;
    WarpQueue<T> q;
    q.qx = reinterpret_cast<uint4*>(p);
    q.qw = reinterpret_cast<uint4*>(p + kQueue * 16 * C::kXVec);
    q.qm = reinterpret_cast<uint2*>(p + kQueue * (16 * C::kXVec + 16));
    q.sum = reinterpret_cast<int32_t*>(p + kQueue * (16 * C::kXVec + 16 + 8));
    return q;
}

// Largest magnitude of a row-group as an fp32 value (NaN stays NaN: integer maximum of the
// magnitude bits; a trusted norm rules NaN out, so fp32 maxima of |x| are used there).
template <typename T, bool TRUSTED>
__device__ __forceinline__ float group_max_abs(const uint4 (&raw)[CompactCfg<T>::kXVec]) {
    if (sizeof(T) == 2 && TRUSTED) {
        // bf16 pairs: max.xorsign.abs gives max(|a|, |b|) per half (its sign bit, the xor of
        // the operands' signs, is dropped by the final fabsf)
        const uint4 r = raw[0];
        uint32_t m1, m2, m;
        asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(m1) : "r"(r.x), "r"(r.y));
        asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(m2) : "r"(r.z), "r"(r.w));
        asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(m) : "r"(m1), "r"(m2));
        return fmaxf(fabsf(__uint_as_float(m << 16)), fabsf(__uint_as_float(m & 0xFFFF0000u)));
    } else if (sizeof(T) == 2) {
        const uint4 r = raw[0];
        const uint32_t m = __vmaxu2(__vmaxu2(r.x & 0x7FFF7FFFu, r.y & 0x7FFF7FFFu),
                                    __vmaxu2(r.z & 0x7FFF7FFFu, r.w & 0x7FFF7FFFu));
        return __uint_as_float(max(m & 0xFFFFu, m >> 16) << 16);
    } else if (TRUSTED) {
        float m = 0.0f;
#pragma unroll
        for (int h = 0; h < CompactCfg<T>::kXVec; ++h) {
            const uint4 r = raw[h];
            m = fmaxf(m, fmaxf(fmaxf(fabsf(__uint_as_float(r.x)), fabsf(__uint_as_float(r.y))),
                               fmaxf(fabsf(__uint_as_float(r.z)), fabsf(__uint_as_float(r.w)))));
        }
        return m;
    } else {
        uint32_t m = 0u;
#pragma unroll
        for (int h = 0; h < CompactCfg<T>::kXVec; ++h) {
            const uint4 r = raw[h];
            m = max(m, max(max(r.x & 0x7FFFFFFFu, r.y & 0x7FFFFFFFu),
                           max(r.z & 0x7FFFFFFFu, r.w & 0x7FFFFFFFu)));
        }
        return __uint_as_float(m);
    }
}

template <typename T>
__device__ __forceinline__ void widen_raw(const uint4 (&raw)[CompactCfg<T>::kXVec],
                                          float (&v)[kQCols]) {
    if (sizeof(T) == 2) {
        const uint32_t w[4] = {raw[0].x, raw[0].y, raw[0].z, raw[0].w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            v[2 * k] = __uint_as_float(w[k] << 16);
            v[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
        }
    } else {
        const uint32_t w[8] = {raw[0].x, raw[0].y, raw[0].z, raw[0].w,
                               raw[CompactCfg<T>::kXVec - 1].x, raw[CompactCfg<T>::kXVec - 1].y,
                               raw[CompactCfg<T>::kXVec - 1].z, raw[CompactCfg<T>::kXVec - 1].w};
#pragma unroll
        for (int c = 0; c < kQCols; ++c) v[c] = __uint_as_float(w[c]);
    }
}

// Decide the first `cnt` queued row-groups, one per lane, and add their code values (Global-L:
// the signed level index; Global-E: sign 2^(k-1), 0 for k = 0) to their owners' sums.
template <typename T, int SCHEME, bool TRUSTED>
__device__ __forceinline__ void flush_queue(const WarpQueue<T>& q, int cnt, int lane,
                                            const QuantArgs& a, const Decide& dc) {
    __syncwarp();
    if (lane < cnt) {
        uint4 raw[CompactCfg<T>::kXVec];
#pragma unroll
        for (int h = 0; h < CompactCfg<T>::kXVec; ++h) raw[h] = q.qx[lane * CompactCfg<T>::kXVec + h];
        const uint4 w = q.qw[lane];
        const uint2 m = q.qm[lane];
        float v[1][kQCols];
        widen_raw<T>(raw, v[0]);
        const uint32_t aw[1][4] = {{w.x, w.y, w.z, w.w}};
        uint32_t yk[1][kQCols];
        decide_rows<SCHEME, TRUSTED, 1>(v, dc, a, m.x & 0x7FFFFFFFu, m.y, aw, yk);
        int32_t* sum = q.sum + (m.x >> 31) * (kQCols * 32) + (m.x & 31u) * 4;
#pragma unroll
        for (int c = 0; c < kQCols; ++c) {
            const int32_t k = static_cast<int32_t>(yk[0][c] >> 16) - 0x4300;
            int32_t units = SCHEME == kLinear ? k : ((1 << k) >> 1);
            if (__float_as_uint(v[0][c]) >> 31) units = -units;
            if (units != 0) atomicAdd(&sum[(c >> 2) * 128 + (c & 3)], units);
        }
    }
    __syncwarp();
}

// The rare flush when one stage alone queues more than a queue's worth of row-groups: kept out of
// line so that the common path holds one inlined copy of the full decision.
template <typename T, int SCHEME, bool TRUSTED>
__device__ __noinline__ void flush_queue_cold(const WarpQueue<T>& q, int cnt, int lane,
                                              const QuantArgs& a, const Decide& dc) {
    flush_queue<T, SCHEME, TRUSTED>(q, cnt, lane, a, dc);
}

template <typename T>
__device__ __forceinline__ void push_item(const WarpQueue<T>& q, int pos,
                                          const uint4 (&raw)[CompactCfg<T>::kXVec], uint4 wd,
                                          uint32_t g32, uint32_t worker) {
#pragma unroll
    for (int h = 0; h < CompactCfg<T>::kXVec; ++h) q.qx[pos * CompactCfg<T>::kXVec + h] = raw[h];
    q.qw[pos] = wd;
    q.qm[pos] = make_uint2(g32, worker);
}

// One stage (rows r0 .. r0 + nrows - 1 of this thread's group) through the compacting
// consumer: every row-group's largest magnitude, the rows' random words (independent chains the
// scheduler interleaves), the certainty test, then the row-groups that fail it are queued (one
// ballot per row, one position each; the queue is flushed first if they would not fit).
// g32: the group index with the chunk's sum buffer in bit 31 (what a queued item records).
// count: queued row-groups of the warp (warp-uniform).
// ROW_BYTES: the stage's row pitch; release: run by lane 0 once every row of the stage is in
// registers (frees the stage for the next copy).
// RB: the rows this copy handles (nrows <= RB); COLD: decide an overflowing queue out of line.
template <typename T, int SCHEME, bool TRUSTED, int ROW_BYTES, int RB, bool COLD,
          typename Release>
__device__ __forceinline__ void tma_consume_compact_rows(const unsigned char* stage, int lane,
                                                         bool active, uint32_t r0, uint32_t nrows,
                                                         uint32_t g32, const PhiloxGroup& pg,
                                                         const QuantArgs& a, const Decide& dc,
                                                         const Release& release,
                                                         const WarpQueue<T>& q, int& count) {
    using C = CompactCfg<T>;
    uint4 raw[RB][C::kXVec];
#pragma unroll
    for (int u = 0; u < RB; ++u) {
        const uint4* p = reinterpret_cast<const uint4*>(stage + u * ROW_BYTES);
#pragma unroll
        for (int h = 0; h < C::kXVec; ++h) raw[u][h] = p[h];  // rows past nrows are ignored
    }
    __syncwarp();
    if (lane == 0) release();  // every row of the stage is in registers
    float mx[RB];
    uint32_t any = 0u;
#pragma unroll
    for (int u = 0; u < RB; ++u) {
        const float m = group_max_abs<T, TRUSTED>(raw[u]);
        mx[u] = (active && static_cast<uint32_t>(u) < nrows) ? m : 0.0f;
        any |= __float_as_uint(mx[u]);
    }
    // a stage that is zero across the warp (sparse layers) needs no random words at all
    if (!__any_sync(0xFFFFFFFFu, any != 0u)) return;
    const uint32_t w0 = r0 + a.row0;
    uint4 wd[RB];
    if (nrows == RB) {
#pragma unroll
        for (int u = 0; u < RB; ++u) wd[u] = philox_row(pg, w0 + u, a.step_lo, a.rk);
    } else {
#pragma unroll
        for (int u = 0; u < RB; ++u)
            wd[u] = static_cast<uint32_t>(u) < nrows ? philox_row(pg, w0 + u, a.step_lo, a.rk)
                                                     : make_uint4(0u, 0u, 0u, 0u);
    }
    unsigned mk[RB];
    int tot = 0;
#pragma unroll
    for (int u = 0; u < RB; ++u) {
        const uint4 w = wd[u];
        const uint32_t h2 = __vminu2(__vminu2(w.x, w.y), __vminu2(w.z, w.w));
        const uint32_t minh = min(h2 & 0xFFFFu, h2 >> 16);
        const uint32_t pbm = __float_as_uint(__fmaf_rn(mx[u], dc.c1, dc.c0));
        // P_c + 3 > min H (unsigned: a NaN, infinite or P_c >= 1 estimate always queues)
        const bool nd = __float_as_uint(mx[u]) != 0u && (!dc.fast || pbm - dc.lsub > minh);
        mk[u] = __ballot_sync(0xFFFFFFFFu, nd);
        tot += __popc(mk[u]);
    }
    if (tot == 0) return;
    const unsigned lt = (1u << lane) - 1u;
    if (count + tot > kQueue) {
        if (COLD)
            flush_queue_cold<T, SCHEME, TRUSTED>(q, count, lane, a, dc);
        else
            flush_queue<T, SCHEME, TRUSTED>(q, count, lane, a, dc);
        count = 0;
    }
    if (tot <= kQueue) {
        int base = count;
#pragma unroll
        for (int u = 0; u < RB; ++u) {
            if ((mk[u] >> lane) & 1u)
                push_item<T>(q, base + __popc(mk[u] & lt), raw[u], wd[u], g32, w0 + u);
            base += __popc(mk[u]);
        }
        count += tot;
        return;
    }
    // more than a queue's worth in this one stage (rare): row by row
#pragma unroll
    for (int u = 0; u < RB; ++u) {
        const int c = __popc(mk[u]);
        if (count + c > kQueue) {
            flush_queue_cold<T, SCHEME, TRUSTED>(q, count, lane, a, dc);
            count = 0;
        }
        if ((mk[u] >> lane) & 1u)
            push_item<T>(q, count + __popc(mk[u] & lt), raw[u], wd[u], g32, w0 + u);
        count += c;
    }
}

// Barriers of the ring: full[k] completes when stage k's copies land (the producer's arrival
// plus the bytes), empty[k] when every consumer warp has read it.
template <int STAGES>
__device__ __forceinline__ void tma_init_barriers(uint64_t (&full_bar)[STAGES],
                                                  uint64_t (&empty_bar)[STAGES],
                                                  volatile int* abort_flag) {
    if (threadIdx.x == 0) {
#pragma unroll
        for (int k = 0; k < STAGES; ++k) {
            mbar_init(smem_u32(&full_bar[k]), 1u);
            mbar_init(smem_u32(&empty_bar[k]), static_cast<uint32_t>(kTmaWarps));
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
}

// Producer, item `item` of the block: wait (bounded) until its stage is free, then copy `rows`
// rows of row_bytes starting at src (row stride ld elements) into it.  False if the wait gave up
// or the consumers stopped.  nst stages of stage_bytes each (at most STAGES).
template <typename T, int STAGES>
__device__ __forceinline__ bool tma_issue(uint32_t item, const T* src, int64_t ld, int rows,
                                          uint32_t row_bytes, unsigned char* smem,
                                          uint64_t (&full_bar)[STAGES],
                                          uint64_t (&empty_bar)[STAGES],
                                          volatile int* abort_flag, uint32_t nst = STAGES,
                                          uint32_t stage_bytes = TmaCfg<T>::kStageBytes) {
    using Cfg = TmaCfg<T>;
    const uint32_t st = item % nst;
    if (item >= nst && !mbar_wait(smem_u32(&empty_bar[st]), ((item / nst) - 1u) & 1u))
        return false;
    if (*abort_flag) return false;
    const uint32_t fb = smem_u32(&full_bar[st]);
    mbar_arrive_expect_tx(fb, static_cast<uint32_t>(rows) * row_bytes);
    const uint32_t dst = smem_u32(smem + st * stage_bytes);
    for (int u = 0; u < rows; ++u) bulk_load(dst + u * Cfg::kRowBytes, src + u * ld, row_bytes, fb);
    return true;
}

// Producer epilogue: on failure record the timeout and stop the consumers; then wait (bounded)
// for the last issued stages, so that the block never exits with copies in flight.
template <int STAGES>
__device__ __forceinline__ void tma_drain(bool ok, uint32_t item, uint64_t (&full_bar)[STAGES],
                                          volatile int* abort_flag,
                                          unsigned int* __restrict__ status,
                                          uint32_t nst = STAGES) {
    if (!ok) {
        if (status) atomicCAS(status, 0u, kStatusTimeout);
        *abort_flag = 1;
    }
    const uint32_t inflight = item < nst ? item : nst;
    for (uint32_t k = 0; k < inflight; ++k) {
        const uint32_t it = item - 1 - k;
        mbar_wait(smem_u32(&full_bar[it % nst]), (it / nst) & 1u);
    }
}

// Consumer wait for item `item`: bounded, and decided uniformly by the warp.
template <int STAGES>
__device__ __forceinline__ bool tma_wait_slot(uint32_t slot, uint32_t phase,
                                              uint64_t (&full_bar)[STAGES],
                                              volatile int* abort_flag) {
    const bool got = mbar_wait(smem_u32(&full_bar[slot]), phase);
    return __all_sync(0xFFFFFFFFu, got && !*abort_flag);
}
template <int STAGES>
__device__ __forceinline__ bool tma_wait_full(uint32_t item, uint64_t (&full_bar)[STAGES],
                                              volatile int* abort_flag) {
    const bool got = mbar_wait(smem_u32(&full_bar[item % STAGES]), (item / STAGES) & 1u);
    return __all_sync(0xFFFFFFFFu, got && !*abort_flag);
}

// ZSKIP: rows that are zero across the whole warp skip their random words.  COMPACT (no codes):
// the compacting consumer above; the dynamic shared memory then holds its queues after the ring.
// RS: rows per ring stage (TmaCfg<T>::kRows; 1 or 2 for one or two workers: as many stages
// as the ring holds, so that as many bytes stay in flight as with full stages and the
// compacting consumer spends no work on empty row slots).
template <typename T, int SCHEME, int CODE_BITS, bool WRITE_OUT, bool TRUSTED, int SUB,
          bool ZSKIP = false, bool COMPACT = false, int RS = TmaCfg<T>::kRows>
__global__ void __launch_bounds__(kTmaBlock, 1)
quantize_tma_kernel(const T* __restrict__ x, QuantArgs a, int64_t groups,
                    unsigned char* __restrict__ codes, void* __restrict__ out,
                    unsigned int* __restrict__ status) {
    using Cfg = TmaCfg<T>;
    constexpr int RB = Cfg::kRows;
    constexpr int NS = COMPACT ? CompactCfg<T>::kStages : Cfg::kStages;  // stages of RB rows
    static_assert(RS == RB || RS == 2 || RS == 1, "stages of kRows rows, or of two or one");
    constexpr uint32_t NST = static_cast<uint32_t>(NS * RB / RS);  // stages of RS rows
    constexpr uint32_t kStageB = static_cast<uint32_t>(RS * Cfg::kRowBytes);
    extern __shared__ __align__(128) unsigned char tma_smem[];
    __shared__ __align__(8) uint64_t full_bar[NST];
    __shared__ __align__(8) uint64_t empty_bar[NST];
    __shared__ float sh_scale;
    __shared__ volatile int sh_abort;

    const int tid = threadIdx.x;
    pdl_wait();  // the norm of the fused call's first pass
    const float nrm = __ldg(a.norm_ptr);
    const float scale = block_scale<SCHEME>(nrm, a.n, a.s, &sh_scale);
    const bool live = nrm > 0.0f && nrm < __uint_as_float(kInfBits);
    tma_init_barriers<NST>(full_bar, empty_bar, &sh_abort);

    const int64_t full = live ? a.d / kQCols : 0;  // groups taken through shared memory
    const int64_t nchunks = (full + kTmaConsumers - 1) / kTmaConsumers;
    const int64_t nbatch = (a.n + RS - 1) / RS;
    GQ_BOUND(RS == RB || a.n <= RS);  // short stages hold every worker of a chunk

    if (tid >= kTmaConsumers) {
        if (tid == kTmaConsumers) {  // producer: lane 0 of the last warp
            uint32_t item = 0;
            bool ok = true;
            for (int64_t q = blockIdx.x; q < nchunks && ok; q += gridDim.x) {
                const int64_t g0 = (nchunks - 1 - q) * kTmaConsumers;
                const int64_t ng = min(static_cast<int64_t>(kTmaConsumers), full - g0);
                const uint32_t row_bytes = static_cast<uint32_t>(ng * kQCols * sizeof(T));
                for (int64_t b = 0; b < nbatch; ++b) {
                    const int rows = static_cast<int>(min(static_cast<int64_t>(RS), a.n - b * RS));
                    GQ_BOUND(rows >= 1 && b * RS + rows <= a.n && g0 >= 0 && ng >= 1 &&
                             (g0 + ng) * kQCols <= a.d);
                    ok = tma_issue<T, NST>(item, x + b * RS * a.d + g0 * kQCols, a.d, rows,
                                           row_bytes, tma_smem, full_bar, empty_bar, &sh_abort,
                                           NST, kStageB);
                    if (!ok) break;
                    ++item;  // counts the stages actually issued
                }
            }
            tma_drain<NST>(ok, item, full_bar, &sh_abort, status);
        }
    } else if (COMPACT && nchunks > 0) {  // consumers, compacting
        static_assert(!COMPACT || CODE_BITS == 0, "the compacting consumer writes no codes");
        using C = CompactCfg<T>;
        const Decide dc = make_decide<SCHEME>(nrm, a.s, a.u16);
        const int lane = tid & 31;
        const WarpQueue<T> wq = warp_queue<T>(tma_smem + NS * Cfg::kStageBytes, tid >> 5);
        int4* const lsum = reinterpret_cast<int4*>(wq.sum) + lane;  // this lane's 16-byte pieces
#pragma unroll
        for (int h = 0; h < C::kSumBufs * 2; ++h) lsum[h * 32] = make_int4(0, 0, 0, 0);
        // a chunk's output: its sums (complete after a flush) scaled, and the buffer cleared
        const auto emit = [&](int64_t gg, bool act, uint32_t buf) {
            const int4 lo = lsum[buf * 64], hi = lsum[buf * 64 + 32];
            lsum[buf * 64] = make_int4(0, 0, 0, 0);
            lsum[buf * 64 + 32] = make_int4(0, 0, 0, 0);
            // exact: integers below 2^24
            float S[kQCols] = {static_cast<float>(lo.x), static_cast<float>(lo.y),
                               static_cast<float>(lo.z), static_cast<float>(lo.w),
                               static_cast<float>(hi.x), static_cast<float>(hi.y),
                               static_cast<float>(hi.z), static_cast<float>(hi.w)};
            if (act && WRITE_OUT) store_out(out, a.sums, a.sums_i8, a.out_dtype, gg, a.d, scale, S);
        };
        int count = 0;
        uint32_t slot = 0, phase = 0;  // ring position of the next stage
        uint32_t buf = 0;              // sum buffer of the current chunk
        bool pending = false;          // the previous chunk's output waits for the next flush
        int64_t pend_g = 0;
        bool pend_act = false;
        bool ok = true;
        for (int64_t q = blockIdx.x; q < nchunks; q += gridDim.x) {
            const int64_t g = (nchunks - 1 - q) * kTmaConsumers + tid;
            const bool active = g < full;
            const PhiloxGroup pg = philox_group(static_cast<uint32_t>(g), a.step_lo, a.step_hi, a.rk);
            const uint32_t tag = static_cast<uint32_t>(g) | (buf << 31);
            for (int64_t b = 0; b < nbatch; ++b) {
                if (!tma_wait_slot<NST>(slot, phase, full_bar, &sh_abort)) {
                    ok = false;
                    break;
                }
                const unsigned char* stage = tma_smem + slot * kStageB + tid * kQCols * sizeof(T);
                const uint32_t eb = smem_u32(&empty_bar[slot]);
                tma_consume_compact_rows<T, SCHEME, TRUSTED, Cfg::kRowBytes, RS, (RS < RB)>(
                    stage, lane, active, static_cast<uint32_t>(b * RS),
                    static_cast<uint32_t>(min(static_cast<int64_t>(RS), a.n - b * RS)), tag, pg,
                    a, dc, [eb] { mbar_arrive(eb); }, wq, count);
                if (++slot == NST) {
                    slot = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) break;
            if (C::kSumBufs == 1 || pending) {  // one flush completes this chunk (and the previous)
                flush_queue<T, SCHEME, TRUSTED>(wq, count, lane, a, dc);
                count = 0;
                if (pending) emit(pend_g, pend_act, buf ^ 1u);
                emit(g, active, buf);
                pending = false;
            } else {
                pending = true;
                pend_g = g;
                pend_act = active;
            }
            buf ^= static_cast<uint32_t>(C::kSumBufs - 1);
        }
        if (ok && pending) {
            flush_queue<T, SCHEME, TRUSTED>(wq, count, lane, a, dc);
            emit(pend_g, pend_act, buf ^ 1u);
        }
        if (!ok) {
            if (status) atomicCAS(status, 0u, kStatusTimeout);
            sh_abort = 1;
        }
    } else if (nchunks > 0) {  // consumers
        const Decide dc = make_decide<SCHEME>(nrm, a.s, a.u16);
        const int lane = tid & 31;
        uint32_t slot = 0, phase = 0;  // ring position of the next stage
        bool ok = true;
        for (int64_t q = blockIdx.x; q < nchunks && ok; q += gridDim.x) {
            const int64_t g = (nchunks - 1 - q) * kTmaConsumers + tid;
            const bool active = g < full;
            const PhiloxGroup pg = philox_group(static_cast<uint32_t>(g), a.step_lo, a.step_hi, a.rk);
            float S[kQCols];
#pragma unroll
            for (int c = 0; c < kQCols; ++c) S[c] = 0.0f;
            bool probe = true;
            // (stage b holds rows b RB ..; short stages hold all the workers: b = 0)
            for (int64_t b = 0; b < nbatch; ++b) {
                if (!tma_wait_slot<NST>(slot, phase, full_bar, &sh_abort)) {
                    ok = false;
                    break;
                }
                const unsigned char* stage = tma_smem + slot * kStageB + tid * kQCols * sizeof(T);
                tma_consume_stage<T, SCHEME, CODE_BITS, TRUSTED, SUB, ZSKIP>(
                    stage, lane, active, b, g, pg, a, dc, smem_u32(&empty_bar[slot]), S, codes,
                    &probe);
                if (++slot == NST) {
                    slot = 0;
                    phase ^= 1u;
                }
            }
            if (ok && active && WRITE_OUT)
                store_out(out, a.sums, a.sums_i8, a.out_dtype, g, a.d, scale, S);
        }
        if (!ok) {
            if (status) atomicCAS(status, 0u, kStatusTimeout);
            sh_abort = 1;
        }
    }
    if (tid >= kTmaConsumers) return;

    // ---- the groups [full, groups): ragged last group, code padding, or all of them when the
    // norm is 0 or not finite; direct loads by the consumer threads
    const Decide dc = make_decide<SCHEME>(nrm, a.s, a.u16);
    const int64_t rest = groups - full;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kTmaConsumers;
    for (int64_t it = static_cast<int64_t>(blockIdx.x) * kTmaConsumers + tid; it < rest;
         it += stride) {
        const int64_t g = groups - 1 - it;
        float S[kQCols];
        if (live) {
            quantize_group<T, SCHEME, CODE_BITS, TRUSTED>(x, a, dc, g, codes, S);
        } else {
#pragma unroll
            for (int c = 0; c < kQCols; ++c) S[c] = 0.0f;
            if (CODE_BITS) {
                const int32_t zero[kQCols] = {0, 0, 0, 0, 0, 0, 0, 0};
                for (int64_t i = 0; i < a.n; ++i) store_codes<CODE_BITS>(codes, i, g, a.pitch, zero);
            }
        }
        if (WRITE_OUT) store_out(out, a.sums, a.sums_i8, a.out_dtype, g, a.d, scale, S);
    }
}

// The segmented form of the bulk-copy pass: the chunks of all segments of a launch (segment k
// owns chunks L.seg[k].b0 .. b0 + nb - 1 of 3840 columns; nb = 0 for a segment whose rows are
// not 16-byte aligned) run through one ring, last chunk first; each chunk takes its segment's
// norm and scale (written by norm_segments_kernel) and its random stream (step << 16) | l.  The
// groups outside the chunks (a ragged last group, or every group of an unaligned segment) are
// done afterwards with direct loads.  No codes; trusted norms.
template <typename T, int SCHEME>
__global__ void __launch_bounds__(kTmaBlock, 1)
quantize_seg_tma_kernel(const __grid_constant__ SegLaunch L, QuantArgs base, int32_t nchunks,
                        unsigned char* __restrict__ ws) {
    using Cfg = TmaCfg<T>;
    constexpr int RB = Cfg::kRows;
    constexpr int NS = Cfg::kStages;
    extern __shared__ __align__(128) unsigned char tma_smem[];
    __shared__ __align__(8) uint64_t full_bar[NS];
    __shared__ __align__(8) uint64_t empty_bar[NS];
    __shared__ volatile int sh_abort;

    const int tid = threadIdx.x;
    unsigned int* status = &reinterpret_cast<WsHeader*>(ws)->status;
    const float* norms = reinterpret_cast<const float*>(ws + kSegNormsOff);
    const float* scales = reinterpret_cast<const float*>(ws + kSegScalesOff);
    tma_init_barriers<NS>(full_bar, empty_bar, &sh_abort);
    const int64_t nbatch = (base.n + RB - 1) / RB;

    if (tid >= kTmaConsumers) {
        if (tid == kTmaConsumers) {  // producer: lane 0 of the last warp
            uint32_t item = 0;
            bool ok = true;
            int k = -1;
            for (int32_t q = blockIdx.x; q < nchunks && ok; q += gridDim.x) {
                const int32_t cg = nchunks - 1 - q;
                // chunks come in decreasing order: search only when cg leaves segment k
                if (k < 0 || cg < L.seg[k].b0) k = find_segment(L, cg);
                const SegDesc& sd = L.seg[k];
                const int64_t g0 = static_cast<int64_t>(cg - sd.b0) * kTmaConsumers;
                const int64_t ng = min(static_cast<int64_t>(kTmaConsumers), sd.d / kQCols - g0);
                const uint32_t row_bytes = static_cast<uint32_t>(ng * kQCols * sizeof(T));
                const T* x = static_cast<const T*>(sd.x);
                GQ_BOUND(k >= 0 && k < L.nseg && g0 >= 0 && ng >= 1 &&
                         (g0 + ng) * kQCols <= sd.d);
                for (int64_t b = 0; b < nbatch; ++b) {
                    const int rows = static_cast<int>(min(static_cast<int64_t>(RB), base.n - b * RB));
                    ok = tma_issue<T, NS>(item, x + b * RB * sd.d + g0 * kQCols, sd.d, rows,
                                          row_bytes, tma_smem, full_bar, empty_bar, &sh_abort);
                    if (!ok) break;
                    ++item;
                }
            }
            tma_drain<NS>(ok, item, full_bar, &sh_abort, status);
        }
        return;
    }

    // consumers; the segment of the current chunk, its arguments and decision constants are
    // kept while consecutive chunks stay in it
    const int lane = tid & 31;
    uint32_t item = 0;
    bool ok = true;
    int k = -1;
    QuantArgs a = base;
    Decide dc;
    float scale = 0.0f;
    for (int32_t q = blockIdx.x; q < nchunks && ok; q += gridDim.x) {
        const int32_t cg = nchunks - 1 - q;
        if (k < 0 || cg < L.seg[k].b0) {
            k = find_segment(L, cg);
            a.d = L.seg[k].d;
            a.step_lo = base.step_lo | static_cast<uint32_t>(L.seg0 + k);
            dc = make_decide<SCHEME>(norms[k], a.s, a.u16);
            scale = scales[k];
        }
        const SegDesc& sd = L.seg[k];
        const int64_t g = static_cast<int64_t>(cg - sd.b0) * kTmaConsumers + tid;
        const bool active = g < sd.d / kQCols;
        const PhiloxGroup pg = philox_group(static_cast<uint32_t>(g), a.step_lo, a.step_hi, a.rk);
        float S[kQCols];
#pragma unroll
        for (int c = 0; c < kQCols; ++c) S[c] = 0.0f;
        for (int64_t b = 0; b < nbatch; ++b, ++item) {
            if (!tma_wait_full<NS>(item, full_bar, &sh_abort)) {
                ok = false;
                break;
            }
            const unsigned char* stage =
                tma_smem + (item % NS) * Cfg::kStageBytes + tid * kQCols * sizeof(T);
            tma_consume_stage<T, SCHEME, 0, true, 2>(stage, lane, active, b, g, pg, a, dc,
                                                     smem_u32(&empty_bar[item % NS]), S, nullptr);
        }
        if (ok && active) store_out(sd.out, nullptr, 0, base.out_dtype, g, sd.d, scale, S);
    }
    if (!ok) {
        atomicCAS(status, 0u, kStatusTimeout);
        sh_abort = 1;
        return;
    }

    // groups outside the chunks, numbered across the launch (segment k owns t0 .. t0 + its
    // count - 1, last group first), direct loads
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kTmaConsumers;
    k = -1;
    for (int64_t it = static_cast<int64_t>(blockIdx.x) * kTmaConsumers + tid; it < L.ntail;
         it += stride) {
        const int kt = find_tail_segment(L, it);
        const SegDesc& sd = L.seg[kt];
        if (kt != k) {
            k = kt;
            a.d = sd.d;
            a.pitch = (sd.d + 31) / 32 * 32;
            a.vec_rows = sd.nb > 0;
            a.step_lo = base.step_lo | static_cast<uint32_t>(L.seg0 + k);
            a.norm_ptr = norms + k;
            dc = make_decide<SCHEME>(norms[k], a.s, a.u16);
            scale = scales[k];
        }
        const int64_t g = (sd.d + kQCols - 1) / kQCols - 1 - (it - sd.t0);
        float S[kQCols];
        quantize_group<T, SCHEME, 0, true>(static_cast<const T*>(sd.x), a, dc, g, nullptr, S);
        store_out(sd.out, nullptr, 0, base.out_dtype, g, sd.d, scale, S);
    }
}

// ------------------------------------------------------------------------------------------
// Single-launch form for problems whose n x d matrix fits in the grid's shared memory.  Each
// block copies its slice of columns (all n rows, 16-byte aligned rows) into shared memory with
// bulk copies, takes its partial of the norm from there, meets the other blocks at a grid
// barrier (cooperative launch: every block resident; the wait is bounded), combines the partials
// into the same norm in every block, and then quantises, sums over the workers and dequantises
// from shared memory: the matrix crosses DRAM once, in one launch.  Random words, decisions and
// outputs are those of the two-pass kernels; the (2,2) and (inf,2) norms are sums whose rounding
// depends on how the blocks split them (the others are maxima and equal the two-pass norm).
// ------------------------------------------------------------------------------------------
constexpr int kResThreads = 512;
constexpr int kResTileBytes = 200 * 1024;  // at most this much of a block's slice

__device__ __forceinline__ unsigned int ld_acquire_u32(const unsigned int* p) {
    unsigned int v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ unsigned int atom_add_acq_rel(unsigned int* p, unsigned int v) {
    unsigned int old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v)
                 : "memory");
    return old;
}
__device__ __forceinline__ void red_add_release(unsigned int* p, unsigned int v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Barrier of the nblk (< 256) blocks of a cooperative launch on one workspace word holding
// generation << 8 | arrivals.  Thread 0 of each block arrives with an acquire-release add
// (releasing the block's writes made by thread 0); the last arrival adds 256 - nblk, which
// clears the arrivals and advances the generation in one release, and the others wait, with
// acquire loads, for the generation to move.  Only writes of thread 0 before the barrier are
// published to the other blocks.  A block that waits longer than kWaitLimitNs records
// GQ_ERR_TIMEOUT and gets false (the same in all its threads).
__device__ __forceinline__ bool grid_barrier(WsHeader* hdr, unsigned int nblk,
                                             volatile int* sh_flag) {
    __syncthreads();
    if (threadIdx.x == 0) {
        const unsigned int old = atom_add_acq_rel(&hdr->bar, 1u);
        bool ok = true;
        if ((old & 0xFFu) == nblk - 1u) {
            red_add_release(&hdr->bar, 256u - nblk);
        } else {
            const unsigned int gen = old >> 8;
            const uint64_t t0 = global_ns();
            while ((ld_acquire_u32(&hdr->bar) >> 8) == gen) {
                if (global_ns() - t0 > kWaitLimitNs) {
                    ok = false;
                    break;
                }
                __nanosleep(20);
            }
            if (!ok) atomicCAS(&hdr->status, 0u, kStatusTimeout);
        }
        *sh_flag = ok ? 1 : 0;
    }
    __syncthreads();
    return *sh_flag != 0;
}

// The fixed-order combine of nb block partials by one warp (valid in lane 0): their max or sum.
template <int MODE>
__device__ __forceinline__ double warp_combine(const uint64_t* partials, int nb) {
    const int lane = threadIdx.x & 31;
    if (MODE == kMaxMax || MODE == kL2Max) {
        uint64_t m = 0;
        for (int b = lane; b < nb; b += 32) {
            const uint64_t v = __ldcg(reinterpret_cast<const unsigned long long*>(partials + b));
            m = v > m ? v : m;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const uint64_t t = __shfl_down_sync(0xFFFFFFFFu, m, o);
            m = t > m ? t : m;
        }
        return __longlong_as_double(static_cast<long long>(m));
    } else {
        double v = 0.0;
        for (int b = lane; b < nb; b += 32)
            v += __longlong_as_double(static_cast<long long>(
                __ldcg(reinterpret_cast<const unsigned long long*>(partials + b))));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_down_sync(0xFFFFFFFFu, v, o);
        return v;
    }
}

// One element of a shared-memory tile, widened to fp32.
__device__ __forceinline__ float smem_one(const float* p) { return *p; }
__device__ __forceinline__ float smem_one(const uint16_t* p) {
    return __uint_as_float(static_cast<uint32_t>(*p) << 16);
}

// Block b owns column groups [b gpb, (b + 1) gpb) of kQCols columns, all n rows, as an n x
// (gpb kQCols) tile in dynamic shared memory.
template <typename T, int SCHEME, int MODE>
__global__ void __launch_bounds__(kResThreads, 1)
resident_kernel(const T* __restrict__ x, QuantArgs a, int64_t gpb, void* __restrict__ out,
                float* __restrict__ norm_user, unsigned char* __restrict__ ws) {
    extern __shared__ __align__(128) unsigned char res_smem[];
    __shared__ __align__(8) uint64_t bar;
    __shared__ double sh_d[kResThreads / 32];
    __shared__ uint64_t sh_u[kResThreads / 32];
    __shared__ float sh_norm, sh_scale;
    __shared__ Decide sh_dc;
    __shared__ volatile int sh_flag;
    __shared__ float sh_S[kResThreads / 2][kQCols];  // split row pairs' sums (ng <= 256)
    WsHeader* hdr = reinterpret_cast<WsHeader*>(ws);
    uint64_t* partials = reinterpret_cast<uint64_t*>(ws + kHeaderBytes);
    const int tid = threadIdx.x;
    const int64_t n = a.n, d = a.d;
    const int64_t groups = (d + kQCols - 1) / kQCols;
    const int64_t g0 = static_cast<int64_t>(blockIdx.x) * gpb;
    const int64_t ng = max(min(groups - g0, gpb), static_cast<int64_t>(0));
    const int64_t c0 = g0 * kQCols;
    const int64_t cols = ng > 0 ? min(d - c0, gpb * kQCols) : 0;  // columns present
    const int64_t pitch = gpb * kQCols;                              // tile row, elements
    const T* tile = reinterpret_cast<const T*>(res_smem);

    // 1. the slice into shared memory: bulk copies of up to 8 KB of a row, issued by the lanes
    // of the first warp and counted on one mbarrier
    if (tid == 0) {
        mbar_init(smem_u32(&bar), 1u);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    bool ok = true;
    if (ng > 0) {
        constexpr uint32_t kPiece = 8192;
        const uint32_t row_bytes = static_cast<uint32_t>(cols * static_cast<int64_t>(sizeof(T)));
        const uint32_t pieces = (row_bytes + kPiece - 1) / kPiece;  // per row
        if (tid < 32) {
            if (tid == 0)
                mbar_arrive_expect_tx(smem_u32(&bar), static_cast<uint32_t>(n) * row_bytes);
            __syncwarp();
            for (uint32_t q = tid; q < static_cast<uint32_t>(n) * pieces; q += 32) {
                const uint32_t i = q / pieces, k = q - i * pieces;
                const uint32_t off = k * kPiece;  // bytes into the row, a multiple of 16
                const uint32_t len = min(kPiece, row_bytes - off);
                bulk_load(smem_u32(reinterpret_cast<const unsigned char*>(tile + i * pitch) + off),
                          reinterpret_cast<const unsigned char*>(x + i * d + c0) + off, len,
                          smem_u32(&bar));
            }
        }
        ok = mbar_wait(smem_u32(&bar), 0u, kWaitLimitNs);
    }
    ok = __syncthreads_and(ok) != 0;
    if (!ok) {
        if (tid == 0) {
            atomicCAS(&hdr->status, 0u, kStatusTimeout);
            mbar_wait(smem_u32(&bar), 0u, kWaitLimitNs);  // let the copies in flight land
        }
    } else if (ng * kQCols > cols) {
        // the ragged last group: zero the columns past d (they add nothing to the norm)
        T* t = reinterpret_cast<T*>(res_smem);
        for (int64_t e = tid; e < n * (ng * kQCols - cols); e += kResThreads) {
            const int64_t i = e / (ng * kQCols - cols), c = cols + e % (ng * kQCols - cols);
            t[i * pitch + c] = T(0);
        }
    }
    __syncthreads();

    // 2. this block's partial of the norm
    uint32_t maxbits = 0;
    ScaledSumSq ssq;
    ssq.init();
    int64_t best_key = INT64_MIN;
    uint32_t bad_col = 0;
    if (ok && (MODE == kMaxMax || MODE == kL2L2)) {
        // these two do not depend on the column: the tile's n x (8 ng) elements, 16 bytes per
        // thread step, all threads busy however few the column groups
        constexpr int V = 16 / static_cast<int>(sizeof(T));
        const uint32_t vrow = static_cast<uint32_t>(ng * kQCols / V);
        const uint32_t nv = static_cast<uint32_t>(n) * vrow;  // <= 200 KB / 16
        for (uint32_t e = tid; e < nv; e += kResThreads) {
            const uint32_t i = e / vrow, vc = e - i * vrow;
            float v[Elem<T>::kCols];
            widen16<T>(*reinterpret_cast<const uint4*>(tile + i * pitch + vc * V), v);
            if (MODE == kMaxMax) {
#pragma unroll
                for (int c = 0; c < Elem<T>::kCols; ++c) {
                    const uint32_t b = __float_as_uint(v[c]) & 0x7FFFFFFFu;
                    maxbits = b > maxbits ? b : maxbits;
                }
            } else {
                ssq.add<Elem<T>::kCols>(v);
            }
        }
    } else if (ok) {
        for (int64_t gl = tid; gl < ng; gl += kResThreads) {
            const T* col0 = tile + gl * kQCols;
            if (MODE == kMaxL2) {
                uint32_t colmax[kQCols];
#pragma unroll
                for (int c = 0; c < kQCols; ++c) colmax[c] = 0u;
                for (int64_t i = 0; i < n; ++i) {
                    float v[kQCols];
                    const uint4* p = reinterpret_cast<const uint4*>(col0 + i * pitch);
                    unstage<T>(p, p + 1, v);
#pragma unroll
                    for (int c = 0; c < kQCols; ++c) {
                        const uint32_t b = __float_as_uint(v[c]) & 0x7FFFFFFFu;
                        colmax[c] = b > colmax[c] ? b : colmax[c];
                    }
                }
                float m[kQCols];
#pragma unroll
                for (int c = 0; c < kQCols; ++c) m[c] = __uint_as_float(colmax[c]);
                ssq.add<kQCols>(m);
            } else {
                // (2, inf): column sums of squares with the arithmetic of norm_kernel (plain FMA
                // into NA interleaved accumulators, row i into accumulator i mod NA, when
                // n <= 16 NA; a scaled sum for the rest and for columns outside the normal range)
                constexpr int NA = Elem<T>::kCols == 8 ? 2 : 4;
                if (n <= 16 * NA) {
                    float acc[NA][kQCols];
#pragma unroll
                    for (int q = 0; q < NA; ++q)
#pragma unroll
                        for (int c = 0; c < kQCols; ++c) acc[q][c] = 0.0f;
                    for (int64_t i0 = 0; i0 < n; i0 += NA) {
#pragma unroll
                        for (int q = 0; q < NA; ++q) {
                            if (i0 + q >= n) break;
                            float v[kQCols];
                            const uint4* p = reinterpret_cast<const uint4*>(col0 + (i0 + q) * pitch);
                            unstage<T>(p, p + 1, v);
#pragma unroll
                            for (int c = 0; c < kQCols; ++c) acc[q][c] = __fmaf_rn(v[c], v[c], acc[q][c]);
                        }
                    }
#pragma unroll
                    for (int c = 0; c < kQCols; ++c) {
                        float sum = acc[0][c];
#pragma unroll
                        for (int q = 1; q < NA; ++q) sum = sum + acc[q][c];
                        if (sum >= 0x1p-100f && sum < __uint_as_float(kInfBits)) {
                            const int64_t key = scaled_key(sum, 0);
                            best_key = key > best_key ? key : best_key;
                            continue;
                        }
                        if (sum == 0.0f) continue;
                        ScaledSumSq cs;
                        cs.init();
                        for (int64_t i = 0; i < n; ++i) {
                            const float one[1] = {smem_one(col0 + i * pitch + c)};
                            cs.add<1>(one);
                        }
                        const float ssum = cs.sum();
                        if (!(ssum < __uint_as_float(kInfBits))) {
                            const uint32_t b = __float_as_uint(ssum) & 0x7FFFFFFFu;
                            bad_col = b > bad_col ? b : bad_col;
                        } else if (ssum > 0.0f) {
                            const int64_t key = scaled_key(ssum, cs.e);
                            best_key = key > best_key ? key : best_key;
                        }
                    }
                } else {
                    ScaledSumSq col[kQCols];
#pragma unroll
                    for (int c = 0; c < kQCols; ++c) col[c].init();
                    for (int64_t i = 0; i < n; ++i) {
                        float v[kQCols];
                        const uint4* p = reinterpret_cast<const uint4*>(col0 + i * pitch);
                        unstage<T>(p, p + 1, v);
#pragma unroll
                        for (int c = 0; c < kQCols; ++c) {
                            const float one[1] = {v[c]};
                            col[c].add<1>(one);
                        }
                    }
#pragma unroll
                    for (int c = 0; c < kQCols; ++c) {
                        const float sum = col[c].sum();
                        if (!(sum < __uint_as_float(kInfBits))) {
                            const uint32_t b = __float_as_uint(sum) & 0x7FFFFFFFu;
                            bad_col = b > bad_col ? b : bad_col;
                        } else if (sum > 0.0f) {
                            const int64_t key = scaled_key(sum, col[c].e);
                            best_key = key > best_key ? key : best_key;
                        }
                    }
                }
            }
        }
    }

    // 3. the partials of all blocks, the same norm in every block
    const uint64_t part =
        block_partial<MODE, kResThreads>(maxbits, ssq, best_key, bad_col, sh_d, sh_u);
    GQ_BOUND(blockIdx.x < static_cast<unsigned>(kMaxPartials));
    if (tid == 0) partials[blockIdx.x] = part;
    if (!grid_barrier(hdr, gridDim.x, &sh_flag)) return;
    double comb = 0.0;
    if (tid < 32) comb = warp_combine<MODE>(partials, static_cast<int>(gridDim.x));
    if (tid == 0) {  // the norm, the scale and the decision constants once per block
        const float n32 = norm_from_combined<MODE>(comb);
        sh_norm = n32;
        sh_scale = dequant_scale(SCHEME, n32, n, a.s);
        sh_dc = make_decide<SCHEME>(n32, a.s, a.u16);
        if (blockIdx.x == 0) {
            hdr->norm = n32;
            if (norm_user) *norm_user = n32;
            if (!(fabsf(n32) < __uint_as_float(kInfBits))) atomicCAS(&hdr->status, 0u, 4u);
        }
    }
    __syncthreads();
    if (!ok) return;
    const float nrm = sh_norm;
    const bool live = nrm > 0.0f && nrm < __uint_as_float(kInfBits);
    const float scale = sh_scale;
    const Decide dc = sh_dc;

    // 4. quantise, sum over the workers and dequantise, two rows per decision.  With fewer
    // column groups than half the threads, each group's row pairs are split P ways and the
    // partial sums (exact integers in fp32, so the order of the additions does not matter)
    // meet in shared memory.
    const int64_t npairs = (n + 1) / 2;
    int64_t P = 1;
    if (ng <= kResThreads / 2) P = min(npairs, static_cast<int64_t>(kResThreads) / ng);
    if (P > 1) {
        for (int64_t e = tid; e < ng * kQCols; e += kResThreads) sh_S[e / kQCols][e % kQCols] = 0.0f;
        __syncthreads();
    }
    for (int64_t u = tid; u < ng * P; u += kResThreads) {
        const uint32_t u32 = static_cast<uint32_t>(u), ng32 = static_cast<uint32_t>(ng);
        const int64_t part = u32 / ng32, gl = u32 - static_cast<uint32_t>(part) * ng32;
        const int64_t g = g0 + gl;
        float S[kQCols];
#pragma unroll
        for (int c = 0; c < kQCols; ++c) S[c] = 0.0f;
        if (live) {
            const uint32_t g32 = static_cast<uint32_t>(g);
            const PhiloxGroup pg = philox_group(g32, a.step_lo, a.step_hi, a.rk);
            const T* col0 = tile + gl * kQCols;
            for (int64_t r0 = 2 * part; r0 < n; r0 += 2 * P) {
                float v[2][kQCols];
                uint32_t aw[2][4];
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    if (r0 + u < n) {
                        const uint4* p = reinterpret_cast<const uint4*>(col0 + (r0 + u) * pitch);
                        unstage<T>(p, p + 1, v[u]);
                    } else {
#pragma unroll
                        for (int c = 0; c < kQCols; ++c) v[u][c] = 0.0f;
                    }
                    const uint4 ra = philox_row(pg, static_cast<uint32_t>(r0 + u) + a.row0,
                                                a.step_lo, a.rk);
                    aw[u][0] = ra.x; aw[u][1] = ra.y; aw[u][2] = ra.z; aw[u][3] = ra.w;
                }
                uint32_t yk[2][kQCols];
                decide_rows<SCHEME, true, 2>(v, dc, a, g32, static_cast<uint32_t>(r0) + a.row0,
                                             aw, yk);
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    if (r0 + u >= n) break;
                    int32_t code[kQCols];
                    accumulate_row<SCHEME>(v[u], yk[u], S, code);
                }
            }
        }
        if (P == 1) {
            store_out(out, nullptr, 0, a.out_dtype, g, d, scale, S);
        } else {
#pragma unroll
            for (int c = 0; c < kQCols; ++c) atomicAdd(&sh_S[gl][c], S[c]);
        }
    }
    if (P > 1) {
        __syncthreads();
        for (int64_t gl = tid; gl < ng; gl += kResThreads) {
            float S[kQCols];
#pragma unroll
            for (int c = 0; c < kQCols; ++c) S[c] = sh_S[gl][c];
            store_out(out, nullptr, 0, a.out_dtype, g0 + gl, d, scale, S);
        }
    }
}

// Signed contribution of a code to the integer sum: L sums the level index; E sums
// 2^(k-1) units of 2^-(s-1) for level index k >= 1.
template <int SCHEME>
__device__ __forceinline__ int32_t code_units(uint32_t k, bool neg) {
    const int32_t u = (SCHEME == kLinear) ? static_cast<int32_t>(k)
                                          : static_cast<int32_t>((1u << k) >> 1);
    return neg ? -u : u;
}

// ------------------------------------------------------------------------------------------
// Step 3 unfused: integer sum of the code matrix over the workers.  Each thread owns 16 bytes
// of every code row (16 int8 or 32 int4 codes).
// ------------------------------------------------------------------------------------------
template <int CODE_BITS, int SCHEME>
__global__ void __launch_bounds__(kThreads)
reduce_codes_kernel(const unsigned char* __restrict__ codes, int64_t n, int64_t d,
                    int64_t row_bytes, int64_t chunks, int32_t* __restrict__ sums) {
    constexpr int K = (CODE_BITS == 8) ? 16 : 32;  // codes per 16-byte chunk
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
    for (int64_t q = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; q < chunks;
         q += stride) {
        int32_t S[K];
#pragma unroll
        for (int k = 0; k < K; ++k) S[k] = 0;
        const unsigned char* base = codes + q * 16;
        int64_t i = 0;
        for (; i < n; i += 4) {
            uint4 w[4];
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (i + u < n) w[u] = __ldg(reinterpret_cast<const uint4*>(base + (i + u) * row_bytes));
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                if (i + u >= n) break;
                const uint32_t word[4] = {w[u].x, w[u].y, w[u].z, w[u].w};
#pragma unroll
                for (int k = 0; k < K; ++k) {
                    int32_t c;
                    if (CODE_BITS == 8)
                        c = static_cast<int32_t>(word[k >> 2] << (24 - 8 * (k & 3))) >> 24;
                    else
                        c = static_cast<int32_t>(word[k >> 3] << (28 - 4 * (k & 7))) >> 28;
                    const bool neg = c < 0;
                    const uint32_t lvl = static_cast<uint32_t>(neg ? -c : c);
                    S[k] += code_units<SCHEME>(lvl, neg);
                }
            }
        }
        const int64_t j0 = q * K;
        GQ_BOUND((q + 1) * 16 <= row_bytes);  // chunks of the code pitch (padding stores nothing)
        if (j0 + K <= d) {
#pragma unroll
            for (int h = 0; h < K / 4; ++h)
                reinterpret_cast<int4*>(sums + j0)[h] = make_int4(S[4 * h], S[4 * h + 1], S[4 * h + 2], S[4 * h + 3]);
        } else {
#pragma unroll
            for (int k = 0; k < K; ++k)
                if (j0 + k < d) sums[j0 + k] = S[k];
        }
    }
}

// Step 4 unfused: out_j = scale * S_j, the sums S int32 or (SUM_I8) int8.
template <int SCHEME, bool SUM_I8>
__global__ void __launch_bounds__(kThreads)
dequantize_kernel(const void* __restrict__ sums_v, const float* __restrict__ norm_ptr,
                  int64_t n, uint32_t s, int64_t d, void* __restrict__ out, int dt) {
    __shared__ float sh_scale;
    const float scale = block_scale<SCHEME>(__ldg(norm_ptr), n, s, &sh_scale);
    const int64_t quads = (d + 3) / 4;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
    const int32_t* sums = static_cast<const int32_t*>(sums_v);
    const int8_t* sums8 = static_cast<const int8_t*>(sums_v);
    for (int64_t q = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; q < quads;
         q += stride) {
        const int64_t j0 = q * 4;
        GQ_BOUND(j0 < d);
        if (j0 + 4 <= d) {
            int4 t;
            if (SUM_I8) {
                const uint32_t w = __ldg(reinterpret_cast<const unsigned int*>(sums8 + j0));
                t = make_int4(static_cast<int8_t>(w), static_cast<int8_t>(w >> 8),
                              static_cast<int8_t>(w >> 16), static_cast<int8_t>(w >> 24));
            } else {
                t = __ldg(reinterpret_cast<const int4*>(sums + j0));
            }
            const float v0 = scale * static_cast<float>(t.x), v1 = scale * static_cast<float>(t.y);
            const float v2 = scale * static_cast<float>(t.z), v3 = scale * static_cast<float>(t.w);
            if (dt == kOutF32)
                reinterpret_cast<float4*>(out)[q] = make_float4(v0, v1, v2, v3);
            else
                reinterpret_cast<uint2*>(out)[q] = make_uint2(pack16(dt, v0, v1), pack16(dt, v2, v3));
        } else {
            for (int64_t j = j0; j < d; ++j)
                store1(out, dt, j, scale * static_cast<float>(SUM_I8 ? static_cast<int32_t>(sums8[j])
                                                                      : __ldg(sums + j)));
        }
    }
}

// Philox check kernel: one call per thread.
static __global__ void philox_kernel(const uint32_t* __restrict__ ck, uint32_t* __restrict__ out,
                              int64_t count) {
    const int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (t >= count) return;
    const uint32_t* p = ck + 6 * t;
    const uint4 r = philox4x32_10(make_uint4(p[0], p[1], p[2], p[3]), p[4], p[5]);
    out[4 * t] = r.x; out[4 * t + 1] = r.y; out[4 * t + 2] = r.z; out[4 * t + 3] = r.w;
}

}  // namespace gq

namespace gq {

// ------------------------------------------------------------------------------------------
// Global-E allreduce with re-rounding at every hop (Global-QSGD: the custom reduction of the
// exponential-dithering allreduce; the extra variance of rounding inside the allreduce; the
// tree allreduce preferred for its fewer reduction steps).  A partial sum stays an extended
// Global-E code: level index k stands for 2^(k-1) units of 2^-(s-1).  One step decodes two
// codes, adds them exactly (int64) and rounds |t| between 2^e and 2^(e+1), e = floor(log2 |t|),
// up with probability (|t| - 2^e) / 2^e, keeping the sign.  The random word of coordinate j in
// stream `sid` (counter word 1; worker indices are below 2^31) is built as for the quantiser:
// high half from Philox(j/8, sid, step), low half from Philox(2^31 + j/8, sid, step).
// ------------------------------------------------------------------------------------------

__device__ __forceinline__ int64_t exp_units_dev(int c) {
    const int k = min(c < 0 ? -c : c, 62);  // valid codes have |k| <= 62
    const int64_t u = k ? (static_cast<int64_t>(1) << (k - 1)) : 0;
    return c < 0 ? -u : u;
}

// The same for |c| <= 30: sign 2^(|c|-1) in 32 bits.
__device__ __forceinline__ int32_t exp_units32(int c) {
    const uint32_t k = static_cast<uint32_t>(c < 0 ? -c : c);
    const int32_t u = static_cast<int32_t>((1u << k) >> 1);  // 0 for k = 0
    return c < 0 ? -u : u;
}

// Lower level index and threshold of |t| units on the extended grid (exact).
__device__ __forceinline__ void exp_split_dev(uint64_t a, uint32_t& lo, uint32_t& T) {
    if (a == 0) {
        lo = 0;
        T = 0;
        return;
    }
    const int e = 63 - __clzll(static_cast<long long>(a));
    const uint64_t frac = a - (static_cast<uint64_t>(1) << e);
    lo = static_cast<uint32_t>(e + 1);
    T = e <= 32 ? static_cast<uint32_t>(frac << (32 - e)) : static_cast<uint32_t>(frac >> (e - 32));
}

struct ExpArgs {
    uint32_t rk[20];  // Philox round keys of the seed
    uint32_t step_lo, step_hi;
};

// The same split for a 32-bit magnitude (|t| < 2^31).
__device__ __forceinline__ void exp_split32(uint32_t a, uint32_t& lo, uint32_t& T) {
    const int e = 31 - __clz(static_cast<int>(a));  // -1 for a = 0
    lo = static_cast<uint32_t>(e + 1);
    T = e > 0 ? (a - (1u << e)) << (32 - e) : 0u;   // 2^32 (a - 2^e) / 2^e, exact; 0 for a <= 1
}

// Re-rounded signed codes of eight sums t[c] (coordinates 8 g8 + c) in stream sid.  TI: int64_t
// for any extended codes, int32_t when every |t| < 2^31 (codes with |k| <= 30).
template <typename TI>
__device__ __forceinline__ void exp_reround8(const TI (&t)[8], uint32_t g8, uint32_t sid,
                                             const ExpArgs& ea, int32_t (&code)[8]) {
    const uint4 ra = philox4x32_10_rk(make_uint4(g8, sid, ea.step_lo, ea.step_hi), ea.rk);
    const uint32_t aw[4] = {ra.x, ra.y, ra.z, ra.w};
    uint32_t lo[8], T[8];
    bool tie = false;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        if (sizeof(TI) == 8)
            exp_split_dev(static_cast<uint64_t>(t[c] < 0 ? -t[c] : t[c]), lo[c], T[c]);
        else
            exp_split32(static_cast<uint32_t>(t[c] < 0 ? -t[c] : t[c]), lo[c], T[c]);
        const uint32_t h = half16(aw, c);
        tie |= h == (T[c] >> 16);
        code[c] = static_cast<int32_t>(lo[c] + (h < (T[c] >> 16) ? 1u : 0u));
    }
    if (tie) {  // the high half equals the threshold's: the low half decides (rare)
        const uint4 rb = philox4x32_10_rk(make_uint4(g8 | 0x80000000u, sid, ea.step_lo, ea.step_hi),
                                          ea.rk);
        const uint32_t bw[4] = {rb.x, rb.y, rb.z, rb.w};
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const uint32_t r = (half16(aw, c) << 16) | half16(bw, c);
            code[c] = static_cast<int32_t>(lo[c] + (r < T[c] ? 1u : 0u));
        }
    }
#pragma unroll
    for (int c = 0; c < 8; ++c)
        if (t[c] < 0) code[c] = -code[c];
}

// Codes with |k| <= kExpTab (every code a quantiser writes, s <= 24) combine through a table in
// shared memory: entry (ka + kExpTab) kExpTabN + (kb + kExpTab) holds the split of the exact sum
// t = units(ka) + units(kb) (|t| <= 2^24): the lower level index, the sign of t (bit 8) and the
// threshold T, computed in the block's prologue with the same integer arithmetic as the split.
constexpr int kExpTab = 24;
constexpr int kExpTabN = 2 * kExpTab + 1;

// Re-rounded signed codes of eight coordinates from their table entries (as exp_reround8).
__device__ __forceinline__ void exp_reround8_tab(const uint2 (&e)[8], uint32_t g8, uint32_t sid,
                                                 const ExpArgs& ea, int32_t (&code)[8]) {
    const uint4 ra = philox4x32_10_rk(make_uint4(g8, sid, ea.step_lo, ea.step_hi), ea.rk);
    const uint32_t aw[4] = {ra.x, ra.y, ra.z, ra.w};
    bool tie = false;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const uint32_t h = half16(aw, c);
        tie |= h == (e[c].y >> 16);
        code[c] = static_cast<int32_t>((e[c].x & 0xFFu) + (h < (e[c].y >> 16) ? 1u : 0u));
    }
    if (tie) {  // the high half equals the threshold's: the low half decides (rare)
        const uint4 rb = philox4x32_10_rk(make_uint4(g8 | 0x80000000u, sid, ea.step_lo, ea.step_hi),
                                          ea.rk);
        const uint32_t bw[4] = {rb.x, rb.y, rb.z, rb.w};
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const uint32_t r = (half16(aw, c) << 16) | half16(bw, c);
            code[c] = static_cast<int32_t>((e[c].x & 0xFFu) + (r < e[c].y ? 1u : 0u));
        }
    }
#pragma unroll
    for (int c = 0; c < 8; ++c)
        if (e[c].x >> 8) code[c] = -code[c];
}

// One step on d coordinates: out = re-round(decode(a) + decode(b)); coordinate j of the buffers
// is coordinate jbase + j of the whole vector (jbase a multiple of 8), which keys its random
// word.  Each thread owns 16 coordinates (one 16-byte load of a and of b, one 16-byte store).
static __global__ void __launch_bounds__(kThreads, 3)
exp_combine_kernel(const int8_t* __restrict__ a, const int8_t* __restrict__ b, int64_t d,
                   int64_t jbase, uint32_t sid, ExpArgs ea, int8_t* __restrict__ out) {
    __shared__ uint2 tab[kExpTabN * kExpTabN];
    for (int i = threadIdx.x; i < kExpTabN * kExpTabN; i += kThreads) {
        const int32_t t = exp_units32(i / kExpTabN - kExpTab) + exp_units32(i % kExpTabN - kExpTab);
        uint32_t lo, T;
        exp_split32(static_cast<uint32_t>(t < 0 ? -t : t), lo, T);
        tab[i] = make_uint2(lo | (t < 0 ? 0x100u : 0u), T);
    }
    __syncthreads();
    const int64_t chunks = (d + 15) / 16;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
    for (int64_t q = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; q < chunks;
         q += stride) {
        const int64_t j0 = q * 16;
        const bool full = j0 + 16 <= d;
        int8_t av[16], bv[16];
        if (full) {
            *reinterpret_cast<uint4*>(av) = __ldg(reinterpret_cast<const uint4*>(a + j0));
            *reinterpret_cast<uint4*>(bv) = __ldg(reinterpret_cast<const uint4*>(b + j0));
        } else {
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                av[c] = j0 + c < d ? a[j0 + c] : 0;
                bv[c] = j0 + c < d ? b[j0 + c] : 0;
            }
        }
        // codes up to |k| = 24 take the table, up to 30 sum in 32 bits, larger in 64 bits
        int32_t mag = 0;  // largest |c| of the 32 codes
#pragma unroll
        for (int c = 0; c < 16; ++c) mag = max(mag, max(abs(int32_t{av[c]}), abs(int32_t{bv[c]})));
        const bool big = mag > 30;
        const bool tabled = mag <= kExpTab;
        int8_t ov[16];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            int32_t code[8];
            if (tabled) {
                uint2 e[8];
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const int i = (av[8 * h + c] + kExpTab) * kExpTabN + (bv[8 * h + c] + kExpTab);
                    GQ_BOUND(i >= 0 && i < kExpTabN * kExpTabN);
                    e[c] = tab[i];
                }
                exp_reround8_tab(e, static_cast<uint32_t>((jbase + j0) / 8 + h), sid, ea, code);
            } else if (!big) {
                int32_t t[8];
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    t[c] = exp_units32(av[8 * h + c]) + exp_units32(bv[8 * h + c]);
                exp_reround8(t, static_cast<uint32_t>((jbase + j0) / 8 + h), sid, ea, code);
            } else {
                int64_t t[8];
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    t[c] = exp_units_dev(av[8 * h + c]) + exp_units_dev(bv[8 * h + c]);
                exp_reround8(t, static_cast<uint32_t>((jbase + j0) / 8 + h), sid, ea, code);
            }
#pragma unroll
            for (int c = 0; c < 8; ++c) ov[8 * h + c] = static_cast<int8_t>(code[c]);
        }
        GQ_BOUND(j0 >= 0 && j0 < d);
        if (full) {
            *reinterpret_cast<uint4*>(out + j0) = *reinterpret_cast<const uint4*>(ov);
        } else {
#pragma unroll
            for (int c = 0; c < 16; ++c)
                if (j0 + c < d) out[j0 + c] = ov[c];
        }
    }
}

// Re-rounded signed code of one sum t at coordinate j in stream sid (one thread, one column).
__device__ __forceinline__ int32_t exp_reround1(int64_t t, int64_t j, uint32_t sid,
                                                const ExpArgs& ea) {
    uint32_t lo, T;
    exp_split_dev(static_cast<uint64_t>(t < 0 ? -t : t), lo, T);
    const uint32_t g8 = static_cast<uint32_t>(j >> 3);
    const int c = static_cast<int>(j & 7);
    const uint4 ra = philox4x32_10_rk(make_uint4(g8, sid, ea.step_lo, ea.step_hi), ea.rk);
    const uint32_t aw[4] = {ra.x, ra.y, ra.z, ra.w};
    const uint32_t h = half16(aw, c);
    uint32_t up = h < (T >> 16) ? 1u : 0u;
    if (h == (T >> 16)) {
        const uint4 rb = philox4x32_10_rk(make_uint4(g8 | 0x80000000u, sid, ea.step_lo, ea.step_hi),
                                          ea.rk);
        const uint32_t bw[4] = {rb.x, rb.y, rb.z, rb.w};
        up = ((h << 16) | half16(bw, c)) < T ? 1u : 0u;
    }
    const int32_t k = static_cast<int32_t>(lo + up);
    return t < 0 ? -k : k;
}

// Dequantise extended Global-E codes (the root of a re-rounding allreduce over n workers):
// out_j = scale * sign 2^(|k|-1) with scale = fp32(N 2^-(s-1) / n), 0 for k = 0.  Each thread
// owns 16 coordinates.
static __global__ void __launch_bounds__(kThreads)
exp_dequantize_kernel(const int8_t* __restrict__ codes, int64_t d,
                      const float* __restrict__ norm_ptr, uint32_t s, int64_t n,
                      void* __restrict__ out, int dt) {
    __shared__ float sh_scale;
    const float scale = block_scale<kExp>(__ldg(norm_ptr), n, s, &sh_scale);
    const int64_t chunks = (d + 15) / 16;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
    for (int64_t q = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; q < chunks;
         q += stride) {
        const int64_t j0 = q * 16;
        GQ_BOUND(j0 < d);
        if (j0 + 16 <= d) {
            const uint4 w = __ldg(reinterpret_cast<const uint4*>(codes + j0));
            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                float v[4];
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    v[c] = scale * static_cast<float>(
                                       exp_units_dev(static_cast<int8_t>(ws[h] >> (8 * c))));
                if (dt == kOutF32)
                    reinterpret_cast<float4*>(static_cast<float*>(out) + j0)[h] =
                        make_float4(v[0], v[1], v[2], v[3]);
                else
                    reinterpret_cast<uint2*>(static_cast<uint16_t*>(out) + j0)[h] =
                        make_uint2(pack16(dt, v[0], v[1]), pack16(dt, v[2], v[3]));
            }
        } else {
            for (int64_t j = j0; j < d; ++j)
                store1(out, dt, j, scale * static_cast<float>(exp_units_dev(codes[j])));
        }
    }
}

constexpr int kExpMaxWorkers = 64;  // rows the one-GPU allreduce simulation holds per column

// Code of worker i at coordinate j from the quantiser's layout (int8, or int4 nibbles).
template <int CODE_BITS>
__device__ __forceinline__ int read_code(const unsigned char* __restrict__ codes, int64_t i,
                                         int64_t j, int64_t pitch) {
    if (CODE_BITS == 8) return static_cast<int>(reinterpret_cast<const int8_t*>(codes)[i * pitch + j]);
    const int byte = codes[i * (pitch / 2) + (j >> 1)];
    const int nib = (j & 1) ? (byte >> 4) : (byte & 0xF);
    return (nib ^ 8) - 8;
}

// The whole Global-E allreduce of the code matrix, one thread per coordinate: tree (ORDER 0:
// level l, row i a multiple of 2^l takes row i + 2^(l-1), stream 2^31 + l 2^24 + i / 2^l) or
// ring (ORDER 1: chunk c = j / chunk, chunk = ceil(d/n) rounded up to a multiple of 16, starts
// at worker c + 1 and visits c + 2, ..., c;
// stream of step h: 2^31 + 2^30 + h 2^12 + c); then out = scale * (root units).
template <int ORDER, int CODE_BITS>
__global__ void __launch_bounds__(kThreads)
exp_allreduce_kernel(const unsigned char* __restrict__ codes, int64_t n, int64_t d, int64_t pitch,
                     ExpArgs ea, const float* __restrict__ norm_ptr, uint32_t s,
                     float* __restrict__ out, int8_t* __restrict__ root_codes) {
    __shared__ float sh_scale;
    const float scale = block_scale<kExp>(__ldg(norm_ptr), n, s, &sh_scale);
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
    const int64_t chunk = ((d + n - 1) / n + 15) / 16 * 16;
    for (int64_t j = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; j < d; j += stride) {
        int32_t root;
        if (ORDER == 0) {
            int64_t u[kExpMaxWorkers];
            int32_t c0 = 0;
            for (int64_t i = 0; i < n; ++i) {
                const int c = read_code<CODE_BITS>(codes, i, j, pitch);
                if (i == 0) c0 = c;
                u[i] = exp_units_dev(c);
            }
            root = c0;
            for (int l = 1; (static_cast<int64_t>(1) << (l - 1)) < n; ++l) {
                const int64_t half = static_cast<int64_t>(1) << (l - 1);
                for (int64_t i = 0; i + half < n; i += 2 * half) {
                    const uint32_t sid = 0x80000000u + (static_cast<uint32_t>(l) << 24) +
                                         static_cast<uint32_t>(i >> l);
                    root = exp_reround1(u[i] + u[i + half], j, sid, ea);
                    u[i] = exp_units_dev(root);
                }
            }
            if (n > 1) {  // row 0 now holds one level
                uint32_t lo, T;
                exp_split_dev(static_cast<uint64_t>(u[0] < 0 ? -u[0] : u[0]), lo, T);
                root = u[0] < 0 ? -static_cast<int32_t>(lo) : static_cast<int32_t>(lo);
            }
        } else {
            const int64_t c = j / chunk;
            int32_t code = read_code<CODE_BITS>(codes, (c + 1) % n, j, pitch);
            for (int64_t h = 1; h < n; ++h) {
                const int64_t t = exp_units_dev(code) +
                                  exp_units_dev(read_code<CODE_BITS>(codes, (c + 1 + h) % n, j, pitch));
                const uint32_t sid = 0xC0000000u + (static_cast<uint32_t>(h) << 12) +
                                     static_cast<uint32_t>(c);
                code = exp_reround1(t, j, sid, ea);
            }
            root = code;
        }
        GQ_BOUND(j >= 0 && j < d);
        out[j] = scale * static_cast<float>(exp_units_dev(root));
        if (root_codes) root_codes[j] = static_cast<int8_t>(root);
    }
}

}  // namespace gq
