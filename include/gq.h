/*
 * gq.h -- C ABI of the GB300 (sm_103a) Global-QSGD compress / aggregate / decompress library.
 *
 * The method: "Global-QSGD: Practical Floatless Quantization for Distributed Learning with
 * Theoretical Guarantees" (Xin, Canini, Richtarik, Horvath; arXiv 2305.18627), cited below as
 * "Global-QSGD".  n workers' gradients x_1..x_n in R^d are held as one n x d matrix X on one GPU
 * (row i = worker i, element (i, j) at i*d + j: the concatenated vector x = [x_1, ..., x_n] of
 * the notation paragraph).  The pipeline:
 *   1. N = ||x||_{q,p}: the q-norm over the workers of every coordinate, then the p-norm of those
 *      d values (notation paragraph); q, p in {2, inf}.
 *   2. every element is normalised, v = |x_ij| / N in fp32, and rounded at random, without bias,
 *      to one of the two adjacent levels of the grid (Global-Q operator):
 *        GQ_LINEAR  Global-L_s, standard dithering, levels m/s, m = 0..s;
 *        GQ_EXP     Global-E_s, exponential dithering, levels 0 and 2^-(s-k), k = 1..s
 *      (the paragraph introducing the two forms of the operator, with its footnote on base 2).
 *      The code is the signed level index c = sign(x) * k.
 *   3. the codes are summed over the workers in integer arithmetic: the allreduce of the
 *      communication hook, on one GPU.  Global-E codes are summed as fixed-point values:
 *      level k counts 2^(k-1) units of 2^-(s-1), so the sum stays exact.
 *   4. the sum is dequantised to the estimate of the mean gradient:
 *        out_j = N * S_j / (n * s)            (Global-L_s)
 *        out_j = N * S_j * 2^-(s-1) / n       (Global-E_s)
 *      (implementation paragraph: quantisation, allreduce, dequantisation).
 * Round up iff r < T, where T = floor(P(up) * 2^32) is computed exactly from v and r is a
 * uniform 32-bit word from Philox4x32-10 (Salmon et al., SC'11) with key (low, high 32 bits of
 * seed): its high 16 bits are half (j mod 8) of the call at counter (j / 8, i, low 32 bits of
 * step, high 32 bits of step), its low 16 bits half (j mod 8) of the call at counter
 * (2^31 + j / 8, i, step); half h is the low half of word h/2 for even h, the high half for odd h.
 *
 * Conventions for every call:
 *   - All buffers are caller-owned device memory (grads, codes, sums, out, norm, ws), 16-byte
 *     aligned (cudaMalloc and PyTorch give 256 bytes).  The library allocates no memory.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).  Every call
 *     is asynchronous on that stream; argument errors are returned synchronously before anything
 *     is enqueued.  Calls on different streams may run concurrently if they use different
 *     workspaces.
 *   - Device-detected conditions (a non-finite norm; a bounded wait of a bulk-copy kernel or of
 *     the single-launch form's grid barrier that gave up) are recorded in the workspace status
 *     word and read with gq_get_status.  On a non-finite norm every output is written as zeros.
 *   - Sizes: n >= 1, 1 <= d < 2^34 (the Philox counter holds j / 8 in 31 bits), n < 2^31.
 *   - Codes: int8 when the code needs more than 4 bits (s > 7), else int4 (two's-complement
 *     nibbles, element 2m in the low nibble of byte m).  Code rows have a pitch of
 *     gq_code_pitch(d) = round_up(d, 32) elements; padding codes are written as 0.
 */
#ifndef GQ_H
#define GQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GQ_OK = 0,
    GQ_ERR_INVALID = 1,     /* null pointer, bad size, bad enum, misaligned buffer */
    GQ_ERR_UNSUPPORTED = 2, /* s outside [1, 127] (Global-L) or [1, 24] (Global-E) */
    GQ_ERR_OVERFLOW = 3,    /* n * s >= 2^24 (L) or n * 2^(s-1) >= 2^24 (E): the code sum
                               would not convert to fp32 exactly */
    GQ_ERR_NONFINITE = 4,   /* device: the norm is NaN or infinite */
    GQ_ERR_TIMEOUT = 5,     /* device: a bounded wait of a bulk-copy kernel gave up (~1 s) */
    GQ_ERR_CUDA = 6,        /* a CUDA runtime call or kernel launch failed */
    GQ_ERR_WORKSPACE = 7    /* workspace null, too small or misaligned */
} gq_status;

/* Element types: gradients are GQ_F32 or GQ_BF16; the dequantised mean (the *_to entry points
 * and the segmented form) may also be GQ_BF16 or GQ_F16. */
typedef enum { GQ_F32 = 0, GQ_BF16 = 1, GQ_F16 = 2 } gq_dtype;

/* Integer type of the code sums that ranks exchange (gq_quantize_sum, gq_dequantize_sums):
 * int32 always holds them; int8 holds them when the total number of workers n satisfies
 * n s <= 127 (Global-L) or n 2^(s-1) <= 127 (Global-E), and then the allreduce moves one byte
 * per coordinate, a quarter of an fp32 gradient's. */
typedef enum { GQ_SUM_I32 = 0, GQ_SUM_I8 = 1 } gq_sum_type;

typedef enum {
    GQ_LINEAR = 0, /* Global-L_s, standard dithering */
    GQ_EXP = 1     /* Global-E_s, exponential dithering */
} gq_scheme;

/*
 * Rounding mode, added to the scheme argument of any call (GQ_LINEAR | GQ_ROUND_U16): the
 * 16-bit-uniform mode.  The pages require an unbiased random rounding and fix no random source;
 * by default the decision is exact (round up iff r < T, r the full 32-bit word).  In this mode
 * element (i, j) rounds up iff H < F, where H is the high 16 bits of its word r and F a 16-bit
 * fraction of its grid position computed without a division:
 *   Global-L_s: P16 = |x| fp32(s / N) 2^16 rounded to the nearest integer, ties to the odd one,
 *               at most s 2^16; lower level P16 >> 16, F = P16 & 0xFFFF;
 *   Global-E_s: w = min(fp32(|x| fp32(1 / N)), 1); for w >= 2^-(s-1) lower level s + e with
 *               2^e <= w < 2^(e+1) and F the top 16 of w's 23 fraction bits; below, P16 =
 *               |x| fp32(1 / N) 2^(s-1) 2^16 rounded as for L, lower level P16 >> 16,
 *               F = P16 & 0xFFFF.
 * P(up) = F / 2^16, so the estimate's bias is below 2^-16 + 2^-22 of a level spacing per
 * element.  A NaN element gets code 0; for a norm outside [2^-100, 2^100] the decision is the
 * exact mode's.  Codes, sums and outputs have the same layout; gq_reduce_codes and the
 * dequantising calls ignore the flag.  No counterpart in the paper beyond its unbiased rounding:
 * an option of this library.
 */
#define GQ_ROUND_U16 16

/* Norm orders for q and p. */
#define GQ_NORM_INF 0
#define GQ_NORM_L2 2

/* Version of this ABI (incremented on incompatible change). */
int gq_abi_version(void);

/* Bytes of workspace the norm step needs for an n x d problem (a small constant today,
 * 36,096 bytes).  The workspace holds the device status word, the block partials of the norm,
 * a completion ticket and the last norm, the grid-barrier words of the single-launch form of
 * gq_allreduce_mean, and per-segment tickets, norms and dequantisation scales for
 * gq_allreduce_mean_segments. */
size_t gq_workspace_bytes(int64_t n, int64_t d);

/* Zero a freshly allocated workspace (enqueued on `stream`).  Required once before its first
 * use; every later call leaves the ticket at zero and the status word sticky. */
gq_status gq_workspace_init(void *ws, size_t ws_bytes, void *stream);

/* 4 or 8: bits per stored code for this scheme and s; 0 if s is unsupported. */
int gq_code_bits(int scheme, int s);

/* Kernel launches of one gq_allreduce_mean call on the current device for an n x d matrix of
 * dtype, with (with_codes != 0) or without a code output: 1 for the single-launch form, 2 for
 * the norm pass + quantise pass; 0 for invalid sizes.  (16-byte aligned grads assumed.) */
int gq_fused_launches(int dtype, int64_t n, int64_t d, int with_codes);

/* Row pitch of the code matrix in elements: round_up(d, 32); 0 if d < 1. */
int64_t gq_code_pitch(int64_t d);

/* Bytes of the n x pitch code matrix: n * gq_code_pitch(d) * gq_code_bits / 8; 0 if invalid. */
size_t gq_code_bytes(int scheme, int s, int64_t n, int64_t d);

/*
 * Step 1: the global norm N = ||x||_{q,p} (Global-QSGD, notation paragraph) of the n x d
 * gradient matrix `grads` (dtype GQ_F32 or GQ_BF16), written as fp32 to *norm_dev.
 * q, p: GQ_NORM_L2 or GQ_NORM_INF.  One kernel: a grid-wide pass with a fixed-order block
 * combine (deterministic on a given GPU).  The l2 forms are accurate to ~1e-7 relative over the
 * whole fp32 range (sums of squares are carried in fp32 with a per-thread power-of-two scale and
 * compensation, combined in fp64).  A NaN or infinite element makes the norm non-finite and
 * sets GQ_ERR_NONFINITE in the workspace status.
 */
gq_status gq_global_norm(const void *grads, int dtype, int64_t n, int64_t d, int q, int p,
                         float *norm_dev, void *ws, size_t ws_bytes, void *stream);

/*
 * Step 2: quantise every element to its signed level-index code (Global-QSGD, Global-Q
 * operator and the two level grids), using the fp32 norm at *norm_dev (device memory; a norm
 * below some |x_ij| saturates that element at level s).  `codes` receives the n x pitch code
 * matrix (gq_code_bytes bytes).  NaN elements get code 0.  A norm of 0 gives all-zero codes; a
 * non-finite norm gives all-zero codes (and no status: this call has no workspace).
 * seed and step key the Philox stream (see the file comment).
 */
gq_status gq_quantize(const void *grads, int dtype, int64_t n, int64_t d, const float *norm_dev,
                      int scheme, int s, uint64_t seed, uint64_t step, void *codes,
                      void *stream);

/*
 * gq_quantize with a workspace (ws, ws_bytes as for gq_allreduce_mean; caller-owned, 16-byte
 * aligned, at least gq_workspace_bytes(n, d) bytes, else GQ_ERR_WORKSPACE): large problems with
 * 16-byte aligned rows take the bulk-copy kernel, whose bounded waits report GQ_ERR_TIMEOUT in
 * the workspace's status word.  ws NULL is gq_quantize; the codes are bit-identical either way.
 * Calls that share a workspace must not overlap on the GPU.
 */
gq_status gq_quantize_ws(const void *grads, int dtype, int64_t n, int64_t d,
                         const float *norm_dev, int scheme, int s, uint64_t seed, uint64_t step,
                         void *codes, void *ws, size_t ws_bytes, void *stream);

/*
 * Step 3: sum the code matrix over the n workers into int32 sums[d] (the allreduce reduction
 * of the communication hook: the native integer sum for Global-L; for Global-E each level index
 * k is summed as 2^(k-1) units of 2^-(s-1)).  Exact.
 */
gq_status gq_reduce_codes(const void *codes, int scheme, int s, int64_t n, int64_t d,
                          int32_t *sum_dev, void *stream);

/*
 * Step 4: dequantise the sums to the mean-gradient estimate out[d] (fp32):
 * out_j = fp32(scale * S_j) with scale = fp32(N / (n s)) (L) or fp32(N 2^-(s-1) / n) (E), the
 * scale computed in fp64 from the fp32 norm at *norm_dev.  |out_j - exact| <= 2^-23 |out_j|.
 * A non-finite norm gives all zeros.
 */
gq_status gq_dequantize(const int32_t *sum_dev, const float *norm_dev, int scheme, int s,
                        int64_t n, int64_t d, float *out_dev, void *stream);

/*
 * gq_dequantize with the output type out_dtype (GQ_F32, GQ_BF16 or GQ_F16): the fp32 value above
 * rounded to nearest even, so a 16-bit output adds at most half a unit in its last place (fp16:
 * magnitudes past 65504 become infinite, as IEEE rounding gives).  out_dev: d elements of that
 * type, 16-byte aligned.  Any other out_dtype: GQ_ERR_INVALID.
 */
gq_status gq_dequantize_to(const int32_t *sum_dev, const float *norm_dev, int scheme, int s,
                           int64_t n, int64_t d, void *out_dev, int out_dtype, void *stream);

/*
 * gq_dequantize_to with the sums given as sum_type (GQ_SUM_I32 or GQ_SUM_I8, d elements, 16-byte
 * aligned).  GQ_SUM_I8 needs n s <= 127 (L) or n 2^(s-1) <= 127 (E), else GQ_ERR_OVERFLOW.
 */
gq_status gq_dequantize_sums(const void *sum_dev, int sum_type, const float *norm_dev, int scheme,
                             int s, int64_t n, int64_t d, void *out_dev, int out_dtype,
                             void *stream);

/*
 * Steps 1-4 fused: the norm pass, then one pass that quantises, sums over the workers in
 * registers and dequantises, so codes and sums never touch memory.  Traffic: X is read twice,
 * out written once.  norm_dev (nullable) receives the fp32 norm; codes (nullable) receives the
 * code matrix as gq_quantize would write it.  Bit-identical to gq_global_norm + gq_quantize +
 * gq_reduce_codes + gq_dequantize on the same stream.
 *
 * Small problems take one launch instead (gq_fused_launches says which): when codes is NULL,
 * the rows are 16-byte aligned (d a multiple of 4 for fp32, 8 for bf16) and the matrix fits in
 * the GPU's shared memory (n * 8 * ceil(ceil(d / 8) / SMs) * element bytes <= 204,800: about
 * 30 MB on 152 SMs), each SM holds its slice of columns on chip, the blocks meet at a grid
 * barrier (cooperative launch; the wait is bounded and reports GQ_ERR_TIMEOUT) to combine the
 * norm, and X is read once.  Decisions, random words and outputs are the same; for the
 * (inf, inf) and (2, inf) norms (maxima) the norm is bit-identical too, while the (2, 2) and
 * (inf, 2) norms are sums that the single launch splits differently, so their last bits may
 * differ from gq_global_norm's (both within its error bound): the outputs are then exactly
 * those of gq_allreduce_mean_with_norm given the norm written to norm_dev.  Calls that share a
 * workspace must not overlap on the GPU (they share its completion ticket and barrier words).
 */
gq_status gq_allreduce_mean(const void *grads, int dtype, int64_t n, int64_t d, int q, int p,
                            int scheme, int s, uint64_t seed, uint64_t step, float *out_dev,
                            float *norm_dev, void *codes, void *ws, size_t ws_bytes,
                            void *stream);

/*
 * gq_allreduce_mean with the output type out_dtype (GQ_F32, GQ_BF16 or GQ_F16), rounded as in
 * gq_dequantize_to; a 16-bit output halves the bytes written.
 */
gq_status gq_allreduce_mean_to(const void *grads, int dtype, int64_t n, int64_t d, int q, int p,
                               int scheme, int s, uint64_t seed, uint64_t step, void *out_dev,
                               int out_dtype, float *norm_dev, void *codes, void *ws,
                               size_t ws_bytes, void *stream);

/*
 * Steps 2-4 fused with a norm supplied in device memory (*norm_dev), e.g. one agreed on by a
 * separate scalar collective.  Same outputs as gq_quantize + gq_reduce_codes + gq_dequantize.
 * codes is nullable.
 */
gq_status gq_allreduce_mean_with_norm(const void *grads, int dtype, int64_t n, int64_t d,
                                      const float *norm_dev, int scheme, int s, uint64_t seed,
                                      uint64_t step, float *out_dev, void *codes, void *stream);

/*
 * gq_allreduce_mean_with_norm with a workspace (ws, ws_bytes as for gq_allreduce_mean; the
 * caller owns it; 16-byte aligned, at least gq_workspace_bytes(n, d) bytes, else
 * GQ_ERR_WORKSPACE): large problems with 16-byte aligned rows then take the bulk-copy quantise
 * kernel, whose bounded waits report GQ_ERR_TIMEOUT in the workspace's status word (read by
 * gq_get_status).  ws NULL is gq_allreduce_mean_with_norm.  Outputs are bit-identical to it:
 * the norm is not trusted (|x| above it saturates, a NaN element gives code 0).  Calls that
 * share a workspace must not overlap on the GPU.
 */
gq_status gq_allreduce_mean_with_norm_ws(const void *grads, int dtype, int64_t n, int64_t d,
                                         const float *norm_dev, int scheme, int s, uint64_t seed,
                                         uint64_t step, float *out_dev, void *codes, void *ws,
                                         size_t ws_bytes, void *stream);

/*
 * Global-E allreduce with re-rounding at every hop (Global-QSGD: the custom reduction the
 * implementation paragraph uses for exponential dithering; the extra variance of "stochastic
 * rounding during AllReduce" counted in the theta worked example; the tree allreduce of the
 * performance model, chosen for its fewer reduction steps).  A partial sum stays an extended
 * Global-E code: level index k stands for 2^(k-1) units of 2^-(s-1), k = 0 for 0.  One step
 * decodes two codes, adds them exactly and rounds |t| between 2^e and 2^(e+1) (e = floor(log2
 * |t|)), up with probability (|t| - 2^e) / 2^e, keeping the sign: unbiased.  Random word of
 * coordinate j in stream `stream_id`: as for gq_quantize with the worker index replaced by the
 * stream identifier (counter word 1), so every step has its own independent stream.
 */
#define GQ_ORDER_TREE 0
#define GQ_ORDER_RING 1

/* Stream identifier of the tree step at level `level` (1-based) that combines into node m:
 * 2^31 + level 2^24 + m.  Of ring step h (1-based) of chunk c: 2^31 + 2^30 + h 2^12 + c. */
uint32_t gq_exp_tree_stream(int level, int64_t m);
uint32_t gq_exp_ring_stream(int64_t h, int64_t c);

/*
 * One reduction step on d coordinates: out[j] = re-round(decode(a[j]) + decode(b[j])).  a, b,
 * out: int8 extended Global-E codes in device memory (16-byte aligned), |k| <= 62 on input (the
 * result for larger codes is unspecified).  Element j is coordinate j0 + j of the whole vector
 * (its random word is that coordinate's); j0 >= 0 is a multiple of 8 (a ring chunk's start).
 * d >= 1.
 */
gq_status gq_exp_combine(const int8_t *a, const int8_t *b, int64_t d, int64_t j0, uint64_t seed,
                         uint64_t step, uint32_t stream_id, int8_t *out, void *stream);

/*
 * The whole Global-E allreduce of the n x pitch code matrix written by gq_quantize (Global-E_s,
 * int4 or int8 by s), simulated on one GPU, then dequantised: out_j = N * R_j * 2^-(s-1) / n
 * with R_j the reduced value in units (fp32, exact scale as gq_dequantize) from the fp32 norm at
 * *norm_dev.  order GQ_ORDER_TREE: level l = 1, 2, ...: row i (a multiple of 2^l) takes
 * re-round(row i + row i + 2^(l-1)) when that row exists.  GQ_ORDER_RING: the coordinates form n
 * chunks of ceil(d/n); chunk c starts at worker c + 1 and adds workers c + 2, ..., c (mod n),
 * re-rounding after each step (reduce-scatter; the allgather only copies).  root_codes
 * (nullable, int8 x d) receives the reduced codes.  1 <= n <= 64; s and n as for gq_quantize
 * (n 2^(s-1) < 2^24, so every partial sum stays below 2^24 units).
 */
gq_status gq_exp_allreduce(const void *codes, int s, int64_t n, int64_t d, int order,
                           const float *norm_dev, uint64_t seed, uint64_t step, float *out_dev,
                           int8_t *root_codes, void *stream);

/*
 * gq_allreduce_mean without a workspace argument, for callers that cannot allocate device
 * memory where they need the allreduce (for example code running inside a framework's caching
 * allocator or communication hook, which may not call back into the allocator, or a process
 * whose device memory is planned in full ahead of time).  The paper has no counterpart to this
 * call; it exists for those callers only.
 *
 * Same arguments, kernels and results as gq_allreduce_mean minus ws / ws_bytes (the single
 * launch for small problems without codes, else the norm pass and the same quantise kernel).
 * Its scratch (status word, completion ticket, norm, the single launch's barrier word and up to
 * 1,024 per-block partials: 8,448 bytes) lives in a fixed array in the library's device memory,
 * which every GPU that loads the library holds until the process exits.  Nothing is allocated:
 * no cudaMalloc, cudaFree or allocating library call.  The first call on a device looks up that
 * array's device address (cudaGetSymbolAddress) with the device current and keeps it for the
 * process: make that first call before any stream capture, and do not call it again on a device
 * after cudaDeviceReset (the address kept would be stale).  A problem whose norm step would
 * launch more than gq_noalloc_max_blocks() = 1,024 blocks (gq_norm_blocks tells) is refused with
 * GQ_ERR_WORKSPACE; on GB300 the norm step launches at most 608.  Every call shares the one array:
 * each call clears its header first, and calls that overlap on the GPU (other streams, other host
 * threads) race, so serialise them.  A non-finite norm gives all-zero outputs; there is no status
 * word to read, so test the norm written to norm_dev (nullable) instead.
 */
gq_status gq_allreduce_mean_noalloc(const void *grads, int dtype, int64_t n, int64_t d, int q,
                                    int p, int scheme, int s, uint64_t seed, uint64_t step,
                                    float *out_dev, float *norm_dev, void *codes, void *stream);

/* Blocks the norm step launches for an n x d matrix of dtype under norm orders (q, p) on the
 * current device (gq_global_norm, gq_allreduce_mean and its allocation-free form all use this
 * count); 0 for invalid arguments.  And the most that gq_allreduce_mean_noalloc accepts (the
 * partials its fixed scratch holds: 1,024).  No counterpart in the paper: sizing queries. */
int64_t gq_norm_blocks(int dtype, int64_t n, int64_t d, int q, int p);
int64_t gq_noalloc_max_blocks(void);

/*
 * Segmented form (per layer or per gradient bucket, as the DDP hook of Global-QSGD's
 * implementation paragraph applies the method bucket by bucket): nseg independent problems, each
 * its own row-major n x d[l] matrix at grads[l] (device, 16-byte aligned, dtype as gq_quantize)
 * with its own norm ||x_l||_{q,p}, quantised, summed over the n workers and dequantised into
 * out[l] (device, d[l] elements of out_dtype as in gq_dequantize_to, 16-byte aligned).
 * grads, d and out are HOST arrays of nseg
 * entries.  Segment l draws its random words with step (step << 16) | l, so it equals
 * gq_allreduce_mean(grads[l], ..., step * 65536 + l) bit for bit; the DDP hook uses the same
 * numbering for its buckets.  norms_dev (nullable, device) receives the nseg fp32 norms.  Two
 * launches per 256 segments, whatever their sizes.  1 <= nseg <= 65536, step < 2^48; other
 * errors as gq_allreduce_mean.  Codes are not written.
 */
gq_status gq_allreduce_mean_segments(int64_t nseg, const void *const *grads, const int64_t *d,
                                     int dtype, int64_t n, int q, int p, int scheme, int s,
                                     uint64_t seed, uint64_t step, void *const *out,
                                     int out_dtype, float *norms_dev, void *ws, size_t ws_bytes,
                                     void *stream);

/*
 * The global norm when the workers sit on different GPUs.  gq_norm_partial writes this rank's
 * share of N = ||x||_{q,p} over its m x d rows as one fp64 value at *part_dev: the sum of squares
 * (q = p = 2) or the largest magnitude (q = p = inf).  Combine the ranks' values with a sum or a
 * maximum allreduce, then gq_norm_finish turns the combined value into the fp32 norm at *norm_dev
 * (the square root of the sum, or the maximum itself, rounded to fp32).  For q = p = inf this is
 * exactly gq_global_norm of the stacked rows; for q = p = 2 it agrees to the l2 forms' relative
 * 1e-6.  The mixed orders need a d-vector exchange and are refused with GQ_ERR_UNSUPPORTED.  The
 * workspace is used as by gq_global_norm.
 */
gq_status gq_norm_partial(const void *grads, int dtype, int64_t m, int64_t d, int q, int p,
                          double *part_dev, void *ws, size_t ws_bytes, void *stream);
gq_status gq_norm_finish(const double *part_dev, int q, int p, float *norm_dev, void *stream);

/*
 * One rank's share of the allreduce when the workers sit on different GPUs (the communication
 * hook of Global-QSGD's implementation paragraph: quantise, allreduce, dequantise per gradient
 * bucket).  Quantises the m x d rows at grads, whose workers are worker0 .. worker0 + m - 1 (the
 * worker index keys the random words, as row i does in gq_quantize), with the fp32 global norm
 * at *norm_dev, and writes the integer sum of their codes (Global-L: the level indices; Global-E:
 * 2^(k-1) units of 2^-(s-1)) to sum_dev[d] as sum_type (int32, or int8 when m s <= 127 for L,
 * m 2^(s-1) <= 127 for E, else GQ_ERR_OVERFLOW; the caller keeps the total over ranks in range
 * too).  Summing these over all ranks (an integer allreduce, exact) and calling
 * gq_dequantize_sums with n = the total number of workers gives the same result as
 * gq_allreduce_mean on the stacked matrix with the same norm.  ws (nullable; as for
 * gq_global_norm) lets a large problem take the bulk-copy kernel, whose bounded waits report
 * GQ_ERR_TIMEOUT in its status word.  Errors as gq_quantize; worker0 >= 0 and
 * worker0 + m <= 2^31.
 */
gq_status gq_quantize_sum(const void *grads, int dtype, int64_t m, int64_t d, int64_t worker0,
                          const float *norm_dev, int scheme, int s, uint64_t seed, uint64_t step,
                          void *sum_dev, int sum_type, void *ws, size_t ws_bytes, void *stream);

/*
 * Philox4x32-10 on the device, for checking the random stream: `count` calls, input
 * ctr_key[6*c .. 6*c+5] = counter words 0..3 then key words 0..1, output out[4*c .. 4*c+3].
 */
gq_status gq_philox4x32_10(const uint32_t *ctr_key_dev, uint32_t *out_dev, int64_t count,
                           void *stream);

/* Synchronise `stream`, read the workspace status word, clear it, and return it (GQ_OK if no
 * device-detected condition occurred since the last read). */
gq_status gq_get_status(void *ws, void *stream);

/* Static string naming a status value. */
const char *gq_status_string(int status);

/* Bounds checks of a debug build (the library compiled with -DGQ_DEBUG; the stand-in for a
 * memory checker): every kernel store and bulk copy is checked against the logical extent of its
 * buffer (d, the code pitch, the partials, the matrix), and a failed check records its source
 * line instead of trapping.  Returns -1 in a normal build; in a debug build synchronises the
 * device, returns and clears the first recorded line (0: none; -2: the word could not be read).
 * No counterpart in the paper. */
int gq_debug_status(void);

/*
 * One rank's codes for a multi-GPU allreduce that moves codes rather than sums (the Global-E
 * re-rounding allreduce of Global-QSGD's performance-model paragraph): the m x d rows at grads,
 * whose workers are worker0 .. worker0 + m - 1, quantised as gq_quantize would quantise those
 * rows of the stacked matrix, written as m x gq_code_pitch(d) codes of code_bits (8, or 4 when
 * s <= 7; int8 whatever s is, for gq_exp_combine).  ws (nullable) as for gq_quantize_sum.
 */
gq_status gq_quantize_codes(const void *grads, int dtype, int64_t m, int64_t d, int64_t worker0,
                            const float *norm_dev, int scheme, int s, uint64_t seed,
                            uint64_t step, void *codes, int code_bits, void *ws, size_t ws_bytes,
                            void *stream);

/*
 * Dequantise d extended Global-E codes (int8, |k| <= 62, 16-byte aligned; the result of a
 * re-rounding allreduce over n workers) into out (d elements of out_dtype):
 * out_j = fp32(N 2^-(s-1) / n) * sign 2^(|k|-1), 0 for k = 0, N the fp32 norm at *norm_dev.
 */
gq_status gq_exp_dequantize(const int8_t *codes, int64_t d, const float *norm_dev, int s,
                            int64_t n, void *out_dev, int out_dtype, void *stream);

/*
 * Self-test of the bounded waits of the bulk-copy kernels: one GPU thread waits on an mbarrier
 * that nothing completes, gives up after limit_ns nanoseconds (1,000 .. 4e9) of global time and
 * records GQ_ERR_TIMEOUT in the workspace status word (read it with gq_get_status), exactly as a
 * quantise kernel whose copies never arrive would.  *elapsed_dev (device, 8 bytes) receives the
 * time waited.  The kernel then returns normally: the context stays usable.
 */
gq_status gq_selftest_wait_timeout(void *ws, size_t ws_bytes, uint64_t limit_ns,
                                   unsigned long long *elapsed_dev, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* GQ_H */
