/*
 * jetq: block-scaled FP8 (E4M3) quantize-and-GEMM for one GB300 (sm_103a).
 *
 * One quantizer and one set of GEMMs serve both RL rollout and RL training, so
 * the rollout forward and the training forward see bit-identical quantized
 * operands and return bit-identical outputs ("unified precision flow",
 * Jet-RL, section 4.1 of the papercache summary; on-policy weight sync, SkyRL
 * FP8 post, "On-Policy FP8 weight sync").
 *
 * Conventions for every entry point:
 *  - All pointers are DEVICE pointers, allocated and owned by the caller.  The
 *    library allocates nothing, frees nothing and keeps no pointer after the
 *    call returns.
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = the legacy default
 *    stream) and the call returns without synchronizing.
 *  - Arguments are validated on the host before anything is launched; a
 *    failed check returns an error code and launches nothing.  Outputs are
 *    undefined after a JETQ_ERR_CUDA return.
 *  - Every wait inside a kernel is bounded.  A kernel that gives up records
 *    the fact in a device error word, which jetq_check_device_error() reads.
 *  - Codes are E4M3 bytes (OCP "FN" variant: bias 7, no infinities, largest
 *    finite value 448).  BF16 inputs are uint16_t bit patterns.
 *  - Row strides (ld*) are in elements of the pointed-to type and must keep
 *    every row 16-byte aligned; base pointers must be 16-byte aligned.
 *  - C (channels), D (output features) are multiples of 128.  N (tokens) is
 *    any value >= 0.
 *
 * Quantization readings (the pages are silent or garbled on these; the
 * oracle uses the same ones):
 *  - FP32-scale recipe: S = fl32(amax / 448); q = E4M3_rne_satfinite(fl32(x / S)).
 *    An all-zero group has S = 0 and codes 0x00.
 *  - MXFP8 recipe: e = smallest integer with amax <= 448 * 2^e, clamped to
 *    [-127, 127]; scale byte = e + 127 (E8M0); q = E4M3_rne_satfinite(x * 2^-e).
 *    An all-zero block has scale byte 127 and codes 0x00.
 */
#ifndef JETQ_H
#define JETQ_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define JETQ_API __attribute__((visibility("default")))
#else
#define JETQ_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    JETQ_OK = 0,
    JETQ_ERR_INVALID_ARG = 1,       /* null pointer, negative size, bad enum */
    JETQ_ERR_UNSUPPORTED_SHAPE = 2, /* C or D not a multiple of 128, ld too small */
    JETQ_ERR_MISALIGNED = 3,        /* pointer or row stride not 16-byte aligned */
    JETQ_ERR_ARCH = 4,              /* current device is not compute capability 10.3 */
    JETQ_ERR_CUDA = 5,              /* a CUDA runtime call or a launch failed */
    JETQ_ERR_TIMEOUT = 6            /* a kernel gave up a bounded wait (device error word) */
} jetq_status;

typedef enum {
    JETQ_RECIPE_BLOCK128 = 0,     /* 1x128 activation groups, 128x128 weight blocks, FP32 scales */
    JETQ_RECIPE_MXFP8 = 1,        /* 1x32 blocks, E8M0 power-of-two scales rounded up */
    JETQ_RECIPE_BLOCK128_POW2 = 2 /* 1x128 groups, 128x128 blocks, scales constrained to powers of
                                     two (E8M0 atoms, each 32-element sub-block byte carrying its
                                     group's exponent); runs the block-scaled MMA like MXFP8 */
} jetq_recipe;

typedef enum {
    JETQ_PATH_AUTO = 0,   /* DECODE when N <= 256 tokens, else TRAIN */
    JETQ_PATH_TRAIN = 1,  /* wide tiles for large N */
    JETQ_PATH_DECODE = 2  /* few-token kernels that stream the weight: 1-64 tokens against >= 32
                             weight row blocks run with weight rows as the MMA's M; otherwise
                             narrow 32-row weight tiles; same per-element arithmetic as TRAIN */
} jetq_path;

typedef enum {
    JETQ_GEMM_FPROP = 0,
    JETQ_GEMM_DGRAD = 1,
    JETQ_GEMM_WGRAD = 2
} jetq_gemm_kind;

typedef enum {
    JETQ_OUT_F32 = 0,
    JETQ_OUT_BF16 = 1 /* round-to-nearest-even of the FP32 result */
} jetq_out_dtype;

/* Human-readable name of a status code (static storage). */
JETQ_API const char *jetq_status_string(jetq_status status);

/* Library version, major * 10000 + minor * 100 + patch. */
JETQ_API int jetq_version(void);

/*
 * Synchronize `stream`, then read and clear the device error word of every
 * kernel family.  Returns JETQ_ERR_TIMEOUT if any kernel gave up a bounded
 * wait since the last call, JETQ_ERR_CUDA if the synchronization failed.
 * The read and the clear are separate copies: call it when no jetq kernel is
 * running on another stream, or a word set in between would be lost.
 */
JETQ_API jetq_status jetq_check_device_error(void *stream);

/*
 * Diagnostic for the bounded waits (the pages have no counterpart: their
 * kernels are not shown waiting at all).  Launches one CTA whose two waiters
 * wait on shared-memory mbarriers that nothing ever completes, using the same
 * wait primitive as the GEMM kernels: waiter 0 gives up after limit_ns of wall
 * clock, raises the CTA's abort flag and records a timeout in the device error
 * word; waiter 1 (limit 8 * limit_ns) gives up as soon as it sees the abort
 * flag.  Each waiter writes the nanoseconds it waited to elapsed_ns[0..1]
 * (caller-owned device memory, two int64).  The kernel faults nothing and
 * leaves the context usable; jetq_check_device_error() afterwards returns
 * JETQ_ERR_TIMEOUT once and clears the word.
 * Limits: 1 ms <= limit_ns <= 1 s; elapsed_ns 8-byte aligned.
 */
JETQ_API jetq_status jetq_selftest_bounded_wait(uint64_t limit_ns, int64_t *elapsed_ns, void *stream);

/* ======================================================================== */
/* Layouts                                                                  */
/* ======================================================================== */
/*
 * Row-wise FP32-scale copy of an [R x K] tensor (groups of 128 along K):
 *   codes  q[r * K + k]                        (dense, K-major)
 *   scales s[(k / 128) * R + r]                (group-major, rows contiguous)
 *
 * Column-wise FP32-scale copy of an [N x C] tensor (groups of 128 along N,
 * never crossing a segment bound), stored transposed:
 *   codes  qc[c * ldqc + p]    p = position in the column copy
 *   scales sc[(p / 128) * C + c]
 * Segment e (tokens off[e] .. off[e+1]-1) starts at column-copy position
 * pad[e] = sum_{j<e} ceil(n_j / 128) * 128, so every 128-group of positions
 * belongs to one segment.  Positions of a segment's last, partial group past
 * its tokens hold code 0x00.  Positions from pad[nseg] up to the capacity are
 * not written.  Capacity: jetq_colcopy_capacity(N, nseg).
 *
 * 128x128 weight copy of W [D x C]:
 *   codes  q[d * C + c],  scales s[(d / 128) * (C / 128) + c / 128]
 *   transposed copy (for DGrad): qT[c * D + d],  sT[(c / 128) * (D / 128) + d / 128]
 *
 * MXFP8 scale bytes of a K-major payload with R rows and K columns (one byte
 * per row and 32 columns, K a multiple of 128) are kept in 512-byte atoms,
 * one per 128-row band and 128-column K-block: the unit the tensor core's
 * block-scaled MMA reads (32 lanes x 16 bytes; lane r % 32 holds rows
 * r % 32 + 32 * i, i = 0..3, four K sub-blocks each):
 *   RB = ceil(R / 128) bands;  j = k / 32 (K sub-block), kb = j / 4
 *   byte(r, j) at (kb * RB + r / 128) * 512 + (r % 32) * 16 + ((r % 128) / 32) * 4 + j % 4
 *   size = RB * (K / 128) * 512 bytes (jetq_mx_scale_bytes)
 * Bytes for rows >= R inside a band are not written.
 */

/* Capacity (positions, a multiple of 128) a column copy of N tokens in nseg segments needs. */
JETQ_API int64_t jetq_colcopy_capacity(int64_t n, int nseg);

/* Bytes of the MX scale-atom array for a K-major payload of `rows` x `k`. */
JETQ_API int64_t jetq_mx_scale_bytes(int64_t rows, int64_t k);

/* ======================================================================== */
/* Quantizers                                                               */
/* ======================================================================== */

/*
 * Activation / gradient quantizer, FP32-scale recipe, one pass over X.
 * Jet-RL (paper-graph-ui explainer), "GEMM Quantization": 1x128 per-group
 * activation scales S = max|X[n, c:c+128]| / 448; papercache summary 4.2: the
 * backward GEMMs need 1x128 and 128x1 quantizations of the same tensor, which
 * are fused; Miles Blackwell post, MXFP8 section: both copies are quantized
 * from full precision.
 *
 *   x       BF16 [n x c], row stride ldx (elements, multiple of 8)
 *   q_row   codes [n x c] and s_row [c/128 x n]        (nullable pair: skip)
 *   q_col   codes [c x ldq_col] and s_col [ldq_col/128 x c] (nullable pair: skip);
 *           ldq_col >= jetq_colcopy_capacity(n, nseg), a multiple of 128
 *   seg_offsets  device int64 [nseg + 1], 0 = off[0] <= ... <= off[nseg] = n;
 *           NULL means one segment [0, n) (nseg is then ignored)
 * Row-wise groups ignore segments.  Offsets are read on the device; values
 * outside [0, n] are clamped.  n == 0 is a no-op.
 */
JETQ_API jetq_status jetq_quant_act_1x128(const uint16_t *x, int64_t n, int64_t c, int64_t ldx,
                                 uint8_t *q_row, float *s_row,
                                 uint8_t *q_col, float *s_col, int64_t ldq_col,
                                 const int64_t *seg_offsets, int nseg, void *stream);

/*
 * Activation quantizer fused with its producer: RMSNorm.
 * Jet-RL explainer, "The Three GEMM Operations and Their Quantization
 * Configuration" (the activation quantizer is fused with the preceding
 * operator, typically RMSNorm) and "Implementation Details: Frameworks,
 * Kernels, and Weight Synchronization" (fused_rmsnorm_quantize: RMSNorm, then
 * 1x128 quantization, with no BF16 write in between).
 *
 * The quantized tensor is y = BF16(fl32(fl32(x * rstd[r]) * w[col])) with
 * rstd[r] = 1 / sqrt(fl32(sum_sq(x[r]) / c) + eps), every operation a
 * correctly rounded binary32 one and the sum of squares taken in a fixed
 * order: each 128-column group left to right by fma, then the group sums
 * left to right.  y is quantized exactly as jetq_quant_act_1x128 quantizes
 * BF16 input; y itself is not stored.
 *
 *   x, n, c, ldx   BF16 input [n x c], row stride ldx (multiple of 8); c <= 32768
 *   w              BF16 weight [c] (16-byte aligned)
 *   eps            in [0, 1]
 *   rstd           float [n], device: written with rstd[r] (kept for the
 *                  backward pass); written even when both copies are skipped
 *   q_row ... nseg as for jetq_quant_act_1x128
 * Two launches on `stream`: the per-row statistics, then the quantizer.
 */
JETQ_API jetq_status jetq_quant_act_1x128_rmsnorm(const uint16_t *x, int64_t n, int64_t c, int64_t ldx,
                                 const uint16_t *w, float eps, float *rstd,
                                 uint8_t *q_row, float *s_row,
                                 uint8_t *q_col, float *s_col, int64_t ldq_col,
                                 const int64_t *seg_offsets, int nseg, void *stream);

/*
 * Activation quantizer fused with its producer: the SwiGLU product feeding
 * the down projection (Jet-RL explainer, "Summary of What Jet-RL Changes
 * Versus BF16 Training", MLP block: SiLU of the gate output times the up
 * output, then 1x128 quantization before the down projection; papercache
 * summary 4.3: fused activation and RMSNorm kernels beside the quantizers).
 *
 * The quantized tensor is h = BF16(fl32(fl32(g * fl32(1 / fl32(1 + e))) * u))
 * with e = exp(-g) in binary32 by Cody-Waite reduction and a degree-7 Taylor
 * polynomial evaluated by fma (the same function on every machine; +inf for
 * -g > 88, 0 for -g < -87).  h is quantized exactly as jetq_quant_act_1x128
 * quantizes BF16 input and is not stored.
 *
 *   gate, up       BF16 [n x c], row strides ldg, ldu (multiples of 8)
 *   q_row ... nseg as for jetq_quant_act_1x128
 */
JETQ_API jetq_status jetq_quant_act_1x128_swiglu(const uint16_t *gate, const uint16_t *up, int64_t n, int64_t c,
                                 int64_t ldg, int64_t ldu,
                                 uint8_t *q_row, float *s_row,
                                 uint8_t *q_col, float *s_col, int64_t ldq_col,
                                 const int64_t *seg_offsets, int nseg, void *stream);

/*
 * NVFP4 (Miles "Blackwell-native RL recipes" post, NVFP4 section): FP4 E2M1
 * values, one E4M3 scale per block of 16 consecutive values (rounded to the
 * nearest E4M3 value), one FP32 scale for a larger scope: per token (row) for
 * activations, per tensor for weights (a gate/up pair shares one).  The post
 * gives no formula; the library computes
 *   S_g = fl32(amax_scope / 2688)                     (2688 = 448 * 6)
 *   e_b = E4M3(fl32(fl32(amax_b / 6) / S_g)),  D_b = fl32(decode(e_b) * S_g)
 *   q   = E2M1(fl32(x / D_b))   (nearest, ties to even, saturating at 6;
 *                                every code 0 where D_b = 0)
 *
 *   x, rows, cols, ldx  BF16 [rows x cols], row stride ldx (multiple of 8); cols % 16 == 0
 *   scope_amax  device float: max |x| of the tensor scope (e.g. from
 *               jetq_amax_bf16 over gate and up); NULL: one scope per row
 *   q    packed codes [rows x cols/2], element 2j in the low nibble of byte j (4-byte aligned)
 *   sb   E4M3 block scales [rows x cols/16], row-major
 *   sg   FP32 scope scales: [rows] (per row) or [1] (written from row 0's pass)
 * One warp per row; with a per-row scope it reads the row twice.
 */
JETQ_API jetq_status jetq_quant_nvfp4(const uint16_t *x, int64_t rows, int64_t cols, int64_t ldx,
                                 const float *scope_amax, uint8_t *q, uint8_t *sb, float *sg, void *stream);

/*
 * max |x| over a BF16 tensor, folded into *amax (device float, at least 0 on
 * entry; a non-negative float compares as its bits): call it on gate and on
 * up with one *amax for a shared NVFP4 tensor scope.  cols % 8 == 0.
 */
JETQ_API jetq_status jetq_amax_bf16(const uint16_t *x, int64_t rows, int64_t cols, int64_t ldx, float *amax,
                                 void *stream);

/*
 * BF16 dequantization of an NVFP4 copy (the post's dequantized-backward mode:
 * BF16 GEMMs on BF16 values of the exact low-precision operands):
 * out = BF16(e2m1 * decode(e_b) * S_g), rounded once.
 *   q, sb, sg   as jetq_quant_nvfp4 writes them; per_row = 1: sg has one scale
 *               per row, 0: one scale for the tensor
 *   out         BF16 [rows x cols], row stride ldo (multiple of 8), 16-byte aligned
 */
JETQ_API jetq_status jetq_dequant_nvfp4_bf16(const uint8_t *q, const uint8_t *sb, const float *sg, int per_row,
                                 int64_t rows, int64_t cols, uint16_t *out, int64_t ldo, void *stream);

/*
 * Weight quantizer, 128x128 blocks (Jet-RL explainer, "GEMM Quantization":
 * S_W(i,j) = max|W_tile(i,j)| / 448; the DGrad operand is the same FP8
 * weight, only transposed).  Runs after every optimizer step; its output is
 * what training and rollout both consume.
 *
 *   w      BF16 [d x c], row stride ldw
 *   q, s   codes [d x c], scales [d/128 x c/128]
 *   qT, sT transposed codes [c x d], scales [c/128 x d/128] (nullable pair)
 */
JETQ_API jetq_status jetq_quant_w_128x128(const uint16_t *w, int64_t d, int64_t c, int64_t ldw,
                                 uint8_t *q, float *s, uint8_t *qT, float *sT, void *stream);

/*
 * MXFP8 quantizer (Miles Blackwell post, MXFP8 section: 32 consecutive E4M3
 * values share one E8M0 scale rounded up; row-wise and column-wise copies are
 * each quantized from BF16).
 *
 *   x        BF16 [rows x cols], row stride ldx; cols a multiple of 128
 *   q_row    codes [rows x cols], e8_row scale atoms for (rows, cols)   (nullable pair)
 *   q_col    codes [cols x ldq_col], e8_col scale atoms for (cols, ldq_col) (nullable pair);
 *            segments start on multiples of 128 exactly as in the FP32-scale
 *            column copy; whole 32-blocks past a segment's end have scale
 *            byte 127 and codes 0x00
 *   seg_offsets, nseg  as for jetq_quant_act_1x128
 */
JETQ_API jetq_status jetq_quant_mx32(const uint16_t *x, int64_t rows, int64_t cols, int64_t ldx,
                            uint8_t *q_row, uint8_t *e8_row,
                            uint8_t *q_col, uint8_t *e8_col, int64_t ldq_col,
                            const int64_t *seg_offsets, int nseg, void *stream);

/*
 * 128-block recipe with power-of-two scales (SkyRL "Deep dive: FP8
 * quantization with FP32 and power-of-two block scales": the blockwise
 * recipe's FP32 scales constrained to powers of two, the only block scaling
 * Blackwell tensor cores take).  Per 1x128 row group / 128x1 column group /
 * 128x128 weight block: e = smallest integer with amax <= 448 * 2^e (the MX
 * rule), q = E4M3(x * 2^-e).  Scales are written in the MX atom layout for
 * the same (rows, K) as MXFP8 (jetq_mx_scale_bytes), the byte e + 127 repeated
 * in the four 32-element sub-blocks of each group, so the GEMMs read them
 * with JETQ_RECIPE_BLOCK128_POW2 (or MXFP8) unchanged.
 *
 * Activations: arguments and layouts as jetq_quant_mx32 (groups of 128).
 * Weights: q [d x c] (dense), e8 atoms for (d, c); optional qT [c x d] and e8T
 *          atoms for (c, d) (the DGrad operand), both or neither.
 */
JETQ_API jetq_status jetq_quant_act_1x128_pow2(const uint16_t *x, int64_t rows, int64_t cols, int64_t ldx,
                                      uint8_t *q_row, uint8_t *e8_row,
                                      uint8_t *q_col, uint8_t *e8_col, int64_t ldq_col,
                                      const int64_t *seg_offsets, int nseg, void *stream);
JETQ_API jetq_status jetq_quant_w_128x128_pow2(const uint16_t *w, int64_t d, int64_t c, int64_t ldw,
                                      uint8_t *q, uint8_t *e8, uint8_t *qT, uint8_t *e8T, void *stream);

/*
 * Column copy re-quantized from the FP8 row copy (JetRL's
 * requantize_for_dgrad: the 1x128 copy goes back through dequantization and
 * is quantized again along the token dimension; the Miles post traces this
 * to DeepSeek-V3 and contrasts it with taking both copies from BF16).  Each value
 * is rebuilt in binary32, v = fl32(decode(q_row[r,k]) * s_row[k/128, r]),
 * then quantized as the column copy of jetq_quant_act_1x128 quantizes BF16:
 * S = fl32(amax/448) per 128x1 group inside each segment, q = E4M3(fl32(v/S)).
 *
 *   q_row, s_row   the row copy of an [n x c] tensor (layouts above)
 *   q_col, s_col   column copy [c x ldq_col] and its scales, exactly the
 *                  layout jetq_quant_act_1x128 writes (same capacity rule)
 *   seg_offsets, nseg  as for jetq_quant_act_1x128
 */
JETQ_API jetq_status jetq_requant_col_from_row(const uint8_t *q_row, const float *s_row, int64_t n, int64_t c,
                                      uint8_t *q_col, float *s_col, int64_t ldq_col,
                                      const int64_t *seg_offsets, int nseg, void *stream);

/*
 * Dequantization to BF16 (the dequant side of the pages' dequant-requant
 * boundary and of a dequantized backward pass): out[r, k] = BF16 of the
 * exact product decode(q[r, k]) * S, rounded once to nearest-even.
 *   layout ROWGROUPS_1X128: s [cols/128 x rows] (a row copy's scales)
 *   layout BLOCKS_128X128:  s [rows/128 x cols/128] (a weight's scales)
 *   q [rows x cols] dense; out BF16 bit patterns [rows x ldo].
 */
typedef enum {
    JETQ_SCALES_ROWGROUPS_1X128 = 0,
    JETQ_SCALES_BLOCKS_128X128 = 1
} jetq_scale_layout;
JETQ_API jetq_status jetq_dequant_bf16(const uint8_t *q, const float *s, int64_t rows, int64_t cols,
                              jetq_scale_layout layout, uint16_t *out, int64_t ldo, void *stream);

/* ======================================================================== */
/* GEMMs                                                                    */
/* ======================================================================== */
/*
 * The three linear-layer GEMMs (papercache summary 2.2):
 *   FProp  Y  = X W^T    [N x D] = [N x C] [C x D]
 *   DGrad  dX = dY W     [N x C] = [N x D] [D x C]
 *   WGrad  dW = dY^T X   [D x C] = [D x N] [N x C]
 * Every operand is K-major (the contraction dimension contiguous).
 *
 * BLOCK128 arithmetic, identical for every path and tile shape (this is what
 * makes rollout FProp bitwise equal to training FProp):
 *   acc = 0;  for kb = 0, 1, ... (K-blocks of 128, ascending):
 *       P  = sum over the block of qa * qb   (tensor core, FP32, fresh accumulator)
 *       s  = fl32(Sa[row, kb] * Sb[col, kb])
 *       acc = fma(P, s, acc)
 *   out = acc (F32) or bf16_rne(acc); WGrad with accumulate: out = fl32(out_old + acc).
 * MXFP8 arithmetic: the tensor core's block-scaled MMA over all of K into one
 * FP32 accumulator.
 *
 * Output stride ld* is in output elements (a multiple of 4 for F32, 8 for BF16).
 */

/*
 * FProp.  BLOCK128: qx = row copy of X [n x c], sx [c/128 x n]; qw [d x c],
 * sw [d/128 x c/128].  MXFP8: qx row MX copy of X, sx its scale atoms (n, c);
 * qw row MX copy of W [d x c], sw its scale atoms (d, c).
 */
JETQ_API jetq_status jetq_gemm_fprop(jetq_recipe recipe,
                            const uint8_t *qx, const void *sx,
                            const uint8_t *qw, const void *sw,
                            int64_t n, int64_t d, int64_t c,
                            void *y, jetq_out_dtype y_dtype, int64_t ldy,
                            jetq_path path, void *stream);

/*
 * FProp with a caller-owned workspace, for rollout-sized batches.  The SkyRL
 * post ("On-Policy FP8 weight sync") has the rollout engine run the trainer's
 * FP8 weights, and the Jet-RL explainer's rollout keeps 128 sequences in
 * flight: each decode step multiplies a few tokens by whole weights.  When the
 * decode path applies (BLOCK128, 1 <= n <= 64, a weight of at least 32 and at
 * most 152 128-row bands), a cluster of SMs shares each band's K range and
 * the partial sums pass through `workspace`; the fold order is unchanged, so
 * the result equals jetq_gemm_fprop's bit for bit.  Otherwise (another recipe
 * or path, other sizes, a null or too small workspace) it runs exactly what
 * jetq_gemm_fprop runs.
 *
 * workspace: device memory, 16-byte aligned, at least
 * jetq_decode_workspace_bytes(n, d, c) bytes (0 when the shape does not use
 * one; currently d * c/128 * n * 4 bytes).  No initial contents are needed;
 * the call overwrites it.  Calls that share a workspace must not overlap on
 * the GPU.  Errors as jetq_gemm_fprop, plus JETQ_ERR_MISALIGNED for the
 * workspace.
 */
JETQ_API size_t jetq_decode_workspace_bytes(int64_t n, int64_t d, int64_t c);
JETQ_API jetq_status jetq_gemm_fprop_ws(jetq_recipe recipe,
                            const uint8_t *qx, const void *sx,
                            const uint8_t *qw, const void *sw,
                            int64_t n, int64_t d, int64_t c,
                            void *y, jetq_out_dtype y_dtype, int64_t ldy,
                            void *workspace, size_t workspace_bytes,
                            jetq_path path, void *stream);

/*
 * Rollout FProp that allocates nothing (BLOCK128, the decode path).  The
 * paper has no counterpart to it: it is a library convenience.  Some callers
 * cannot hand out device memory for a workspace: a framework whose caching
 * allocator must own every device allocation, a serving loop that cannot
 * afford the device-wide synchronization of cudaMalloc/cudaFree, or a host
 * that gives a plugin only a stream and its input/output buffers.  This call
 * computes exactly what jetq_gemm_fprop(JETQ_RECIPE_BLOCK128, ...,
 * JETQ_PATH_DECODE, ...) and jetq_gemm_fprop_ws compute, bit for bit, with
 * the split-K decode's partial sums kept in a scratch array built into the
 * library (JETQ_NOALLOC_SCRATCH_BYTES of device memory, held by every GPU
 * that loads the library until the process exits).  It calls no allocator.
 *
 * Arguments as jetq_gemm_fprop (qx [n x c], sx [c/128 x n], qw [d x c],
 * sw [d/128 x c/128], y [n x ldy]).  Returns JETQ_ERR_UNSUPPORTED_SHAPE when
 * the split-K partials of this shape, jetq_decode_workspace_bytes(n, d, c),
 * exceed JETQ_NOALLOC_SCRATCH_BYTES (e.g. more than 10 tokens against a
 * 4096 x 12288 weight); shapes that need no partials run without the array.
 * The first call on a device looks up the array's device address (with that
 * device current) and caches it; make that first call before any stream
 * capture.  Every call shares the one array: calls that overlap on the GPU
 * (other streams, or several host threads) race on it.  Nothing in it needs
 * an initial value: each call writes every partial before reading it.
 */
#define JETQ_NOALLOC_SCRATCH_BYTES (16u << 20)
JETQ_API jetq_status jetq_gemm_fprop_noalloc(const uint8_t *qx, const float *sx,
                            const uint8_t *qw, const float *sw,
                            int64_t n, int64_t d, int64_t c,
                            void *y, jetq_out_dtype y_dtype, int64_t ldy,
                            void *stream);

/*
 * DGrad.  BLOCK128: qdy = row copy of dY [n x d], sdy [d/128 x n]; qwt = the
 * transposed weight copy [c x d], swt [c/128 x d/128].  MXFP8: qdy row MX
 * copy of dY (n, d); qwt = column MX copy of W ([c x d], blocks of 32 along d).
 */
JETQ_API jetq_status jetq_gemm_dgrad(jetq_recipe recipe,
                            const uint8_t *qdy, const void *sdy,
                            const uint8_t *qwt, const void *swt,
                            int64_t n, int64_t d, int64_t c,
                            void *dx, jetq_out_dtype dx_dtype, int64_t lddx,
                            void *stream);

/*
 * WGrad.  Both operands are column copies along the token axis with the same
 * segment layout: qdyc [d x ldk] (scales sdyc [k/128 x d]), qxc [c x ldk]
 * (scales sxc [k/128 x c]); k = column-copy length (a multiple of 128, the
 * zero-padded positions contribute nothing), ldk >= k a multiple of 16.
 * MXFP8: the same codes with scale atoms (d, k) and (c, k).
 * dw is FP32 [d x c], stride lddw; accumulate != 0 adds into it.
 */
JETQ_API jetq_status jetq_gemm_wgrad(jetq_recipe recipe,
                            const uint8_t *qdyc, const void *sdyc,
                            const uint8_t *qxc, const void *sxc,
                            int64_t k, int64_t ldk, int64_t d, int64_t c,
                            float *dw, int64_t lddw, int accumulate, void *stream);

/*
 * Grouped GEMMs for MoE experts (Miles Blackwell post: MoE expert GEMMs are
 * quantized like every other linear layer).  Routed rows are sorted by expert:
 * expert e owns rows seg_offsets[e] .. seg_offsets[e+1]-1 (device int64
 * [num_experts + 1], from 0 to the routed-row count; values are clamped on the
 * device, so bad offsets give wrong sums but never out-of-bounds accesses).
 * Every expert runs the same arithmetic as the matching dense GEMM.
 *
 *   FPROP  a = routed activations, row copy [m x ldk] (K = k);  b = expert
 *          weights stacked [num_experts x n x ldk];  out [m x n], row r of
 *          expert e = a[r] * W_e^T.
 *   DGRAD  a = routed output gradients, row copy [m x ldk] (K = k = D);
 *          b = expert transposed weights stacked [num_experts x n x ldk]
 *          (n = C); out [m x n].
 *   WGRAD  a = output-gradient column copy [m x ldk] (m = D), b = activation
 *          column copy [n x ldk] (n = C), both made by the quantizers with
 *          these segment offsets (k = column-copy length); out = FP32 expert
 *          gradients stacked [num_experts x m x n] (expert stride m * ldo);
 *          an expert with no rows gets zeros (or is left unchanged with
 *          accumulate).
 *
 * Scales.  BLOCK128: FPROP/DGRAD sa [k/128 x m], sb [num_experts x n/128 x
 * k/128] (each expert's 128x128 grid); WGRAD sa [k/128 x m], sb [k/128 x n].
 * MXFP8: FPROP/DGRAD sa = atoms for (m, k), sb = each expert's atoms for
 * (n, k) stacked jetq_mx_scale_bytes(n, k) apart; WGRAD sa, sb = atoms of the
 * two column copies.
 * Limits: 1 <= num_experts <= 256; n, k multiples of 128; ldk >= k, a
 * multiple of 16.
 */
JETQ_API jetq_status jetq_gemm_grouped(jetq_gemm_kind kind, jetq_recipe recipe,
                                       const uint8_t *a, const void *sa, const uint8_t *b, const void *sb,
                                       int64_t m, int64_t n, int64_t k, int64_t ldk,
                                       const int64_t *seg_offsets, int num_experts,
                                       void *out, jetq_out_dtype out_dtype, int64_t ldo, int accumulate,
                                       void *stream);

/* ======================================================================== */
/* NVFP4 GEMM                                                               */
/* ======================================================================== */
/*
 * Scale atoms of an NVFP4 payload with R rows and K columns (K a multiple of
 * 256): the E4M3 block scales (one per row and 16 columns) regrouped into the
 * 512-byte unit the tensor core's block-scaled FP4 MMA reads, one atom per
 * 256-column K-block kb, 128-row band rb and 64-column step s:
 *   RB = ceil(R / 128);  atom (kb, rb, s) at ((kb * RB + rb) * 4 + s) * 512
 *   byte of (r, k) inside it: (r % 32) * 16 + ((r % 128) / 32) * 4 + (k % 64) / 16
 * Rows past R in the last band are zero.
 */
JETQ_API int64_t jetq_nvfp4_atom_bytes(int64_t rows, int64_t k);

/*
 * Row-major block scales sb [rows x k/16] (as jetq_quant_nvfp4 writes them) ->
 * scale atoms (layout above, jetq_nvfp4_atom_bytes(rows, k) bytes).  A pure
 * byte permutation.  k % 256 == 0; sb and atoms 16-byte aligned.
 */
JETQ_API jetq_status jetq_nvfp4_scale_atoms(const uint8_t *sb, int64_t rows, int64_t k, uint8_t *atoms,
                                            void *stream);

/*
 * NVFP4 FProp with the scope scales in the epilogue (Miles "Blackwell-native
 * RL recipes" post, NVFP4 section: activations carry a per-token FP32 scale,
 * which that post's path applied in a step of its own, outside the GEMM):
 *   acc[i, j] = sum_k (e2m1(qa[i, k]) * e4m3(sba[i, k/16])) * (e2m1(qb[j, k]) * e4m3(sbb[j, k/16]))
 *               (tensor core: block-scaled FP4 MMA, FP32 accumulation over all of K)
 *   out[i, j] = fl32(fl32(sga[per_row_a ? i : 0] * sgb[0]) * acc[i, j]), F32 or BF16 (RNE of that)
 *   qa    packed E2M1 codes of A [m x k/2] (activations: jetq_quant_nvfp4, element 2j
 *         in the low nibble of byte j); sfa = its scale atoms (m, k); sga [m] (per-token
 *         scope, per_row_a = 1) or [1]
 *   qb    packed codes of B [n x k/2] (the weight, Y = X W^T); sfb = its atoms (n, k);
 *         sgb [1] (tensor scope)
 *   out   [m x n], row stride ldo
 * Limits: m >= 0; n a multiple of 128; k a multiple of 256; qa, qb, sfa, sfb,
 * out 16-byte aligned; sga, sgb 4-byte aligned.
 */
JETQ_API jetq_status jetq_gemm_nvfp4(const uint8_t *qa, const uint8_t *sfa, const float *sga, int per_row_a,
                                     const uint8_t *qb, const uint8_t *sfb, const float *sgb,
                                     int64_t m, int64_t n, int64_t k,
                                     void *out, jetq_out_dtype out_dtype, int64_t ldo, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* JETQ_H */
