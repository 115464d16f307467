// Internal declarations shared by the jetq translation units (host side).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/jetq.h"

namespace jetq {

// ---------------------------------------------------------------- quantizers
// Producer fused ahead of the activation quantizer: the quantized tensor is
// x itself, RMSNorm(x) * w, or silu(x) * up, rounded to BF16.
enum ActProducer : int { kProducePlain = 0, kProduceRms = 1, kProduceSwiglu = 2 };

struct ActQuantArgs {
    const uint16_t *x;
    int64_t n, c, ldx;
    uint8_t *q_row;
    float *s_row;
    uint8_t *q_col;
    float *s_col;
    int64_t ldq_col;
    const int64_t *seg; // device, nseg + 1 entries, or nullptr
    int nseg;
    int producer = kProducePlain;
    const uint16_t *up = nullptr; // SwiGLU: the up projection [n x ldup]
    int64_t ldup = 0;
    const uint16_t *w = nullptr;  // RMSNorm: per-column weight [c]
    const float *rstd = nullptr;  // RMSNorm: per-row 1 / rms, from launch_rms_rstd
};

// RMSNorm statistics: rstd[r] = 1 / sqrt(sum_sq(x[r]) / c + eps), the sum of
// squares in binary32 in a fixed order (each 128-column group left to right
// by fma, then the group sums left to right); c a multiple of 128, <= 32768.
cudaError_t launch_rms_rstd(const uint16_t *x, int64_t n, int64_t c, int64_t ldx, float eps, float *rstd,
                            cudaStream_t st);

struct WeightQuantArgs {
    const uint16_t *w;
    int64_t d, c, ldw;
    uint8_t *q;
    float *s;
    uint8_t *qT;
    float *sT;
};

struct MxQuantArgs {
    const uint16_t *x;
    int64_t rows, cols, ldx;
    uint8_t *q_row;
    uint8_t *e8_row;
    uint8_t *q_col;
    uint8_t *e8_col;
    int64_t ldq_col;
    const int64_t *seg;
    int nseg;
};

cudaError_t launch_quant_act(const ActQuantArgs &a, cudaStream_t st);
cudaError_t launch_quant_weight(const WeightQuantArgs &a, cudaStream_t st);
// group: 32 (MXFP8) or 128 (power-of-two 128-block recipe)
cudaError_t launch_quant_mx(const MxQuantArgs &a, int group, cudaStream_t st);

struct WeightPow2Args {
    const uint16_t *w;
    int64_t d, c, ldw;
    uint8_t *q;
    uint8_t *e8;  // MX scale atoms of W (rows d, K = c)
    uint8_t *qT;  // optional
    uint8_t *e8T; // MX scale atoms of W^T (rows c, K = d), with qT
};
cudaError_t launch_quant_weight_pow2(const WeightPow2Args &a, cudaStream_t st);

// Column copy re-quantized from a 1x128 row copy (v = fl32(decode(q) * S_row)).
struct RequantArgs {
    const uint8_t *q_row;
    const float *s_row;
    int64_t n, c;
    uint8_t *q_col;
    float *s_col;
    int64_t ldq_col;
    const int64_t *seg;
    int nseg;
};
cudaError_t launch_requant_col(const RequantArgs &a, cudaStream_t st);

// BF16 of decode(q) * S, rounded once; blocks = false: 1x128 row groups
// (s [cols/128 x rows]), true: 128x128 blocks (s [rows/128 x cols/128]).
struct DequantArgs {
    const uint8_t *q;
    const float *s;
    int64_t rows, cols;
    bool blocks;
    uint16_t *out;
    int64_t ldo;
};
cudaError_t launch_dequant_bf16(const DequantArgs &a, cudaStream_t st);

// --------------------------------------------------------------------- GEMMs
// One block-scaled GEMM problem: out[M x N] = A[M x K] * B[N x K]^T, both
// operands K-major FP8 with per-128-K-block scales.
enum class BScale : int {
    Block128 = 0, // sb[(n / 128) * (K / 128) + kb]           (128x128 weight blocks)
    PerRow = 1    // sb[kb * N + n]                           (column copy along K)
};

enum class GroupKind : int {
    None = 0, // one problem
    Rows = 1, // per-expert FProp/DGrad: A rows split by segments, B = experts' weights stacked [E*N x K]
    K = 2     // per-expert WGrad: K-blocks split by segments (column copies), out = experts stacked [E x M x N]
};

struct GemmProblem {
    const uint8_t *a;  // [M x lda] codes
    const float *sa;   // [K/128 x M]
    const uint8_t *b;  // [N x ldb] codes
    const float *sb;   // see BScale
    int64_t M, N, K;
    int64_t lda, ldb;  // bytes
    BScale bscale;
    void *out;
    int64_t ldo;       // elements
    jetq_out_dtype out_dtype;
    int accumulate;    // F32 only: out = out + acc
    GroupKind group = GroupKind::None;
    const int64_t *seg = nullptr; // device [num_experts + 1]
    int num_experts = 1;
    void *ws = nullptr;           // device workspace of the split-K decode (optional)
    size_t ws_bytes = 0;
};

enum class GemmShape : int { Train = 0, Decode = 1 };

// Launch with programmatic stream serialization: the kernel's prologue may
// overlap the stream's previous kernel (the kernel calls griddepcontrol.wait
// before it touches global memory, and launch_dependents once its own
// prologue is done).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<Args &&>(args)...);
}

cudaError_t launch_gemm_block128(const GemmProblem &p, GemmShape shape, cudaStream_t st);

// MXFP8 GEMM: both operands K-major E4M3 with E8M0 scale atoms (include/jetq.h
// layout; atom of (row band rb, K-block kb) at sf + (kb * RB + rb) * 512).
struct MxGemmProblem {
    const uint8_t *a;
    const uint8_t *sfa; // atoms for (M rows, K)
    const uint8_t *b;
    const uint8_t *sfb; // atoms for (N rows, K)
    int64_t M, N, K;
    int64_t lda, ldb;
    void *out;
    int64_t ldo;
    jetq_out_dtype out_dtype;
    int accumulate;
    GroupKind group = GroupKind::None;
    const int64_t *seg = nullptr;
    int num_experts = 1;
};

cudaError_t launch_gemm_mx(const MxGemmProblem &p, cudaStream_t st);
cudaError_t gemm_mx_read_and_clear_error(cudaStream_t st, unsigned *out);

// One CTA whose two waiters time out on mbarriers nothing completes (the
// bounded-wait diagnostic); records the timeout in the 128-block error word.
cudaError_t launch_selftest_wait(unsigned long long limit_ns, long long *elapsed_ns, cudaStream_t st);

// Decode-shaped 128-block FProp/DGrad with the operands swapped (weight rows
// as the MMA's M, tokens as its N): dense, B-block scales, 1 <= M <= 64
// tokens, N a multiple of 128 with at least kDecodeSwappedMinTiles 128-row
// weight tiles, K a multiple of 128.  Bitwise equal to launch_gemm_block128.
constexpr int64_t kDecodeSwappedMinTiles = 32;
bool gemm_decode_swapped_applies(const GemmProblem &g);
// Split-K decode (a cluster of CTAs per 128-row band; partial sums through a
// workspace): cluster size for a shape (1 = not used) and workspace bytes.
int decode_split_factor(int64_t M, int64_t N, int64_t K);
size_t decode_split_workspace_bytes(int64_t M, int64_t N, int64_t K);
// The same FProp with the partial sums in a device array built into the
// library (no allocation; see jetq_gemm_fprop_noalloc): its size, and the
// launch (cudaErrorInvalidValue when the shape needs more than the array).
size_t decode_static_scratch_bytes();
cudaError_t launch_gemm_decode_static(GemmProblem g, cudaStream_t st);
cudaError_t launch_gemm_decode_swapped(const GemmProblem &g, cudaStream_t st);
cudaError_t gemm_decode_read_and_clear_error(cudaStream_t st, unsigned *out);

cudaError_t gemm_read_and_clear_error(cudaStream_t st, unsigned *out);

// NVFP4 (E2M1 values, E4M3 scale per 16, FP32 scope scale per row or tensor)
cudaError_t launch_amax_bf16(const uint16_t *x, int64_t rows, int64_t cols, int64_t ldx, float *amax,
                             cudaStream_t st);
cudaError_t launch_quant_nvfp4(const uint16_t *x, int64_t rows, int64_t cols, int64_t ldx, const float *scope_amax,
                               uint8_t *q, uint8_t *sb, float *sg, cudaStream_t st);
cudaError_t launch_dequant_nvfp4(const uint8_t *q, const uint8_t *sb, const float *sg, int per_row, int64_t rows,
                                 int64_t cols, uint16_t *out, int64_t ldo, cudaStream_t st);

// NVFP4 FProp: packed E2M1 operands [M x K/2], [N x K/2] bytes, scale atoms
// (include/jetq.h layout), FP32 scope scales applied in the epilogue.
struct Nvfp4GemmProblem {
    const uint8_t *a;
    const uint8_t *sfa;
    const float *sga;
    int per_row_a;
    const uint8_t *b;
    const uint8_t *sfb;
    const float *sgb;
    int64_t M, N, K;
    void *out;
    int64_t ldo;
    jetq_out_dtype out_dtype;
};
cudaError_t launch_gemm_nvfp4(const Nvfp4GemmProblem &p, cudaStream_t st);
cudaError_t launch_nvfp4_atoms(const uint8_t *sb, int64_t rows, int64_t k, uint8_t *atoms, cudaStream_t st);
cudaError_t gemm_nvfp4_read_and_clear_error(cudaStream_t st, unsigned *out);

// TMA descriptor for a BF16 matrix [rows x cols], row stride ld elements:
// 128 x 128 boxes (32 KB, rows of 256 bytes, no swizzle), zero fill out of bounds.
cudaError_t make_bf16_tile_map(CUtensorMap *map, const void *base, int64_t cols, int64_t rows, int64_t ld);

// device error word of the quantizers (bounded waits of the TMA-fed kernels)
cudaError_t quant_read_and_clear_error(cudaStream_t st, unsigned *out);

// TMA descriptor for a K-major byte matrix [rows x k_extent], row stride ld,
// boxes of 128 bytes x box_rows (x kb_per_box consecutive K-blocks, as a 3-D
// map, when kb_per_box > 1), 128-byte swizzle, zero fill out of bounds.
cudaError_t make_kmajor_map(CUtensorMap *map, const void *base, int64_t k_extent, int64_t rows, int64_t ld,
                            int box_rows, int kb_per_box = 1);

// Number of SMs of the current device (cached per device).
int sm_count();

} // namespace jetq
