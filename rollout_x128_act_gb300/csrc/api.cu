// The C ABI (include/jetq.h): host-side validation, then one launch on the
// caller's stream.  Nothing here allocates, synchronizes (except
// jetq_check_device_error) or keeps pointers.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "jetq_internal.h"

namespace jetq {

int sm_count()
{
    static std::atomic<int> cached[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return 1;
    int v = cached[dev].load(std::memory_order_relaxed);
    if (v == 0) {
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
            v = 1;
        cached[dev].store(v, std::memory_order_relaxed);
    }
    return v;
}

namespace {

// 1 = sm_103, -1 = other, 0 = unknown yet
std::atomic<int> g_arch_ok[64];

jetq_status check_arch()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return JETQ_ERR_CUDA;
    int v = g_arch_ok[dev].load(std::memory_order_relaxed);
    if (v == 0) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return JETQ_ERR_CUDA;
        v = (major == 10 && minor == 3) ? 1 : -1;
        g_arch_ok[dev].store(v, std::memory_order_relaxed);
    }
    return v == 1 ? JETQ_OK : JETQ_ERR_ARCH;
}

bool aligned16(const void *p)
{
    return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

jetq_status from_cuda(cudaError_t e)
{
    return e == cudaSuccess ? JETQ_OK : JETQ_ERR_CUDA;
}

#define JQ_REQUIRE(cond, code)                                                                                       \
    do {                                                                                                             \
        if (!(cond))                                                                                                 \
            return (code);                                                                                           \
    } while (0)

jetq_status check_out(const void *out, jetq_out_dtype dt, int64_t ld, int64_t cols)
{
    JQ_REQUIRE(out != nullptr, JETQ_ERR_INVALID_ARG);
    JQ_REQUIRE(dt == JETQ_OUT_F32 || dt == JETQ_OUT_BF16, JETQ_ERR_INVALID_ARG);
    JQ_REQUIRE(ld >= cols, JETQ_ERR_UNSUPPORTED_SHAPE);
    JQ_REQUIRE(aligned16(out) && ld % (dt == JETQ_OUT_F32 ? 4 : 8) == 0, JETQ_ERR_MISALIGNED);
    return JETQ_OK;
}

} // namespace
} // namespace jetq

using namespace jetq;

extern "C" {

const char *jetq_status_string(jetq_status status)
{
    switch (status) {
    case JETQ_OK: return "ok";
    case JETQ_ERR_INVALID_ARG: return "invalid argument";
    case JETQ_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case JETQ_ERR_MISALIGNED: return "pointer or stride not 16-byte aligned";
    case JETQ_ERR_ARCH: return "device is not compute capability 10.3 (GB300)";
    case JETQ_ERR_CUDA: return "CUDA runtime error";
    case JETQ_ERR_TIMEOUT: return "a kernel gave up a bounded wait";
    }
    return "unknown status";
}

int jetq_version(void)
{
    return 100; // 0.1.0
}

int64_t jetq_colcopy_capacity(int64_t n, int nseg)
{
    if (n <= 0)
        return 0;
    const int64_t bound = nseg <= 1 ? n : n + 127 * (int64_t)nseg;
    return (bound + 127) / 128 * 128;
}

int64_t jetq_mx_scale_bytes(int64_t rows, int64_t k)
{
    if (rows <= 0 || k <= 0)
        return 0;
    return (rows + 127) / 128 * ((k + 127) / 128) * 512;
}

int64_t jetq_nvfp4_atom_bytes(int64_t rows, int64_t k)
{
    if (rows <= 0 || k <= 0)
        return 0;
    return (rows + 127) / 128 * ((k + 255) / 256) * 4 * 512;
}

jetq_status jetq_nvfp4_scale_atoms(const uint8_t *sb, int64_t rows, int64_t k, uint8_t *atoms, void *stream)
{
    JQ_REQUIRE(rows >= 0 && k > 0, JETQ_ERR_INVALID_ARG);
    JQ_REQUIRE(k % 256 == 0, JETQ_ERR_UNSUPPORTED_SHAPE);
    if (rows == 0)
        return JETQ_OK;
    JQ_REQUIRE(sb != nullptr && atoms != nullptr, JETQ_ERR_INVALID_ARG);
    JQ_REQUIRE(aligned16(sb) && aligned16(atoms), JETQ_ERR_MISALIGNED);
    const jetq_status a = check_arch();
    if (a != JETQ_OK)
        return a;
    return from_cuda(launch_nvfp4_atoms(sb, rows, k, atoms, static_cast<cudaStream_t>(stream)));
}

jetq_status jetq_gemm_nvfp4(const uint8_t *qa, const uint8_t *sfa, const float *sga, int per_row_a,
                            const uint8_t *qb, const uint8_t *sfb, const float *sgb, int64_t m, int64_t n, int64_t k,
                            void *out, jetq_out_dtype out_dtype, int64_t ldo, void *stream)
{
    JQ_REQUIRE(m >= 0 && n > 0 && k > 0 && (per_row_a == 0 || per_row_a == 1), JETQ_ERR_INVALID_ARG);
    JQ_REQUIRE(out_dtype == JETQ_OUT_F32 || out_dtype == JETQ_OUT_BF16, JETQ_ERR_INVALID_ARG);
    JQ_REQUIRE(n % 128 == 0 && k % 256 == 0 && ldo >= n, JETQ_ERR_UNSUPPORTED_SHAPE);
    if (m == 0)
        return JETQ_OK;
    JQ_REQUIRE(qa != nullptr && sfa != nullptr && sga != nullptr && qb != nullptr && sfb != nullptr &&
                   sgb != nullptr && out != nullptr,
               JETQ_ERR_INVALID_ARG);
    JQ_REQUIRE(aligned16(qa) && aligned16(qb) && aligned16(sfa) && aligned16(sfb) &&
                   (reinterpret_cast<uintptr_t>(sga) & 3u) == 0 && (reinterpret_cast<uintptr_t>(sgb) & 3u) == 0 &&
                   aligned16(out) && ldo % (out_dtype == JETQ_OUT_F32 ? 4 : 8) == 0,
               JETQ_ERR_MISALIGNED);
    const jetq_status a = check_arch();
    if (a != JETQ_OK)
        return a;
    Nvfp4GemmProblem g{qa, sfa, sga, per_row_a, qb, sfb, sgb, m, n, k, out, ldo, out_dtype};
    return from_cuda(launch_gemm_nvfp4(g, static_cast<cudaStream_t>(stream)));
}

jetq_status jetq_check_device_error(void *stream)
{
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    unsigned word = 0;
    if (gemm_read_and_clear_error(st, &word) != cudaSuccess || gemm_mx_read_and_clear_error(st, &word) != cudaSuccess ||
        gemm_decode_read_and_clear_error(st, &word) != cudaSuccess || quant_read_and_clear_error(st, &word) != cudaSuccess ||
        gemm_nvfp4_read_and_clear_error(st, &word) != cudaSuccess)
        return JETQ_ERR_CUDA;
    return word ? JETQ_ERR_TIMEOUT : JETQ_OK;
}

jetq_status jetq_selftest_bounded_wait(uint64_t limit_ns, int64_t *elapsed_ns, void *stream)
{
    JQ_REQUIRE(limit_ns >= 1000000ull && limit_ns <= 1000000000ull, JETQ_ERR_INVALID_ARG);
    JQ_REQUIRE(elapsed_ns != nullptr, JETQ_ERR_INVALID_ARG);
    JQ_REQUIRE(reinterpret_cast<uintptr_t>(elapsed_ns) % 8 == 0, JETQ_ERR_MISALIGNED);
    const jetq_status a = check_arch();
    if (a != JETQ_OK)
        return a;
    return from_cuda(launch_selftest_wait(limit_ns, reinterpret_cast<long long *>(elapsed_ns),
                                          static_cast<cudaStream_t>(stream)));
}

jetq_status jetq_quant_act_1x128(const uint16_t *x, int64_t n, int64_t c, int64_t ldx, uint8_t *q_row, float *s_row,
                                 uint8_t *q_col, float *s_col, int64_t ldq_col, const int64_t *seg_offsets, int nseg,
                                 void *stream)
{
    JQ_REQUIRE(n >= 0 && c > 0, JETQ_ERR_INVALID_ARG);
    JQ_REQUIRE((q_row == nullptr) == (s_row == nullptr), JETQ_ERR_INVALID_ARG);
    JQ_REQUIRE((q_col == nullptr) == (s_col == nullptr), JETQ_ERR_INVALID_ARG);
    JQ_REQUIRE(seg_offsets == nullptr || nseg >= 1, JETQ_ERR_INVALID_ARG);
    JQ_REQUIRE(c % 128 == 0 && ldx >= c, JETQ_ERR_UNSUPPORTED_SHAPE);
    const int nseg_eff = seg_offsets ? nseg : 1;
    if (q_col)
        JQ_REQUIRE(ldq_col % 128 == 0 && ldq_col >= jetq_colcopy_capacity(n, nseg_eff), JETQ_ERR_UNSUPPORTED_SHAPE);
    if (n == 0 || (!q_row && !q_col))
        return JETQ_OK;
    JQ_REQUIRE(x != nullptr, JETQ_ERR_INVALID_ARG);
    JQ_REQUIRE(aligned16(x) && ldx % 8 == 0 && aligned16(q_row) && aligned16(s_row) && aligned16(q_col) &&
                   aligned16(s_col) && (reinterpret_cast<uintptr_t>(seg_offsets) & 7u) == 0,
               JETQ_ERR_MISALIGNED);
    const jetq_status a = check_arch();
    if (a != JETQ_OK)
        return a;
    ActQuantArgs args{x, n, c, ldx, q_row, s_row, q_col, s_col, ldq_col, seg_offsets, nseg_eff};
    return from_cuda(launch_quant_act(args, static_cast<cudaStream_t>(stream)));
}

namespace {

// validation shared by the activation quantizer and its fused-producer forms
jetq_status check_act_copies(int64_t n, int64_t c, uint8_t *q_row, float *s_row, uint8_t *q_col, float *s_col,
                             int64_t ldq_col, const int64_t *seg_offsets, int nseg)
{
    JQ_REQUIRE(n >= 0 && c > 0, JETQ_ERR_INVALID_ARG);
    JQ_REQUIRE((q_row == nullptr) == (s_row == nullptr), JETQ_ERR_INVALID_ARG);
    JQ_REQUIRE((q_col == nullptr) == (s_col == nullptr), JETQ_ERR_INVALID_ARG);
    JQ_REQUIRE(seg_offsets == nullptr || nseg >= 1, JETQ_ERR_INVALID_ARG);
    JQ_REQUIRE(c % 128 == 0, JETQ_ERR_UNSUPPORTED_SHAPE);
    if (q_col)
        JQ_REQUIRE(ldq_col % 128 == 0 && ldq_col >= jetq_colcopy_capacity(n, seg_offsets ? nseg : 1),
                   JETQ_ERR_UNSUPPORTED_SHAPE);
    JQ_REQUIRE(aligned16(q_row) && aligned16(s_row) && aligned16(q_col) && aligned16(s_col) &&
                   (reinterpret_cast<uintptr_t>(seg_offsets) & 7u) == 0,
               JETQ_ERR_MISALIGNED);
    return JETQ_OK;
}

} // namespace

jetq_status jetq_quant_act_1x128_rmsnorm(const uint16_t *x, int64_t n, int64_t c, int64_t ldx, const uint16_t *w,
                                         float eps, float *rstd, uint8_t *q_row, float *s_row, uint8_t *q_col,
                                         float *s_col, int64_t ldq_col, const int64_t *seg_offsets, int nseg,
                                         void *stream)
{
    const jetq_status v = check_act_copies(n, c, q_row, s_row, q_col, s_col, ldq_col, seg_offsets, nseg);
    if (v != JETQ_OK)
        return v;
    JQ_REQUIRE(ldx >= c && c <= 32768, JETQ_ERR_UNSUPPORTED_SHAPE);
    JQ_REQUIRE(eps >= 0.0f && eps <= 1.0f, JETQ_ERR_INVALID_ARG);
    if (n == 0)
        return JETQ_OK;
    JQ_REQUIRE(x != nullptr && w != nullptr && rstd != nullptr, JETQ_ERR_INVALID_ARG);
    JQ_REQUIRE(aligned16(x) && ldx % 8 == 0 && aligned16(w) && (reinterpret_cast<uintptr_t>(rstd) & 3u) == 0,
               JETQ_ERR_MISALIGNED);
    const jetq_status a = check_arch();
    if (a != JETQ_OK)
        return a;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = launch_rms_rstd(x, n, c, ldx, eps, rstd, st);
    if (e != cudaSuccess || (!q_row && !q_col))
        return from_cuda(e);
    ActQuantArgs args{x, n, c, ldx, q_row, s_row, q_col, s_col, ldq_col, seg_offsets, seg_offsets ? nseg : 1};
    args.producer = kProduceRms;
    args.w = w;
    args.rstd = rstd;
    return from_cuda(launch_quant_act(args, st));
}

jetq_status jetq_quant_act_1x128_swiglu(const uint16_t *gate, const uint16_t *up, int64_t n, int64_t c,
                                        int64_t ldg, int64_t ldu, uint8_t *q_row, float *s_row, uint8_t *q_col,
                                        float *s_col, int64_t ldq_col, const int64_t *seg_offsets, int nseg,
                                        void *stream)
{
    const jetq_status v = check_act_copies(n, c, q_row, s_row, q_col, s_col, ldq_col, seg_offsets, nseg);
    if (v != JETQ_OK)
        return v;
    JQ_REQUIRE(ldg >= c && ldu >= c, JETQ_ERR_UNSUPPORTED_SHAPE);
    if (n == 0 || (!q_row && !q_col))
        return JETQ_OK;
    JQ_REQUIRE(gate != nullptr && up != nullptr, JETQ_ERR_INVALID_ARG);
    JQ_REQUIRE(aligned16(gate) && ldg % 8 == 0 && aligned16(up) && ldu % 8 == 0, JETQ_ERR_MISALIGNED);
    const jetq_status a = check_arch();
    if (a != JETQ_OK)
        return a;
    ActQuantArgs args{gate, n, c, ldg, q_row, s_row, q_col, s_col, ldq_col, seg_offsets, seg_offsets ? nseg : 1};
    args.producer = kProduceSwiglu;
    args.up = up;
    args.ldup = ldu;
    return from_cuda(launch_quant_act(args, static_cast<cudaStream_t>(stream)));
}

jetq_status jetq_amax_bf16(const uint16_t *x, int64_t rows, int64_t cols, int64_t ldx, float *amax, void *stream)
{
    JQ_REQUIRE(rows >= 0 && cols > 0 && amax != nullptr, JETQ_ERR_INVALID_ARG);
    JQ_REQUIRE(cols % 8 == 0 && ldx >= cols, JETQ_ERR_UNSUPPORTED_SHAPE);
    if (rows == 0)
        return JETQ_OK;
    JQ_REQUIRE(x != nullptr, JETQ_ERR_INVALID_ARG);
    JQ_REQUIRE(aligned16(x) && ldx % 8 == 0 && (reinterpret_cast<uintptr_t>(amax) & 3u) == 0, JETQ_ERR_MISALIGNED);
    const jetq_status a = check_arch();
    if (a != JETQ_OK)
        return a;
    return from_cuda(launch_amax_bf16(x, rows, cols, ldx, amax, static_cast<cudaStream_t>(stream)));
}

jetq_status jetq_quant_nvfp4(const uint16_t *x, int64_t rows, int64_t cols, int64_t ldx, const float *scope_amax,
                             uint8_t *q, uint8_t *sb, float *sg, void *stream)
{
    JQ_REQUIRE(rows >= 0 && cols > 0, JETQ_ERR_INVALID_ARG);
    JQ_REQUIRE(cols % 16 == 0 && ldx >= cols, JETQ_ERR_UNSUPPORTED_SHAPE);
    if (rows == 0)
        return JETQ_OK;
    JQ_REQUIRE(x != nullptr && q != nullptr && sb != nullptr && sg != nullptr, JETQ_ERR_INVALID_ARG);
    JQ_REQUIRE(aligned16(x) && ldx % 8 == 0 && (reinterpret_cast<uintptr_t>(q) & 3u) == 0 &&
                   (reinterpret_cast<uintptr_t>(sg) & 3u) == 0 && (reinterpret_cast<uintptr_t>(scope_amax) & 3u) == 0,
               JETQ_ERR_MISALIGNED);
    const jetq_status a = check_arch();
    if (a != JETQ_OK)
        return a;
    return from_cuda(launch_quant_nvfp4(x, rows, cols, ldx, scope_amax, q, sb, sg, static_cast<cudaStream_t>(stream)));
}

jetq_status jetq_dequant_nvfp4_bf16(const uint8_t *q, const uint8_t *sb, const float *sg, int per_row, int64_t rows,
                                    int64_t cols, uint16_t *out, int64_t ldo, void *stream)
{
    JQ_REQUIRE(rows >= 0 && cols > 0 && (per_row == 0 || per_row == 1), JETQ_ERR_INVALID_ARG);
    JQ_REQUIRE(cols % 16 == 0 && ldo >= cols, JETQ_ERR_UNSUPPORTED_SHAPE);
    if (rows == 0)
        return JETQ_OK;
    JQ_REQUIRE(q != nullptr && sb != nullptr && sg != nullptr && out != nullptr, JETQ_ERR_INVALID_ARG);
    JQ_REQUIRE((reinterpret_cast<uintptr_t>(q) & 3u) == 0 && (reinterpret_cast<uintptr_t>(sg) & 3u) == 0 &&
                   aligned16(out) && ldo % 8 == 0,
               JETQ_ERR_MISALIGNED);
    const jetq_status a = check_arch();
    if (a != JETQ_OK)
        return a;
    return from_cuda(launch_dequant_nvfp4(q, sb, sg, per_row, rows, cols, out, ldo, static_cast<cudaStream_t>(stream)));
}

jetq_status jetq_quant_w_128x128(const uint16_t *w, int64_t d, int64_t c, int64_t ldw, uint8_t *q, float *s,
                                 uint8_t *qT, float *sT, void *stream)
{
    JQ_REQUIRE(w != nullptr && q != nullptr && s != nullptr && d > 0 && c > 0, JETQ_ERR_INVALID_ARG);
    JQ_REQUIRE((qT == nullptr) == (sT == nullptr), JETQ_ERR_INVALID_ARG);
    JQ_REQUIRE(d % 128 == 0 && c % 128 == 0 && ldw >= c, JETQ_ERR_UNSUPPORTED_SHAPE);
    JQ_REQUIRE(aligned16(w) && ldw % 8 == 0 && aligned16(q) && aligned16(qT) &&
                   (reinterpret_cast<uintptr_t>(s) & 3u) == 0 && (reinterpret_cast<uintptr_t>(sT) & 3u) == 0,
               JETQ_ERR_MISALIGNED);
    const jetq_status a = check_arch();
    if (a != JETQ_OK)
        return a;
    WeightQuantArgs args{w, d, c, ldw, q, s, qT, sT};
    return from_cuda(launch_quant_weight(args, static_cast<cudaStream_t>(stream)));
}

namespace {

// E8M0-scaled row and column copies with groups of `group` (32 or 128) elements
jetq_status quant_e8m0_groups(const uint16_t *x, int64_t rows, int64_t cols, int64_t ldx, uint8_t *q_row,
                              uint8_t *e8_row, uint8_t *q_col, uint8_t *e8_col, int64_t ldq_col,
                              const int64_t *seg_offsets, int nseg, int group, void *stream)
{
    JQ_REQUIRE(rows >= 0 && cols > 0, JETQ_ERR_INVALID_ARG);
    JQ_REQUIRE((q_row == nullptr) == (e8_row == nullptr), JETQ_ERR_INVALID_ARG);
    JQ_REQUIRE((q_col == nullptr) == (e8_col == nullptr), JETQ_ERR_INVALID_ARG);
    JQ_REQUIRE(seg_offsets == nullptr || nseg >= 1, JETQ_ERR_INVALID_ARG);
    JQ_REQUIRE(cols % 128 == 0 && ldx >= cols, JETQ_ERR_UNSUPPORTED_SHAPE);
    const int nseg_eff = seg_offsets ? nseg : 1;
    if (q_col)
        JQ_REQUIRE(ldq_col % 128 == 0 && ldq_col >= jetq_colcopy_capacity(rows, nseg_eff), JETQ_ERR_UNSUPPORTED_SHAPE);
    if (rows == 0 || (!q_row && !q_col))
        return JETQ_OK;
    JQ_REQUIRE(x != nullptr, JETQ_ERR_INVALID_ARG);
    JQ_REQUIRE(aligned16(x) && ldx % 8 == 0 && aligned16(q_row) && aligned16(e8_row) && aligned16(q_col) &&
                   aligned16(e8_col) && (reinterpret_cast<uintptr_t>(seg_offsets) & 7u) == 0,
               JETQ_ERR_MISALIGNED);
    const jetq_status a = check_arch();
    if (a != JETQ_OK)
        return a;
    MxQuantArgs args{x, rows, cols, ldx, q_row, e8_row, q_col, e8_col, ldq_col, seg_offsets, nseg_eff};
    return from_cuda(launch_quant_mx(args, group, static_cast<cudaStream_t>(stream)));
}

} // namespace

jetq_status jetq_quant_mx32(const uint16_t *x, int64_t rows, int64_t cols, int64_t ldx, uint8_t *q_row,
                            uint8_t *e8_row, uint8_t *q_col, uint8_t *e8_col, int64_t ldq_col,
                            const int64_t *seg_offsets, int nseg, void *stream)
{
    return quant_e8m0_groups(x, rows, cols, ldx, q_row, e8_row, q_col, e8_col, ldq_col, seg_offsets, nseg, 32,
                             stream);
}

jetq_status jetq_quant_act_1x128_pow2(const uint16_t *x, int64_t rows, int64_t cols, int64_t ldx, uint8_t *q_row,
                                      uint8_t *e8_row, uint8_t *q_col, uint8_t *e8_col, int64_t ldq_col,
                                      const int64_t *seg_offsets, int nseg, void *stream)
{
    return quant_e8m0_groups(x, rows, cols, ldx, q_row, e8_row, q_col, e8_col, ldq_col, seg_offsets, nseg, 128,
                             stream);
}

jetq_status jetq_quant_w_128x128_pow2(const uint16_t *w, int64_t d, int64_t c, int64_t ldw, uint8_t *q, uint8_t *e8,
                                      uint8_t *qT, uint8_t *e8T, void *stream)
{
    JQ_REQUIRE(w != nullptr && q != nullptr && e8 != nullptr && d > 0 && c > 0, JETQ_ERR_INVALID_ARG);
    JQ_REQUIRE((qT == nullptr) == (e8T == nullptr), JETQ_ERR_INVALID_ARG);
    JQ_REQUIRE(d % 128 == 0 && c % 128 == 0 && ldw >= c, JETQ_ERR_UNSUPPORTED_SHAPE);
    JQ_REQUIRE(aligned16(w) && ldw % 8 == 0 && aligned16(q) && aligned16(qT) && aligned16(e8) && aligned16(e8T),
               JETQ_ERR_MISALIGNED);
    const jetq_status a = check_arch();
    if (a != JETQ_OK)
        return a;
    WeightPow2Args args{w, d, c, ldw, q, e8, qT, e8T};
    return from_cuda(launch_quant_weight_pow2(args, static_cast<cudaStream_t>(stream)));
}

jetq_status jetq_requant_col_from_row(const uint8_t *q_row, const float *s_row, int64_t n, int64_t c, uint8_t *q_col,
                                      float *s_col, int64_t ldq_col, const int64_t *seg_offsets, int nseg,
                                      void *stream)
{
    JQ_REQUIRE(n >= 0 && c > 0, JETQ_ERR_INVALID_ARG);
    JQ_REQUIRE(seg_offsets == nullptr || nseg >= 1, JETQ_ERR_INVALID_ARG);
    JQ_REQUIRE(c % 128 == 0, JETQ_ERR_UNSUPPORTED_SHAPE);
    const int nseg_eff = seg_offsets ? nseg : 1;
    JQ_REQUIRE(ldq_col % 128 == 0 && ldq_col >= jetq_colcopy_capacity(n, nseg_eff), JETQ_ERR_UNSUPPORTED_SHAPE);
    if (n == 0)
        return JETQ_OK;
    JQ_REQUIRE(q_row && s_row && q_col && s_col, JETQ_ERR_INVALID_ARG);
    JQ_REQUIRE(aligned16(q_row) && aligned16(q_col) && (reinterpret_cast<uintptr_t>(s_row) & 3u) == 0 &&
                   (reinterpret_cast<uintptr_t>(s_col) & 3u) == 0 &&
                   (reinterpret_cast<uintptr_t>(seg_offsets) & 7u) == 0,
               JETQ_ERR_MISALIGNED);
    const jetq_status a = check_arch();
    if (a != JETQ_OK)
        return a;
    RequantArgs args{q_row, s_row, n, c, q_col, s_col, ldq_col, seg_offsets, nseg_eff};
    return from_cuda(launch_requant_col(args, static_cast<cudaStream_t>(stream)));
}

jetq_status jetq_dequant_bf16(const uint8_t *q, const float *s, int64_t rows, int64_t cols, jetq_scale_layout layout,
                              uint16_t *out, int64_t ldo, void *stream)
{
    JQ_REQUIRE(layout == JETQ_SCALES_ROWGROUPS_1X128 || layout == JETQ_SCALES_BLOCKS_128X128, JETQ_ERR_INVALID_ARG);
    JQ_REQUIRE(rows >= 0 && cols > 0, JETQ_ERR_INVALID_ARG);
    JQ_REQUIRE(cols % 128 == 0 && ldo >= cols && (layout == JETQ_SCALES_ROWGROUPS_1X128 || rows % 128 == 0),
               JETQ_ERR_UNSUPPORTED_SHAPE);
    if (rows == 0)
        return JETQ_OK;
    JQ_REQUIRE(q && s && out, JETQ_ERR_INVALID_ARG);
    JQ_REQUIRE(aligned16(q) && aligned16(out) && ldo % 8 == 0 && (reinterpret_cast<uintptr_t>(s) & 3u) == 0,
               JETQ_ERR_MISALIGNED);
    const jetq_status a = check_arch();
    if (a != JETQ_OK)
        return a;
    DequantArgs args{q, s, rows, cols, layout == JETQ_SCALES_BLOCKS_128X128, out, ldo};
    return from_cuda(launch_dequant_bf16(args, static_cast<cudaStream_t>(stream)));
}

static jetq_status fprop_impl(jetq_recipe recipe, const uint8_t *qx, const void *sx, const uint8_t *qw,
                              const void *sw, int64_t n, int64_t d, int64_t c, void *y, jetq_out_dtype y_dtype,
                              int64_t ldy, void *workspace, size_t workspace_bytes, jetq_path path, void *stream)
{
    JQ_REQUIRE(recipe == JETQ_RECIPE_BLOCK128 || recipe == JETQ_RECIPE_MXFP8 ||
                   recipe == JETQ_RECIPE_BLOCK128_POW2,
               JETQ_ERR_INVALID_ARG);
    JQ_REQUIRE(path == JETQ_PATH_AUTO || path == JETQ_PATH_TRAIN || path == JETQ_PATH_DECODE, JETQ_ERR_INVALID_ARG);
    JQ_REQUIRE(n >= 0 && d > 0 && c > 0, JETQ_ERR_INVALID_ARG);
    JQ_REQUIRE(d % 128 == 0 && c % 128 == 0, JETQ_ERR_UNSUPPORTED_SHAPE);
    jetq_status st = check_out(y, y_dtype, ldy, d);
    if (st != JETQ_OK)
        return st;
    if (n == 0)
        return JETQ_OK;
    JQ_REQUIRE(qx && sx && qw && sw, JETQ_ERR_INVALID_ARG);
    JQ_REQUIRE(aligned16(qx) && aligned16(qw) && aligned16(sx) && aligned16(sw), JETQ_ERR_MISALIGNED);
    if ((st = check_arch()) != JETQ_OK)
        return st;
    if (recipe != JETQ_RECIPE_BLOCK128) { // E8M0 scale atoms: the block-scaled MMA
        MxGemmProblem m{qx, static_cast<const uint8_t *>(sx), qw, static_cast<const uint8_t *>(sw), n, d, c, c, c,
                        y, ldy, y_dtype, 0};
        return from_cuda(launch_gemm_mx(m, static_cast<cudaStream_t>(stream)));
    }
    GemmProblem g{qx, static_cast<const float *>(sx), qw, static_cast<const float *>(sw), n, d, c, c, c,
                  BScale::Block128, y, ldy, y_dtype, 0};
    const bool decode = path == JETQ_PATH_DECODE || (path == JETQ_PATH_AUTO && n <= 256);
    if (decode && workspace) {
        g.ws = workspace;
        g.ws_bytes = workspace_bytes;
    }
    return from_cuda(launch_gemm_block128(g, decode ? GemmShape::Decode : GemmShape::Train,
                                          static_cast<cudaStream_t>(stream)));
}

jetq_status jetq_gemm_fprop(jetq_recipe recipe, const uint8_t *qx, const void *sx, const uint8_t *qw, const void *sw,
                            int64_t n, int64_t d, int64_t c, void *y, jetq_out_dtype y_dtype, int64_t ldy,
                            jetq_path path, void *stream)
{
    return fprop_impl(recipe, qx, sx, qw, sw, n, d, c, y, y_dtype, ldy, nullptr, 0, path, stream);
}

size_t jetq_decode_workspace_bytes(int64_t n, int64_t d, int64_t c)
{
    if (n < 1 || d <= 0 || c <= 0 || d % 128 != 0 || c % 128 != 0 || check_arch() != JETQ_OK)
        return 0;
    return decode_split_workspace_bytes(n, d, c);
}

jetq_status jetq_gemm_fprop_ws(jetq_recipe recipe, const uint8_t *qx, const void *sx, const uint8_t *qw,
                               const void *sw, int64_t n, int64_t d, int64_t c, void *y, jetq_out_dtype y_dtype,
                               int64_t ldy, void *workspace, size_t workspace_bytes, jetq_path path, void *stream)
{
    JQ_REQUIRE(workspace == nullptr || aligned16(workspace), JETQ_ERR_MISALIGNED);
    return fprop_impl(recipe, qx, sx, qw, sw, n, d, c, y, y_dtype, ldy, workspace, workspace_bytes, path, stream);
}

jetq_status jetq_gemm_fprop_noalloc(const uint8_t *qx, const float *sx, const uint8_t *qw, const float *sw, int64_t n,
                                    int64_t d, int64_t c, void *y, jetq_out_dtype y_dtype, int64_t ldy, void *stream)
{
    JQ_REQUIRE(n >= 0 && d > 0 && c > 0, JETQ_ERR_INVALID_ARG);
    JQ_REQUIRE(d % 128 == 0 && c % 128 == 0, JETQ_ERR_UNSUPPORTED_SHAPE);
    jetq_status st = check_out(y, y_dtype, ldy, d);
    if (st != JETQ_OK)
        return st;
    if (n == 0)
        return JETQ_OK;
    JQ_REQUIRE(qx && sx && qw && sw, JETQ_ERR_INVALID_ARG);
    JQ_REQUIRE(aligned16(qx) && aligned16(qw) && aligned16(sx) && aligned16(sw), JETQ_ERR_MISALIGNED);
    if ((st = check_arch()) != JETQ_OK)
        return st;
    // the built-in array must hold this shape's partial sums
    JQ_REQUIRE(decode_split_workspace_bytes(n, d, c) <= decode_static_scratch_bytes(), JETQ_ERR_UNSUPPORTED_SHAPE);
    GemmProblem g{qx, sx, qw, sw, n, d, c, c, c, BScale::Block128, y, ldy, y_dtype, 0};
    return from_cuda(launch_gemm_decode_static(g, static_cast<cudaStream_t>(stream)));
}

jetq_status jetq_gemm_dgrad(jetq_recipe recipe, const uint8_t *qdy, const void *sdy, const uint8_t *qwt,
                            const void *swt, int64_t n, int64_t d, int64_t c, void *dx, jetq_out_dtype dx_dtype,
                            int64_t lddx, void *stream)
{
    JQ_REQUIRE(recipe == JETQ_RECIPE_BLOCK128 || recipe == JETQ_RECIPE_MXFP8 ||
                   recipe == JETQ_RECIPE_BLOCK128_POW2,
               JETQ_ERR_INVALID_ARG);
    JQ_REQUIRE(n >= 0 && d > 0 && c > 0, JETQ_ERR_INVALID_ARG);
    JQ_REQUIRE(d % 128 == 0 && c % 128 == 0, JETQ_ERR_UNSUPPORTED_SHAPE);
    jetq_status st = check_out(dx, dx_dtype, lddx, c);
    if (st != JETQ_OK)
        return st;
    if (n == 0)
        return JETQ_OK;
    JQ_REQUIRE(qdy && sdy && qwt && swt, JETQ_ERR_INVALID_ARG);
    JQ_REQUIRE(aligned16(qdy) && aligned16(qwt) && aligned16(sdy) && aligned16(swt), JETQ_ERR_MISALIGNED);
    if ((st = check_arch()) != JETQ_OK)
        return st;
    if (recipe != JETQ_RECIPE_BLOCK128) { // E8M0 scale atoms: the block-scaled MMA
        MxGemmProblem m{qdy, static_cast<const uint8_t *>(sdy), qwt, static_cast<const uint8_t *>(swt), n, c, d, d, d,
                        dx, lddx, dx_dtype, 0};
        return from_cuda(launch_gemm_mx(m, static_cast<cudaStream_t>(stream)));
    }
    GemmProblem g{qdy, static_cast<const float *>(sdy), qwt, static_cast<const float *>(swt), n, c, d, d, d,
                  BScale::Block128, dx, lddx, dx_dtype, 0};
    return from_cuda(launch_gemm_block128(g, n <= 256 ? GemmShape::Decode : GemmShape::Train,
                                          static_cast<cudaStream_t>(stream)));
}

jetq_status jetq_gemm_wgrad(jetq_recipe recipe, const uint8_t *qdyc, const void *sdyc, const uint8_t *qxc,
                            const void *sxc, int64_t k, int64_t ldk, int64_t d, int64_t c, float *dw, int64_t lddw,
                            int accumulate, void *stream)
{
    JQ_REQUIRE(recipe == JETQ_RECIPE_BLOCK128 || recipe == JETQ_RECIPE_MXFP8 ||
                   recipe == JETQ_RECIPE_BLOCK128_POW2,
               JETQ_ERR_INVALID_ARG);
    JQ_REQUIRE(k >= 0 && d > 0 && c > 0, JETQ_ERR_INVALID_ARG);
    JQ_REQUIRE(d % 128 == 0 && c % 128 == 0 && k % 128 == 0 && ldk >= k, JETQ_ERR_UNSUPPORTED_SHAPE);
    jetq_status st = check_out(dw, JETQ_OUT_F32, lddw, c);
    if (st != JETQ_OK)
        return st;
    if (k == 0) {
        if (accumulate)
            return JETQ_OK;
        return from_cuda(cudaMemset2DAsync(dw, (size_t)lddw * 4, 0, (size_t)c * 4, (size_t)d,
                                           static_cast<cudaStream_t>(stream)));
    }
    JQ_REQUIRE(qdyc && sdyc && qxc && sxc, JETQ_ERR_INVALID_ARG);
    JQ_REQUIRE(aligned16(qdyc) && aligned16(qxc) && aligned16(sdyc) && aligned16(sxc) && ldk % 16 == 0,
               JETQ_ERR_MISALIGNED);
    if ((st = check_arch()) != JETQ_OK)
        return st;
    if (recipe != JETQ_RECIPE_BLOCK128) { // E8M0 scale atoms: the block-scaled MMA
        MxGemmProblem m{qdyc, static_cast<const uint8_t *>(sdyc), qxc, static_cast<const uint8_t *>(sxc), d, c, k, ldk,
                        ldk, dw, lddw, JETQ_OUT_F32, accumulate ? 1 : 0};
        return from_cuda(launch_gemm_mx(m, static_cast<cudaStream_t>(stream)));
    }
    GemmProblem g{qdyc, static_cast<const float *>(sdyc), qxc, static_cast<const float *>(sxc), d, c, k, ldk, ldk,
                  BScale::PerRow, dw, lddw, JETQ_OUT_F32, accumulate ? 1 : 0};
    return from_cuda(launch_gemm_block128(g, GemmShape::Train, static_cast<cudaStream_t>(stream)));
}

jetq_status jetq_gemm_grouped(jetq_gemm_kind kind, jetq_recipe recipe, const uint8_t *a, const void *sa,
                              const uint8_t *b, const void *sb, int64_t m, int64_t n, int64_t k, int64_t ldk,
                              const int64_t *seg_offsets, int num_experts, void *out, jetq_out_dtype out_dtype,
                              int64_t ldo, int accumulate, void *stream)
{
    JQ_REQUIRE(kind == JETQ_GEMM_FPROP || kind == JETQ_GEMM_DGRAD || kind == JETQ_GEMM_WGRAD, JETQ_ERR_INVALID_ARG);
    JQ_REQUIRE(recipe == JETQ_RECIPE_BLOCK128 || recipe == JETQ_RECIPE_MXFP8 ||
                   recipe == JETQ_RECIPE_BLOCK128_POW2,
               JETQ_ERR_INVALID_ARG);
    JQ_REQUIRE(m >= 0 && n > 0 && k >= 0 && seg_offsets != nullptr, JETQ_ERR_INVALID_ARG);
    JQ_REQUIRE(num_experts >= 1 && num_experts <= 256, JETQ_ERR_UNSUPPORTED_SHAPE);
    JQ_REQUIRE(n % 128 == 0 && k % 128 == 0 && ldk >= k, JETQ_ERR_UNSUPPORTED_SHAPE);
    const bool wgrad = kind == JETQ_GEMM_WGRAD;
    JQ_REQUIRE(!wgrad || m % 128 == 0, JETQ_ERR_UNSUPPORTED_SHAPE);
    JQ_REQUIRE(!(accumulate && (!wgrad || out_dtype != JETQ_OUT_F32)), JETQ_ERR_INVALID_ARG);
    jetq_status st = check_out(out, wgrad ? JETQ_OUT_F32 : out_dtype, ldo, n);
    if (st != JETQ_OK)
        return st;
    if (wgrad)
        JQ_REQUIRE(out_dtype == JETQ_OUT_F32, JETQ_ERR_INVALID_ARG);
    if (m == 0 || (k == 0 && !wgrad))
        return JETQ_OK;
    if (k == 0) { // WGrad over no tokens: every expert's gradient is zero
        if (accumulate)
            return JETQ_OK;
        return from_cuda(cudaMemset2DAsync(out, (size_t)ldo * 4, 0, (size_t)n * 4, (size_t)(m * num_experts),
                                           static_cast<cudaStream_t>(stream)));
    }
    JQ_REQUIRE(a && sa && b && sb, JETQ_ERR_INVALID_ARG);
    JQ_REQUIRE(aligned16(a) && aligned16(b) && aligned16(sa) && aligned16(sb) && ldk % 16 == 0 &&
                   (reinterpret_cast<uintptr_t>(seg_offsets) & 7u) == 0,
               JETQ_ERR_MISALIGNED);
    if ((st = check_arch()) != JETQ_OK)
        return st;
    const cudaStream_t cs = static_cast<cudaStream_t>(stream);
    if (recipe != JETQ_RECIPE_BLOCK128) { // E8M0 scale atoms: the block-scaled MMA
        MxGemmProblem mp{a, static_cast<const uint8_t *>(sa), b, static_cast<const uint8_t *>(sb), m, n, k, ldk, ldk,
                         out, ldo, wgrad ? JETQ_OUT_F32 : out_dtype, accumulate ? 1 : 0};
        mp.group = wgrad ? GroupKind::K : GroupKind::Rows;
        mp.seg = seg_offsets;
        mp.num_experts = num_experts;
        return from_cuda(launch_gemm_mx(mp, cs));
    }
    GemmProblem g{a, static_cast<const float *>(sa), b, static_cast<const float *>(sb), m, n, k, ldk, ldk,
                  wgrad ? BScale::PerRow : BScale::Block128, out, ldo, wgrad ? JETQ_OUT_F32 : out_dtype,
                  accumulate ? 1 : 0};
    g.group = wgrad ? GroupKind::K : GroupKind::Rows;
    g.seg = seg_offsets;
    g.num_experts = num_experts;
    return from_cuda(launch_gemm_block128(g, GemmShape::Train, cs));
}

} // extern "C"
