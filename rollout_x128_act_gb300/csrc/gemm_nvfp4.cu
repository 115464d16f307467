// NVFP4 GEMM on sm_103a tensor cores (kind::mxf4nvf4, native block scaling).
//
//   out[m, n] = fl32(fl32(sga[m] * sgb) * acc[m, n])
//   acc[m, n] = sum_k (e2m1(qa[m, k]) * e4m3(sfa[m, k/16])) * (e2m1(qb[n, k]) * e4m3(sfb[n, k/16]))
//
// The Miles post on Blackwell-native RL recipes (NVFP4 section) quantizes MoE
// expert operands to E2M1 with one E4M3 scale per 16 values and one FP32
// scale for a larger scope (per token for activations, per tensor for
// weights), and traces part of its training gap to applying the per-token
// scale as a separate step outside the GEMM.  Here it is inside: the block
// scales ride the tensor core's block-scaled MMA
// (scale_vec::4X: four E4M3 scales per 64-element K step), the whole K loop
// accumulates in TMEM, and the epilogue applies the two FP32 scope scales once.
//
//   warp 0    TMA producer: A and B K-block tiles (256 FP4 values = 128 bytes a
//             row, 128-byte swizzle) and the K-block's scale atoms (1-D bulk
//             copies) into a STAGES-deep shared-memory ring
//   warp 1    MMA issuer: tcgen05.cp of the stage's scale atoms into TMEM, then
//             4 x tcgen05.mma.kind::mxf4nvf4.block_scale.scale_vec::4X (K = 64)
//             into the tile accumulator; commits release the stage and, after
//             the last K-block, signal the epilogue
//   warps 4.. epilogue: TMEM -> registers, release the accumulator (the next
//             tile's MMAs start), scale by the scope scales, store
//
// Scale atoms (the layout the block-scaled MMA reads through tcgen05.cp
// 32x128b.warpx4): for K-block kb (256 values), 128-row band rb and 64-value
// step s, a 512-byte atom at ((kb * RB + rb) * 4 + s) * 512 holding byte
// (r % 32) * 16 + ((r % 128) / 32) * 4 + (k % 64) / 16 for row r, column k.
// k_nvfp4_atoms builds it from the quantizer's row-major block scales.
//
// TMEM: accumulator in columns [0, 256); scale factors of stage s at 256 + 48 s
// (A: 4 steps x 4 columns, B: 4 steps x 8 columns).  Every wait is bounded.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "jetq_internal.h"
#include "ptx.cuh"
#include "sched.cuh"

namespace jetq {

__device__ unsigned g_gemm_nvfp4_error;

namespace {

constexpr unsigned kErrTimeout = 1u;
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

struct Nvf4Params {
    int mt, nt, num_kb;
    int64_t M;
    int N;
    const uint8_t *sfa, *sfb;
    int rba, rbb;            // 128-row bands of A and B
    const float *sga;        // [M] (per-row scope) or [1]
    const float *sgb;        // [1]
    int per_row_a;
    int box_a_rows, box_b_rows;
    void *out;
    int64_t ldo;
    int out_bf16;
    unsigned long long limit_ns;
};

template <int BN, int EPI_WARPS, int STAGES>
struct Nvf4Cfg {
    static constexpr int kABytes = 128 * 128;
    static constexpr int kBBytes = BN * 128;
    static constexpr int kStage = kABytes + kBBytes;
    static constexpr int kSfaBytes = 4 * 512;              // 4 steps x one band
    static constexpr int kSfbBytes = (BN / 128) * 4 * 512; // 4 steps x BN/128 bands
    static constexpr int kSfStage = kSfaBytes + kSfbBytes;
    static constexpr int kThreads = 128 + 32 * EPI_WARPS;
    static constexpr int kCols = BN / (EPI_WARPS / 4);
    static constexpr int kSfCols = 4 * 4 + 4 * 4 * (BN / 128); // TMEM columns per stage
    static constexpr int kTmemCols = 512;
    static constexpr int kBars = 2 * STAGES + 3;
    static constexpr size_t kSmem = 1024 + (size_t)STAGES * kStage + (size_t)STAGES * kSfStage + 256;
    static_assert(BN % 128 == 0 && BN <= 256, "B tile is whole 128-row scale bands");
    static_assert(BN + STAGES * kSfCols <= kTmemCols, "TMEM budget");
    static_assert(kCols % 32 == 0, "epilogue split");
    static_assert(kBars * 8 + 16 <= 256, "barrier area");
    static_assert(kSmem <= 232448, "shared memory");
};

// Instruction descriptor, kind::mxf4nvf4 block-scaled: E2M1 x E2M1 -> F32,
// UE4M3 scale factors (scale_vec::4X uses the whole 32-bit scale word, so both
// scale-factor ids are 0), both operands K-major.
__host__ __device__ constexpr uint32_t idesc_nvf4(int m, int n)
{
    return (1u << 7) | (1u << 10)           // A, B format: E2M1
           | ((uint32_t)(n >> 3) << 17)     // N / 8
           | (0u << 23)                     // scale format: UE4M3
           | ((uint32_t)(m >> 4) << 24);    // M / 16
}

__device__ __forceinline__ void mma_mxf4nvf4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                             uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
            d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

template <int BN, int EPI_WARPS, int STAGES>
__global__ void __launch_bounds__(128 + 32 * EPI_WARPS, 1)
    k_gemm_nvfp4(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, const Nvf4Params p)
{
    using C = Nvf4Cfg<BN, EPI_WARPS, STAGES>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *tiles = ptx::align_smem<1024>(smem_raw);
    uint8_t *sf = tiles + (size_t)STAGES * C::kStage; // STAGES x (SFA atoms, SFB atoms)
    uint64_t *bars = reinterpret_cast<uint64_t *>(sf + (size_t)STAGES * C::kSfStage);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + C::kBars);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const uint32_t bar0 = ptx::smem_addr(bars);
    auto full = [&](int s) { return bar0 + 8u * s; };
    auto empty = [&](int s) { return bar0 + 8u * (STAGES + s); };
    const uint32_t acc_full = bar0 + 8u * (2 * STAGES);
    const uint32_t acc_empty = acc_full + 8u;
    const uint32_t done = acc_full + 16u;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    unsigned *err = &g_gemm_nvfp4_error;
    const int num_tiles = p.mt * p.nt;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(full(s), 1);
            ptx::mbar_init(empty(s), 1);
        }
        ptx::mbar_init(acc_full, 1);
        ptx::mbar_init(acc_empty, EPI_WARPS);
        ptx::mbar_init(done, 1);
        *abort_flag = 0;
        ptx::fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tensormap(&tmA);
        ptx::prefetch_tensormap(&tmB);
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_addr(tmem_slot), C::kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp < 4) {
        if (warp == 0 && lane == 0) {
            // -------------------------------------------------- TMA producer
            uint32_t it = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
                int mi, ni;
                dense_coords(t, p.mt, p.nt, mi, ni);
                const int b_bands = min(BN / 128, p.rbb - ni * (BN / 128));
                const uint32_t tx = (uint32_t)((p.box_a_rows + p.box_b_rows) * 128 + C::kSfaBytes +
                                               b_bands * 4 * 512);
                for (int kb = 0; kb < p.num_kb; ++kb, ++it) {
                    const int s = (int)(it % STAGES);
                    const uint32_t ph = (it / STAGES) & 1u;
                    if (!ptx::mbar_wait(empty(s), ph ^ 1u, abort_flag, err, kErrTimeout, p.limit_ns)) {
                        ok = false;
                        break;
                    }
                    ptx::mbar_arrive_expect_tx(full(s), tx);
                    const uint32_t dst = ptx::smem_addr(tiles + (size_t)s * C::kStage);
                    ptx::tma_load_2d(dst, &tmA, full(s), kb * 128, mi * 128);
                    ptx::tma_load_2d(dst + C::kABytes, &tmB, full(s), kb * 128, ni * BN);
                    const uint32_t sdst = ptx::smem_addr(sf + (size_t)s * C::kSfStage);
                    ptx::bulk_load(sdst, p.sfa + ((int64_t)kb * p.rba + mi) * 4 * 512, (uint32_t)C::kSfaBytes,
                                   full(s));
                    ptx::bulk_load(sdst + C::kSfaBytes, p.sfb + ((int64_t)kb * p.rbb + ni * (BN / 128)) * 4 * 512,
                                   (uint32_t)b_bands * 4u * 512u, full(s));
                }
            }
            for (int s = 0; s < STAGES; ++s) {
                if (it > (uint32_t)s) {
                    const uint32_t last = (uint32_t)s + ((it - 1u - (uint32_t)s) / STAGES) * STAGES;
                    ptx::mbar_wait(full(s), (last / STAGES) & 1u, abort_flag, err, kErrTimeout, p.limit_ns, false);
                }
            }
        } else if (warp == 1 && lane == 0) {
            // -------------------------------------------------- MMA issuer
            constexpr uint32_t idesc = idesc_nvf4(128, BN);
            uint32_t it = 0, tc = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x, ++tc) {
                if (!ptx::mbar_wait(acc_empty, (tc & 1u) ^ 1u, abort_flag, err, kErrTimeout, p.limit_ns))
                    break;
                ptx::tc_fence_after();
                for (int kb = 0; kb < p.num_kb; ++kb, ++it) {
                    const int s = (int)(it % STAGES);
                    const uint32_t ph = (it / STAGES) & 1u;
                    if (!ptx::mbar_wait(full(s), ph, abort_flag, err, kErrTimeout, p.limit_ns)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t sf_smem = ptx::smem_addr(sf + (size_t)s * C::kSfStage);
                    const uint32_t sfa_t = tmem_base + (uint32_t)(BN + s * C::kSfCols);
                    const uint32_t sfb_t = sfa_t + 16u;
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        ptx::tmem_cp_32x128b_warpx4(sfa_t + 4u * k, ptx::desc_kmajor_noswizzle_16b(sf_smem + 512u * k));
#pragma unroll
                        for (int band = 0; band < BN / 128; ++band)
                            ptx::tmem_cp_32x128b_warpx4(
                                sfb_t + (uint32_t)(k * 4 * (BN / 128) + 4 * band),
                                ptx::desc_kmajor_noswizzle_16b(sf_smem + C::kSfaBytes + 2048u * band + 512u * k));
                    }
                    const uint32_t a_addr = ptx::smem_addr(tiles + (size_t)s * C::kStage);
                    const uint64_t adesc = ptx::desc_kmajor_sw128(a_addr);
                    const uint64_t bdesc = ptx::desc_kmajor_sw128(a_addr + C::kABytes);
#pragma unroll
                    for (int k = 0; k < 4; ++k) // 64 FP4 values (32 bytes) per MMA
                        mma_mxf4nvf4(tmem_base, adesc + 2u * k, bdesc + 2u * k, idesc, sfa_t + 4u * k,
                                     sfb_t + (uint32_t)(k * 4 * (BN / 128)), (kb > 0 || k > 0) ? 1u : 0u);
                    ptx::mma_commit(empty(s));
                }
                if (!ok)
                    break;
                ptx::mma_commit(acc_full);
            }
            ptx::mma_commit(done);
            ptx::mbar_wait(done, 0u, abort_flag, err, kErrTimeout, p.limit_ns, false);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------ epilogue
        const int ew = warp - 4;
        const int quarter = warp & 3;
        const int col0 = (ew >> 2) * C::kCols;
        const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
        const float sgb = __ldg(p.sgb);
        uint32_t tc = 0;
        for (int t = blockIdx.x; t < num_tiles; t += gridDim.x, ++tc) {
            int mi, ni;
            dense_coords(t, p.mt, p.nt, mi, ni);
            const int64_t m = (int64_t)mi * 128 + quarter * 32 + lane;
            const int n0 = ni * BN + col0;
            const float sga = m < p.M ? __ldg(p.sga + (p.per_row_a ? m : 0)) : 0.0f;
            const float s = __fmul_rn(sga, sgb);
            const bool got = ptx::mbar_wait(acc_full, tc & 1u, abort_flag, err, kErrTimeout, p.limit_ns);
            if (!__all_sync(0xFFFFFFFFu, got))
                break;
            ptx::tc_fence_after();
            uint32_t v[C::kCols];
#pragma unroll
            for (int ch = 0; ch < C::kCols / 32; ++ch)
                ptx::tmem_ld_32x32b_x32(tmem_base + lane_addr + (uint32_t)(col0 + ch * 32),
                                        *reinterpret_cast<uint32_t(*)[32]>(&v[ch * 32]));
            ptx::tmem_ld_wait();
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0)
                ptx::mbar_arrive(acc_empty); // the MMA may start the next tile
            if (m < p.M && n0 < p.N) {
                if (p.out_bf16) {
                    __nv_bfloat16 *o = reinterpret_cast<__nv_bfloat16 *>(p.out) + m * p.ldo + n0;
#pragma unroll
                    for (int j8 = 0; j8 < C::kCols / 8; ++j8) {
                        uint4 w;
                        uint32_t *wp = reinterpret_cast<uint32_t *>(&w);
#pragma unroll
                        for (int h = 0; h < 4; ++h) {
                            const float2 y = __fmul2_rn(make_float2(__uint_as_float(v[8 * j8 + 2 * h]),
                                                                    __uint_as_float(v[8 * j8 + 2 * h + 1])),
                                                        make_float2(s, s));
                            const __nv_bfloat162 b2 = __floats2bfloat162_rn(y.x, y.y);
                            wp[h] = *reinterpret_cast<const uint32_t *>(&b2);
                        }
                        *reinterpret_cast<uint4 *>(o + 8 * j8) = w;
                    }
                } else {
                    float *o = reinterpret_cast<float *>(p.out) + m * p.ldo + n0;
#pragma unroll
                    for (int j4 = 0; j4 < C::kCols / 4; ++j4) {
                        const float2 y0 = __fmul2_rn(
                            make_float2(__uint_as_float(v[4 * j4]), __uint_as_float(v[4 * j4 + 1])), make_float2(s, s));
                        const float2 y1 = __fmul2_rn(
                            make_float2(__uint_as_float(v[4 * j4 + 2]), __uint_as_float(v[4 * j4 + 3])),
                            make_float2(s, s));
                        *reinterpret_cast<float4 *>(o + 4 * j4) = make_float4(y0.x, y0.y, y1.x, y1.y);
                    }
                }
            }
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_base, C::kTmemCols);
    }
}

// Row-major E4M3 block scales [rows x k/16] -> scale atoms (layout above); one
// thread per 32-bit word (row r, 64-value step); rows past `rows` in the last
// band are zero.
__global__ void k_nvfp4_atoms(const uint8_t *sb, int64_t rows, int64_t k, uint8_t *atoms)
{
    const int64_t steps = k / 64;
    const int64_t rb_count = (rows + 127) / 128;
    const int64_t total = rb_count * 128 * steps;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = i / steps, sg = i % steps;
        const uint32_t w = r < rows ? *reinterpret_cast<const uint32_t *>(sb + r * (k / 16) + 4 * sg) : 0u;
        const int64_t kb = sg / 4, s = sg % 4;
        const int64_t off = ((kb * rb_count + r / 128) * 4 + s) * 512 + (r % 32) * 16 + ((r % 128) / 32) * 4;
        *reinterpret_cast<uint32_t *>(atoms + off) = w;
    }
}

template <int BN, int EPI_WARPS, int STAGES>
cudaError_t run_nvfp4(const Nvfp4GemmProblem &g, cudaStream_t st)
{
    using C = Nvf4Cfg<BN, EPI_WARPS, STAGES>;
    auto kern = k_gemm_nvfp4<BN, EPI_WARPS, STAGES>;
    static int configured_device = -1;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (configured_device != dev) {
        if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::kSmem)) !=
            cudaSuccess)
            return e;
        configured_device = dev;
    }
    const int box_a = g.M >= 128 ? 128 : (int)((g.M + 7) / 8 * 8);
    const int box_b = g.N >= BN ? BN : (int)((g.N + 7) / 8 * 8);
    CUtensorMap ta, tbm;
    // packed codes: K/2 bytes a row, 128-byte (256-value) K-blocks
    if ((e = make_kmajor_map(&ta, g.a, g.K / 2, g.M, g.K / 2, box_a)) != cudaSuccess)
        return e;
    if ((e = make_kmajor_map(&tbm, g.b, g.K / 2, g.N, g.K / 2, box_b)) != cudaSuccess)
        return e;
    Nvf4Params kp;
    kp.mt = (int)((g.M + 127) / 128);
    kp.nt = (int)((g.N + BN - 1) / BN);
    kp.num_kb = (int)(g.K / 256);
    kp.M = g.M;
    kp.N = (int)g.N;
    kp.sfa = g.sfa;
    kp.sfb = g.sfb;
    kp.rba = (int)((g.M + 127) / 128);
    kp.rbb = (int)((g.N + 127) / 128);
    kp.sga = g.sga;
    kp.sgb = g.sgb;
    kp.per_row_a = g.per_row_a;
    kp.box_a_rows = box_a;
    kp.box_b_rows = box_b;
    kp.out = g.out;
    kp.ldo = g.ldo;
    kp.out_bf16 = g.out_dtype == JETQ_OUT_BF16;
    kp.limit_ns = kWaitLimitNs;
    const int tiles = kp.mt * kp.nt;
    const int grid = tiles < sm_count() ? tiles : sm_count();
    kern<<<grid, C::kThreads, C::kSmem, st>>>(ta, tbm, kp);
    return cudaGetLastError();
}

} // namespace

cudaError_t launch_gemm_nvfp4(const Nvfp4GemmProblem &g, cudaStream_t st)
{
    if (g.M == 0)
        return cudaSuccess;
    return run_nvfp4<256, 8, 4>(g, st);
}

cudaError_t launch_nvfp4_atoms(const uint8_t *sb, int64_t rows, int64_t k, uint8_t *atoms, cudaStream_t st)
{
    const int64_t words = (rows + 127) / 128 * 128 * (k / 64);
    if (words == 0)
        return cudaSuccess;
    int64_t blocks = (words + 255) / 256;
    const int64_t cap = (int64_t)sm_count() * 8;
    if (blocks > cap)
        blocks = cap;
    k_nvfp4_atoms<<<(unsigned)blocks, 256, 0, st>>>(sb, rows, k, atoms);
    return cudaGetLastError();
}

cudaError_t gemm_nvfp4_read_and_clear_error(cudaStream_t st, unsigned *out)
{
    unsigned v = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(&v, g_gemm_nvfp4_error, sizeof v, 0, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(st);
    if (e != cudaSuccess)
        return e;
    *out |= v;
    if (v) {
        const unsigned zero = 0;
        e = cudaMemcpyToSymbolAsync(g_gemm_nvfp4_error, &zero, sizeof zero, 0, cudaMemcpyHostToDevice, st);
        if (e == cudaSuccess)
            e = cudaStreamSynchronize(st);
    }
    return e;
}

} // namespace jetq
