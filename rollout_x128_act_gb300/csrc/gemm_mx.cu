// MXFP8 GEMM on sm_103a tensor cores (kind::mxf8f6f4, native block scaling).
//
//   out[m, n] = sum_k (2^ea[m, k/32] * qa[m, k]) * (2^eb[n, k/32] * qb[n, k])
//
// The Blackwell MXFP8 recipe (Miles Blackwell-recipes post, MXFP8 section:
// one E8M0 scale per 32 consecutive E4M3 values) is what the tensor core's
// block-scaled MMA consumes directly, so unlike the FP32-scale recipe the
// whole K loop accumulates in TMEM and the epilogue runs once per tile.
//
//   warp 0    TMA producer: A and B K-block tiles (128-byte swizzle) plus the
//             K-block's scale atoms (one 512-byte atom per 128 rows, a 1-D bulk
//             copy each) into a STAGES-deep shared-memory ring
//   warp 1    MMA issuer: tcgen05.cp of the stage's scale atoms into TMEM, then
//             4 x tcgen05.mma.kind::mxf8f6f4.block_scale (K = 32, scale byte =
//             sub-block) into the tile accumulator; tcgen05.commit releases the
//             stage, and after the last K-block signals the epilogue
//   warps 4.. epilogue: TMEM -> registers, release the accumulator (the next
//             tile's MMAs start), convert and store
//
// TMEM: accumulator in columns [0, BN); scale factors of stage s at
// BN + 12 s (A: 4 columns, B: 8 columns).  Every wait is bounded as in the
// 128-block GEMM.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "jetq_internal.h"
#include "ptx.cuh"

namespace jetq {

__device__ unsigned g_gemm_mx_error;

namespace {

constexpr int kGroupM = 8;
constexpr unsigned kErrTimeout = 1u;
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

struct MxParams {
    const uint8_t *sfa;
    const uint8_t *sfb;
    int64_t M, N;
    int num_kb;
    int mt, nt;
    int rba, rbb; // row bands of A and B (atoms per K-block)
    int box_a_rows, box_b_rows;
    void *out;
    int64_t ldo;
    int out_bf16;
    int accumulate;
    unsigned long long limit_ns;
};

__device__ __forceinline__ void tile_coords(int t, int mt, int nt, int &mi, int &ni)
{
    const int group = kGroupM * nt;
    const int first_m = (t / group) * kGroupM;
    const int gm = min(mt - first_m, kGroupM);
    const int r = t % group;
    mi = first_m + r % gm;
    ni = r / gm;
}

template <int BN, int EPI_WARPS, int STAGES>
struct MxCfg {
    static constexpr int kABytes = 128 * 128;
    static constexpr int kBBytes = BN * 128;
    static constexpr int kStage = kABytes + kBBytes;
    static constexpr int kSfaBytes = 512;
    static constexpr int kSfbBytes = (BN / 128) * 512;
    static constexpr int kSfStage = kSfaBytes + kSfbBytes;
    static constexpr int kThreads = 128 + 32 * EPI_WARPS;
    static constexpr int kCols = BN / (EPI_WARPS / 4);
    static constexpr int kSfCols = 4 + 4 * (BN / 128); // TMEM columns per stage
    static constexpr int kTmemCols = 512;
    static constexpr int kBars = 2 * STAGES + 3;
    static constexpr size_t kSmem = 1024 + (size_t)STAGES * kStage + (size_t)STAGES * kSfStage + 1024;
    static_assert(BN % 128 == 0 && BN <= 256, "B tile is whole 128-row scale bands");
    static_assert(BN + STAGES * kSfCols <= kTmemCols, "TMEM budget");
    static_assert(kCols % 32 == 0, "epilogue split");
};

template <int BN, int EPI_WARPS, int STAGES>
__global__ void __launch_bounds__(128 + 32 * EPI_WARPS, 1)
    k_gemm_mx(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, const MxParams p)
{
    using C = MxCfg<BN, EPI_WARPS, STAGES>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *tiles = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t *sf = tiles + (size_t)STAGES * C::kStage; // STAGES x (SFA atom, SFB atoms)
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
    const int num_tiles = p.mt * p.nt;
    unsigned *err = &g_gemm_mx_error;

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
            for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
                int mi, ni;
                tile_coords(tile, p.mt, p.nt, mi, ni);
                const int b_bands = min(BN / 128, p.rbb - ni * (BN / 128)); // scale atoms that exist
                const uint32_t tx = (uint32_t)((p.box_a_rows + p.box_b_rows) * 128 + 512 + b_bands * 512);
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
                    ptx::bulk_load(sdst, p.sfa + ((int64_t)kb * p.rba + mi) * 512, 512u, full(s));
                    ptx::bulk_load(sdst + C::kSfaBytes, p.sfb + ((int64_t)kb * p.rbb + ni * (BN / 128)) * 512,
                                   (uint32_t)b_bands * 512u, full(s));
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
            uint32_t it = 0, tc = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x, ++tc) {
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
                    const uint32_t sfb_t = sfa_t + 4u;
                    ptx::tmem_cp_32x128b_warpx4(sfa_t, ptx::desc_kmajor_noswizzle_16b(sf_smem));
#pragma unroll
                    for (int band = 0; band < BN / 128; ++band)
                        ptx::tmem_cp_32x128b_warpx4(sfb_t + 4u * band,
                                                    ptx::desc_kmajor_noswizzle_16b(sf_smem + C::kSfaBytes + 512u * band));
                    const uint32_t a_addr = ptx::smem_addr(tiles + (size_t)s * C::kStage);
                    const uint64_t adesc = ptx::desc_kmajor_sw128(a_addr);
                    const uint64_t bdesc = ptx::desc_kmajor_sw128(a_addr + C::kABytes);
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        ptx::mma_mxf8f6f4(tmem_base, adesc + 2u * k, bdesc + 2u * k, ptx::idesc_mx_e4m3(128, BN, k),
                                          sfa_t, sfb_t, (kb > 0 || k > 0) ? 1u : 0u);
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
        uint32_t tc = 0;
        for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++tc) {
            int mi, ni;
            tile_coords(tile, p.mt, p.nt, mi, ni);
            const int64_t m = (int64_t)mi * 128 + quarter * 32 + lane;
            const int64_t n0 = (int64_t)ni * BN + col0;
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
                            const __nv_bfloat162 b2 = __floats2bfloat162_rn(__uint_as_float(v[8 * j8 + 2 * h]),
                                                                            __uint_as_float(v[8 * j8 + 2 * h + 1]));
                            wp[h] = *reinterpret_cast<const uint32_t *>(&b2);
                        }
                        *reinterpret_cast<uint4 *>(o + 8 * j8) = w;
                    }
                } else {
                    float *o = reinterpret_cast<float *>(p.out) + m * p.ldo + n0;
#pragma unroll
                    for (int j4 = 0; j4 < C::kCols / 4; ++j4) {
                        float4 w = make_float4(__uint_as_float(v[4 * j4]), __uint_as_float(v[4 * j4 + 1]),
                                               __uint_as_float(v[4 * j4 + 2]), __uint_as_float(v[4 * j4 + 3]));
                        if (p.accumulate) {
                            const float4 old = *reinterpret_cast<const float4 *>(o + 4 * j4);
                            w.x = __fadd_rn(old.x, w.x);
                            w.y = __fadd_rn(old.y, w.y);
                            w.z = __fadd_rn(old.z, w.z);
                            w.w = __fadd_rn(old.w, w.w);
                        }
                        *reinterpret_cast<float4 *>(o + 4 * j4) = w;
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

template <int BN, int EPI_WARPS, int STAGES>
cudaError_t run_mx(const MxGemmProblem &g, cudaStream_t st)
{
    using C = MxCfg<BN, EPI_WARPS, STAGES>;
    auto kern = k_gemm_mx<BN, EPI_WARPS, STAGES>;
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
    if ((e = make_kmajor_map(&ta, g.a, g.K, g.M, g.lda, box_a)) != cudaSuccess)
        return e;
    if ((e = make_kmajor_map(&tbm, g.b, g.K, g.N, g.ldb, box_b)) != cudaSuccess)
        return e;
    MxParams kp;
    kp.sfa = g.sfa;
    kp.sfb = g.sfb;
    kp.M = g.M;
    kp.N = g.N;
    kp.num_kb = (int)(g.K / 128);
    kp.mt = (int)((g.M + 127) / 128);
    kp.nt = (int)((g.N + BN - 1) / BN);
    kp.rba = (int)((g.M + 127) / 128);
    kp.rbb = (int)((g.N + 127) / 128);
    kp.box_a_rows = box_a;
    kp.box_b_rows = box_b;
    kp.out = g.out;
    kp.ldo = g.ldo;
    kp.out_bf16 = g.out_dtype == JETQ_OUT_BF16;
    kp.accumulate = g.accumulate;
    kp.limit_ns = kWaitLimitNs;
    const int tiles = kp.mt * kp.nt;
    const int grid = tiles < sm_count() ? tiles : sm_count();
    kern<<<grid, C::kThreads, C::kSmem, st>>>(ta, tbm, kp);
    return cudaGetLastError();
}

} // namespace

cudaError_t launch_gemm_mx(const MxGemmProblem &g, cudaStream_t st)
{
    if (g.M == 0)
        return cudaSuccess;
    return run_mx<256, 8, 4>(g, st);
}

cudaError_t gemm_mx_read_and_clear_error(cudaStream_t st, unsigned *out)
{
    unsigned v = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(&v, g_gemm_mx_error, sizeof v, 0, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(st);
    if (e != cudaSuccess)
        return e;
    *out |= v;
    if (v) {
        const unsigned zero = 0;
        e = cudaMemcpyToSymbolAsync(g_gemm_mx_error, &zero, sizeof zero, 0, cudaMemcpyHostToDevice, st);
        if (e == cudaSuccess)
            e = cudaStreamSynchronize(st);
    }
    return e;
}

} // namespace jetq
