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
//   warp 2    grouped FProp/DGrad only: an expert's rows need not start on a
//             128-row scale band, so the A scale words of the tile's 128 rows
//             are gathered into an atom in shared memory
//   warp 3    builds the per-expert tile tables of a grouped launch
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
#include "sched.cuh"

namespace jetq {

__device__ unsigned g_gemm_mx_error;

namespace {

constexpr unsigned kErrTimeout = 1u;
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

struct MxParams {
    Sched sched;
    const uint8_t *sfa;
    const uint8_t *sfb;
    int rba, rbb;          // row bands of A and B (atoms per K-block)
    int64_t sfb_e_stride;  // bytes between experts' B scale atoms (grouped rows)
    int box_a_rows, box_b_rows;
    void *out;
    int64_t ldo;
    int64_t out_e_stride;  // elements between experts' outputs (grouped K)
    int out_bf16;
    int accumulate;
    unsigned long long limit_ns;
};

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
    static constexpr size_t kSmem =
        1024 + (size_t)STAGES * kStage + (size_t)STAGES * kSfStage + 1024 + sizeof(GroupTables);
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
    uint8_t *tiles = ptx::align_smem<1024>(smem_raw);
    uint8_t *sf = tiles + (size_t)STAGES * C::kStage; // STAGES x (SFA atom, SFB atoms)
    uint64_t *bars = reinterpret_cast<uint64_t *>(sf + (size_t)STAGES * C::kSfStage);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + C::kBars);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    GroupTables *gt = reinterpret_cast<GroupTables *>(reinterpret_cast<uint8_t *>(bars) + 1024);

    const uint32_t bar0 = ptx::smem_addr(bars);
    auto full = [&](int s) { return bar0 + 8u * s; };
    auto empty = [&](int s) { return bar0 + 8u * (STAGES + s); };
    const uint32_t acc_full = bar0 + 8u * (2 * STAGES);
    const uint32_t acc_empty = acc_full + 8u;
    const uint32_t done = acc_full + 16u;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const Sched &sc = p.sched;
    const bool gather_a = sc.mode == kGroupedRows; // A scale atoms are assembled by warp 2
    unsigned *err = &g_gemm_mx_error;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(full(s), gather_a ? 2 : 1);
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
    if (warp == 3 && sc.mode != kDense)
        build_group_tables(sc, gt);
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int num_tiles = total_tiles(sc, gt);

    if (warp < 4) {
        if (warp == 0 && lane == 0) {
            // -------------------------------------------------- TMA producer
            uint32_t it = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
                const TileInfo ti = get_tile(sc, gt, t);
                const int brb0 = ti.n0 / 128; // first B scale band inside the (expert's) B operand
                const int b_bands = min(BN / 128, p.rbb - brb0);
                const uint8_t *sfb_e = p.sfb + (int64_t)ti.e * p.sfb_e_stride;
                const uint32_t tx = (uint32_t)((p.box_a_rows + p.box_b_rows) * 128 + (gather_a ? 0 : 512) +
                                               b_bands * 512);
                for (int kb = 0; kb < ti.num_kb; ++kb, ++it) {
                    const int s = (int)(it % STAGES);
                    const uint32_t ph = (it / STAGES) & 1u;
                    if (!ptx::mbar_wait(empty(s), ph ^ 1u, abort_flag, err, kErrTimeout, p.limit_ns)) {
                        ok = false;
                        break;
                    }
                    const int kg = ti.kb0 + kb;
                    ptx::mbar_arrive_expect_tx(full(s), tx);
                    const uint32_t dst = ptx::smem_addr(tiles + (size_t)s * C::kStage);
                    ptx::tma_load_2d(dst, &tmA, full(s), kg * 128, ti.a_row0);
                    ptx::tma_load_2d(dst + C::kABytes, &tmB, full(s), kg * 128, ti.b_row0);
                    const uint32_t sdst = ptx::smem_addr(sf + (size_t)s * C::kSfStage);
                    if (!gather_a)
                        ptx::bulk_load(sdst, p.sfa + ((int64_t)kg * p.rba + ti.a_row0 / 128) * 512, 512u, full(s));
                    ptx::bulk_load(sdst + C::kSfaBytes, sfb_e + ((int64_t)kg * p.rbb + brb0) * 512,
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
            for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x, ++tc) {
                const TileInfo ti = get_tile(sc, gt, t);
                if (!ptx::mbar_wait(acc_empty, (tc & 1u) ^ 1u, abort_flag, err, kErrTimeout, p.limit_ns))
                    break;
                ptx::tc_fence_after();
                for (int kb = 0; kb < ti.num_kb; ++kb, ++it) {
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
                ptx::mma_commit(acc_full); // also for an empty expert: the epilogue writes zeros
            }
            ptx::mma_commit(done);
            ptx::mbar_wait(done, 0u, abort_flag, err, kErrTimeout, p.limit_ns, false);
        } else if (warp == 2 && gather_a) {
            // -------------------------------------------------- A scale gather (grouped rows)
            // row a_row0 + i (i = lane + 32 j) of the tile -> byte lane * 16 + j * 4 of the atom.
            // The words of the next kGather K-blocks of the CTA's (tile, K-block)
            // sequence are loaded while a group is stored, so the global-load
            // latency is paid once per group.
            constexpr int kGather = 4;
            int ft = blockIdx.x, fkb = 0; // fetch cursor
            TileInfo fti{};
            bool fvalid = ft < num_tiles;
            if (fvalid)
                fti = get_tile(sc, gt, ft);
            auto settle = [&]() { // skip to the next (tile, K-block) that exists
                while (fvalid && fkb >= fti.num_kb) {
                    ft += gridDim.x;
                    fkb = 0;
                    fvalid = ft < num_tiles;
                    if (fvalid)
                        fti = get_tile(sc, gt, ft);
                }
            };
            auto fetch = [&](uint32_t (&w)[4]) {
                settle();
                if (!fvalid) {
                    w[0] = w[1] = w[2] = w[3] = 0u;
                    return;
                }
                const int64_t kg = fti.kb0 + fkb;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int64_t r = (int64_t)fti.a_row0 + lane + 32 * j;
                    w[j] = r < sc.M ? __ldg(reinterpret_cast<const uint32_t *>(
                                          p.sfa + (kg * p.rba + (r >> 7)) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4))
                                    : 0u;
                }
                ++fkb;
            };
            uint32_t total = 0; // the CTA's K-blocks
            for (int t = blockIdx.x; t < num_tiles; t += gridDim.x)
                total += (uint32_t)get_tile(sc, gt, t).num_kb;
            uint32_t cur[kGather][4];
#pragma unroll
            for (int u = 0; u < kGather; ++u)
                fetch(cur[u]);
            bool ok = true;
            for (uint32_t it0 = 0; it0 < total && ok; it0 += kGather) {
                uint32_t nxt[kGather][4];
#pragma unroll
                for (int u = 0; u < kGather; ++u)
                    fetch(nxt[u]);
#pragma unroll
                for (int u = 0; u < kGather; ++u) {
                    const uint32_t it = it0 + (uint32_t)u;
                    if (it < total && ok) {
                        const int s = (int)(it % STAGES);
                        const uint32_t ph = (it / STAGES) & 1u;
                        const bool got = ptx::mbar_wait(empty(s), ph ^ 1u, abort_flag, err, kErrTimeout, p.limit_ns);
                        if (!__all_sync(0xFFFFFFFFu, got)) {
                            ok = false;
                        } else {
                            *reinterpret_cast<uint4 *>(sf + (size_t)s * C::kSfStage + lane * 16) =
                                make_uint4(cur[u][0], cur[u][1], cur[u][2], cur[u][3]);
                            asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); // visible to tcgen05.cp
                            __syncwarp();
                            if (lane == 0)
                                ptx::mbar_arrive(full(s));
                        }
                    }
                }
#pragma unroll
                for (int u = 0; u < kGather; ++u)
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        cur[u][j] = nxt[u][j];
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------ epilogue
        const int ew = warp - 4;
        const int quarter = warp & 3;
        const int col0 = (ew >> 2) * C::kCols;
        const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
        uint32_t tc = 0;
        for (int t = blockIdx.x; t < num_tiles; t += gridDim.x, ++tc) {
            const TileInfo ti = get_tile(sc, gt, t);
            const int64_t m = (int64_t)ti.a_row0 + quarter * 32 + lane;
            const int n0 = ti.n0 + col0;
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
            if (ti.num_kb == 0) {            // an expert without rows: its gradient is zero
#pragma unroll
                for (int j = 0; j < C::kCols; ++j)
                    v[j] = 0u;
            }
            if (m < ti.m_end && n0 < sc.N) {
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
                    float *o = reinterpret_cast<float *>(p.out) + ti.e * p.out_e_stride + m * p.ldo + n0;
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
    const int64_t b_rows = g.group == GroupKind::Rows ? g.N * g.num_experts : g.N;
    const int box_a = g.M >= 128 ? 128 : (int)((g.M + 7) / 8 * 8);
    const int box_b = b_rows >= BN ? BN : (int)((b_rows + 7) / 8 * 8);
    CUtensorMap ta, tbm;
    if ((e = make_kmajor_map(&ta, g.a, g.K, g.M, g.lda, box_a)) != cudaSuccess)
        return e;
    if ((e = make_kmajor_map(&tbm, g.b, g.K, b_rows, g.ldb, box_b)) != cudaSuccess)
        return e;
    MxParams kp;
    Sched &s = kp.sched;
    s.mode = g.group == GroupKind::None ? kDense : (g.group == GroupKind::Rows ? kGroupedRows : kGroupedK);
    s.mt = (int)((g.M + 127) / 128);
    s.nt = (int)((g.N + BN - 1) / BN);
    s.num_kb = (int)(g.K / 128);
    s.M = g.M;
    s.N = (int)g.N;
    s.bn = BN;
    s.seg = g.seg;
    // routed rows for FProp/DGrad; column-copy positions (>= routed rows) for WGrad
    s.seg_max = g.group == GroupKind::K ? g.K : g.M;
    s.E = g.num_experts;
    kp.sfa = g.sfa;
    kp.sfb = g.sfb;
    kp.rba = (int)((g.M + 127) / 128);
    kp.rbb = (int)((g.N + 127) / 128);
    kp.sfb_e_stride = g.group == GroupKind::Rows ? (int64_t)kp.rbb * (g.K / 128) * 512 : 0;
    kp.box_a_rows = box_a;
    kp.box_b_rows = box_b;
    kp.out = g.out;
    kp.ldo = g.ldo;
    kp.out_e_stride = g.group == GroupKind::K ? g.M * g.ldo : 0;
    kp.out_bf16 = g.out_dtype == JETQ_OUT_BF16;
    kp.accumulate = g.accumulate;
    kp.limit_ns = kWaitLimitNs;
    int grid = sm_count();
    if (g.group == GroupKind::None) {
        const int tiles = s.mt * s.nt;
        grid = tiles < grid ? tiles : grid;
    } else if (g.group == GroupKind::K) {
        const int tiles = s.mt * s.nt * g.num_experts;
        grid = tiles < grid ? tiles : grid;
    }
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
