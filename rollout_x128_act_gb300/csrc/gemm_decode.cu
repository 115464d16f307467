// Decode-shaped FP8 GEMM, 128-block recipe, with the operands swapped.
//
//   y[t, o] = sum over K-blocks kb of  fl32(Sx[t,kb] * Sw[o/128,kb]) * P_kb[t, o]
//   P_kb[t, o] = sum_{k in kb} qx[t, k] * qw[o, k]        (E4M3 x E4M3 -> FP32)
//
// A rollout step multiplies a handful of tokens (n <= 64) by a whole weight,
// so the weight stream is the work.  Here the weight is the MMA's A operand
// (M = 128 weight rows per tile) and the tokens its N operand (NB = 16, 32 or
// 64 columns, the rows past n zero-filled by TMA): one tcgen05.mma then
// covers 4 KB of weight, four times what the token-row orientation covers,
// and every TMEM lane holds a live output feature.  The per-element
// operation sequence is the training kernel's (ascending K-blocks, one fresh
// FP32 partial per K-block, acc = fma(P_kb, fl32(Sx * Sw), acc)), so a row of
// this kernel's output equals the training kernel's row bit for bit.
//
//   warp 0      TMA producer: per stage KBP K-blocks of the 128-row weight
//               tile and of the token rows, one 3-D box each
//   warp 1      MMA issuer: per K-block 4 x tcgen05.mma (K = 32) into its own
//               TMEM buffer; one commit per stage releases the smem stage
//               and hands the stage's buffer group to the epilogue
//   warp 2      scale producer: the NB products fl32(Sx * Sw) of each
//               K-block into a shared-memory ring, eight K-blocks a slot
//   warps 4-7   epilogue: per K-block tcgen05.ld the partial (TMEM lanes =
//               weight rows, columns = tokens), acc = fma(P, s, acc); after
//               the last K-block, store y[t, o] for t < n (coalesced along o)
//
// One CTA per SM, persistent over 128-row weight tiles.  Weights with few
// row bands (the down projection has 32) leave most SMs idle that way; with
// a caller's workspace they take the split-K kernel further down (a cluster
// of CTAs per band, partial sums through the workspace, the same fold).
// Both kernels are launched so that their prologue overlaps the stream's
// previous kernel (programmatic dependent launch) and wait for it before
// touching global memory.  Every mbarrier wait is bounded; a CTA that gives
// up raises its abort flag, records the error in the device error word,
// drains its TMA copies and MMAs (bounded) and frees its TMEM.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "jetq_internal.h"
#include "ptx.cuh"

namespace jetq {

__device__ unsigned g_gemm_decode_error;

namespace {

constexpr unsigned kErrTimeout = 1u;
constexpr unsigned long long kWaitLimitNs = 2000000000ull; // 2 s per wait

// Scale ring: each slot holds the products fl32(Sx * Sw) of kScaleGroup
// consecutive K-blocks, so producer and epilogue meet once per group.
constexpr int kScaleGroup = 8;
constexpr int kScaleSlots = 4;

__host__ __device__ constexpr int gcd_i(int a, int b) { return b ? gcd_i(b, a % b) : a; }
__host__ __device__ constexpr int lcm_i(int a, int b) { return a / gcd_i(a, b) * b; }

struct DParams {
    const float *sx;  // token scales [K-blocks x n]
    const float *sw;  // weight block scales [D/128 x num_kb]
    int n;            // tokens
    int tiles;        // D / 128
    int num_kb;       // K / 128
    void *out;        // y [n x ldo]
    int64_t ldo;
    int out_bf16;
    unsigned long long limit_ns;
};

// Scale producer (one warp): slot i of the ring holds, for kScaleGroup
// consecutive K-blocks c of the CTA's sequence, s[t] = fl32(Sx[t, kb] *
// Sw[tile, kb]) for t < NB (0 past the batch).  fetch(c, x0, x1, w) loads
// the lane's two token scales and the weight scale of K-block c; the next
// group's loads are in flight while a group is stored.
template <int NB, class Fetch, class BarF, class BarE>
__device__ __forceinline__ void scale_producer(int total, Fetch &&fetch, float *srow, BarF &&sfull, BarE &&sempty,
                                               volatile int *abort_flag, unsigned *err, uint64_t limit_ns, int lane)
{
    constexpr int G = kScaleGroup;
    float cx0[G], cx1[G], cw[G];
#pragma unroll
    for (int u = 0; u < G; ++u)
        if (u < total)
            fetch(u, cx0[u], cx1[u], cw[u]);
    for (int g = 0; g * G < total; ++g) {
        const int c0 = g * G;
        float nx0[G], nx1[G], nw[G];
#pragma unroll
        for (int u = 0; u < G; ++u)
            if (c0 + G + u < total)
                fetch(c0 + G + u, nx0[u], nx1[u], nw[u]);
        const int i = g % kScaleSlots;
        const bool got = ptx::mbar_wait(sempty(i), ((uint32_t)(g / kScaleSlots) & 1u) ^ 1u, abort_flag, err,
                                        kErrTimeout, limit_ns);
        if (!__all_sync(0xFFFFFFFFu, got))
            return;
#pragma unroll
        for (int u = 0; u < G; ++u) {
            if (c0 + u < total) {
                float *row = srow + (i * G + u) * NB;
                if (lane < NB)
                    row[lane] = __fmul_rn(cx0[u], cw[u]);
                if (NB > 32 && lane + 32 < NB)
                    row[lane + 32] = __fmul_rn(cx1[u], cw[u]);
            }
        }
        ptx::mbar_arrive(sfull(i));
#pragma unroll
        for (int u = 0; u < G; ++u) {
            cx0[u] = nx0[u];
            cx1[u] = nx1[u];
            cw[u] = nw[u];
        }
    }
}

template <int NB, int STAGES, int KBP, int TMEM_BUFS>
struct DCfg {
    static constexpr int kWBytes = 128 * 128; // one K-block of the 128-row weight tile
    static constexpr int kXBytes = NB * 128;  // one K-block of the token rows
    static constexpr int NG = TMEM_BUFS / KBP; // accumulator groups: one per stage, KBP buffers each
    static constexpr int kSlots = kScaleSlots; // scale ring: kScaleGroup K-blocks per slot
    static constexpr int kThreads = 256;
    static constexpr int kBars = 2 * STAGES + 2 * NG + 2 * kSlots + 1;
    static constexpr size_t kSmem = 1024 + (size_t)STAGES * KBP * (kWBytes + kXBytes) +
                                    (size_t)kSlots * kScaleGroup * NB * 4 + 1024;
    static_assert(NB % 16 == 0 && NB >= 16 && NB <= 64, "token columns");
    static_assert(TMEM_BUFS % KBP == 0 && TMEM_BUFS * NB <= 512, "TMEM buffers");
    static_assert(kBars * 8 + 16 <= 1024, "barrier area");
    static_assert(kSmem <= 232448, "shared memory");
};

template <int NB, int STAGES, int KBP, int TMEM_BUFS>
__global__ void __launch_bounds__(256, 1)
    k_gemm_decode(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX, const DParams p)
{
    using C = DCfg<NB, STAGES, KBP, TMEM_BUFS>;
    constexpr int NG = C::NG;
    constexpr int SL = C::kSlots;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *tiles_w = ptx::align_smem<1024>(smem_raw);
    uint8_t *tiles_x = tiles_w + (size_t)STAGES * KBP * C::kWBytes;
    float *srow = reinterpret_cast<float *>(tiles_x + (size_t)STAGES * KBP * C::kXBytes);
    uint64_t *bars = reinterpret_cast<uint64_t *>(srow + SL * kScaleGroup * NB);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + C::kBars);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const uint32_t bar0 = ptx::smem_addr(bars);
    auto full = [&](int s) { return bar0 + 8u * s; };
    auto empty = [&](int s) { return bar0 + 8u * (STAGES + s); };
    auto tfull = [&](int g) { return bar0 + 8u * (2 * STAGES + g); };
    auto tempty = [&](int g) { return bar0 + 8u * (2 * STAGES + NG + g); };
    auto sfull = [&](int i) { return bar0 + 8u * (2 * STAGES + 2 * NG + i); };
    auto sempty = [&](int i) { return bar0 + 8u * (2 * STAGES + 2 * NG + SL + i); };
    const uint32_t done = bar0 + 8u * (2 * STAGES + 2 * NG + 2 * SL);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    unsigned *err = &g_gemm_decode_error;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(full(s), 1);
            ptx::mbar_init(empty(s), 1);
        }
        for (int g = 0; g < NG; ++g) {
            ptx::mbar_init(tfull(g), 1);
            ptx::mbar_init(tempty(g), 4);
        }
        for (int i = 0; i < SL; ++i) {
            ptx::mbar_init(sfull(i), 32);
            ptx::mbar_init(sempty(i), 4);
        }
        ptx::mbar_init(done, 1);
        *abort_flag = 0;
        ptx::fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tensormap(&tmW);
        ptx::prefetch_tensormap(&tmX);
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_addr(tmem_slot), 512);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // the prologue above overlaps the stream's previous kernel; global memory
    // only after it has completed
    ptx::grid_dep_launch();
    ptx::grid_dep_wait();

    const int nkb = p.num_kb;
    const int spt = (nkb + KBP - 1) / KBP; // stages per tile
    const int last_nk = nkb - (spt - 1) * KBP;
    int my_tiles = 0;
    for (int t = blockIdx.x; t < p.tiles; t += gridDim.x)
        ++my_tiles;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------------------------------------------- TMA producer
            // a box past the last K-block is zero-filled and still counts in full
            constexpr uint32_t tx = (uint32_t)(KBP * (C::kWBytes + C::kXBytes));
            uint32_t it = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < p.tiles && ok; t += gridDim.x) {
                for (int q = 0; q < spt; ++q, ++it) {
                    const int s = (int)(it % STAGES);
                    if (!ptx::mbar_wait(empty(s), ((it / STAGES) & 1u) ^ 1u, abort_flag, err, kErrTimeout, p.limit_ns)) {
                        ok = false;
                        break;
                    }
                    ptx::mbar_arrive_expect_tx(full(s), tx);
                    ptx::tma_load_3d(ptx::smem_addr(tiles_w + (size_t)s * KBP * C::kWBytes), &tmW, full(s), 0, t * 128,
                                     q * KBP);
                    ptx::tma_load_3d(ptx::smem_addr(tiles_x + (size_t)s * KBP * C::kXBytes), &tmX, full(s), 0, 0,
                                     q * KBP);
                }
            }
            // drain: every copy this thread started must have landed before exit
            for (int s = 0; s < STAGES; ++s) {
                if (it > (uint32_t)s) {
                    const uint32_t last = (uint32_t)s + ((it - 1u - (uint32_t)s) / STAGES) * STAGES;
                    ptx::mbar_wait(full(s), (last / STAGES) & 1u, abort_flag, err, kErrTimeout, p.limit_ns, false);
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------------------------------------------- MMA issuer
            // operands are base registers plus compile-time offsets (the loop is
            // unrolled so stage and buffer indices are constants): an operand
            // computed inside the loop slows each issue by a few hundred cycles
            constexpr uint32_t idesc = ptx::idesc_e4m3_f32(128, NB);
            constexpr int U = lcm_i(STAGES, NG);
            const uint64_t wdesc0 = ptx::desc_kmajor_sw128(ptx::smem_addr(tiles_w));
            const uint64_t xdesc0 = ptx::desc_kmajor_sw128(ptx::smem_addr(tiles_x));
            const int total = my_tiles * spt;
            bool ok = true;
            for (int q0 = 0; q0 < total && ok; q0 += U) {
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int q = q0 + u;
                    if (q < total && ok) {
                        const int s = u % STAGES;
                        const int gi = u % NG;
                        const int nk = q % spt == spt - 1 ? last_nk : KBP;
                        if (!ptx::mbar_wait(tempty(gi), (((uint32_t)q / NG) & 1u) ^ 1u, abort_flag, err, kErrTimeout,
                                            p.limit_ns) ||
                            !ptx::mbar_wait(full(s), ((uint32_t)q / STAGES) & 1u, abort_flag, err, kErrTimeout,
                                            p.limit_ns)) {
                            ok = false;
                        } else {
                            ptx::tc_fence_after();
#pragma unroll
                            for (int j = 0; j < KBP; ++j) {
                                if (j < nk) {
                                    // descriptors address 16-byte units
                                    const uint64_t wd = wdesc0 + (uint64_t)(((s * KBP + j) * C::kWBytes) >> 4);
                                    const uint64_t xd = xdesc0 + (uint64_t)(((s * KBP + j) * C::kXBytes) >> 4);
                                    const uint32_t d = tmem_base + (uint32_t)((gi * KBP + j) * NB);
#pragma unroll
                                    for (int k = 0; k < 4; ++k) // 4 x K=32 (32 bytes) in the 128-byte swizzle row
                                        ptx::mma_f8f6f4(d, wd + 2u * k, xd + 2u * k, idesc, k > 0 ? 1u : 0u);
                                }
                            }
                            ptx::mma_commit(empty(s));
                            ptx::mma_commit(tfull(gi));
                        }
                    }
                }
            }
            ptx::mma_commit(done);
            ptx::mbar_wait(done, 0u, abort_flag, err, kErrTimeout, p.limit_ns, false);
        }
        __syncwarp();
    } else if (warp == 2) {
        // ---------------------------------------------------- scale producer
        const int total = my_tiles * nkb; // this CTA's K-blocks, tile after tile
        auto fetch = [&](int gk, float &xv0, float &xv1, float &wv) {
            const int lt = gk / nkb, kb = gk - lt * nkb;
            wv = __ldg(p.sw + (int64_t)(blockIdx.x + lt * gridDim.x) * nkb + kb);
            xv0 = lane < p.n ? __ldg(p.sx + (int64_t)kb * p.n + lane) : 0.0f;
            xv1 = NB > 32 && lane + 32 < p.n ? __ldg(p.sx + (int64_t)kb * p.n + lane + 32) : 0.0f;
        };
        scale_producer<NB>(total, fetch, srow, sfull, sempty, abort_flag, err, p.limit_ns, lane);
    } else if (warp >= 4) {
        // ---------------------------------------------------- epilogue
        const int quarter = warp & 3; // TMEM lanes 32*quarter .. +31 = weight rows of the tile
        const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
        uint32_t c = 0, qg = 0;
        const int total_kb = my_tiles * nkb;
        bool ok = true;
        for (int t = blockIdx.x; t < p.tiles && ok; t += gridDim.x) {
            float2 acc[NB / 2];
#pragma unroll
            for (int j = 0; j < NB / 2; ++j)
                acc[j] = make_float2(0.0f, 0.0f);
            for (int q = 0; q < spt && ok; ++q, ++qg) {
                const int gi = (int)(qg % NG);
                const int nk = q == spt - 1 ? last_nk : KBP;
                bool got = ptx::mbar_wait(tfull(gi), (qg / NG) & 1u, abort_flag, err, kErrTimeout, p.limit_ns);
                if (!__all_sync(0xFFFFFFFFu, got)) { // keep the warp converged for tcgen05.ld
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
#pragma unroll
                for (int j = 0; j < KBP; ++j) {
                    if (j < nk && ok) {
                        const int gq = (int)(c / kScaleGroup), u = (int)(c % kScaleGroup), i = gq % SL;
                        if (u == 0)
                            got = ptx::mbar_wait(sfull(i), (uint32_t)(gq / SL) & 1u, abort_flag, err, kErrTimeout,
                                                 p.limit_ns);
                        if (!__all_sync(0xFFFFFFFFu, got)) {
                            ok = false;
                        } else {
                            uint32_t P[NB / 16][16];
                            const uint32_t col = tmem_base + lane_addr + (uint32_t)((gi * KBP + j) * NB);
#pragma unroll
                            for (int h = 0; h < NB / 16; ++h)
                                ptx::tmem_ld_32x32b_x16(col + 16u * h, P[h]);
                            ptx::tmem_ld_wait();
                            const float4 *s4 =
                                reinterpret_cast<const float4 *>(srow + (i * kScaleGroup + u) * NB);
#pragma unroll
                            for (int h = 0; h < NB / 4; ++h) {
                                const float4 sv = s4[h];
                                const uint32_t *ph = &P[h / 4][(h % 4) * 4];
                                acc[2 * h] = __ffma2_rn(make_float2(__uint_as_float(ph[0]), __uint_as_float(ph[1])),
                                                        make_float2(sv.x, sv.y), acc[2 * h]);
                                acc[2 * h + 1] = __ffma2_rn(make_float2(__uint_as_float(ph[2]), __uint_as_float(ph[3])),
                                                            make_float2(sv.z, sv.w), acc[2 * h + 1]);
                            }
                            ++c;
                            if (u == kScaleGroup - 1 || (int)c == total_kb) { // the slot's last K-block
                                __syncwarp();
                                if (lane == 0)
                                    ptx::mbar_arrive(sempty(i));
                            }
                        }
                    }
                }
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    ptx::mbar_arrive(tempty(gi));
            }
            if (!ok)
                break;
            const int64_t o = (int64_t)t * 128 + quarter * 32 + lane;
            if (p.out_bf16) {
                __nv_bfloat16 *y = reinterpret_cast<__nv_bfloat16 *>(p.out) + o;
#pragma unroll
                for (int h = 0; h < NB / 2; ++h) {
                    if (2 * h < p.n)
                        y[(int64_t)(2 * h) * p.ldo] = __float2bfloat16_rn(acc[h].x);
                    if (2 * h + 1 < p.n)
                        y[(int64_t)(2 * h + 1) * p.ldo] = __float2bfloat16_rn(acc[h].y);
                }
            } else {
                float *y = reinterpret_cast<float *>(p.out) + o;
#pragma unroll
                for (int h = 0; h < NB / 2; ++h) {
                    if (2 * h < p.n)
                        y[(int64_t)(2 * h) * p.ldo] = acc[h].x;
                    if (2 * h + 1 < p.n)
                        y[(int64_t)(2 * h + 1) * p.ldo] = acc[h].y;
                }
            }
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_base, 512);
    }
}

template <int NB, int STAGES, int KBP, int TMEM_BUFS>
cudaError_t run_decode(const GemmProblem &g, cudaStream_t st)
{
    using C = DCfg<NB, STAGES, KBP, TMEM_BUFS>;
    auto kern = k_gemm_decode<NB, STAGES, KBP, TMEM_BUFS>;
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
    // weight: 128-row boxes; tokens: NB-row boxes (rows past n arrive zero-filled)
    CUtensorMap tw, tx;
    if ((e = make_kmajor_map(&tw, g.b, g.K, g.N, g.ldb, 128, KBP)) != cudaSuccess)
        return e;
    if ((e = make_kmajor_map(&tx, g.a, g.K, g.M, g.lda, NB, KBP)) != cudaSuccess)
        return e;
    DParams p;
    p.sx = g.sa;
    p.sw = g.sb;
    p.n = (int)g.M;
    p.tiles = (int)(g.N / 128);
    p.num_kb = (int)(g.K / 128);
    p.out = g.out;
    p.ldo = g.ldo;
    p.out_bf16 = g.out_dtype == JETQ_OUT_BF16;
    p.limit_ns = kWaitLimitNs;
    const int grid = p.tiles < sm_count() ? p.tiles : sm_count();
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(C::kThreads);
    cfg.dynamicSmemBytes = C::kSmem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization; // prologue overlaps the previous kernel
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if ((e = cudaLaunchKernelEx(&cfg, kern, tw, tx, p)) != cudaSuccess)
        return e;
    return cudaGetLastError();
}


// ---------------------------------------------------------------------------
// Split-K variant for weights with few 128-row bands (the down projection has
// 32): a cluster of S CTAs per band, so that S times as many SMs stream the
// weight.  The band's K range is cut into chunks of KBP K-blocks; chunk q is
// computed by CTA q % S of the cluster.
//
//   phase 1     warp 0 (TMA) and warp 1 (MMA) run this CTA's chunks through
//               TMEM; warps 4-7 read each finished K-block's FP32 partials
//               P_kb (TMEM lanes = rows 32(w-4)..) and store the n real token
//               columns to the workspace, layout [band][kb][token][row]
//   barrier     the cluster's CTAs meet (release / acquire at cluster scope),
//               so every partial of the band is visible to all of them
//   phase 2     CTA r folds rows [r * 128 / S, (r + 1) * 128 / S) of the band,
//               every token: acc = fma(P_kb, fl32(Sx * Sw), acc) over the
//               K-blocks in ascending order, the training kernel's chain, so
//               the output equals the single-CTA kernel's and the training
//               kernel's bit for bit
//
// The workspace holds N x (K / 128) x n floats (L2-resident for decode batch
// sizes).  Every mbarrier wait is bounded, and every CTA reaches the cluster
// barrier whatever happened before it.
template <int NB, int S, int STAGES, int KBP, int TMEM_BUFS>
struct SCfg {
    static constexpr int kWBytes = 128 * 128;
    static constexpr int kXBytes = NB * 128;
    static constexpr int NG = TMEM_BUFS / KBP;
    static constexpr int kThreads = 256;
    static constexpr int kRows = 128 / S; // rows of the band folded per CTA
    // CTAs per SM the launch must allow: two when shared memory lets two share an SM
    static constexpr int kMinBlocks = S == 2 ? 2 : 1;
    static constexpr int kBars = 2 * STAGES + 2 * NG + 1;
    static constexpr int kTmemCols = TMEM_BUFS * NB <= 32    ? 32
                                     : TMEM_BUFS * NB <= 64  ? 64
                                     : TMEM_BUFS * NB <= 128 ? 128
                                     : TMEM_BUFS * NB <= 256 ? 256
                                                             : 512;
    static constexpr size_t kSmem = 1024 + (size_t)STAGES * KBP * (kWBytes + kXBytes) + 1024;
    static_assert(S >= 2 && S <= 8 && 128 % S == 0 && (128 / S) % 16 == 0, "portable cluster");
    static_assert(NB == 16 || NB == 32, "token columns (the fold covers up to 32 tokens)");
    static_assert(TMEM_BUFS % KBP == 0 && TMEM_BUFS * NB <= 512, "TMEM buffers");
    static_assert(kBars * 8 + 16 <= 1024, "barrier area");
    static_assert(kSmem <= 232448, "shared memory");
    // CTAs that share an SM must never wait for each other's TMEM
    static_assert(kTmemCols * (int)(232448 / kSmem) <= 512, "TMEM of co-resident CTAs");
};

// Phase 2 of the split-K decode, over this CTA's R rows of the band: in
// passes of up to `cap` K-blocks, the partials [kb][token][R rows] and the
// products fl32(Sx[kb, t] * Sw[band, kb]) are copied into shared memory (the
// idle stage buffers; every copy of a pass in flight at once), then element
// e = threadIdx.x + T i (token e / R, row rank * R + e % R) runs
// acc = fma(P_kb, s, acc) over the pass's K-blocks in ascending order.
template <int R, int E, int T>
__device__ __forceinline__ void fold_rows(const DParams &p, const float *wsb, float *smem, int cap, int rank, int n,
                                          int nkb, int band)
{
    const int elems = R * n;
    const float *swb = p.sw + (size_t)band * nkb;
    const uint32_t sbase = ptx::smem_addr(smem);
    float acc[E];
#pragma unroll
    for (int i = 0; i < E; ++i)
        acc[i] = 0.0f;
    for (int kb0 = 0; kb0 < nkb; kb0 += cap) {
        const int kn = min(cap, nkb - kb0);
        const int units = kn * n * (R / 4); // 16-byte units of partials
        for (int u = (int)threadIdx.x; u < units; u += T) {
            const int rq = u % (R / 4), rest = u / (R / 4); // rest = kbl * n + t
            const float *src = wsb + (size_t)(kb0 * n + rest) * 128 + rank * R + rq * 4;
            ptx::cp_async_16(sbase + (uint32_t)(rest * R + rq * 4) * 4u, src, 16u);
        }
        float *sprod = smem + (size_t)kn * n * R;
        for (int v = (int)threadIdx.x; v < kn * n; v += T) {
            const int kbl = v / n, t = v - kbl * n;
            sprod[v] = __fmul_rn(__ldg(p.sx + (size_t)(kb0 + kbl) * n + t), __ldg(swb + kb0 + kbl));
        }
        ptx::cp_async_wait_all();
        __syncthreads();
#pragma unroll
        for (int i = 0; i < E; ++i) {
            const int e = (int)threadIdx.x + T * i;
            if (e < elems) {
                const int t = e / R, r = e - t * R;
                const float *pp = smem + t * R + r;
                const float *ss = sprod + t;
                float a = acc[i];
#pragma unroll 8
                for (int kbl = 0; kbl < kn; ++kbl)
                    a = __fmaf_rn(pp[(size_t)kbl * n * R], ss[kbl * n], a);
                acc[i] = a;
            }
        }
        __syncthreads(); // the next pass overwrites the buffers
    }
#pragma unroll
    for (int i = 0; i < E; ++i) {
        const int e = (int)threadIdx.x + T * i;
        if (e < elems) {
            const int t = e / R, row = rank * R + (e - t * R);
            const int64_t o = (int64_t)t * p.ldo + (int64_t)band * 128 + row;
            if (p.out_bf16)
                reinterpret_cast<__nv_bfloat16 *>(p.out)[o] = __float2bfloat16_rn(acc[i]);
            else
                reinterpret_cast<float *>(p.out)[o] = acc[i];
        }
    }
}

template <int NB, int S, int STAGES, int KBP, int TMEM_BUFS>
__global__ void __launch_bounds__(256, (SCfg<NB, S, STAGES, KBP, TMEM_BUFS>::kMinBlocks))
    k_gemm_decode_split(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                        const DParams p, float *__restrict__ ws)
{
    using C = SCfg<NB, S, STAGES, KBP, TMEM_BUFS>;
    constexpr int NG = C::NG;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *tiles_w = ptx::align_smem<1024>(smem_raw);
    uint8_t *tiles_x = tiles_w + (size_t)STAGES * KBP * C::kWBytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(tiles_x + (size_t)STAGES * KBP * C::kXBytes);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + C::kBars);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const uint32_t bar0 = ptx::smem_addr(bars);
    auto full = [&](int s) { return bar0 + 8u * s; };
    auto empty = [&](int s) { return bar0 + 8u * (STAGES + s); };
    auto tfull = [&](int g) { return bar0 + 8u * (2 * STAGES + g); };
    auto tempty = [&](int g) { return bar0 + 8u * (2 * STAGES + NG + g); };
    const uint32_t done = bar0 + 8u * (2 * STAGES + 2 * NG);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    unsigned *err = &g_gemm_decode_error;
    const int rank = (int)ptx::cluster_ctarank();
    const int band = (int)blockIdx.x / S;
    const int n = p.n;
    const int nkb = p.num_kb;
    float *wsb = ws + (size_t)band * nkb * n * 128; // this band's partials [kb][token][row]

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(full(s), 1);
            ptx::mbar_init(empty(s), 1);
        }
        for (int g = 0; g < NG; ++g) {
            ptx::mbar_init(tfull(g), 1);
            ptx::mbar_init(tempty(g), 4);
        }
        ptx::mbar_init(done, 1);
        *abort_flag = 0;
        ptx::fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tensormap(&tmW);
        ptx::prefetch_tensormap(&tmX);
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_addr(tmem_slot), C::kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // the prologue above overlaps the stream's previous kernel; global memory
    // (the workspace included) only after it has completed
    ptx::grid_dep_launch();
    ptx::grid_dep_wait();

    const int nch = (nkb + KBP - 1) / KBP; // chunks of the band
    const int last_nk = nkb - (nch - 1) * KBP;
    const int my_chunks = rank < nch ? (nch - 1 - rank) / S + 1 : 0;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------------------------------------------- TMA producer
            constexpr uint32_t tx = (uint32_t)(KBP * (C::kWBytes + C::kXBytes));
            uint32_t it = 0;
            for (int j = 0; j < my_chunks; ++j, ++it) {
                const int s = (int)(it % STAGES);
                if (!ptx::mbar_wait(empty(s), ((it / STAGES) & 1u) ^ 1u, abort_flag, err, kErrTimeout, p.limit_ns))
                    break;
                const int q = rank + j * S;
                ptx::mbar_arrive_expect_tx(full(s), tx);
                const uint32_t dw = ptx::smem_addr(tiles_w + (size_t)s * KBP * C::kWBytes);
                const uint32_t dx = ptx::smem_addr(tiles_x + (size_t)s * KBP * C::kXBytes);
                if constexpr (KBP == 1) { // plain 2-D maps (x = byte offset along K)
                    ptx::tma_load_2d(dw, &tmW, full(s), q * 128, band * 128);
                    ptx::tma_load_2d(dx, &tmX, full(s), q * 128, 0);
                } else { // 3-D maps: (byte in K-block, row, K-block)
                    ptx::tma_load_3d(dw, &tmW, full(s), 0, band * 128, q * KBP);
                    ptx::tma_load_3d(dx, &tmX, full(s), 0, 0, q * KBP);
                }
            }
            for (int s = 0; s < STAGES; ++s) {
                if (it > (uint32_t)s) {
                    const uint32_t last = (uint32_t)s + ((it - 1u - (uint32_t)s) / STAGES) * STAGES;
                    ptx::mbar_wait(full(s), (last / STAGES) & 1u, abort_flag, err, kErrTimeout, p.limit_ns, false);
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------------------------------------------- MMA issuer
            constexpr uint32_t idesc = ptx::idesc_e4m3_f32(128, NB);
            constexpr int UU = lcm_i(STAGES, NG);
            const uint64_t wdesc0 = ptx::desc_kmajor_sw128(ptx::smem_addr(tiles_w));
            const uint64_t xdesc0 = ptx::desc_kmajor_sw128(ptx::smem_addr(tiles_x));
            bool ok = true;
            for (int q0 = 0; q0 < my_chunks && ok; q0 += UU) {
#pragma unroll
                for (int u = 0; u < UU; ++u) {
                    const int j = q0 + u;
                    if (j < my_chunks && ok) {
                        const int s = u % STAGES;
                        const int gi = u % NG;
                        const int nk = rank + j * S == nch - 1 ? last_nk : KBP;
                        if (!ptx::mbar_wait(tempty(gi), (((uint32_t)j / NG) & 1u) ^ 1u, abort_flag, err, kErrTimeout,
                                            p.limit_ns) ||
                            !ptx::mbar_wait(full(s), ((uint32_t)j / STAGES) & 1u, abort_flag, err, kErrTimeout,
                                            p.limit_ns)) {
                            ok = false;
                        } else {
                            ptx::tc_fence_after();
#pragma unroll
                            for (int jj = 0; jj < KBP; ++jj) {
                                if (jj < nk) {
                                    const uint64_t wd = wdesc0 + (uint64_t)(((s * KBP + jj) * C::kWBytes) >> 4);
                                    const uint64_t xd = xdesc0 + (uint64_t)(((s * KBP + jj) * C::kXBytes) >> 4);
                                    const uint32_t d = tmem_base + (uint32_t)((gi * KBP + jj) * NB);
#pragma unroll
                                    for (int k = 0; k < 4; ++k)
                                        ptx::mma_f8f6f4(d, wd + 2u * k, xd + 2u * k, idesc, k > 0 ? 1u : 0u);
                                }
                            }
                            ptx::mma_commit(empty(s));
                            ptx::mma_commit(tfull(gi));
                        }
                    }
                }
            }
            ptx::mma_commit(done);
            ptx::mbar_wait(done, 0u, abort_flag, err, kErrTimeout, p.limit_ns, false);
        }
        __syncwarp();
    } else if (warp >= 4) {
        // ---------------------------------------------------- partials out
        const int quarter = warp - 4; // TMEM lanes 32*quarter .. +31 = rows of the band
        const int row = quarter * 32 + lane;
        const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
        for (int j = 0; j < my_chunks; ++j) {
            const int q = rank + j * S;
            const int nk = q == nch - 1 ? last_nk : KBP;
            const int gi = j % NG;
            const bool got =
                ptx::mbar_wait(tfull(gi), ((uint32_t)j / NG) & 1u, abort_flag, err, kErrTimeout, p.limit_ns);
            if (!__all_sync(0xFFFFFFFFu, got))
                break;
            ptx::tc_fence_after();
#pragma unroll
            for (int jj = 0; jj < KBP; ++jj) {
                if (jj < nk) {
                    uint32_t P[NB];
                    const uint32_t col = tmem_base + lane_addr + (uint32_t)((gi * KBP + jj) * NB);
#pragma unroll
                    for (int h = 0; h < NB / 16; ++h)
                        ptx::tmem_ld_32x32b_x16(col + 16u * h, *reinterpret_cast<uint32_t(*)[16]>(P + 16 * h));
                    ptx::tmem_ld_wait();
                    float *dst = wsb + (size_t)(q * KBP + jj) * n * 128 + row;
#pragma unroll
                    for (int t = 0; t < NB; ++t)
                        if (t < n)
                            __stcg(dst + (size_t)t * 128, __uint_as_float(P[t]));
                }
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0)
                ptx::mbar_arrive(tempty(gi));
        }
    }

    // ---------------------------------------------------------- cluster barrier
    __syncwarp();
    ptx::tc_fence_before();
    ptx::cluster_sync(); // release / acquire at cluster scope: the band's partials are visible
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_base, C::kTmemCols);
    }

    // ---------------------------------------------------------- phase 2: fold
    if (*abort_flag == 0) {
        // the stage buffers are idle: every TMA copy has landed and every MMA
        // has completed before the cluster barrier
        float *fsm = reinterpret_cast<float *>(tiles_w);
        const int cap = (int)(((size_t)STAGES * KBP * (C::kWBytes + C::kXBytes)) / ((size_t)(C::kRows + 1) * n * 4));
        const int per_thread = (C::kRows * n + C::kThreads - 1) / C::kThreads; // <= 8 (n <= 32)
        if (per_thread <= 1)
            fold_rows<C::kRows, 1, C::kThreads>(p, wsb, fsm, cap, rank, n, nkb, band);
        else if (per_thread <= 2)
            fold_rows<C::kRows, 2, C::kThreads>(p, wsb, fsm, cap, rank, n, nkb, band);
        else if (per_thread <= 4)
            fold_rows<C::kRows, 4, C::kThreads>(p, wsb, fsm, cap, rank, n, nkb, band);
        else
            fold_rows<C::kRows, 8, C::kThreads>(p, wsb, fsm, cap, rank, n, nkb, band);
    }
}

template <int NB, int S, int STAGES, int KBP, int TMEM_BUFS>
cudaError_t run_decode_split(const GemmProblem &g, cudaStream_t st)
{
    using C = SCfg<NB, S, STAGES, KBP, TMEM_BUFS>;
    auto kern = k_gemm_decode_split<NB, S, STAGES, KBP, TMEM_BUFS>;
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
    CUtensorMap tw, tx;
    if ((e = make_kmajor_map(&tw, g.b, g.K, g.N, g.ldb, 128, KBP)) != cudaSuccess)
        return e;
    if ((e = make_kmajor_map(&tx, g.a, g.K, g.M, g.lda, NB, KBP)) != cudaSuccess)
        return e;
    DParams p;
    p.sx = g.sa;
    p.sw = g.sb;
    p.n = (int)g.M;
    p.tiles = (int)(g.N / 128);
    p.num_kb = (int)(g.K / 128);
    p.out = g.out;
    p.ldo = g.ldo;
    p.out_bf16 = g.out_dtype == JETQ_OUT_BF16;
    p.limit_ns = kWaitLimitNs;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(p.tiles * S));
    cfg.blockDim = dim3(C::kThreads);
    cfg.dynamicSmemBytes = C::kSmem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = S;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization; // prologue overlaps the previous kernel
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    if ((e = cudaLaunchKernelEx(&cfg, kern, tw, tx, p, static_cast<float *>(g.ws))) != cudaSuccess)
        return e;
    return cudaGetLastError();
}

} // namespace

// Cluster size of the split-K decode for a shape (1: the single-CTA kernel):
// weights of few row bands, whose one-CTA-a-band launch leaves most SMs idle,
// and at least two chunks of K-blocks per CTA.
int decode_split_factor(int64_t M, int64_t N, int64_t K)
{
    // partial sums grow with the batch: past 32 tokens they outweigh the weight
    if (M < 1 || M > 32 || N % 128 != 0 || K % 128 != 0)
        return 1;
    const int64_t bands = N / 128, nkb = K / 128, sms = sm_count();
    if (bands < kDecodeSwappedMinTiles)
        return 1;
    // (measured: a weight of 96 bands runs faster one CTA a band than split
    // over two CTAs a band, two CTAs an SM)
    if (bands * 4 <= sms && nkb >= 16)
        return 4;
    if (bands * 2 <= sms && nkb >= 8)
        return 2;
    return 1;
}

size_t decode_split_workspace_bytes(int64_t M, int64_t N, int64_t K)
{
    if (decode_split_factor(M, N, K) == 1)
        return 0;
    return (size_t)N * (size_t)(K / 128) * (size_t)M * sizeof(float);
}

bool gemm_decode_swapped_applies(const GemmProblem &g)
{
    return g.group == GroupKind::None && g.bscale == BScale::Block128 && g.M >= 1 && g.M <= 64 &&
           g.N % 128 == 0 && g.K % 128 == 0 && g.K > 0 && g.N / 128 >= kDecodeSwappedMinTiles && !g.accumulate;
}

cudaError_t launch_gemm_decode_swapped(const GemmProblem &g, cudaStream_t st)
{
    if (!gemm_decode_swapped_applies(g))
        return cudaErrorInvalidValue;
    // with a workspace: a cluster of S CTAs per row band splits its K range
    if (g.ws && g.ws_bytes >= decode_split_workspace_bytes(g.M, g.N, g.K)) {
        const int S = decode_split_factor(g.M, g.N, g.K);
        if (S == 4)
            return g.M <= 16 ? run_decode_split<16, 4, 4, 2, 16>(g, st) : run_decode_split<32, 4, 4, 2, 16>(g, st);
        if (S == 2) // two CTAs fit on an SM (shared memory, TMEM and registers)
            return g.M <= 16 ? run_decode_split<16, 2, 3, 2, 16>(g, st) : run_decode_split<32, 2, 2, 2, 8>(g, st);
    }
    // few large copies in flight (three stages of 3-4 K-blocks fill shared memory)
    if (g.M <= 16)
        return run_decode<16, 3, 4, 12>(g, st);
    if (g.M <= 32)
        return run_decode<32, 3, 3, 9>(g, st);
    return run_decode<64, 3, 3, 6>(g, st);
}

// ---------------------------------------------------------------------------
// Allocation-free split-K decode (jetq_gemm_fprop_noalloc): the partial sums
// live in this file-scope device array instead of a caller's workspace.
// Every GPU that loads the library holds it until the process exits; every
// call shares it (overlapping calls race), and no element needs an initial
// value (each call writes every partial it reads).
namespace {
constexpr size_t kStaticScratchBytes = JETQ_NOALLOC_SCRATCH_BYTES;
constexpr int kStaticScratchDevices = 64;
static __device__ __align__(256) float g_decode_static_scratch[kStaticScratchBytes / sizeof(float)];

// The array's device address on the current device.  In host code the
// array's name is only a host-side handle, so the address comes from
// cudaGetSymbolAddress, once per device with that device current, cached.
cudaError_t static_scratch_address(float **out)
{
    static std::mutex mu;
    static float *addr[kStaticScratchDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= kStaticScratchDevices)
        return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void *p = nullptr;
        if ((e = cudaGetSymbolAddress(&p, g_decode_static_scratch)) != cudaSuccess)
            return e;
        addr[dev] = static_cast<float *>(p);
    }
    *out = addr[dev];
    return cudaSuccess;
}
} // namespace

size_t decode_static_scratch_bytes() { return kStaticScratchBytes; }

cudaError_t launch_gemm_decode_static(GemmProblem g, cudaStream_t st)
{
    if (decode_split_workspace_bytes(g.M, g.N, g.K) > kStaticScratchBytes)
        return cudaErrorInvalidValue;
    float *scratch = nullptr;
    cudaError_t e = static_scratch_address(&scratch);
    if (e != cudaSuccess)
        return e;
    g.ws = scratch;
    g.ws_bytes = kStaticScratchBytes;
    return launch_gemm_block128(g, GemmShape::Decode, st);
}

cudaError_t gemm_decode_read_and_clear_error(cudaStream_t st, unsigned *out)
{
    unsigned v = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(&v, g_gemm_decode_error, sizeof v, 0, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(st);
    if (e != cudaSuccess)
        return e;
    *out |= v;
    if (v) {
        const unsigned zero = 0;
        e = cudaMemcpyToSymbolAsync(g_gemm_decode_error, &zero, sizeof zero, 0, cudaMemcpyHostToDevice, st);
        if (e == cudaSuccess)
            e = cudaStreamSynchronize(st);
    }
    return e;
}

} // namespace jetq
