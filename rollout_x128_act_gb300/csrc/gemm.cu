// Block-scaled FP8 GEMM (128-block recipe) on sm_103a tensor cores.
//
//   out[m, n] = sum over K-blocks kb of  fl32(Sa[m,kb] * Sb[n,kb]) * P_kb[m, n]
//   P_kb[m, n] = sum_{k in kb} qa[m, k] * qb[n, k]      (E4M3 x E4M3 -> FP32)
//
// Per-128-K-block FP32 scales (Jet-RL: 1x128 activation groups, 128x128
// weight blocks; FP32 scales are applied outside the tensor core on
// Blackwell, as the Miles Blackwell-recipes post notes) cannot ride the
// native block-scaled MMA, so each K-block is one MMA group into a fresh TMEM
// accumulator and the scale is applied ("promoted") by CUDA cores:
//
//   warp 0        TMA producer: A and B K-block tiles (128-byte swizzle) into
//                 a STAGES-deep shared-memory ring
//   warp 1        MMA issuer: 4 x tcgen05.mma (K = 32 each) per K-block into
//                 its TMEM buffer, then tcgen05.commit to release the smem
//                 stage and to signal the epilogue (one commit per stage of
//                 KBP K-blocks)
//   warp 2        (WGrad) bulk copies of the per-column scales into a ring
//   warp 3        builds the per-expert tile tables of a grouped launch
//   warps 4..     epilogue: tcgen05.ld the K-block partial, acc = fma(P, s, acc)
//                 in registers (packed f32x2), release the TMEM buffer; after
//                 the last K-block, store the tile
//
// One CTA per SM, persistent over output tiles.  The same template serves the
// training shape (BN = 256, 8 epilogue warps, 2 TMEM buffers) and a narrow
// decode shape (BN = 32 weight rows per tile, 4 epilogue warps, four K-blocks
// per TMA copy) for token batches that gemm_decode.cu does not take.  Both
// perform the identical per-element operation sequence, so a decode row
// equals the corresponding training row bit for bit.  Grouped launches (MoE
// experts) run the same loop over per-expert tiles (sched.cuh).
//
// Every mbarrier wait is bounded (wall clock); a CTA that gives up raises a
// shared abort flag, records the fact in the device error word, drains its
// own TMA copies and MMAs (again bounded) and frees its TMEM.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>

#include "jetq_internal.h"
#include "ptx.cuh"
#include "sched.cuh"


namespace jetq {

__device__ unsigned g_gemm_error;

namespace {

constexpr unsigned kErrTimeout = 1u;
constexpr unsigned kErrLayout = 2u;
constexpr unsigned long long kWaitLimitNs = 2000000000ull; // 2 s per wait

struct KParams {
    Sched sched;
    const float *sa;        // [K-blocks x sa_ld]
    const float *sb;        // Block128: [E x N/128 x kb_total]; PerRow: [K-blocks x N]
    int64_t sa_ld;          // rows of the A scale grid
    int kb_total;           // K-blocks of one weight's scale grid (Block128)
    int64_t sb_e_stride;    // floats between experts' weight scales
    int box_a_rows;
    int box_b_rows;
    void *out;
    int64_t ldo;
    int64_t out_e_stride;   // elements between experts' outputs (grouped K)
    int out_bf16;
    int accumulate;
    int tma_out;            // BF16 tiles leave through the output tensor map
    unsigned long long limit_ns;
};

__host__ __device__ constexpr int gcd_int(int a, int b) { return b ? gcd_int(b, a % b) : a; }
__host__ __device__ constexpr int lcm_int(int a, int b) { return a / gcd_int(a, b) * b; }

// Epilogue of the narrow decode tiles: 16-column TMEM loads, the next one in
// flight while the current one is folded; 2 KB per-warp store staging.
struct EpiNarrow {
    static constexpr bool kWide = false;
    static constexpr int STG_BUFS = 1;
    static constexpr int LDX = 16, REG_WG0 = 0, REG_EPI = 0, DEPTH = 1;
    static constexpr int TMA_OUT = 0;
};

// Epilogue of the training tiles: the producer/MMA warpgroup hands registers
// to the epilogue warpgroups (REG_WG0 / REG_EPI per thread); TMEM is read in
// groups of DEPTH loads of LDX columns per wait; the K-blocks' scales arrive
// in a shared-memory ring filled ahead by warp 2 (per-thread asynchronous
// copies), so no global load sits on the fold's path; tiles leave through
// TMA stores of 32-row x 64-byte boxes from a per-warp staging area.
template <int LDX_, int DEPTH_, int REG_WG0_, int REG_EPI_, int STG_BUFS_ = 1>
struct EpiWide {
    static constexpr bool kWide = true;
    static constexpr int LDX = LDX_, DEPTH = DEPTH_, REG_WG0 = REG_WG0_, REG_EPI = REG_EPI_;
    static constexpr int TMA_OUT = 1;
    // 2 KB staging buffers per epilogue warp: with two, a pass is written while
    // the previous pass's TMA store still reads the other one
    static constexpr int STG_BUFS = STG_BUFS_;
};

template <int BN, int EPI_WARPS, int STAGES, int TMEM_BUFS, int A_STRIDE_MAX = 16384, int KBP = 1,
          bool PER_ROW_B = false, class E = EpiNarrow>
struct Cfg {
    static constexpr int kABytes = 128 * 128;
    static constexpr int kBBytes = BN * 128;
    // A stage holds KBP K-blocks and B stage KBP K-blocks (one TMA box each when
    // KBP > 1: a decode slice of 32 weight rows moves 4 KB per K-block, too little
    // per copy to keep HBM busy).  A K-blocks sit A_STRIDE_MAX (or less, for a
    // decode batch of <= A_STRIDE_MAX/128 rows) apart; an M = 128 MMA reads 16 KB
    // from a K-block's base, so the rows past a short A tile are the next
    // K-blocks' bytes: don't-care rows whose results are never stored.  The
    // region keeps every such read inside it.
    static constexpr int kARegion = (STAGES * KBP - 1) * A_STRIDE_MAX + kABytes;
    // warpgroup 0: TMA producer (warp 0), MMA issuer (warp 1), column-scale
    // producer (warp 2, WGrad), group tables (warp 3); warpgroups 1..: epilogue
    static constexpr int kThreads = 128 + 32 * EPI_WARPS;
    static constexpr int kCols = BN / (EPI_WARPS / 4); // accumulator columns per epilogue thread
    static constexpr int kTmemCols = 512;
    // scale ring: narrow tiles, WGrad column scales only (bulk copies); training
    // tiles, each slot the K-block's 128 row scales then its column scales
    // (per-row B) or weight-block scales (4 floats)
    static constexpr int kSbSlots = E::kWide ? 8 : 4;
    static constexpr int kSlotFloats = E::kWide ? 128 + (PER_ROW_B ? BN : 4) : BN;
    static constexpr int kBars = 2 * STAGES + 2 * TMEM_BUFS + 2 * kSbSlots + 1;
    static constexpr size_t kSbBytes =
        (E::kWide || PER_ROW_B) ? ((size_t)kSbSlots * kSlotFloats * 4 + 1023) / 1024 * 1024 : 0;
    // output staging per epilogue warp: 32 rows x 64 bytes (the stores' unit)
    static constexpr size_t kStgWarp = 2048 * (size_t)E::STG_BUFS;
    static constexpr size_t kStageOutBytes = (size_t)EPI_WARPS * kStgWarp;
    // layout: barriers (512 B) and group tables first, then 1024-aligned tiles,
    // the column-scale ring and the output staging.  With TMA stores the size
    // assumes the dynamic shared memory starts on a 1024-byte boundary (the
    // kernel checks that the layout fits before it touches anything).
    static constexpr size_t kFront = 512 + sizeof(GroupTables);
    static constexpr size_t kFrontAligned = (kFront + 1023) / 1024 * 1024;
    static constexpr size_t kSmem = kFrontAligned + (size_t)kARegion + (size_t)STAGES * KBP * kBBytes + kSbBytes +
                                    kStageOutBytes + (E::TMA_OUT ? 0 : 1024);
    static_assert(!E::kWide || (KBP == 1 && kCols % 64 == 0 && kCols % (E::LDX * E::DEPTH) == 0 &&
                                (kSlotFloats * 4) % 16 == 0),
                  "wide epilogue");
    static_assert(!E::kWide || E::REG_WG0 == 0 ||
                      E::REG_WG0 * 128 + E::REG_EPI * 32 * EPI_WARPS <= 65536, "register split exceeds the SM");
    static_assert(TMEM_BUFS * BN <= kTmemCols, "TMEM buffers exceed 512 columns");
    static_assert(EPI_WARPS % 4 == 0 && kCols % 32 == 0, "epilogue split");
    static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "MMA N for M = 128");
    static_assert(kBars * 8 + 16 <= 512, "barrier area");
    static_assert(kSbBytes % 1024 == 0, "staging alignment");
    static_assert(E::kWide || !PER_ROW_B, "per-row B scales are folded by the training-tile epilogue");
    static_assert(A_STRIDE_MAX % 1024 == 0 && A_STRIDE_MAX <= kABytes, "A stages on 1024-byte swizzle atoms");
    static_assert(kSmem <= 232448, "shared memory");
};

template <int BN, int EPI_WARPS, int STAGES, int TMEM_BUFS, bool PER_ROW_B, int A_STRIDE_MAX, int KBP, int PF,
          class E>
__global__ void __launch_bounds__(128 + 32 * EPI_WARPS, 1)
    k_gemm_b128(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmO, const KParams p)
{
    using C = Cfg<BN, EPI_WARPS, STAGES, TMEM_BUFS, A_STRIDE_MAX, KBP, PER_ROW_B, E>;
    constexpr int SB = C::kSbSlots;
    extern __shared__ uint8_t smem_raw[];
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem_raw);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + C::kBars);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    GroupTables *gt = reinterpret_cast<GroupTables *>(smem_raw + 512);
    uint8_t *tiles_a = ptx::align_smem<1024>(smem_raw + C::kFront);
    uint8_t *tiles_b = tiles_a + C::kARegion;
    float *sb_ring = reinterpret_cast<float *>(tiles_b + (size_t)STAGES * KBP * C::kBBytes);
    uint8_t *stage_out = reinterpret_cast<uint8_t *>(sb_ring) + C::kSbBytes;
    // the layout must fit the allocation (it does unless the dynamic shared
    // memory starts far off a 1024-byte boundary): otherwise report and stop
    if (ptx::smem_addr(stage_out + C::kStageOutBytes) - ptx::smem_addr(smem_raw) > (uint32_t)C::kSmem) {
        if (threadIdx.x == 0)
            atomicOr(&g_gemm_error, kErrLayout);
        return;
    }

    const uint32_t bar0 = ptx::smem_addr(bars);
    auto full = [&](int s) { return bar0 + 8u * s; };
    auto empty = [&](int s) { return bar0 + 8u * (STAGES + s); };
    auto tfull = [&](int b) { return bar0 + 8u * (2 * STAGES + b); };
    auto tempty = [&](int b) { return bar0 + 8u * (2 * STAGES + TMEM_BUFS + b); };
    auto sfull = [&](int s) { return bar0 + 8u * (2 * STAGES + 2 * TMEM_BUFS + s); };
    auto sempty = [&](int s) { return bar0 + 8u * (2 * STAGES + 2 * TMEM_BUFS + SB + s); };
    const uint32_t done = bar0 + 8u * (2 * STAGES + 2 * TMEM_BUFS + 2 * SB);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const Sched &sc = p.sched;
    unsigned *err = &g_gemm_error;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(full(s), 1);
            ptx::mbar_init(empty(s), 1);
        }
        for (int b = 0; b < TMEM_BUFS; ++b) {
            ptx::mbar_init(tfull(b), 1);
            ptx::mbar_init(tempty(b), EPI_WARPS * 32); // every epilogue thread arrives
        }
        for (int s = 0; s < SB; ++s) {
            ptx::mbar_init(sfull(s), E::kWide ? 32 : 1); // training tiles: one cp.async arrival per lane
            ptx::mbar_init(sempty(s), EPI_WARPS * 32);
        }
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
    // the prologue above overlaps the stream's previous kernel; global memory
    // (the segment offsets included) only after it has completed
    ptx::grid_dep_launch();
    ptx::grid_dep_wait();
    if (warp == 3 && sc.mode != kDense)
        build_group_tables(sc, gt);
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int num_tiles = total_tiles(sc, gt);
    if constexpr (E::REG_WG0 > 0) {
        if (warp < 4)
            ptx::setmaxnreg_dec<E::REG_WG0>();
        else
            ptx::setmaxnreg_inc<E::REG_EPI>();
    }

    if (warp < 4) {
        if (warp == 0 && lane == 0) {
            // -------------------------------------------------- TMA producer
            // a box past the last K-block is zero-filled and still counts in full
            const uint32_t tx = (uint32_t)(KBP * (p.box_a_rows + p.box_b_rows) * 128);
            uint32_t it = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
                const TileInfo ti = get_tile(sc, gt, t);
                for (int kb = 0; kb < ti.num_kb; kb += KBP, ++it) {
                    const int s = (int)(it % STAGES);
                    const uint32_t ph = (it / STAGES) & 1u;
                    if (!ptx::mbar_wait(empty(s), ph ^ 1u, abort_flag, err, kErrTimeout, p.limit_ns)) {
                        ok = false;
                        break;
                    }
                    ptx::mbar_arrive_expect_tx(full(s), tx);
                    const uint32_t da = ptx::smem_addr(tiles_a + (size_t)s * KBP * A_STRIDE_MAX);
                    const uint32_t db = ptx::smem_addr(tiles_b + (size_t)s * KBP * C::kBBytes);
                    if constexpr (KBP == 1) {
                        ptx::tma_load_2d(da, &tmA, full(s), (ti.kb0 + kb) * 128, ti.a_row0);
                        ptx::tma_load_2d(db, &tmB, full(s), (ti.kb0 + kb) * 128, ti.b_row0);
                    } else {
                        ptx::tma_load_3d(da, &tmA, full(s), 0, ti.a_row0, ti.kb0 + kb);
                        ptx::tma_load_3d(db, &tmB, full(s), 0, ti.b_row0, ti.kb0 + kb);
                    }
                }
            }
            // drain: every copy this thread started must have landed before exit
            for (int s = 0; s < STAGES; ++s) {
                if (it > (uint32_t)s) {
                    const uint32_t last = (uint32_t)s + ((it - 1u - (uint32_t)s) / STAGES) * STAGES;
                    ptx::mbar_wait(full(s), (last / STAGES) & 1u, abort_flag, err, kErrTimeout, p.limit_ns, false);
                }
            }
        } else if (warp == 1 && lane == 0) {
            // -------------------------------------------------- MMA issuer
            // Every MMA operand is a base register plus a compile-time offset
            // (the loop below is unrolled so that stage and buffer indices are
            // constants): an operand computed inside the loop costs the issue a
            // few hundred cycles, more than a narrow MMA takes to run.
            constexpr uint32_t idesc = ptx::idesc_e4m3_f32(128, BN);
            constexpr int NG = TMEM_BUFS / KBP; // accumulator groups: one per stage, KBP buffers each
            constexpr int U = lcm_int(STAGES, NG);
            static_assert(TMEM_BUFS % KBP == 0, "buffer groups");
            const uint64_t adesc0 = ptx::desc_kmajor_sw128(ptx::smem_addr(tiles_a));
            const uint64_t bdesc0 = ptx::desc_kmajor_sw128(ptx::smem_addr(tiles_b));
            // the stages this CTA consumes, in order; with KBP > 1 (dense
            // problems only) every tile takes spt stages, the last holding
            // last_nk K-blocks; the buffers of missing K-blocks stay unused
            int total = 0;
            for (int t = blockIdx.x; t < num_tiles; t += gridDim.x)
                total += (get_tile(sc, gt, t).num_kb + KBP - 1) / KBP;
            const int spt = (sc.num_kb + KBP - 1) / KBP;
            const int last_nk = sc.num_kb - (spt - 1) * KBP;
            bool ok = true;
            for (int q0 = 0; q0 < total && ok; q0 += U) {
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int q = q0 + u;
                    if (q < total && ok) {
                        const int s = u % STAGES;
                        const int gi = u % NG;
                        const int nk = KBP == 1 ? 1 : (q % spt == spt - 1 ? last_nk : KBP);
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
                                    const uint64_t ad = adesc0 + (uint64_t)(((s * KBP + j) * A_STRIDE_MAX) >> 4);
                                    const uint64_t bd = bdesc0 + (uint64_t)(((s * KBP + j) * C::kBBytes) >> 4);
                                    const uint32_t d = tmem_base + (uint32_t)((gi * KBP + j) * BN);
#pragma unroll
                                    for (int k = 0; k < 4; ++k) // 4 x K=32 (32 bytes) in the 128-byte swizzle row
                                        ptx::mma_f8f6f4(d, ad + 2u * k, bd + 2u * k, idesc, k > 0 ? 1u : 0u);
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
        } else if (E::kWide && warp == 2) {
            // -------------------------------------------------- scale producer (training tiles)
            // Per K-block: the tile's 128 row scales and its column scales (per-row B:
            // BN of them) or weight-block scales, copied by the 32 lanes with cp.async
            // into a ring slot; each lane's copies complete as one arrival on sfull.
            uint32_t it = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
                const TileInfo ti = get_tile(sc, gt, t);
                for (int kb = 0; kb < ti.num_kb; ++kb, ++it) {
                    const int slot = (int)(it % SB);
                    if (!ptx::mbar_wait(sempty(slot), ((it / SB) & 1u) ^ 1u, abort_flag, err, kErrTimeout,
                                        p.limit_ns)) {
                        ok = false;
                        break;
                    }
                    const int kbg = ti.kb0 + kb;
                    float *ring = sb_ring + (size_t)slot * C::kSlotFloats;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int64_t m = (int64_t)ti.a_row0 + lane + 32 * i;
                        const bool in = m < sc.M;
                        ptx::cp_async_4(ptx::smem_addr(ring + lane + 32 * i),
                                        p.sa + (in ? (int64_t)kbg * p.sa_ld + m : 0), in ? 4u : 0u);
                    }
                    if constexpr (PER_ROW_B) {
                        for (int c4 = lane; c4 < BN / 4; c4 += 32) {
                            const int n = ti.n0 + 4 * c4;
                            const bool in = n < sc.N; // N is a multiple of 64
                            ptx::cp_async_16(ptx::smem_addr(ring + 128 + 4 * c4),
                                             p.sb + (in ? (int64_t)kbg * sc.N + n : 0), in ? 16u : 0u);
                        }
                    } else {
                        if (lane < BN / 128) {
                            const int n = ti.n0 + 128 * lane;
                            const bool in = n < sc.N;
                            ptx::cp_async_4(ptx::smem_addr(ring + 128 + lane),
                                            p.sb + (in ? ti.e * p.sb_e_stride + (int64_t)(n >> 7) * p.kb_total + kbg
                                                       : 0),
                                            in ? 4u : 0u);
                        }
                    }
                    ptx::cp_async_mbar_arrive(sfull(slot));
                }
            }
            ptx::cp_async_wait_all();
        }
        __syncwarp();
    } else if constexpr (E::kWide) {
        // ------------------------------------------------------ epilogue (training tiles)
        constexpr int LDX = E::LDX;
        constexpr int GC = LDX * E::DEPTH;   // columns per TMEM wait
        constexpr int NGR = C::kCols / GC;
        const int ew = warp - 4;
        const int quarter = warp & 3; // TMEM lanes 32*quarter .. +31
        const int col0 = (ew >> 2) * C::kCols;
        const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
        uint8_t *stg = stage_out + (size_t)ew * C::kStgWarp;

        uint32_t tb = 0; // K-blocks folded so far (TMEM buffer tb % TMEM_BUFS, scale slot tb % SB)
        bool ok = true;
        uint32_t npass = 0; // store passes of this warp so far (staging buffer npass % STG_BUFS)
        for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
            const TileInfo ti = get_tile(sc, gt, t);
            const int64_t mw = (int64_t)ti.a_row0 + quarter * 32; // the warp's first row
            const int n0 = ti.n0 + col0;
            const bool col_ok = n0 < sc.N; // a slice past N (N % BN != 0) computes nothing it stores
            float2 acc[C::kCols / 2];
#pragma unroll
            for (int j = 0; j < C::kCols / 2; ++j)
                acc[j] = make_float2(0.0f, 0.0f);

            for (int kb = 0; kb < ti.num_kb; ++kb) {
                const int b = (int)(tb % TMEM_BUFS);
                const int slot = (int)(tb % SB);
                bool got = ptx::mbar_wait(sfull(slot), (tb / SB) & 1u, abort_flag, err, kErrTimeout, p.limit_ns);
                got = got && ptx::mbar_wait(tfull(b), (tb / TMEM_BUFS) & 1u, abort_flag, err, kErrTimeout, p.limit_ns);
                if (!__all_sync(0xFFFFFFFFu, got)) { // keep the warp converged for tcgen05.ld
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const float *ring = sb_ring + (size_t)slot * C::kSlotFloats;
                const float sa = ring[quarter * 32 + lane];
                const float *sbs = ring + 128 + col0;              // per-row B: this slice's column scales
                const float s = PER_ROW_B ? 0.0f : __fmul_rn(sa, ring[128 + (col0 >> 7)]);
                const uint32_t tbase = tmem_base + lane_addr + (uint32_t)(b * BN + col0);
                uint32_t Q[GC];
#pragma unroll
                for (int gr = 0; gr < NGR; ++gr) {
#pragma unroll
                    for (int d = 0; d < E::DEPTH; ++d)
                        ptx::tmem_ld_x(tbase + (uint32_t)(gr * GC + d * LDX),
                                       *reinterpret_cast<uint32_t(*)[LDX]>(&Q[d * LDX]));
                    ptx::tmem_ld_wait_tie(Q);
                    if (gr == NGR - 1) {
                        // every load of buffer b has completed: hand it back to the MMA
                        ptx::tc_fence_before();
                        ptx::mbar_arrive(tempty(b));
                    }
                    if constexpr (PER_ROW_B) {
#pragma unroll
                        for (int q = 0; q < GC / 4; ++q) {
                            const float4 sb4 = *reinterpret_cast<const float4 *>(sbs + gr * GC + 4 * q);
                            const float2 s01 = __fmul2_rn(make_float2(sa, sa), make_float2(sb4.x, sb4.y));
                            const float2 s23 = __fmul2_rn(make_float2(sa, sa), make_float2(sb4.z, sb4.w));
                            float2 &a0 = acc[gr * (GC / 2) + 2 * q];
                            float2 &a1 = acc[gr * (GC / 2) + 2 * q + 1];
                            a0 = __ffma2_rn(make_float2(__uint_as_float(Q[4 * q]), __uint_as_float(Q[4 * q + 1])), s01,
                                            a0);
                            a1 = __ffma2_rn(make_float2(__uint_as_float(Q[4 * q + 2]), __uint_as_float(Q[4 * q + 3])),
                                            s23, a1);
                        }
                    } else {
                        const float2 s2 = make_float2(s, s);
#pragma unroll
                        for (int h = 0; h < GC / 2; ++h)
                            acc[gr * (GC / 2) + h] = __ffma2_rn(
                                make_float2(__uint_as_float(Q[2 * h]), __uint_as_float(Q[2 * h + 1])), s2,
                                acc[gr * (GC / 2) + h]);
                    }
                }
                ptx::mbar_arrive(sempty(slot)); // the slot's scales have been read
                ++tb;
            }
            if (!ok)
                break;

            // ---- store the tile: passes of 64 bytes per row (32 BF16 or 16 FP32 columns),
            // each written into the warp's staging area with its 16-byte chunks swizzled by
            // row (the 64-byte swizzle of the output tensor map: conflict-free), then stored
            // by one TMA box of 32 rows, or (rows past a problem's end, accumulation) read
            // back as 8 rows x 64 contiguous bytes per store instruction
            const bool tma = p.tma_out && !p.accumulate && col_ok &&
                             (mw + 32 <= ti.m_end || (ti.m_end == sc.M && sc.mode != kGroupedK));
            const int64_t out_row0 = (sc.mode == kGroupedK ? (int64_t)ti.e * sc.M : 0) + mw;
            auto pass = [&](int px, auto chunk, auto store) {
                uint8_t *buf = stg + (size_t)(npass % E::STG_BUFS) * 2048;
                ++npass;
                // the store that last used this buffer must have finished reading it
                if (lane == 0)
                    ptx::bulk_wait_group_read<E::STG_BUFS - 1>();
                __syncwarp();
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    *reinterpret_cast<uint4 *>(buf + lane * 64 + ((c ^ ((lane >> 1) & 3)) << 4)) = chunk(c);
                if (tma) {
                    ptx::fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        ptx::tma_store_2d(&tmO, ptx::smem_addr(buf), px, (int)out_row0);
                        ptx::bulk_commit_group();
                    }
                } else {
                    __syncwarp();
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int pc = lane + 32 * i, r = pc >> 2, c = pc & 3;
                        const uint4 v = *reinterpret_cast<const uint4 *>(buf + r * 64 + ((c ^ ((r >> 1) & 3)) << 4));
                        if (col_ok && mw + r < ti.m_end)
                            store(mw + r, c, v);
                    }
                    __syncwarp();
                }
            };
            if (p.out_bf16) {
#pragma unroll
                for (int ps = 0; ps < C::kCols / 32; ++ps) // 32 BF16 columns a pass
                    pass(
                        n0 + ps * 32,
                        [&](int c) {
                            uint32_t w[4];
#pragma unroll
                            for (int h = 0; h < 4; ++h) {
                                const float2 a = acc[ps * 16 + 4 * c + h];
                                const __nv_bfloat162 b2 = __floats2bfloat162_rn(a.x, a.y);
                                w[h] = *reinterpret_cast<const uint32_t *>(&b2);
                            }
                            return make_uint4(w[0], w[1], w[2], w[3]);
                        },
                        [&](int64_t row, int c, const uint4 &v) {
                            *reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(p.out) + row * p.ldo + n0 +
                                                       ps * 32 + c * 8) = v;
                        });
            } else if (!p.accumulate) {
#pragma unroll
                for (int ps = 0; ps < C::kCols / 16; ++ps) // 16 FP32 columns a pass
                    pass(
                        n0 + ps * 16,
                        [&](int c) {
                            const float2 a = acc[ps * 8 + 2 * c], b2 = acc[ps * 8 + 2 * c + 1];
                            return make_uint4(__float_as_uint(a.x), __float_as_uint(a.y), __float_as_uint(b2.x),
                                              __float_as_uint(b2.y));
                        },
                        [&](int64_t row, int c, const uint4 &v) {
                            *reinterpret_cast<uint4 *>(reinterpret_cast<float *>(p.out) + ti.e * p.out_e_stride +
                                                       row * p.ldo + n0 + ps * 16 + c * 4) = v;
                        });
            } else {
                const int64_t m = mw + lane;
                if (m < ti.m_end && col_ok) {
                    float *o = reinterpret_cast<float *>(p.out) + ti.e * p.out_e_stride + m * p.ldo + n0;
#pragma unroll
                    for (int j4 = 0; j4 < C::kCols / 4; ++j4) {
                        float4 v = make_float4(acc[2 * j4].x, acc[2 * j4].y, acc[2 * j4 + 1].x, acc[2 * j4 + 1].y);
                        const float4 old = *reinterpret_cast<const float4 *>(o + 4 * j4);
                        v.x = __fadd_rn(old.x, v.x);
                        v.y = __fadd_rn(old.y, v.y);
                        v.z = __fadd_rn(old.z, v.z);
                        v.w = __fadd_rn(old.w, v.w);
                        *reinterpret_cast<float4 *>(o + 4 * j4) = v;
                    }
                }
            }
        }
        // every TMA store of this warp must complete before the CTA exits
        if (lane == 0)
            ptx::bulk_wait_group0();
        __syncwarp();
    } else {
        // ------------------------------------------------------ epilogue (narrow decode tiles)
        static_assert(!PER_ROW_B && BN < 128 && PF > 1, "narrow epilogue: decode tiles only");
        const int ew = warp - 4;
        const int quarter = warp & 3; // TMEM lanes 32*quarter .. +31
        const int col0 = (ew >> 2) * C::kCols;
        const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;

        uint32_t tb = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
            const TileInfo ti = get_tile(sc, gt, t);
            const int64_t m = (int64_t)ti.a_row0 + quarter * 32 + lane;
            const bool row_ok = m < ti.m_end;
            const bool load_ok = m < sc.M;
            const int n0 = ti.n0 + col0;
            const bool col_ok = n0 < sc.N; // a slice past N (N % BN != 0) computes nothing it stores
            const float *sa_ptr = p.sa + (load_ok ? m : 0);
            const float *sb_ptr = p.sb + ti.e * p.sb_e_stride + (col_ok ? (int64_t)(n0 >> 7) * p.kb_total : 0);
            float2 acc[C::kCols / 2];
#pragma unroll
            for (int j = 0; j < C::kCols / 2; ++j)
                acc[j] = make_float2(0.0f, 0.0f);

            // fold one K-block's accumulator buffer into acc with scale s; buffers come in
            // groups of KBP, one group per stage, waited for at the group's first K-block and
            // released after its last (use = false: a K-block past the tile's end, whose
            // buffer only passes through)
            auto fold = [&](float s, bool use) -> bool {
                constexpr int NG = TMEM_BUFS / KBP;
                const int j = (int)(tb % KBP);
                const int gi = (int)((tb / KBP) % NG);
                const int b = (int)(tb % TMEM_BUFS);
                bool got = true;
                if (j == 0)
                    got = ptx::mbar_wait(tfull(gi), ((tb / KBP) / NG) & 1u, abort_flag, err, kErrTimeout, p.limit_ns);
                if (!__all_sync(0xFFFFFFFFu, got)) // keep the warp converged for tcgen05.ld
                    return false;
                ptx::tc_fence_after();
                // 16-column chunks, the next one in flight while the current one is folded (a
                // warp whose 32 rows are all past the tile's rows has nothing to keep)
                if (use && ti.a_row0 + quarter * 32 < ti.m_end) {
                    constexpr int NCH = C::kCols / 16;
                    uint32_t PP[2][16];
                    const uint32_t tbase = tmem_base + lane_addr + (uint32_t)(b * BN + col0);
                    ptx::tmem_ld_32x32b_x16(tbase, PP[0]);
                    ptx::tmem_ld_wait_regs(PP[0]);
#pragma unroll
                    for (int ch = 0; ch < NCH; ++ch) {
                        if (ch + 1 < NCH)
                            ptx::tmem_ld_32x32b_x16(tbase + (uint32_t)((ch + 1) * 16), PP[(ch + 1) & 1]);
                        const uint32_t (&P)[16] = PP[ch & 1];
                        const float2 s2 = make_float2(s, s);
#pragma unroll
                        for (int h = 0; h < 8; ++h)
                            acc[ch * 8 + h] = __ffma2_rn(
                                make_float2(__uint_as_float(P[2 * h]), __uint_as_float(P[2 * h + 1])), s2, acc[ch * 8 + h]);
                        if (ch + 1 < NCH)
                            ptx::tmem_ld_wait_regs(PP[(ch + 1) & 1]);
                    }
                }
                ptx::tc_fence_before();
                if (j == KBP - 1)
                    ptx::mbar_arrive(tempty(gi));
                ++tb;
                return true;
            };
            // the scales of PF K-blocks in flight: a decode slice spends too little
            // time per K-block to hide one global load behind the next
            float qa[PF], qb[PF];
#pragma unroll
            for (int u = 0; u < PF; ++u) {
                const bool in = u < ti.num_kb;
                qa[u] = in && load_ok ? __ldg(sa_ptr + (int64_t)(ti.kb0 + u) * p.sa_ld) : 0.0f;
                qb[u] = in && col_ok ? __ldg(sb_ptr + ti.kb0 + u) : 0.0f;
            }
            for (int kb0 = 0; kb0 < ti.num_kb && ok; kb0 += PF) {
#pragma unroll
                for (int u = 0; u < PF; ++u) {
                    const int kb = kb0 + u;
                    if (kb < ti.num_kb && ok) {
                        const float s = __fmul_rn(qa[u], qb[u]);
                        const int kn = kb + PF;
                        if (kn < ti.num_kb) {
                            qa[u] = load_ok ? __ldg(sa_ptr + (int64_t)(ti.kb0 + kn) * p.sa_ld) : 0.0f;
                            qb[u] = col_ok ? __ldg(sb_ptr + ti.kb0 + kn) : 0.0f;
                        }
                        ok = fold(s, true);
                    }
                }
            }
            if constexpr (KBP > 1) {
                const int padded = (ti.num_kb + KBP - 1) / KBP * KBP;
                for (int kb = ti.num_kb; kb < padded && ok; ++kb)
                    ok = fold(0.0f, false);
            }
            if (!ok)
                break;
            if (row_ok && col_ok) {
                if (p.out_bf16) {
                    __nv_bfloat16 *o = reinterpret_cast<__nv_bfloat16 *>(p.out) + m * p.ldo + n0;
#pragma unroll
                    for (int j8 = 0; j8 < C::kCols / 8; ++j8) {
                        uint4 v;
                        uint32_t *w = reinterpret_cast<uint32_t *>(&v);
#pragma unroll
                        for (int h = 0; h < 4; ++h) {
                            const __nv_bfloat162 b2 = __floats2bfloat162_rn(acc[4 * j8 + h].x, acc[4 * j8 + h].y);
                            w[h] = *reinterpret_cast<const uint32_t *>(&b2);
                        }
                        *reinterpret_cast<uint4 *>(o + 8 * j8) = v;
                    }
                } else {
                    float *o = reinterpret_cast<float *>(p.out) + m * p.ldo + n0;
#pragma unroll
                    for (int j4 = 0; j4 < C::kCols / 4; ++j4) {
                        float4 v = make_float4(acc[2 * j4].x, acc[2 * j4].y, acc[2 * j4 + 1].x, acc[2 * j4 + 1].y);
                        if (p.accumulate) {
                            const float4 old = *reinterpret_cast<const float4 *>(o + 4 * j4);
                            v.x = __fadd_rn(old.x, v.x);
                            v.y = __fadd_rn(old.y, v.y);
                            v.z = __fadd_rn(old.z, v.z);
                            v.w = __fadd_rn(old.w, v.w);
                        }
                        *reinterpret_cast<float4 *>(o + 4 * j4) = v;
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

// Two waiters on mbarriers nothing completes (see jetq_selftest_bounded_wait).
__global__ void __launch_bounds__(64, 1) k_selftest_wait(unsigned long long limit_ns, long long *elapsed_ns)
{
    __shared__ __align__(8) uint64_t bars[2];
    __shared__ int abort_word;
    if (threadIdx.x == 0) {
        ptx::mbar_init(ptx::smem_addr(&bars[0]), 1);
        ptx::mbar_init(ptx::smem_addr(&bars[1]), 1);
        abort_word = 0;
        ptx::fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0 || threadIdx.x == 32) {
        const int w = threadIdx.x >> 5;
        const uint64_t t0 = ptx::globaltimer();
        ptx::mbar_wait(ptx::smem_addr(&bars[w]), 0u, &abort_word, &g_gemm_error, kErrTimeout,
                       w == 0 ? limit_ns : 8ull * limit_ns, w == 1);
        elapsed_ns[w] = (long long)(ptx::globaltimer() - t0);
    }
}

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
    });
    return fn;
}

} // namespace

cudaError_t make_bf16_tile_map(CUtensorMap *map, const void *base, int64_t cols, int64_t rows, int64_t ld)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn)
        return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)ld * 2u};
    const cuuint32_t box[2] = {128u, 128u};
    const cuuint32_t estr[2] = {1u, 1u};
    const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Output map for the training tiles' TMA stores: [rows x cols] of BF16 or
// FP32, boxes of 64 bytes x 32 rows, 64-byte swizzle.
cudaError_t make_store_map(CUtensorMap *map, const void *base, int64_t cols, int64_t rows, int64_t ld, bool bf16)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn)
        return cudaErrorNotSupported;
    const int esize = bf16 ? 2 : 4;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)ld * esize};
    const cuuint32_t box[2] = {(cuuint32_t)(64 / esize), 32u};
    const cuuint32_t estr[2] = {1u, 1u};
    const CUresult r =
        fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void *>(base),
           dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
           CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t make_kmajor_map(CUtensorMap *map, const void *base, int64_t k_extent, int64_t rows, int64_t ld,
                            int box_rows, int kb_per_box)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn)
        return cudaErrorNotSupported;
    CUresult r;
    if (kb_per_box <= 1) {
        const cuuint64_t dims[2] = {(cuuint64_t)k_extent, (cuuint64_t)rows};
        const cuuint64_t strides[1] = {(cuuint64_t)ld};
        const cuuint32_t box[2] = {128u, (cuuint32_t)box_rows};
        const cuuint32_t estr[2] = {1u, 1u};
        r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    } else {
        // (128 bytes of a K-block, row, K-block): the K-block axis steps 128 bytes
        // along the row, so one box lands as kb_per_box consecutive 128-byte-wide
        // swizzled tiles, each the layout a single K-block box would give
        if (k_extent % 128 != 0)
            return cudaErrorInvalidValue;
        const cuuint64_t dims[3] = {128u, (cuuint64_t)rows, (cuuint64_t)(k_extent / 128)};
        const cuuint64_t strides[2] = {(cuuint64_t)ld, 128u};
        const cuuint32_t box[3] = {128u, (cuuint32_t)box_rows, (cuuint32_t)kb_per_box};
        const cuuint32_t estr[3] = {1u, 1u, 1u};
        r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

namespace {

template <int BN, int EPI_WARPS, int STAGES, int TMEM_BUFS, bool PER_ROW_B, int A_STRIDE_MAX = 16384, int KBP = 1,
          int PF = 1, class E = EpiNarrow>
cudaError_t run(const GemmProblem &g, cudaStream_t st)
{
    using C = Cfg<BN, EPI_WARPS, STAGES, TMEM_BUFS, A_STRIDE_MAX, KBP, PER_ROW_B, E>;
    auto kern = k_gemm_b128<BN, EPI_WARPS, STAGES, TMEM_BUFS, PER_ROW_B, A_STRIDE_MAX, KBP, PF, E>;
    if (KBP > 1 && g.group != GroupKind::None)
        return cudaErrorInvalidValue; // multi-K-block boxes serve dense problems only
    static int configured_device = -1;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (configured_device != dev) {
        if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::kSmem)) !=
            cudaSuccess)
            return e;
        if constexpr (E::REG_WG0 > 0) {
            // setmaxnreg.inc waits until the CTA's register pool can serve it: the
            // launch must provide every warpgroup's share, or the kernel would stall
            cudaFuncAttributes fa;
            if ((e = cudaFuncGetAttributes(&fa, kern)) != cudaSuccess)
                return e;
            if (fa.numRegs < E::REG_WG0 || fa.numRegs > E::REG_EPI ||
                fa.numRegs * C::kThreads < E::REG_WG0 * 128 + E::REG_EPI * 32 * EPI_WARPS)
                return cudaErrorInvalidConfiguration;
        }
        configured_device = dev;
    }
    // an epilogue thread stores kCols consecutive columns once the first is in
    // range, so N must be a multiple of that slice
    if (g.N % C::kCols != 0)
        return cudaErrorInvalidValue;
    // B rows the map covers: one weight, or every expert's stacked
    const int64_t b_rows = g.group == GroupKind::Rows ? g.N * g.num_experts : g.N;
    // single-K-block boxes are never taller than the tensor: rows of a stage
    // past the box keep stale bytes, which only reach accumulator rows/columns
    // that are not stored.  A multi-K-block box lays its K-blocks one box
    // height apart, so its A box is exactly as tall as the K-block stride
    // (rows past the batch arrive zero-filled).
    if (KBP > 1 && (b_rows < BN || g.M > A_STRIDE_MAX / 128))
        return cudaErrorInvalidValue;
    const int box_a = KBP > 1 ? A_STRIDE_MAX / 128 : (g.M >= 128 ? 128 : (int)((g.M + 7) / 8 * 8));
    const int box_b = b_rows >= BN ? BN : (int)((b_rows + 7) / 8 * 8);
    CUtensorMap ta, tbm;
    if ((e = make_kmajor_map(&ta, g.a, g.K, g.M, g.lda, box_a, KBP)) != cudaSuccess)
        return e;
    if ((e = make_kmajor_map(&tbm, g.b, g.K, b_rows, g.ldb, box_b, KBP)) != cudaSuccess)
        return e;
    KParams kp;
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
    kp.sa = g.sa;
    kp.sb = g.sb;
    kp.sa_ld = g.M;
    kp.kb_total = (int)(g.K / 128);
    kp.sb_e_stride = g.group == GroupKind::Rows ? (g.N / 128) * (g.K / 128) : 0;
    kp.box_a_rows = box_a;
    kp.box_b_rows = box_b;

    kp.out = g.out;
    kp.ldo = g.ldo;
    kp.out_e_stride = g.group == GroupKind::K ? g.M * g.ldo : 0;
    kp.out_bf16 = g.out_dtype == JETQ_OUT_BF16;
    kp.accumulate = g.accumulate;
    kp.limit_ns = kWaitLimitNs;
    // output tiles leave by TMA when the output rows are 16-byte aligned (a
    // grouped WGrad's experts are stacked: one map over their E x M rows)
    CUtensorMap to;
    memset(&to, 0, sizeof to);
    kp.tma_out = 0;
    if (E::TMA_OUT && !g.accumulate && (g.ldo * (kp.out_bf16 ? 2 : 4)) % 16 == 0 &&
        (reinterpret_cast<uintptr_t>(g.out) & 15u) == 0) {
        const int64_t rows = g.group == GroupKind::K ? g.M * g.num_experts : g.M;
        if ((e = make_store_map(&to, g.out, g.N, rows, g.ldo, kp.out_bf16)) != cudaSuccess)
            return e;
        kp.tma_out = 1;
    }
    int grid = sm_count();
    if (g.group == GroupKind::None) {
        const int tiles = s.mt * s.nt;
        grid = tiles < grid ? tiles : grid;
    } else if (g.group == GroupKind::K) {
        const int tiles = s.mt * s.nt * g.num_experts;
        grid = tiles < grid ? tiles : grid;
    }
    if ((e = launch_pdl(kern, dim3(grid), dim3(C::kThreads), C::kSmem, st, ta, tbm, to, kp)) != cudaSuccess)
        return e;
    return cudaGetLastError();
}

// FProp / DGrad training tiles: 128 x 256, 8 epilogue warps (one row x 128
// columns a thread, 216 registers after the split), TMEM read in 32-column
// groups (two 16-column loads per wait).
cudaError_t run_train(const GemmProblem &g, cudaStream_t st)
{
    // MoE experts' tiles are short (K = hidden): three stages and four staging
    // buffers a warp, so a whole tile's output is staged and its stores drain
    // while the next tile folds (30B-A3B FProp +6%, DGrad +8% measured; the
    // dense shapes keep four stages, which measured as fast or faster)
    if (g.group == GroupKind::Rows)
        return run<256, 8, 3, 2, false, 16384, 1, 1, EpiWide<16, 2, 72, 216, 4>>(g, st);
    return run<256, 8, 4, 2, false, 16384, 1, 1, EpiWide<16, 2, 72, 216>>(g, st);
}

// WGrad (per-column B scales): 128 x 192 tiles folded by three epilogue
// warpgroups (64 columns a thread, one 16-column TMEM load per wait), two
// staging buffers a warp (FP32 tiles are twice the bytes; a MoE expert's WGrad
// tiles can be a few K-blocks long, so the store is a large share).
cudaError_t run_wgrad(const GemmProblem &g, cudaStream_t st)
{
    return run<192, 12, 4, 2, true, 16384, 1, 1, EpiWide<16, 1, 0, 0, 2>>(g, st);
}

} // namespace

cudaError_t launch_gemm_block128(const GemmProblem &g, GemmShape shape, cudaStream_t st)
{
    if (g.M == 0)
        return cudaSuccess;
    // per-row B scales come with WGrad, which always runs the training shape:
    // 192-column tiles folded by three epilogue warpgroups (64 columns a
    // thread, no register spills) and row scales two K-blocks ahead
    if (g.bscale == BScale::PerRow)
        return run_wgrad(g, st);
    if (shape == GemmShape::Train)
        return run_train(g, st);
    if (gemm_decode_swapped_applies(g))
        return launch_gemm_decode_swapped(g, st);
    // past the swapped kernel's 64 tokens the training tiles stream the weight
    // faster once they cover 32 CTAs (same per-element arithmetic either way)
    if (g.group == GroupKind::None && ((g.M + 127) / 128) * ((g.N + 255) / 256) >= 32)
        return run_train(g, st);
    // decode: 32 weight rows per tile, four K-blocks per copy, scales eight
    // K-blocks ahead; a batch of up to 32 (64) tokens packs its A K-blocks
    // 4 KB (8 KB) apart
    if (g.M <= 32)
        return run<32, 4, 6, 8, false, 4096, 4, 8>(g, st);
    if (g.M <= 64)
        return run<32, 4, 4, 8, false, 8192, 4, 8>(g, st);
    return run<32, 4, 8, 8, false, 16384, 1, 8>(g, st);
}

cudaError_t launch_selftest_wait(unsigned long long limit_ns, long long *elapsed_ns, cudaStream_t st)
{
    k_selftest_wait<<<1, 64, 0, st>>>(limit_ns, elapsed_ns);
    return cudaGetLastError();
}

cudaError_t gemm_read_and_clear_error(cudaStream_t st, unsigned *out)
{
    unsigned v = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(&v, g_gemm_error, sizeof v, 0, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(st);
    if (e != cudaSuccess)
        return e;
    *out |= v;
    if (v) {
        const unsigned zero = 0;
        e = cudaMemcpyToSymbolAsync(g_gemm_error, &zero, sizeof zero, 0, cudaMemcpyHostToDevice, st);
        if (e == cudaSuccess)
            e = cudaStreamSynchronize(st);
    }
    return e;
}

} // namespace jetq
