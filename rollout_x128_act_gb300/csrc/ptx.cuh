// Inline-PTX wrappers for the sm_103a features the GEMM kernels use:
// mbarriers, TMA tiled loads, tcgen05 (TMEM allocation, MMA, loads, fences).
#pragma once

#include <cstdint>
#include <cuda.h>

namespace jetq {
namespace ptx {

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// The dynamic shared-memory base rounded up to ALIGN bytes by pointer
// arithmetic on the shared array itself, so that the compiler still knows the
// result is a shared address (plain accesses become shared-memory loads and
// stores, not generic ones).
template <uint32_t ALIGN>
__device__ __forceinline__ uint8_t *align_smem(uint8_t *raw)
{
    const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(raw));
    return raw + ((ALIGN - (a & (ALIGN - 1))) & (ALIGN - 1));
}

__device__ __forceinline__ uint64_t globaltimer()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ------------------------------------------------------------------ mbarrier

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Orders this thread's generic-proxy accesses to shared memory against later
// async-proxy accesses (TMA / bulk copies, tcgen05.cp) to the same bytes.
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// The same with acquire at cluster scope: for phases completed by arrivals of
// other CTAs of the cluster (their writes to this CTA's shared memory before
// the arrive are visible after the wait).
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits for the phase with the given parity.  Gives up after limit_ns of
// wall time, or (when honor_abort) as soon as another thread of the CTA has
// given up (abort flag in shared memory); on timing out it raises the abort
// flag, records `code` in the device error word and returns false.
template <bool kClusterAcquire = false>
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                          unsigned *err_word, unsigned code, uint64_t limit_ns,
                                          bool honor_abort = true)
{
    auto poll = [&]() { return kClusterAcquire ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity); };
    if (poll())
        return true;
    const uint64_t t0 = globaltimer();
    for (uint32_t i = 1;; ++i) {
        if (poll())
            return true;
        if ((i & 31u) == 0u) {
            if (honor_abort && *abort_flag)
                return false;
            if (globaltimer() - t0 > limit_ns) {
                *abort_flag = 1;
                atomicOr(err_word, code);
                return false;
            }
        }
    }
}

// ------------------------------------------------------------------ TMA

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, uint32_t bar, int x, int y)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
        : "memory");
}

// 1-D bulk copy global -> shared (both 16-byte aligned, size a multiple of 16),
// completion counted on the mbarrier in bytes.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

// 3-D tiled load: coordinates (x, y, z) in the map's element units
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, uint32_t bar, int x, int y, int z)
{
    asm volatile("cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                 " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
                 "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
                 : "memory");
}

__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Shared-memory address of the same offset in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_cta(uint32_t saddr, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}

// Arrive on an mbarrier of another CTA of the cluster (release at cluster scope).
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr)
{
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// Bulk copy from this CTA's shared memory into the shared memory of a CTA of
// the cluster; completion (bytes) is signalled on an mbarrier of the
// destination CTA.  dst and bar come from map_to_cta; addresses 16-byte
// aligned, size a multiple of 16.
__device__ __forceinline__ void bulk_copy_to_cta(uint32_t dst_cluster, uint32_t src, uint32_t bytes,
                                                 uint32_t bar_cluster)
{
    asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     dst_cluster),
                 "r"(src), "r"(bytes), "r"(bar_cluster)
                 : "memory");
}

// 16-byte store to this CTA's shared memory (shared-window address).
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d)
{
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// Arrive on an mbarrier of another CTA of the cluster with the default
// (CTA-scope release) semantics: the consumer release of a pipeline slot that
// the peer next overwrites with a bulk copy; the releasing threads have
// consumed the slot's values before they arrive.
__device__ __forceinline__ void mbar_arrive_remote_cta(uint32_t cluster_addr)
{
    asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// Programmatic dependent launch.  grid_dep_wait: the executing thread waits
// until the kernels this one may overlap (the stream's preceding kernel, when
// the launch allowed it) have completed and their memory is visible; a no-op
// otherwise.  grid_dep_launch: this CTA allows the stream's next kernel to
// start (its own prologue; it waits in grid_dep_wait before touching memory).
__device__ __forceinline__ void grid_dep_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void grid_dep_launch()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Named barrier `id` (1..15) over `count` threads (whole warps) of the CTA;
// the threads of a warp may arrive apart (non-aligned form).
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t count)
{
    asm volatile("barrier.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Hardware cluster barrier (every thread of every CTA of the cluster).
__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Per-thread asynchronous copies global -> shared of 4 or 16 bytes; src_size
// bytes are read (0 reads nothing) and the rest of the destination is zeroed.
__device__ __forceinline__ void cp_async_4(uint32_t dst, const void *src, uint32_t src_size)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(src_size) : "memory");
}

__device__ __forceinline__ void cp_async_16(uint32_t dst, const void *src, uint32_t src_size)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_size) : "memory");
}

// One arrival on the mbarrier once every cp.async this thread issued so far
// has completed (the arrival is counted in the barrier's expected count).
__device__ __forceinline__ void cp_async_mbar_arrive(uint32_t bar)
{
    asm volatile("cp.async.mbarrier.arrive.noinc.shared.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all()
{
    asm volatile("cp.async.wait_all;" ::: "memory");
}

// Tiled 2-D store shared -> global (bulk-group completion).  Elements outside
// the tensor's bounds are not written; coordinates must be non-negative.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, uint32_t src, int x, int y)
{
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(src), "r"(x), "r"(y)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit_group()
{
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Waits until at most N of the bulk groups this thread committed are still
// reading their shared-memory sources (the others' buffers may be overwritten).
template <int N>
__device__ __forceinline__ void bulk_wait_group_read()
{
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Waits until every bulk group this thread committed has completed.
__device__ __forceinline__ void bulk_wait_group0()
{
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Register split between warpgroups: every warp of a warpgroup executes the
// same instruction.  dec returns registers to the CTA's pool; inc waits until
// the pool holds enough (the launch must have provided them).
template <int N>
__device__ __forceinline__ void setmaxnreg_dec()
{
    static_assert(N >= 24 && N <= 256 && N % 8 == 0, "setmaxnreg count");
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

template <int N>
__device__ __forceinline__ void setmaxnreg_inc()
{
    static_assert(N >= 24 && N <= 256 && N % 8 == 0, "setmaxnreg count");
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ------------------------------------------------------------------ tcgen05

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before()
{
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after()
{
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, kind::f8f6f4, one CTA.
__device__ __forceinline__ void mma_f8f6f4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Block-scaled D[tmem] (+)= (A * 2^SFA)[smem] * (B * 2^SFB)[smem]^T, kind::mxf8f6f4,
// one E8M0 scale per row and 32 K-elements, scale factors read from TMEM.
__device__ __forceinline__ void mma_mxf8f6f4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                             uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
            d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

// Copies a 32-row x 16-byte shared-memory matrix into 4 TMEM columns of lanes
// 0-31, replicated into each of the four 32-lane quarters.
__device__ __forceinline__ void tmem_cp_32x128b_warpx4(uint32_t taddr, uint64_t sdesc)
{
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// Descriptor of a K-major shared-memory matrix without swizzle whose rows are
// 16 bytes apart (8-row core matrices 128 bytes apart).
__device__ __forceinline__ uint64_t desc_kmajor_noswizzle_16b(uint32_t saddr)
{
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)(128 >> 4) << 16) | ((uint64_t)(128 >> 4) << 32) |
           ((uint64_t)1 << 46);
}

// Instruction descriptor, kind::mxf8f6f4 block-scaled: E4M3 x E4M3 -> F32,
// UE8M0 scales, both K-major; sf_id selects the byte of each 32-bit scale
// column (the K sub-block of 32 inside a 128-wide K-block).
__host__ __device__ constexpr uint32_t idesc_mx_e4m3(int m, int n, int sf_id)
{
    return ((uint32_t)sf_id << 4)           // B scale-factor id
           | (0u << 7) | (0u << 10)         // A, B format: E4M3
           | ((uint32_t)(n >> 3) << 17)     // N / 8
           | (1u << 23)                     // scale format: UE8M0
           | ((uint32_t)(m >> 4) << 24)     // M / 16
           | ((uint32_t)sf_id << 29);       // A scale-factor id
}

// Arrives once on `bar` when every tcgen05 operation this thread issued so far has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: thread i of the warp gets lane
// (taddr.lane + i), columns taddr.col .. +31.
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
          "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
          "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

// 32 lanes x 16 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait()
{
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// The same wait, tied to the registers of the load it completes: every later
// use of r depends on it, so the compiler cannot read r before the data lands.
__device__ __forceinline__ void tmem_ld_wait_regs(uint32_t (&r)[16])
{
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                   "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                   "+r"(r[15])
                 :
                 : "memory");
}

__device__ __forceinline__ void tmem_ld_wait_regs(uint32_t (&r)[32])
{
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                   "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                   "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                   "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]),
                   "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
                 :
                 : "memory");
}

// Ties 32 registers to the preceding instruction (no code): later uses of r
// cannot move above it.
__device__ __forceinline__ void reg_fence(uint32_t (&r)[32])
{
    asm volatile(""
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                   "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                   "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                   "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]),
                   "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
                 :
                 : "memory");
}

// tcgen05.wait::ld tied to N (a multiple of 32, or 16) loaded registers.
template <int N>
__device__ __forceinline__ void tmem_ld_wait_tie(uint32_t (&r)[N])
{
    if constexpr (N == 16) {
        tmem_ld_wait_regs(r);
    } else {
        static_assert(N % 32 == 0, "tie width");
        tmem_ld_wait_regs(*reinterpret_cast<uint32_t(*)[32]>(&r[0]));
#pragma unroll
        for (int i = 32; i < N; i += 32)
            reg_fence(*reinterpret_cast<uint32_t(*)[32]>(&r[i]));
    }
}

__device__ __forceinline__ void tmem_ld_x(uint32_t taddr, uint32_t (&r)[16]) { tmem_ld_32x32b_x16(taddr, r); }
__device__ __forceinline__ void tmem_ld_x(uint32_t taddr, uint32_t (&r)[32]) { tmem_ld_32x32b_x32(taddr, r); }

// Shared-memory matrix descriptor for a K-major operand tile written by TMA
// with 128-byte swizzle: rows of 128 bytes, 8-row groups 1024 bytes apart,
// tile base 1024-byte aligned.  Fields: start address >> 4 (bits 0-13),
// leading byte offset >> 4 (16-29, unused for this layout), stride byte
// offset >> 4 (32-45), descriptor version 1 (46-47), swizzle mode 2 =
// 128-byte (61-63).
__device__ __forceinline__ uint64_t desc_kmajor_sw128(uint32_t saddr)
{
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor, kind::f8f6f4: E4M3 x E4M3 -> F32, both K-major.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int m, int n)
{
    return (1u << 4)                        // accumulator format: F32
           | (0u << 7) | (0u << 10)         // A, B format: E4M3
           | ((uint32_t)(n >> 3) << 17)     // N / 8
           | ((uint32_t)(m >> 4) << 24);    // M / 16
}

} // namespace ptx
} // namespace jetq
