// Fused FP8 (E4M3) quantizers for sm_103a: one pass over a BF16 tile emits
// the row-wise copy, the transposed column-wise copy and their scales.
//
// Work unit: a 128-row x 128-column BF16 tile (32 KB), 256 threads.  Thread t
// owns rows 8*(t/16) .. +7 and columns 8*(t%16) .. +7 of the tile as an 8x8
// register block, loaded with eight coalesced 16-byte loads (a warp covers two
// full 256-byte row segments per load).  Row maxima are warp shuffles over 16
// lanes; column maxima are a shuffle plus an 8-warp shared-memory reduction.
// The column copy is staged transposed in a swizzled 16 KB shared tile and
// written out as coalesced 16-byte stores, so HBM sees each byte once.
//
// Quotient x / S (FP32-scale recipe).  The exact IEEE quotient fl32(x / S) is
// obtained without a division per element: with r = RN(1/S) (one correctly
// rounded reciprocal per group), q0 = RN(x * r), the FMA residual
// e = x - S * q0 and one correction q1 = RN(q0 + e * r) (Markstein,
// "Computation of elementary functions on the IBM RISC System/6000
// processor", IBM J. R&D 1990) give RN(x / S) for every finite BF16 x with
// |x| <= amax and every S = fl32(amax / 448) >= 2^-96; the sign of a zero
// quotient is restored from x.  This was checked exhaustively over all BF16
// pairs (tests/test_division_domain.py).  Groups with S < 2^-96 use the
// IEEE division itself.
#include <cuda_bf16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "jetq_internal.h"
#include "ptx.cuh"

namespace jetq {

__device__ unsigned g_quant_error;

namespace {

constexpr int kThreads = 256;
constexpr float kE4M3Max = 448.0f;

__device__ __forceinline__ uint4 ldg_stream(const uint16_t *p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void unpack8(const uint4 &u, float (&v)[8])
{
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        v[2 * k] = __uint_as_float(w[k] << 16);
        v[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
    }
}

// the same 8 values negated (sign bit flipped: exact)
__device__ __forceinline__ void unpack8_neg(const uint4 &u, float (&v)[8])
{
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        v[2 * k] = __uint_as_float((w[k] << 16) ^ 0x80000000u);
        v[2 * k + 1] = __uint_as_float((w[k] & 0xFFFF0000u) ^ 0x80000000u);
    }
}

// ------------------------------------------------------------ FP32 recipe

struct Fp32Scale {
    float s;   // the group scale, fl32(amax / 448)
    float r;   // RN(1 / s)
    bool zero; // all-zero group: codes 0x00
    bool slow; // s < 2^-96: use the IEEE division
};

__device__ __forceinline__ Fp32Scale make_scale(float amax)
{
    Fp32Scale sc;
    sc.s = __fdiv_rn(amax, kE4M3Max);
    sc.zero = !(sc.s > 0.0f);
    sc.slow = sc.s < 0x1p-96f;
    sc.r = sc.zero ? 0.0f : __frcp_rn(sc.s);
    return sc;
}

__device__ __forceinline__ uint32_t cvt4(float a, float b, float c, float d)
{
    const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
    const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
    return lo | (hi << 16);
}

__device__ __forceinline__ float with_sign_of(float q, float x)
{
    return __uint_as_float((__float_as_uint(q) & 0x7FFFFFFFu) | (__float_as_uint(x) & 0x80000000u));
}

// 8 values with one scale each (s8[k], r8[k] per value) -> 8 codes, for scales
// >= 2^-96: q0 = x*r, e = x - s*q0 (exact), q1 = q0 + e*r, two values at a time.
__device__ __forceinline__ uint2 quant8_fast(const float (&v)[8], const float (&s8)[8], const float (&r8)[8])
{
    float q[8];
#pragma unroll
    for (int k = 0; k < 8; k += 2) {
        const float2 x2 = make_float2(v[k], v[k + 1]);
        const float2 q0 = __fmul2_rn(x2, make_float2(r8[k], r8[k + 1]));
        const float2 e = __ffma2_rn(q0, make_float2(-s8[k], -s8[k + 1]), x2);
        const float2 q1 = __ffma2_rn(e, make_float2(r8[k], r8[k + 1]), q0);
        q[k] = with_sign_of(q1.x, v[k]);
        q[k + 1] = with_sign_of(q1.y, v[k + 1]);
    }
    return make_uint2(cvt4(q[0], q[1], q[2], q[3]), cvt4(q[4], q[5], q[6], q[7]));
}

// One value, any scale: zero groups give 0x00, tiny scales use the IEEE division.
__device__ __forceinline__ float quotient_general(float x, float s, float r)
{
    if (!(s > 0.0f))
        return 0.0f;
    if (s < 0x1p-96f)
        return __fdiv_rn(x, s);
    const float q0 = __fmul_rn(x, r);
    const float e = __fmaf_rn(-q0, s, x);
    return with_sign_of(__fmaf_rn(e, r, q0), x);
}

// ------------------------------------------------------------ MX recipe

// Smallest e with amax <= 448 * 2^e, clamped to [-127, 127]; 0 for amax == 0.
// 448 = 1.75 * 2^8: for amax = m * 2^E (m in [1, 2)), e = E - 8 + (m > 1.75).
__device__ __forceinline__ int e8m0_exponent(float amax)
{
    uint32_t bits = __float_as_uint(amax);
    if (bits == 0u)
        return 0;
    int E = (int)(bits >> 23) - 127;
    uint32_t mant = bits & 0x7FFFFFu;
    if ((bits >> 23) == 0u) { // subnormal amax = mant * 2^-149: normalise the significand
        const int lz = __clz(mant); // top set bit at 31 - lz
        E = -118 - lz;
        mant = (mant << (lz - 8)) & 0x7FFFFFu;
    }
    int e = E - 8 + (mant > 0x600000u ? 1 : 0);
    return max(-127, min(127, e));
}

__device__ __forceinline__ uint2 quant8_mx(const float (&v)[8], float mult, bool zero)
{
    if (zero)
        return make_uint2(0u, 0u);
    float q[8];
#pragma unroll
    for (int k = 0; k < 8; k += 2) { // exact: a power of two in the normal range
        const float2 p = __fmul2_rn(make_float2(v[k], v[k + 1]), make_float2(mult, mult));
        q[k] = p.x;
        q[k + 1] = p.y;
    }
    return make_uint2(cvt4(q[0], q[1], q[2], q[3]), cvt4(q[4], q[5], q[6], q[7]));
}

// 2^-e as a float, e in [-127, 127] (2^127 .. 2^-127; 2^-127 is subnormal but
// never needed: e <= 120 for finite inputs).
__device__ __forceinline__ float exp2_neg(int e)
{
    const int be = 127 - e;
    return be >= 1 && be <= 254 ? __uint_as_float((uint32_t)be << 23) : __uint_as_float(1u << (22 + be));
}

// byte offset of MX scale (row r, 32-block j) in the 512-byte atom layout; rb = bands
__device__ __forceinline__ int64_t mx_atom_offset(int64_t r, int64_t j, int64_t rb)
{
    return ((j >> 2) * rb + (r >> 7)) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (j & 3);
}

// ------------------------------------------------------------ shared tiles

// Transposed code tile: row = column of the source tile (128 B = 128 source
// rows).  8-byte chunk k of row c is stored at chunk k ^ (c >> 3), which makes
// the per-thread 8-byte stores and the 16-byte read-back conflict-free.
__device__ __forceinline__ void tileT_put(uint8_t *tileT, int col, int chunk, uint2 v)
{
    *reinterpret_cast<uint2 *>(tileT + col * 128 + ((chunk ^ (col >> 3)) & 15) * 8) = v;
}

__device__ __forceinline__ uint4 tileT_get16(const uint8_t *tileT, int col, int u)
{
    const int s = (col >> 3) & 15;
    uint4 v = *reinterpret_cast<const uint4 *>(tileT + col * 128 + (((2 * u) ^ (s & 14)) * 8));
    if (s & 1) {
        uint32_t t0 = v.x, t1 = v.y;
        v.x = v.z;
        v.y = v.w;
        v.z = t0;
        v.w = t1;
    }
    return v;
}

// ------------------------------------------------------------ group mapping

struct Group {
    int64_t t0;  // first source row of the tile
    int cnt;     // valid rows (0 .. 128)
    int64_t p0;  // position of the tile in the column copy
};

// Maps padded group index g to its source rows.  Segment e owns groups
// G_e .. G_{e+1}-1 with G_e = sum_{j<e} ceil(n_j / 128).  Warp 0 computes it
// and publishes through shared memory; cnt = 0 marks a group past the end.
__device__ void map_group(int64_t g, int64_t n, const int64_t *seg, int nseg, Group *out)
{
    const int lane = threadIdx.x & 31;
    if (threadIdx.x >= 32)
        return;
    if (seg == nullptr) {
        if (lane == 0) {
            out->t0 = g * 128;
            const int64_t rem = n - g * 128;
            out->cnt = rem <= 0 ? 0 : (rem >= 128 ? 128 : (int)rem);
            out->p0 = g * 128;
        }
        return;
    }
    const int per = (nseg + 31) / 32;
    const int e0 = min(nseg, lane * per), e1 = min(nseg, e0 + per);
    auto clampo = [&](int64_t v) { return v < 0 ? (int64_t)0 : (v > n ? n : v); };
    int64_t mine = 0;
    for (int e = e0; e < e1; ++e) {
        const int64_t ne = clampo(seg[e + 1]) - clampo(seg[e]);
        if (ne > 0)
            mine += (ne + 127) / 128;
    }
    int64_t incl = mine;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int64_t v = __shfl_up_sync(0xFFFFFFFFu, incl, d);
        if (lane >= d)
            incl += v;
    }
    const int64_t total = __shfl_sync(0xFFFFFFFFu, incl, 31);
    if (lane == 0 && g >= total)
        out->cnt = 0;
    const int64_t excl = incl - mine;
    if (g >= excl && g < incl) {
        int64_t gg = excl;
        for (int e = e0; e < e1; ++e) {
            const int64_t lo = clampo(seg[e]), ne = clampo(seg[e + 1]) - lo;
            if (ne <= 0)
                continue;
            const int64_t ge = (ne + 127) / 128;
            if (g < gg + ge) {
                const int64_t t = g - gg;
                out->t0 = lo + t * 128;
                const int64_t rem = ne - t * 128;
                out->cnt = rem >= 128 ? 128 : (int)rem;
                out->p0 = g * 128;
                break;
            }
            gg += ge;
        }
    }
}

// loads the thread's 8x8 block (rows >= cnt read as +0)
__device__ __forceinline__ void load_block(const uint16_t *x, int64_t ldx, int64_t row0, int64_t col0, int cnt,
                                           int rg, int cc, float (&v)[8][8])
{
    uint4 raw[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int r = rg * 8 + i;
        raw[i] = r < cnt ? ldg_stream(x + (row0 + r) * ldx + col0 + cc * 8) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i)
        unpack8(raw[i], v[i]);
}

// ------------------------------------------------------------ fused producers
//
// The quantized tensor may be produced in the same pass (the activation
// quantizer sits in the kernel that produces the activation): RMSNorm(x) * w
// with a per-row rstd from k_rms_rstd, or the SwiGLU product silu(g) * u.
// Each is the BF16 value the unfused layer would store, computed operation by
// operation in binary32 with explicitly rounded intrinsics, so it is
// reproducible on any IEEE machine.

__device__ __forceinline__ float bf16_round(float f)
{
    return __bfloat162float(__float2bfloat16_rn(f));
}

// exp in binary32: Cody-Waite reduction r = x - n ln2 (ln2 in two parts),
// n = rint(x log2 e), and the degree-7 Taylor polynomial of exp(r) in Horner
// form (Muller, "Elementary Functions", ch. 11); p * 2^n with 2^n built from
// its bits.  Above 88: +inf; below -87: 0.
__device__ __forceinline__ float exp_taylor7(float x)
{
    if (x > 88.0f)
        return __int_as_float(0x7F800000);
    if (x < -87.0f)
        return 0.0f;
    const float n = rintf(__fmul_rn(x, 1.44269502f));
    float r = __fmaf_rn(-n, 0.693145751953125f, x);
    r = __fmaf_rn(-n, 1.42860677e-06f, r);
    float p = 0.000198412701f;
    p = __fmaf_rn(p, r, 0.00138888892f);
    p = __fmaf_rn(p, r, 0.00833333377f);
    p = __fmaf_rn(p, r, 0.0416666679f);
    p = __fmaf_rn(p, r, 0.166666672f);
    p = __fmaf_rn(p, r, 0.5f);
    p = __fmaf_rn(p, r, 1.0f);
    p = __fmaf_rn(p, r, 1.0f);
    return __fmul_rn(p, __int_as_float(((int)n + 127) << 23));
}

// h = BF16(fl32(fl32(g * fl32(1 / fl32(1 + exp(-g)))) * u))
__device__ __forceinline__ float swiglu_bf16(float g, float u)
{
    const float sg = __frcp_rn(__fadd_rn(1.0f, exp_taylor7(-g)));
    return bf16_round(__fmul_rn(__fmul_rn(g, sg), u));
}

// Producer P on one loaded 8-column segment of a row.  With NEG the result is
// negated (the fast tile path works on -y, see quant_tile): the negation is
// folded into the unpacking of x, of the RMSNorm weights or of the SwiGLU up
// values, so it costs nothing.  aux holds the 8 up values (SwiGLU), rs the
// row's rstd and w8 the 8 weights, already carrying the NEG sign (RMSNorm).
template <int P, bool NEG>
__device__ __forceinline__ void produce8(const uint4 &raw, const uint4 &aux, float rs, const float (&w8)[8],
                                         float (&v)[8])
{
    if (P == kProducePlain) {
        if (NEG)
            unpack8_neg(raw, v);
        else
            unpack8(raw, v);
    } else if (P == kProduceRms) {
        float x[8];
        unpack8(raw, x);
#pragma unroll
        for (int k = 0; k < 8; ++k)
            v[k] = bf16_round(__fmul_rn(__fmul_rn(x[k], rs), w8[k]));
    } else {
        float gt[8], u[8];
        unpack8(raw, gt);
        if (NEG)
            unpack8_neg(aux, u);
        else
            unpack8(aux, u);
#pragma unroll
        for (int k = 0; k < 8; ++k)
            v[k] = swiglu_bf16(gt[k], u[k]);
    }
}

// the 8 RMSNorm weights of columns col .. col+7, negated with NEG (zeros for other producers)
template <int P, bool NEG>
__device__ __forceinline__ void load_weights8(const ActQuantArgs &a, int64_t col, float (&w8)[8])
{
    if (P == kProduceRms) {
        const uint4 raw = __ldg(reinterpret_cast<const uint4 *>(a.w + col));
        if (NEG)
            unpack8_neg(raw, w8);
        else
            unpack8(raw, w8);
    } else {
#pragma unroll
        for (int k = 0; k < 8; ++k)
            w8[k] = 0.0f;
    }
}

// one produced 8-column segment of row `row`, sign as is (zeros when !in)
template <int P>
__device__ __forceinline__ void load_row8_produced(const ActQuantArgs &a, int64_t row, int64_t col, bool in,
                                                   float (&v)[8])
{
    float w8[8];
    load_weights8<P, false>(a, col, w8);
    const uint4 raw = in ? ldg_stream(a.x + row * a.ldx + col) : make_uint4(0, 0, 0, 0);
    const uint4 aux = (P == kProduceSwiglu && in) ? ldg_stream(a.up + row * a.ldup + col) : make_uint4(0, 0, 0, 0);
    const float rs = (P == kProduceRms && in) ? __ldg(a.rstd + row) : 0.0f;
    produce8<P, false>(raw, aux, rs, w8, v);
}

__device__ __forceinline__ float absmax8(const float (&v)[8])
{
    float m = fabsf(v[0]);
#pragma unroll
    for (int k = 1; k < 8; ++k)
        m = fmaxf(m, fabsf(v[k]));
    return m;
}

// writes the transposed tile (128 columns x 128 rows of codes) to qc
__device__ __forceinline__ void store_tileT(const uint8_t *tileT, uint8_t *qc, int64_t ldq, int64_t ch0, int64_t pos0)
{
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int L = threadIdx.x + kThreads * k;
        const int ch = L >> 3, u = L & 7;
        *reinterpret_cast<uint4 *>(qc + (ch0 + ch) * ldq + pos0 + u * 16) = tileT_get16(tileT, ch, u);
    }
}

// ============================================================ kernels

// The act tile again, element by element, for any scale (zero groups, scales
// below 2^-96).  Reloads its inputs; scales come from shared memory.
template <int P>
__device__ __noinline__ void quant_act_tile_general(const ActQuantArgs &a, int64_t t0, int cnt, int64_t p0,
                                                    int64_t c0, bool row, bool col, const float *scS,
                                                    const float *scR, uint8_t *tileT)
{
    const int t = threadIdx.x, rg = t >> 4, cc = t & 15;
    for (int i = 0; i < 8; ++i) {
        const int r = rg * 8 + i;
        float v[8];
        load_row8_produced<P>(a, t0 + r, c0 + cc * 8, r < cnt, v);
        if (row && r < cnt) {
            float q[8];
#pragma unroll
            for (int k = 0; k < 8; ++k)
                q[k] = quotient_general(v[k], scS[r], scR[r]);
            *reinterpret_cast<uint2 *>(a.q_row + (t0 + r) * a.c + c0 + cc * 8) =
                make_uint2(cvt4(q[0], q[1], q[2], q[3]), cvt4(q[4], q[5], q[6], q[7]));
        }
        if (col) {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int c = cc * 8 + k;
                const float qv = quotient_general(v[k], scS[128 + c], scR[128 + c]);
                const uint32_t code = __nv_cvt_float2_to_fp8x2(make_float2(qv, 0.0f), __NV_SATFINITE, __NV_E4M3) & 0xFFu;
                tileT[c * 128 + ((rg ^ (c >> 3)) & 15) * 8 + i] = (uint8_t)code;
            }
        }
    }
    if (col) {
        __syncthreads();
        store_tileT(tileT, a.q_col, a.ldq_col, c0, p0);
    }
}

// Shared working set of one 128 x 128 activation tile.
struct TileSmem {
    uint8_t tileT[128 * 128]; // transposed column codes (swizzled)
    float redR[16][132];      // row partial maxima [column chunk][row]
    float redC[8][128];       // column partial maxima [warp][column]
    float4 rowSc[128];        // per row: (S, S, -1/S, -1/S), packed operand pairs
    float colS[128];          // per column: S
    float colNR[128];         // per column: -1/S
    float scS[2][128];        // S and 1/S for the general path: [0] rows, [1] columns
    float scR[2][128];
};

// Both quotients of a pair, from the negated values nx = -x:
// q0 = RN(x * r), e' = S*q0 - x (exact by FMA), q1 = RN(q0 - e' * r), which is
// the residual-corrected quotient of the file header with e' = -e.  Working on
// -x also gives zero quotients the sign of x: x = -0 yields -0 + -0 = -0.
__device__ __forceinline__ float2 quotient2_neg(float2 nx, float2 S, float2 NR)
{
    const float2 q0 = __fmul2_rn(nx, NR);
    const float2 e = __ffma2_rn(S, q0, nx);
    return __ffma2_rn(e, NR, q0);
}

// The tile computation both activation-quantizer kernels share, from the
// thread's 8x8 block of negated values (rows >= cnt zero).  Each of the 256
// scales of the tile is computed once, by one thread, and published through
// shared memory.  after_sync() runs once every thread holds its block in
// registers (its input buffer may then be refilled).
template <bool ROW, bool COL, int P, typename AfterSync>
__device__ __forceinline__ void quant_tile(const ActQuantArgs &a, TileSmem &ts, float (&nv)[8][8], int64_t t0,
                                           int cnt, int64_t p0, int64_t c0, AfterSync after_sync)
{
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int rg = t >> 4, cc = t & 15;

    // ---- partial maxima
    if (ROW) {
        float rm[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            rm[i] = absmax8(nv[i]);
        *reinterpret_cast<float4 *>(&ts.redR[cc][rg * 8]) = make_float4(rm[0], rm[1], rm[2], rm[3]);
        *reinterpret_cast<float4 *>(&ts.redR[cc][rg * 8 + 4]) = make_float4(rm[4], rm[5], rm[6], rm[7]);
    }
    if (COL) {
        float cm[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            float m = fabsf(nv[0][j]);
#pragma unroll
            for (int i = 1; i < 8; ++i)
                m = fmaxf(m, fabsf(nv[i][j]));
            cm[j] = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 16));
        }
        if (lane < 16) {
            *reinterpret_cast<float4 *>(&ts.redC[warp][cc * 8]) = make_float4(cm[0], cm[1], cm[2], cm[3]);
            *reinterpret_cast<float4 *>(&ts.redC[warp][cc * 8 + 4]) = make_float4(cm[4], cm[5], cm[6], cm[7]);
        }
    }
    __syncthreads();
    after_sync();

    // ---- one scale per thread: threads 0..127 rows, 128..255 columns
    int special = 0;
    {
        const bool is_row = t < 128;
        const int k = t & 127;
        if (is_row ? ROW : COL) {
            float m = 0.0f;
            if (is_row) {
#pragma unroll
                for (int w = 0; w < 16; ++w)
                    m = fmaxf(m, ts.redR[w][k]);
            } else {
#pragma unroll
                for (int w = 0; w < 8; ++w)
                    m = fmaxf(m, ts.redC[w][k]);
            }
            const Fp32Scale sc = make_scale(m);
            ts.scS[is_row ? 0 : 1][k] = sc.s;
            ts.scR[is_row ? 0 : 1][k] = sc.r;
            special = (sc.zero || sc.slow) && (!is_row || k < cnt); // rows past cnt are never stored
            if (is_row) {
                ts.rowSc[k] = make_float4(sc.s, sc.s, -sc.r, -sc.r);
                if (k < cnt)
                    a.s_row[(c0 >> 7) * a.n + t0 + k] = sc.s;
            } else {
                ts.colS[k] = sc.s;
                ts.colNR[k] = -sc.r;
                a.s_col[(p0 >> 7) * a.c + c0 + k] = sc.s;
            }
        }
    }
    if (__syncthreads_or(special)) { // a zero or tiny scale somewhere in the tile (rare): slow, general path
        quant_act_tile_general<P>(a, t0, cnt, p0, c0, ROW, COL, &ts.scS[0][0], &ts.scR[0][0], ts.tileT);
        return;
    }

    // ---- row codes straight to global (16 lanes write one 128-byte row); the
    // column quotients replace the block in place, row by row
    float cs[8], cnr[8];
    if (COL) {
        *reinterpret_cast<float4 *>(cs) = *reinterpret_cast<const float4 *>(&ts.colS[cc * 8]);
        *reinterpret_cast<float4 *>(cs + 4) = *reinterpret_cast<const float4 *>(&ts.colS[cc * 8 + 4]);
        *reinterpret_cast<float4 *>(cnr) = *reinterpret_cast<const float4 *>(&ts.colNR[cc * 8]);
        *reinterpret_cast<float4 *>(cnr + 4) = *reinterpret_cast<const float4 *>(&ts.colNR[cc * 8 + 4]);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int r = rg * 8 + i;
        if (ROW) {
            const float4 rs4 = ts.rowSc[r];
            const float2 S2 = make_float2(rs4.x, rs4.y), NR2 = make_float2(rs4.z, rs4.w);
            float q[8];
#pragma unroll
            for (int k = 0; k < 8; k += 2) {
                const float2 q2 = quotient2_neg(make_float2(nv[i][k], nv[i][k + 1]), S2, NR2);
                q[k] = q2.x;
                q[k + 1] = q2.y;
            }
            if (r < cnt)
                *reinterpret_cast<uint2 *>(a.q_row + (t0 + r) * a.c + c0 + cc * 8) =
                    make_uint2(cvt4(q[0], q[1], q[2], q[3]), cvt4(q[4], q[5], q[6], q[7]));
        }
        if (COL) {
#pragma unroll
            for (int k = 0; k < 8; k += 2) {
                const float2 q2 = quotient2_neg(make_float2(nv[i][k], nv[i][k + 1]), make_float2(cs[k], cs[k + 1]),
                                                make_float2(cnr[k], cnr[k + 1]));
                nv[i][k] = q2.x;
                nv[i][k + 1] = q2.y;
            }
        }
    }

    // ---- column codes transposed through shared memory
    if (COL) {
#pragma unroll
        for (int j = 0; j < 8; ++j)
            tileT_put(ts.tileT, cc * 8 + j, rg,
                      make_uint2(cvt4(nv[0][j], nv[1][j], nv[2][j], nv[3][j]),
                                 cvt4(nv[4][j], nv[5][j], nv[6][j], nv[7][j])));
        __syncthreads();
        store_tileT(ts.tileT, a.q_col, a.ldq_col, c0, p0);
    }
}

// ------------------------------------------------------------ SwiGLU-fused quantizer
//
// The sigmoid factor fl32(1 / fl32(1 + exp(-g))) depends on the BF16 gate g
// alone, so each CTA tabulates it once, with the same device function, for the
// 8192 gates of magnitude 2^-25 .. 2^7 (32 binades, both signs; 32 KB of shared
// memory), and looks it up per element; other gates (zeros, tiny or large
// magnitudes) take the direct computation.  The table entries are that
// computation's results, so the product is unchanged bit for bit.  The kernel
// is persistent (two CTAs per SM walk the tiles) so the table is built once
// per CTA.

constexpr int kSigTable = 8192;
constexpr uint32_t kSigE8Lo = 102; // 2^-25

__device__ __forceinline__ float sigmoid_factor(float g)
{
    return __frcp_rn(__fadd_rn(1.0f, exp_taylor7(-g)));
}

// table slot of the BF16 gate with bits b, or -1 outside the tabulated binades:
// |b| - (102 << 7) is (binade - 102) << 7 | mantissa inside them
__device__ __forceinline__ int sigmoid_slot(uint32_t b)
{
    const uint32_t d = (b & 0x7FFFu) - (kSigE8Lo << 7);
    return d < 4096u ? (int)(((b >> 3) & 0x1000u) | d) : -1;
}

// the direct computation, out of line: every element has a call site and
// almost none take it, so inlining would only crowd the instruction cache
__device__ __noinline__ float sigmoid_factor_slow(float g)
{
    return sigmoid_factor(g);
}

// -h for 8 columns of one row: gate bits in graw, up values in uraw
__device__ __forceinline__ void swiglu8_neg(const uint4 &graw, const uint4 &uraw, const float *tab, float (&nv)[8])
{
    const uint32_t gw[4] = {graw.x, graw.y, graw.z, graw.w};
    float gv[8], nu[8], sg[8];
    unpack8(graw, gv);
    unpack8_neg(uraw, nu);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const int slot = sigmoid_slot((k & 1) ? (gw[k >> 1] >> 16) : (gw[k >> 1] & 0xFFFFu));
        sg[k] = slot >= 0 ? tab[slot] : sigmoid_factor_slow(gv[k]);
    }
#pragma unroll
    for (int k = 0; k < 8; k += 2) {
        const float2 sl = __fmul2_rn(make_float2(gv[k], gv[k + 1]), make_float2(sg[k], sg[k + 1]));
        const float2 h = __fmul2_rn(sl, make_float2(nu[k], nu[k + 1]));
        const __nv_bfloat162 hb = __float22bfloat162_rn(h);
        nv[k] = __low2float(hb);
        nv[k + 1] = __high2float(hb);
    }
}

struct SwiSmem {
    TileSmem ts;
    float tab[kSigTable];
    Group grp[2];
};

template <bool ROW, bool COL>
__global__ void __launch_bounds__(kThreads, 2)
    k_quant_act_swiglu(const __grid_constant__ ActQuantArgs a, int64_t ngroups, int ncb)
{
    extern __shared__ uint8_t smem_raw[];
    SwiSmem &sm = *reinterpret_cast<SwiSmem *>(ptx::align_smem<16>(smem_raw));
    const int t = threadIdx.x, warp = t >> 5;
    const int rg = t >> 4, cc = t & 15;
    const int64_t total = ngroups * ncb;

    for (int i = t; i < kSigTable; i += kThreads) {
        const uint32_t b = ((uint32_t)(i >> 12) << 15) | ((kSigE8Lo + (uint32_t)((i >> 7) & 31)) << 7) | (uint32_t)(i & 127);
        sm.tab[i] = sigmoid_factor(__uint_as_float(b << 16));
    }

    for (int64_t k = 0;; ++k) {
        const int64_t T = blockIdx.x + k * (int64_t)gridDim.x;
        if (T >= total)
            break;
        if (warp == 0)
            map_group(T / ncb, a.n, a.seg, a.nseg, &sm.grp[k & 1]);
        __syncthreads(); // the group (and, the first time, the table) visible to all
        const int cnt = sm.grp[k & 1].cnt;
        if (cnt == 0)
            continue;
        const int64_t t0 = sm.grp[k & 1].t0, p0 = sm.grp[k & 1].p0;
        const int64_t c0 = (T % ncb) * 128;
        uint4 graw[8], uraw[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int r = rg * 8 + i;
            const bool in = r < cnt;
            graw[i] = in ? ldg_stream(a.x + (t0 + r) * a.ldx + c0 + cc * 8) : make_uint4(0, 0, 0, 0);
            uraw[i] = in ? ldg_stream(a.up + (t0 + r) * a.ldup + c0 + cc * 8) : make_uint4(0, 0, 0, 0);
        }
        float nv[8][8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            swiglu8_neg(graw[i], uraw[i], sm.tab, nv[i]);
        quant_tile<ROW, COL, kProduceSwiglu>(a, sm.ts, nv, t0, cnt, p0, c0, [] {});
    }
}

// ------------------------------------------------------------ TMA-fed activation quantizer
//
// The same tile computation in a persistent loop: each CTA walks tiles
// blockIdx.x, blockIdx.x + gridDim.x, ...; warp 0 keeps the next tiles' BF16
// input in flight with TMA (one 32 KB box per tile, a two-stage ring per CTA,
// two CTAs per SM), so HBM sees requests while the previous tile is reduced,
// quantized and stored.  A stage is refilled once every thread has moved its
// 8x8 block into registers (the first barrier of the tile).

constexpr int kPipeStages = 2;
constexpr uint32_t kPipeTileBytes = 128 * 128 * 2;
constexpr unsigned long long kQuantWaitLimitNs = 2000000000ull; // 2 s per wait
constexpr unsigned kQuantErrTimeout = 1u;

struct PipeSmem {
    uint16_t stage[kPipeStages][128 * 128]; // BF16 input tiles, rows of 256 bytes
    TileSmem ts;
    Group grp[kPipeStages]; // the tile each stage holds
    unsigned long long full[kPipeStages];
    int issued[kPipeStages];
    int abort;
};
constexpr size_t kPipeSmemBytes = sizeof(PipeSmem) + 1024;

template <bool ROW, bool COL, int P>
__global__ void __launch_bounds__(kThreads, 2)
    k_quant_act_tma(const __grid_constant__ ActQuantArgs a, const __grid_constant__ CUtensorMap tmx,
                    int64_t ngroups, int ncb)
{
    static_assert(P != kProduceSwiglu, "the TMA path stages one input tensor");
    extern __shared__ uint8_t smem_raw[];
    PipeSmem &sm = *reinterpret_cast<PipeSmem *>(ptx::align_smem<1024>(smem_raw));
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int rg = t >> 4, cc = t & 15;
    const int64_t total = ngroups * ncb;
    unsigned *err = &g_quant_error;

    // warp 0: map the CTA's k-th tile to its rows and start its load into stage k % kPipeStages
    auto issue = [&](int64_t k) {
        const int64_t T = blockIdx.x + k * (int64_t)gridDim.x;
        if (T >= total || sm.abort)
            return;
        const int s = (int)(k % kPipeStages);
        map_group(T / ncb, a.n, a.seg, a.nseg, &sm.grp[s]);
        __syncwarp();
        if (lane == 0) {
            const uint32_t bar = ptx::smem_addr(&sm.full[s]);
            sm.issued[s] += 1;
            if (sm.grp[s].cnt > 0) {
                ptx::mbar_arrive_expect_tx(bar, kPipeTileBytes);
                ptx::tma_load_2d(ptx::smem_addr(sm.stage[s]), &tmx, bar, (int)((T % ncb) * 128), (int)sm.grp[s].t0);
            } else {
                ptx::mbar_arrive(bar);
            }
        }
        __syncwarp();
    };

    if (t == 0) {
        for (int s = 0; s < kPipeStages; ++s) {
            ptx::mbar_init(ptx::smem_addr(&sm.full[s]), 1);
            sm.issued[s] = 0;
        }
        sm.abort = 0;
        ptx::fence_barrier_init();
    }
    __syncthreads();
    // global memory only after the stream's previous kernel has completed (no
    // early launch_dependents: the next kernel starts as these CTAs exit, which
    // measured faster in a decode step than letting it in at once)
    ptx::grid_dep_wait();
    if (warp == 0) {
        if (lane == 0)
            ptx::prefetch_tensormap(&tmx);
        for (int s = 0; s < kPipeStages; ++s)
            issue(s);
    }

    for (int64_t k = 0;; ++k) {
        const int64_t T = blockIdx.x + k * (int64_t)gridDim.x;
        if (T >= total)
            break;
        const int s = (int)(k % kPipeStages);
        ptx::mbar_wait(ptx::smem_addr(&sm.full[s]), (uint32_t)((k / kPipeStages) & 1), &sm.abort, err,
                       kQuantErrTimeout, kQuantWaitLimitNs);
        const int cnt = sm.grp[s].cnt;
        const int64_t t0 = sm.grp[s].t0, p0 = sm.grp[s].p0;
        const int64_t c0 = (T % ncb) * 128;
        if (cnt == 0) { // a padded group past the last segment
            __syncthreads();
            if (warp == 0)
                issue(k + kPipeStages);
            continue;
        }

        float nv[8][8];
        {
            float w8[8];
            load_weights8<P, true>(a, c0 + cc * 8, w8);
            const uint16_t *st = sm.stage[s];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int r = rg * 8 + i;
                const bool in = r < cnt;
                const uint4 raw = in ? *reinterpret_cast<const uint4 *>(st + r * 128 + cc * 8) : make_uint4(0, 0, 0, 0);
                const float rs = (P == kProduceRms && in) ? __ldg(a.rstd + t0 + r) : 0.0f;
                produce8<P, true>(raw, make_uint4(0, 0, 0, 0), rs, w8, nv[i]);
            }
        }
        ptx::fence_proxy_async_smem(); // the stage's generic reads before the next TMA write into it
        quant_tile<ROW, COL, P>(a, sm.ts, nv, t0, cnt, p0, c0, [&] {
            if (warp == 0)
                issue(k + kPipeStages);
        });
    }

    // after a timed-out wait no new loads were started; wait (bounded) for the
    // ones still in flight before the CTA's shared memory is released
    if (t == 0 && sm.abort) {
        for (int s = 0; s < kPipeStages; ++s)
            if (sm.issued[s] > 0)
                ptx::mbar_wait(ptx::smem_addr(&sm.full[s]), (uint32_t)((sm.issued[s] - 1) & 1), &sm.abort, err,
                               kQuantErrTimeout, kQuantWaitLimitNs, false);
    }
}


// RMSNorm statistics, one warp per row.  Lane l sums the 128-column groups
// l, l + 32, ... (each left to right by fma); the group sums are then added
// left to right by every lane through shuffles, so the binary32 result
// follows one fixed order: rstd = 1 / sqrt(total / c + eps).  A batch of 32
// groups (8 KB) is loaded coalesced (one warp load = 512 contiguous bytes)
// and regrouped through shared memory, each group padded to 272 bytes so that
// both the regrouping stores and the per-lane group reads are conflict-free.
// Warps walk rows grid-stride; the next batch's loads are in flight while the
// current batch is summed.
constexpr int kRmsWarps = 4;
constexpr int kRmsPitch = 272;

__global__ void __launch_bounds__(kRmsWarps * 32) k_rms_rstd(const uint16_t *__restrict__ x, int64_t n, int64_t c,
                                                             int64_t ldx, float eps, float *__restrict__ rstd)
{
    __shared__ __align__(16) uint8_t stage[kRmsWarps][32 * kRmsPitch];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t stride = (int64_t)gridDim.x * kRmsWarps;
    int64_t row = (int64_t)blockIdx.x * kRmsWarps + warp;
    if (row >= n)
        return;
    uint8_t *sw = stage[warp];
    const int groups = (int)(c >> 7);
    // batch (row, g0): its live * 16 chunks of 16 bytes; chunk q is slot q % 16 of group q / 16
    uint4 raw[16];
    auto load = [&](int64_t r, int g0) {
        const uint4 *xr = reinterpret_cast<const uint4 *>(x + r * ldx) + (int64_t)g0 * 16;
        const int chunks = min(32, groups - g0) * 16;
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            const int q = k * 32 + lane;
            raw[k] = q < chunks ? __ldg(xr + q) : make_uint4(0, 0, 0, 0);
        }
    };
    int g0 = 0;
    float total = 0.0f;
    load(row, 0);
    while (row < n) {
        const int live = min(32, groups - g0);
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            const int q = k * 32 + lane;
            if (q < live * 16)
                *reinterpret_cast<uint4 *>(sw + (q >> 4) * kRmsPitch + (q & 15) * 16) = raw[k];
        }
        __syncwarp();
        int64_t nrow = row;
        int ng0 = g0 + 32;
        if (ng0 >= groups) {
            nrow = row + stride;
            ng0 = 0;
        }
        if (nrow < n)
            load(nrow, ng0);
        float part = 0.0f;
        if (lane < live) {
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                float v[8];
                unpack8(*reinterpret_cast<const uint4 *>(sw + lane * kRmsPitch + k * 16), v);
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    part = __fmaf_rn(v[j], v[j], part);
            }
        }
        __syncwarp(); // every lane has read its group before the next batch is staged
        for (int j = 0; j < live; ++j)
            total = __fadd_rn(total, __shfl_sync(0xFFFFFFFFu, part, j));
        if (ng0 == 0) {
            if (lane == 0)
                rstd[row] = __frcp_rn(__fsqrt_rn(__fadd_rn(__fdiv_rn(total, (float)c), eps)));
            total = 0.0f;
        }
        row = nrow;
        g0 = ng0;
    }
}

// 8x8 byte transpose: in[i] holds bytes (row i, cols 0..7); out[j] holds
// bytes (rows 0..7, col j).
__device__ __forceinline__ void transpose8x8(const uint2 (&in)[8], uint2 (&out)[8])
{
    // interleave row pairs: p[k] = rows (2k, 2k+1)
    uint32_t lo0[4], lo1[4], hi0[4], hi1[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        lo0[k] = __byte_perm(in[2 * k].x, in[2 * k + 1].x, 0x5140); // c0: r0 r1, c1: r0 r1
        lo1[k] = __byte_perm(in[2 * k].x, in[2 * k + 1].x, 0x7362); // c2, c3
        hi0[k] = __byte_perm(in[2 * k].y, in[2 * k + 1].y, 0x5140); // c4, c5
        hi1[k] = __byte_perm(in[2 * k].y, in[2 * k + 1].y, 0x7362); // c6, c7
    }
    const uint32_t *src[4] = {lo0, lo1, hi0, hi1};
#pragma unroll
    for (int h = 0; h < 4; ++h) {
        const uint32_t *p = src[h];
        // column 2h: bytes 0,1 of each pair word; column 2h+1: bytes 2,3
        out[2 * h].x = __byte_perm(p[0], p[1], 0x5410);
        out[2 * h].y = __byte_perm(p[2], p[3], 0x5410);
        out[2 * h + 1].x = __byte_perm(p[0], p[1], 0x7632);
        out[2 * h + 1].y = __byte_perm(p[2], p[3], 0x7632);
    }
}

// Weight quantizer: one scale per 128x128 block, codes + transposed codes.
// One 128 x 128 weight block (rows d0.., columns c0..), the thread's 8 x 8
// block in v; red (8 floats) and tileT (16 KB) are the CTA's shared scratch.
// Leaves with every thread past the block's last shared-memory access.
__device__ __forceinline__ void quant_weight_tile(const WeightQuantArgs &a, float *red, uint8_t *tileT,
                                                  const float (&v)[8][8], int64_t d0, int64_t c0)
{
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int rg = t >> 4, cc = t & 15;

    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i)
        m = fmaxf(m, absmax8(v[i]));
#pragma unroll
    for (int d = 1; d < 32; d <<= 1)
        m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, d));
    if (lane == 0)
        red[warp] = m;
    __syncthreads();
    m = red[0];
#pragma unroll
    for (int w = 1; w < 8; ++w)
        m = fmaxf(m, red[w]);
    const Fp32Scale sc = make_scale(m);
    if (t == 0) {
        a.s[(d0 >> 7) * (a.c >> 7) + (c0 >> 7)] = sc.s;
        if (a.sT)
            a.sT[(c0 >> 7) * (a.d >> 7) + (d0 >> 7)] = sc.s;
    }

    uint2 rows[8];
    if (sc.zero || sc.slow) { // rare: all-zero block or a scale below 2^-96
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            float q[8];
#pragma unroll
            for (int k = 0; k < 8; ++k)
                q[k] = quotient_general(v[i][k], sc.s, sc.r);
            rows[i] = make_uint2(cvt4(q[0], q[1], q[2], q[3]), cvt4(q[4], q[5], q[6], q[7]));
        }
    } else {
        float s8[8], r8[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            s8[k] = sc.s;
            r8[k] = sc.r;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i)
            rows[i] = quant8_fast(v[i], s8, r8);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i)
        *reinterpret_cast<uint2 *>(a.q + (d0 + rg * 8 + i) * a.c + c0 + cc * 8) = rows[i];
    if (a.qT) {
        uint2 cols[8];
        transpose8x8(rows, cols);
#pragma unroll
        for (int j = 0; j < 8; ++j)
            tileT_put(tileT, cc * 8 + j, rg, cols[j]);
        __syncthreads();
        store_tileT(tileT, a.qT, a.d, c0, d0);
    }
}

// Weight quantizer, persistent: two CTAs of 256 threads per SM walk the
// 128 x 128 blocks, warp 0 keeping the next block's BF16 input in flight by
// TMA (a two-stage ring).
struct WPipeSmem {
    uint16_t stage[2][128 * 128];
    uint8_t tileT[128 * 128];
    float red[8];
    unsigned long long full[2];
    int issued[2];
    int abort;
};
constexpr size_t kWPipeSmemBytes = sizeof(WPipeSmem) + 1024;

__global__ void __launch_bounds__(kThreads, 2)
    k_quant_weight_tma(const __grid_constant__ WeightQuantArgs a, const __grid_constant__ CUtensorMap tmw)
{
    extern __shared__ uint8_t smem_raw[];
    WPipeSmem &sm = *reinterpret_cast<WPipeSmem *>(ptx::align_smem<1024>(smem_raw));
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int rg = t >> 4, cc = t & 15;
    const int ncb = (int)(a.c / 128);
    const int64_t total = (a.d / 128) * ncb;
    unsigned *err = &g_quant_error;

    auto issue = [&](int64_t k) { // warp 0, lane 0
        const int64_t T = blockIdx.x + k * (int64_t)gridDim.x;
        if (T >= total || sm.abort)
            return;
        const int s = (int)(k & 1);
        const uint32_t bar = ptx::smem_addr(&sm.full[s]);
        sm.issued[s] += 1;
        ptx::mbar_arrive_expect_tx(bar, kPipeTileBytes);
        ptx::tma_load_2d(ptx::smem_addr(sm.stage[s]), &tmw, bar, (int)((T % ncb) * 128), (int)((T / ncb) * 128));
    };

    if (t == 0) {
        for (int s = 0; s < 2; ++s) {
            ptx::mbar_init(ptx::smem_addr(&sm.full[s]), 1);
            sm.issued[s] = 0;
        }
        sm.abort = 0;
        ptx::fence_barrier_init();
    }
    __syncthreads();
    // global memory only after the stream's previous kernel has completed (no
    // early launch_dependents: the next kernel starts as these CTAs exit, which
    // measured faster in a decode step than letting it in at once)
    ptx::grid_dep_wait();
    if (t == 0) {
        ptx::prefetch_tensormap(&tmw);
        issue(0);
        issue(1);
    }
    for (int64_t k = 0;; ++k) {
        const int64_t T = blockIdx.x + k * (int64_t)gridDim.x;
        if (T >= total)
            break;
        const int s = (int)(k & 1);
        ptx::mbar_wait(ptx::smem_addr(&sm.full[s]), (uint32_t)((k >> 1) & 1), &sm.abort, err, kQuantErrTimeout,
                       kQuantWaitLimitNs);
        float v[8][8];
        const uint16_t *st = sm.stage[s];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            unpack8(*reinterpret_cast<const uint4 *>(st + (rg * 8 + i) * 128 + cc * 8), v[i]);
        // every thread has its block (and finished the previous block's shared-memory work)
        ptx::fence_proxy_async_smem();
        __syncthreads();
        if (t == 0)
            issue(k + 2);
        quant_weight_tile(a, sm.red, sm.tileT, v, (T / ncb) * 128, (T % ncb) * 128);
    }
    if (t == 0 && sm.abort) {
        for (int s = 0; s < 2; ++s)
            if (sm.issued[s] > 0)
                ptx::mbar_wait(ptx::smem_addr(&sm.full[s]), (uint32_t)((sm.issued[s] - 1) & 1), &sm.abort, err,
                               kQuantErrTimeout, kQuantWaitLimitNs, false);
    }
}

// Power-of-two 128x128 weight blocks: one E8M0 exponent per block, written
// into the MX scale atoms of W (rows D, K = C) and of W^T (rows C, K = D),
// each 32-element sub-block byte carrying its block's exponent.
__global__ void __launch_bounds__(kThreads, 2) k_quant_weight_pow2(WeightPow2Args a)
{
    __shared__ float red[8];
    __shared__ __align__(16) uint8_t tileT[128 * 128];

    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int rg = t >> 4, cc = t & 15;
    const int64_t d0 = (int64_t)blockIdx.x * 128, c0 = (int64_t)blockIdx.y * 128;

    float v[8][8];
    load_block(a.w, a.ldw, d0, c0, 128, rg, cc, v);

    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i)
        m = fmaxf(m, absmax8(v[i]));
#pragma unroll
    for (int d = 1; d < 32; d <<= 1)
        m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, d));
    if (lane == 0)
        red[warp] = m;
    __syncthreads();
    m = red[0];
#pragma unroll
    for (int w = 1; w < 8; ++w)
        m = fmaxf(m, red[w]);
    const int e = e8m0_exponent(m);
    const float f = exp2_neg(e);
    const uint32_t word = (uint32_t)(e + 127) * 0x01010101u;
    if (t < 128)
        *reinterpret_cast<uint32_t *>(a.e8 + mx_atom_offset(d0 + t, c0 >> 5, (a.d + 127) / 128)) = word;
    else if (a.e8T)
        *reinterpret_cast<uint32_t *>(a.e8T + mx_atom_offset(c0 + (t - 128), d0 >> 5, (a.c + 127) / 128)) = word;

    uint2 rows[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
        rows[i] = quant8_mx(v[i], f, m == 0.0f);
#pragma unroll
    for (int i = 0; i < 8; ++i)
        *reinterpret_cast<uint2 *>(a.q + (d0 + rg * 8 + i) * a.c + c0 + cc * 8) = rows[i];
    if (a.qT) {
        uint2 cols[8];
        transpose8x8(rows, cols);
#pragma unroll
        for (int j = 0; j < 8; ++j)
            tileT_put(tileT, cc * 8 + j, rg, cols[j]);
        __syncthreads();
        store_tileT(tileT, a.qT, a.d, c0, d0);
    }
}

// MX-style quantizer with E8M0 scales: 1xG row blocks and Gx1 column blocks,
// G = 32 (MXFP8) or 128 (the 128-block recipe with power-of-two scales; each
// 32-element sub-block byte of the scale atoms then carries its group's exponent).
// Shared memory of one MX tile: column partial maxima, the transposed column
// codes and the column scale bytes.
struct MxTileSmem {
    float red[8][128];
    uint8_t tileT[128 * 128];
    uint32_t e8T[128];
};

// One 128 x 128 tile (rows t0 .. t0 + cnt of a segment, columns c0 .. c0 + 127):
// the thread holds its 8 x 8 block v (rows rg * 8 + i, columns cc * 8 + j).
// Leaves with every thread past the tile's last shared-memory access.
template <bool ROW, bool COL, int G>
__device__ __forceinline__ void quant_mx_tile(const MxQuantArgs &a, MxTileSmem &ts, const float (&v)[8][8],
                                              int64_t t0, int cnt, int64_t p0, int64_t c0)
{
    float (&red)[8][128] = ts.red;
    uint8_t *tileT = ts.tileT;
    uint32_t *e8T = ts.e8T;
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int rg = t >> 4, cc = t & 15;

    if (ROW) {
        const int64_t ka = (a.rows + 127) / 128; // row bands of the row copy
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            float m = absmax8(v[i]);
            m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
            m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
            if (G == 128) { // the 16 lanes of a half-warp span the tile's 128 columns
                m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 4));
                m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 8));
            }
            const int e = e8m0_exponent(m);
            const uint2 codes = quant8_mx(v[i], exp2_neg(e), m == 0.0f);
            // the four 32-blocks of this row sit in lanes with cc = 0, 4, 8, 12 of the half-warp
            const uint32_t byte = (uint32_t)(e + 127);
            const int base = lane & 16;
            const uint32_t b0 = __shfl_sync(0xFFFFFFFFu, byte, base + 0);
            const uint32_t b1 = __shfl_sync(0xFFFFFFFFu, byte, base + 4);
            const uint32_t b2 = __shfl_sync(0xFFFFFFFFu, byte, base + 8);
            const uint32_t b3 = __shfl_sync(0xFFFFFFFFu, byte, base + 12);
            const int r = rg * 8 + i;
            if (r < cnt) {
                const int64_t row = t0 + r;
                *reinterpret_cast<uint2 *>(a.q_row + row * a.cols + c0 + cc * 8) = codes;
                if (cc == i)
                    *reinterpret_cast<uint32_t *>(a.e8_row + mx_atom_offset(row, c0 >> 5, ka)) =
                        b0 | (b1 << 8) | (b2 << 16) | (b3 << 24);
            }
        }
    }

    if (COL) {
        float cm[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            float m = fabsf(v[0][j]);
#pragma unroll
            for (int i = 1; i < 8; ++i)
                m = fmaxf(m, fabsf(v[i][j]));
            cm[j] = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 16)); // rows 16w .. 16w+15
        }
        if (lane < 16) {
            *reinterpret_cast<float4 *>(&red[warp][cc * 8]) = make_float4(cm[0], cm[1], cm[2], cm[3]);
            *reinterpret_cast<float4 *>(&red[warp][cc * 8 + 4]) = make_float4(cm[4], cm[5], cm[6], cm[7]);
        }
        __syncthreads();
        // 32-row block k = warp / 2 covers warps 2k and 2k+1 (G = 128: all eight warps)
#pragma unroll
        for (int w = 0; w < 8; ++w) {
            if (G == 128 ? w == warp : w != (warp ^ 1))
                continue;
            const float4 p = *reinterpret_cast<const float4 *>(&red[w][cc * 8]);
            const float4 q = *reinterpret_cast<const float4 *>(&red[w][cc * 8 + 4]);
            cm[0] = fmaxf(cm[0], p.x); cm[1] = fmaxf(cm[1], p.y);
            cm[2] = fmaxf(cm[2], p.z); cm[3] = fmaxf(cm[3], p.w);
            cm[4] = fmaxf(cm[4], q.x); cm[5] = fmaxf(cm[5], q.y);
            cm[6] = fmaxf(cm[6], q.z); cm[7] = fmaxf(cm[7], q.w);
        }
        const int k = warp >> 1;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int e = e8m0_exponent(cm[j]);
            float col[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
                col[i] = v[i][j];
            tileT_put(tileT, cc * 8 + j, rg, quant8_mx(col, exp2_neg(e), cm[j] == 0.0f));
            if ((warp & 1) == 0 && lane < 16)
                reinterpret_cast<uint8_t *>(e8T)[(cc * 8 + j) * 4 + k] = (uint8_t)(e + 127);
        }
        __syncthreads();
        store_tileT(tileT, a.q_col, a.ldq_col, c0, p0);
        if (t < 128) {
            const int64_t ka = (a.cols + 127) / 128; // row bands of the column copy (rows = channels)
            *reinterpret_cast<uint32_t *>(a.e8_col + mx_atom_offset(c0 + t, p0 >> 5, ka)) = e8T[t];
        }
    }
}

// MX quantizer, persistent: two CTAs of 256 threads per SM walk the 128 x 128
// tiles; warp 0 keeps the next tile's BF16 input in flight by TMA (a two-stage
// ring, as in the FP8 activation quantizer), so HBM sees requests while a tile
// is reduced, quantized and stored.
constexpr int kMxStages = 2;
struct MxPipeSmem {
    uint16_t stage[kMxStages][128 * 128];
    MxTileSmem ts;
    Group grp[kMxStages];
    unsigned long long full[kMxStages];
    int issued[kMxStages];
    int abort;
};
constexpr size_t kMxPipeSmemBytes = sizeof(MxPipeSmem) + 1024;

template <bool ROW, bool COL, int G>
__global__ void __launch_bounds__(kThreads, 2)
    k_quant_mx_tma(const __grid_constant__ MxQuantArgs a, const __grid_constant__ CUtensorMap tmx, int64_t ngroups,
                   int ncb)
{
    extern __shared__ uint8_t smem_raw[];
    MxPipeSmem &sm = *reinterpret_cast<MxPipeSmem *>(ptx::align_smem<1024>(smem_raw));
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int rg = t >> 4, cc = t & 15;
    const int64_t total = ngroups * ncb;
    unsigned *err = &g_quant_error;

    // warp 0: map the CTA's k-th tile to its rows and start its load into stage k % kMxStages
    auto issue = [&](int64_t k) {
        const int64_t T = blockIdx.x + k * (int64_t)gridDim.x;
        if (T >= total || sm.abort)
            return;
        const int s = (int)(k % kMxStages);
        map_group(T / ncb, a.rows, a.seg, a.nseg, &sm.grp[s]);
        __syncwarp();
        if (lane == 0) {
            const uint32_t bar = ptx::smem_addr(&sm.full[s]);
            sm.issued[s] += 1;
            if (sm.grp[s].cnt > 0) {
                ptx::mbar_arrive_expect_tx(bar, kPipeTileBytes);
                ptx::tma_load_2d(ptx::smem_addr(sm.stage[s]), &tmx, bar, (int)((T % ncb) * 128), (int)sm.grp[s].t0);
            } else {
                ptx::mbar_arrive(bar);
            }
        }
        __syncwarp();
    };

    if (t == 0) {
        for (int s = 0; s < kMxStages; ++s) {
            ptx::mbar_init(ptx::smem_addr(&sm.full[s]), 1);
            sm.issued[s] = 0;
        }
        sm.abort = 0;
        ptx::fence_barrier_init();
    }
    __syncthreads();
    if (warp == 0) {
        if (lane == 0)
            ptx::prefetch_tensormap(&tmx);
        for (int s = 0; s < kMxStages; ++s)
            issue(s);
    }

    for (int64_t k = 0;; ++k) {
        const int64_t T = blockIdx.x + k * (int64_t)gridDim.x;
        if (T >= total)
            break;
        const int s = (int)(k % kMxStages);
        ptx::mbar_wait(ptx::smem_addr(&sm.full[s]), (uint32_t)((k / kMxStages) & 1), &sm.abort, err,
                       kQuantErrTimeout, kQuantWaitLimitNs);
        const int cnt = sm.grp[s].cnt;
        const int64_t t0 = sm.grp[s].t0, p0 = sm.grp[s].p0;
        const int64_t c0 = (T % ncb) * 128;
        float v[8][8];
        if (cnt > 0) {
            const uint16_t *st = sm.stage[s];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int r = rg * 8 + i;
                const uint4 raw = r < cnt ? *reinterpret_cast<const uint4 *>(st + r * 128 + cc * 8) : make_uint4(0, 0, 0, 0);
                unpack8(raw, v[i]);
            }
        }
        // every thread has its block (and finished the previous tile's shared-memory
        // work): the stage can be refilled
        ptx::fence_proxy_async_smem();
        __syncthreads();
        if (warp == 0)
            issue(k + kMxStages);
        if (cnt > 0)
            quant_mx_tile<ROW, COL, G>(a, sm.ts, v, t0, cnt, p0, c0);
    }

    // after a timed-out wait no new loads were started; wait (bounded) for the
    // ones still in flight before the CTA's shared memory is released
    if (t == 0 && sm.abort) {
        for (int s = 0; s < kMxStages; ++s)
            if (sm.issued[s] > 0)
                ptx::mbar_wait(ptx::smem_addr(&sm.full[s]), (uint32_t)((sm.issued[s] - 1) & 1), &sm.abort, err,
                               kQuantErrTimeout, kQuantWaitLimitNs, false);
    }
}

// E4M3 codes -> binary32 values (exact: every E4M3 value is an FP16 value)
__device__ __forceinline__ void decode8(uint2 codes, float (&f)[8])
{
    const uint32_t w[2] = {codes.x, codes.y};
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w[h] >> (16 * k)), __NV_E4M3);
            const float2 v = __half22float2(*reinterpret_cast<const __half2 *>(&hr));
            f[4 * h + 2 * k] = v.x;
            f[4 * h + 2 * k + 1] = v.y;
        }
}

// E4M3(fl32(v / s)) for any binary32 v, s >= 2^-96 (r = RN(1/s)): the
// residual-corrected quotient is within one binary32 ulp of fl32(v / s), so
// its E4M3 code is the same unless it lies within two ulps of an E4M3 rounding
// midpoint (bit 19 of the significand set, bits 18..0 clear) or in the E4M3
// subnormal range; those take the IEEE division.  Two values at a time.
__device__ __forceinline__ float2 quotient2_for_e4m3(float2 v, float s, float r)
{
    const float2 q0 = __fmul2_rn(v, make_float2(r, r));
    const float2 e = __ffma2_rn(q0, make_float2(-s, -s), v);
    float2 q = __ffma2_rn(e, make_float2(r, r), q0);
    const uint32_t ux = __float_as_uint(q.x) & 0x7FFFFFFFu, uy = __float_as_uint(q.y) & 0x7FFFFFFFu;
    if (ux < 0x3C800000u || ((ux & 0xFFFFFu) - 0x7FFFEu) <= 4u)
        q.x = __fdiv_rn(v.x, s);
    if (uy < 0x3C800000u || ((uy & 0xFFFFFu) - 0x7FFFEu) <= 4u)
        q.y = __fdiv_rn(v.y, s);
    return q;
}

// Column copy re-quantized from the row copy: one CTA per 128-token group x
// 128 channels; v = fl32(decode(q_row) * S_row), 128x1 column groups on v,
// q = E4M3(fl32(v / S)) (quotient2_for_e4m3; v is not a BF16 value, for which
// the plain corrected quotient is proven exact).
__global__ void __launch_bounds__(kThreads, 2) k_requant_col(const __grid_constant__ RequantArgs a)
{
    __shared__ __align__(16) float red[8][128];
    __shared__ __align__(16) float scS[128], scR[128]; // column scales and their reciprocals
    __shared__ __align__(16) uint8_t tileT[128 * 128];
    __shared__ Group grp;

    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int rg = t >> 4, cc = t & 15;
    const int64_t c0 = (int64_t)blockIdx.y * 128;

    map_group(blockIdx.x, a.n, a.seg, a.nseg, &grp);
    __syncthreads();
    const int cnt = grp.cnt;
    if (cnt == 0)
        return;
    const int64_t t0 = grp.t0, p0 = grp.p0;

    // all eight rows' loads first (rows past the group read as codes 0, scale 0)
    uint2 codes[8];
    float srow[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int r = rg * 8 + i;
        const bool in = r < cnt;
        codes[i] = in ? __ldg(reinterpret_cast<const uint2 *>(a.q_row + (t0 + r) * a.c + c0 + cc * 8))
                      : make_uint2(0u, 0u);
        srow[i] = in ? __ldg(a.s_row + (c0 >> 7) * a.n + t0 + r) : 0.0f;
    }
    float v[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        float d[8];
        decode8(codes[i], d);
#pragma unroll
        for (int j = 0; j < 8; j += 2) {
            const float2 p2 = __fmul2_rn(make_float2(d[j], d[j + 1]), make_float2(srow[i], srow[i]));
            v[i][j] = p2.x;
            v[i][j + 1] = p2.y;
        }
    }
    float cm[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        float m = fabsf(v[0][j]);
#pragma unroll
        for (int i = 1; i < 8; ++i)
            m = fmaxf(m, fabsf(v[i][j]));
        cm[j] = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 16));
    }
    if (lane < 16) {
        *reinterpret_cast<float4 *>(&red[warp][cc * 8]) = make_float4(cm[0], cm[1], cm[2], cm[3]);
        *reinterpret_cast<float4 *>(&red[warp][cc * 8 + 4]) = make_float4(cm[4], cm[5], cm[6], cm[7]);
    }
    __syncthreads();
    // each column's scale once, by one thread
    if (t < 128) {
        float m = red[0][t];
#pragma unroll
        for (int w = 1; w < 8; ++w)
            m = fmaxf(m, red[w][t]);
        const float s = __fdiv_rn(m, kE4M3Max);
        scS[t] = s;
        scR[t] = (s >= 0x1p-96f) ? __frcp_rn(s) : 0.0f;
        a.s_col[(p0 >> 7) * a.c + c0 + t] = s;
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const float s = scS[cc * 8 + j];
        const bool zero = !(s > 0.0f);
        float q[8];
        if (zero) {
#pragma unroll
            for (int i = 0; i < 8; ++i)
                q[i] = 0.0f;
        } else if (s < 0x1p-96f) {
#pragma unroll
            for (int i = 0; i < 8; ++i)
                q[i] = __fdiv_rn(v[i][j], s);
        } else {
            const float r = scR[cc * 8 + j];
#pragma unroll
            for (int i = 0; i < 8; i += 2) {
                const float2 qq = quotient2_for_e4m3(make_float2(v[i][j], v[i + 1][j]), s, r);
                q[i] = qq.x;
                q[i + 1] = qq.y;
            }
        }
        tileT_put(tileT, cc * 8 + j, rg, make_uint2(cvt4(q[0], q[1], q[2], q[3]), cvt4(q[4], q[5], q[6], q[7])));
    }
    __syncthreads();
    store_tileT(tileT, a.q_col, a.ldq_col, c0, p0);
}

// BF16 of decode(q) * S rounded once: the FP32 product is exact or within half
// an FP32 ulp, so only a product that lands exactly on a BF16 midpoint needs
// the sign of its (exact, FMA) residual; products below 2^-100, whose residual
// may not be exact, take the binary64 route.
__device__ __forceinline__ uint32_t bf16_of_product(float d, float s)
{
    const float p = __fmul_rn(d, s);
    if (p != 0.0f && fabsf(p) < 0x1p-100f)
        return __bfloat16_as_ushort(__double2bfloat16((double)d * (double)s));
    const uint32_t b = __float_as_uint(p);
    const float e = __fmaf_rn(d, s, -p);
    if ((b & 0xFFFFu) == 0x8000u && e != 0.0f)
        return (b >> 16) + (((e > 0.0f) == (p > 0.0f)) ? 1u : 0u);
    return __bfloat16_as_ushort(__float2bfloat16_rn(p));
}

// One block per (row, 4096-column segment): thread t converts columns
// 16t .. 16t+15 of the segment (no index division anywhere).
__global__ void __launch_bounds__(256) k_dequant_bf16(const __grid_constant__ DequantArgs a)
{
    const int64_t r = blockIdx.y;
    const int64_t c = (int64_t)blockIdx.x * 4096 + threadIdx.x * 16;
    if (c >= a.cols)
        return;
    const uint4 codes = __ldg(reinterpret_cast<const uint4 *>(a.q + r * a.cols + c));
    const float s = a.blocks ? __ldg(a.s + (r >> 7) * (a.cols >> 7) + (c >> 7)) : __ldg(a.s + (c >> 7) * a.rows + r);
    float d[16];
    decode8(make_uint2(codes.x, codes.y), *reinterpret_cast<float(*)[8]>(&d[0]));
    decode8(make_uint2(codes.z, codes.w), *reinterpret_cast<float(*)[8]>(&d[8]));
    uint32_t o[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        // packed product and rounding; a midpoint tie or a tiny product takes the exact route
        const float2 p2 = __fmul2_rn(make_float2(d[2 * j], d[2 * j + 1]), make_float2(s, s));
        const uint32_t bx = __float_as_uint(p2.x), by = __float_as_uint(p2.y);
        const bool odd = (bx & 0xFFFFu) == 0x8000u || (by & 0xFFFFu) == 0x8000u ||
                         ((bx & 0x7FFFFFFFu) - 1u) < 0x0D7FFFFFu || ((by & 0x7FFFFFFFu) - 1u) < 0x0D7FFFFFu;
        if (odd) {
            o[j] = bf16_of_product(d[2 * j], s) | (bf16_of_product(d[2 * j + 1], s) << 16);
        } else {
            const __nv_bfloat162 h2 = __floats2bfloat162_rn(p2.x, p2.y);
            o[j] = *reinterpret_cast<const uint32_t *>(&h2);
        }
    }
    uint4 *dst = reinterpret_cast<uint4 *>(a.out + r * a.ldo + c);
    dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
    dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
}

// ------------------------------------------------------------ NVFP4
//
// E2M1 values, one E4M3 scale per block of 16 consecutive values and an FP32
// scope scale (per row, or one for the tensor): S_g = fl32(amax / 2688),
// e_b = E4M3(fl32(fl32(amax_b / 6) / S_g)), D_b = fl32(decode(e_b) * S_g),
// q = E2M1(fl32(x / D_b)), every code 0 where D_b = 0.  One warp per row:
// lane l holds elements 256k + 8l .. +7 of the row, so a block is a lane pair.

__device__ __forceinline__ float e4m3_value(uint32_t code)
{
    const __half_raw h = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)code, __NV_E4M3);
    return __half2float(*reinterpret_cast<const __half *>(&h));
}

// 8 consecutive E2M1 codes of the quotients fl32(x / d) (d != 0), element 0 in
// the low nibble.  With r = RN(1/d): q0 = RN(x * -r), e = x + d*q0 (exact by
// FMA), q1 = RN(q0 + e * -r) is the residual-corrected quotient, negated (zero
// quotients then come out with the sign of -x; the sign bits are flipped back
// on the packed codes).  It is within one binary32 ulp of fl32(x / d), so its
// E2M1 code is the same unless it lies within two ulps of an E2M1 midpoint
// (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5: significand bits 20..0 clear); those
// quotients, and some harmless neighbours, take the IEEE division.
__device__ __forceinline__ uint32_t e2m1_codes8(const float (&v)[8], float d)
{
    const float nr = -__frcp_rn(d);
    uint32_t w = 0;
#pragma unroll
    for (int k = 0; k < 8; k += 2) {
        const float2 x2 = make_float2(v[k], v[k + 1]);
        const float2 q0 = __fmul2_rn(x2, make_float2(nr, nr));
        const float2 e = __ffma2_rn(make_float2(d, d), q0, x2);
        float2 q = __ffma2_rn(e, make_float2(nr, nr), q0);
        if (((__float_as_uint(q.x) + 2u) & 0x1FFFFFu) <= 4u)
            q.x = -__fdiv_rn(v[k], d);
        if (((__float_as_uint(q.y) + 2u) & 0x1FFFFFu) <= 4u)
            q.y = -__fdiv_rn(v[k + 1], d);
        const __nv_fp4x2_storage_t b = __nv_cvt_float2_to_fp4x2(q, __NV_E2M1, cudaRoundNearest);
        w |= (uint32_t)b << (4 * k);
    }
    return w ^ 0x88888888u; // the codes of fl32(x / d)
}

// max |x| over the tensor, folded into *amax (a non-negative float compared as its bits)
__global__ void __launch_bounds__(256) k_amax_bf16(const uint16_t *__restrict__ x, int64_t rows, int64_t cols,
                                                   int64_t ldx, float *amax)
{
    const int64_t per_row = cols / 8;
    float m = 0.0f;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < rows * per_row;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = i / per_row, c = (i - r * per_row) * 8;
        float v[8];
        unpack8(ldg_stream(x + r * ldx + c), v);
        m = fmaxf(m, absmax8(v));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    if ((threadIdx.x & 31) == 0 && m > 0.0f)
        atomicMax(reinterpret_cast<unsigned *>(amax), __float_as_uint(m));
}

// quantizes the lane's chunk (8 values at column c) with scope scale s; the block
// maximum is a lane-pair shuffle, so every lane of the warp calls it in step
__device__ __forceinline__ void nvfp4_chunk(const float (&v)[8], bool in, float s, int64_t row, int64_t c,
                                            int64_t cols, int lane, uint8_t *q, uint8_t *sb)
{
    const float own = absmax8(v);
    const float ab = fmaxf(own, __shfl_xor_sync(0xFFFFFFFFu, own, 1));
    uint32_t e = 0;
    if (s > 0.0f)
        e = __nv_cvt_float2_to_fp8x2(make_float2(__fdiv_rn(__fdiv_rn(ab, 6.0f), s), 0.0f), __NV_SATFINITE, __NV_E4M3) &
            0xFFu;
    const float d = __fmul_rn(e4m3_value(e), s);
    const uint32_t codes = d != 0.0f ? e2m1_codes8(v, d) : 0u;
    if (in) {
        *reinterpret_cast<uint32_t *>(q + row * (cols / 2) + c / 2) = codes;
        if ((lane & 1) == 0)
            sb[row * (cols / 16) + c / 16] = (uint8_t)e;
    }
}

// One warp per row, two passes over it in 256-column steps (its maximum, then
// the quantization; the second read mostly hits L1).  A lane past the row's end
// holds zeros and stores nothing (cols % 16 == 0 keeps both lanes of a block
// pair on the same side).  Holding a row in registers between the passes cut
// the warps per SM and measured slower.
template <bool PER_ROW>
__global__ void __launch_bounds__(256) k_quant_nvfp4(const uint16_t *__restrict__ x, int64_t rows, int64_t cols,
                                                     int64_t ldx, const float *scope_amax, uint8_t *__restrict__ q,
                                                     uint8_t *__restrict__ sb, float *__restrict__ sg)
{
    const int lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (row >= rows)
        return;
    const uint16_t *xr = x + row * ldx;
    float amax;
    if (PER_ROW) {
        float m = 0.0f;
        for (int64_t c = (int64_t)lane * 8; c < cols; c += 256) {
            float v[8];
            unpack8(__ldg(reinterpret_cast<const uint4 *>(xr + c)), v);
            m = fmaxf(m, absmax8(v));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
        amax = m;
    } else {
        amax = __ldg(scope_amax);
    }
    const float s = __fdiv_rn(amax, 2688.0f);
    if (lane == 0 && (PER_ROW || row == 0))
        sg[PER_ROW ? row : 0] = s;
    for (int64_t c0 = 0; c0 < cols; c0 += 256) {
        const int64_t c = c0 + lane * 8;
        const bool in = c < cols;
        float v[8];
        unpack8(in ? __ldg(reinterpret_cast<const uint4 *>(xr + c)) : make_uint4(0, 0, 0, 0), v);
        nvfp4_chunk(v, in, s, row, c, cols, lane, q, sb);
    }
}

// BF16 of e2m1 * decode(e_b) * S_g, rounded once (bf16_of_product on the exact
// binary32 product e2m1 * decode(e_b)).  Grid (column segments of 2048, groups
// of kDqRows rows): thread t converts elements 8t .. 8t+7 of its segment in
// each row of the group, the group's loads issued together.
constexpr int kDqRows = 8;

__global__ void __launch_bounds__(256) k_dequant_nvfp4(const uint8_t *__restrict__ q, const uint8_t *__restrict__ sb,
                                                       const float *__restrict__ sg, int per_row, int64_t rows,
                                                       int64_t cols, uint16_t *__restrict__ out, int64_t ldo)
{
    const int64_t r0 = (int64_t)blockIdx.y * kDqRows;
    const int64_t c = (int64_t)blockIdx.x * 2048 + threadIdx.x * 8;
    if (c >= cols)
        return;
    uint32_t w[kDqRows];
    float bs[kDqRows], s[kDqRows];
#pragma unroll
    for (int i = 0; i < kDqRows; ++i) {
        const int64_t r = r0 + i;
        const bool in = r < rows;
        w[i] = in ? __ldg(reinterpret_cast<const uint32_t *>(q + r * (cols / 2) + c / 2)) : 0u;
        bs[i] = in ? e4m3_value(__ldg(sb + r * (cols / 16) + c / 16)) : 0.0f;
        s[i] = in ? __ldg(sg + (per_row ? r : 0)) : 0.0f;
    }
#pragma unroll
    for (int i = 0; i < kDqRows; ++i) {
        if (r0 + i >= rows)
            break;
        uint32_t o[4];
#pragma unroll
        for (int k = 0; k < 8; k += 2) {
            const __half2_raw hr =
                __nv_cvt_fp4x2_to_halfraw2((__nv_fp4x2_storage_t)((w[i] >> (4 * k)) & 0xFFu), __NV_E2M1);
            const float2 e2 = __half22float2(*reinterpret_cast<const __half2 *>(&hr));
            o[k / 2] = bf16_of_product(__fmul_rn(e2.x, bs[i]), s[i]) |
                       (bf16_of_product(__fmul_rn(e2.y, bs[i]), s[i]) << 16);
        }
        *reinterpret_cast<uint4 *>(out + (r0 + i) * ldo + c) = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

int64_t groups_upper_bound(int64_t n, const int64_t *seg, int nseg)
{
    const int64_t g = (n + 127) / 128;
    return seg ? g + nseg : g;
}

} // namespace

namespace {

template <bool ROW, bool COL, int P>
cudaError_t launch_quant_act_tma(const ActQuantArgs &a, const CUtensorMap &map, int64_t ngroups, int ncb,
                                 cudaStream_t st)
{
    auto kern = k_quant_act_tma<ROW, COL, P>;
    static int configured_device = -1;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (configured_device != dev) {
        if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kPipeSmemBytes)) !=
            cudaSuccess)
            return e;
        configured_device = dev;
    }
    const int64_t tiles = ngroups * ncb;
    const int64_t cap = 2 * (int64_t)sm_count();
    if ((e = launch_pdl(kern, dim3((unsigned)(tiles < cap ? tiles : cap)), dim3(kThreads), kPipeSmemBytes, st, a, map,
                        ngroups, ncb)) != cudaSuccess)
        return e;
    return cudaGetLastError();
}

template <bool ROW, bool COL, int G>
cudaError_t launch_quant_mx_tma(const MxQuantArgs &a, const CUtensorMap &map, int64_t ngroups, int ncb,
                                cudaStream_t st)
{
    auto kern = k_quant_mx_tma<ROW, COL, G>;
    static int configured_device = -1;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (configured_device != dev) {
        if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kMxPipeSmemBytes)) !=
            cudaSuccess)
            return e;
        configured_device = dev;
    }
    const int64_t tiles = ngroups * ncb;
    const int64_t cap = 2 * (int64_t)sm_count();
    kern<<<(unsigned)(tiles < cap ? tiles : cap), kThreads, kMxPipeSmemBytes, st>>>(a, map, ngroups, ncb);
    return cudaGetLastError();
}

template <int P>
cudaError_t launch_quant_act_tma_p(const ActQuantArgs &a, cudaStream_t st)
{
    if (a.n > 2147483647 - 128 || a.c > 2147483647)
        return cudaErrorInvalidValue; // TMA coordinates are 32-bit
    CUtensorMap map;
    cudaError_t e = make_bf16_tile_map(&map, a.x, a.c, a.n, a.ldx);
    if (e != cudaSuccess)
        return e;
    const int64_t ngroups = groups_upper_bound(a.n, a.seg, a.nseg);
    const int ncb = (int)(a.c / 128);
    if (a.q_row && a.q_col)
        return launch_quant_act_tma<true, true, P>(a, map, ngroups, ncb, st);
    if (a.q_row)
        return launch_quant_act_tma<true, false, P>(a, map, ngroups, ncb, st);
    return launch_quant_act_tma<false, true, P>(a, map, ngroups, ncb, st);
}

template <bool ROW, bool COL>
cudaError_t launch_quant_act_swiglu_rc(const ActQuantArgs &a, int64_t ngroups, int ncb, cudaStream_t st)
{
    auto kern = k_quant_act_swiglu<ROW, COL>;
    constexpr size_t smem = sizeof(SwiSmem) + 16;
    static int configured_device = -1;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (configured_device != dev) {
        if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
            return e;
        configured_device = dev;
    }
    const int64_t tiles = ngroups * ncb;
    const int64_t cap = 2 * (int64_t)sm_count();
    kern<<<(unsigned)(tiles < cap ? tiles : cap), kThreads, smem, st>>>(a, ngroups, ncb);
    return cudaGetLastError();
}

cudaError_t launch_quant_act_swiglu(const ActQuantArgs &a, cudaStream_t st)
{
    const int64_t ngroups = groups_upper_bound(a.n, a.seg, a.nseg);
    const int ncb = (int)(a.c / 128);
    if (a.q_row && a.q_col)
        return launch_quant_act_swiglu_rc<true, true>(a, ngroups, ncb, st);
    if (a.q_row)
        return launch_quant_act_swiglu_rc<true, false>(a, ngroups, ncb, st);
    return launch_quant_act_swiglu_rc<false, true>(a, ngroups, ncb, st);
}

} // namespace

cudaError_t launch_quant_act(const ActQuantArgs &a, cudaStream_t st)
{
    if (a.n == 0 || (!a.q_row && !a.q_col))
        return cudaSuccess;
    switch (a.producer) {
    case kProducePlain:
        return launch_quant_act_tma_p<kProducePlain>(a, st);
    case kProduceRms:
        if (!a.w || !a.rstd)
            return cudaErrorInvalidValue;
        return launch_quant_act_tma_p<kProduceRms>(a, st);
    case kProduceSwiglu:
        if (!a.up)
            return cudaErrorInvalidValue;
        return launch_quant_act_swiglu(a, st);
    default:
        return cudaErrorInvalidValue;
    }
}

cudaError_t launch_rms_rstd(const uint16_t *x, int64_t n, int64_t c, int64_t ldx, float eps, float *rstd,
                            cudaStream_t st)
{
    if (n == 0)
        return cudaSuccess;
    if (c <= 0 || c % 128 != 0 || c > 32768)
        return cudaErrorInvalidValue;
    // as many CTAs as are resident at once (registers and stages permitting); warps then walk the rows
    static int per_sm = 0;
    if (per_sm == 0) {
        int v = 0;
        const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, k_rms_rstd, kRmsWarps * 32, 0);
        if (e != cudaSuccess)
            return e;
        per_sm = v > 0 ? v : 1;
    }
    const int64_t blocks = (n + kRmsWarps - 1) / kRmsWarps, cap = (int64_t)per_sm * sm_count();
    k_rms_rstd<<<(unsigned)(blocks < cap ? blocks : cap), kRmsWarps * 32, 0, st>>>(x, n, c, ldx, eps, rstd);
    return cudaGetLastError();
}

cudaError_t quant_read_and_clear_error(cudaStream_t st, unsigned *out)
{
    unsigned v = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(&v, g_quant_error, sizeof v, 0, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(st);
    if (e != cudaSuccess)
        return e;
    *out |= v;
    if (v) {
        const unsigned zero = 0;
        e = cudaMemcpyToSymbolAsync(g_quant_error, &zero, sizeof zero, 0, cudaMemcpyHostToDevice, st);
        if (e == cudaSuccess)
            e = cudaStreamSynchronize(st);
    }
    return e;
}

cudaError_t launch_quant_weight(const WeightQuantArgs &a, cudaStream_t st)
{
    if (a.d > 2147483647 || a.c > 2147483647)
        return cudaErrorInvalidValue; // TMA coordinates are 32-bit
    static int configured_device = -1;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (configured_device != dev) {
        if ((e = cudaFuncSetAttribute(k_quant_weight_tma, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)kWPipeSmemBytes)) != cudaSuccess)
            return e;
        configured_device = dev;
    }
    CUtensorMap map;
    if ((e = make_bf16_tile_map(&map, a.w, a.c, a.d, a.ldw)) != cudaSuccess)
        return e;
    const int64_t tiles = (a.d / 128) * (a.c / 128);
    const int64_t cap = 2 * (int64_t)sm_count();
    if ((e = launch_pdl(k_quant_weight_tma, dim3((unsigned)(tiles < cap ? tiles : cap)), dim3(kThreads),
                        kWPipeSmemBytes, st, a, map)) != cudaSuccess)
        return e;
    return cudaGetLastError();
}

cudaError_t launch_quant_mx(const MxQuantArgs &a, int group, cudaStream_t st)
{
    if (a.rows == 0 || (!a.q_row && !a.q_col))
        return cudaSuccess;
    if (group != 32 && group != 128)
        return cudaErrorInvalidValue;
    if (a.rows > 2147483647 - 128 || a.cols > 2147483647)
        return cudaErrorInvalidValue; // TMA coordinates are 32-bit
    CUtensorMap map;
    cudaError_t e = make_bf16_tile_map(&map, a.x, a.cols, a.rows, a.ldx);
    if (e != cudaSuccess)
        return e;
    const int64_t ngroups = groups_upper_bound(a.rows, a.seg, a.nseg);
    const int ncb = (int)(a.cols / 128);
    if (group == 32) {
        if (a.q_row && a.q_col)
            return launch_quant_mx_tma<true, true, 32>(a, map, ngroups, ncb, st);
        if (a.q_row)
            return launch_quant_mx_tma<true, false, 32>(a, map, ngroups, ncb, st);
        return launch_quant_mx_tma<false, true, 32>(a, map, ngroups, ncb, st);
    }
    if (a.q_row && a.q_col)
        return launch_quant_mx_tma<true, true, 128>(a, map, ngroups, ncb, st);
    if (a.q_row)
        return launch_quant_mx_tma<true, false, 128>(a, map, ngroups, ncb, st);
    return launch_quant_mx_tma<false, true, 128>(a, map, ngroups, ncb, st);
}

cudaError_t launch_requant_col(const RequantArgs &a, cudaStream_t st)
{
    if (a.n == 0)
        return cudaSuccess;
    dim3 grid((unsigned)groups_upper_bound(a.n, a.seg, a.nseg), (unsigned)(a.c / 128));
    k_requant_col<<<grid, kThreads, 0, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_amax_bf16(const uint16_t *x, int64_t rows, int64_t cols, int64_t ldx, float *amax,
                             cudaStream_t st)
{
    if (rows == 0)
        return cudaSuccess;
    const int64_t threads = rows * (cols / 8), cap = 4 * (int64_t)sm_count();
    const int64_t blocks = (threads + 255) / 256;
    k_amax_bf16<<<(unsigned)(blocks < cap ? blocks : cap), 256, 0, st>>>(x, rows, cols, ldx, amax);
    return cudaGetLastError();
}

cudaError_t launch_quant_nvfp4(const uint16_t *x, int64_t rows, int64_t cols, int64_t ldx, const float *scope_amax,
                               uint8_t *q, uint8_t *sb, float *sg, cudaStream_t st)
{
    if (rows == 0)
        return cudaSuccess;
    const int64_t blocks = (rows + 7) / 8;
    if (blocks > 2147483647)
        return cudaErrorInvalidValue;
    if (scope_amax)
        k_quant_nvfp4<false><<<(unsigned)blocks, 256, 0, st>>>(x, rows, cols, ldx, scope_amax, q, sb, sg);
    else
        k_quant_nvfp4<true><<<(unsigned)blocks, 256, 0, st>>>(x, rows, cols, ldx, nullptr, q, sb, sg);
    return cudaGetLastError();
}

cudaError_t launch_dequant_nvfp4(const uint8_t *q, const uint8_t *sb, const float *sg, int per_row, int64_t rows,
                                 int64_t cols, uint16_t *out, int64_t ldo, cudaStream_t st)
{
    if (rows == 0)
        return cudaSuccess;
    // row groups on grid.y (at most 65535 per launch), column segments of 2048 on grid.x
    constexpr int64_t kRowsPerLaunch = (int64_t)65535 * kDqRows;
    for (int64_t r0 = 0; r0 < rows; r0 += kRowsPerLaunch) {
        const int64_t nr = rows - r0 < kRowsPerLaunch ? rows - r0 : kRowsPerLaunch;
        dim3 grid((unsigned)((cols + 2047) / 2048), (unsigned)((nr + kDqRows - 1) / kDqRows));
        k_dequant_nvfp4<<<grid, 256, 0, st>>>(q + r0 * (cols / 2), sb + r0 * (cols / 16), per_row ? sg + r0 : sg,
                                              per_row, nr, cols, out + r0 * ldo, ldo);
    }
    return cudaGetLastError();
}

cudaError_t launch_dequant_bf16(const DequantArgs &a, cudaStream_t st)
{
    if (a.rows == 0)
        return cudaSuccess;
    if (a.rows > 2147483647)
        return cudaErrorInvalidValue;
    dim3 grid((unsigned)((a.cols + 4095) / 4096), (unsigned)a.rows);
    k_dequant_bf16<<<grid, 256, 0, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_quant_weight_pow2(const WeightPow2Args &a, cudaStream_t st)
{
    dim3 grid((unsigned)(a.d / 128), (unsigned)(a.c / 128));
    k_quant_weight_pow2<<<grid, kThreads, 0, st>>>(a);
    return cudaGetLastError();
}

} // namespace jetq
