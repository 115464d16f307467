// Persistent tile schedules shared by the GEMM kernels: one dense problem,
// or a group of per-expert problems whose segment bounds live on the device.
#pragma once

#include <cstdint>

namespace jetq {

constexpr int kMaxExperts = 256;
constexpr int kGroupM = 8;

enum SchedMode : int {
    kDense = 0,       // one problem, tiles over [M x N]
    kGroupedRows = 1, // FProp/DGrad: expert e owns routed rows seg[e] .. seg[e+1]-1 and weight rows e*N ..
    kGroupedK = 2     // WGrad: expert e owns K-blocks kb_off[e] .. kb_off[e+1]-1 of the column copies
};

struct Sched {
    int mode;
    int mt, nt;         // dense: tile grid; grouped: m-tiles (K mode) / n-tiles per expert
    int num_kb;         // K-blocks per tile (dense, grouped rows); K-blocks of the column copies (grouped K)
    int64_t M;          // rows of A: dense M, routed rows R, or D
    int N;              // output columns of one problem
    int bn;             // tile width
    const int64_t *seg; // grouped: device segment bounds [E + 1]
    int64_t seg_max;    // segment bounds are clamped into [0, seg_max]
    int E;
};

struct TileInfo {
    int a_row0; // first A row (TMA coordinate)
    int b_row0; // first B row (TMA coordinate)
    int kb0;    // first K-block
    int num_kb; // K-blocks of this tile (0: an empty expert, output is zero)
    int m_end;  // rows a_row0 .. m_end-1 belong to this tile's problem
    int n0;     // first output column inside the problem
    int e;      // expert (0 for dense)
};

// Per-CTA tables for the grouped modes, built once at kernel start.
struct GroupTables {
    int tile_prefix[kMaxExperts + 1]; // tiles before expert e
    int row_off[kMaxExperts + 1];     // grouped rows: first routed row of e; grouped K: first K-block of e
};

__device__ __forceinline__ void dense_coords(int t, int mt, int nt, int &mi, int &ni)
{
    const int group = kGroupM * nt;
    const int first_m = (t / group) * kGroupM;
    const int gm = min(mt - first_m, kGroupM);
    const int r = t % group;
    mi = first_m + r % gm;
    ni = r / gm;
}

// One warp builds the tables (segment bounds clamped into [0, seg_max]; a
// decreasing pair is an empty segment), so any device contents give an
// in-bounds schedule.
__device__ __forceinline__ void build_group_tables(const Sched &s, GroupTables *g)
{
    const int lane = threadIdx.x & 31;
    const int per = (s.E + 31) / 32;
    const int e0 = min(s.E, lane * per), e1 = min(s.E, e0 + per);
    auto bound = [&](int e) -> int64_t {
        int64_t v = s.seg[e];
        return v < 0 ? 0 : (v > s.seg_max ? s.seg_max : v);
    };
    // chunk sums: tiles (rows mode) or K-blocks (K mode)
    int sum = 0;
    for (int e = e0; e < e1; ++e) {
        const int64_t lo = bound(e), hi = bound(e + 1);
        const int64_t n = hi > lo ? hi - lo : 0;
        sum += (int)((n + 127) / 128) * (s.mode == kGroupedRows ? s.nt : 1);
    }
    int incl = sum;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int v = __shfl_up_sync(0xFFFFFFFFu, incl, d);
        if (lane >= d)
            incl += v;
    }
    int acc = incl - sum;
    for (int e = e0; e < e1; ++e) {
        const int64_t lo = bound(e), hi = bound(e + 1);
        const int64_t n = hi > lo ? hi - lo : 0;
        const int units = (int)((n + 127) / 128) * (s.mode == kGroupedRows ? s.nt : 1);
        if (s.mode == kGroupedRows) {
            g->tile_prefix[e] = acc;
            g->row_off[e] = (int)lo;
        } else {
            g->tile_prefix[e] = e * s.mt * s.nt;
            g->row_off[e] = acc; // first K-block of the expert in the column copies
        }
        acc += units;
    }
    if (lane == 31) {
        if (s.mode == kGroupedRows) {
            g->tile_prefix[s.E] = acc;
            g->row_off[s.E] = (int)bound(s.E);
        } else {
            g->tile_prefix[s.E] = s.E * s.mt * s.nt;
            g->row_off[s.E] = acc;
        }
    }
}

__device__ __forceinline__ int total_tiles(const Sched &s, const GroupTables *g)
{
    return s.mode == kDense ? s.mt * s.nt : g->tile_prefix[s.E];
}

__device__ __forceinline__ TileInfo get_tile(const Sched &s, const GroupTables *g, int t)
{
    TileInfo ti;
    if (s.mode == kDense) {
        int mi, ni;
        dense_coords(t, s.mt, s.nt, mi, ni);
        ti.a_row0 = mi * 128;
        ti.b_row0 = ni * s.bn;
        ti.kb0 = 0;
        ti.num_kb = s.num_kb;
        ti.m_end = (int)(s.M < (int64_t)ti.a_row0 + 128 ? s.M : ti.a_row0 + 128);
        ti.n0 = ni * s.bn;
        ti.e = 0;
    } else if (s.mode == kGroupedRows) {
        int lo = 0, hi = s.E; // largest e with tile_prefix[e] <= t
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (g->tile_prefix[mid] <= t)
                lo = mid;
            else
                hi = mid - 1;
        }
        const int e = lo;
        const int local = t - g->tile_prefix[e];
        const int mt_e = (g->tile_prefix[e + 1] - g->tile_prefix[e]) / s.nt;
        const int mi = local % mt_e, ni = local / mt_e;
        ti.a_row0 = g->row_off[e] + mi * 128;
        ti.m_end = min(g->row_off[e + 1], ti.a_row0 + 128);
        ti.b_row0 = e * s.N + ni * s.bn;
        ti.kb0 = 0;
        ti.num_kb = s.num_kb;
        ti.n0 = ni * s.bn;
        ti.e = e;
    } else {
        const int per = s.mt * s.nt;
        const int e = t / per, local = t % per;
        const int mi = local % s.mt, ni = local / s.mt;
        ti.a_row0 = mi * 128;
        ti.m_end = (int)(s.M < (int64_t)ti.a_row0 + 128 ? s.M : ti.a_row0 + 128);
        ti.b_row0 = ni * s.bn;
        // never past the K-blocks the column copies hold, whatever the offsets say
        ti.kb0 = min(g->row_off[e], s.num_kb);
        ti.num_kb = min(g->row_off[e + 1], s.num_kb) - ti.kb0;
        ti.n0 = ni * s.bn;
        ti.e = e;
    }
    return ti;
}

} // namespace jetq
