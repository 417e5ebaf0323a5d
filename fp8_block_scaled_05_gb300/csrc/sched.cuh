// Output-tile schedule shared by the persistent large-M GEMM kernels (dense
// and grouped): tile index -> (rows, weight rows, output columns, expert).
#pragma once
#include <cstdint>

namespace fp8bs {

struct Tile {
    int32_t m0, row_end, brow, n0, g;
};

// Rows [lo, hi) of expert g: the offsets clamped to [0, M], each range
// starting where the previous one ends or later.
__device__ __forceinline__ void group_rows(const int32_t* __restrict__ offsets, int g, int M, int& lo, int& hi) {
    lo = min(max(offsets[g], 0), M);
    hi = min(max(offsets[g + 1], lo), M);
}

// Tile t -> coordinates.  Dense: the operand that is re-read once per tile
// column (or row) of the other is the smaller one, so that it stays in L2:
// with M <= N m-tiles vary fastest (CTAs running at the same time share the
// B tile, and A is re-read per column of tiles); with M > N (e.g. a weight
// gradient, M = out-features, N = in-features) n-tiles vary fastest and B is
// the one re-read.  Grouped: tiles of expert g follow
// those of expert g-1; inside an expert, m-tiles vary fastest.  cum[g] is the
// number of tiles of experts before g (shared memory, from
// build_group_table).
template <int BM, int BN, bool GROUPED>
__device__ __forceinline__ Tile decode_tile(int t, int M, int N, const int32_t* cum,
                                            const int32_t* __restrict__ offsets, int G) {
    Tile r;
    if (!GROUPED) {
        int mt, nt;
        if (M > N) {
            const int NT = (N + BN - 1) / BN;
            mt = t / NT;
            nt = t % NT;
        } else {
            const int MT = (M + BM - 1) / BM;
            mt = t % MT;
            nt = t / MT;
        }
        r.m0 = mt * BM;
        r.row_end = M;
        r.brow = nt * BN;
        r.n0 = nt * BN;
        r.g = 0;
    } else {
        int lo = 0, hi = G;   // largest g with cum[g] <= t
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (cum[mid] <= t) lo = mid; else hi = mid;
        }
        const int g = lo;
        int rlo, rhi;
        group_rows(offsets, g, M, rlo, rhi);
        const int local = t - cum[g];
        const int MTg = (rhi - rlo + BM - 1) / BM;
        const int mt = local % MTg, nt = local / MTg;
        r.m0 = rlo + mt * BM;
        r.row_end = rhi;
        r.brow = g * N + nt * BN;
        r.n0 = nt * BN;
        r.g = g;
    }
    return r;
}

// Executed by one whole warp: the running tile count cum[0..G] of the
// experts (NT output-column tiles per row tile); returns the total number of
// tiles on every lane.
template <int BM>
__device__ __forceinline__ int build_group_table(const int32_t* __restrict__ offsets, int G, int M, int NT,
                                                 int32_t* cum) {
    const int lane = threadIdx.x & 31;
    int carry = 0;
    if (lane == 0) cum[0] = 0;
    for (int g0 = 0; g0 < G; g0 += 32) {
        const int g = g0 + lane;
        int tiles = 0;
        if (g < G) {
            int lo, hi;
            group_rows(offsets, g, M, lo, hi);
            tiles = ((hi - lo + BM - 1) / BM) * NT;
        }
        int incl = tiles;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (lane >= o) incl += v;
        }
        if (g < G) cum[g + 1] = carry + incl;
        carry += __shfl_sync(0xFFFFFFFFu, incl, 31);
    }
    return carry;
}

// Tail split of the persistent large-M kernels: the last, partial wave of
// output tiles (dense only) is split along K so that it fills the GPU.
// Tiles [0, n_full) are computed whole; each tile n_full + i is computed as
// `parts` items over K-block ranges [p KB / parts, (p + 1) KB / parts), whose
// fp32 results meet in `part` ([tile][part][column][row]) and are added in
// part order by the warp that completes the tile slice's ticket (one slice
// per epilogue warp).  parts <= 1: no split.
struct SplitTail {
    int n_full;
    int parts;
    float* part;
    int* ticket;      // one per (split tile, epilogue warp); zero between calls
};

struct Item {
    int tile, kb0, kb1, part, parts;
};

__host__ __device__ __forceinline__ int work_items(int n_tiles, const SplitTail& sp) {
    return sp.parts > 1 ? sp.n_full + (n_tiles - sp.n_full) * sp.parts : n_tiles;
}

__device__ __forceinline__ Item decode_item(int t, const SplitTail& sp, int KB) {
    Item w;
    if (sp.parts <= 1 || t < sp.n_full) {
        w.tile = t;
        w.kb0 = 0;
        w.kb1 = KB;
        w.part = 0;
        w.parts = 1;
    } else {
        const int j = t - sp.n_full;
        w.tile = sp.n_full + j / sp.parts;
        w.part = j % sp.parts;
        w.parts = sp.parts;
        w.kb0 = w.part * KB / sp.parts;
        w.kb1 = (w.part + 1) * KB / sp.parts;
    }
    return w;
}

}  // namespace fp8bs
