// Tile table of a grouped GEMM, built on the device from the expert offsets.
//
// Group g < E is routed expert g (rows offsets[g] .. offsets[g+1]-1 of A0);
// group E + s is shared expert s (T rows of A1). Each group is cut into
// ceil(M_g / BM) row tiles and nt column tiles. Tiles are numbered group by
// group. Inside a group the row tiles are taken in blocks of rb
// (GroupedGemm::row_block; 0: one block of all of them), and inside a block
// column-tile-major with the block's row tiles consecutive: CTAs that run at
// the same time share a weight tile through L2, and a block's token rows stay
// in L2 while every weight tile of the expert passes over them.
#pragma once

#include "moe_internal.cuh"

namespace moe {

struct GroupTile {
    int g;        // group
    int m0;       // first row of the tile inside the group
    int n_tile;   // column tile
    int rows;     // valid rows of the group from m0 (may exceed BM)
    int a_row;    // first A row of the tile
    int out_row;  // first output row of the tile (in out0 for routed, out1 for shared)
    int b_row;    // first B row of the group (in B0 or B1)
};

// Whether a group of `rows` rows takes part in this launch (GroupedGemm::
// rows_lo / rows_hi: a layer can run its many-row and its few-row experts as
// two launches with different tile shapes; 0 means no bound).
__device__ __forceinline__ bool in_launch(const GroupedGemm& p, int rows) {
    return rows >= p.rows_lo && (p.rows_hi <= 0 || rows <= p.rows_hi);
}

// L2: read the offsets from L2 (ld.global.cg), for reads made before the wait
// for the preceding kernel (the offsets are final by then, but an L1 line
// could predate them); otherwise plain loads.
template <bool L2 = false>
__device__ __forceinline__ int group_rows(const GroupedGemm& p, int g, int* a_row, int* out_row,
                                          bool* bad) {
    if (g < p.E) {
        const int lo = L2 ? __ldcg(p.offsets + g) : p.offsets[g];
        const int hi = L2 ? __ldcg(p.offsets + g + 1) : p.offsets[g + 1];
        if (lo < 0 || hi < lo || hi > p.max_rows0) {
            *bad = true;
            *a_row = 0;
            *out_row = 0;
            return 0;
        }
        *a_row = lo;
        *out_row = lo;
        return in_launch(p, hi - lo) ? hi - lo : 0;
    }
    const int s = g - p.E;
    *a_row = p.a1_row0 + s * p.a1_stride;
    *out_row = s * p.T;
    return in_launch(p, p.T) ? p.T : 0;
}

// Warp 0 of the block fills mt_start[0..G] (row-tile prefix) and, if grows is
// not NULL, grows[g] = rows of group g. Caller syncs.
template <bool L2 = false>
__device__ __forceinline__ void build_tile_table(const GroupedGemm& p, int BM, int* mt_start,
                                                 int* grows = nullptr) {
    if (threadIdx.x >= 32) return;
    const int lane = threadIdx.x;
    const int G = p.E + p.S;
    int running = 0;
    bool bad = false;
    for (int base = 0; base < G; base += 32) {
        const int g = base + lane;
        int mt = 0;
        if (g < G) {
            int ar, orow;
            int M = group_rows<L2>(p, g, &ar, &orow, &bad);
            mt = (M + BM - 1) / BM;
            if (grows) grows[g] = M;
        }
        int incl = mt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int n = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += n;
        }
        if (g < G) mt_start[g] = running + incl - mt;
        running += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) mt_start[G] = running;
    if (__any_sync(0xffffffffu, bad) && lane == 0) flag_status(p.status, DEV_BAD_ARG);
}

// (row tile, column tile) of the local-th tile of a group of mt row tiles
// and nt column tiles, in blocks of rb row tiles (rb <= 0: one block).
__device__ __forceinline__ void tile_position(int local, int mt, int nt, int rb, int* m,
                                              int* n) {
    if (rb <= 0 || rb >= mt) {
        *n = local / mt;
        *m = local - *n * mt;
        return;
    }
    const int blk = local / (rb * nt);
    const int within = local - blk * rb * nt;
    const int rows = min(rb, mt - blk * rb);  // row tiles of this block
    *n = within / rows;
    *m = blk * rb + (within - *n * rows);
}

// Valid rows of tile `tile` (at most BM) from the shared-memory tables alone.
__device__ __forceinline__ int tile_rows(const int* mt_start, const int* grows, int G, int nt,
                                         int BM, int tile, int rb) {
    int lo = 0, hi = G - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (mt_start[mid] * nt <= tile) lo = mid;
        else hi = mid - 1;
    }
    const int mt = mt_start[lo + 1] - mt_start[lo];
    int m, n;
    tile_position(tile - mt_start[lo] * nt, mt, nt, rb, &m, &n);
    return min(BM, grows[lo] - m * BM);
}

template <bool L2 = false>
__device__ __forceinline__ GroupTile decode_tile(const GroupedGemm& p, const int* mt_start,
                                                 int nt, int BM, int tile) {
    const int G = p.E + p.S;
    // largest g with mt_start[g] * nt <= tile
    int lo = 0, hi = G - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (mt_start[mid] * nt <= tile) lo = mid;
        else hi = mid - 1;
    }
    GroupTile t;
    t.g = lo;
    const int mt = mt_start[lo + 1] - mt_start[lo];
    int m;
    tile_position(tile - mt_start[lo] * nt, mt, nt, p.row_block, &m, &t.n_tile);
    t.m0 = m * BM;
    bool bad = false;
    int a_row, out_row;
    const int M = group_rows<L2>(p, lo, &a_row, &out_row, &bad);
    t.rows = M - t.m0;
    t.a_row = a_row + t.m0;
    t.out_row = out_row + t.m0;
    t.b_row = (lo < p.E ? lo : lo - p.E) * p.b_rows_group;
    return t;
}

}  // namespace moe
