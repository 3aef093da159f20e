// gemm_tiles.cuh -- the ragged tile schedule of the persistent grouped GEMMs
// (bf16 and 3xTF32): a per-group tile table built on the device from the
// group row offsets (no host synchronisation), and tile -> (group, n-tile,
// m-tile) decoding.
#pragma once

#include "common.cuh"

namespace moe {
namespace tiles {

constexpr int kMaxGroups = 256;  // one warp builds the table: 8 groups per lane

// Tile -> (group, n-tile, m-tile) from the per-group tile table.
struct TileInfo {
    int g, m_tile, n_tile, row0, rows;
    int kb0, nkb;  // K blocks of the tile
};

// Exclusive prefix sum over a warp.
__device__ __forceinline__ int warp_excl_scan(int v, int lane, int* total) {
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
    }
    *total = __shfl_sync(0xffffffffu, incl, 31);
    return incl - v;
}

// The per-group tile table, built by one warp (lane l covers groups [8l, 8l+8)).
// Row-offset mode: tstart[g] = first tile of group g, mt[g] = its m-tiles (at
// least 1), rowoff/grows = its first row and row count; groups own rows
// [offsets[g], offsets[g+1]) (one group of m_rows rows when offsets is null).
// K-grouped mode: every group has ceil(kg_M / BM) m-tiles over the K blocks
// its rows fill (rows padded to BK); rowoff/grows = its first K block and
// K-block count.  *total_s = number of tiles.
template <bool KG, int BM, int BK>
__device__ __forceinline__ void build_tile_table(const int32_t* offsets, int64_t m_rows, int G,
                                                 int n_tiles, int kg_M, int lane, int* tstart,
                                                 int* mt, int* rowoff, int* grows, int* total_s) {
    int cnt[8], kbs[8];
    int sum = 0, ksum = 0;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const int g = lane * 8 + q;
        cnt[q] = 0;
        kbs[q] = 0;
        if (g < G) {
            const int lo = offsets ? offsets[g] : 0;
            const int hi = offsets ? offsets[g + 1] : (int)m_rows;
            if (KG) {
                const int m = (kg_M + BM - 1) / BM;
                kbs[q] = (hi - lo + BK - 1) / BK;
                mt[g] = m;
                grows[g] = kbs[q];
                cnt[q] = m * n_tiles;  // a group without rows gets zero tiles written
            } else {
                const int m = (hi - lo + BM - 1) / BM;
                mt[g] = m > 0 ? m : 1;
                rowoff[g] = lo;
                grows[g] = hi - lo;
                cnt[q] = m * n_tiles;
            }
            sum += cnt[q];
            ksum += kbs[q];
        }
    }
    int total_tiles, total_kb;
    int run = warp_excl_scan(sum, lane, &total_tiles);
    int krun = warp_excl_scan(ksum, lane, &total_kb);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const int g = lane * 8 + q;
        if (g < G) {
            tstart[g] = run;
            if (KG) rowoff[g] = krun;
        }
        run += cnt[q];
        krun += kbs[q];
    }
    if (lane == 31) *total_s = total_tiles;
}

// Row-offset mode: rowoff/grows hold each group's first row and row count.
// K-grouped mode: they hold each group's first K block and K-block count.
// P supplies kg_M, band, n_tiles and num_kb.  With p.band > 0 a group's tiles
// run in bands of p.band n-tiles, m-tile fastest inside a band; otherwise
// n-tile by n-tile, m-tile fastest.
template <bool KG, int BM, class P>
__device__ __forceinline__ TileInfo decode_tile(int tile, int G, const int* tstart, const int* mt,
                                                const int* rowoff, const int* grows, const P& p) {
    int lo = 0, hi = G - 1;  // last g with tstart[g] <= tile
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (tstart[mid] <= tile) lo = mid;
        else hi = mid - 1;
    }
    TileInfo ti;
    ti.g = lo;
    const int local = tile - tstart[lo];
    ti.n_tile = local / mt[lo];
    ti.m_tile = local - ti.n_tile * mt[lo];
    if (KG) {
        ti.row0 = ti.m_tile * BM;
        ti.rows = p.kg_M - ti.row0;
        ti.kb0 = rowoff[lo];
        ti.nkb = grows[lo];
    } else {
        if (p.band > 0) {
            // band b holds n-tiles [b*band, b*band + wb); its tiles run m-fastest
            const int b = local / (mt[lo] * p.band);
            const int wb = min(p.band, p.n_tiles - b * p.band);
            const int lb = local - b * mt[lo] * p.band;
            ti.m_tile = lb / wb;
            ti.n_tile = b * p.band + (lb - ti.m_tile * wb);
        }
        ti.row0 = rowoff[lo] + ti.m_tile * BM;
        ti.rows = grows[lo] - ti.m_tile * BM;
        ti.kb0 = 0;
        ti.nkb = p.num_kb;
    }
    if (ti.rows > BM) ti.rows = BM;
    return ti;
}

}  // namespace tiles
}  // namespace moe
