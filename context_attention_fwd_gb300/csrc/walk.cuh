// walk.cuh -- the order in which a CTA visits the tiles of the other operand.
//
// Forward (a CTA holds query rows of ring chunk r): at ring iteration it the
// queries meet KV chunk (r - it) mod P (diffusers issue #14265, "Root cause":
// the query stays put while the K/V chunks rotate); with the all-gather order
// they meet chunk it.  Backward (a CTA holds one KV tile of chunk c): the
// query chunks (c + it) mod P, i.e. the chunks that met c at iteration it.
// With causal masking, tiles entirely above the diagonal are skipped.
#pragma once

#include "internal.h"

namespace ctxattn {

// ------------------------------------------------------------ launch order
// (tile, head, z) of this CTA: the grid is (tiles, heads, z) in the tile-major
// order and (heads, z, tiles) in the head-major one, which launches tile 0 of
// every head before tile 1 of any (the host picks the order per launch).
struct GridPos {
    int tile, head, z;
};
template <bool kHeadMajor>
__device__ __forceinline__ GridPos grid_pos() {
    if (kHeadMajor) return {(int)blockIdx.z, (int)blockIdx.x, (int)blockIdx.y};
    return {(int)blockIdx.x, (int)blockIdx.y, (int)blockIdx.z};
}
inline dim3 grid_dims(bool head_major, int tiles, int heads, int z) {
    return head_major ? dim3(heads, z, tiles) : dim3(tiles, heads, z);
}

// ------------------------------------------------------------ forward walk
struct KvWalk {
    int it, c, t, t0, t1;
};
struct WalkCfg {
    int r, P, causal, allgather, q_last;  // q_last: the CTA's last query row (global)
};
__device__ __forceinline__ void kv_set_chunk(const ChunkTable& ct, const WalkCfg& g, KvWalk& w) {
    w.c = g.allgather ? w.it : (g.r - w.it + g.P) % g.P;
    w.t0 = w.t = ct.tile_off[w.c];
    w.t1 = ct.tile_off[w.c + 1];
}
__device__ __forceinline__ bool kv_visible(const ChunkTable& ct, const WalkCfg& g, const KvWalk& w) {
    if (!g.causal || w.c < g.r) return true;
    if (w.c > g.r) return false;
    return ct.off[w.c] + (w.t - w.t0) * kTile <= g.q_last;
}
__device__ __forceinline__ void kv_adv(const ChunkTable& ct, const WalkCfg& g, KvWalk& w) {
    if (g.causal && w.c > g.r) w.t = w.t1 - 1;  // the whole chunk is masked
    if (++w.t == w.t1 && ++w.it < g.P) kv_set_chunk(ct, g, w);
}
__device__ __forceinline__ void kv_first(const ChunkTable& ct, const WalkCfg& g, KvWalk& w) {
    w.it = 0;
    kv_set_chunk(ct, g, w);
    while (w.it < g.P && !kv_visible(ct, g, w)) kv_adv(ct, g, w);
}
__device__ __forceinline__ void kv_next(const ChunkTable& ct, const WalkCfg& g, KvWalk& w) {
    do kv_adv(ct, g, w);
    while (w.it < g.P && !kv_visible(ct, g, w));
}
// The visited tile is the last one the walk visits in its chunk (the end of
// that chunk's partial): the chunk's last tile, or with causal masking in the
// query chunk itself the last tile starting at or before the CTA's last row.
__device__ __forceinline__ bool kv_chunk_last(const ChunkTable& ct, const WalkCfg& g, const KvWalk& w) {
    int last = w.t1 - 1;
    if (g.causal && w.c == g.r) last = min(last, w.t0 + ((g.q_last - ct.off[w.c]) >> 7));
    return w.t == last;
}
// Number of KV tiles the walk visits.
__device__ __forceinline__ int kv_count(const ChunkTable& ct, const WalkCfg& g) {
    if (!g.causal) return ct.ntiles;
    return ct.tile_off[g.r] + ((g.q_last - ct.off[g.r]) >> 7) + 1;
}

// ----------------------------------------------------------- backward walk
// Query tiles visited by one KV tile (chunk c, first row kv_start): for each
// query head of the GQA group, ring iterations it = 0..P-1 (query chunk
// (c + it) mod P) and that chunk's 128-row tiles.
struct QTileIter {
    int h, t, it, r;
};
struct QWalk {
    const ChunkTable* ct;
    int c, causal, kv_start, h_end;
    __device__ __forceinline__ int first_row(const QTileIter& q) const {
        return ct->off[q.r] + (q.t - ct->tile_off[q.r]) * kTile;
    }
    __device__ __forceinline__ bool visible(const QTileIter& q) const {
        if (!causal || q.r > c) return true;
        if (q.r < c) return false;
        const int qs = first_row(q);
        return qs + min(kTile, ct->off[q.r + 1] - qs) - 1 >= kv_start;
    }
    __device__ __forceinline__ void adv(QTileIter& q) const {
        if (causal && q.r < c) q.t = ct->tile_off[q.r + 1] - 1;  // the whole chunk is masked
        ++q.t;
        if (q.t == ct->tile_off[q.r + 1]) {
            if (++q.it == ct->P) {
                q.it = 0;
                ++q.h;
            }
            q.r = (c + q.it) % ct->P;
            q.t = ct->tile_off[q.r];
        }
    }
    __device__ __forceinline__ void next(QTileIter& q) const {
        do adv(q);
        while (q.h < h_end && !visible(q));
    }
    __device__ __forceinline__ QTileIter first(int h0) const {
        QTileIter q;
        q.h = h0;
        q.it = 0;
        q.r = c;
        q.t = ct->tile_off[c];
        while (!visible(q)) adv(q);
        return q;
    }
    // number of query tiles visited, over G query heads
    __device__ __forceinline__ int count(int G) const {
        if (!causal) return G * ct->ntiles;
        int per = ct->tile_off[c + 1] - ct->tile_off[c] - ((kv_start - ct->off[c]) >> 7);
        for (int r2 = c + 1; r2 < ct->P; ++r2) per += ct->tile_off[r2 + 1] - ct->tile_off[r2];
        return G * per;
    }
};

}  // namespace ctxattn
