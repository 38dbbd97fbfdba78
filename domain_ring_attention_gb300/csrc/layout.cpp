// Shard-layout descriptor (host code, no CUDA calls).
//
// Sharding shapes: ShardTensor summary, section 2 -- each rank holds a local
// chunk of its own length along the sharded axis; lengths may be uneven.
// Zigzag: TSP summary, section 2, attention layer -- the sequence is cut into
// 2D natural-order chunks and rank r holds chunks r and 2D-1-r.  With uneven
// shapes chunk r and chunk 2D-1-r both take L_r / 2 rows, which reduces to the
// equal split when every L_r is the same.
#include <climits>
#include <new>

#include "common.h"

extern "C" int st_layout_create(const int64_t* shard_lens, int D, int zigzag,
                                st_layout_t** out) {
    if (!shard_lens || !out) return ST_ERR_NULL;
    *out = nullptr;
    if (D < 1 || D > ST_MAX_SHARDS) return ST_ERR_INVALID_LAYOUT;
    if (zigzag != 0 && zigzag != 1) return ST_ERR_INVALID_ARG;
    int64_t S = 0;
    for (int r = 0; r < D; ++r) {
        const int64_t L = shard_lens[r];
        if (L < 1) return ST_ERR_INVALID_LAYOUT;
        if (zigzag && (L % 2) != 0) return ST_ERR_INVALID_LAYOUT;
        S += L;
        if (S >= (int64_t)INT_MAX) return ST_ERR_INVALID_LAYOUT;
    }
    st_layout* L = new (std::nothrow) st_layout();
    if (!L) return ST_ERR_INVALID_ARG;
    L->D = D;
    L->zigzag = zigzag;
    L->S = S;
    L->lens.assign(shard_lens, shard_lens + D);
    L->off.assign(D + 1, 0);
    for (int r = 0; r < D; ++r) L->off[r + 1] = L->off[r] + shard_lens[r];

    L->shard_seg.assign(D + 1, 0);
    if (!zigzag) {
        for (int r = 0; r < D; ++r) {
            L->shard_seg[r] = r;
            L->seg_buf.push_back(L->off[r]);
            L->seg_nat.push_back(L->off[r]);
        }
        L->shard_seg[D] = D;
    } else {
        // natural start of chunk c, with c_r = c_{2D-1-r} = L_r / 2
        std::vector<int64_t> chunk(2 * D), start(2 * D + 1, 0);
        for (int r = 0; r < D; ++r) chunk[r] = chunk[2 * D - 1 - r] = shard_lens[r] / 2;
        for (int c = 0; c < 2 * D; ++c) start[c + 1] = start[c] + chunk[c];
        for (int r = 0; r < D; ++r) {
            L->shard_seg[r] = 2 * r;
            L->seg_buf.push_back(L->off[r]);
            L->seg_nat.push_back(start[r]);
            L->seg_buf.push_back(L->off[r] + shard_lens[r] / 2);
            L->seg_nat.push_back(start[2 * D - 1 - r]);
        }
        L->shard_seg[D] = 2 * D;
    }
    L->seg_buf.push_back(S);
    *out = L;
    return ST_OK;
}

extern "C" int st_layout_destroy(st_layout_t* layout) {
    delete layout;
    return ST_OK;
}

extern "C" int st_layout_query(const st_layout_t* L, int64_t* S, int64_t* offsets,
                               int64_t* pos, int* D, int* zigzag) {
    if (!L) return ST_ERR_NULL;
    if (S) *S = L->S;
    if (D) *D = L->D;
    if (zigzag) *zigzag = L->zigzag;
    if (offsets)
        for (int r = 0; r <= L->D; ++r) offsets[r] = L->off[r];
    if (pos) {
        const int nseg = (int)L->seg_nat.size();
        for (int s = 0; s < nseg; ++s)
            for (int64_t t = L->seg_buf[s]; t < L->seg_buf[s + 1]; ++t)
                pos[t] = L->seg_nat[s] + (t - L->seg_buf[s]);
    }
    return ST_OK;
}

namespace st {

void fill_segtable(const st_layout& L, int tile_rows, SegTable* t) {
    const int nseg = (int)L.seg_nat.size();
    t->nseg = nseg;
    t->D = L.D;
    t->S = (int32_t)L.S;
    int tiles = 0;
    for (int s = 0; s < nseg; ++s) {
        t->seg_buf[s] = (int32_t)L.seg_buf[s];
        t->seg_nat[s] = (int32_t)L.seg_nat[s];
        t->seg_tile[s] = tiles;
        const int64_t len = L.seg_buf[s + 1] - L.seg_buf[s];
        tiles += (int)((len + tile_rows - 1) / tile_rows);
    }
    t->seg_buf[nseg] = (int32_t)L.S;
    t->seg_tile[nseg] = tiles;
    t->ntiles = tiles;
    for (int r = 0; r <= L.D; ++r) t->shard_seg[r] = L.shard_seg[r];
}

st_layout shard_layout(const st_layout& L, int r) {
    st_layout s;
    s.D = 1;
    s.zigzag = L.zigzag;
    s.S = L.lens[r];
    s.lens = {L.lens[r]};
    s.off = {0, L.lens[r]};
    for (int g = L.shard_seg[r]; g < L.shard_seg[r + 1]; ++g) {
        s.seg_buf.push_back(L.seg_buf[g] - L.off[r]);
        s.seg_nat.push_back(L.seg_nat[g]);
    }
    s.seg_buf.push_back(L.lens[r]);
    s.shard_seg = {0, L.shard_seg[r + 1] - L.shard_seg[r]};
    return s;
}

}  // namespace st
