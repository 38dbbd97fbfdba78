// Device-side helpers shared by the attention kernels: where a query tile
// lives, and the ring-order walk over KV tiles.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "common.h"

namespace st {

// A query tile: `nq` valid rows starting at buffer row `row0`, all inside one
// segment, so their natural positions are nat0, nat0+1, ...
struct QTile {
    int seg;
    int shard;
    int row0;
    int nq;
    int nat0;
};

__device__ __forceinline__ QTile locate_qtile(const SegTable& T, int tile, int tile_rows) {
    int s = 0;
    while (s + 1 < T.nseg && T.seg_tile[s + 1] <= tile) ++s;
    int r = 0;
    while (r + 1 < T.D && T.shard_seg[r + 1] <= s) ++r;
    QTile q;
    q.seg = s;
    q.shard = r;
    const int local = (tile - T.seg_tile[s]) * tile_rows;
    q.row0 = T.seg_buf[s] + local;
    q.nq = min(tile_rows, T.seg_buf[s + 1] - q.row0);
    q.nat0 = T.seg_nat[s] + local;
    return q;
}

// Classification of a (query tile, KV tile) pair.
enum TileKind { kSkip = 0, kFull = 1, kPartial = 2 };

// A partial pair on the causal diagonal: some of its keys come after the first
// query.  Its rows and keys have few partners, so P and dS there get the extra
// hi / lo precision; a pair that is partial only because its KV tile is ragged
// needs the key mask alone.
__device__ __forceinline__ bool on_diagonal(int causal, int nat_q0, int nat_k0, int nk) {
    return causal && nat_k0 + nk - 1 > nat_q0;
}

__device__ __forceinline__ int classify(int causal, int nat_q0, int nq, int nat_k0, int nk,
                                        int tile_cols) {
    if (causal && nat_k0 > nat_q0 + nq - 1) return kSkip;
    if (nk == tile_cols && (!causal || nat_k0 + tile_cols - 1 <= nat_q0)) return kFull;
    return kPartial;
}

// Walk the KV tiles met by a query tile of shard `r` in ring order: KV shards
// r, r-1, ..., r+1 (mod D) -- rank r receives its neighbour's K/V at every
// ring step -- and inside each shard its segments and `tile_cols`-row tiles in
// buffer order.  f(kv_shard, kv_row0, nk, nat_k0, last_tile_of_shard).
template <int kCols, typename F>
__device__ __forceinline__ void ring_walk(const SegTable& T, int r, F&& f) {
    for (int t = 0; t < T.D; ++t) {
        int j = r - t;
        if (j < 0) j += T.D;
        const int s_end = T.shard_seg[j + 1];
        for (int s = T.shard_seg[j]; s < s_end; ++s) {
            const int b0 = T.seg_buf[s], b1 = T.seg_buf[s + 1], nat = T.seg_nat[s];
            for (int kv0 = b0; kv0 < b1; kv0 += kCols) {
                const int nk = min(kCols, b1 - kv0);
                const bool last = (s + 1 == s_end) && (kv0 + kCols >= b1);
                f(j, kv0, nk, nat + (kv0 - b0), last);
            }
        }
    }
}

template <typename T>
__device__ __forceinline__ float to_f32(T x);
template <>
__device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

}  // namespace st
