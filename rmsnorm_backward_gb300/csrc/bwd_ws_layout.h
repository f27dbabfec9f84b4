// bwd_ws_layout.h -- launch shape and shared-memory layout of the
// warp-specialised backward (bwd_ws.cuh), shared by the host planner and the
// kernel.
#pragma once

#include <stddef.h>

#include "gbn_launch.h"

namespace gbn {

// warps of each role: one producer, kSumWarps sum warps (whole rows, taken
// in turn), kOutWarps output warps (fixed column slices of every row)
constexpr int kSumWarps = 5;
constexpr int kOutWarps = 16;
constexpr int kWsThreads = 32 * (1 + kSumWarps + kOutWarps);

struct WsLayout {
    size_t gam, stat, cval, bars, total;
};

// ring [S][2 * rowb] | gamma [rowb] | saved rstd, mean [stat_rows] |
// per stage the row's {rstd, mean, c1, c2} [S] float4, issued-row count |
// mbarriers full, ready, consumed [S] and gamma's
__host__ __device__ inline WsLayout ws_layout(bool ln, size_t rowb, int S, int stat_rows) {
    WsLayout L;
    L.gam = (size_t)S * 2 * rowb;
    L.stat = L.gam + round_up(rowb, 16);
    L.cval = L.stat + round_up((size_t)stat_rows * 4 * (ln ? 2 : 1), 16);
    L.bars = L.cval + (size_t)S * 16 + 16;
    L.total = L.bars + ((size_t)3 * S + 1) * 8;
    return L;
}

// 16-byte vectors per output lane for a row of nvec vectors: the row must
// split into kOutWarps warps x 32 lanes x 1 or 2 vectors
__host__ __device__ inline bool ws_shape(int nvec, int *vec_per_lane) {
    if (nvec % (32 * kOutWarps) != 0) return false;
    const int vo = nvec / (32 * kOutWarps);
    if (vo != 1 && vo != 2) return false;
    *vec_per_lane = vo;
    return true;
}

}  // namespace gbn
