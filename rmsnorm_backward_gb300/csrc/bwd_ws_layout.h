// bwd_ws_layout.h -- launch shape and shared-memory layout of the
// warp-specialised backward (bwd_ws.cuh), shared by the host planner and the
// kernel.
#pragma once

#include <stddef.h>

#include "gbn_launch.h"

namespace gbn {

// warps of each role: one producer, kSumWarps sum warps (every row's sums
// split over all of them), kOutWarps output warps (fixed column slices)
constexpr int kSumWarps = 4;
constexpr int kOutWarps = 16;
constexpr int kWsThreads = 32 * (1 + kSumWarps + kOutWarps);

struct WsLayout {
    size_t gam, cval, xch, bars, total;
};

// ring [S][2 * rowb] | gamma [rowb] | per stage: the sum warps' partial sums
// [S][kSumWarps] float4 and the row's statistics [S] float4 |
// save-nothing LayerNorm exchange [2][kSumWarps] floats + abort flags [2] |
// mbarriers full, ready, consumed [S] and gamma's
__host__ __device__ inline WsLayout ws_layout(size_t rowb, int S) {
    WsLayout L;
    L.gam = (size_t)S * 2 * rowb;
    L.cval = L.gam + round_up(rowb, 16);
    L.xch = L.cval + (size_t)S * (kSumWarps + 1) * 16;
    L.bars = L.xch + round_up((size_t)2 * kSumWarps * 4 + 8, 16);
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
