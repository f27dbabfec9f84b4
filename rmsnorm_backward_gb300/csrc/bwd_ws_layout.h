// bwd_ws_layout.h -- launch shape and shared-memory layout of the
// warp-specialised backward (bwd_ws.cuh), shared by the host planner and the
// kernel.
#pragma once

#include <stddef.h>

#include "gbn_launch.h"

namespace gbn {

constexpr int kSumWarps = 5;

struct WsLayout {
    size_t gam, stat, cval, bars, total;
};

// ring [S][2 * rowb] | gamma [rowb] | rstd, mean [stat_rows] | sums [S][2], issued count |
// full, ready, consumed [S]
__host__ __device__ inline WsLayout ws_layout(bool ln, size_t rowb, int S, int stat_rows) {
    WsLayout L;
    L.gam = (size_t)S * 2 * rowb;
    L.stat = L.gam + round_up(rowb, 16);
    L.cval = L.stat + round_up((size_t)stat_rows * 4 * (ln ? 2 : 1), 16);
    L.bars = L.cval + round_up((size_t)S * 2 * 4 + 4, 16);
    L.total = L.bars + (size_t)3 * S * 8;
    return L;
}

// output warps and 16-byte vectors per lane for a row of nvec vectors
__host__ __device__ inline bool ws_shape(int nvec, int *out_warps, int *vec_per_lane) {
    if (nvec % 32 != 0) return false;
    const int lanes = nvec / 32;  // vectors per lane if one warp held the row
    const int no = lanes < 16 ? lanes : 16;
    if (lanes % no != 0) return false;
    const int vo = lanes / no;
    if (vo != 1 && vo != 2) return false;
    *out_warps = no;
    *vec_per_lane = vo;
    return true;
}

}  // namespace gbn
