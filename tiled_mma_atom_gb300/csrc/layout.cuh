// layout.cuh — crd2idx of a rank-2 (Shape, Stride) layout on the device:
// index = sum of coordinate x stride over the modes ("FlyDSL Kernel Authoring
// Skill", §2 "Layout System", "Coordinate Mapping"); the scalar coordinate of
// a nested mode (s0, s1):(d0, d1) splits first-sub-mode-fastest,
// c = c0 + s0 * c1 (the order of the page's idx2crd example).
#pragma once

#include "internal.h"

namespace tmg {

__device__ __forceinline__ int64_t mode_off(const DevLayout &L, int t, int64_t c)
{
    if (L.depth[t] == 1)
        return c * L.stride[t][0];
    const int64_t s0 = L.shape[t][0];
    return (c % s0) * L.stride[t][0] + (c / s0) * L.stride[t][1];
}

__device__ __forceinline__ int64_t crd2idx(const DevLayout &L, int64_t r, int64_t c)
{
    return mode_off(L, 0, r) + mode_off(L, 1, c);
}

// Elements the layout spans: one past its largest offset (strides are >= 0,
// checked by the host), the limit of the debug build's bounds checks.
__device__ __forceinline__ int64_t layout_extent(const DevLayout &L)
{
    int64_t e = 1;
    for (int t = 0; t < 2; ++t)
        for (int j = 0; j < L.depth[t]; ++j)
            e += (L.shape[t][j] - 1) * L.stride[t][j];
    return e;
}

}  // namespace tmg
