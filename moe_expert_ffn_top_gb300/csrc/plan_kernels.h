// Kernels of the routing plan (plan.cu), shared by the plan entry points.
#pragma once
#include <cuda_runtime.h>

#include "launch.h"

namespace moelora {

__global__ void plan_count(const int* __restrict__ ids, int64_t TK, int k, int E, int G, AdapterTable at,
                           int* __restrict__ chunk_base, int nchunks, int* err);
__global__ void plan_scan(int* __restrict__ chunk_base, int nchunks, int G, int* __restrict__ counts,
                          int* __restrict__ offsets);
__global__ void plan_scatter(const int* __restrict__ ids, int64_t TK, int k, int E, int G, AdapterTable at,
                             const int* __restrict__ chunk_base, const int* __restrict__ offsets, int nchunks,
                             int* __restrict__ row_of_route, int* __restrict__ route_of_row, int* err);
__global__ void plan_finish(int G, int E, const int* __restrict__ counts, const int* __restrict__ offsets,
                            int* __restrict__ route_of_row, int* __restrict__ tile_group,
                            int2* __restrict__ tile_span, AdapterTable at, int* __restrict__ tok_off,
                            int* __restrict__ tok_tile);

// 256-row tiles: each group's 128-row tiles in pairs (a lone last tile is a half).
__global__ void plan_wide(int G, int A, int E, const int* __restrict__ offsets, int* __restrict__ wtile_off,
                          int4* __restrict__ wtile);

}  // namespace moelora
