// Routing plan on the device: a stable counting sort of the live routes by
// (expert, adapter, token, slot), each (expert, adapter) group padded to a
// multiple of 128 rows (plan slot q = e*A + a; one adapter: q = e).  Deterministic: the row of every route is a function of
// the ids alone (the pages' atomic dispatch reordered rows between replays,
// "feat(mega): add fused shared side-LoRA kernels", review thread on
// repeatability; this plan does not).
//
// Routes are cut into chunks of kPlanChunk (flattened t*k+j order), one warp each:
//   1. plan_count   : per-chunk group histogram -> chunk_base[g][c]
//   2. plan_scan    : per-group sums and prefix over chunks, padded group offsets
//   3. plan_scatter : in-order ranking inside each chunk (warp match), rows out
//   4. plan_finish  : padding rows -> -1, tile -> group table, adapter tables
//   5. plan_wide    : 256-row tiles (pairs of a group's 128-row tiles)
#include <cuda_runtime.h>

#include "common.cuh"
#include "launch.h"
#include "prof.h"

namespace moelora {

__device__ __forceinline__ int group_of(const int* ids, int64_t rt, int k, int E, const AdapterTable& at,
                                        int* err) {
  const int e = ids[rt];
  if (e < -1 || e >= E) {
    atomicOr(err, MOE_LORA_DEV_BAD_ID);
    return -1;
  }
  if (e < 0) return -1;
  const int64_t t = rt / k;
  int a = 0;
  while (a + 1 < at.n && t >= at.tok_off[a + 1]) ++a;
  return e * at.n + a;
}

// one warp per chunk; smem histogram of G counters
__global__ void plan_count(const int* __restrict__ ids, int64_t TK, int k, int E, int G, AdapterTable at,
                           int* __restrict__ chunk_base, int nchunks, int* err) {
  extern __shared__ int hist[];
  const int c = blockIdx.x;
  for (int g = threadIdx.x; g < G; g += blockDim.x) hist[g] = 0;
  __syncwarp();
  const int64_t r0 = (int64_t)c * kPlanChunk;
  const int64_t r1 = r0 + kPlanChunk < TK ? r0 + kPlanChunk : TK;
  for (int64_t rt = r0 + threadIdx.x; rt < r1; rt += 32) {
    const int g = group_of(ids, rt, k, E, at, err);
    if (g >= 0) atomicAdd(&hist[g], 1);
  }
  __syncwarp();
  for (int g = threadIdx.x; g < G; g += blockDim.x) chunk_base[(int64_t)g * nchunks + c] = hist[g];
}

// one block: per-group totals and exclusive prefix over chunks; group offsets.
__global__ void plan_scan(int* __restrict__ chunk_base, int nchunks, int G, int* __restrict__ counts,
                          int* __restrict__ offsets) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
  for (int g = warp; g < G; g += nwarps) {
    int* row = chunk_base + (int64_t)g * nchunks;
    int carry = 0;
    for (int c0 = 0; c0 < nchunks; c0 += 32) {
      const int c = c0 + lane;
      const int v = c < nchunks ? row[c] : 0;
      int incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
      }
      if (c < nchunks) row[c] = carry + incl - v;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) counts[g] = carry;
  }
  __syncthreads();
  // exclusive scan of padded counts over groups (warp 0)
  if (warp == 0) {
    int carry = 0;
    for (int g0 = 0; g0 < G; g0 += 32) {
      const int g = g0 + lane;
      const int v = g < G ? (counts[g] + kBlockM - 1) / kBlockM * kBlockM : 0;
      int incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
      }
      if (g < G) offsets[g] = carry + incl - v;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) offsets[G] = carry;
  }
}

// one warp per chunk: stable in-order ranks with __match_any_sync.
__global__ void plan_scatter(const int* __restrict__ ids, int64_t TK, int k, int E, int G, AdapterTable at,
                             const int* __restrict__ chunk_base, const int* __restrict__ offsets, int nchunks,
                             int* __restrict__ row_of_route, int* __restrict__ route_of_row, int* err) {
  extern __shared__ int cursor[];
  const int c = blockIdx.x, lane = threadIdx.x;
  for (int g = lane; g < G; g += 32) cursor[g] = offsets[g] + chunk_base[(int64_t)g * nchunks + c];
  __syncwarp();
  const int64_t r0 = (int64_t)c * kPlanChunk;
  const int64_t r1 = r0 + kPlanChunk < TK ? r0 + kPlanChunk : TK;
  for (int64_t b = r0; b < r1; b += 32) {
    const int64_t rt = b + lane;
    const bool in = rt < r1;
    int g = -1;
    if (in) {
      const int e = ids[rt];
      if (e >= 0 && e < E) {
        const int64_t t = rt / k;
        int a = 0;
        while (a + 1 < at.n && t >= at.tok_off[a + 1]) ++a;
        g = e * at.n + a;
      }
    }
    const unsigned peers = __match_any_sync(0xffffffffu, g);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    int row = -1;
    if (g >= 0) row = cursor[g] + rank;
    __syncwarp();
    if (g >= 0 && (peers >> lane) == 1u) cursor[g] += __popc(peers);  // highest peer lane advances
    __syncwarp();
    if (in) {
      row_of_route[rt] = row;
      if (row >= 0) route_of_row[row] = (int)rt;
    }
  }
  (void)err;
}

// padding rows -> -1; tile -> group; adapter tables into the workspace.
__global__ void plan_finish(int G, int E, const int* __restrict__ counts, const int* __restrict__ offsets,
                            int* __restrict__ route_of_row, int* __restrict__ tile_group,
                            int2* __restrict__ tile_span, AdapterTable at, int* __restrict__ tok_off,
                            int* __restrict__ tok_tile) {
  for (int g = blockIdx.x; g < G; g += gridDim.x) {
    const int beg = offsets[g], end = offsets[g + 1], live = beg + counts[g];
    for (int p = live + threadIdx.x; p < end; p += blockDim.x) route_of_row[p] = -1;
    const int2 span = make_int2(beg / kBlockM, (end - beg) / kBlockM);
    const int wg = group_weight_index(g, at.n, E);
    for (int m = beg / kBlockM + threadIdx.x; m < end / kBlockM; m += blockDim.x) {
      tile_group[m] = wg;
      tile_span[m] = span;
    }
  }
  if (blockIdx.x == 0) {
    for (int a = threadIdx.x; a <= at.n; a += blockDim.x) {
      tok_off[a] = at.tok_off[a];
      tok_tile[a] = at.tok_tile[a];
    }
  }
}

__global__ void plan_wide(int G, int A, int E, const int* __restrict__ offsets, int* __restrict__ wtile_off,
                          int4* __restrict__ wtile) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == 0) {
    int carry = 0;
    for (int g0 = 0; g0 < G; g0 += 32) {
      const int g = g0 + lane;
      const int v = g < G ? ((offsets[g + 1] - offsets[g]) / kBlockM + 1) / 2 : 0;
      int incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
      }
      if (g < G) wtile_off[g] = carry + incl - v;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) wtile_off[G] = carry;
  }
  __syncthreads();
  for (int g = threadIdx.x; g < G; g += blockDim.x) {
    const int m = offsets[g] / kBlockM, n = (offsets[g + 1] - offsets[g]) / kBlockM, base = wtile_off[g];
    const int nw = (n + 1) / 2;
    const int wg = group_weight_index(g, A, E);
    for (int j = 0; j < nw; ++j)
      wtile[base + j] = make_int4(((m + 2 * j) << 1) | (n - 2 * j >= 2 ? 1 : 0), wg, base, nw);
  }
}

cudaError_t launch_plan(const moe_lora_dims* d, const int32_t* ids, const AdapterTable& at, void* ws,
                        int* chunk_base, cudaStream_t stream) {
  const PlanLayout L = plan_layout(d);
  char* b = static_cast<char*>(ws);
  int* err = (int*)(b + L.err);
  int* counts = (int*)(b + L.counts);
  int* offsets = (int*)(b + L.offsets);
  int* row_of_route = (int*)(b + L.row_of_route);
  int* route_of_row = (int*)(b + L.route_of_row);
  int* tile_group = (int*)(b + L.tile_group);
  int2* tile_span = (int2*)(b + L.tile_span);
  int* tok_off = (int*)(b + L.tok_off);
  int* tok_tile = (int*)(b + L.tok_tile);
  int* wtile_off = (int*)(b + L.wtile_off);
  int4* wtile = (int4*)(b + L.wtile);
  const int G = d->A * d->E;
  const int64_t TK = d->T * d->k;
  const int nchunks = (int)plan_chunks(d);
  cudaError_t e = cudaMemsetAsync(err, 0, 16, stream);
  if (e != cudaSuccess) return e;
  const size_t hist_bytes = sizeof(int) * (size_t)G;
  if (hist_bytes > 48 * 1024) {
    e = cudaFuncSetAttribute(plan_count, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)hist_bytes);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(plan_scatter, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)hist_bytes);
    if (e != cudaSuccess) return e;
  }
  // plan_count rewrites every histogram entry that plan_scan and plan_scatter read,
  // so chunk_base may hold anything on entry (the fixed array of the no-allocation
  // entry point keeps the previous call's values); with no routes at all, the G
  // entries plan_scan reads are cleared instead.
  if (nchunks > 0) {
    prof_begin(K_PLAN_COUNT, stream);
    plan_count<<<nchunks, 32, hist_bytes, stream>>>(ids, TK, d->k, d->E, G, at, chunk_base, nchunks, err);
    prof_end(K_PLAN_COUNT, stream);
  } else {
    e = cudaMemsetAsync(chunk_base, 0, sizeof(int) * (size_t)G, stream);
    if (e != cudaSuccess) return e;
  }
  prof_begin(K_PLAN_SCAN, stream);
  plan_scan<<<1, 1024, 0, stream>>>(chunk_base, nchunks > 0 ? nchunks : 1, G, counts, offsets);
  prof_end(K_PLAN_SCAN, stream);
  if (nchunks > 0) {
    prof_begin(K_PLAN_SCATTER, stream);
    plan_scatter<<<nchunks, 32, hist_bytes, stream>>>(ids, TK, d->k, d->E, G, at, chunk_base, offsets, nchunks,
                                                      row_of_route, route_of_row, err);
    prof_end(K_PLAN_SCATTER, stream);
  }
  prof_begin(K_PLAN_FINISH, stream);
  plan_finish<<<G < 1024 ? G : 1024, 128, 0, stream>>>(G, d->E, counts, offsets, route_of_row, tile_group, tile_span,
                                                  at, tok_off, tok_tile);
  prof_end(K_PLAN_FINISH, stream);
  prof_begin(K_PLAN_WIDE, stream);
  plan_wide<<<1, 1024, 0, stream>>>(G, d->A, d->E, offsets, wtile_off, wtile);
  prof_end(K_PLAN_WIDE, stream);
  return cudaGetLastError();
}

}  // namespace moelora
