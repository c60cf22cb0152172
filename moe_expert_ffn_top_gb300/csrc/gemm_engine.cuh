// Persistent, warp-specialised BF16 GEMM engine for sm_103a.
//
//   warp 0 (one lane)  : TMA producer, fills a kStages-deep ring of (A, B) tiles
//   warp 1 (one lane)  : tcgen05.mma issuer; also owns the TMEM allocation
//   warps 2..          : P::kEpiWarps epilogue warps (4 or 8); warp w may read TMEM
//                        lane quarter w%4 (one accumulator row per thread); with 8
//                        warps, warps w and w+4 take alternate 32-column chunks
//
// Accumulators are 128 x 256 fp32 in tensor memory, double buffered (512
// columns), so the epilogue of tile i overlaps the main loop of tile i+1.
// Every output tile is 128 rows (M) by up to 256 columns (N); the K loop runs in
// steps of 64.  What a tile means -- its rows, which operand tiles each K step
// loads, and what the epilogue does with the accumulator -- is supplied by a
// problem type P (see gemm_problems.cuh):
//
//   static constexpr bool kAmn, kBmn;      operand majorness (true = MN-major)
//   static constexpr int  kEpiWarps;       4 or 8 epilogue warps
//   int*  err;                              device error word
//   int      num_tiles() const;             read from device plan data
//   TileInfo tile(int t) const;
//   void     prefetch() const;              tensor-map prefetch
//   void     load(const TileInfo&, int ks, uint8_t* sA, uint8_t* sB, uint64_t* bar) const;
//   MmaStep  mma_step(const TileInfo&, int ks) const;
//   void     epilogue(const TileInfo&, int row, uint32_t tmem_lane_addr, int c0, int cs,
//                     uint32_t* stg) const;    stg: the warp's staging buffer
//   void     epilogue_empty(const TileInfo&, int row, int c0, int cs) const;   (tiles with nk == 0)
//   static constexpr bool kWide;           256-row tiles (see EngineShape)
// An epilogue warp handles the 32-column chunks c = c0, c0 + cs, ... of its row.
//
// Operand tiles in shared memory use the 128-byte swizzle written by TMA:
//   A K-major : 128 rows x 128 B                         (one 16 KB box)
//   A MN-major: two boxes of 64 K-rows x 64 M, 8 KB apart
//   B K-major : N rows x 128 B
//   B MN-major: N/64 boxes of 64 K-rows x 64 N, 8 KB apart
#pragma once
#include "common.cuh"
#include "prof.h"
#include "sm100_ptx.cuh"

namespace moelora {

constexpr int kBK = 64;
constexpr int kBStageBytes = 256 * 128;  // 32 KB: up to 256 rows x 64 bf16
constexpr int kAccCols = 256;
// Per epilogue warp: a 4 KB staging buffer (1024-byte aligned) used to turn
// row-per-thread accumulator data into coalesced row segments: bf16 rows at a pitch
// of 17 words, fp32 rows at 32 words with the column index XORed by the row (both
// conflict-free), or two 2 KB tiles of 32 x 32 bf16 for TMA stores.
constexpr int kStgPitch = 17;
constexpr int kStgWordsPerWarp = 1024;
constexpr int kStgBytes = 8 * kStgWordsPerWarp * 4;
// pipeline stages (at most 192 KB), staging, barriers, and slack to align the base
constexpr int kGemmSmemBytes = 192 * 1024 + kStgBytes + 256 + 1024;

// Per-problem pipeline shape.  Narrow problems: 128-row tiles, 4 stages of
// (A 16 KB + B 32 KB), two TMEM accumulators (the epilogue of one tile overlaps the
// main loop of the next).  Wide problems (P::kWide): 256-row tiles as two M=128
// MMAs sharing each B tile, 3 stages of (A 32 KB + B 32 KB), one accumulator pair
// using all 512 TMEM columns -- a third fewer operand bytes per FLOP streamed into
// the SM, at the price of an epilogue that no longer overlaps the main loop.
template <class P>
struct EngineShape {
  static constexpr bool kWide = P::kWide;
  static constexpr int kAStage = kWide ? 2 * 128 * 128 : 128 * 128;
  static constexpr int kStage = kAStage + kBStageBytes;
  static constexpr int kStages = kWide ? 3 : 4;
  static constexpr int kAccBufs = kWide ? 1 : 2;
  static_assert(kStages * kStage <= 192 * 1024, "pipeline exceeds shared memory budget");
};

struct TileInfo {
  int m0;    // first output row
  int n0;    // first output column
  int g;     // plan group or adapter index
  int sub;   // problem-specific tile variant
  int nk;    // number of 64-wide K steps (0 = empty tile)
  int k0;    // first K index for K-grouped problems
  int mend;  // one past the last valid output row
  int mh;    // wide problems: 128-row halves present (1 or 2)
};

struct MmaStep {
  int n;      // MMA N (multiple of 16, <= 256)
  int col;    // TMEM column of D inside the accumulator
  int b_off;  // byte offset of B inside the B stage
  int first;  // 1: the step's first MMA overwrites D instead of accumulating
};

template <class P>
__global__ void __launch_bounds__(64 + 32 * P::kEpiWarps, 1) gemm_kernel(const __grid_constant__ P p) {
  using S = EngineShape<P>;
  static_assert(P::kEpiWarps == 4 || P::kEpiWarps == 8, "4 or 8 epilogue warps");
  static_assert(!P::kWide || (P::kEpiWarps == 8 && !P::kAmn), "wide tiles: 8 epilogue warps, K-major A");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S::kStages * S::kStage + kStgBytes);
  uint64_t* empty = full + S::kStages;
  uint64_t* tfull = empty + S::kStages;
  uint64_t* tempty = tfull + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);
  uint32_t* stg_base = reinterpret_cast<uint32_t*>(smem + S::kStages * S::kStage);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int* err = p.err;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], P::kEpiWarps);
    }
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 2 * kAccCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int ntiles = p.num_tiles();

  if (warp == 0) {
    if (lane == 0) {
      p.prefetch();
      int s = 0;
      uint32_t ph = 0;
      bool ok = true;
      uint32_t issued = 0;   // bit s: stage s has received a load
      uint32_t last_ph = 0;  // bit s: phase parity of stage s's last load
      for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
        const TileInfo ti = p.tile(t);
        for (int ks = 0; ks < ti.nk; ++ks) {
          if (!mbar_wait(&empty[s], ph ^ 1u, err)) {
            ok = false;
            break;
          }
          uint8_t* sa = smem + s * S::kStage;
          p.load(ti, ks, sa, sa + S::kAStage, &full[s]);
          issued |= 1u << s;
          last_ph = (last_ph & ~(1u << s)) | (ph << s);
          if (++s == S::kStages) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      // No TMA copy may still be landing in shared memory when the CTA exits
      // (matters only if a wait above gave up): wait, bounded, for each stage's
      // last load to complete.
      for (int i = 0; i < S::kStages; ++i)
        if (issued & (1u << i)) mbar_wait(&full[i], (last_ph >> i) & 1u, err, 100000000ull);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      int s = 0, acc = 0;
      uint32_t ph = 0, aph = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
        const TileInfo ti = p.tile(t);
        if (ti.nk == 0) continue;
        if (!mbar_wait(&tempty[acc], aph ^ 1u, err)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + (uint32_t)(S::kWide ? 0 : acc * kAccCols);
        for (int ks = 0; ks < ti.nk; ++ks) {
          if (!mbar_wait(&full[s], ph, err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const MmaStep st = p.mma_step(ti, ks);
          const uint32_t idesc = idesc_bf16_f32(128, st.n, P::kAmn, P::kBmn);
          const uint32_t sa = smem_u32(smem + s * S::kStage);
          const uint32_t sb = sa + S::kAStage + (uint32_t)st.b_off;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            const uint64_t ad = P::kAmn ? sw128_desc(sa + kk * 2048, 8192, 1024) : sw128_desc(sa + kk * 32, 16, 1024);
            const uint64_t bd = P::kBmn ? sw128_desc(sb + kk * 2048, 8192, 1024) : sw128_desc(sb + kk * 32, 16, 1024);
            const uint32_t accum = (st.first && kk == 0) ? 0u : 1u;
            mma_bf16(d + (uint32_t)st.col, ad, bd, idesc, accum);
            if (S::kWide && ti.mh == 2)  // rows 128..255 of the tile: second A half, same B
              mma_bf16(d + kAccCols + (uint32_t)st.col, sw128_desc(sa + 128 * 128 + kk * 32, 16, 1024), bd, idesc,
                       accum);
          }
          mma_commit(&empty[s]);
          if (++s == S::kStages) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit(&tfull[acc]);
        if (++acc == S::kAccBufs) {
          acc = 0;
          aph ^= 1u;
        }
      }
    }
  } else {
    const int q = warp & 3;            // TMEM lane quarter this warp may access
    const int half = (warp - 2) >> 2;  // 0 for warps 2..5, 1 for warps 6..9
    // Narrow: warps sharing a quarter split the columns.  Wide: half selects the
    // 128-row half of the tile (its own accumulator), all columns.
    const int row = (S::kWide ? half * 128 : 0) + q * 32 + lane;
    const int c0 = S::kWide ? 0 : 32 * half;
    const int cs = S::kWide ? 32 : 32 * (P::kEpiWarps / 4);
    int acc = 0;
    uint32_t aph = 0;
    for (int t = blockIdx.x; t < ntiles; t += gridDim.x) {
      const TileInfo ti = p.tile(t);
      if (ti.nk == 0) {
        p.epilogue_empty(ti, row, c0, cs);
        continue;
      }
      const bool ok = __all_sync(0xffffffffu, mbar_wait(&tfull[acc], aph, err));
      if (!ok) break;
      tc_fence_after();
      if (!S::kWide || half < ti.mh) {
        const uint32_t col = (uint32_t)(S::kWide ? half * kAccCols : acc * kAccCols);
        p.epilogue(ti, row, tmem_base + col + ((uint32_t)(q * 32) << 16), c0, cs,
                   stg_base + (warp - 2) * kStgWordsPerWarp);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[acc]);
      if (++acc == S::kAccBufs) {
        acc = 0;
        aph ^= 1u;
      }
    }
    if (lane == 0) bulk_wait_group<0>();  // epilogue TMA stores complete before exit
  }
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, 2 * kAccCols);
  }
}

// Host launch: one CTA per SM (or fewer if the problem has fewer tiles).
template <class P>
cudaError_t launch_gemm(const P& p, int max_tiles, int num_sms, cudaStream_t stream, int slot) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(gemm_kernel<P>, cudaFuncAttributeMaxDynamicSharedMemorySize, kGemmSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  if (max_tiles <= 0) return cudaSuccess;
  const int grid = max_tiles < num_sms ? max_tiles : num_sms;
  prof_begin(slot, stream);
  gemm_kernel<P><<<grid, 64 + 32 * P::kEpiWarps, kGemmSmemBytes, stream>>>(p);
  prof_end(slot, stream);
  return cudaGetLastError();
}

}  // namespace moelora
