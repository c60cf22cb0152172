// Two-SM variant of the persistent GEMM engine (gemm_engine.cuh): a cluster of two
// CTAs shares each 256-row output tile through tcgen05.mma.cta_group::2.
//
//   CTA rank 0 (leader) and rank 1 each hold, per 64-wide K step, their own 128 rows
//   of A (16 KB) and their half of the N columns of B (up to 16 KB) at identical
//   shared-memory offsets; the leader's single MMA thread multiplies the 256 x N x 64
//   step, and each CTA receives its 128 accumulator rows (all N columns) in its own
//   tensor memory.  Per SM that is 32 KB of operands per 64-wide K step for a
//   128 x 256 share of the output (48 KB in the one-SM engine), six pipeline stages
//   instead of four, and still two accumulator buffers, so the epilogue of one tile
//   overlaps the main loop of the next.
//
//   warp 0 (one lane, both CTAs): TMA producer of this CTA's operands; every load
//       completes on the LEADER's full barrier, which the leader arms with the bytes
//       of both CTAs
//   warp 1 (one lane, leader only): MMA issuer; commits release the stage in both
//       CTAs and publish the accumulator to both CTAs' epilogues; warp 1 of each
//       CTA allocates (jointly) the pair's tensor memory
//   warps 2..: P::kEpiWarps epilogue warps per CTA, each CTA on its own 128 rows;
//       they report a drained accumulator on the leader's tempty barrier
//
// Tiles are 256 rows (two plan tiles of 128 rows of one group, or a group's odd last
// tile alone: then the rank-1 CTA loads no A rows and its epilogue stores nothing)
// by up to 256 columns.  A problem type P for this engine provides:
//
//   static constexpr bool kAmn, kBmn;  static constexpr int kEpiWarps;
//   int* err;
//   int      num_tiles() const;                    256-row tiles
//   int4     tile_fetch(int t) const;              the tile's plan entry (global loads only)
//   TileInfo tile_at(int t, int4 w) const;         decode (no memory access): m0 = first row of
//                                                  the 256-row tile, mh = halves
//   TileInfo tile(int t) const;                    tile_at(t, tile_fetch(t))
//   static constexpr bool kIssuerNeedsTile;        false: nk and the MMA steps do not depend on
//                                                  the entry, and the issuer decodes with zeros
//   void     prefetch() const;
//   uint32_t tx_bytes(const TileInfo&, int ks) const;   bytes BOTH CTAs load at step ks
//   void     load_pair(const TileInfo&, int ks, int rank, uint8_t* sA, uint8_t* sB, uint32_t cbar) const;
//   MmaStep  mma_step(const TileInfo&, int ks) const;   n = the full N of the pair MMA
//   void     epilogue(const TileInfo&, int row, uint32_t taddr, int c0, int cs, uint32_t* stg) const;
//            (called with m0 = this CTA's first row, row in [0, 128))
#pragma once
#include "gemm_engine.cuh"

namespace moelora {

constexpr int kPairAStage = 128 * 128;  // this CTA's 128 rows x 64 bf16
constexpr int kPairBStage = 128 * 128;  // this CTA's half of B: up to 128 rows x 64 bf16
constexpr int kPairStage = kPairAStage + kPairBStage;
constexpr int kPairStages = 6;
static_assert(kPairStages * kPairStage <= 192 * 1024, "pair pipeline exceeds shared memory budget");

// P::kBmnCompact: an MN-major B half sits as 8-K-row groups of its two 64-column chunks
// (chunk stride 1 KB, group stride 2 KB) instead of whole chunks 8 KB apart.  With whole
// chunks the pair MMA reads MN-major B slowly (plain 8192^3 GEMM: 1,197-1,529 against
// 1,644-1,706 TFLOP/s K-major); with the groups at the K-major rate (1,627-1,678).
template <class P, class = void>
struct BmnCompactOf : std::false_type {};
template <class P>
struct BmnCompactOf<P, std::void_t<decltype(P::kBmnCompact)>> : std::integral_constant<bool, P::kBmnCompact> {};

template <class P>
__global__ void __launch_bounds__(64 + 32 * P::kEpiWarps, 1) gemm_pair_kernel(const __grid_constant__ P p) {
  static_assert(P::kEpiWarps == 4 || P::kEpiWarps == 8, "4 or 8 epilogue warps");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kPairStages * kPairStage + kStgBytes);
  uint64_t* empty = full + kPairStages;
  uint64_t* tfull = empty + kPairStages;
  uint64_t* tempty = tfull + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);
  uint32_t* stg_base = reinterpret_cast<uint32_t*>(smem + kPairStages * kPairStage);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
  int* err = p.err;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPairStages; ++s) {
      mbar_init(&full[s], 1);   // leader only: its own arrive.expect_tx + both CTAs' bytes
      mbar_init(&empty[s], 1);  // both: one multicast commit per use
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);                  // both: one multicast commit per tile
      mbar_init(&tempty[a], 2 * P::kEpiWarps);  // leader only: every epilogue warp of the pair
    }
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, 2 * kAccCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync_all();  // barriers initialised and tensor memory allocated in both CTAs
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int ntiles = p.num_tiles();

  if (warp == 0) {
    if (lane == 0) {
      p.prefetch();
      int s = 0;
      uint32_t ph = 0;
      bool ok = true;
      uint32_t issued = 0, last_ph = 0;  // leader: stages armed, and the parity of their last use
      // The next tile's plan entry is loaded at K step 2 of the current tile, when the
      // stage ring is already full, so no tile start waits on a global load.
      int4 w = pair < ntiles ? p.tile_fetch(pair) : make_int4(0, 0, 0, 0);
      for (int t = pair; t < ntiles && ok; t += npairs) {
        const TileInfo ti = p.tile_at(t, w);
        const bool more = t + npairs < ntiles;
        const int fks = ti.nk > 2 ? 2 : ti.nk - 1;
        if (ti.nk == 0 && more) w = p.tile_fetch(t + npairs);
        for (int ks = 0; ks < ti.nk; ++ks) {
          if (!mbar_wait(&empty[s], ph ^ 1u, err)) {
            ok = false;
            break;
          }
          if (rank == 0) {
            mbar_arrive_expect_tx(&full[s], p.tx_bytes(ti, ks));
            issued |= 1u << s;
            last_ph = (last_ph & ~(1u << s)) | (ph << s);
          }
          uint8_t* sa = smem + s * kPairStage;
          p.load_pair(ti, ks, (int)rank, sa, sa + kPairAStage, mapa_shared(smem_u32(&full[s]), 0));
          if (ks == fks && more) w = p.tile_fetch(t + npairs);
          if (++s == kPairStages) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      // Only after a wait gave up can copies still be in flight here: the leader's
      // full barriers count both CTAs' bytes, so the leader waits (bounded) for each
      // armed stage; the closing cluster barrier keeps the peer resident meanwhile.
      if (rank == 0)
        for (int i = 0; i < kPairStages; ++i)
          if (issued & (1u << i)) mbar_wait(&full[i], (last_ph >> i) & 1u, err, 100000000ull);
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      int s = 0, acc = 0;
      uint32_t ph = 0, aph = 0;
      bool ok = true;
      int4 w = P::kIssuerNeedsTile && pair < ntiles ? p.tile_fetch(pair) : make_int4(0, 0, 0, 0);
      for (int t = pair; t < ntiles && ok; t += npairs) {
        const TileInfo ti = p.tile_at(t, w);
        const bool more = P::kIssuerNeedsTile && t + npairs < ntiles;
        const int fks = ti.nk > 2 ? 2 : ti.nk - 1;
        if (ti.nk == 0) {
          if (more) w = p.tile_fetch(t + npairs);
          continue;
        }
        if (!mbar_wait_cluster(&tempty[acc], aph ^ 1u, err)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + (uint32_t)(acc * kAccCols);
        for (int ks = 0; ks < ti.nk; ++ks) {
          if (!mbar_wait(&full[s], ph, err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const MmaStep st = p.mma_step(ti, ks);
          const uint32_t idesc = idesc_bf16_f32(256, st.n, P::kAmn, P::kBmn);
          const uint32_t sa = smem_u32(smem + s * kPairStage);
          const uint32_t sb = sa + kPairAStage + (uint32_t)st.b_off;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            const uint64_t ad = P::kAmn ? sw128_desc(sa + kk * 2048, 8192, 1024) : sw128_desc(sa + kk * 32, 16, 1024);
            const uint64_t bd = BmnCompactOf<P>::value ? sw128_desc(sb + kk * 4096, 1024, 2048)
                                : P::kBmn              ? sw128_desc(sb + kk * 2048, 8192, 1024)
                                                       : sw128_desc(sb + kk * 32, 16, 1024);
            mma_bf16_pair(d + (uint32_t)st.col, ad, bd, idesc, (st.first && kk == 0) ? 0u : 1u);
          }
          mma_commit_pair_both(&empty[s]);
          if (ks == fks && more) w = p.tile_fetch(t + npairs);
          if (++s == kPairStages) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit_pair_both(&tfull[acc]);
        if (++acc == 2) {
          acc = 0;
          aph ^= 1u;
        }
      }
    }
  } else {
    const int q = warp & 3;            // TMEM lane quarter this warp may access
    const int half = (warp - 2) >> 2;  // with 8 warps: which alternate 32-column chunks
    const int row = q * 32 + lane;
    const int c0 = 32 * half;
    const int cs = 32 * (P::kEpiWarps / 4);
    int acc = 0;
    uint32_t aph = 0;
    for (int t = pair; t < ntiles; t += npairs) {
      TileInfo ti = p.tile(t);
      if (ti.nk == 0) continue;
      const bool ok = __all_sync(0xffffffffu, mbar_wait(&tfull[acc], aph, err));
      if (!ok) break;
      tc_fence_after();
      if ((int)rank < ti.mh) {
        ti.m0 += (int)rank * 128;
        p.epilogue(ti, row, tmem_base + (uint32_t)(acc * kAccCols) + ((uint32_t)(q * 32) << 16), c0, cs,
                   stg_base + (warp - 2) * kStgWordsPerWarp);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&tempty[acc]), 0));
      if (++acc == 2) {
        acc = 0;
        aph ^= 1u;
      }
    }
    if (lane == 0) bulk_wait_group<0>();  // epilogue TMA stores complete before exit
  }
  __syncthreads();
  tc_fence_before();
  cluster_sync_all();  // no CTA leaves while its peer may still signal or read it
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, 2 * kAccCols);
  }
}

// Host launch: clusters of two CTAs, at most as many clusters as fit at once
// (one CTA per SM, within num_sms), never more than the problem's 256-row tiles.
template <class P>
cudaError_t launch_gemm_pair(const P& p, int max_tiles, int num_sms, cudaStream_t stream, int slot) {
  static int max_clusters = 0;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(64 + 32 * P::kEpiWarps);
  cfg.dynamicSmemBytes = kGemmSmemBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (max_clusters == 0) {
    cudaError_t e = cudaFuncSetAttribute(gemm_pair_kernel<P>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kGemmSmemBytes);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    cfg.gridDim = dim3(sms & ~1);
    int n = 0;
    if ((e = cudaOccupancyMaxActiveClusters(&n, gemm_pair_kernel<P>, &cfg)) != cudaSuccess) return e;
    if (n < 1) return cudaErrorInvalidConfiguration;
    max_clusters = n;
  }
  if (max_tiles <= 0) return cudaSuccess;
  int clusters = max_tiles < max_clusters ? max_tiles : max_clusters;
  if (clusters > num_sms / 2) clusters = num_sms / 2 > 0 ? num_sms / 2 : 1;
  cfg.gridDim = dim3(2 * clusters);
  prof_begin(slot, stream);
  cudaError_t e = cudaLaunchKernelEx(&cfg, gemm_pair_kernel<P>, p);
  prof_end(slot, stream);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace moelora
