// The contractions of the routed MoE side-LoRA FFN, each expressed as a problem
// type for the GEMM engine (gemm_engine.cuh): which 128-row x N-column tiles exist,
// which TMA boxes every 64-wide K step loads, and the fused epilogue.
//
// Notation (row-major): x [T,H], Xp [P,H] routed rows (zero on padding rows),
// W1/W3 [E,I,H], W2 [E,H,I], A1/A3 [A,r,H], B1/B3 [A*E,I,r], A2 [A*E,r,I], B2 [A,H,r].
// A group (adapter a, expert e) has weight index g = a*E + e (TileInfo::g) and plan
// slot q = e*A + a; its rows are [offsets[q], offsets[q+1]), a multiple of 128 long.
//
// The side-LoRA contract ("feat(mega): add fused shared side-LoRA kernels",
// DeepGEMM PR #9, Summary): A1/A3 and B2 are shared, so the rank-r shrink
// x A^T and the expand Z B2^T run once per TOKEN; B1/B3/A2 are expert-local and
// run per routed row, fused into the expert GEMMs as extra K steps (B1/B3) or an
// extra N tile (A2).
#pragma once
#include "gemm_engine.cuh"


namespace moelora {

constexpr int kAStage128 = 128 * 128;  // bytes of one 128-row x 64 bf16 operand tile

// MN-major weight tiles of the dgrads (256 columns = four 64 x 64 boxes, 8 KB apart):
// one 4D copy over the weight seen as 64-column chunks (tmap_mn4) instead of four 3D
// copies -- the producer's TMA issue is what held the W2 dgrad (in-kernel counters:
// 69% of the kernel issuing copies, the MMA waiting for operands 32%).
constexpr bool kMnChunkCopy = true;

__device__ __forceinline__ int adapter_of_tile(const PlanView& pl, int t) {
  int a = 0;
  while (a + 1 < pl.A && t >= pl.tok_tile[a + 1]) ++a;
  return a;
}

// 256-row tile of an M-grouped problem from its plan entry w: rows
// [m0, m0 + 128*mh) of the group with weight index w.y (mh = 2, or 1 for a group's
// odd last tile).
__device__ __forceinline__ void wide_tile_from(int4 w, TileInfo& ti) {
  const int mt = w.x >> 1;
  ti.mh = (w.x & 1) + 1;
  ti.m0 = mt * 128;
  ti.mend = ti.m0 + 128 * ti.mh;
  ti.g = w.y;
  ti.k0 = 0;
}

// 128-row tile t of an M-grouped problem with ntn column tiles (row-tile-major).
__device__ __forceinline__ void narrow_tile(const PlanView& pl, int t, int ntn, TileInfo& ti) {
  const int mt = t / ntn;
  ti.mh = 1;
  ti.m0 = mt * 128;
  ti.mend = ti.m0 + 128;
  ti.g = pl.tile_group[mt];
  ti.k0 = 0;
}

// Column-tile-major order inside row chunks of each group: the base expert GEMMs walk
// a chunk of up to kChunkRows of a group's rows for one block of weight columns, then
// the next block, then the next chunk.  The CTAs running at the same time then share
// a few weight blocks (read once from DRAM) and one chunk of routed rows (16 MB at
// H = 4096, held in L2 across the column blocks); a group of up to kChunkRows rows --
// the usual case -- is a single chunk.  A group's tiles are the contiguous range
// [first*ntn, (first+count)*ntn) of tile indices, so t / ntn names a row tile of the
// right group.
constexpr int kChunkRows = 2048;

// Row tile (offset from the group's first) and column tile of the group's tile u, for
// a group of `count` row tiles cut into chunks of `chunk` row tiles.
__device__ __forceinline__ void chunked_order(int u, int count, int chunk, int ntn, int& mt, int& nt) {
  const int c = u / (chunk * ntn);
  const int v = u - c * chunk * ntn;
  const int cs = count - c * chunk < chunk ? count - c * chunk : chunk;
  mt = c * chunk + v % cs;
  nt = v / cs;
}

// 128-row tiles: the plan entry of tile t (loads only: group, first row tile and
// row-tile count of the group) ...
__device__ __forceinline__ int4 nmajor_narrow_fetch(const PlanView& pl, int t, int ntn) {
  const int l = t / ntn;
  const int2 sp = pl.tile_span[l];
  return make_int4(pl.tile_group[l], sp.x, sp.y, 0);
}
// ... and its decode (no memory access); returns the column tile.
__device__ __forceinline__ int nmajor_narrow_decode(int4 e, int t, int ntn, TileInfo& ti) {
  int mt, nt;
  chunked_order(t - e.y * ntn, e.z, kChunkRows / 128, ntn, mt, nt);
  ti.g = e.x;
  ti.m0 = (e.y + mt) * 128;
  ti.mend = ti.m0 + 128;
  ti.mh = 1;
  ti.k0 = 0;
  return nt;
}
// 256-row tiles: the entry of tile t (two dependent loads: any 256-row tile of the
// group gives the group's first tile and count, then the tile itself; z = column tile).
__device__ __forceinline__ int4 nmajor_wide_fetch(const PlanView& pl, int t, int ntn) {
  const int4 a = pl.wtile[t / ntn];
  int mt, nt;
  chunked_order(t - a.z * ntn, a.w, kChunkRows / 256, ntn, mt, nt);
  const int4 w = pl.wtile[a.z + mt];
  return make_int4(w.x, w.y, nt, 0);
}
// Decode of a 256-row tile entry (x, y as in the plan, z = column tile); returns the column tile.
__device__ __forceinline__ int wide_entry_decode(int4 e, TileInfo& ti) {
  wide_tile_from(e, ti);
  return e.z;
}

// A-operand rows of a wide tile: one 128-row box per half present.
__device__ __forceinline__ void load_a_wide(const TileInfo& ti, uint8_t* sa, const CUtensorMap* m, uint64_t* bar,
                                            int kx) {
  tma_load_2d(sa, m, bar, kx, ti.m0);
  if (ti.mh == 2) tma_load_2d(sa + kAStage128, m, bar, kx, ti.m0 + 128);
}

// Gated activations: ACT 0 = silu (SwiGLU), 1 = exact erf GELU (GeGLU); the
// clamp c > 0 limits gate and up pre-activations to [-c, c] (0 = no clamp).
// silu runs on the fast exponential and division (a few fp32 ulp, far below the
// bf16 rounding of what is saved): the accurate forms put a dependent chain with a
// slow-path branch on every element, which the epilogue warp (alone on its
// scheduler) cannot hide.  For z -> -inf the denominator is +inf and the quotient 0.
template <int ACT>
__device__ __forceinline__ float act_fwd(float z) {
  if (ACT == 1) return 0.5f * z * (1.0f + erff(z * 0.70710678118654752f));
  return __fdividef(z, 1.0f + __expf(-z));
}
// f(z) and f'(z) together (one exponential and one division for silu).
template <int ACT>
__device__ __forceinline__ void act_pair(float z, float& f, float& df) {
  if (ACT == 1) {
    const float cdf = 0.5f * (1.0f + erff(z * 0.70710678118654752f));
    f = z * cdf;
    df = cdf + z * 0.39894228040143268f * expf(-0.5f * z * z);
  } else {
    const float sg = __fdividef(1.0f, 1.0f + __expf(-z));
    f = z * sg;
    df = sg * (1.0f + z * (1.0f - sg));
  }
}
__device__ __forceinline__ float clamp_act(float v, float c) { return fminf(fmaxf(v, -c), c); }
// derivative of the clamp: 1 on [-c, c], ends included
__device__ __forceinline__ float clamp_pass(float v, float c) { return (v >= -c && v <= c) ? 1.0f : 0.0f; }

// Forward of one 32-column chunk: a = act(cl(g)) * cl(u), then g/u replaced by
// the values to save (clamp_encode, defined below).
__device__ __forceinline__ float clamp_encode(float v, float c);
template <int ACT, bool CL>
__device__ __forceinline__ void act_fwd_chunk(float (&g)[32], float (&u)[32], float (&a)[32], float c) {
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    a[i] = CL ? act_fwd<ACT>(clamp_act(g[i], c)) * clamp_act(u[i], c) : act_fwd<ACT>(g[i]) * u[i];
    if (CL) {
      g[i] = clamp_encode(g[i], c);
      u[i] = clamp_encode(u[i], c);
    }
  }
}
__device__ __forceinline__ void act_fwd_chunk(int act, float c, float (&g)[32], float (&u)[32], float (&a)[32]) {
  if (act == 1) {
    if (c > 0.0f) act_fwd_chunk<1, true>(g, u, a, c); else act_fwd_chunk<1, false>(g, u, a, c);
  } else {
    if (c > 0.0f) act_fwd_chunk<0, true>(g, u, a, c); else act_fwd_chunk<0, false>(g, u, a, c);
  }
}

// Backward of one chunk from the upstream dAct = w * q:
//   dG = dAct * cl(U) * act'(cl(G)) * [G in clamp],  dU = dAct * act(cl(G)) * [U in clamp]
// (dead rows give zeros).  G/U are the saved values, whose clamp test matches the
// forward's fp32 decision.
// Also returns sum_i q_i * act(cl(g_i)) * cl(u_i): the chunk's share of the router
// dot <Q, Act>, with the activation recomputed from the saved G and U (so the saved
// activation is not read again; it differs from the saved bf16 value by the
// rounding of G and U, far inside the tolerance).
template <int ACT, bool CL>
__device__ __forceinline__ float act_bwd_chunk(const float (&q)[32], const float (&g)[32], const float (&u)[32],
                                               float w, bool live, float c, float (&og)[32], float (&ou)[32]) {
  float dot = 0.0f;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const float da = w * q[i];
    float f, df;
    act_pair<ACT>(CL ? clamp_act(g[i], c) : g[i], f, df);
    const float uc = CL ? clamp_act(u[i], c) : u[i];
    dot += q[i] * (f * uc);
    og[i] = live ? da * uc * df * (CL ? clamp_pass(g[i], c) : 1.0f) : 0.0f;
    ou[i] = live ? da * f * (CL ? clamp_pass(u[i], c) : 1.0f) : 0.0f;
  }
  return dot;
}
__device__ __forceinline__ float act_bwd_chunk(int act, float c, const float (&q)[32], const float (&g)[32],
                                               const float (&u)[32], float w, bool live, float (&og)[32],
                                               float (&ou)[32]) {
  if (act == 1) {
    if (c > 0.0f) return act_bwd_chunk<1, true>(q, g, u, w, live, c, og, ou);
    return act_bwd_chunk<1, false>(q, g, u, w, live, c, og, ou);
  }
  if (c > 0.0f) return act_bwd_chunk<0, true>(q, g, u, w, live, c, og, ou);
  return act_bwd_chunk<0, false>(q, g, u, w, live, c, og, ou);
}
// Value saved (as bf16) for a gate/up pre-activation v so that the backward sees
// the forward's fp32 clamp decision: a clamped element (|v| > c) is saved as the
// smallest bf16 magnitude above c, an element inside [-c, c] as its bf16 value,
// rounded toward zero when rounding to nearest would cross c.  The result is a
// bf16 value; |saved| <= c exactly when the forward did not clamp.
__device__ __forceinline__ float clamp_encode(float v, float c) {
  if (fabsf(v) > c) {
    const uint32_t above = (__float_as_uint(c) & 0xFFFF0000u) + 0x10000u;  // next bf16 above trunc(c)
    return copysignf(__uint_as_float(above), v);
  }
  const float r = __bfloat162float(__float2bfloat16_rn(v));
  return fabsf(r) > c ? __uint_as_float(__float_as_uint(v) & 0xFFFF0000u) : r;
}

// Stores n (multiple of 8, <= 32) bf16 values v[i] * mul.
__device__ __forceinline__ void store_row_bf16(uint16_t* dst, const float (&v)[32], float mul, int n) {
#pragma unroll
  for (int j = 0; j < 32; j += 8) {
    if (j < n) {
      float t[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) t[i] = v[j + i] * mul;
      st_bf16x8(dst + j, t);
    }
  }
}
// Stores n (multiple of 4, <= 32) fp32 values v[i] * mul.
__device__ __forceinline__ void store_row_f32(float* dst, const float (&v)[32], float mul, int n) {
#pragma unroll
  for (int j = 0; j < 32; j += 4) {
    if (j < n) {
      float t[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) t[i] = v[j + i] * mul;
      st_f32x4(dst + j, t);
    }
  }
}

__device__ __forceinline__ int round16(int r) { return (r + 15) & ~15; }
// Tiles of `b` covering `n` (H and I are multiples of 64, not of the tile widths:
// TMA loads past the tensor edge read zeros, and epilogues skip the 32-column chunks
// -- or rows -- that lie past it).
__host__ __device__ __forceinline__ int cdiv(int n, int b) { return (n + b - 1) / b; }
// N of a two-SM (M = 256) MMA: a multiple of 32, so each CTA holds a multiple of 16 columns.
__device__ __forceinline__ int round32(int r) { return (r + 31) & ~31; }

// Coalesced epilogue row access.  An epilogue warp owns 32 consecutive
// accumulator rows, one per lane.  Storing "my row" directly makes every 16-byte
// warp store touch 32 different rows; instead the warp stages its 32 x 32-column
// chunk in shared memory and writes it back 4 lanes per row (8 rows of 64
// contiguous bytes per instruction).  Loads go the same way in reverse.

// dst0: row 0 of the warp, first column of the chunk; rows >= nvalid are skipped.
__device__ __forceinline__ void warp_store_rows_bf16(uint16_t* dst0, int64_t ld, int nvalid, const float (&v)[32],
                                                     float mul, uint32_t* stg) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int j = 0; j < 16; ++j) stg[lane * kStgPitch + j] = pack_bf16x2(v[2 * j] * mul, v[2 * j + 1] * mul);
  __syncwarp();
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    const int r = s * 8 + (lane >> 2), w = (lane & 3) * 4;
    const uint32_t* src = stg + r * kStgPitch + w;
    const uint4 u = make_uint4(src[0], src[1], src[2], src[3]);
    if (r < nvalid) *reinterpret_cast<uint4*>(dst0 + (int64_t)r * ld + 2 * w) = u;
  }
  __syncwarp();
}

// fp32 version: n (<= 32, multiple of 4) columns of v * mul, 8 lanes per row
// (4 rows of 128 contiguous bytes per instruction).
__device__ __forceinline__ void warp_store_rows_f32(float* dst0, int64_t ld, int nvalid, const float (&v)[32],
                                                    float mul, int n, uint32_t* stg) {
  const int lane = threadIdx.x & 31;
  // row i, column j at word 32 i + (j ^ i): conflict-free row writes and reads
#pragma unroll
  for (int j = 0; j < 32; ++j) stg[lane * 32 + (j ^ lane)] = __float_as_uint(v[j] * mul);
  __syncwarp();
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    const int r = s * 4 + (lane >> 3), w = (lane & 7) * 4;
    const uint32_t* src = stg + r * 32;
    const uint4 u = make_uint4(src[w ^ r], src[(w + 1) ^ r], src[(w + 2) ^ r], src[(w + 3) ^ r]);
    if (r < nvalid && w < n) *reinterpret_cast<uint4*>(dst0 + (int64_t)r * ld + w) = u;
  }
  __syncwarp();
}

// Epilogue stores through TMA: the warp writes its 32 rows x 32 bf16 columns into
// one of two 2 KB staging tiles (64-byte swizzle, conflict-free), one lane issues
// the bulk tensor store, and the warp goes on while the copy engine writes the
// rows out.  A tile is rewritten only after the store that last read it has
// finished reading.  Constructed once per tile epilogue (waits for the warp's
// earlier stores to finish reading the staging tiles).
// TMA stores for the large bf16 epilogue outputs (false: the staged warp stores).
// Same box, 65,536 tokens: step 31.9 -> 30.8 ms, W13 8.79 -> 8.31 ms, W13 dgrad
// 8.70 -> 7.93 ms.
constexpr bool kEpiTmaStore = true;
struct TmaStoreRing {
  uint8_t* base;
  int cur;
  __device__ __forceinline__ explicit TmaStoreRing(uint32_t* stg) : base(reinterpret_cast<uint8_t*>(stg)), cur(0) {
    if ((threadIdx.x & 31) == 0) bulk_wait_group_read<0>();
    __syncwarp();
  }
  // rows y0..y0+31 (one per lane), columns x0..x0+31 of the tensor of map m: v * mul
  __device__ __forceinline__ void store_bf16(const CUtensorMap* m, int x0, int y0, const float (&v)[32],
                                             float mul = 1.0f) {
    const int lane = threadIdx.x & 31;
    uint8_t* buf = base + cur * 2048;
    if (lane == 0) bulk_wait_group_read<1>();
    __syncwarp();
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint4 q;
      q.x = pack_bf16x2(v[8 * j + 0] * mul, v[8 * j + 1] * mul);
      q.y = pack_bf16x2(v[8 * j + 2] * mul, v[8 * j + 3] * mul);
      q.z = pack_bf16x2(v[8 * j + 4] * mul, v[8 * j + 5] * mul);
      q.w = pack_bf16x2(v[8 * j + 6] * mul, v[8 * j + 7] * mul);
      *reinterpret_cast<uint4*>(buf + lane * 64 + ((j ^ ((lane >> 1) & 3)) << 4)) = q;
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_2d(m, buf, x0, y0);
      bulk_commit_group();
    }
    cur ^= 1;
  }
};

// Issues the coalesced global loads of a warp's 32 rows x 32 bf16 columns.
__device__ __forceinline__ void warp_load_rows_issue(const uint16_t* src0, int64_t ld, uint4 (&u)[4]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    const int r = s * 8 + (lane >> 2);
    u[s] = __ldg(reinterpret_cast<const uint4*>(src0 + (int64_t)r * ld + (lane & 3) * 8));
  }
}
// Redistributes loaded rows so each lane holds its own row's 32 values.
__device__ __forceinline__ void warp_rows_to_lane(const uint4 (&u)[4], uint32_t* stg, float (&out)[32]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    uint32_t* d = stg + (s * 8 + (lane >> 2)) * kStgPitch + (lane & 3) * 4;
    d[0] = u[s].x;
    d[1] = u[s].y;
    d[2] = u[s].z;
    d[3] = u[s].w;
  }
  __syncwarp();
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const uint32_t w = stg[lane * kStgPitch + j];
    out[2 * j] = bf16_lo(w);
    out[2 * j + 1] = bf16_hi(w);
  }
  __syncwarp();
}

// =====================================================================================
// Forward F1 -- shared shrink, once per token:  Y13[t] = bf16(s * x_t [A1_a; A3_a]^T).
// M = tokens of adapter a, N = 2r (y1 | y3), K = H.  A: x K-major; B: A1/A3 K-major.
// =====================================================================================
struct ProbShrink {
  static constexpr bool kAmn = false, kBmn = false;
  static constexpr int kEpiWarps = 4;
  static constexpr bool kWide = false;
  CUtensorMap mx, mA1, mA3;  // x (H,T) box(64,128); A1/A3 (H,r,A) box(64,r,1)
  PlanView pl;
  int* err;
  uint16_t* Y13;
  int H, r;
  float s;
  __device__ int num_tiles() const { return pl.tok_tile[pl.A]; }
  __device__ TileInfo tile(int t) const {
    const int a = adapter_of_tile(pl, t);
    TileInfo ti;
    ti.g = a;
    ti.m0 = pl.tok_off[a] + (t - pl.tok_tile[a]) * 128;
    ti.mend = pl.tok_off[a + 1];
    ti.n0 = 0;
    ti.sub = 0;
    ti.nk = H / kBK;
    ti.k0 = 0;
    return ti;
  }
  __device__ void prefetch() const {
    tma_prefetch_map(&mx);
    tma_prefetch_map(&mA1);
    tma_prefetch_map(&mA3);
  }
  __device__ void load(const TileInfo& ti, int ks, uint8_t* sa, uint8_t* sb, uint64_t* bar) const {
    mbar_arrive_expect_tx(bar, kAStage128 + 2 * r * 128);
    tma_load_2d(sa, &mx, bar, ks * kBK, ti.m0);
    tma_load_3d(sb, &mA1, bar, ks * kBK, 0, ti.g);
    tma_load_3d(sb + r * 128, &mA3, bar, ks * kBK, 0, ti.g);
  }
  __device__ MmaStep mma_step(const TileInfo&, int ks) const { return MmaStep{2 * r, 0, 0, ks == 0}; }
  __device__ void epilogue(const TileInfo& ti, int row, uint32_t taddr, int c0, int cs, uint32_t* stg) const {
    const int64_t t = (int64_t)ti.m0 + row;
    const bool ok = t < ti.mend;
    for (int c = c0; c < 2 * r; c += cs) {
      float v[32];
      tmem_ld32(taddr + c, v);
      const int n = 2 * r - c < 32 ? 2 * r - c : 32;
      if (ok) store_row_bf16(Y13 + t * (2 * r) + c, v, s, n);
    }
  }
  __device__ void epilogue_empty(const TileInfo&, int, int, int) const {}
};

// =====================================================================================
// Forward F3 -- W13 expert GEMM with the expert-local B1/B3 expand and SwiGLU:
//   G = Xp W1_e^T + Y1p B1_ae^T,  U = Xp W3_e^T + Y3p B3_ae^T   (s folded into Y13)
//   Act = bf16(act(cl(G)) * cl(U)); G and U are kept (bf16) for the backward, with
//   the forward's clamp decision encoded (clamp_encode).
// Tile: 128 rows x 128 columns of I; the accumulator holds the gate columns in
// TMEM [0,128) and the up columns in [128,256).  K steps: H/64 base steps (one
// N=256 MMA over W1|W3 rows), then ceil(r/64) steps per side for the expand
// (N=128 into the gate half with Y1p/B1, then into the up half with Y3p/B3).
// =====================================================================================
// 256-row tiles: a third fewer operand bytes per FLOP than 128-row tiles, at the
// price of an epilogue that no longer overlaps the next tile's main loop.  With the
// fast silu that trade pays (same-box 9.33 -> 9.04 ms at 65,536 tokens, E256).
constexpr bool kW13Wide = true;
// MX: W1/W3 are MXFP4, decoded into the stage by the epilogue warps (no TMA for them).
// W13's epilogue stores through the TMA-store ring.  Measured against 64-byte row
// segments straight from registers (same box, two alternations, 65,536 tokens): W13
// 8.7-8.9 ms with the ring, 9.7-9.9 ms with row stores (the native W13, without staging
// buffers and with a fourth stage, prefers row stores).  Handing the accumulator back
// to the MMA right after the last tensor-memory read of a tile (before the last chunk's
// activation and stores) was measured too: 8.58-8.59 ms against 8.55-8.57 ms, no gain,
// since the next tile's loads and MMAs already overlap the epilogue of the other buffer.
template <bool MX>
struct ProbW13T {
  static constexpr bool kAmn = false, kBmn = false;
  static constexpr bool kWide = kW13Wide;
  static constexpr bool kDecode = MX;
  static constexpr bool kMxMN = false;
  static constexpr int kEpiWarps = kWide ? 8 : 4;
  const uint8_t *S1q, *S3q;  // MX: scales [E,I,H/32]
  CUtensorMap mW1q, mW3q;    // MX: packed [E,I,H/2] bytes, box (32, 128, 1)
  CUtensorMap mXp, mY13p, mW1, mW3, mB1, mB3;  // Xp (H,P) box(64,128); Y13p (2r,P) box(64,128);
                                               // W1/W3 (H,I,E) box(64,128,1); B1/B3 (r,I,G) box(64,128,1)
  CUtensorMap mG, mU, mAct;                    // outputs (I,P), 32 x 32 store boxes
  PlanView pl;
  int* err;
  uint16_t *G, *U, *Act;
  int H, I, r;
  int act;      // 0 = SwiGLU, 1 = GeGLU
  float clamp;  // activation clamp (0 = none)
  __device__ int ntn() const { return cdiv(I, 128); }
  __device__ int nkr() const { return (r + 63) / 64; }
  __device__ int num_tiles() const {
    return (kWide ? pl.wtile_off[pl.G] : pl.offsets[pl.G] / 128) * ntn();
  }
  __device__ TileInfo tile(int t) const {  // column-tile-major inside each group
    TileInfo ti;
    if (kWide)
      ti.n0 = wide_entry_decode(nmajor_wide_fetch(pl, t, ntn()), ti) * 128;
    else
      ti.n0 = nmajor_narrow_decode(nmajor_narrow_fetch(pl, t, ntn()), t, ntn(), ti) * 128;
    ti.sub = 0;
    ti.nk = H / kBK + 2 * nkr();
    return ti;
  }
  __device__ void prefetch() const {
    tma_prefetch_map(&mXp);
    tma_prefetch_map(&mY13p);
    tma_prefetch_map(&mW1);
    tma_prefetch_map(&mW3);
    tma_prefetch_map(&mB1);
    tma_prefetch_map(&mB3);
  }
  __device__ void load(const TileInfo& ti, int ks, uint8_t* sa, uint8_t* sb, uint64_t* bar) const {
    const int nb = H / kBK;
    const int e = ti.g % pl.E;
    if (ks < nb) {
      mbar_arrive_expect_tx(bar, ti.mh * kAStage128 + (MX ? 2 * 128 * 32 : 2 * 128 * 128));
      load_a_wide(ti, sa, &mXp, bar, ks * kBK);
      if (MX) {  // packed rows: W1's into rows 0..127, W3's into rows 128..255
        tma_load_3d(sb + kMxRaw, &mW1q, bar, ks * (kBK / 2), ti.n0, e);
        tma_load_3d(sb + kMxRaw + 128 * 32, &mW3q, bar, ks * (kBK / 2), ti.n0, e);
      } else {
        tma_load_3d(sb, &mW1, bar, ks * kBK, ti.n0, e);
        tma_load_3d(sb + 128 * 128, &mW3, bar, ks * kBK, ti.n0, e);
      }
    } else {
      const int j = ks - nb, half = j / nkr(), kb = j % nkr();
      mbar_arrive_expect_tx(bar, ti.mh * kAStage128 + 128 * 128);
      load_a_wide(ti, sa, &mY13p, bar, half * r + kb * kBK);
      tma_load_3d(sb, half ? &mB3 : &mB1, bar, kb * kBK, ti.n0, ti.g);
    }
  }
  // MX, base K steps: rows 0..127 of the B tile are W1 rows n0.., 128..255 W3 rows
  __device__ bool decodes(const TileInfo&, int ks) const { return MX && ks < H / kBK; }
  __device__ MxScales mx_scales(const TileInfo& ti, int ks) const {
    const int64_t so = ((int64_t)(ti.g % pl.E) * I + ti.n0) * (H / 32) + ks * (kBK / 32);
    const int lim = I - ti.n0 < 128 ? I - ti.n0 : 128;
    return MxScales{{S1q + so, S3q + so}, H / 32, {lim, lim}};
  }
  __device__ MmaStep mma_step(const TileInfo&, int ks) const {
    const int nb = H / kBK;
    if (ks < nb) return MmaStep{256, 0, 0, ks == 0};
    const int half = (ks - nb) / nkr();
    return MmaStep{128, half * 128, 0, 0};
  }
  __device__ void epilogue(const TileInfo& ti, int row, uint32_t taddr, int c0, int cs, uint32_t* stg) const {
    const int y0 = ti.m0 + row - (threadIdx.x & 31);  // warp's first row
    TmaStoreRing out(stg);
    const int64_t base = (int64_t)y0 * I + ti.n0;
    for (int c = c0; c < 128 && ti.n0 + c < I; c += cs) {
      float g[32], u[32], a[32];
      tmem_ld32(taddr + c, g);
      tmem_ld32(taddr + 128 + c, u);
      act_fwd_chunk(act, clamp, g, u, a);
      if (kEpiTmaStore) {
        out.store_bf16(&mG, ti.n0 + c, y0, g);
        out.store_bf16(&mU, ti.n0 + c, y0, u);
        out.store_bf16(&mAct, ti.n0 + c, y0, a);
      } else {
        warp_store_rows_bf16(G + base + c, I, 32, g, 1.0f, stg);
        warp_store_rows_bf16(U + base + c, I, 32, u, 1.0f, stg);
        warp_store_rows_bf16(Act + base + c, I, 32, a, 1.0f, stg);
      }
    }
  }
  __device__ void epilogue_empty(const TileInfo&, int, int, int) const {}
};
using ProbW13 = ProbW13T<false>;

// =====================================================================================
// Native FP4 forward F3 (block-scaled MMAs; see ProbW13Nv below)
// =====================================================================================
// 32 consecutive values of one row as bf16 (64 bytes, 16-byte aligned) from registers.
__device__ __forceinline__ void store_row_bf16(uint16_t* dst, const float (&v)[32]) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint4 q;
    q.x = pack_bf16x2(v[8 * j + 0], v[8 * j + 1]);
    q.y = pack_bf16x2(v[8 * j + 2], v[8 * j + 3]);
    q.z = pack_bf16x2(v[8 * j + 4], v[8 * j + 5]);
    q.w = pack_bf16x2(v[8 * j + 6], v[8 * j + 7]);
    *reinterpret_cast<uint4*>(dst + 8 * j) = q;
  }
}

// Native FP4 forward F3: the gate/up base products on block-scaled FP4 tensor cores,
//   G = q8(Xp) W1_e^T + s (Y1p B1_e^T),   U = q8(Xp) W3_e^T + s (Y3p B3_e^T)
// with q8(Xp) the routed rows as MXFP8 (E4M3 codes Xq + scale words Xs, from
// launch_gather_fwd_mxfp8) and W1/W3 in MXFP4 as stored -- no decoded copy.  128-row
// tiles x (128 W1 rows + 128 W3 rows): H/128 native K steps, then the BF16 side-LoRA
// steps of ProbW13 into the same accumulator; the same epilogue.  H, I multiples of 128.
// Epilogue of the native W13, measured (65,536 tokens, E256): 16-byte row stores from
// registers with four stages 6.68 ms; TMA bulk stores out of staging tiles with three
// stages 6.81 ms; 16 epilogue warps releasing the accumulator as soon as it is read
// (the next tile's MMAs overlapping the activation and the stores) 6.90 ms; the
// activation computed and stored 8 columns at a time (fewer live registers) 7.29 ms;
// gate and up read with one tensor-memory wait or one each: no difference.  In-kernel cycle
// counters put the MMA issuer at ~98% of the FP8 rate while it has operands, waiting
// for them 31% of the kernel with the producer's ring full: operand delivery (each
// stage's A and weight tiles landing from L2/HBM) is what holds it, not the epilogue.
struct ProbW13Nv {
  static constexpr bool kAmn = false, kBmn = false, kWide = false, kNative = true;
  static constexpr int kEpiWarps = 8;
  static constexpr int kNvLayout = kNvLayoutCopy;  // scale words copied by the MMA thread
  const uint8_t* Xs;          // [P/128][H/128][128][4] scale bytes of Xq
  const uint8_t *S1t, *S3t;   // [E*I/128][H/128][128][4] scale bytes of W1/W3 (launch_scales_to_tiles)
  CUtensorMap mXq;            // Xq (H,P) bytes, box (128,128)
  CUtensorMap mW1f, mW3f;     // W1/W3 E2M1 (H,I,E), box (128 codes, 128, 1)
  CUtensorMap mY13p, mB1, mB3;  // as ProbW13
  PlanView pl;
  int* err;
  uint16_t *G, *U, *Act;  // [P,I] outputs
  uint8_t *Actq, *Acts;   // the activation as MXFP8 for the native W2: codes [P,I], scale
                          // words [P/128][I/128][32][4][4] (as launch_scales_to_tiles lays them)
  int H, I, r;
  int act;
  float clamp;
  __device__ int ntn() const { return I / 128; }
  __device__ int nkr() const { return (r + 63) / 64; }
  __device__ int num_tiles() const { return pl.offsets[pl.G] / 128 * ntn(); }
  __device__ TileInfo tile(int t) const {
    TileInfo ti;
    ti.n0 = nmajor_narrow_decode(nmajor_narrow_fetch(pl, t, ntn()), t, ntn(), ti) * 128;
    ti.sub = 0;
    ti.nk = H / 128 + 2 * nkr();
    return ti;
  }
  __device__ void prefetch() const {
    tma_prefetch_map(&mXq);
    tma_prefetch_map(&mW1f);
    tma_prefetch_map(&mW3f);
    tma_prefetch_map(&mY13p);
    tma_prefetch_map(&mB1);
    tma_prefetch_map(&mB3);
  }
  __device__ void load(const TileInfo& ti, int ks, uint8_t* sa, uint8_t* sb, uint8_t* sf, uint64_t* bar) const {
    const int nb = H / 128;
    if (ks < nb) {
      const int e = ti.g % pl.E;
      const int64_t kt = H / 128;
      const int64_t wt = ((int64_t)e * (I / 128) + (ti.n0 >> 7)) * kt + ks;  // weight row tile, K step
      mbar_arrive_expect_tx(bar, 128 * 128 + 2 * 128 * 64 + kNvSfBytes);  // E2M1 boxes count packed bytes
      tma_load_2d(sa, &mXq, bar, ks * 128, ti.m0);
      tma_load_3d(sb, &mW1f, bar, ks * 128, ti.n0, e);
      tma_load_3d(sb + 128 * 128, &mW3f, bar, ks * 128, ti.n0, e);
      bulk_load(sf, Xs + ((int64_t)(ti.m0 >> 7) * kt + ks) * 512, 512, bar);
      bulk_load(sf + 512, S1t + wt * 512, 512, bar);
      bulk_load(sf + 1024, S3t + wt * 512, 512, bar);
    } else {
      const int j = ks - nb, half = j / nkr(), kb = j % nkr();
      mbar_arrive_expect_tx(bar, kAStage128 + 128 * 128);
      tma_load_2d(sa, &mY13p, bar, half * r + kb * kBK, ti.m0);
      tma_load_3d(sb, half ? &mB3 : &mB1, bar, kb * kBK, ti.n0, ti.g);
    }
  }
  __device__ bool native_step(const TileInfo&, int ks) const { return ks < H / 128; }
  __device__ MmaStep mma_step(const TileInfo&, int ks) const {
    const int nb = H / 128;
    if (ks < nb) return MmaStep{256, 0, 0, ks == 0};
    return MmaStep{128, ((ks - nb) / nkr()) * 128, 0, 0};
  }
  __device__ void epilogue(const TileInfo& ti, int row, uint32_t taddr, int c0, int cs, uint32_t*) const {
    const int64_t o = ((int64_t)ti.m0 + row) * I + ti.n0;  // this thread's row: 64-byte row segments
    const int64_t p = (int64_t)ti.m0 + row;
    uint8_t* sw = Acts + ((p >> 7) * (I / 128) + (ti.n0 >> 7)) * 512 + nv_word((int)(p & 127)) * 4;
    for (int c = c0; c < 128; c += cs) {
      float g[32], u[32], a[32];
      tmem_ld32(taddr + c, g);
      tmem_ld32(taddr + 128 + c, u);
      act_fwd_chunk(act, clamp, g, u, a);
      store_row_bf16(G + o + c, g);
      store_row_bf16(U + o + c, u);
      store_row_bf16(Act + o + c, a);
      // q8 of the stored (bf16-rounded) activation: this thread's 32 columns are one
      // MXFP8 block, byte c / 32 of the row's scale word for this 128-wide K step
#pragma unroll
      for (int i = 0; i < 32; ++i) a[i] = __bfloat162float(__float2bfloat16_rn(a[i]));
      uint4 q[2];
      sw[c >> 5] = (uint8_t)mxfp8_block_f32(a, q);
      uint4* dq = reinterpret_cast<uint4*>(Actq + o + c);
      dq[0] = q[0];
      dq[1] = q[1];
    }
  }
  __device__ void epilogue_empty(const TileInfo&, int, int, int) const {}
};

// =====================================================================================
// Forward F4/F5 -- W2 expert GEMM with the expert-local A2 shrink:
//   O = Act W2_e^T  [P,H] (unweighted),   Z2 = bf16(Act A2_ae^T) [P,r]
// N tiles: H/256 base tiles over W2 rows, then one tile of round16(r) over A2 rows.
// =====================================================================================
// The forward W2 GEMM on the one-SM engine with 256-row tiles (true) or on the
// two-SM engine (ProbW2Pair, false).  With the TMA-store epilogue: 4.22 vs 4.47 ms
// (same box, 65,536 tokens, E256).
constexpr bool kW2OneSmWide = true;
// MX: W2 is MXFP4, decoded into the stage by the epilogue warps (no TMA for it).
template <bool MX>
struct ProbW2T {
  static constexpr bool kAmn = false, kBmn = false;
  static constexpr bool kWide = kW2OneSmWide;
  static constexpr bool kDecode = MX;
  static constexpr bool kMxMN = false;
  static constexpr int kEpiWarps = kWide ? 8 : 4;
  const uint8_t* S2q;  // MX: scales [E,H,I/32]
  CUtensorMap mW2q;    // MX: packed [E,H,I/2] bytes, box (32, 256, 1)
  CUtensorMap mAct, mW2, mA2;  // Act (I,P) box(64,128); W2 (I,H,E) box(64,256,1); A2 (I,r,G) box(64,r16,1)
  CUtensorMap mO;              // output (H,P), 32 x 32 store boxes
  PlanView pl;
  int* err;
  uint16_t *O, *Z2;
  int H, I, r;
  __device__ int ntn() const { return cdiv(H, 256) + 1; }
  __device__ int num_tiles() const {
    return (kWide ? pl.wtile_off[pl.G] : pl.offsets[pl.G] / 128) * ntn();
  }
  __device__ TileInfo tile(int t) const {  // column-tile-major inside each group
    TileInfo ti;
    const int nt = kWide ? wide_entry_decode(nmajor_wide_fetch(pl, t, ntn()), ti)
                         : nmajor_narrow_decode(nmajor_narrow_fetch(pl, t, ntn()), t, ntn(), ti);
    ti.sub = nt == cdiv(H, 256);
    ti.n0 = ti.sub ? 0 : nt * 256;
    ti.nk = I / kBK;
    return ti;
  }
  __device__ void prefetch() const {
    tma_prefetch_map(&mAct);
    tma_prefetch_map(&mW2);
    tma_prefetch_map(&mA2);
  }
  __device__ void load(const TileInfo& ti, int ks, uint8_t* sa, uint8_t* sb, uint64_t* bar) const {
    if (!ti.sub) {
      mbar_arrive_expect_tx(bar, ti.mh * kAStage128 + (MX ? 256 * 32 : 256 * 128));
      load_a_wide(ti, sa, &mAct, bar, ks * kBK);
      if (MX)
        tma_load_3d(sb + kMxRaw, &mW2q, bar, ks * (kBK / 2), ti.n0, ti.g % pl.E);
      else
        tma_load_3d(sb, &mW2, bar, ks * kBK, ti.n0, ti.g % pl.E);
    } else {
      mbar_arrive_expect_tx(bar, ti.mh * kAStage128 + round16(r) * 128);
      load_a_wide(ti, sa, &mAct, bar, ks * kBK);
      tma_load_3d(sb, &mA2, bar, ks * kBK, 0, ti.g);
    }
  }
  // MX, base tiles: B rows are W2 rows h = n0 + rho
  __device__ bool decodes(const TileInfo& ti, int) const { return MX && !ti.sub; }
  __device__ MxScales mx_scales(const TileInfo& ti, int ks) const {
    const int64_t so = ((int64_t)(ti.g % pl.E) * H + ti.n0) * (I / 32) + ks * (kBK / 32);
    const int left = H - ti.n0;
    return MxScales{{S2q + so, S2q + so + 128 * (int64_t)(I / 32)}, I / 32,
                    {left < 128 ? left : 128, left - 128 < 0 ? 0 : (left - 128 < 128 ? left - 128 : 128)}};
  }
  __device__ MmaStep mma_step(const TileInfo& ti, int ks) const {
    return MmaStep{ti.sub ? round16(r) : 256, 0, 0, ks == 0};
  }
  __device__ void epilogue(const TileInfo& ti, int row, uint32_t taddr, int c0, int cs, uint32_t* stg) const {
    const int64_t p = (int64_t)ti.m0 + row;
    TmaStoreRing out(stg);  // before any use of the staging buffer
    if (!ti.sub) {
      const int y0 = (int)(p - (threadIdx.x & 31));  // warp's first row
      uint16_t* o0 = O + (int64_t)y0 * H + ti.n0;
      for (int c = c0; c < 256 && ti.n0 + c < H; c += cs) {
        float v[32];
        tmem_ld32(taddr + c, v);
        if (kEpiTmaStore)
          out.store_bf16(&mO, ti.n0 + c, y0, v);
        else
          warp_store_rows_bf16(o0 + c, H, 32, v, 1.0f, stg);
      }
    } else {
      for (int c = c0; c < r; c += cs) {
        float v[32];
        tmem_ld32(taddr + c, v);
        store_row_bf16(Z2 + p * r + c, v, 1.0f, r - c < 32 ? r - c : 32);
      }
    }
  }
  __device__ void epilogue_empty(const TileInfo&, int, int, int) const {}
};
using ProbW2 = ProbW2T<false>;

// =====================================================================================
// Native FP4 forward F4/F5
// =====================================================================================
// Native FP4 forward F4/F5: the down base product on block-scaled FP4 tensor cores,
//   O = q8(Act) W2_e^T   [P,H] (unweighted),   Z2 = bf16(Act A2_ae^T) [P,r]
// with q8(Act) the activation as MXFP8 (written by ProbW13Nv's epilogue) and W2 in
// MXFP4 as stored.  128-row tiles: H/256 native tiles over W2 rows (I/128 steps), then
// one BF16 tile over A2 rows on the bf16 activation (the side shrink stays BF16).  H, I
// multiples of 128; a last native tile with 128 valid rows reads zero codes past H.
struct ProbW2Nv {
  static constexpr bool kAmn = false, kBmn = false, kWide = false, kNative = true;
  static constexpr int kEpiWarps = 8;
  static constexpr int kNvLayout = kNvLayoutCopy;
  const uint8_t* Acts;       // [P/128][I/128][512] scale words of Actq
  const uint8_t* S2t;        // [E*H/128][I/128][512] scale words of W2 (launch_scales_to_tiles)
  CUtensorMap mActq;         // Actq (I,P) bytes, box (128,128)
  CUtensorMap mW2f;          // W2 E2M1 (I,H,E), box (128 codes, 256, 1)
  CUtensorMap mAct, mA2;     // Act (I,P) box(64,128); A2 (I,r,G) box(64,r16,1)
  PlanView pl;
  int* err;
  uint16_t *O, *Z2;
  int H, I, r;
  __device__ int ntn() const { return cdiv(H, 256) + 1; }
  __device__ int num_tiles() const { return pl.offsets[pl.G] / 128 * ntn(); }
  __device__ TileInfo tile(int t) const {
    TileInfo ti;
    const int nt = nmajor_narrow_decode(nmajor_narrow_fetch(pl, t, ntn()), t, ntn(), ti);
    ti.sub = nt == cdiv(H, 256);
    ti.n0 = ti.sub ? 0 : nt * 256;
    ti.nk = ti.sub ? I / kBK : I / 128;
    return ti;
  }
  __device__ void prefetch() const {
    tma_prefetch_map(&mActq);
    tma_prefetch_map(&mW2f);
    tma_prefetch_map(&mAct);
    tma_prefetch_map(&mA2);
  }
  __device__ void load(const TileInfo& ti, int ks, uint8_t* sa, uint8_t* sb, uint8_t* sf, uint64_t* bar) const {
    if (!ti.sub) {
      const int e = ti.g % pl.E;
      const int64_t kt = I / 128, hb = H / 128;
      const int64_t b0 = (int64_t)e * hb + (ti.n0 >> 7);
      const int64_t b1 = (ti.n0 >> 7) + 1 < hb ? b0 + 1 : b0;  // past H: any valid block (codes there are 0)
      mbar_arrive_expect_tx(bar, 128 * 128 + 256 * 64 + kNvSfBytes);  // E2M1 boxes count packed bytes
      tma_load_2d(sa, &mActq, bar, ks * 128, ti.m0);
      tma_load_3d(sb, &mW2f, bar, ks * 128, ti.n0, e);
      bulk_load(sf, Acts + ((int64_t)(ti.m0 >> 7) * kt + ks) * 512, 512, bar);
      bulk_load(sf + 512, S2t + (b0 * kt + ks) * 512, 512, bar);
      bulk_load(sf + 1024, S2t + (b1 * kt + ks) * 512, 512, bar);
    } else {
      mbar_arrive_expect_tx(bar, kAStage128 + round16(r) * 128);
      tma_load_2d(sa, &mAct, bar, ks * kBK, ti.m0);
      tma_load_3d(sb, &mA2, bar, ks * kBK, 0, ti.g);
    }
  }
  __device__ bool native_step(const TileInfo& ti, int) const { return !ti.sub; }
  __device__ MmaStep mma_step(const TileInfo& ti, int ks) const {
    return MmaStep{ti.sub ? round16(r) : 256, 0, 0, ks == 0};
  }
  __device__ void epilogue(const TileInfo& ti, int row, uint32_t taddr, int c0, int cs, uint32_t*) const {
    const int64_t p = (int64_t)ti.m0 + row;
    if (!ti.sub) {
      for (int c = c0; c < 256 && ti.n0 + c < H; c += cs) {
        float v[32];
        tmem_ld32(taddr + c, v);
        store_row_bf16(O + p * H + ti.n0 + c, v);
      }
    } else {
      for (int c = c0; c < r; c += cs) {
        float v[32];
        tmem_ld32(taddr + c, v);
        store_row_bf16(Z2 + p * r + c, v, 1.0f, r - c < 32 ? r - c : 32);
      }
    }
  }
  __device__ void epilogue_empty(const TileInfo&, int, int, int) const {}
};

// =====================================================================================
// Forward F6 (first half) -- shared B2 expand, once per token:
//   Yl_t = bf16( s * Z2w_t B2_a^T )   [T,H]
// M = tokens of adapter a, N = H (tiles of 256), K = r.  The routing-weighted sum
// of the routed rows is added by combine_rows (mem_kernels.cu), which reads them
// one whole row per warp: a TMEM-row-per-thread epilogue would touch 32 scattered
// rows per warp instruction.
// =====================================================================================
struct ProbB2Expand {
  static constexpr bool kAmn = false, kBmn = false;
  // 8 epilogue warps (TMA-store epilogue; same box: 0.109 vs 0.143 ms with 4)
  static constexpr int kEpiWarps = 8;
  static constexpr bool kWide = false;
  CUtensorMap mZ2w, mB2;  // Z2w (r,T) box(64,128); B2 (r,H,A) box(64,256,1)
  CUtensorMap mYl;        // output (H,T), 32 x 32 store boxes
  PlanView pl;
  int* err;
  uint16_t* Yl;
  int H, r;
  float s;
  __device__ int ntn() const { return cdiv(H, 256); }
  __device__ int num_tiles() const { return pl.tok_tile[pl.A] * ntn(); }
  __device__ TileInfo tile(int t) const {
    const int mt = t / ntn(), nt = t % ntn();
    const int a = adapter_of_tile(pl, mt);
    TileInfo ti;
    ti.g = a;
    ti.m0 = pl.tok_off[a] + (mt - pl.tok_tile[a]) * 128;
    ti.mend = pl.tok_off[a + 1];
    ti.n0 = nt * 256;
    ti.sub = 0;
    ti.nk = (r + kBK - 1) / kBK;
    ti.k0 = 0;
    return ti;
  }
  __device__ void prefetch() const {
    tma_prefetch_map(&mZ2w);
    tma_prefetch_map(&mB2);
  }
  __device__ void load(const TileInfo& ti, int ks, uint8_t* sa, uint8_t* sb, uint64_t* bar) const {
    mbar_arrive_expect_tx(bar, kAStage128 + 256 * 128);
    tma_load_2d(sa, &mZ2w, bar, ks * kBK, ti.m0);
    tma_load_3d(sb, &mB2, bar, ks * kBK, ti.n0, ti.g);
  }
  __device__ MmaStep mma_step(const TileInfo&, int ks) const { return MmaStep{256, 0, 0, ks == 0}; }
  __device__ void epilogue(const TileInfo& ti, int row, uint32_t taddr, int c0, int cs, uint32_t* stg) const {
    const int64_t t0 = (int64_t)ti.m0 + row - (threadIdx.x & 31);  // warp's first row
    const int nvalid = (int)(ti.mend - t0 < 32 ? ti.mend - t0 : 32);
    // A tile ends early only at the last token: adapters start on 128-token
    // boundaries, so a whole-box store never reaches another adapter's rows, and
    // the map clips rows past T.
    TmaStoreRing out(stg);
    for (int c = c0; c < 256 && ti.n0 + c < H; c += cs) {
      float v[32];
      tmem_ld32(taddr + c, v);
      if (nvalid <= 0) continue;
      if (kEpiTmaStore)
        out.store_bf16(&mYl, ti.n0 + c, (int)t0, v, s);
      else
        warp_store_rows_bf16(Yl + t0 * H + ti.n0 + c, H, nvalid, v, s, stg);
    }
  }
  __device__ void epilogue_empty(const TileInfo&, int, int, int) const {}
};

// =====================================================================================
// Backward B1a -- dyB2 = bf16(dy B2_a) [T,r], per token (B2 shared).
// A: dy K-major; B: (n=q, k=h) = B2[a][h][q], MN-major.
// =====================================================================================
struct ProbDyB2 {
  static constexpr bool kAmn = false, kBmn = true;
  static constexpr int kEpiWarps = 4;
  static constexpr bool kWide = false;
  CUtensorMap mdy, mB2;  // dy (H,T) box(64,128); B2 (r,H,A) box(64,64,1)
  PlanView pl;
  int* err;
  uint16_t* dyB2;
  int H, r;
  __device__ int num_tiles() const { return pl.tok_tile[pl.A]; }
  __device__ TileInfo tile(int t) const {
    const int a = adapter_of_tile(pl, t);
    TileInfo ti;
    ti.g = a;
    ti.m0 = pl.tok_off[a] + (t - pl.tok_tile[a]) * 128;
    ti.mend = pl.tok_off[a + 1];
    ti.n0 = 0;
    ti.sub = 0;
    ti.nk = H / kBK;
    ti.k0 = 0;
    return ti;
  }
  __device__ void prefetch() const {
    tma_prefetch_map(&mdy);
    tma_prefetch_map(&mB2);
  }
  __device__ void load(const TileInfo& ti, int ks, uint8_t* sa, uint8_t* sb, uint64_t* bar) const {
    const int nbox = (round16(r) + 63) / 64;
    mbar_arrive_expect_tx(bar, kAStage128 + nbox * 8192);
    tma_load_2d(sa, &mdy, bar, ks * kBK, ti.m0);
    for (int c = 0; c < nbox; ++c) tma_load_3d(sb + c * 8192, &mB2, bar, c * 64, ks * kBK, ti.g);
  }
  __device__ MmaStep mma_step(const TileInfo&, int ks) const { return MmaStep{round16(r), 0, 0, ks == 0}; }
  __device__ void epilogue(const TileInfo& ti, int row, uint32_t taddr, int c0, int cs, uint32_t* stg) const {
    const int64_t t = (int64_t)ti.m0 + row;
    const bool ok = t < ti.mend;
    for (int c = c0; c < r; c += cs) {
      float v[32];
      tmem_ld32(taddr + c, v);
      if (ok) store_row_bf16(dyB2 + t * r + c, v, 1.0f, r - c < 32 ? r - c : 32);
    }
  }
  __device__ void epilogue_empty(const TileInfo&, int, int, int) const {}
};

// =====================================================================================
// Backward B1b -- dB2_a = s * dy^T Z2w over the adapter's tokens  [H,r] fp32.
// M = H, N = r, K = tokens.  A: (m=h, k=t) = dy[t][h] MN-major; B: (n=q, k=t) = Z2w[t][q] MN-major.
// The token range is cut into `split` slices of whole 64-token steps (few output
// tiles, very long K); slice s writes out + s*split_stride, summed afterwards in
// slice order by reduce_splits.
// =====================================================================================
struct ProbDB2 {
  static constexpr bool kAmn = true, kBmn = true;
  static constexpr int kEpiWarps = 4;
  static constexpr bool kWide = false;
  CUtensorMap mdy, mZ2w;  // dy (H,T) box(64,64); Z2w (r,T) box(64,64)
  PlanView pl;
  int* err;
  float* out;  // dB2, or the split partials
  int64_t split_stride;
  int H, r, split;
  float s;
  __device__ int num_tiles() const { return split * pl.A * cdiv(H, 128); }
  __device__ TileInfo tile(int t) const {
    const int ntm = cdiv(H, 128), per = pl.A * ntm;
    const int sp = t / per, a = (t % per) / ntm, mt = t % ntm;
    TileInfo ti;
    ti.g = a;
    ti.m0 = mt * 128;
    ti.mend = H;
    ti.n0 = 0;
    ti.sub = sp;
    const int nk = (pl.tok_off[a + 1] - pl.tok_off[a] + kBK - 1) / kBK, cs = (nk + split - 1) / split;
    ti.k0 = pl.tok_off[a] + sp * cs * kBK;
    ti.nk = max(0, min(cs, nk - sp * cs));
    return ti;
  }
  __device__ float* row_ptr(const TileInfo& ti, int64_t h) const {
    return out + ti.sub * split_stride + ((int64_t)ti.g * H + h) * r;
  }
  __device__ void prefetch() const {
    tma_prefetch_map(&mdy);
    tma_prefetch_map(&mZ2w);
  }
  __device__ void load(const TileInfo& ti, int ks, uint8_t* sa, uint8_t* sb, uint64_t* bar) const {
    const int nbox = (round16(r) + 63) / 64;
    const int kt = ti.k0 + ks * kBK;
    mbar_arrive_expect_tx(bar, kAStage128 + nbox * 8192);
    tma_load_2d(sa, &mdy, bar, ti.m0, kt);
    tma_load_2d(sa + 8192, &mdy, bar, ti.m0 + 64, kt);
    for (int c = 0; c < nbox; ++c) tma_load_2d(sb + c * 8192, &mZ2w, bar, c * 64, kt);
  }
  __device__ MmaStep mma_step(const TileInfo&, int ks) const { return MmaStep{round16(r), 0, 0, ks == 0}; }
  __device__ void epilogue(const TileInfo& ti, int row, uint32_t taddr, int c0, int cs, uint32_t* stg) const {
    const int h0 = ti.m0 + row - (threadIdx.x & 31);  // warp's first row
    if (h0 >= H) return;                                // rows past H (H % 128 == 64)
    float* o0 = row_ptr(ti, h0);
    for (int c = c0; c < r; c += cs) {
      float v[32];
      tmem_ld32(taddr + c, v);
      warp_store_rows_f32(o0 + c, r, 32, v, s, r - c < 32 ? r - c : 32, stg);
    }
  }
  __device__ void epilogue_empty(const TileInfo& ti, int row, int c0, int cs) const {
    const float z[32] = {};
    const int64_t h = (int64_t)ti.m0 + row;
    if (h >= H) return;
    for (int c = c0; c < r; c += cs) store_row_f32(row_ptr(ti, h) + c, z, 0.f, r - c < 32 ? r - c : 32);
  }
};

// =====================================================================================
// Backward B3/B4 -- W2^T dgrad with the A2 path, SwiGLU backward and router dots:
//   Q  = Dp W2_e + D2p A2_ae              [P,I]   (D2p = s * dyB2 of the row's token)
//   dAct = w * Q;  dG = dAct * cl(U) * act'(cl(G)) * [G in clamp];  dU = dAct * act(cl(G)) * [U in clamp]
//   part[p, 2*n-tile + half] = <Q, Act> over the columns one epilogue warp handles
//   (router-gradient partial sums, reduced in a fixed order by the dw kernel)
// Padding rows produce exact zeros.  A: Dp/D2p K-major; B: W2/A2 MN-major.
// =====================================================================================
// 128-row tiles: its epilogue loads the saved G, U and activation from DRAM, and on
// 256-row tiles those loads no longer overlap the main loop (same-box 5.55 -> 6.77 ms
// at 65,536 tokens, E256).
constexpr bool kW2DgradWide = false;
// MX: W2 is MXFP4, decoded into the stage (MN-major boxes) by the epilogue warps; on
// 256-row tiles (the decoding warps are the epilogue warps, idle during the main loop
// only there, and each decoded weight tile then serves 256 rows instead of 128).
template <bool MX>
struct ProbW2DgradT {
  static constexpr bool kAmn = false, kBmn = true;
  static constexpr bool kWide = MX || kW2DgradWide;
  static constexpr bool kDecode = MX;
  static constexpr bool kMxMN = true;
  const uint8_t* S2q;  // MX: scales [E,H,I/32]
  CUtensorMap mW2q;    // MX: packed [E,H,I/2] bytes, box (128, 64, 1)
  // On the two-SM engine (each CTA copying its 128 rows of dY and its 128 of the tile's
  // 256 I columns with one 4D copy: 32 KB per SM per 64-wide K step instead of 48 KB)
  // this GEMM measured 5.23-5.25 ms against 4.86-4.88 ms here (65,536 tokens, E256,
  // same box, two alternations), and 5.58-5.64 against 5.02 with 8 epilogue warps per
  // CTA, and 5.23-5.26 against 4.84-4.85 with W2 copied as 8-row groups of chunk pairs
  // (the layout that brings the two-SM engine's plain GEMM with MN-major B from
  // 1,197-1,529 to 1,627-1,678 TFLOP/s), so the one-SM form stays.  That engine runs a
  // plain 8192^3 GEMM faster than the one-SM 128-row form (1,627-1,715 vs 1,430-1,517
  // TFLOP/s): the loss comes with this problem (its epilogue's DRAM loads and stores, its
  // grouped tiles), not with the engine; which of them was not isolated.  Clusters of
  // two CTAs on neighbouring row tiles, each copying half of the shared W2 tile and
  // multicasting it to both (a third fewer L2 reads), measured 5.08-5.10 against
  // 4.95-4.97 ms: the shared L2 reads are not what holds it.
  // 4 epilogue warps: with the fast silu they keep up with the main loop, and fewer
  // loads in flight leave the operand copies more of the memory system (same box:
  // 5.22 vs 5.36 ms with 8 warps, 65,536 tokens, E256); 256-row tiles need 8
  static constexpr int kEpiWarps = kWide ? 8 : 4;
  // router-gradient partial sums per row and column tile (one per epilogue column stripe)
  static constexpr int kPartsPerTile = kWide ? 1 : kEpiWarps / 4;
  CUtensorMap mDp, mD2p, mW2, mA2;  // Dp (H,P) box(64,128); D2p (r,P) box(64,128);
                                    // W2 (I,H,E), A2 (I,r,G): box(64,64,1), or 64-column
                                    // chunks box(64,64,4,1) with kMnChunkCopy
  CUtensorMap mdG, mdU;             // outputs (I,P), 32 x 32 store boxes (4 epilogue warps)
  PlanView pl;
  int* err;
  const float* topk_w;
  const uint16_t *G, *U;
  uint16_t *dG, *dU;
  float* part;
  int H, I, r;
  int act;      // 0 = SwiGLU, 1 = GeGLU
  float clamp;  // activation clamp (0 = none)
  __device__ int ntn() const { return cdiv(I, 256); }
  __device__ int nkr() const { return (r + 63) / 64; }
  __device__ int num_tiles() const {
    return (kWide ? pl.wtile_off[pl.G] : pl.offsets[pl.G] / 128) * ntn();
  }
  __device__ TileInfo tile(int t) const {  // column-tile-major inside each group
    TileInfo ti;
    const int nt = kWide ? wide_entry_decode(nmajor_wide_fetch(pl, t, ntn()), ti)
                         : nmajor_narrow_decode(nmajor_narrow_fetch(pl, t, ntn()), t, ntn(), ti);
    ti.n0 = nt * 256;
    ti.sub = nt;
    ti.nk = H / kBK + nkr();
    return ti;
  }
  __device__ void prefetch() const {
    tma_prefetch_map(&mDp);
    tma_prefetch_map(&mD2p);
    tma_prefetch_map(&mW2);
    tma_prefetch_map(&mA2);
  }
  __device__ void load(const TileInfo& ti, int ks, uint8_t* sa, uint8_t* sb, uint64_t* bar) const {
    const int nb = H / kBK;
    mbar_arrive_expect_tx(bar, ti.mh * kAStage128 + (MX && ks < nb ? 64 * 128 : 4 * 8192));
    if (ks < nb) {
      load_a_wide(ti, sa, &mDp, bar, ks * kBK);
      if (MX)  // 64 rows of W2 (h) x 256 packed columns (i)
        tma_load_3d(sb + kMxRaw, &mW2q, bar, ti.n0 / 2, ks * kBK, ti.g % pl.E);
      else
        if (kMnChunkCopy)
          tma_load_4d(sb, &mW2, bar, 0, ks * kBK, ti.n0 / 64, ti.g % pl.E);
        else
          for (int c = 0; c < 4; ++c) tma_load_3d(sb + c * 8192, &mW2, bar, ti.n0 + c * 64, ks * kBK, ti.g % pl.E);
    } else {
      const int kb = ks - nb;
      load_a_wide(ti, sa, &mD2p, bar, kb * kBK);
      if (kMnChunkCopy)
        tma_load_4d(sb, &mA2, bar, 0, kb * kBK, ti.n0 / 64, ti.g);
      else
        for (int c = 0; c < 4; ++c) tma_load_3d(sb + c * 8192, &mA2, bar, ti.n0 + c * 64, kb * kBK, ti.g);
    }
  }
  // MX, base K steps: box b holds W2[e][h][i] for i = n0 + 64 b.., h = 64 ks + (rho % 64)
  __device__ bool decodes(const TileInfo&, int ks) const { return MX && ks < H / kBK; }
  __device__ MxScales mx_scales(const TileInfo& ti, int ks) const {
    const int64_t so = ((int64_t)(ti.g % pl.E) * H + ks * kBK) * (I / 32) + ti.n0 / 32;
    const int boxes = (I - ti.n0) / 64;
    return MxScales{{S2q + so, S2q + so}, I / 32, {boxes < 4 ? boxes : 4, 0}};
  }
  __device__ MmaStep mma_step(const TileInfo&, int ks) const { return MmaStep{256, 0, 0, ks == 0}; }
  __device__ void epilogue(const TileInfo& ti, int row, uint32_t taddr, int c0, int cs, uint32_t* stg) const {
    const int64_t p = (int64_t)ti.m0 + row;
    const int rt = pl.route_of_row[p];
    const bool live = rt >= 0;
    const float w = live ? topk_w[rt] : 0.0f;
    const int y0 = (int)(p - (threadIdx.x & 31));  // warp's first row
    const int64_t base0 = (int64_t)y0 * I + ti.n0;
    // With 4 epilogue warps the staging slots of warps 4..7 are free: each warp keeps
    // its load-transposition buffer and gets a TMA-store ring in the slot 4 further on.
    constexpr bool kTmaOut = kEpiTmaStore && kEpiWarps == 4;
    TmaStoreRing out(stg + (kTmaOut ? 4 * kStgWordsPerWarp : 0));
    float dot = 0.0f;
    for (int c = c0; c < 256 && ti.n0 + c < I; c += cs) {
      // the chunk's saved G and U: coalesced loads, all in flight, then redistributed
      // so each lane holds its own row
      uint4 lg[4], lu[4];
      warp_load_rows_issue(G + base0 + c, I, lg);
      warp_load_rows_issue(U + base0 + c, I, lu);
      float q[32];
      tmem_ld32(taddr + c, q);
      float g[32], u[32];
      warp_rows_to_lane(lg, stg, g);
      warp_rows_to_lane(lu, stg, u);
      float og[32], ou[32];
      dot += act_bwd_chunk(act, clamp, q, g, u, w, live, og, ou);
      if (kTmaOut) {
        out.store_bf16(&mdG, ti.n0 + c, y0, og);
        out.store_bf16(&mdU, ti.n0 + c, y0, ou);
      } else {  // staged warp stores: the loads use the staging buffer
        warp_store_rows_bf16(dG + base0 + c, I, 32, og, 1.0f, stg);
        warp_store_rows_bf16(dU + base0 + c, I, 32, ou, 1.0f, stg);
      }
    }
    part[(p * ntn() + ti.sub) * kPartsPerTile + c0 / 32] = live ? dot : 0.0f;
  }
  __device__ void epilogue_empty(const TileInfo&, int, int, int) const {}
};
using ProbW2Dgrad = ProbW2DgradT<false>;

// =====================================================================================
// Backward -- expert-local A2 gradient, K-grouped over each group's rows:
//   dA2_ae = dZ2p^T Act  [r,I] fp32,  dZ2p = s * w * dyB2 of the row's token.
// M = r (one tile), N = I (tiles of 256), K = the group's padded rows (zero on padding).
// =====================================================================================
struct ProbDA2 {
  static constexpr bool kAmn = true, kBmn = true;
  static constexpr int kEpiWarps = 4;
  static constexpr bool kWide = false;
  CUtensorMap mdZ2p, mAct;  // dZ2p (r,P) box(64,64); Act (I,P) box(64,64)
  PlanView pl;
  int* err;
  float* dA2;
  int I, r;
  __device__ int ntn() const { return cdiv(I, 256); }
  __device__ int num_tiles() const { return pl.G * ntn(); }
  __device__ TileInfo tile(int t) const {
    const int q = t / ntn(), nt = t % ntn();  // plan slot of the group
    TileInfo ti;
    ti.g = group_weight_index(q, pl.A, pl.E);
    ti.m0 = 0;
    ti.mend = r;
    ti.n0 = nt * 256;
    ti.sub = 0;
    ti.k0 = pl.offsets[q];
    ti.nk = (pl.offsets[q + 1] - pl.offsets[q]) / kBK;
    return ti;
  }
  __device__ void prefetch() const {
    tma_prefetch_map(&mdZ2p);
    tma_prefetch_map(&mAct);
  }
  __device__ void load(const TileInfo& ti, int ks, uint8_t* sa, uint8_t* sb, uint64_t* bar) const {
    const int kt = ti.k0 + ks * kBK;
    mbar_arrive_expect_tx(bar, kAStage128 + 4 * 8192);
    tma_load_2d(sa, &mdZ2p, bar, 0, kt);
    tma_load_2d(sa + 8192, &mdZ2p, bar, 64, kt);
    for (int c = 0; c < 4; ++c) tma_load_2d(sb + c * 8192, &mAct, bar, ti.n0 + c * 64, kt);
  }
  __device__ MmaStep mma_step(const TileInfo&, int ks) const { return MmaStep{256, 0, 0, ks == 0}; }
  __device__ void epilogue(const TileInfo& ti, int row, uint32_t taddr, int c0, int cs, uint32_t* stg) const {
    const int rb = row - (threadIdx.x & 31);  // warp's first row
    float* o0 = dA2 + ((int64_t)ti.g * r + rb) * I + ti.n0;
    for (int c = c0; c < 256 && ti.n0 + c < I; c += cs) {
      float v[32];
      tmem_ld32(taddr + c, v);
      warp_store_rows_f32(o0 + c, I, r - rb, v, 1.0f, 32, stg);
    }
  }
  __device__ void epilogue_empty(const TileInfo& ti, int row, int c0, int cs) const {
    if (row >= r) return;
    const float z[32] = {};
    for (int c = c0; c < 256 && ti.n0 + c < I; c += cs)
      store_row_f32(dA2 + ((int64_t)ti.g * r + row) * I + ti.n0 + c, z, 0.f, 32);
  }
};

// =====================================================================================
// Backward B5 -- W13^T dgrad with the B1/B3 path:
//   dXp = dG W1_e + dU W3_e                 [P,H] bf16     (N tiles of 256, K = 2I)
//   dY13 = s * [dG B1_ae | dU B3_ae]        [P,2r] fp32    (one extra N tile)
// A: dG/dU K-major; B: W1/W3/B1/B3 MN-major.  In the extra tile dY1 accumulates
// in TMEM columns [0,r) and dY3 in [128,128+r).
// =====================================================================================
// MX: W1/W3 are MXFP4, decoded into the stage (MN-major boxes) by the epilogue warps.
template <bool MX>
struct ProbW13DgradT {
  static constexpr bool kAmn = false, kBmn = true;
  static constexpr int kEpiWarps = 8;
  static constexpr bool kWide = true;
  static constexpr bool kDecode = MX;
  static constexpr bool kMxMN = true;
  static constexpr bool kNoinlineEpilogue = MX;  // see epilogue_call
  const uint8_t *S1q, *S3q;  // MX: scales [E,I,H/32]
  CUtensorMap mW1q, mW3q;    // MX: packed [E,I,H/2] bytes, box (128, 64, 1)
  CUtensorMap mdXp;                          // output (H,P), 32 x 32 store boxes
  CUtensorMap mdG, mdU, mW1, mW3, mB1, mB3;  // dG/dU (I,P) box(64,128); W1/W3 (H,I,E) box(64,64,1)
                                             // or chunks box(64,64,4,1) (kMnChunkCopy);
                                             // B1/B3 (r,I,G) box(64,64,1)
  PlanView pl;
  int* err;
  uint16_t* dXp;
  float* dY13;
  int H, I, r;
  float s;
  __device__ int ntn() const { return cdiv(H, 256) + 1; }
  __device__ int num_tiles() const { return pl.wtile_off[pl.G] * ntn(); }
  __device__ TileInfo tile(int t) const {  // column-tile-major inside each group
    TileInfo ti;
    const int nt = wide_entry_decode(nmajor_wide_fetch(pl, t, ntn()), ti);
    ti.sub = nt == cdiv(H, 256);
    ti.n0 = ti.sub ? 0 : nt * 256;
    ti.nk = 2 * (I / kBK);
    return ti;
  }
  __device__ void prefetch() const {
    tma_prefetch_map(&mdG);
    tma_prefetch_map(&mdU);
    tma_prefetch_map(&mW1);
    tma_prefetch_map(&mW3);
    tma_prefetch_map(&mB1);
    tma_prefetch_map(&mB3);
  }
  __device__ void load(const TileInfo& ti, int ks, uint8_t* sa, uint8_t* sb, uint64_t* bar) const {
    const int nb = I / kBK;
    const bool second = ks >= nb;
    const int kk = (second ? ks - nb : ks) * kBK;
    if (!ti.sub) {
      mbar_arrive_expect_tx(bar, ti.mh * kAStage128 + (MX ? 64 * 128 : 4 * 8192));
      load_a_wide(ti, sa, second ? &mdU : &mdG, bar, kk);
      const int e = ti.g % pl.E;
      if (MX)  // 64 rows of W1 / W3 (i) x 256 packed columns (h)
        tma_load_3d(sb + kMxRaw, second ? &mW3q : &mW1q, bar, ti.n0 / 2, kk, e);
      else
        if (kMnChunkCopy)
          tma_load_4d(sb, second ? &mW3 : &mW1, bar, 0, kk, ti.n0 / 64, e);
        else
          for (int c = 0; c < 4; ++c) tma_load_3d(sb + c * 8192, second ? &mW3 : &mW1, bar, ti.n0 + c * 64, kk, e);
    } else {
      const int nbox = (round16(r) + 63) / 64;
      mbar_arrive_expect_tx(bar, ti.mh * kAStage128 + nbox * 8192);
      load_a_wide(ti, sa, second ? &mdU : &mdG, bar, kk);
      const CUtensorMap* mb = second ? &mB3 : &mB1;
      for (int c = 0; c < nbox; ++c) tma_load_3d(sb + c * 8192, mb, bar, c * 64, kk, ti.g);
    }
  }
  // MX, base tiles: box b holds W1[e][i][h] (W3 in the second half of K) for
  // h = n0 + 64 b.., i = 64 ks' + (rho % 64)
  __device__ bool decodes(const TileInfo& ti, int) const { return MX && !ti.sub; }
  __device__ MxScales mx_scales(const TileInfo& ti, int ks) const {
    const int nb = I / kBK;
    const bool second = ks >= nb;
    const int64_t row = (int64_t)(ti.g % pl.E) * I + (second ? ks - nb : ks) * kBK;
    const uint8_t* sq = (second ? S3q : S1q) + row * (H / 32) + ti.n0 / 32;
    const int boxes = (H - ti.n0) / 64;
    return MxScales{{sq, sq}, H / 32, {boxes < 4 ? boxes : 4, 0}};
  }
  __device__ MmaStep mma_step(const TileInfo& ti, int ks) const {
    const int nb = I / kBK;
    if (!ti.sub) return MmaStep{256, 0, 0, ks == 0};
    const bool second = ks >= nb;
    return MmaStep{round16(r), second ? 128 : 0, 0, ks == 0 || ks == nb};
  }
  __device__ void epilogue(const TileInfo& ti, int row, uint32_t taddr, int c0, int cs, uint32_t* stg) const {
    const int64_t p = (int64_t)ti.m0 + row;
    TmaStoreRing out(stg);  // before any use of the staging buffer
    if (!ti.sub) {
      const int y0 = (int)(p - (threadIdx.x & 31));  // warp's first row
      uint16_t* o0 = dXp + (int64_t)y0 * H + ti.n0;
      for (int c = c0; c < 256 && ti.n0 + c < H; c += cs) {
        float v[32];
        tmem_ld32(taddr + c, v);
        if (kEpiTmaStore)
          out.store_bf16(&mdXp, ti.n0 + c, y0, v);
        else
          warp_store_rows_bf16(o0 + c, H, 32, v, 1.0f, stg);
      }
    } else {
      float* o0 = dY13 + (p - (threadIdx.x & 31)) * (2 * r);  // warp's first row
      for (int hh = 0; hh < 2; ++hh) {
        for (int c = c0; c < r; c += cs) {
          float v[32];
          tmem_ld32(taddr + hh * 128 + c, v);
          warp_store_rows_f32(o0 + hh * r + c, 2 * r, 32, v, s, r - c < 32 ? r - c : 32, stg);
        }
      }
    }
  }
  __device__ void epilogue_empty(const TileInfo&, int, int, int) const {}
};
using ProbW13Dgrad = ProbW13DgradT<false>;

// =====================================================================================
// Backward -- expert-local B1/B3 gradients, K-grouped over each group's rows:
//   dB1_ae = dG^T Y1p,  dB3_ae = dU^T Y3p   [I,r] fp32   (s already inside Y13p)
// M = I (tiles of 128), N = round16(r), K = the group's padded rows.
// =====================================================================================
struct ProbDB13 {
  static constexpr bool kAmn = true, kBmn = true;
  static constexpr int kEpiWarps = 4;
  static constexpr bool kWide = false;
  CUtensorMap mdG, mdU, mY13p;  // dG/dU (I,P) box(64,64); Y13p (2r,P) box(64,64)
  PlanView pl;
  int* err;
  float *dB1, *dB3;
  int I, r;
  __device__ int ntm() const { return cdiv(I, 128); }
  __device__ int num_tiles() const { return 2 * pl.G * ntm(); }
  __device__ TileInfo tile(int t) const {
    const int which = t / (pl.G * ntm());
    const int rem = t % (pl.G * ntm());
    const int q = rem / ntm(), mt = rem % ntm();  // plan slot of the group
    TileInfo ti;
    ti.g = group_weight_index(q, pl.A, pl.E);
    ti.m0 = mt * 128;
    ti.mend = I;
    ti.n0 = 0;
    ti.sub = which;
    ti.k0 = pl.offsets[q];
    ti.nk = (pl.offsets[q + 1] - pl.offsets[q]) / kBK;
    return ti;
  }
  __device__ void prefetch() const {
    tma_prefetch_map(&mdG);
    tma_prefetch_map(&mdU);
    tma_prefetch_map(&mY13p);
  }
  __device__ void load(const TileInfo& ti, int ks, uint8_t* sa, uint8_t* sb, uint64_t* bar) const {
    const int kt = ti.k0 + ks * kBK;
    const int nbox = (round16(r) + 63) / 64;
    const CUtensorMap* ma = ti.sub ? &mdU : &mdG;
    mbar_arrive_expect_tx(bar, kAStage128 + nbox * 8192);
    tma_load_2d(sa, ma, bar, ti.m0, kt);
    tma_load_2d(sa + 8192, ma, bar, ti.m0 + 64, kt);
    for (int c = 0; c < nbox; ++c) tma_load_2d(sb + c * 8192, &mY13p, bar, ti.sub * r + c * 64, kt);
  }
  __device__ MmaStep mma_step(const TileInfo&, int ks) const { return MmaStep{round16(r), 0, 0, ks == 0}; }
  __device__ void epilogue(const TileInfo& ti, int row, uint32_t taddr, int c0, int cs, uint32_t* stg) const {
    const int64_t i0 = (int64_t)ti.m0 + row - (threadIdx.x & 31);  // warp's first row
    if (i0 >= I) return;                                              // rows past I (I % 128 == 64)
    float* o0 = (ti.sub ? dB3 : dB1) + ((int64_t)ti.g * I + i0) * r;
    for (int c = c0; c < r; c += cs) {
      float v[32];
      tmem_ld32(taddr + c, v);
      warp_store_rows_f32(o0 + c, r, 32, v, 1.0f, r - c < 32 ? r - c : 32, stg);
    }
  }
  __device__ void epilogue_empty(const TileInfo& ti, int row, int c0, int cs) const {
    const int64_t i = (int64_t)ti.m0 + row;
    if (i >= I) return;
    float* out = (ti.sub ? dB3 : dB1) + ((int64_t)ti.g * I + i) * r;
    const float z[32] = {};
    for (int c = c0; c < r; c += cs) store_row_f32(out + c, z, 0.f, r - c < 32 ? r - c : 32);
  }
};

// =====================================================================================
// Backward B6 (first half) -- grad-x through the shared A1/A3, once per token:
//   dXl_t = bf16( dY13w_t [A1_a; A3_a] )   [T,H]
// M = tokens of adapter a, N = H (tiles of 256), K = 2r (dY1 steps with A1, then dY3
// with A3).  A: dY13w K-major; B: (n=h, k=q) = A1[a][q][h], MN-major.  The source
// combine of the routed dXp rows is added by combine_rows.
// =====================================================================================
struct ProbA13Expand {
  static constexpr bool kAmn = false, kBmn = true;
  // 4 epilogue warps (TMA-store epilogue; same box: 0.147 vs 0.160 ms with 8)
  static constexpr int kEpiWarps = 4;
  static constexpr bool kWide = false;
  CUtensorMap mdY13w, mA1, mA3;  // dY13w (2r,T) box(64,128); A1/A3 (H,r,A) box(64,64,1)
  CUtensorMap mdXl;               // output (H,T), 32 x 32 store boxes
  PlanView pl;
  int* err;
  uint16_t* dXl;
  int H, r;
  __device__ int ntn() const { return cdiv(H, 256); }
  __device__ int nkr() const { return (r + 63) / 64; }
  __device__ int num_tiles() const { return pl.tok_tile[pl.A] * ntn(); }
  __device__ TileInfo tile(int t) const {
    const int mt = t / ntn(), nt = t % ntn();
    const int a = adapter_of_tile(pl, mt);
    TileInfo ti;
    ti.g = a;
    ti.m0 = pl.tok_off[a] + (mt - pl.tok_tile[a]) * 128;
    ti.mend = pl.tok_off[a + 1];
    ti.n0 = nt * 256;
    ti.sub = 0;
    ti.nk = 2 * nkr();
    ti.k0 = 0;
    return ti;
  }
  __device__ void prefetch() const {
    tma_prefetch_map(&mdY13w);
    tma_prefetch_map(&mA1);
    tma_prefetch_map(&mA3);
  }
  __device__ void load(const TileInfo& ti, int ks, uint8_t* sa, uint8_t* sb, uint64_t* bar) const {
    const int half = ks / nkr(), kb = ks % nkr();
    mbar_arrive_expect_tx(bar, kAStage128 + 4 * 8192);
    tma_load_2d(sa, &mdY13w, bar, half * r + kb * kBK, ti.m0);
    const CUtensorMap* m = half ? &mA3 : &mA1;
    for (int c = 0; c < 4; ++c) tma_load_3d(sb + c * 8192, m, bar, ti.n0 + c * 64, kb * kBK, ti.g);
  }
  __device__ MmaStep mma_step(const TileInfo&, int ks) const { return MmaStep{256, 0, 0, ks == 0}; }
  __device__ void epilogue(const TileInfo& ti, int row, uint32_t taddr, int c0, int cs, uint32_t* stg) const {
    const int64_t t0 = (int64_t)ti.m0 + row - (threadIdx.x & 31);  // warp's first row
    const int nvalid = (int)(ti.mend - t0 < 32 ? ti.mend - t0 : 32);
    TmaStoreRing out(stg);  // whole-box stores: see ProbB2Expand
    for (int c = c0; c < 256 && ti.n0 + c < H; c += cs) {
      float v[32];
      tmem_ld32(taddr + c, v);
      if (nvalid <= 0) continue;
      if (kEpiTmaStore)
        out.store_bf16(&mdXl, ti.n0 + c, (int)t0, v);
      else
        warp_store_rows_bf16(dXl + t0 * H + ti.n0 + c, H, nvalid, v, 1.0f, stg);
    }
  }
  __device__ void epilogue_empty(const TileInfo&, int, int, int) const {}
};

// =====================================================================================
// Backward -- shared A1/A3 gradients, per adapter over its tokens:
//   [dA1; dA3]_a = dY13w^T x   [2r,H] fp32
// M = 2r (tiles of 128), N = H (tiles of 256), K = tokens.  Both operands MN-major.
// Split over the token range like dB2: slice s writes dA1 rows to out1 and dA3
// rows to out3, each offset by s*split_stride.
// =====================================================================================
struct ProbDA13 {
  static constexpr bool kAmn = true, kBmn = true;
  static constexpr int kEpiWarps = 4;
  static constexpr bool kWide = false;
  CUtensorMap mdY13w, mx;  // dY13w (2r,T) box(64,64); x (H,T) box(64,64)
  PlanView pl;
  int* err;
  float *out1, *out3;  // dA1 / dA3, or the split partials
  int64_t split_stride;
  int H, r, split;
  __device__ int ntm() const { return (2 * r + 127) / 128; }
  __device__ int ntn() const { return cdiv(H, 256); }
  __device__ int num_tiles() const { return split * pl.A * ntm() * ntn(); }
  __device__ TileInfo tile(int t) const {
    const int per = ntm() * ntn();
    const int sp = t / (pl.A * per), ta = t % (pl.A * per);
    const int a = ta / per, rem = ta % per;
    const int mt = rem / ntn(), nt = rem % ntn();
    TileInfo ti;
    ti.g = a;
    ti.m0 = mt * 128;
    ti.mend = 2 * r;
    ti.n0 = nt * 256;
    ti.sub = sp;
    const int nk = (pl.tok_off[a + 1] - pl.tok_off[a] + kBK - 1) / kBK, cs = (nk + split - 1) / split;
    ti.k0 = pl.tok_off[a] + sp * cs * kBK;
    ti.nk = max(0, min(cs, nk - sp * cs));
    return ti;
  }
  __device__ void prefetch() const {
    tma_prefetch_map(&mdY13w);
    tma_prefetch_map(&mx);
  }
  __device__ void load(const TileInfo& ti, int ks, uint8_t* sa, uint8_t* sb, uint64_t* bar) const {
    const int kt = ti.k0 + ks * kBK;
    mbar_arrive_expect_tx(bar, kAStage128 + 4 * 8192);
    tma_load_2d(sa, &mdY13w, bar, ti.m0, kt);
    tma_load_2d(sa + 8192, &mdY13w, bar, ti.m0 + 64, kt);
    for (int c = 0; c < 4; ++c) tma_load_2d(sb + c * 8192, &mx, bar, ti.n0 + c * 64, kt);
  }
  __device__ MmaStep mma_step(const TileInfo&, int ks) const { return MmaStep{256, 0, 0, ks == 0}; }
  __device__ float* out_row(const TileInfo& ti, int m) const {
    const int64_t so = ti.sub * split_stride;
    return (m < r ? out1 + so + ((int64_t)ti.g * r + m) * H : out3 + so + ((int64_t)ti.g * r + (m - r)) * H) + ti.n0;
  }
  __device__ void epilogue(const TileInfo& ti, int row, uint32_t taddr, int c0, int cs, uint32_t* stg) const {
    const int m = ti.m0 + row;
    const bool ok = m < 2 * r;
    for (int c = c0; c < 256 && ti.n0 + c < H; c += cs) {
      float v[32];
      tmem_ld32(taddr + c, v);
      if (ok) store_row_f32(out_row(ti, m) + c, v, 1.0f, 32);
    }
  }
  __device__ void epilogue_empty(const TileInfo& ti, int row, int c0, int cs) const {
    const int m = ti.m0 + row;
    if (m >= 2 * r) return;
    const float z[32] = {};
    for (int c = c0; c < 256 && ti.n0 + c < H; c += cs) store_row_f32(out_row(ti, m) + c, z, 0.f, 32);
  }
};

// =====================================================================================
// Two-SM (cta_group::2) form of the W2 expert GEMM, for gemm_pair.cuh.
// A tile is 256 rows of one plan group: rank-0 CTA rows [m0, m0+128), rank-1 CTA
// rows [m0+128, m0+256) (absent on a group's odd last tile).  The N columns of every
// pair MMA are split in halves: rank v holds B columns [v*N/2, (v+1)*N/2).  Each
// CTA's accumulator has the same column meaning as the one-SM problem's, so the
// fused epilogues are inherited unchanged.
// =====================================================================================

// F4/F5: base tiles split 256 W2 rows 128 / 128; the A2 tile (N = round32(r))
// splits the A2 rows in halves of round32(r)/2 (rows past r read as zeros).
// Row-tile-major on the two-SM engine.  Column-tile-major (2,048-row chunks) halves
// its DRAM reads in a cold-cache capture (14.8 -> 8.0 GB per launch at 65,536 tokens)
// but measured slower inside the step (4.50 vs 4.39 ms, same box, two alternations).
constexpr bool kW2PairNmajor = false;
struct ProbW2Pair : ProbW2 {
  CUtensorMap mW2h, mA2h;  // W2 (I,H,E) box(64,128,1); A2 (I,r,G) box(64,round32(r)/2,1),
                           // in place of the one-SM mW2/mA2
  static constexpr bool kIssuerNeedsTile = true;  // the A2 tile has its own MMA N
  __device__ int num_tiles() const { return pl.wtile_off[pl.G] * ntn(); }
  __device__ int4 tile_fetch(int t) const {
    if (kW2PairNmajor) return nmajor_wide_fetch(pl, t, ntn());
    const int4 w = pl.wtile[t / ntn()];  // row-tile-major
    return make_int4(w.x, w.y, t % ntn(), 0);
  }
  __device__ TileInfo tile_at(int, int4 w) const {
    TileInfo ti;
    const int nt = wide_entry_decode(w, ti);
    ti.sub = nt == cdiv(H, 256);
    ti.n0 = ti.sub ? 0 : nt * 256;
    ti.nk = I / kBK;
    return ti;
  }
  __device__ TileInfo tile(int t) const { return tile_at(t, tile_fetch(t)); }
  __device__ void prefetch() const {
    tma_prefetch_map(&mAct);
    tma_prefetch_map(&mW2h);
    tma_prefetch_map(&mA2h);
  }
  __device__ uint32_t tx_bytes(const TileInfo& ti, int) const {
    return (uint32_t)(ti.mh * kAStage128 + (ti.sub ? round32(r) : 256) * 128);
  }
  __device__ void load_pair(const TileInfo& ti, int ks, int rank, uint8_t* sa, uint8_t* sb, uint32_t bar) const {
    if (rank < ti.mh) tma_load_2d_pair(sa, &mAct, bar, ks * kBK, ti.m0 + rank * 128);
    if (!ti.sub)
      tma_load_3d_pair(sb, &mW2h, bar, ks * kBK, ti.n0 + rank * 128, ti.g % pl.E);
    else
      tma_load_3d_pair(sb, &mA2h, bar, ks * kBK, rank * (round32(r) / 2), ti.g);
  }
  __device__ MmaStep mma_step(const TileInfo& ti, int ks) const {
    return MmaStep{ti.sub ? round32(r) : 256, 0, 0, ks == 0};
  }
};

// =====================================================================================
// Plain GEMM for engine self-tests: C[M,N] fp32 = sum_k A(m,k) B(n,k).
// A is [M,K] (K-major) or [K,M] (MN-major); B is [N,K] or [K,N].  M % 128 == 0,
// K % 64 == 0, N % 256 == 0 or N <= 256 with N % 16 == 0.
// =====================================================================================
template <bool AMN, bool BMN>
struct ProbPlain {
  static constexpr bool kAmn = AMN, kBmn = BMN;
  static constexpr int kEpiWarps = 4;
  static constexpr bool kWide = false;
  CUtensorMap mA, mB;  // K-major: (K,rows) box(64,128 | N); MN-major: (rows,K) box(64,64)
  int* err;
  float* C;
  int M, N, K;
  int starve;  // 1: issue no operand copy (the bounded waits must expire; error-path self-test)
  __device__ int tn() const { return N < 256 ? N : 256; }
  __device__ int ntn() const { return (N + 255) / 256; }
  __device__ int num_tiles() const { return M / 128 * ntn(); }
  __device__ TileInfo tile(int t) const {
    TileInfo ti;
    ti.m0 = t / ntn() * 128;
    ti.n0 = t % ntn() * 256;
    ti.mend = M;
    ti.g = 0;
    ti.sub = 0;
    ti.nk = K / kBK;
    ti.k0 = 0;
    return ti;
  }
  __device__ void prefetch() const {
    tma_prefetch_map(&mA);
    tma_prefetch_map(&mB);
  }
  __device__ void load(const TileInfo& ti, int ks, uint8_t* sa, uint8_t* sb, uint64_t* bar) const {
    if (starve) return;
    const int kt = ks * kBK;
    const int nbox = (tn() + 63) / 64;
    mbar_arrive_expect_tx(bar, kAStage128 + (BMN ? nbox * 8192 : tn() * 128));
    if (AMN) {
      tma_load_2d(sa, &mA, bar, ti.m0, kt);
      tma_load_2d(sa + 8192, &mA, bar, ti.m0 + 64, kt);
    } else {
      tma_load_2d(sa, &mA, bar, kt, ti.m0);
    }
    if (BMN) {
      for (int c = 0; c < nbox; ++c) tma_load_2d(sb + c * 8192, &mB, bar, ti.n0 + c * 64, kt);
    } else {
      tma_load_2d(sb, &mB, bar, kt, ti.n0);
    }
  }
  __device__ MmaStep mma_step(const TileInfo&, int ks) const { return MmaStep{tn(), 0, 0, ks == 0}; }
  __device__ void epilogue(const TileInfo& ti, int row, uint32_t taddr, int c0, int cs, uint32_t* stg) const {
    float* o0 = C + ((int64_t)ti.m0 + row - (threadIdx.x & 31)) * N + ti.n0;  // warp's first row
    for (int c = c0; c < tn(); c += cs) {
      float v[32];
      tmem_ld32(taddr + c, v);
      warp_store_rows_f32(o0 + c, N, 32, v, 1.0f, tn() - c < 32 ? tn() - c : 32, stg);
    }
  }
  __device__ void epilogue_empty(const TileInfo&, int, int, int) const {}
};

// Block-scaled plain GEMM (self-test of the native FP4 path):
//   C[M,N] = (Aq x 2^(As-127)) (Bq x 2^(Bs-127))^T   in fp32
// with Aq [M,K] E4M3 codes, Bq [N,K/2] packed E2M1 codes (low nibble = lower K), and
// As, Bs the UE8M0 bytes (one per 32 K elements) in the tile-major layout
// [rows/128][K/128][128 rows][4].  M % 128 == 0, N % 256 == 0, K % 128 == 0.
// L: layout of the scale words in tensor memory.
template <int L>
struct ProbPlainNv {
  static constexpr bool kAmn = false, kBmn = false, kWide = false, kNative = true;
  static constexpr int kEpiWarps = 8;
  static constexpr int kNvLayout = L;
  CUtensorMap mA, mB;  // Aq (K,M) bytes, box (128,128); Bq (K,N) E2M1, box (128,256)
  const uint8_t *As, *Bs;
  int* err;
  float* C;
  int M, N, K;
  __device__ int ntn() const { return N / 256; }
  __device__ int num_tiles() const { return M / 128 * ntn(); }
  __device__ TileInfo tile(int t) const {
    TileInfo ti;
    ti.m0 = t / ntn() * 128;
    ti.n0 = t % ntn() * 256;
    ti.mend = ti.m0 + 128;
    ti.g = 0;
    ti.sub = 0;
    ti.nk = K / 128;
    ti.k0 = 0;
    ti.mh = 1;
    return ti;
  }
  __device__ void prefetch() const {
    tma_prefetch_map(&mA);
    tma_prefetch_map(&mB);
  }
  __device__ void load(const TileInfo& ti, int ks, uint8_t* sa, uint8_t* sb, uint8_t* sf, uint64_t* bar) const {
    mbar_arrive_expect_tx(bar, 128 * 128 + 256 * 64 + kNvSfBytes);  // E2M1 boxes count packed bytes
    tma_load_2d(sa, &mA, bar, ks * 128, ti.m0);
    tma_load_3d(sb, &mB, bar, ks * 128, ti.n0, 0);
    const int64_t kt = K / 128;
    bulk_load(sf, As + ((int64_t)(ti.m0 >> 7) * kt + ks) * 512, 512, bar);
    bulk_load(sf + 512, Bs + ((int64_t)(ti.n0 >> 7) * kt + ks) * 512, 512, bar);
    bulk_load(sf + 1024, Bs + ((int64_t)((ti.n0 >> 7) + 1) * kt + ks) * 512, 512, bar);
  }
  __device__ bool native_step(const TileInfo&, int) const { return true; }
  __device__ MmaStep mma_step(const TileInfo&, int ks) const { return MmaStep{256, 0, 0, ks == 0}; }
  __device__ void epilogue(const TileInfo& ti, int row, uint32_t taddr, int c0, int cs, uint32_t*) const {
    float* o = C + ((int64_t)ti.m0 + row) * N + ti.n0;  // this thread's row (no staging: native shape)
    for (int c = c0; c < 256; c += cs) {
      float v[32];
      tmem_ld32(taddr + c, v);
#pragma unroll
      for (int j = 0; j < 8; ++j)
        *reinterpret_cast<float4*>(o + c + 4 * j) = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
    }
  }
  __device__ void epilogue_empty(const TileInfo&, int, int, int) const {}
};

// Plain GEMM on the two-SM engine (self-test): 256-row tiles, the MMA N (tn rounded
// up to 32) split in halves.  M % 128 == 0 (an odd last 128-row tile runs on the
// rank-0 CTA alone).
// CB (MN-major B, N % 256 == 0): each CTA's B half copied as 8-K-row groups of its two
// 64-column chunks (tmap_mn_k8), the layout the two-SM MMA reads at full rate.
template <bool AMN, bool BMN, bool CB = false>
struct ProbPlainPair : ProbPlain<AMN, BMN> {
  using Base = ProbPlain<AMN, BMN>;
  static constexpr bool kBmnCompact = BMN && CB;
  CUtensorMap mB5;  // kBmnCompact: B [K,N] (tmap_mn_k8, two chunks)
  // B maps: K-major box(64, tn/2); MN-major box(64,64) as in the one-SM form.
  __device__ int num_tiles() const { return (this->M + 255) / 256 * this->ntn(); }
  static constexpr bool kIssuerNeedsTile = false;
  __device__ int4 tile_fetch(int) const { return make_int4(0, 0, 0, 0); }
  __device__ TileInfo tile_at(int t, int4) const { return tile(t); }
  __device__ TileInfo tile(int t) const {
    TileInfo ti;
    ti.m0 = t / this->ntn() * 256;
    ti.mh = this->M - ti.m0 >= 256 ? 2 : 1;
    ti.n0 = t % this->ntn() * 256;
    ti.mend = this->M;
    ti.g = 0;
    ti.sub = 0;
    ti.nk = this->K / kBK;
    ti.k0 = 0;
    return ti;
  }
  __device__ int half_n() const { return round32(this->tn()) / 2; }
  __device__ int nbox() const { return (half_n() + 63) / 64; }
  __device__ uint32_t tx_bytes(const TileInfo& ti, int) const {
    return (uint32_t)(ti.mh * kAStage128 + 2 * (BMN ? nbox() * 8192 : half_n() * 128));
  }
  __device__ void load_pair(const TileInfo& ti, int ks, int rank, uint8_t* sa, uint8_t* sb, uint32_t bar) const {
    if (this->starve) return;
    const int kt = ks * kBK, mrow = ti.m0 + rank * 128, nc = ti.n0 + rank * half_n();
    if (rank < ti.mh) {
      if (AMN) {
        tma_load_2d_pair(sa, &this->mA, bar, mrow, kt);
        tma_load_2d_pair(sa + 8192, &this->mA, bar, mrow + 64, kt);
      } else {
        tma_load_2d_pair(sa, &this->mA, bar, kt, mrow);
      }
    }
    if (kBmnCompact) {
      tma_load_5d_pair(sb, &mB5, bar, 0, 0, nc / 64, kt / 8, 0);
    } else if (BMN) {
      for (int c = 0; c < nbox(); ++c) tma_load_2d_pair(sb + c * 8192, &this->mB, bar, nc + c * 64, kt);
    } else {
      tma_load_2d_pair(sb, &this->mB, bar, kt, nc);
    }
  }
  __device__ MmaStep mma_step(const TileInfo&, int ks) const { return MmaStep{round32(this->tn()), 0, 0, ks == 0}; }
};

}  // namespace moelora
