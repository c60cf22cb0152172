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
//   static constexpr bool kDecode;         B operand decoded from MXFP4 (wide problems only);
//   (kDecode only:)
//   static constexpr bool kMxMN;           layout of the packed rows (below)
//   bool  decodes(const TileInfo&, int ks) const;   false: the producer loads B with TMA
//   MxScales mx_scales(const TileInfo&, int ks) const;   where the stage's scale bytes are
//   and load() copies the stage's packed E2M1 rows with TMA into the last 12 KB of the
//   B buffer (kMxRaw), counted on the stage's full barrier
// An epilogue warp handles the 32-column chunks c = c0, c0 + cs, ... of its row.
//
// With kDecode the epilogue warps are also the decoders.  On 256-row tiles they are
// idle while the main loop runs (one accumulator, no overlap): for every K step of a
// tile they wait for the stage's full barrier (its A tile and its packed weight rows
// have landed), decode the packed rows into the stage's bf16 B tile (in the swizzled
// layout TMA would write) and arrive on the stage's decoded barrier, which the MMA
// waits on instead; after a tile's last K step they run its epilogue.  The packed
// rows travel by TMA with the rest of the stage, so the ring's depth hides their
// latency; the scale bytes (rows too narrow for TMA in general) are loaded by the
// decoding threads one K step ahead.
//
// Block-scaled FP4 problems (P::kNative): 128-row tiles with one 128 x 256
// accumulator (columns 0..255); tensor-memory columns 256.. hold each stage's scale
// words (kNvSfCols per stage).  On a native K step (K = 128) the A tile holds 128 rows
// of 128 E4M3 codes and the B tile 256 rows of 128 E2M1 codes, each code in its own
// byte position as TMA's 16U4_ALIGN16B type writes them (16 codes in 8 bytes, then 8
// bytes of gap); every row carries one UE8M0 scale per 32 K elements.  Such a copy
// counts its PACKED bytes on the stage barrier (64 per row of 128 codes), not the
// bytes it writes to shared memory (measured: expecting the latter never completes).
// The epilogue warps walk the K steps like decoders: for a native step they copy the
// stage's scale words (which the producer brought with the operands) into tensor
// memory and arrive on the stage's decoded barrier, which the MMA waits on; it then
// issues four kind::mxf8f6f4 MMAs of K = 32 (scale byte kk of each word for step kk).
// Other K steps of such a problem are ordinary BF16 steps.  Four stages of 48 KB
// (A 16 KB, B 32 KB) and four 1.5 KB blocks of scale words after them; no epilogue
// staging buffers (the epilogue stores rows from registers), which is what makes room
// for the fourth stage.
//   static constexpr bool kNative;
//   bool     native_step(const TileInfo&, int ks) const;
//   void     load(const TileInfo&, int ks, uint8_t* sA, uint8_t* sB, uint8_t* sSf, uint64_t* bar) const;
//            copies the step's scale words to sSf: 128 words of A rows 0..127, then 256
//            words of B rows 0..255 (one word = the step's 4 scale bytes)
//
// Operand tiles in shared memory use the 128-byte swizzle written by TMA:
//   A K-major : 128 rows x 128 B                         (one 16 KB box)
//   A MN-major: two boxes of 64 K-rows x 64 M, 8 KB apart
//   B K-major : N rows x 128 B
//   B MN-major: N/64 boxes of 64 K-rows x 64 N, 8 KB apart
#pragma once
#include <type_traits>

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

// P::kNative when the problem declares it, else false.
template <class P, class = void>
struct NativeOf : std::false_type {};
template <class P>
struct NativeOf<P, std::void_t<decltype(P::kNative)>> : std::integral_constant<bool, P::kNative> {};

// Per-problem pipeline shape.  Narrow problems: 128-row tiles, 4 stages of
// (A 16 KB + B 32 KB), two TMEM accumulators (the epilogue of one tile overlaps the
// main loop of the next).  Wide problems (P::kWide): 256-row tiles as two M=128
// MMAs sharing each B tile, 3 stages of (A 32 KB + B 32 KB), one accumulator pair
// using all 512 TMEM columns -- a third fewer operand bytes per FLOP streamed into
// the SM, at the price of an epilogue that no longer overlaps the main loop.
constexpr int kNvSfBytes = 384 * 4;  // scale words of one native stage
template <class P>
struct EngineShape {
  static constexpr bool kWide = P::kWide;
  static constexpr bool kNat = NativeOf<P>::value;
  static constexpr int kAStage = kWide ? 2 * 128 * 128 : 128 * 128;
  static constexpr int kStage = kAStage + kBStageBytes;
  static constexpr int kStages = kWide ? 3 : 4;
  static constexpr int kAccBufs = kWide || kNat ? 1 : 2;
  static constexpr int kSfArea = kNat ? kStages * kNvSfBytes : 0;  // after the ring
  static constexpr int kStg = kNat ? 0 : kStgBytes;                // epilogue staging, after that
  static constexpr int kBarOff = kStages * kStage + kSfArea + kStg;
  static constexpr int kSmem = kBarOff + 256 + 1024;  // barriers and TMEM slot, alignment slack
  static_assert(kStages * kStage <= 192 * 1024, "pipeline exceeds shared memory budget");
  static_assert(kSmem <= kGemmSmemBytes, "shared memory exceeds the launch size");
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

// ------------------------------------------------------------------ MXFP4 decoder
// The B tile of a stage is 256 rows of 64 bf16 in the 128-byte swizzle -- row rho at
// rho * 128, its 16-byte chunk c (elements 8c..8c+7) at chunk position c ^ (rho & 7)
// -- which is the layout TMA writes for a K-major tile of 256 rows and for four
// MN-major boxes of 64 x 64 (rho = 64 * box + K row) alike.  The producer copies the
// stage's packed rows (64 E2M1 codes = 32 bytes per B row, 8 KB) into the last 12 KB
// of the same buffer (kMxRaw):
//   K-major (kMxMN false): B row rho's 32 bytes at rho * 32;
//   MN-major (kMxMN true):  one box of 64 K rows x 128 bytes, B row rho = 64 b + kk's
//                           32 bytes at kk * 128 + 32 b.
// Each decoding thread (dt of NT = 256) takes two 32-element halves (items): it reads
// their packed bytes, the decoding warps meet at a reducing barrier (decoded rows
// 160..255 overwrite the packed bytes), and it writes 2 x 64 bytes of bf16.  The item
// mapping puts the 32 lanes of a warp on distinct banks for the reads and the writes.
//
// The barrier also carries each warp's "my bounded wait for this stage succeeded" and
// returns their AND to all of them, so the decoding warps always leave the loop
// together and every barrier they enter is entered by all of them: a hardware barrier
// with no way to be left waiting (one mbarrier-based alternative measured 7% slower).
constexpr int kMxRaw = 20480;  // offset of the packed rows in the 32 KB B buffer
template <bool MN>
__device__ __forceinline__ void mx_item(int dt, int j, int& rho, int& half) {
  half = dt & 1;
  rho = MN ? ((dt >> 1) & 3) * 64 + (dt >> 3) + 32 * j : (dt >> 1) + 128 * j;
}
// Where a stage's UE8M0 bytes are: B row rho's two bytes (one per 32-element half).
//   K-major: rows 0..127 at s[0] + rho * rs, rows 128..255 at s[1] + (rho - 128) * rs,
//            valid below lim[0] / lim[1] rows;
//   MN-major: row 64 b + kk at s[0] + kk * rs + 2 b, valid for b < lim[0].
// Rows past the tensor's edge (zeros from the zero-filled TMA copy) take scale 1.
struct MxScales {
  const uint8_t* s[2];
  int64_t rs;
  int lim[2];
};
// Read-only byte loads issued exactly where written (volatile asm keeps them ahead of
// the stage wait that follows, so they overlap the current step's decode).
__device__ __forceinline__ uint32_t ldg_issue_u8(const void* p) {
  uint32_t v;
  asm volatile("ld.global.nc.u8 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}
template <bool MN>
__device__ __forceinline__ void mx_load_scales(const MxScales& sc, int dt, uint32_t (&out)[2]) {
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    int rho, half;
    mx_item<MN>(dt, j, rho, half);
    const int h = MN ? 0 : rho >> 7;
    const int r = MN ? (rho & 63) : (rho & 127);
    const int b = MN ? rho >> 6 : 0;
    const bool ok = MN ? b < sc.lim[0] : r < (h ? sc.lim[1] : sc.lim[0]);
    const uint8_t* sp = (h ? sc.s[1] : sc.s[0]) + r * sc.rs + 2 * b + half;
    out[j] = ok ? ldg_issue_u8(sp) : 127u;
  }
}
// AND of `ok` over the NT threads of the decoding warps (named barrier 1); every one of
// them must execute it the same number of times.
template <int NT>
__device__ __forceinline__ bool decoders_agree(bool ok) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "bar.red.and.pred p, 1, %2, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"(ok ? 1u : 0u), "n"(NT)
      : "memory");
  return r != 0;
}
// Decodes a stage whose full barrier this warp has waited for (ok: the wait
// succeeded).  Returns false, with nothing written, unless every decoding warp's wait
// succeeded.
template <int NT, bool MN>
__device__ __forceinline__ bool mx_decode_stage(uint8_t* sb, int dt, const uint32_t (&scale)[2], bool ok) {
  static_assert(NT == 256, "two items per decoding thread");
  const uint8_t* raw = sb + kMxRaw;
  uint4 pk[2];
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    int rho, half;
    mx_item<MN>(dt, j, rho, half);
    const int off = MN ? (rho & 63) * 128 + (rho >> 6) * 32 + half * 16 : rho * 32 + half * 16;
    pk[j] = *reinterpret_cast<const uint4*>(raw + off);
  }
  // every packed byte read (by all decoding warps) before decoded rows overwrite them
  if (!decoders_agree<NT>(ok)) return false;
  // One choice per warp and stage between the permute route (scale bytes 2..252: all
  // but the extremes) and the exact fp32 route, so that the common case is one
  // straight-line block whose eight independent word decodes the compiler interleaves.
  const bool fast = scale[0] - 2u <= 250u && scale[1] - 2u <= 250u;
  uint4 o[2][4];
  if (__all_sync(0xffffffffu, fast)) {
    const uint32_t s2[2] = {(scale[0] << 7) * 0x10001u, (scale[1] << 7) * 0x10001u};
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      o[j][0] = mx_decode8_fast(pk[j].x, s2[j]);
      o[j][1] = mx_decode8_fast(pk[j].y, s2[j]);
      o[j][2] = mx_decode8_fast(pk[j].z, s2[j]);
      o[j][3] = mx_decode8_fast(pk[j].w, s2[j]);
    }
  } else {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      o[j][0] = mx_decode8_any(pk[j].x, scale[j]);
      o[j][1] = mx_decode8_any(pk[j].y, scale[j]);
      o[j][2] = mx_decode8_any(pk[j].z, scale[j]);
      o[j][3] = mx_decode8_any(pk[j].w, scale[j]);
    }
  }
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    int rho, half;
    mx_item<MN>(dt, j, rho, half);
#pragma unroll
    for (int w = 0; w < 4; ++w)
      *reinterpret_cast<uint4*>(sb + rho * 128 + (((half * 4 + w) ^ (rho & 7)) << 4)) = o[j][w];
  }
  return true;
}

// ------------------------------------------------------------------ block-scaled FP4
// Scale words of a native K step: 4 UE8M0 bytes (the step's four 32-element blocks,
// byte j for K elements 32j..32j+31) per operand row, in blocks of 128 rows (A rows
// 0..127, then B rows 0..127 and 128..255).  Inside a block the word of row i sits at
// position nv_word(i) = 4 (i % 32) + i / 32: 16-byte row j holds the words of rows j,
// 32 + j, 64 + j, 96 + j, which is what the tensor-memory layout below wants per lane.
constexpr int kNvSfCols = 12;  // per stage: A 4 columns, then B 8 columns
__host__ __device__ constexpr int nv_word(int i) { return 4 * (i & 31) + (i >> 5); }
// Layout of the scale words in tensor memory.  kNvLayoutGroups (the one the MMAs use):
// the words of operand row i sit in column i / 32 of that operand's block at lane i % 32
// of every lane quarter (each quarter holds all rows), written by the epilogue warps
// with tcgen05.st.  kNvLayoutCopy: the same layout, copied by the MMA thread itself with
// tcgen05.cp (no epilogue-warp work in the main loop).  kNvLayoutRows (self-test
// comparison only): row i at lane i % 128 of column i / 128.
constexpr int kNvLayoutGroups = 0, kNvLayoutRows = 1, kNvLayoutCopy = 2;
// The six words this thread (lane of a quarter; half 0 / 1 = the first / second warp
// of that quarter) stores for one step, from the stage's words sw.  kNvLayoutGroups:
// half 0 takes A columns 0..3 and B columns 0..1, half 1 B columns 2..7 (A/B row
// 32c + lane for column c); consecutive lanes read consecutive words.
template <int L>
__device__ __forceinline__ void nv_load_scales(const uint32_t* sw, int q, int half, int lane, uint32_t (&w)[6]) {
  const uint32_t* sa = sw;
  const uint32_t* sb = sw + 128;
  if (L == kNvLayoutGroups) {
    if (half == 0) {
#pragma unroll
      for (int c = 0; c < 4; ++c) w[c] = sa[nv_word(32 * c + lane)];
#pragma unroll
      for (int c = 0; c < 2; ++c) w[4 + c] = sb[nv_word(32 * c + lane)];
    } else {
#pragma unroll
      for (int c = 2; c < 8; ++c) w[c - 2] = sb[128 * (c >> 2) + nv_word(32 * (c & 3) + lane)];
    }
  } else {
    const int row = 32 * q + lane;
    w[0] = sa[nv_word(row)];
    w[1] = sb[nv_word(row)];
    w[2] = sb[128 + nv_word(row)];
    w[3] = w[4] = w[5] = 0;
  }
}
// Stores them at the stage's scale columns (sf: tensor-memory address of column 0 of
// the stage's block, lane 0) in this warp's lane quarter.
template <int L>
__device__ __forceinline__ void nv_store_scales(uint32_t sf, int q, int half, const uint32_t (&w)[6]) {
  const uint32_t qa = sf + ((uint32_t)(32 * q) << 16);
  if (L == kNvLayoutGroups) {
    if (half == 0) {
      tmem_st4(qa, w[0], w[1], w[2], w[3]);
      tmem_st2(qa + 4, w[4], w[5]);
    } else {
      tmem_st2(qa + 6, w[0], w[1]);
      tmem_st4(qa + 8, w[2], w[3], w[4], w[5]);
    }
  } else if (half == 0) {
    tmem_st4(qa, w[0], w[0], w[0], w[0]);
    tmem_st2(qa + 4, w[1], w[2]);
  }
  tmem_wait_st();
}

// P::kNoinlineEpilogue when the problem declares it, else false (see epilogue_call).
template <class P, class = void>
struct NoinlineEpilogueOf : std::false_type {};
template <class P>
struct NoinlineEpilogueOf<P, std::void_t<decltype(P::kNoinlineEpilogue)>>
    : std::integral_constant<bool, P::kNoinlineEpilogue> {};

// P::kDecode when the problem declares it, else false.
template <class P, class = void>
struct DecodeOf : std::false_type {};
template <class P>
struct DecodeOf<P, std::void_t<decltype(P::kDecode)>> : std::integral_constant<bool, P::kDecode> {};
// P::kNvLayout (self-test problems) or the layout the MMAs use.
template <class P, class = void>
struct NvLayoutOf : std::integral_constant<int, kNvLayoutGroups> {};
template <class P>
struct NvLayoutOf<P, std::void_t<decltype(P::kNvLayout)>> : std::integral_constant<int, P::kNvLayout> {};
template <class P>
constexpr int gemm_threads() {
  return 64 + 32 * P::kEpiWarps;
}

// The epilogue as a separately compiled call (P::kNoinlineEpilogue), for kernels whose
// epilogue warps also decode: the decode loop and the epilogue then get their own
// register allocations; the call saves the loop's live registers once per tile.
// Measured per problem (MXFP4 base, 65,536 tokens, E256): the W13 dgrad 45.8 -> 29.5
// ms with the call (global-load decoders); W13 (37.0 -> 56.5 ms then, 20.3 -> 22.0 ms
// with the TMA-fed decoders) and the W2 dgrad (11.3 -> 19.7) keep the epilogue inline.
template <class P>
__device__ __noinline__ void epilogue_call(const P& p, const TileInfo& ti, int row, uint32_t taddr, int c0, int cs,
                                           uint32_t* stg) {
  p.epilogue(ti, row, taddr, c0, cs, stg);
}

template <class P>
__global__ void __launch_bounds__(gemm_threads<P>(), 1) gemm_kernel(const __grid_constant__ P p) {
  using S = EngineShape<P>;
  static_assert(P::kEpiWarps == 4 || P::kEpiWarps == 8, "4 or 8 epilogue warps");
  static_assert(!P::kWide || (P::kEpiWarps == 8 && !P::kAmn), "wide tiles: 8 epilogue warps, K-major A");
  static_assert(!DecodeOf<P>::value || P::kWide, "decoding epilogue warps need 256-row tiles");
  static_assert(!NativeOf<P>::value || (!P::kWide && !P::kAmn && !P::kBmn && !DecodeOf<P>::value && P::kEpiWarps == 8),
                "block-scaled problems: 128-row tiles, K-major operands, 8 epilogue warps");
  static_assert(!NativeOf<P>::value || kAccCols + S::kStages * kNvSfCols <= 2 * kAccCols, "scale words exceed TMEM");
  // The epilogue warps walk the K steps (and the MMA waits for them) in decoding and
  // block-scaled problems -- unless the MMA thread copies the scale words itself.
  constexpr bool kNvCopy = NativeOf<P>::value && NvLayoutOf<P>::value == kNvLayoutCopy;
  constexpr bool kWalk = DecodeOf<P>::value || (NativeOf<P>::value && !kNvCopy);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S::kBarOff);
  uint64_t* empty = full + S::kStages;
  uint64_t* tfull = empty + S::kStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* dec = tempty + 2;  // kDecode: the stage's B tile has been decoded
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(dec + S::kStages);
  uint32_t* stg_base = reinterpret_cast<uint32_t*>(smem + S::kStages * S::kStage + S::kSfArea);
  uint8_t* sf_base = smem + S::kStages * S::kStage;  // native: scale words of stage s at + s * kNvSfBytes
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int* err = p.err;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
      mbar_init(&dec[s], P::kEpiWarps);
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
          if constexpr (NativeOf<P>::value)
            p.load(ti, ks, sa, sa + S::kAStage, sf_base + s * kNvSfBytes, &full[s]);
          else
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
          if (!mbar_wait(kWalk ? &dec[s] : &full[s], ph, err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const MmaStep st = p.mma_step(ti, ks);
          const uint32_t sa = smem_u32(smem + s * S::kStage);
          const uint32_t sb = sa + S::kAStage + (uint32_t)st.b_off;
          if constexpr (NativeOf<P>::value) {
            if (p.native_step(ti, ks)) {
              // 128 K elements of one-byte codes: four K = 32 steps, 32 bytes apart,
              // step kk using byte kk of every scale word
              const uint32_t sfa = tmem_base + (uint32_t)(kAccCols + s * kNvSfCols);
              if constexpr (kNvCopy) {
                // the stage's three 512-byte blocks of words (A, B rows 0..127, B rows
                // 128..255) into columns 0..3, 4..7, 8..11 of the stage's scale block
                const uint32_t sw = smem_u32(sf_base + s * kNvSfBytes);
#pragma unroll
                for (int b = 0; b < 3; ++b) tmem_cp_32x128b_x4(sfa + 4 * b, plain_desc(sw + 512 * b, 128, 128));
              }
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                mma_mx(d + (uint32_t)st.col, sw128_desc(sa + kk * 32, 16, 1024), sw128_desc(sb + kk * 32, 16, 1024),
                       idesc_mx_f32(128, st.n, kMxTypeE4M3, kMxTypeE2M1, kk, kk), sfa, sfa + 4,
                       (st.first && kk == 0) ? 0u : 1u);
              mma_commit(&empty[s]);
              if (++s == S::kStages) {
                s = 0;
                ph ^= 1u;
              }
              continue;
            }
          }
          const uint32_t idesc = idesc_bf16_f32(128, st.n, P::kAmn, P::kBmn);
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
    // The epilogue of one tile with K steps; false if a bounded wait gave up.
    auto run_epilogue = [&](const TileInfo& ti) -> bool {
      if (!__all_sync(0xffffffffu, mbar_wait(&tfull[acc], aph, err))) return false;
      tc_fence_after();
      if (!S::kWide || half < ti.mh) {
        const uint32_t col = (uint32_t)(S::kWide ? half * kAccCols : acc * kAccCols);
        const uint32_t taddr = tmem_base + col + ((uint32_t)(q * 32) << 16);
        uint32_t* stg = stg_base + (warp - 2) * kStgWordsPerWarp;
        if constexpr (NoinlineEpilogueOf<P>::value)
          epilogue_call(p, ti, row, taddr, c0, cs, stg);
        else
          p.epilogue(ti, row, taddr, c0, cs, stg);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[acc]);
      if (++acc == S::kAccBufs) {
        acc = 0;
        aph ^= 1u;
      }
      return true;
    };
    if constexpr (kWalk) {
      // Decode every K step of this CTA's tiles (in the producer's order), or write
      // its scale words, then run each tile's epilogue after its last step.  Tiles
      // without K steps have nothing to decode and no accumulator; they get
      // epilogue_empty.
      constexpr bool kNat = NativeOf<P>::value;
      constexpr int kNvL = NvLayoutOf<P>::value;
      constexpr int kPre = 2;  // decoders: scale bytes loaded one step ahead per thread
      constexpr int NT = 32 * P::kEpiWarps;
      const int dt = threadIdx.x - 64;  // decoder thread 0..NT-1
      int t = blockIdx.x, ks = 0;
      bool fresh = true;  // tile t not fetched yet
      TileInfo ti{};
      auto next = [&]() -> bool {  // advance (t, ks) to the next K step; false at the end
        if (!fresh) {
          if (++ks < ti.nk) return true;
          t += gridDim.x;
        }
        fresh = false;
        for (; t < ntiles; t += gridDim.x) {
          ti = p.tile(t);
          if (ti.nk > 0) {
            ks = 0;
            return true;
          }
          p.epilogue_empty(ti, row, c0, cs);
        }
        ti.nk = 0;  // exhausted: every later call returns false too
        return false;
      };
      // whether step (ti, ks) needs the walkers' work, and its words loaded ahead
      auto step_work = [&]() -> bool {
        if constexpr (kNat)
          return p.native_step(ti, ks);
        else
          return p.decodes(ti, ks);
      };
      auto load_pre = [&](uint32_t (&w)[kPre]) {
        if constexpr (!kNat) mx_load_scales<P::kMxMN>(p.mx_scales(ti, ks), dt, w);
      };
      int s = 0;
      uint32_t ph = 0;
      uint32_t sc[kPre];  // the current step's scale bytes (two items) or words
#pragma unroll
      for (int i = 0; i < kPre; ++i) sc[i] = 127u;
      bool have = next();
      bool cdec = have && step_work();
      if (cdec) load_pre(sc);
      while (have) {
        // The next step's scale bytes are loaded before this step is decoded; after a
        // tile's last step the iterator moves on only once the epilogue has run (the
        // epilogue needs the registers).
        const bool last = ks == ti.nk - 1;
        uint32_t nsc[kPre];
#pragma unroll
        for (int i = 0; i < kPre; ++i) nsc[i] = 127u;
        bool ndec = false;
        if (!last) {
          next();  // ks + 1 of the same tile
          ndec = step_work();
          if (ndec) load_pre(nsc);
        }
        const bool got = __all_sync(0xffffffffu, mbar_wait(&full[s], ph, err));
        if constexpr (kNat) {
          // Each warp writes its own lane quarter: no barrier between the warps, and a
          // warp whose wait gave up simply leaves (the MMA's wait then gives up too).
          if (!got) break;
          if (cdec) {
            uint32_t w[6];
            nv_load_scales<kNvL>(reinterpret_cast<const uint32_t*>(sf_base + s * kNvSfBytes), q, half, lane, w);
            nv_store_scales<kNvL>(tmem_base + (uint32_t)(kAccCols + s * kNvSfCols), q, half, w);
          }
          tc_fence_before();
        } else {
          // Steps that decode agree inside mx_decode_stage; the others here.  Either
          // way all decoding warps pass the same barriers and leave the loop together.
          if (cdec) {
            if (!mx_decode_stage<NT, P::kMxMN>(smem + s * S::kStage + S::kAStage, dt, sc, got)) break;
          } else if (!decoders_agree<NT>(got)) {
            break;
          }
          fence_proxy_async_smem();  // generic-proxy stores before the MMA's reads
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&dec[s]);
        if (++s == S::kStages) {
          s = 0;
          ph ^= 1u;
        }
        if (last) {
          if constexpr (kNat) {
            if (!run_epilogue(ti)) break;
          } else {
            if (!decoders_agree<NT>(run_epilogue(ti))) break;
          }
          have = next();
          ndec = have && step_work();
          if (ndec) load_pre(nsc);
        }
#pragma unroll
        for (int i = 0; i < kPre; ++i) sc[i] = nsc[i];
        cdec = ndec;
      }
    } else {
      for (int t = blockIdx.x; t < ntiles; t += gridDim.x) {
        const TileInfo ti = p.tile(t);
        if (ti.nk == 0) {
          p.epilogue_empty(ti, row, c0, cs);
          continue;
        }
        if (!run_epilogue(ti)) break;
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
    cudaError_t e =
        cudaFuncSetAttribute(gemm_kernel<P>, cudaFuncAttributeMaxDynamicSharedMemorySize, EngineShape<P>::kSmem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  if (max_tiles <= 0) return cudaSuccess;
  const int grid = max_tiles < num_sms ? max_tiles : num_sms;
  prof_begin(slot, stream);
  gemm_kernel<P><<<grid, gemm_threads<P>(), EngineShape<P>::kSmem, stream>>>(p);
  prof_end(slot, stream);
  return cudaGetLastError();
}

}  // namespace moelora
