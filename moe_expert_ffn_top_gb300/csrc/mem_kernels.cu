// HBM-bound kernels of the MoE side-LoRA path: routed-row gathers (with zeroed
// padding rows, so allocator garbage can never reach a shared reduction, the
// padding rule of "feat(mega): add fused shared side-LoRA kernels", Summary) and
// per-token reductions over the k
// routes of a token (fixed slot order, fp32, one bf16 rounding).
// All use 16-byte vector accesses, one warp per row, grid-stride over rows.
#include <cuda_fp16.h>

#include "launch.h"
#include "prof.h"

namespace moelora {

namespace {

constexpr int kThreads = 256;
// 16-byte loads per lane in flight per pass of the routed-row scatters (4,096 bf16
// columns: a whole production-width row)
constexpr int kGatherVec = 16;

__device__ __forceinline__ void copy_row_or_zero(uint16_t* dst, const uint16_t* src, int n, int lane) {
  // n bf16 (multiple of 8), 16 B per lane per step
  for (int c = lane * 8; c < n; c += 32 * 8) {
    uint4 v = src ? *reinterpret_cast<const uint4*>(src + c) : make_uint4(0, 0, 0, 0);
    *reinterpret_cast<uint4*>(dst + c) = v;
  }
}

// Zero the padding rows of each group (rows [offsets[g] + counts[g], offsets[g+1]))
// in up to two routed-row buffers; one warp per padding row.
__device__ __forceinline__ void zero_padding_rows(const PlanView& pl, uint16_t* a, int na, uint16_t* b, int nb) {
  const int lane = threadIdx.x & 31;
  const int warps_per_block = blockDim.x >> 5, wib = threadIdx.x >> 5;
  for (int g = blockIdx.x; g < pl.G; g += gridDim.x) {
    const int beg = pl.offsets[g] + pl.counts[g], end = pl.offsets[g + 1];
    for (int64_t p = beg + wib; p < end; p += warps_per_block) {
      copy_row_or_zero(a + p * na, nullptr, na, lane);
      if (b) copy_row_or_zero(b + p * nb, nullptr, nb, lane);
    }
  }
}

// Forward routed rows by scatter: one warp per token reads its x row (and Y13 row)
// once and writes a copy to each of the token's routed rows; padding rows are
// zeroed.  Reads T*H instead of k*T*H elements compared with a per-row gather.
__global__ void gather_fwd_kernel(PlanView pl, const uint16_t* __restrict__ x, const uint16_t* __restrict__ Y13,
                                  uint16_t* __restrict__ Xp, uint16_t* __restrict__ Y13p, int H, int r2) {
  const int lane = threadIdx.x & 31;
  const int64_t w0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int k = pl.k;
  for (int64_t t = w0; t < pl.T; t += nw) {
    const int* rows = pl.row_of_route + t * k;
    for (int c0 = 0; c0 < H; c0 += 32 * 8 * kGatherVec) {  // kGatherVec x 16 B per lane and pass
      uint4 v[kGatherVec];
#pragma unroll
      for (int i = 0; i < kGatherVec; ++i) {
        const int c = c0 + (i * 32 + lane) * 8;
        v[i] = c < H ? __ldg(reinterpret_cast<const uint4*>(x + t * H + c)) : make_uint4(0, 0, 0, 0);
      }
      for (int j = 0; j < k; ++j) {
        const int R = rows[j];
        if (R < 0) continue;
#pragma unroll
        for (int i = 0; i < kGatherVec; ++i) {
          const int c = c0 + (i * 32 + lane) * 8;
          if (c < H) *reinterpret_cast<uint4*>(Xp + (int64_t)R * H + c) = v[i];
        }
      }
    }
    for (int c = lane * 8; c < r2; c += 32 * 8) {
      const uint4 y = __ldg(reinterpret_cast<const uint4*>(Y13 + t * r2 + c));
      for (int j = 0; j < k; ++j) {
        const int R = rows[j];
        if (R >= 0) *reinterpret_cast<uint4*>(Y13p + (int64_t)R * r2 + c) = y;
      }
    }
  }
  zero_padding_rows(pl, Xp, H, Y13p, r2);
}

// ---------------------------------------------------------------- MXFP8 routed rows
// One MXFP8 block of 32 bf16 (four 16-byte words): mxfp8_block_f32 on their values.
__device__ __forceinline__ uint32_t mxfp8_block(const uint4 (&v)[4], uint4 (&codes)[2]) {
  float f[32];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      f[8 * i + 2 * j] = __uint_as_float(w[j] << 16);
      f[8 * i + 2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
    }
  }
  return mxfp8_block_f32(f, codes);
}

// Forward routed rows for the native FP4 forward, by scatter like gather_fwd_kernel:
// one warp per token quantises its x row once to MXFP8 (lane = one 32-element block)
// and writes the codes to each routed row of Xq [P,H], the scale bytes to Xs in the
// tile-major layout [P/128][H/128][128 rows][4 blocks] (one 4-byte word per row and
// 128-wide K step), and the token's Y13 row to Y13p.  Padding rows get zero codes and
// scale bytes 127.
__global__ void gather_fwd_mxfp8_kernel(PlanView pl, const uint16_t* __restrict__ x,
                                        const uint16_t* __restrict__ Y13, uint8_t* __restrict__ Xq,
                                        uint8_t* __restrict__ Xs, uint16_t* __restrict__ Y13p, int H, int r2) {
  const int lane = threadIdx.x & 31;
  const int64_t w0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int k = pl.k, ks_per_row = H / 128;
  for (int64_t t = w0; t < pl.T; t += nw) {
    const int* rows = pl.row_of_route + t * k;
    for (int b0 = 0; b0 < H / 32; b0 += 32) {  // 32 blocks of 32 per pass
      const int blk = b0 + lane;
      const bool on = blk < H / 32;
      uint4 v[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        v[i] = on ? __ldg(reinterpret_cast<const uint4*>(x + t * H + blk * 32 + 8 * i)) : make_uint4(0, 0, 0, 0);
      uint4 codes[2];
      const uint32_t sb = mxfp8_block(v, codes);
      // the 4 scale bytes of one K step (blocks 4j..4j+3) as one word, on lane 4j; in
      // its 512-byte block the word of row i sits at 4 (i % 32) + i / 32
      const uint32_t word = sb | (__shfl_down_sync(0xffffffffu, sb, 1) << 8) |
                            (__shfl_down_sync(0xffffffffu, sb, 2) << 16) | (__shfl_down_sync(0xffffffffu, sb, 3) << 24);
      for (int j = 0; j < k; ++j) {
        const int R = rows[j];
        if (R < 0 || !on) continue;
        uint4* dst = reinterpret_cast<uint4*>(Xq + (int64_t)R * H + blk * 32);
        dst[0] = codes[0];
        dst[1] = codes[1];
        if ((lane & 3) == 0)
          *reinterpret_cast<uint32_t*>(Xs + ((int64_t)(R >> 7) * ks_per_row + (blk >> 2)) * 512 +
                                       (4 * (R & 31) + ((R >> 5) & 3)) * 4) = word;
      }
    }
    for (int c = lane * 8; c < r2; c += 32 * 8) {
      const uint4 y = __ldg(reinterpret_cast<const uint4*>(Y13 + t * r2 + c));
      for (int j = 0; j < k; ++j) {
        const int R = rows[j];
        if (R >= 0) *reinterpret_cast<uint4*>(Y13p + (int64_t)R * r2 + c) = y;
      }
    }
  }
  // padding rows: zero codes (H bytes = H/2 bf16 of zeros) and neutral scale words
  const int wib = threadIdx.x >> 5, wpb = blockDim.x >> 5;
  for (int g = blockIdx.x; g < pl.G; g += gridDim.x) {
    const int beg = pl.offsets[g] + pl.counts[g], end = pl.offsets[g + 1];
    for (int64_t p = beg + wib; p < end; p += wpb) {
      copy_row_or_zero(reinterpret_cast<uint16_t*>(Xq + p * H), nullptr, H / 2, lane);
      copy_row_or_zero(Y13p + p * r2, nullptr, r2, lane);
      for (int j = lane; j < ks_per_row; j += 32)
        *reinterpret_cast<uint32_t*>(Xs + ((p >> 7) * ks_per_row + j) * 512 + (4 * (p & 31) + ((p >> 5) & 3)) * 4) =
            0x7F7F7F7Fu;
    }
  }
}

// Router-weight gradient of the native FP4 forward, whose down base product ran on
// q8(Act), so that <Q, a> no longer equals <dy, o>: from the forward's saved rows,
//   dw[t,j] = <dy_t, O[row]> + s <dyB2_t, Z2[row]>   (fp32; 0 for a masked slot)
// with row = row_of_route[t*k + j] (o = O + s B2 Z2, and dyB2 = dy B2).  One warp per
// token; H % 256 == 0 is not needed (8 columns per lane and step, H % 8 == 0).
// Measured: 0.80 ms at 65,536 tokens (O and dy read at the copy rate); fusing it into
// the dy gather, which holds each dy row in registers, took that kernel from 0.64 to
// 3.31 ms (246 registers: one block per SM, the per-route reductions serialised).
__global__ void dw_from_o_kernel(PlanView pl, const uint16_t* __restrict__ dy, const uint16_t* __restrict__ dyB2,
                                 const uint16_t* __restrict__ O, const uint16_t* __restrict__ Z2, int H, int r,
                                 float s, float* __restrict__ dw) {
  const int lane = threadIdx.x & 31;
  const int64_t w0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int k = pl.k;
  for (int64_t t = w0; t < pl.T; t += nw) {
    for (int j = 0; j < k; ++j) {
      const int R = pl.row_of_route[t * k + j];
      float acc = 0.f;
      if (R >= 0) {
        for (int c = lane * 8; c < H; c += 256) {
          const uint4 a = __ldg(reinterpret_cast<const uint4*>(dy + t * H + c));
          const uint4 b = __ldg(reinterpret_cast<const uint4*>(O + (int64_t)R * H + c));
          const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
          for (int q = 0; q < 4; ++q)
            acc += bf16_lo(aw[q]) * bf16_lo(bw[q]) + bf16_hi(aw[q]) * bf16_hi(bw[q]);
        }
        float side = 0.f;
        for (int q = lane; q < r; q += 32)
          side += __uint_as_float((uint32_t)dyB2[t * r + q] << 16) * __uint_as_float((uint32_t)Z2[(int64_t)R * r + q] << 16);
        acc += s * side;
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
      if (lane == 0) dw[t * k + j] = acc;
    }
  }
}

// Scale bytes [rows, K/32] (row-major, one per 32 K elements) to the tile-major layout
// [rows/128][K/128][32][4][4]: the 4 bytes of one 128-wide K step of a row become one
// word, the 128 words of a row tile for one K step 512 contiguous bytes (what a
// native GEMM stage copies), row i's word at position 4 (i % 32) + i / 32 of them.
// rows % 128 == 0, K % 128 == 0.
__global__ void scales_to_tiles_kernel(const uint8_t* __restrict__ S, int64_t rows, int kt,
                                       uint8_t* __restrict__ St) {
  const int64_t n = rows * kt;  // words
  for (int64_t w = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; w < n; w += (int64_t)gridDim.x * blockDim.x) {
    const int64_t i = w & 127, j = (w >> 7) % kt, rt = (w >> 7) / kt;  // row in tile, K step, row tile
    const int64_t row = rt * 128 + i;
    *reinterpret_cast<uint32_t*>(St + (w & ~(int64_t)127) * 4 + (4 * (i & 31) + (i >> 5)) * 4) =
        __ldg(reinterpret_cast<const uint32_t*>(S + row * kt * 4 + j * 4));
  }
}

// The same MXFP8 quantisation on its own: one warp per row of x [rows, n], one
// 32-element block per lane, codes [rows, n] and scale bytes [rows, n/32] row-major.
__global__ void quant_mxfp8_kernel(const uint16_t* __restrict__ x, int64_t rows, int n, uint8_t* __restrict__ codes,
                                   uint8_t* __restrict__ scales) {
  const int lane = threadIdx.x & 31;
  const int64_t w0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int nb = n / 32;
  for (int64_t t = w0; t < rows; t += nw) {
    for (int blk = lane; blk < nb; blk += 32) {
      uint4 v[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) v[i] = __ldg(reinterpret_cast<const uint4*>(x + t * n + blk * 32 + 8 * i));
      uint4 c[2];
      const uint32_t sb = mxfp8_block(v, c);
      uint4* dst = reinterpret_cast<uint4*>(codes + t * n + blk * 32);
      dst[0] = c[0];
      dst[1] = c[1];
      scales[t * nb + blk] = (uint8_t)sb;
    }
  }
}

// one warp per token; lane covers r/32.. columns (r <= 128 -> up to 4 per lane)
__global__ void z2w_kernel(PlanView pl, const uint16_t* __restrict__ Z2, const float* __restrict__ topk_w,
                           uint16_t* __restrict__ Z2w, int r) {
  const int lane = threadIdx.x & 31;
  const int64_t w0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t t = w0; t < pl.T; t += nw) {
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int j = 0; j < pl.k; ++j) {
      const int R = pl.row_of_route[t * pl.k + j];
      if (R < 0) continue;
      const float w = topk_w[t * pl.k + j];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int q = lane + 32 * i;
        if (q < r) acc[i] += w * __uint_as_float((uint32_t)Z2[(int64_t)R * r + q] << 16);
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int q = lane + 32 * i;
      if (q < r) {
        __nv_bfloat16 h = __float2bfloat16_rn(acc[i]);
        Z2w[t * r + q] = *reinterpret_cast<uint16_t*>(&h);
      }
    }
  }
}

// Backward routed rows by scatter (as gather_fwd_kernel): Dp gets the token's dy
// row, D2p = bf16(s*dyB2) and dZ2p = bf16(s*w*dyB2) of the token; padding rows zero.
__global__ void gather_bwd_kernel(PlanView pl, const uint16_t* __restrict__ dy, const uint16_t* __restrict__ dyB2,
                                  const float* __restrict__ topk_w, uint16_t* __restrict__ Dp,
                                  uint16_t* __restrict__ D2p, uint16_t* __restrict__ dZ2p, int H, int r, float s) {
  const int lane = threadIdx.x & 31;
  const int64_t w0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int k = pl.k;
  for (int64_t t = w0; t < pl.T; t += nw) {
    const int* rows = pl.row_of_route + t * k;
    for (int c0 = 0; c0 < H; c0 += 32 * 8 * kGatherVec) {
      uint4 v[kGatherVec];
#pragma unroll
      for (int i = 0; i < kGatherVec; ++i) {
        const int c = c0 + (i * 32 + lane) * 8;
        v[i] = c < H ? __ldg(reinterpret_cast<const uint4*>(dy + t * H + c)) : make_uint4(0, 0, 0, 0);
      }
      for (int j = 0; j < k; ++j) {
        const int R = rows[j];
        if (R < 0) continue;
#pragma unroll
        for (int i = 0; i < kGatherVec; ++i) {
          const int c = c0 + (i * 32 + lane) * 8;
          if (c < H) *reinterpret_cast<uint4*>(Dp + (int64_t)R * H + c) = v[i];
        }
      }
    }
    for (int q = lane * 8; q < r; q += 32 * 8) {  // 8 columns per lane (r % 8 == 0)
      float v[8], a[8], b[8];
      ld_bf16x8(dyB2 + t * r + q, v);
#pragma unroll
      for (int i = 0; i < 8; ++i) a[i] = s * v[i];
      for (int j = 0; j < k; ++j) {
        const int R = rows[j];
        if (R < 0) continue;
        const float sw = s * topk_w[t * k + j];
#pragma unroll
        for (int i = 0; i < 8; ++i) b[i] = sw * v[i];
        st_bf16x8(D2p + (int64_t)R * r + q, a);
        st_bf16x8(dZ2p + (int64_t)R * r + q, b);
      }
    }
  }
  zero_padding_rows(pl, Dp, H, nullptr, 0);
  // D2p and dZ2p padding rows (r columns, r % 8 == 0)
  const int wib = threadIdx.x >> 5, wpb = blockDim.x >> 5;
  for (int g = blockIdx.x; g < pl.G; g += gridDim.x) {
    const int beg = pl.offsets[g] + pl.counts[g], end = pl.offsets[g + 1];
    for (int64_t p = beg + wib; p < end; p += wpb) {
      copy_row_or_zero(D2p + p * r, nullptr, r, lane);
      copy_row_or_zero(dZ2p + p * r, nullptr, r, lane);
    }
  }
}

__global__ void dw_kernel(PlanView pl, const float* __restrict__ part, int nparts, float* __restrict__ dw) {
  const int64_t TK = pl.T * pl.k;
  for (int64_t rt = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; rt < TK; rt += (int64_t)gridDim.x * blockDim.x) {
    const int R = pl.row_of_route[rt];
    float acc = 0.0f;
    if (R >= 0)
      for (int n = 0; n < nparts; ++n) acc += part[(int64_t)R * nparts + n];
    dw[rt] = acc;
  }
}

__global__ void dy13w_kernel(PlanView pl, const float* __restrict__ dY13, uint16_t* __restrict__ dY13w, int r2) {
  // one warp per token; lane l sums columns [8l, 8l+8) (+256 per pass; r2 % 16 == 0)
  // with 16-byte loads, up to 8 routes' loads in flight before they are added in
  // slot order
  constexpr int kGroup = 8;
  const int lane = threadIdx.x & 31;
  const int64_t w0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int k = pl.k;
  for (int64_t t = w0; t < pl.T; t += nw) {
    const int R = lane < k ? pl.row_of_route[t * k + lane] : -1;
    for (int c0 = 0; c0 < r2; c0 += 256) {  // warp-uniform loop: every lane takes part in the shuffles
      const int c = c0 + lane * 8;
      const bool on = c < r2;
      float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      for (int j0 = 0; j0 < k; j0 += kGroup) {
        float4 v[kGroup][2];
#pragma unroll
        for (int j = 0; j < kGroup; ++j) {
          const int Rj = __shfl_sync(0xffffffffu, R, (j0 + j) & 31);
          const bool live = on && j0 + j < k && Rj >= 0;
          const float4* p = reinterpret_cast<const float4*>(dY13 + (int64_t)(live ? Rj : 0) * r2 + c);
          v[j][0] = live ? p[0] : make_float4(0.f, 0.f, 0.f, 0.f);
          v[j][1] = live ? p[1] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int j = 0; j < kGroup; ++j) {
          if (j0 + j >= k || __shfl_sync(0xffffffffu, R, (j0 + j) & 31) < 0) continue;
          acc[0] += v[j][0].x;
          acc[1] += v[j][0].y;
          acc[2] += v[j][0].z;
          acc[3] += v[j][0].w;
          acc[4] += v[j][1].x;
          acc[5] += v[j][1].y;
          acc[6] += v[j][1].z;
          acc[7] += v[j][1].w;
        }
      }
      if (on) st_bf16x8(dY13w + t * r2 + c, acc);
    }
  }
}

// out_t = bf16( base_t + sum_j w_tj src[row(t,j)] ), one warp per token: every
// warp access is one contiguous 512-byte piece of one row (coalesced, one page),
// with the 16-byte loads of up to 8 routes in flight before they are summed.
// fp32, slot order j = 0..k-1 after the base term; w = 1 when topk_w is NULL.
__global__ void combine_rows_kernel(PlanView pl, const uint16_t* __restrict__ base, const uint16_t* __restrict__ src,
                                    const float* __restrict__ topk_w, uint16_t* __restrict__ out, int H) {
  const int lane = threadIdx.x & 31;
  const int64_t w0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int k = pl.k;
  for (int64_t t = w0; t < pl.T; t += nw) {
    const int* rows = pl.row_of_route + t * k;
    // two 8-column groups per lane and pass (c and c + 256, the second skipped past H), so up to
    // 2 x 8 routed-row loads are in flight before they are added in slot order
    for (int c = lane * 8; c < H; c += 2 * 32 * 8) {
      const int c2 = c + 32 * 8;
      const bool two = c2 < H;
      float acc[8], acc2[8];
      ld_bf16x8(base + t * H + c, acc);
      if (two) ld_bf16x8(base + t * H + c2, acc2);
      for (int j0 = 0; j0 < k; j0 += 8) {
        int R[8];
        float w[8];
        uint4 u[8], u2[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const bool in = j0 + j < k;
          R[j] = in ? rows[j0 + j] : -1;
          w[j] = (in && topk_w) ? topk_w[t * k + j0 + j] : 1.0f;
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint4* rp = reinterpret_cast<const uint4*>(src + (R[j] >= 0 ? (int64_t)R[j] * H : 0));
          u[j] = R[j] >= 0 ? __ldg(rp + c / 8) : make_uint4(0, 0, 0, 0);
          u2[j] = (R[j] >= 0 && two) ? __ldg(rp + c2 / 8) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (R[j] < 0) continue;
          const uint32_t wd[4] = {u[j].x, u[j].y, u[j].z, u[j].w};
          const uint32_t wd2[4] = {u2[j].x, u2[j].y, u2[j].z, u2[j].w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            acc[2 * e] += w[j] * bf16_lo(wd[e]);
            acc[2 * e + 1] += w[j] * bf16_hi(wd[e]);
            acc2[2 * e] += w[j] * bf16_lo(wd2[e]);
            acc2[2 * e + 1] += w[j] * bf16_hi(wd2[e]);
          }
        }
      }
      st_bf16x8(out + t * H + c, acc);
      if (two) st_bf16x8(out + t * H + c2, acc2);
    }
  }
}

// MXFP4 -> bf16, exactly (32-element groups: 16 packed bytes and one UE8M0 byte in,
// 64 bytes of bf16 out; see the kernel for the thread mapping).  E2M1 magnitudes are
// {0, 0.5, 1, 1.5, 2, 3, 4, 6} (bit 3 = sign); the scale byte b means 2^(b-127)
// (b = 0 is the fp32 subnormal 2^-127, b = 255 is NaN).  Every product is a bf16
// value, so the conversion below rounds nothing.
constexpr bool kDequantCvt = true;  // false: decode the codes with a magnitude table

__global__ void dequant_mxfp4_kernel(const uint8_t* __restrict__ packed, const uint8_t* __restrict__ scales,
                                     uint16_t* __restrict__ out, int64_t groups) {
  const float kMag[8] = {0.0f, 0.5f, 1.0f, 1.5f, 2.0f, 3.0f, 4.0f, 6.0f};
  // one thread per 8 elements (4 packed bytes in, 16 bytes of bf16 out), so a warp
  // reads 128 and writes 512 contiguous bytes per step; 4 consecutive threads share
  // one 32-element scale group
  // Each thread takes kBatch such items a grid stride apart and issues all their
  // loads before decoding any, so a warp keeps kBatch x 128 B of reads in flight.
  constexpr int kBatch = 8;
  const int64_t n8 = groups * 4;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i0 < n8; i0 += stride * kBatch) {
    uint32_t w[kBatch], b[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int64_t i = i0 + u * stride;
      w[u] = i < n8 ? __ldg(reinterpret_cast<const uint32_t*>(packed) + i) : 0u;
      b[u] = i < n8 ? scales[i >> 2] : 0u;
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int64_t i = i0 + u * stride;
      if (i >= n8) break;
      const float sc = ue8m0_to_float(b[u]);
      float v[8];
      if (kDequantCvt) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t h2 = e2m1x2_to_f16x2((w[u] >> (8 * j)) & 0xFFu);
          const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h2));
          v[2 * j] = f.x * sc;
          v[2 * j + 1] = f.y * sc;
        }
      } else {
#pragma unroll
        for (int n = 0; n < 8; ++n) {
          const uint32_t code = (w[u] >> (4 * n)) & 15u;
          const float mag = kMag[code & 7u] * sc;
          v[n] = (code & 8u) ? -mag : mag;
        }
      }
      st_bf16x8(out + i * 8, v);
    }
  }
}

// out[i] = sum over s = 0..split-1 (in order) of in[s * stride + i]; n % 4 == 0.
__global__ void reduce_splits_kernel(const float* __restrict__ in, int64_t stride, int split, int64_t n,
                                     float* __restrict__ out) {
  for (int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 4; i < n; i += (int64_t)gridDim.x * blockDim.x * 4) {
    float4 a = *reinterpret_cast<const float4*>(in + i);
    for (int s = 1; s < split; ++s) {
      const float4 b = *reinterpret_cast<const float4*>(in + s * stride + i);
      a.x += b.x;
      a.y += b.y;
      a.z += b.z;
      a.w += b.w;
    }
    *reinterpret_cast<float4*>(out + i) = a;
  }
}

int grid_for(int num_sms) { return num_sms * 8; }

}  // namespace

cudaError_t launch_combine_rows(const PlanView& pl, const uint16_t* base, const uint16_t* src, const float* topk_w,
                                uint16_t* out, int H, int num_sms, cudaStream_t stream, int slot) {
  prof_begin(slot, stream);
  combine_rows_kernel<<<grid_for(num_sms), kThreads, 0, stream>>>(pl, base, src, topk_w, out, H);
  prof_end(slot, stream);
  return cudaGetLastError();
}

cudaError_t launch_dequant_mxfp4(const uint8_t* packed, const uint8_t* scales, uint16_t* out, int64_t elems,
                                 int num_sms, cudaStream_t stream) {
  prof_begin(K_DEQUANT, stream);
  dequant_mxfp4_kernel<<<grid_for(num_sms), kThreads, 0, stream>>>(packed, scales, out, elems / 32);
  prof_end(K_DEQUANT, stream);
  return cudaGetLastError();
}

cudaError_t launch_reduce_splits(const float* in, int64_t stride, int split, int64_t n, float* out, int num_sms,
                                 cudaStream_t stream) {
  prof_begin(K_SPLIT_REDUCE, stream);
  reduce_splits_kernel<<<grid_for(num_sms), kThreads, 0, stream>>>(in, stride, split, n, out);
  prof_end(K_SPLIT_REDUCE, stream);
  return cudaGetLastError();
}

cudaError_t launch_gather_fwd(const PlanView& pl, const uint16_t* x, const uint16_t* Y13, uint16_t* Xp,
                              uint16_t* Y13p, int H, int r2, int num_sms, cudaStream_t stream) {
  prof_begin(K_GATHER_FWD, stream);
  gather_fwd_kernel<<<grid_for(num_sms), kThreads, 0, stream>>>(pl, x, Y13, Xp, Y13p, H, r2);
  prof_end(K_GATHER_FWD, stream);
  return cudaGetLastError();
}

cudaError_t launch_gather_fwd_mxfp8(const PlanView& pl, const uint16_t* x, const uint16_t* Y13, uint8_t* Xq,
                                    uint8_t* Xs, uint16_t* Y13p, int H, int r2, int num_sms, cudaStream_t stream) {
  prof_begin(K_GATHER_FWD, stream);
  gather_fwd_mxfp8_kernel<<<grid_for(num_sms), kThreads, 0, stream>>>(pl, x, Y13, Xq, Xs, Y13p, H, r2);
  prof_end(K_GATHER_FWD, stream);
  return cudaGetLastError();
}

cudaError_t launch_dw_from_o(const PlanView& pl, const uint16_t* dy, const uint16_t* dyB2, const uint16_t* O,
                             const uint16_t* Z2, int H, int r, float s, float* dw, int num_sms, cudaStream_t stream) {
  prof_begin(K_DW_NV, stream);
  dw_from_o_kernel<<<grid_for(num_sms), kThreads, 0, stream>>>(pl, dy, dyB2, O, Z2, H, r, s, dw);
  prof_end(K_DW_NV, stream);
  return cudaGetLastError();
}

cudaError_t launch_scales_to_tiles(const uint8_t* S, int64_t rows, int K, uint8_t* St, int num_sms,
                                   cudaStream_t stream) {
  scales_to_tiles_kernel<<<grid_for(num_sms), kThreads, 0, stream>>>(S, rows, K / 128, St);
  return cudaGetLastError();
}

cudaError_t launch_quant_mxfp8(const uint16_t* x, int64_t rows, int n, uint8_t* codes, uint8_t* scales,
                               int num_sms, cudaStream_t stream) {
  quant_mxfp8_kernel<<<grid_for(num_sms), kThreads, 0, stream>>>(x, rows, n, codes, scales);
  return cudaGetLastError();
}

cudaError_t launch_z2w(const PlanView& pl, const uint16_t* Z2, const float* topk_w, uint16_t* Z2w, int r,
                       int num_sms, cudaStream_t stream) {
  prof_begin(K_Z2W, stream);
  z2w_kernel<<<grid_for(num_sms), kThreads, 0, stream>>>(pl, Z2, topk_w, Z2w, r);
  prof_end(K_Z2W, stream);
  return cudaGetLastError();
}

cudaError_t launch_gather_bwd(const PlanView& pl, const uint16_t* dy, const uint16_t* dyB2, const float* topk_w,
                              uint16_t* Dp, uint16_t* D2p, uint16_t* dZ2p, int H, int r, float s, int num_sms,
                              cudaStream_t stream) {
  prof_begin(K_GATHER_BWD, stream);
  gather_bwd_kernel<<<grid_for(num_sms), kThreads, 0, stream>>>(pl, dy, dyB2, topk_w, Dp, D2p, dZ2p, H, r, s);
  prof_end(K_GATHER_BWD, stream);
  return cudaGetLastError();
}

cudaError_t launch_dw(const PlanView& pl, const float* part, int nparts, float* dw, int num_sms,
                      cudaStream_t stream) {
  prof_begin(K_DW, stream);
  dw_kernel<<<grid_for(num_sms), kThreads, 0, stream>>>(pl, part, nparts, dw);
  prof_end(K_DW, stream);
  return cudaGetLastError();
}

cudaError_t launch_dy13w(const PlanView& pl, const float* dY13, uint16_t* dY13w, int r2, int num_sms,
                         cudaStream_t stream) {
  prof_begin(K_DY13W, stream);
  dy13w_kernel<<<grid_for(num_sms), kThreads, 0, stream>>>(pl, dY13, dY13w, r2);
  prof_end(K_DY13W, stream);
  return cudaGetLastError();
}

}  // namespace moelora
