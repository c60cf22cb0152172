// Shared definitions of the MoE side-LoRA library: size rules, workspace
// layouts (host), and the device view of a routing plan.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/moe_lora.h"

namespace moelora {

constexpr int kBlockM = 128;       // plan padding unit = GEMM M tile
constexpr int kMaxAdapters = 64;   // adapters sharing one layer
constexpr int kMaxGroups = 16384;  // adapters x experts
constexpr int kPlanChunk = 1024;   // routes per plan chunk (one warp each)
constexpr int kMaxSplit = 8;       // token-range slices of the long-K reductions

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Base formats: 0 bf16; MXFP4 decoded inside the expert GEMMs (1) or once per pass
// into the saved workspace (2); the native FP4 forward with the rest as 1 (3) or as 2 (4).
inline bool fmt_mx(const moe_lora_dims* d) { return d->base_fmt >= 1; }
inline bool fmt_in_gemm(const moe_lora_dims* d) { return d->base_fmt == 1 || d->base_fmt == 3; }
inline bool fmt_once(const moe_lora_dims* d) { return d->base_fmt == 2 || d->base_fmt == 4; }
inline bool fmt_native(const moe_lora_dims* d) { return d->base_fmt >= 3; }

// Returns MOE_LORA_OK when the sizes are supported.
inline int check_dims(const moe_lora_dims* d) {
  if (!d) return MOE_LORA_ERR_NULL;
  if ((d->act != 0 && d->act != 1) || d->base_fmt < 0 || d->base_fmt > 4) return MOE_LORA_ERR_UNSUPPORTED;
  if (!(d->act_clamp >= 0.0f) || d->act_clamp > 3.0e38f) return MOE_LORA_ERR_DIMS;
  if (d->T < 0 || d->T > (int64_t)1 << 30) return MOE_LORA_ERR_DIMS;
  if (d->H < 64 || d->H % 64 || d->I < 64 || d->I % 64) return MOE_LORA_ERR_DIMS;
  // native FP4 forward: whole 128-wide K steps and 128-column tiles
  if (fmt_native(d) && (d->H % 128 || d->I % 128)) return MOE_LORA_ERR_DIMS;
  if (d->r < 8 || d->r > 128 || d->r % 8) return MOE_LORA_ERR_DIMS;
  if (d->k < 1 || d->k > 32 || d->E < 1 || d->A < 1 || d->A > kMaxAdapters) return MOE_LORA_ERR_DIMS;
  if ((int64_t)d->A * d->E > kMaxGroups) return MOE_LORA_ERR_DIMS;
  if (d->block_m != kBlockM) return MOE_LORA_ERR_DIMS;
  if (d->T * d->k + (int64_t)d->A * d->E * kBlockM > ((int64_t)1 << 31) - 1) return MOE_LORA_ERR_DIMS;
  return MOE_LORA_OK;
}

// Upper bound of the padded routed-row count P = sum_g roundup(c_g, 128).
inline int64_t rows_cap(const moe_lora_dims* d) {
  int64_t G = (int64_t)d->A * d->E;
  int64_t p = d->T * d->k + G * (kBlockM - 1);
  return (int64_t)align_up((size_t)p, kBlockM);
}

inline int64_t plan_chunks(const moe_lora_dims* d) {
  return (d->T * d->k + kPlanChunk - 1) / kPlanChunk;
}

// ------------------------------------------------------------------ layouts
struct PlanLayout {
  size_t err, counts, offsets, row_of_route, route_of_row, tile_group, tile_span, tok_off, tok_tile, wtile_off, wtile,
      chunk_base, total;
};
inline PlanLayout plan_layout(const moe_lora_dims* d) {
  PlanLayout L;
  const int64_t G = (int64_t)d->A * d->E, P = rows_cap(d), TK = d->T * d->k;
  size_t o = 0;
  auto take = [&](size_t bytes) { size_t at = o; o = align_up(o + bytes, 256); return at; };
  L.err = take(16);
  L.counts = take(sizeof(int32_t) * G);
  L.offsets = take(sizeof(int32_t) * (G + 1));
  L.row_of_route = take(sizeof(int32_t) * (TK > 0 ? TK : 1));
  L.route_of_row = take(sizeof(int32_t) * P);
  L.tile_group = take(sizeof(int32_t) * (P / kBlockM + 1));
  L.tile_span = take(2 * sizeof(int32_t) * (P / kBlockM + 1));
  L.tok_off = take(sizeof(int32_t) * (kMaxAdapters + 1));
  L.tok_tile = take(sizeof(int32_t) * (kMaxAdapters + 1));
  L.wtile_off = take(sizeof(int32_t) * (G + 1));
  L.wtile = take(4 * sizeof(int32_t) * (P / kBlockM + 1));
  L.chunk_base = take(sizeof(int32_t) * G * (plan_chunks(d) > 0 ? plan_chunks(d) : 1));
  L.total = o;
  return L;
}

// What the forward keeps for the backward (bf16).  An MXFP4 base decoded inside the
// GEMMs (base_fmt 1) is never stored in bf16; decoded once per pass (base_fmt 2) it
// adds the bf16 W1, W3 [E,I,H] and W2 [E,H,I], which the backward reuses.
struct SavedLayout {
  size_t Y13p, G, U, Act, Z2w, O, Z2, W1, W3, W2, total;   // [P,2r], [P,I], [P,I], [P,I], [T,r]
};
inline SavedLayout saved_layout(const moe_lora_dims* d) {
  SavedLayout L;
  const int64_t P = rows_cap(d), T = d->T > 0 ? d->T : 1;
  size_t o = 0;
  auto take = [&](size_t bytes) { size_t at = o; o = align_up(o + bytes, 256); return at; };
  L.Y13p = take(2 * (size_t)P * 2 * d->r);
  L.G = take(2 * (size_t)P * d->I);
  L.U = take(2 * (size_t)P * d->I);
  L.Act = take(2 * (size_t)P * d->I);
  L.Z2w = take(2 * (size_t)T * d->r);
  // native FP4 forward: the forward's routed down rows O [P,H] and the A2 shrink Z2
  // [P,r] (bf16), from which the backward takes the router-weight gradient
  L.O = take(fmt_native(d) ? 2 * (size_t)P * d->H : 0);
  L.Z2 = take(fmt_native(d) ? 2 * (size_t)P * d->r : 0);
  const size_t wbytes = fmt_once(d) ? 2 * (size_t)d->E * d->I * d->H : 0;
  L.W1 = take(wbytes);
  L.W3 = take(wbytes);
  L.W2 = take(wbytes);
  L.total = o;
  return L;
}

struct FwdLayout {
  size_t Y13, Xp, O, Z2, total;   // [T,2r], [P,H], [P,H], [P,r]  (bf16)
  size_t S13t;                    // native FP4 forward: W1/W3 scale bytes, tile-major (2 x E*I*H/32)
  size_t S2t;                     //   W2's, tile-major (E*H*I/32)
  size_t Actq, Acts;              //   the activation as MXFP8: codes [P,I], tile-major scale words
};
inline FwdLayout fwd_layout(const moe_lora_dims* d) {
  FwdLayout L;
  const int64_t P = rows_cap(d), T = d->T > 0 ? d->T : 1;
  size_t o = 0;
  auto take = [&](size_t bytes) { size_t at = o; o = align_up(o + bytes, 256); return at; };
  L.Y13 = take(2 * (size_t)T * 2 * d->r);
  L.Xp = take(2 * (size_t)P * d->H);
  // (native FP4 forward: O and Z2 live in `saved` instead)
  L.O = take(fmt_native(d) ? 0 : 2 * (size_t)P * d->H);
  L.Z2 = take(fmt_native(d) ? 0 : 2 * (size_t)P * d->r);
  L.S13t = take(fmt_native(d) ? 2 * (size_t)d->E * d->I * (d->H / 32) : 0);
  L.S2t = take(fmt_native(d) ? (size_t)d->E * d->H * (d->I / 32) : 0);
  L.Actq = take(fmt_native(d) ? (size_t)P * d->I : 0);
  L.Acts = take(fmt_native(d) ? (size_t)P * (d->I / 32) : 0);
  L.total = o;
  return L;
}

struct BwdLayout {
  // dyB2 [T,r] bf16; Dp [P,H] bf16 (reused for dXp); D2p, dZ2p [P,r] bf16;
  // dG, dU [P,I] bf16; part [P, 2*ceil(I/256)] f32 (router-gradient partial sums: at
  // most two per row and 256-column tile); dY13 [P,2r] f32; dY13w [T,2r] bf16;
  // dXl [T,H] bf16 (grad-x through A1/A3); ksplit: fp32 partials of the
  // token-split dB2 and dA1/dA3 reductions [kMaxSplit][2][A][r][H]
  size_t dyB2, Dp, D2p, dZ2p, dG, dU, part, dY13, dY13w, dXl, ksplit, total;
};
inline BwdLayout bwd_layout(const moe_lora_dims* d) {
  BwdLayout L;
  const int64_t P = rows_cap(d), T = d->T > 0 ? d->T : 1;
  size_t o = 0;
  auto take = [&](size_t bytes) { size_t at = o; o = align_up(o + bytes, 256); return at; };
  L.dyB2 = take(2 * (size_t)T * d->r);
  L.Dp = take(2 * (size_t)P * d->H);
  L.D2p = take(2 * (size_t)P * d->r);
  L.dZ2p = take(2 * (size_t)P * d->r);
  L.dG = take(2 * (size_t)P * d->I);
  L.dU = take(2 * (size_t)P * d->I);
  L.part = take(4 * (size_t)P * 2 * ((d->I + 255) / 256));
  L.dY13 = take(4 * (size_t)P * 2 * d->r);
  L.dY13w = take(2 * (size_t)T * 2 * d->r);
  L.dXl = take(2 * (size_t)T * d->H);
  L.ksplit = take(4 * (size_t)kMaxSplit * 2 * d->A * d->r * d->H);
  L.total = o;
  return L;
}

// Router scratch: error word; dl [T,E] bf16 (dense logit gradient, the tensor-core
// operand of both router-backward contractions); fp32 partials of the token-split
// dW_r reduction [A][kMaxSplit][E][H].
struct RouterLayout {
  size_t err, dl, part, total;
};
inline RouterLayout router_layout(const moe_lora_dims* d) {
  RouterLayout L;
  const int64_t T = d->T > 0 ? d->T : 1;
  size_t o = 0;
  auto take = [&](size_t bytes) { size_t at = o; o = align_up(o + bytes, 256); return at; };
  L.err = take(16);
  L.dl = take(2 * (size_t)T * d->E);
  L.part = take(4 * (size_t)d->A * kMaxSplit * d->E * d->H);
  L.total = o;
  return L;
}

// Extra size rules of the router: 16 <= E <= 256 with E % 16 == 0 (the whole logit
// row is one MMA tile N), k <= E.
inline int check_router_dims(const moe_lora_dims* d) {
  const int rc = check_dims(d);
  if (rc) return rc;
  if (d->E < 16 || d->E > 256 || d->E % 16) return MOE_LORA_ERR_UNSUPPORTED;
  if (d->k > d->E) return MOE_LORA_ERR_DIMS;
  return MOE_LORA_OK;
}

// ------------------------------------------------------------------ device plan view
// Groups are laid out expert-major: plan slot q = e*A + a holds the rows of adapter a
// routed to expert e, so the A groups sharing an expert's base weights are adjacent
// in the padded rows (their tiles run back to back and find those weights in L2).
// Per-group weights and gradients are indexed by g = a*E + e.
__host__ __device__ inline int group_weight_index(int q, int A, int E) { return (q % A) * E + q / A; }

struct PlanView {
  int* err;                  // sticky device error word
  const int* counts;         // [G] live routes per group, in plan-slot order (q = e*A + a)
  const int* offsets;        // [G+1] padded row offsets by plan slot; offsets[G] = P
  const int* row_of_route;   // [T*k] padded row of route t*k+j, or -1
  const int* route_of_row;   // [P] route of a row, or -1 for padding
  const int* tile_group;     // [P/128] weight index g = a*E + e of each 128-row tile's group
  const int2* tile_span;     // [P/128] (first 128-row tile, number of 128-row tiles) of that tile's group
  const int* tok_off;        // [A+1] first token of each adapter
  const int* tok_tile;       // [A+1] first 128-token tile of each adapter
  const int* wtile_off;      // [G+1] first 256-row tile of each group, by plan slot
  const int4* wtile;         // 256-row tiles: x = (first 128-row tile << 1) | (halves - 1), y = weight index,
                             // z = first 256-row tile of the group, w = the group's number of 256-row tiles
  int64_t T;
  int G, E, A, k;
};

inline PlanView make_plan_view(const moe_lora_dims* d, const void* ws) {
  const PlanLayout L = plan_layout(d);
  const char* b = static_cast<const char*>(ws);
  PlanView v;
  v.err = (int*)(b + L.err);
  v.counts = (const int*)(b + L.counts);
  v.offsets = (const int*)(b + L.offsets);
  v.row_of_route = (const int*)(b + L.row_of_route);
  v.route_of_row = (const int*)(b + L.route_of_row);
  v.tile_group = (const int*)(b + L.tile_group);
  v.tile_span = (const int2*)(b + L.tile_span);
  v.tok_off = (const int*)(b + L.tok_off);
  v.tok_tile = (const int*)(b + L.tok_tile);
  v.wtile_off = (const int*)(b + L.wtile_off);
  v.wtile = (const int4*)(b + L.wtile);
  v.T = d->T;
  v.G = d->A * d->E;
  v.E = d->E;
  v.A = d->A;
  v.k = d->k;
  return v;
}

// ------------------------------------------------------------------ bf16 helpers
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}
// ---------------------------------------------------------------- MXFP8 (native FP4 forward)
// E4M3 code of v (already divided by the block scale): round to nearest even,
// saturating at +-448 -- the conversion instruction's own rounding.  Two values per
// instruction; `lo` lands in the low byte.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}
// 2^e as a float for e in [-127, 127] (2^-127 is subnormal)
__device__ __forceinline__ float exp2i(int e) {
  return e >= -126 ? __uint_as_float((uint32_t)(e + 127) << 23) : __uint_as_float(1u << 22);
}
// One MXFP8 block of 32 values (OCP MX: shared scale 2^X, X = floor(log2 max|v|) - 8,
// X = 0 for an all-zero block, clamped to [-127, 127]): the 32 E4M3 codes and the
// scale byte X + 127.
__device__ __forceinline__ uint32_t mxfp8_block_f32(const float (&f)[32], uint4 (&codes)[2]) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(f[i]));
  int X = 0;
  if (amax > 0.f) {
    const uint32_t b = __float_as_uint(amax);
    const int e = (int)(b >> 23);
    const int fl = e ? e - 127 : (31 - __clz((int)b)) - 149;  // floor(log2 amax), subnormals too
    X = min(max(fl - 8, -127), 127);
  }
  const float inv = exp2i(-X);  // exact scaling by a power of two
  uint32_t q[8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
    q[i] = e4m3x2(f[4 * i] * inv, f[4 * i + 1] * inv) | (e4m3x2(f[4 * i + 2] * inv, f[4 * i + 3] * inv) << 16);
  codes[0] = make_uint4(q[0], q[1], q[2], q[3]);
  codes[1] = make_uint4(q[4], q[5], q[6], q[7]);
  return (uint32_t)(X + 127);
}

__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

// 8 bf16 <-> 8 floats through one 16-byte access.
__device__ __forceinline__ void st_bf16x8(uint16_t* dst, const float* v) {
  uint4 u;
  u.x = pack_bf16x2(v[0], v[1]);
  u.y = pack_bf16x2(v[2], v[3]);
  u.z = pack_bf16x2(v[4], v[5]);
  u.w = pack_bf16x2(v[6], v[7]);
  *reinterpret_cast<uint4*>(dst) = u;
}
__device__ __forceinline__ void ld_bf16x8(const uint16_t* src, float* v) {
  const uint4 u = *reinterpret_cast<const uint4*>(src);
  v[0] = bf16_lo(u.x); v[1] = bf16_hi(u.x);
  v[2] = bf16_lo(u.y); v[3] = bf16_hi(u.y);
  v[4] = bf16_lo(u.z); v[5] = bf16_hi(u.z);
  v[6] = bf16_lo(u.w); v[7] = bf16_hi(u.w);
}
__device__ __forceinline__ void st_f32x4(float* dst, const float* v) {
  *reinterpret_cast<float4*>(dst) = make_float4(v[0], v[1], v[2], v[3]);
}

// ------------------------------------------------------------------ MXFP4 (E2M1 + UE8M0)
// Two E2M1 codes (one byte, the lower index in the low nibble) to two f16 values
// (low half = low nibble) with the hardware conversion; every E2M1 value is exact in
// f16.
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte) {
  uint32_t d;
  asm("{ .reg .b8 t; cvt.u8.u16 t, %1; cvt.rn.f16x2.e2m1x2 %0, t; }" : "=r"(d) : "h"((uint16_t)byte));
  return d;
}
// UE8M0 scale byte b -> 2^(b-127) (b = 0: the fp32 subnormal 2^-127; b = 255: NaN).
__device__ __forceinline__ float ue8m0_to_float(uint32_t b) {
  return __uint_as_float(b == 0 ? 0x00400000u : b == 255 ? 0x7FC00000u : b << 23);
}
// Eight E2M1 codes (one 32-bit word, element 0 in the lowest nibble) times the scale
// `sc`, as eight bf16 values in one 16-byte vector.  Every product of an E2M1 value
// and a power of two is a bf16 value (or overflows to inf), so nothing is rounded.
__device__ __forceinline__ uint4 mx_decode8(uint32_t w, float sc) {
  uint32_t o[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t h2 = e2m1x2_to_f16x2((w >> (8 * j)) & 0xFFu);
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h2));
    o[j] = pack_bf16x2(f.x * sc, f.y * sc);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// The same decode without conversion instructions, for scale bytes b in [2, 252]
// (where every product is a normal bf16 value): the bf16 bit patterns of the E2M1
// magnitudes {0, .5, 1, 1.5, 2, 3, 4, 6} are looked up with byte permutes (high
// bytes 00 3F 3F 3F 40 40 40 40, low bytes 00 00 80 C0 00 40 80 C0), each code's sign
// bit is moved to bit 15 of its half with the permute's sign-replicating mode, and
// one bf16x2 multiply by 2^(b-127) (bf16 bits b << 7 in both halves) scales them --
// exactly, as the product of a value of at most two significant bits and a power of
// two is representable.  scale2 = (b << 7) * 0x10001.
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}
__device__ __forceinline__ uint32_t mul_bf16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint4 mx_decode8_fast(uint32_t w, uint32_t scale2) {
  const uint32_t s03 = w & 0x7777u, s47 = (w >> 16) & 0x7777u;  // magnitude codes, 4 per selector
  const uint32_t hA = prmt(0x3F3F3F00u, 0x40404040u, s03), lA = prmt(0xC0800000u, 0xC0804000u, s03);
  const uint32_t hB = prmt(0x3F3F3F00u, 0x40404040u, s47), lB = prmt(0xC0800000u, 0xC0804000u, s47);
  const uint32_t w4 = w << 4;  // byte k's top bit = sign of element 2k (w's own: of element 2k + 1)
  uint32_t o[4] = {prmt(lA, hA, 0x5140u), prmt(lA, hA, 0x7362u), prmt(lB, hB, 0x5140u), prmt(lB, hB, 0x7362u)};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint32_t sg = prmt(w4, w, ((8u | (4u + k)) << 12) | ((8u | k) << 4));  // 0xFF bytes where negative
    o[k] = mul_bf16x2(o[k] | (sg & 0x80008000u), scale2);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}
// Either decode, by the scale byte.
__device__ __forceinline__ uint4 mx_decode8_any(uint32_t w, uint32_t b) {
  if (b >= 2u && b <= 252u) return mx_decode8_fast(w, (b << 7) * 0x10001u);
  return mx_decode8(w, ue8m0_to_float(b));
}

}  // namespace moelora
