// Forward pass of the routed MoE side-LoRA FFN: tensor maps and the launch
// sequence, all on one stream with no host synchronisation.
//   F1 shrink (per token)  ->  F2 gather (routed rows, zero padding)
//   F3 W13 + B1/B3 expand + SwiGLU  ->  F4 W2 + A2 shrink
//   F6a per-token Z2 combine  ->  F6 B2 expand per token  ->  routing-weighted combine
#include "gemm_pair.cuh"
#include "gemm_problems.cuh"
#include "launch.h"
#include "passes.h"
#include "tmap.h"

namespace moelora {

int run_forward(const moe_lora_dims* d, const void* plan_ws, const uint16_t* x, const float* topk_w,
                const moe_lora_weights* w, uint16_t* y, void* saved, void* scratch, int num_sms,
                cudaStream_t stream) {
  const PlanView pl = make_plan_view(d, plan_ws);
  const SavedLayout SL = saved_layout(d);
  const FwdLayout FL = fwd_layout(d);
  char* sv = static_cast<char*>(saved);
  char* sc = static_cast<char*>(scratch);
  uint16_t* Y13p = (uint16_t*)(sv + SL.Y13p);
  uint16_t* Gs = (uint16_t*)(sv + SL.G);
  uint16_t* Us = (uint16_t*)(sv + SL.U);
  uint16_t* Act = (uint16_t*)(sv + SL.Act);
  uint16_t* Z2w = (uint16_t*)(sv + SL.Z2w);
  uint16_t* Y13 = (uint16_t*)(sc + FL.Y13);
  uint16_t* Xp = (uint16_t*)(sc + FL.Xp);
  // native FP4 forward: O and Z2 are kept in `saved` (the backward's router-weight
  // gradient reads them)
  uint16_t* O = (uint16_t*)(fmt_native(d) ? sv + SL.O : sc + FL.O);
  uint16_t* Z2 = (uint16_t*)(fmt_native(d) ? sv + SL.Z2 : sc + FL.Z2);

  const uint64_t T = (uint64_t)d->T, H = d->H, I = d->I, E = d->E, A = d->A, r = d->r;
  const uint64_t P = (uint64_t)rows_cap(d), G = A * E;
  const uint32_t r32 = (uint32_t)((r + 31) / 32 * 32);
  const int max_tok_tiles = (int)((T + 127) / 128) + d->A;
  const int max_row_tiles = (int)(P / 128);
  int rc = 0;
  cudaError_t ce;
  // An MXFP4 base: base_fmt 1 decodes it inside the expert GEMMs, stage by stage,
  // into the same bf16 operand tiles (ProbW13T<true>, ProbW2T<true>), so no decoded
  // copy exists anywhere; base_fmt 2 decodes it once per pass into `saved` (which the
  // backward reuses) and runs the bf16 GEMMs on that copy.  base_fmt 3 (native FP4
  // forward) runs the gate/up base products on block-scaled FP4 tensor cores from
  // MXFP8 routed rows (ProbW13Nv) and the rest as base_fmt 1; base_fmt 4 the same
  // with the rest as base_fmt 2.
  const bool nat = fmt_native(d);
  const bool mx = fmt_in_gemm(d);
  const void* bW1 = w->W1;
  const void* bW3 = w->W3;
  const void* bW2 = w->W2;
  if (fmt_once(d)) {
    uint16_t* q1 = (uint16_t*)(sv + SL.W1);
    uint16_t* q3 = (uint16_t*)(sv + SL.W3);
    uint16_t* q2 = (uint16_t*)(sv + SL.W2);
    const int64_t n = (int64_t)E * I * H;
    if (launch_dequant_mxfp4((const uint8_t*)w->W1, w->S1, q1, n, num_sms, stream) != cudaSuccess ||
        launch_dequant_mxfp4((const uint8_t*)w->W3, w->S3, q3, n, num_sms, stream) != cudaSuccess ||
        launch_dequant_mxfp4((const uint8_t*)w->W2, w->S2, q2, n, num_sms, stream) != cudaSuccess)
      return MOE_LORA_ERR_CUDA;
    bW1 = q1;
    bW3 = q3;
    bW2 = q2;
  }
#define MAP(call)               \
  do {                          \
    if ((rc = (call)) != 0) return MOE_LORA_ERR_CUDA; \
  } while (0)
#define LAUNCH(call)                                  \
  do {                                                \
    if ((ce = (call)) != cudaSuccess) return MOE_LORA_ERR_CUDA; \
  } while (0)

  // F1: Y13 = bf16(s * x [A1; A3]^T), per token
  {
    ProbShrink p;
    MAP(tmap_2d(&p.mx, x, H, T, 64, 128));
    MAP(tmap_3d(&p.mA1, w->A1, H, r, A, 64, (uint32_t)r));
    MAP(tmap_3d(&p.mA3, w->A3, H, r, A, 64, (uint32_t)r));
    p.pl = pl;
    p.err = pl.err;
    p.Y13 = Y13;
    p.H = d->H;
    p.r = d->r;
    p.s = d->scale;
    LAUNCH(launch_gemm(p, max_tok_tiles, num_sms, stream, K_SHRINK));
  }
  // F2: routed rows (native: as MXFP8 codes Xq [P,H] and scale words, in the Xp buffer)
  uint8_t* Xq = reinterpret_cast<uint8_t*>(Xp);
  uint8_t* Xs = Xq + P * H;
  if (nat)
    LAUNCH(launch_gather_fwd_mxfp8(pl, x, Y13, Xq, Xs, Y13p, d->H, 2 * d->r, num_sms, stream));
  else
    LAUNCH(launch_gather_fwd(pl, x, Y13, Xp, Y13p, d->H, 2 * d->r, num_sms, stream));
  // F3: W13 + expert-local expand + SwiGLU
  auto w13 = [&](auto p) -> int {
    MAP(tmap_2d(&p.mXp, Xp, H, P, 64, 128));
    MAP(tmap_2d(&p.mY13p, Y13p, 2 * r, P, 64, 128));
    if (!mx) {
      MAP(tmap_3d(&p.mW1, bW1, H, I, E, 64, 128));
      MAP(tmap_3d(&p.mW3, bW3, H, I, E, 64, 128));
    }
    if (mx) {
      MAP(tmap_3d_u8(&p.mW1q, w->W1, H / 2, I, E, 32, 128));
      MAP(tmap_3d_u8(&p.mW3q, w->W3, H / 2, I, E, 32, 128));
    }
    p.S1q = w->S1;
    p.S3q = w->S3;
    MAP(tmap_3d(&p.mB1, w->B1, r, I, G, 64, 128));
    MAP(tmap_3d(&p.mB3, w->B3, r, I, G, 64, 128));
    MAP(tmap_2d_store32(&p.mG, Gs, I, P));
    MAP(tmap_2d_store32(&p.mU, Us, I, P));
    MAP(tmap_2d_store32(&p.mAct, Act, I, P));
    p.pl = pl;
    p.err = pl.err;
    p.G = Gs;
    p.U = Us;
    p.Act = Act;
    p.H = d->H;
    p.I = d->I;
    p.r = d->r;
    p.act = d->act;
    p.clamp = d->act_clamp;
    LAUNCH(launch_gemm(p, max_row_tiles * cdiv(d->I, 128), num_sms, stream, K_W13));
    return 0;
  };
  if (nat) {
    // the W1/W3 scale bytes in the tile-major layout the native stages copy (per pass)
    uint8_t* S1t = reinterpret_cast<uint8_t*>(sc + FL.S13t);
    uint8_t* S3t = S1t + E * I * (H / 32);
    LAUNCH(launch_scales_to_tiles(w->S1, (int64_t)(E * I), d->H, S1t, num_sms, stream));
    LAUNCH(launch_scales_to_tiles(w->S3, (int64_t)(E * I), d->H, S3t, num_sms, stream));
    ProbW13Nv p;
    MAP(tmap_2d_b8(&p.mXq, Xq, H, P, 128));
    MAP(tmap_fp4_unpacked(&p.mW1f, w->W1, H, I, E, 128));
    MAP(tmap_fp4_unpacked(&p.mW3f, w->W3, H, I, E, 128));
    MAP(tmap_2d(&p.mY13p, Y13p, 2 * r, P, 64, 128));
    MAP(tmap_3d(&p.mB1, w->B1, r, I, G, 64, 128));
    MAP(tmap_3d(&p.mB3, w->B3, r, I, G, 64, 128));
    p.G = Gs;
    p.U = Us;
    p.Act = Act;
    p.Actq = reinterpret_cast<uint8_t*>(sc + FL.Actq);
    p.Acts = reinterpret_cast<uint8_t*>(sc + FL.Acts);
    p.Xs = Xs;
    p.S1t = S1t;
    p.S3t = S3t;
    p.pl = pl;
    p.err = pl.err;
    p.H = d->H;
    p.I = d->I;
    p.r = d->r;
    p.act = d->act;
    p.clamp = d->act_clamp;
    LAUNCH(launch_gemm(p, max_row_tiles * (d->I / 128), num_sms, stream, K_W13_NV));
  } else if ((rc = mx ? w13(ProbW13T<true>{}) : w13(ProbW13T<false>{}))) {
    return rc;
  }
  // F4/F5: W2 + expert-local A2 shrink
  auto w2 = [&](auto p) -> int {
    MAP(tmap_2d(&p.mAct, Act, I, P, 64, 128));
    if (!mx) MAP(tmap_3d(&p.mW2, bW2, I, H, E, 64, 256));
    if (mx) MAP(tmap_3d_u8(&p.mW2q, w->W2, I / 2, H, E, 32, 256));
    p.S2q = w->S2;
    MAP(tmap_3d(&p.mA2, w->A2, I, r, G, 64, (uint32_t)((r + 15) / 16 * 16)));
    MAP(tmap_2d_store32(&p.mO, O, H, P));
    p.pl = pl;
    p.err = pl.err;
    p.O = O;
    p.Z2 = Z2;
    p.H = d->H;
    p.I = d->I;
    p.r = d->r;
    LAUNCH(launch_gemm(p, max_row_tiles * (cdiv(d->H, 256) + 1), num_sms, stream, K_W2));
    return 0;
  };
  if (nat) {
    // W2's scale bytes in the tile-major layout, then the native down product
    uint8_t* S2t = reinterpret_cast<uint8_t*>(sc + FL.S2t);
    LAUNCH(launch_scales_to_tiles(w->S2, (int64_t)(E * H), d->I, S2t, num_sms, stream));
    ProbW2Nv p;
    MAP(tmap_2d_b8(&p.mActq, sc + FL.Actq, I, P, 128));
    MAP(tmap_fp4_unpacked(&p.mW2f, w->W2, I, H, E, 256));
    MAP(tmap_2d(&p.mAct, Act, I, P, 64, 128));
    MAP(tmap_3d(&p.mA2, w->A2, I, r, G, 64, (uint32_t)((r + 15) / 16 * 16)));
    p.Acts = reinterpret_cast<const uint8_t*>(sc + FL.Acts);
    p.S2t = S2t;
    p.pl = pl;
    p.err = pl.err;
    p.O = O;
    p.Z2 = Z2;
    p.H = d->H;
    p.I = d->I;
    p.r = d->r;
    LAUNCH(launch_gemm(p, max_row_tiles * (cdiv(d->H, 256) + 1), num_sms, stream, K_W2_NV));
  } else if (kW2OneSmWide || mx) {
    if ((rc = mx ? w2(ProbW2T<true>{}) : w2(ProbW2T<false>{}))) return rc;
  } else {
    ProbW2Pair p;
    MAP(tmap_2d(&p.mAct, Act, I, P, 64, 128));
    MAP(tmap_3d(&p.mW2h, bW2, I, H, E, 64, 128));
    MAP(tmap_3d(&p.mA2h, w->A2, I, r, G, 64, r32 / 2));
    p.pl = pl;
    p.err = pl.err;
    p.O = O;
    MAP(tmap_2d_store32(&p.mO, O, H, P));
    p.Z2 = Z2;
    p.H = d->H;
    p.I = d->I;
    p.r = d->r;
    LAUNCH(launch_gemm_pair(p, max_row_tiles * (cdiv(d->H, 256) + 1), num_sms, stream, K_W2));
  }
  // F6a: per-token weighted sum of the A2 shrink
  LAUNCH(launch_z2w(pl, Z2, topk_w, Z2w, d->r, num_sms, stream));
  // F6: shared B2 expand per token (into the dead Xp buffer), then the
  // routing-weighted combine of the routed rows on top of it
  uint16_t* Yl = Xp;
  {
    ProbB2Expand p;
    MAP(tmap_2d(&p.mZ2w, Z2w, r, T, 64, 128));
    MAP(tmap_3d(&p.mB2, w->B2, r, H, A, 64, 256));
    p.pl = pl;
    p.err = pl.err;
    p.Yl = Yl;
    MAP(tmap_2d_store32(&p.mYl, Yl, H, T));
    p.H = d->H;
    p.r = d->r;
    p.s = d->scale;
    LAUNCH(launch_gemm(p, max_tok_tiles * cdiv(d->H, 256), num_sms, stream, K_B2_EXPAND));
  }
  LAUNCH(launch_combine_rows(pl, Yl, O, topk_w, y, d->H, num_sms, stream, K_COMBINE_Y));
#undef MAP
#undef LAUNCH
  (void)rc;
  return MOE_LORA_OK;
}

}  // namespace moelora
