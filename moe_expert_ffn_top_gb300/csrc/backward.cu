// Backward pass of the routed MoE side-LoRA FFN: the input gradient, the
// routing-weight gradient and all six factor gradients, nothing for the frozen
// base weights ("feat(mega): add fused shared side-LoRA kernels", Summary).
// Launch sequence, one stream, no host synchronisation:
//   B1a dyB2 = dy B2 (per token)      B1b dB2 = s dy^T Z2w
//   B2  gather dy rows, s*dyB2, s*w*dyB2 (zero padding)
//   B3  W2^T dgrad + A2 path + SwiGLU backward + router partial dots
//       dw reduce;  dA2 (K-grouped per expert)
//   B5  W13^T dgrad + B1/B3 path;  dB1/dB3 (K-grouped per expert)
//   B6a per-token sum of dY13;  B6 grad-x (A1/A3 path per token, then the source
//       combine of the routed dXp rows);  dA1/dA3
#include "gemm_problems.cuh"
#include "launch.h"
#include "passes.h"
#include "tmap.h"

namespace moelora {

int run_backward(const moe_lora_dims* d, const void* plan_ws, const void* saved, const uint16_t* x,
                 const float* topk_w, const uint16_t* dy, const moe_lora_weights* w, uint16_t* dx, float* dw,
                 const moe_lora_grads* gr, void* scratch, int num_sms, cudaStream_t stream) {
  const PlanView pl = make_plan_view(d, plan_ws);
  const SavedLayout SL = saved_layout(d);
  const BwdLayout BL = bwd_layout(d);
  const char* sv = static_cast<const char*>(saved);
  char* sc = static_cast<char*>(scratch);
  const uint16_t* Y13p = (const uint16_t*)(sv + SL.Y13p);
  const uint16_t* Gs = (const uint16_t*)(sv + SL.G);
  const uint16_t* Us = (const uint16_t*)(sv + SL.U);
  const uint16_t* Act = (const uint16_t*)(sv + SL.Act);
  const uint16_t* Z2w = (const uint16_t*)(sv + SL.Z2w);
  uint16_t* dyB2 = (uint16_t*)(sc + BL.dyB2);
  uint16_t* Dp = (uint16_t*)(sc + BL.Dp);
  uint16_t* dXp = Dp;  // Dp is dead once B3 has run
  uint16_t* D2p = (uint16_t*)(sc + BL.D2p);
  uint16_t* dZ2p = (uint16_t*)(sc + BL.dZ2p);
  uint16_t* dG = (uint16_t*)(sc + BL.dG);
  uint16_t* dU = (uint16_t*)(sc + BL.dU);
  float* part = (float*)(sc + BL.part);
  float* dY13 = (float*)(sc + BL.dY13);
  uint16_t* dY13w = (uint16_t*)(sc + BL.dY13w);
  uint16_t* dXl = (uint16_t*)(sc + BL.dXl);
  float* ksplit = (float*)(sc + BL.ksplit);
  // Token-range slices for the two long-K reductions (dB2, dA1/dA3), at least 256
  // K steps (16,384 tokens) each.  The choice depends only on the adapter's own
  // token count, and several adapters are never split, so an adapter's gradients
  // from a shared pass equal its standalone run bit for bit whenever it has fewer
  // than 32,768 tokens.
  auto pick_split = [&]() {
    if (d->A > 1) return 1;
    const int64_t sp = ((d->T + 63) / 64) / 256;
    return (int)(sp < 1 ? 1 : sp > kMaxSplit ? kMaxSplit : sp);
  };

  const uint64_t T = (uint64_t)d->T, H = d->H, I = d->I, E = d->E, A = d->A, r = d->r;
  const uint64_t P = (uint64_t)rows_cap(d), G = A * E;
  const int max_tok_tiles = (int)((T + 127) / 128) + d->A;
  const int max_row_tiles = (int)(P / 128);
  cudaError_t ce;
  // An MXFP4 base: decoded inside the two dgrad GEMMs, stage by stage (base_fmt 1,
  // the ...T<true> problem types), or the bf16 copy the forward decoded into `saved`
  // (base_fmt 2).
  const bool mx = fmt_in_gemm(d);
  const void* bW1 = fmt_once(d) ? (const void*)(sv + SL.W1) : w->W1;
  const void* bW3 = fmt_once(d) ? (const void*)(sv + SL.W3) : w->W3;
  const void* bW2 = fmt_once(d) ? (const void*)(sv + SL.W2) : w->W2;
#define MAP(call)                                 \
  do {                                            \
    if ((call) != 0) return MOE_LORA_ERR_CUDA;    \
  } while (0)
#define LAUNCH(call)                                            \
  do {                                                          \
    if ((ce = (call)) != cudaSuccess) return MOE_LORA_ERR_CUDA; \
  } while (0)

  // B1a: dyB2 = bf16(dy B2)
  {
    ProbDyB2 p;
    MAP(tmap_2d(&p.mdy, dy, H, T, 64, 128));
    MAP(tmap_3d(&p.mB2, w->B2, r, H, A, 64, 64));
    p.pl = pl;
    p.err = pl.err;
    p.dyB2 = dyB2;
    p.H = d->H;
    p.r = d->r;
    LAUNCH(launch_gemm(p, max_tok_tiles, num_sms, stream, K_DYB2));
  }
  // B1b: dB2 = s dy^T Z2w
  {
    ProbDB2 p;
    MAP(tmap_2d(&p.mdy, dy, H, T, 64, 64));
    MAP(tmap_2d(&p.mZ2w, Z2w, r, T, 64, 64));
    p.pl = pl;
    p.err = pl.err;
    p.split = pick_split();
    p.out = p.split > 1 ? ksplit : gr->dB2;
    p.split_stride = (int64_t)A * H * r;
    p.H = d->H;
    p.r = d->r;
    p.s = d->scale;
    LAUNCH(launch_gemm(p, p.split * d->A * cdiv(d->H, 128), num_sms, stream, K_DB2));
    if (p.split > 1) LAUNCH(launch_reduce_splits(ksplit, p.split_stride, p.split, p.split_stride, gr->dB2, num_sms, stream));
  }
  // B2: routed dy rows and the scaled shared-expand gradients
  LAUNCH(launch_gather_bwd(pl, dy, dyB2, topk_w, Dp, D2p, dZ2p, d->H, d->r, d->scale, num_sms, stream));
  // B3/B4: W2^T dgrad + A2 path + SwiGLU backward + router dots
  auto w2d = [&](auto p) -> int {
    MAP(tmap_2d(&p.mDp, Dp, H, P, 64, 128));
    MAP(tmap_2d(&p.mD2p, D2p, r, P, 64, 128));
    if (!mx) MAP(kMnChunkCopy ? tmap_mn4(&p.mW2, bW2, I, H, E) : tmap_3d(&p.mW2, bW2, I, H, E, 64, 64));
    if (mx) MAP(tmap_3d_u8(&p.mW2q, w->W2, I / 2, H, E, 128, 64));
    p.S2q = w->S2;
    MAP(kMnChunkCopy ? tmap_mn4(&p.mA2, w->A2, I, r, G) : tmap_3d(&p.mA2, w->A2, I, r, G, 64, 64));
    p.pl = pl;
    p.err = pl.err;
    p.topk_w = topk_w;
    p.G = Gs;
    p.U = Us;
    p.dG = dG;
    p.dU = dU;
    MAP(tmap_2d_store32(&p.mdG, dG, I, P));
    MAP(tmap_2d_store32(&p.mdU, dU, I, P));
    p.part = part;
    p.H = d->H;
    p.I = d->I;
    p.r = d->r;
    p.act = d->act;
    p.clamp = d->act_clamp;
    LAUNCH(launch_gemm(p, max_row_tiles * cdiv(d->I, 256), num_sms, stream, K_W2_DGRAD));
    return 0;
  };
  if (int rc = mx ? w2d(ProbW2DgradT<true>{}) : w2d(ProbW2DgradT<false>{})) return rc;
  const int parts = mx ? ProbW2DgradT<true>::kPartsPerTile : ProbW2DgradT<false>::kPartsPerTile;
  if (fmt_native(d))  // the down product ran on q8(Act): dw from the forward's O and Z2 rows
    LAUNCH(launch_dw_from_o(pl, dy, dyB2, (const uint16_t*)(sv + SL.O), (const uint16_t*)(sv + SL.Z2), d->H, d->r,
                            d->scale, dw, num_sms, stream));
  else
    LAUNCH(launch_dw(pl, part, parts * cdiv(d->I, 256), dw, num_sms, stream));
  // dA2 per (adapter, expert)
  {
    ProbDA2 p;
    MAP(tmap_2d(&p.mdZ2p, dZ2p, r, P, 64, 64));
    MAP(tmap_2d(&p.mAct, Act, I, P, 64, 64));
    p.pl = pl;
    p.err = pl.err;
    p.dA2 = gr->dA2;
    p.I = d->I;
    p.r = d->r;
    LAUNCH(launch_gemm(p, (int)G * cdiv(d->I, 256), num_sms, stream, K_DA2));
  }
  // B5: W13^T dgrad + B1/B3 path
  auto w13d = [&](auto p) -> int {
    MAP(tmap_2d(&p.mdG, dG, I, P, 64, 128));
    MAP(tmap_2d(&p.mdU, dU, I, P, 64, 128));
    if (!mx) {
      MAP(kMnChunkCopy ? tmap_mn4(&p.mW1, bW1, H, I, E) : tmap_3d(&p.mW1, bW1, H, I, E, 64, 64));
      MAP(kMnChunkCopy ? tmap_mn4(&p.mW3, bW3, H, I, E) : tmap_3d(&p.mW3, bW3, H, I, E, 64, 64));
    }
    if (mx) {
      MAP(tmap_3d_u8(&p.mW1q, w->W1, H / 2, I, E, 128, 64));
      MAP(tmap_3d_u8(&p.mW3q, w->W3, H / 2, I, E, 128, 64));
    }
    p.S1q = w->S1;
    p.S3q = w->S3;
    MAP(tmap_3d(&p.mB1, w->B1, r, I, G, 64, 64));
    MAP(tmap_3d(&p.mB3, w->B3, r, I, G, 64, 64));
    p.pl = pl;
    p.err = pl.err;
    p.dXp = dXp;
    MAP(tmap_2d_store32(&p.mdXp, dXp, H, P));
    p.dY13 = dY13;
    p.H = d->H;
    p.I = d->I;
    p.r = d->r;
    p.s = d->scale;
    LAUNCH(launch_gemm(p, max_row_tiles * (cdiv(d->H, 256) + 1), num_sms, stream, K_W13_DGRAD));
    return 0;
  };
  if (int rc = mx ? w13d(ProbW13DgradT<true>{}) : w13d(ProbW13DgradT<false>{})) return rc;
  // dB1 / dB3 per (adapter, expert)
  {
    ProbDB13 p;
    MAP(tmap_2d(&p.mdG, dG, I, P, 64, 64));
    MAP(tmap_2d(&p.mdU, dU, I, P, 64, 64));
    MAP(tmap_2d(&p.mY13p, Y13p, 2 * r, P, 64, 64));
    p.pl = pl;
    p.err = pl.err;
    p.dB1 = gr->dB1;
    p.dB3 = gr->dB3;
    p.I = d->I;
    p.r = d->r;
    LAUNCH(launch_gemm(p, 2 * (int)G * cdiv(d->I, 128), num_sms, stream, K_DB13));
  }
  // B6a: per-token sum of the shared-shrink gradients
  LAUNCH(launch_dy13w(pl, dY13, dY13w, 2 * d->r, num_sms, stream));
  // B6: grad-x through the shared A1/A3 per token, then the source combine of dXp
  {
    ProbA13Expand p;
    MAP(tmap_2d(&p.mdY13w, dY13w, 2 * r, T, 64, 128));
    MAP(tmap_3d(&p.mA1, w->A1, H, r, A, 64, 64));
    MAP(tmap_3d(&p.mA3, w->A3, H, r, A, 64, 64));
    p.pl = pl;
    p.err = pl.err;
    p.dXl = dXl;
    MAP(tmap_2d_store32(&p.mdXl, dXl, H, T));
    p.H = d->H;
    p.r = d->r;
    LAUNCH(launch_gemm(p, max_tok_tiles * cdiv(d->H, 256), num_sms, stream, K_A13_EXPAND));
  }
  LAUNCH(launch_combine_rows(pl, dXl, dXp, nullptr, dx, d->H, num_sms, stream, K_COMBINE_DX));
  // dA1 / dA3 per adapter
  {
    ProbDA13 p;
    MAP(tmap_2d(&p.mdY13w, dY13w, 2 * r, T, 64, 64));
    MAP(tmap_2d(&p.mx, x, H, T, 64, 64));
    p.pl = pl;
    p.err = pl.err;
    const int tiles = d->A * ((2 * d->r + 127) / 128) * cdiv(d->H, 256);
    p.split = pick_split();
    const int64_t n1 = (int64_t)A * r * H;
    p.out1 = p.split > 1 ? ksplit : gr->dA1;
    p.out3 = p.split > 1 ? ksplit + n1 : gr->dA3;
    p.split_stride = 2 * n1;
    p.H = d->H;
    p.r = d->r;
    LAUNCH(launch_gemm(p, p.split * tiles, num_sms, stream, K_DA13));
    if (p.split > 1) {
      LAUNCH(launch_reduce_splits(ksplit, 2 * n1, p.split, n1, gr->dA1, num_sms, stream));
      LAUNCH(launch_reduce_splits(ksplit + n1, 2 * n1, p.split, n1, gr->dA3, num_sms, stream));
    }
  }
#undef MAP
#undef LAUNCH
  return MOE_LORA_OK;
}

}  // namespace moelora
