// The routing step ahead of the expert path, and its backward.
//
// PR #9 ("feat(mega): add fused shared side-LoRA kernels", Correctness coverage)
// takes the routes as inputs and returns their weight gradient ("grad-route");
// this file makes the routes and carries that gradient to the router:
//
//   forward   l = x W_r^T (fp32), softmax over all E, the k largest (ties to the
//             lower expert id), weights renormalised to sum 1.  One GEMM launch:
//             a 128-token tile holds whole logit rows (N = E <= 256), so the
//             epilogue thread that owns a token row does the softmax and the
//             top-k from tensor memory.
//   backward  dl_t = w_t * (dw_t - <w_t, dw_t>) on the selected experts, 0 elsewhere
//             (w_t is the softmax of the selected logits alone, so the full-softmax
//             normaliser cancels); dx += dl W_r and dW_r = dl^T x on the tensor
//             cores, the dense dl [T,E] as their bf16 operand.
//
// Several adapters (OpenPipe/ART PR #1139, Behavior: one router per adapter) own
// contiguous token ranges starting at multiples of 128; adapter a's tokens use
// W_r[a] and produce dW_r[a].  Every tile lies in one adapter's range, and the
// token-split of each adapter's dW_r reduction depends on that adapter's token
// count alone, so each adapter's results equal its standalone run bit for bit.
#include <algorithm>

#include "gemm_problems.cuh"
#include "launch.h"
#include "passes.h"
#include "tmap.h"

namespace moelora {

// =====================================================================================
// Router forward: logits of 128 tokens x E experts, softmax + top-k in the epilogue.
// A: x K-major; B: W_r K-major (one box of E rows).
// =====================================================================================
// The 128-token tile t of an adapter table: rows [m0, min(m0+128, end of its adapter)).
__device__ __forceinline__ TileInfo adapter_token_tile(const AdapterTable& at, int t) {
  int a = 0;
  while (a + 1 < at.n && t >= at.tok_tile[a + 1]) ++a;
  TileInfo ti;
  ti.g = a;
  ti.m0 = at.tok_off[a] + (t - at.tok_tile[a]) * 128;
  ti.mend = at.tok_off[a + 1] < ti.m0 + 128 ? at.tok_off[a + 1] : ti.m0 + 128;
  ti.n0 = 0;
  ti.sub = 0;
  ti.k0 = 0;
  ti.mh = 1;
  return ti;
}

struct ProbRouter {
  static constexpr bool kAmn = false, kBmn = false;
  static constexpr int kEpiWarps = 4;  // one thread per token row, all E columns
  static constexpr bool kWide = false;
  CUtensorMap mx, mWr;  // x (H,T) box(64,128); W_r (H,E,A) box(64,E,1)
  AdapterTable at;
  int* err;
  int32_t* ids;
  float* w;
  float* logits;  // [T,E] or nullptr
  int64_t T;
  int H, E, k;
  __device__ int num_tiles() const { return at.tok_tile[at.n]; }
  __device__ TileInfo tile(int t) const {
    TileInfo ti = adapter_token_tile(at, t);
    ti.nk = H / kBK;
    return ti;
  }
  __device__ void prefetch() const {
    tma_prefetch_map(&mx);
    tma_prefetch_map(&mWr);
  }
  __device__ void load(const TileInfo& ti, int ks, uint8_t* sa, uint8_t* sb, uint64_t* bar) const {
    mbar_arrive_expect_tx(bar, kAStage128 + E * 128);
    tma_load_2d(sa, &mx, bar, ks * kBK, ti.m0);
    tma_load_3d(sb, &mWr, bar, ks * kBK, 0, ti.g);
  }
  __device__ MmaStep mma_step(const TileInfo&, int ks) const { return MmaStep{E, 0, 0, ks == 0}; }
  __device__ void epilogue(const TileInfo& ti, int row, uint32_t taddr, int, int, uint32_t* stg) const {
    const int lane = threadIdx.x & 31;
    const int64_t t = (int64_t)ti.m0 + row;
    const int64_t t0 = t - lane;  // the warp's first token
    const int nvalid = (int)(ti.mend - t0 < 32 ? ti.mend - t0 : 32);
    const bool ok = t < ti.mend;
    // pass 1: row maximum (and the logits, if asked for)
    float mx = -INFINITY;
    for (int c = 0; c < E; c += 32) {
      float v[32];
      tmem_ld32(taddr + c, v);
      const int n = E - c < 32 ? E - c : 32;
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (i < n) mx = fmaxf(mx, v[i]);
      if (logits) warp_store_rows_f32(logits + t0 * E + c, E, nvalid, v, 1.0f, n, stg);
    }
    // pass 2: softmax normaliser, experts in ascending order
    float z = 0.0f;
    for (int c = 0; c < E; c += 32) {
      float v[32];
      tmem_ld32(taddr + c, v);
      const int n = E - c < 32 ? E - c : 32;
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (i < n) z += expf(v[i] - mx);
    }
    // k selection passes in the order (logit descending, expert id ascending): pass j
    // takes the best element strictly after pass j-1's pick (pv, pi) in that order.
    float pv = INFINITY, S = 0.0f;
    int pi = -1;
    for (int j = 0; j < k; ++j) {
      float bv = -INFINITY;
      int bi = -1;
      for (int c = 0; c < E; c += 32) {
        float v[32];
        tmem_ld32(taddr + c, v);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int e = c + i;
          const float x = v[i];
          const bool after = x < pv || (x == pv && e > pi);
          if (e < E && after && (bi < 0 || x > bv)) {
            bv = x;
            bi = e;
          }
        }
      }
      const float p = bi >= 0 ? expf(bv - mx) / z : 0.0f;
      if (ok) {
        ids[t * k + j] = bi;
        w[t * k + j] = p;
      }
      S += p;
      if (bi >= 0) {
        pv = bv;
        pi = bi;
      } else {  // nothing left (non-finite logits): later passes find nothing either
        pv = -INFINITY;
        pi = 0x7fffffff;
      }
    }
    if (ok)
      for (int j = 0; j < k; ++j) w[t * k + j] = S > 0.0f ? w[t * k + j] / S : 0.0f;
  }
  __device__ void epilogue_empty(const TileInfo&, int, int, int) const {}
};

// =====================================================================================
// Router backward, grad-x part: dx[t, n0:n0+256] <- bf16(dx + dl_t W_r).
// M = tokens, N = H (tiles of 256), K = E.  A: dl K-major; B: W_r MN-major.
// =====================================================================================
struct ProbRouterDx {
  static constexpr bool kAmn = false, kBmn = true;
  static constexpr int kEpiWarps = 8;  // load + store epilogue: two warps per lane quarter
  static constexpr bool kWide = false;
  CUtensorMap mdl, mWr;  // dl (E,T) box(64,128); W_r (H,E,A) box(64,64,1)
  AdapterTable at;
  int* err;
  uint16_t* dx;
  int64_t T;
  int H, E;
  __device__ int ntn() const { return cdiv(H, 256); }
  __device__ int num_tiles() const { return at.tok_tile[at.n] * ntn(); }
  __device__ TileInfo tile(int t) const {
    TileInfo ti = adapter_token_tile(at, t / ntn());
    ti.n0 = t % ntn() * 256;
    ti.nk = (E + kBK - 1) / kBK;
    return ti;
  }
  __device__ void prefetch() const {
    tma_prefetch_map(&mdl);
    tma_prefetch_map(&mWr);
  }
  __device__ void load(const TileInfo& ti, int ks, uint8_t* sa, uint8_t* sb, uint64_t* bar) const {
    mbar_arrive_expect_tx(bar, kAStage128 + 4 * 8192);
    tma_load_2d(sa, &mdl, bar, ks * kBK, ti.m0);
    for (int c = 0; c < 4; ++c) tma_load_3d(sb + c * 8192, &mWr, bar, ti.n0 + c * 64, ks * kBK, ti.g);
  }
  __device__ MmaStep mma_step(const TileInfo&, int ks) const { return MmaStep{256, 0, 0, ks == 0}; }
  __device__ void epilogue(const TileInfo& ti, int row, uint32_t taddr, int c0, int cs, uint32_t* stg) const {
    const int lane = threadIdx.x & 31;
    const int64_t t0 = (int64_t)ti.m0 + row - lane;  // the warp's first token
    const int nvalid = (int)(ti.mend - t0 < 32 ? ti.mend - t0 : 32);
    uint16_t* base = dx + t0 * H + ti.n0;
    for (int c = c0; c < 256 && ti.n0 + c < H; c += cs) {
      uint4 u[4];
#pragma unroll
      for (int s = 0; s < 4; ++s) {  // coalesced loads of the warp's rows, guarded at the tail
        const int r = s * 8 + (lane >> 2);
        u[s] = r < nvalid ? *reinterpret_cast<const uint4*>(base + (int64_t)r * H + c + (lane & 3) * 8)
                          : make_uint4(0, 0, 0, 0);
      }
      float a[32], cur[32];
      tmem_ld32(taddr + c, a);
      warp_rows_to_lane(u, stg, cur);
#pragma unroll
      for (int i = 0; i < 32; ++i) a[i] += cur[i];
      warp_store_rows_bf16(base + c, H, nvalid, a, 1.0f, stg);
    }
  }
  __device__ void epilogue_empty(const TileInfo&, int, int, int) const {}
};

// =====================================================================================
// Router backward, weight part: dW_r[a] = dl^T x over adapter a's tokens  [E,H] fp32.
// K = tokens; adapter a's token range is cut into split[a] slices of whole 64-token
// steps (fp32 partials summed in slice order afterwards when split[a] > 1).
// A: dl MN-major (experts contiguous); B: x MN-major.
// =====================================================================================
struct ProbRouterDW {
  static constexpr bool kAmn = true, kBmn = true;
  static constexpr int kEpiWarps = 4;
  static constexpr bool kWide = false;
  CUtensorMap mdl, mx;  // dl (E,T) box(64,64); x (H,T) box(64,64)
  AdapterTable at;
  int split[kMaxAdapters];      // token slices of each adapter
  int tbase[kMaxAdapters + 1];  // first tile of each adapter
  int* err;
  float* dWr;   // [A,E,H]
  float* part;  // [A][kMaxSplit][E,H] partials
  int64_t T;
  int H, E;
  __device__ int ntm() const { return (E + 127) / 128; }
  __device__ int ntn() const { return cdiv(H, 256); }
  __device__ int num_tiles() const { return tbase[at.n]; }
  __device__ TileInfo tile(int t) const {
    int a = 0;
    while (a + 1 < at.n && t >= tbase[a + 1]) ++a;
    const int per = ntm() * ntn(), u = t - tbase[a];
    const int sp = u / per, rem = u % per;
    TileInfo ti;
    ti.m0 = rem / ntn() * 128;
    ti.n0 = rem % ntn() * 256;
    ti.mend = E;
    ti.g = a;
    ti.sub = sp;
    const int nk = (at.tok_off[a + 1] - at.tok_off[a] + kBK - 1) / kBK, cs = (nk + split[a] - 1) / split[a];
    ti.k0 = at.tok_off[a] + sp * cs * kBK;
    ti.nk = max(0, min(cs, nk - sp * cs));
    ti.mh = 1;
    return ti;
  }
  __device__ void prefetch() const {
    tma_prefetch_map(&mdl);
    tma_prefetch_map(&mx);
  }
  __device__ void load(const TileInfo& ti, int ks, uint8_t* sa, uint8_t* sb, uint64_t* bar) const {
    const int kt = ti.k0 + ks * kBK;
    mbar_arrive_expect_tx(bar, kAStage128 + 4 * 8192);
    tma_load_2d(sa, &mdl, bar, ti.m0, kt);
    tma_load_2d(sa + 8192, &mdl, bar, ti.m0 + 64, kt);
    for (int c = 0; c < 4; ++c) tma_load_2d(sb + c * 8192, &mx, bar, ti.n0 + c * 64, kt);
  }
  __device__ MmaStep mma_step(const TileInfo&, int ks) const { return MmaStep{256, 0, 0, ks == 0}; }
  // adapter a's output (split 1) or its slice's partial
  __device__ float* out_of(const TileInfo& ti) const {
    return split[ti.g] > 1 ? part + ((int64_t)ti.g * kMaxSplit + ti.sub) * E * H : dWr + (int64_t)ti.g * E * H;
  }
  __device__ void epilogue(const TileInfo& ti, int row, uint32_t taddr, int c0, int cs, uint32_t* stg) const {
    const int m0 = ti.m0 + row - (threadIdx.x & 31);  // the warp's first expert row
    float* o0 = out_of(ti) + (int64_t)m0 * H + ti.n0;
    for (int c = c0; c < 256 && ti.n0 + c < H; c += cs) {
      float v[32];
      tmem_ld32(taddr + c, v);
      warp_store_rows_f32(o0 + c, H, E - m0, v, 1.0f, 32, stg);
    }
  }
  // a token slice (or an adapter) with no K steps still owns its output: zeros
  __device__ void epilogue_empty(const TileInfo& ti, int row, int c0, int cs) const {
    const int m = ti.m0 + row;
    if (m >= E) return;
    const float z[32] = {};
    float* o = out_of(ti) + (int64_t)m * H + ti.n0;
    for (int c = c0; c < 256 && ti.n0 + c < H; c += cs) store_row_f32(o + c, z, 0.0f, 32);
  }
};

// dl [T,E] bf16 (and fp32 if asked for): one warp per token, lane j holds slot j.
__global__ void __launch_bounds__(256) router_dl_kernel(const int32_t* __restrict__ ids, const float* __restrict__ w,
                                                        const float* __restrict__ dw, int64_t T, int k, int E,
                                                        uint16_t* __restrict__ dl, float* __restrict__ dl32) {
  const int lane = threadIdx.x & 31;
  const int64_t nw = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t t = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); t < T; t += nw) {
    int id = -1;
    float wj = 0.0f, dwj = 0.0f;
    if (lane < k) {
      id = ids[t * k + lane];
      if (id >= 0 && id < E) {
        wj = w[t * k + lane];
        dwj = dw[t * k + lane];
      } else {
        id = -1;
      }
    }
    float s = wj * dwj;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    const float g = wj * (dwj - s);
    float acc[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) acc[q] = 0.0f;
    for (int j = 0; j < k; ++j) {
      const int idj = __shfl_sync(0xffffffffu, id, j);
      const float gj = __shfl_sync(0xffffffffu, g, j);
#pragma unroll
      for (int q = 0; q < 8; ++q)
        if (idj == lane + 32 * q) acc[q] += gj;
    }
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int e = lane + 32 * q;
      if (e < E) {
        dl[t * E + e] = __bfloat16_as_ushort(__float2bfloat16_rn(acc[q]));
        if (dl32) dl32[t * E + e] = acc[q];
      }
    }
  }
}

#define MAP(call)                                 \
  do {                                            \
    if ((call) != 0) return MOE_LORA_ERR_CUDA;    \
  } while (0)
#define LAUNCH(call)                                     \
  do {                                                   \
    if ((call) != cudaSuccess) return MOE_LORA_ERR_CUDA; \
  } while (0)

int run_router_forward(const moe_lora_dims* d, const AdapterTable& at, const uint16_t* x, const uint16_t* Wr,
                       int32_t* ids, float* w, float* logits, void* scratch, int num_sms, cudaStream_t stream) {
  const RouterLayout L = router_layout(d);
  int* err = (int*)(static_cast<char*>(scratch) + L.err);
  LAUNCH(cudaMemsetAsync(err, 0, 16, stream));
  if (d->T == 0) return MOE_LORA_OK;
  ProbRouter p;
  MAP(tmap_2d(&p.mx, x, d->H, d->T, 64, 128));
  MAP(tmap_3d(&p.mWr, Wr, d->H, d->E, d->A, 64, d->E));
  p.at = at;
  p.err = err;
  p.ids = ids;
  p.w = w;
  p.logits = logits;
  p.T = d->T;
  p.H = d->H;
  p.E = d->E;
  p.k = d->k;
  LAUNCH(launch_gemm(p, at.tok_tile[at.n], num_sms, stream, K_ROUTER_FWD));
  return MOE_LORA_OK;
}

// Token slices of one adapter's dW_r reduction: at least 256 K steps (16,384 tokens)
// each, at most kMaxSplit; a function of that adapter's token count alone.
static int router_split(int64_t tokens) {
  const int64_t nk = (tokens + 63) / 64;
  return (int)std::min<int64_t>(kMaxSplit, std::max<int64_t>(1, nk / 256));
}

int run_router_backward(const moe_lora_dims* d, const AdapterTable& at, const uint16_t* x, const uint16_t* Wr,
                        const int32_t* ids, const float* w, const float* dw, float* dlogits, float* dWr, uint16_t* dx,
                        void* scratch, int num_sms, cudaStream_t stream) {
  const RouterLayout L = router_layout(d);
  char* sc = static_cast<char*>(scratch);
  int* err = (int*)(sc + L.err);
  uint16_t* dl = (uint16_t*)(sc + L.dl);
  float* part = (float*)(sc + L.part);
  const int64_t T = d->T;
  const int H = d->H, E = d->E, A = d->A;
  LAUNCH(cudaMemsetAsync(err, 0, 16, stream));
  if (T == 0) {  // no tokens: dW_r = 0, nothing else to write
    LAUNCH(cudaMemsetAsync(dWr, 0, sizeof(float) * (size_t)A * E * H, stream));
    return MOE_LORA_OK;
  }
  {
    const int64_t blocks = (T + 7) / 8;
    const int grid = (int)(blocks < 8LL * num_sms ? blocks : 8LL * num_sms);
    prof_begin(K_ROUTER_DL, stream);
    router_dl_kernel<<<grid, 256, 0, stream>>>(ids, w, dw, T, d->k, E, dl, dlogits);
    prof_end(K_ROUTER_DL, stream);
    LAUNCH(cudaGetLastError());
  }
  {
    ProbRouterDx p;
    MAP(tmap_2d(&p.mdl, dl, E, T, 64, 128));
    MAP(tmap_3d(&p.mWr, Wr, H, E, A, 64, 64));
    p.at = at;
    p.err = err;
    p.dx = dx;
    p.T = T;
    p.H = H;
    p.E = E;
    LAUNCH(launch_gemm(p, at.tok_tile[at.n] * cdiv(H, 256), num_sms, stream, K_ROUTER_DX));
  }
  {
    ProbRouterDW p;
    MAP(tmap_2d(&p.mdl, dl, E, T, 64, 64));
    MAP(tmap_2d(&p.mx, x, H, T, 64, 64));
    p.at = at;
    const int per = ((E + 127) / 128) * cdiv(H, 256);
    p.tbase[0] = 0;
    for (int a = 0; a < A; ++a) {
      p.split[a] = router_split(at.tok_off[a + 1] - at.tok_off[a]);
      p.tbase[a + 1] = p.tbase[a] + p.split[a] * per;
    }
    p.err = err;
    p.dWr = dWr;
    p.part = part;
    p.T = T;
    p.H = H;
    p.E = E;
    LAUNCH(launch_gemm(p, p.tbase[A], num_sms, stream, K_ROUTER_DW));
    const int64_t n = (int64_t)E * H;
    for (int a = 0; a < A; ++a)
      if (p.split[a] > 1)
        LAUNCH(launch_reduce_splits(part + (int64_t)a * kMaxSplit * n, n, p.split[a], n, dWr + a * n, num_sms,
                                    stream));
  }
  return MOE_LORA_OK;
}

}  // namespace moelora
