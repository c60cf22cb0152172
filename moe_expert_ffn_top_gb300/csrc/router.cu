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
struct ProbRouter {
  static constexpr bool kAmn = false, kBmn = false;
  static constexpr int kEpiWarps = 4;  // one thread per token row, all E columns
  static constexpr bool kWide = false;
  CUtensorMap mx, mWr;  // x (H,T) box(64,128); W_r (H,E) box(64,E)
  int* err;
  int32_t* ids;
  float* w;
  float* logits;  // [T,E] or nullptr
  int64_t T;
  int H, E, k;
  __device__ int num_tiles() const { return (int)((T + 127) / 128); }
  __device__ TileInfo tile(int t) const {
    TileInfo ti;
    ti.m0 = t * 128;
    ti.mend = (int)(T < (int64_t)ti.m0 + 128 ? T : (int64_t)ti.m0 + 128);
    ti.n0 = 0;
    ti.g = 0;
    ti.sub = 0;
    ti.nk = H / kBK;
    ti.k0 = 0;
    ti.mh = 1;
    return ti;
  }
  __device__ void prefetch() const {
    tma_prefetch_map(&mx);
    tma_prefetch_map(&mWr);
  }
  __device__ void load(const TileInfo& ti, int ks, uint8_t* sa, uint8_t* sb, uint64_t* bar) const {
    mbar_arrive_expect_tx(bar, kAStage128 + E * 128);
    tma_load_2d(sa, &mx, bar, ks * kBK, ti.m0);
    tma_load_2d(sb, &mWr, bar, ks * kBK, 0);
  }
  __device__ MmaStep mma_step(const TileInfo&, int ks) const { return MmaStep{E, 0, 0, ks == 0}; }
  __device__ void epilogue(const TileInfo& ti, int row, uint32_t taddr, int, int, uint32_t* stg) const {
    const int lane = threadIdx.x & 31;
    const int64_t t = (int64_t)ti.m0 + row;
    const int64_t t0 = t - lane;  // the warp's first token
    const int nvalid = (int)(T - t0 < 32 ? T - t0 : 32);
    const bool ok = t < T;
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
  CUtensorMap mdl, mWr;  // dl (E,T) box(64,128); W_r (H,E) box(64,64)
  int* err;
  uint16_t* dx;
  int64_t T;
  int H, E;
  __device__ int ntn() const { return H / 256; }
  __device__ int num_tiles() const { return (int)((T + 127) / 128) * ntn(); }
  __device__ TileInfo tile(int t) const {
    TileInfo ti;
    ti.m0 = t / ntn() * 128;
    ti.n0 = t % ntn() * 256;
    ti.mend = (int)(T < (int64_t)ti.m0 + 128 ? T : (int64_t)ti.m0 + 128);
    ti.g = 0;
    ti.sub = 0;
    ti.nk = (E + kBK - 1) / kBK;
    ti.k0 = 0;
    ti.mh = 1;
    return ti;
  }
  __device__ void prefetch() const {
    tma_prefetch_map(&mdl);
    tma_prefetch_map(&mWr);
  }
  __device__ void load(const TileInfo& ti, int ks, uint8_t* sa, uint8_t* sb, uint64_t* bar) const {
    mbar_arrive_expect_tx(bar, kAStage128 + 4 * 8192);
    tma_load_2d(sa, &mdl, bar, ks * kBK, ti.m0);
    for (int c = 0; c < 4; ++c) tma_load_2d(sb + c * 8192, &mWr, bar, ti.n0 + c * 64, ks * kBK);
  }
  __device__ MmaStep mma_step(const TileInfo&, int ks) const { return MmaStep{256, 0, 0, ks == 0}; }
  __device__ void epilogue(const TileInfo& ti, int row, uint32_t taddr, int c0, int cs, uint32_t* stg) const {
    const int lane = threadIdx.x & 31;
    const int64_t t0 = (int64_t)ti.m0 + row - lane;  // the warp's first token
    const int nvalid = (int)(T - t0 < 32 ? T - t0 : 32);
    uint16_t* base = dx + t0 * H + ti.n0;
    for (int c = c0; c < 256; c += cs) {
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
// Router backward, weight part: dW_r = dl^T x  [E,H] fp32, K = tokens, split over
// token slices (fp32 partials summed in slice order afterwards).
// A: dl MN-major (experts contiguous); B: x MN-major.
// =====================================================================================
struct ProbRouterDW {
  static constexpr bool kAmn = true, kBmn = true;
  static constexpr int kEpiWarps = 4;
  static constexpr bool kWide = false;
  CUtensorMap mdl, mx;  // dl (E,T) box(64,64); x (H,T) box(64,64)
  int* err;
  float* out;  // dW_r, or the split partials
  int64_t split_stride;
  int64_t T;
  int H, E, split;
  __device__ int ntm() const { return (E + 127) / 128; }
  __device__ int ntn() const { return H / 256; }
  __device__ int num_tiles() const { return split * ntm() * ntn(); }
  __device__ TileInfo tile(int t) const {
    const int per = ntm() * ntn();
    const int sp = t / per, rem = t % per;
    TileInfo ti;
    ti.m0 = rem / ntn() * 128;
    ti.n0 = rem % ntn() * 256;
    ti.mend = E;
    ti.g = 0;
    ti.sub = sp;
    const int nk = (int)((T + kBK - 1) / kBK), cs = (nk + split - 1) / split;
    ti.k0 = sp * cs * kBK;
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
  __device__ float* warp_rows(const TileInfo& ti, int row, int& nvalid) const {
    const int m0 = ti.m0 + row - (threadIdx.x & 31);  // the warp's first expert row
    nvalid = E - m0;
    return out + ti.sub * split_stride + (int64_t)m0 * H + ti.n0;
  }
  __device__ void epilogue(const TileInfo& ti, int row, uint32_t taddr, int c0, int cs, uint32_t* stg) const {
    int nvalid;
    float* o0 = warp_rows(ti, row, nvalid);
    for (int c = c0; c < 256; c += cs) {
      float v[32];
      tmem_ld32(taddr + c, v);
      warp_store_rows_f32(o0 + c, H, nvalid, v, 1.0f, 32, stg);
    }
  }
  // a token slice with no K steps still owns its partial: zeros
  __device__ void epilogue_empty(const TileInfo& ti, int row, int c0, int cs) const {
    const int m = ti.m0 + row;
    if (m >= E) return;
    const float z[32] = {};
    float* o = out + ti.sub * split_stride + (int64_t)m * H + ti.n0;
    for (int c = c0; c < 256; c += cs) store_row_f32(o + c, z, 0.0f, 32);
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

int run_router_forward(const moe_lora_dims* d, const uint16_t* x, const uint16_t* Wr, int32_t* ids, float* w,
                       float* logits, void* scratch, int num_sms, cudaStream_t stream) {
  const RouterLayout L = router_layout(d);
  int* err = (int*)(static_cast<char*>(scratch) + L.err);
  LAUNCH(cudaMemsetAsync(err, 0, 16, stream));
  if (d->T == 0) return MOE_LORA_OK;
  ProbRouter p;
  MAP(tmap_2d(&p.mx, x, d->H, d->T, 64, 128));
  MAP(tmap_2d(&p.mWr, Wr, d->H, d->E, 64, d->E));
  p.err = err;
  p.ids = ids;
  p.w = w;
  p.logits = logits;
  p.T = d->T;
  p.H = d->H;
  p.E = d->E;
  p.k = d->k;
  LAUNCH(launch_gemm(p, (int)((d->T + 127) / 128), num_sms, stream, K_ROUTER_FWD));
  return MOE_LORA_OK;
}

int run_router_backward(const moe_lora_dims* d, const uint16_t* x, const uint16_t* Wr, const int32_t* ids,
                        const float* w, const float* dw, float* dlogits, float* dWr, uint16_t* dx, void* scratch,
                        int num_sms, cudaStream_t stream) {
  const RouterLayout L = router_layout(d);
  char* sc = static_cast<char*>(scratch);
  int* err = (int*)(sc + L.err);
  uint16_t* dl = (uint16_t*)(sc + L.dl);
  float* part = (float*)(sc + L.part);
  const int64_t T = d->T;
  const int H = d->H, E = d->E;
  LAUNCH(cudaMemsetAsync(err, 0, 16, stream));
  if (T == 0) {  // no tokens: dW_r = 0, nothing else to write
    LAUNCH(cudaMemsetAsync(dWr, 0, sizeof(float) * (size_t)E * H, stream));
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
    MAP(tmap_2d(&p.mWr, Wr, H, E, 64, 64));
    p.err = err;
    p.dx = dx;
    p.T = T;
    p.H = H;
    p.E = E;
    LAUNCH(launch_gemm(p, (int)((T + 127) / 128) * (H / 256), num_sms, stream, K_ROUTER_DX));
  }
  {
    // token slices of at least 256 K steps (16,384 tokens); fixed by the sizes alone
    const int64_t nk = (T + 63) / 64;
    const int split = (int)std::min<int64_t>(kMaxSplit, std::max<int64_t>(1, nk / 256));
    ProbRouterDW p;
    MAP(tmap_2d(&p.mdl, dl, E, T, 64, 64));
    MAP(tmap_2d(&p.mx, x, H, T, 64, 64));
    p.err = err;
    p.split = split;
    p.out = split > 1 ? part : dWr;
    p.split_stride = (int64_t)E * H;
    p.T = T;
    p.H = H;
    p.E = E;
    LAUNCH(launch_gemm(p, split * ((E + 127) / 128) * (H / 256), num_sms, stream, K_ROUTER_DW));
    if (split > 1) LAUNCH(launch_reduce_splits(part, p.split_stride, split, p.split_stride, dWr, num_sms, stream));
  }
  return MOE_LORA_OK;
}

}  // namespace moelora
