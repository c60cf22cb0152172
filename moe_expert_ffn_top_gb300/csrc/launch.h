// Host-side launch interface between the C-ABI entry points and the kernels.
#pragma once
#include <cuda_runtime.h>

#include "common.cuh"

namespace moelora {

// Adapter token ranges, passed by value to the plan kernels.
struct AdapterTable {
  int n;                               // adapters
  int tok_off[kMaxAdapters + 1];       // first token of each adapter; tok_off[n] = T
  int tok_tile[kMaxAdapters + 1];      // first 128-token tile of each adapter
};

// Adapter token ranges from the caller's host offsets [A+1] (NULL allowed when
// A == 1): off[0] = 0, off[A] = T, non-decreasing, and every off[a] with a < A a
// multiple of 128 when A > 1.  Returns MOE_LORA_OK or the rejection code.
inline int make_adapter_table(const moe_lora_dims* d, const int64_t* adapter_offsets, AdapterTable* at) {
  if (d->A > 1 && !adapter_offsets) return MOE_LORA_ERR_NULL;
  *at = AdapterTable{};
  at->n = d->A;
  for (int a = 0; a <= d->A; ++a) {
    const int64_t o = adapter_offsets ? adapter_offsets[a] : (a == 0 ? 0 : d->T);
    if (o < 0 || o > d->T) return MOE_LORA_ERR_DIMS;
    if (a > 0 && o < at->tok_off[a - 1]) return MOE_LORA_ERR_DIMS;
    if (a < d->A && d->A > 1 && o % 128) return MOE_LORA_ERR_DIMS;
    at->tok_off[a] = (int)o;
  }
  if (at->tok_off[0] != 0 || at->tok_off[d->A] != d->T) return MOE_LORA_ERR_DIMS;
  at->tok_tile[0] = 0;
  for (int a = 0; a < d->A; ++a)
    at->tok_tile[a + 1] = at->tok_tile[a] + (at->tok_off[a + 1] - at->tok_off[a] + 127) / 128;
  return MOE_LORA_OK;
}

// The plan kernels' launch sequence.  chunk_base: the per-chunk group histograms,
// A*E*max(1, ceil(T*k/1024)) ints of device memory whose contents on entry do not
// matter (moe_lora_plan passes the end of its workspace, moe_lora_plan_noalloc a
// fixed array inside the library).
cudaError_t launch_plan(const moe_lora_dims* d, const int32_t* ids, const AdapterTable& at, void* ws,
                        int* chunk_base, cudaStream_t stream);

// out[i] = sum_s in[s*stride + i] for s = 0..split-1 in order (fp32, n % 4 == 0).
cudaError_t launch_reduce_splits(const float* in, int64_t stride, int split, int64_t n, float* out, int num_sms,
                                 cudaStream_t stream);

// Decodes `elems` MXFP4 elements (E2M1 nibbles + one UE8M0 byte per 32) to bf16.
cudaError_t launch_dequant_mxfp4(const uint8_t* packed, const uint8_t* scales, uint16_t* out, int64_t elems,
                                 int num_sms, cudaStream_t stream);

// Xp[p] = x[token(p)], Y13p[p] = Y13[token(p)]; zero rows for padding.
cudaError_t launch_gather_fwd(const PlanView& pl, const uint16_t* x, const uint16_t* Y13, uint16_t* Xp,
                              uint16_t* Y13p, int H, int r2, int num_sms, cudaStream_t stream);
// Native FP4 forward: routed rows of x as MXFP8 -- E4M3 codes Xq [P,H] and scale
// bytes Xs in the tile-major layout [P/128][H/128][128][4] (H % 128 == 0) -- and Y13p.
cudaError_t launch_gather_fwd_mxfp8(const PlanView& pl, const uint16_t* x, const uint16_t* Y13, uint8_t* Xq,
                                    uint8_t* Xs, uint16_t* Y13p, int H, int r2, int num_sms, cudaStream_t stream);
// Standalone MXFP8 quantiser (row-major scale bytes [rows, n/32]); n % 32 == 0.
// Native FP4 forward's router-weight gradient from the saved O and Z2 rows:
// dw[t,j] = <dy_t, O[row]> + s <dyB2_t, Z2[row]>  (0 for masked slots).
cudaError_t launch_dw_from_o(const PlanView& pl, const uint16_t* dy, const uint16_t* dyB2, const uint16_t* O,
                             const uint16_t* Z2, int H, int r, float s, float* dw, int num_sms, cudaStream_t stream);
// Scale bytes [rows, K/32] -> tile-major [rows/128][K/128][128][4] (rows, K % 128 == 0).
cudaError_t launch_scales_to_tiles(const uint8_t* S, int64_t rows, int K, uint8_t* St, int num_sms,
                                   cudaStream_t stream);
cudaError_t launch_quant_mxfp8(const uint16_t* x, int64_t rows, int n, uint8_t* codes, uint8_t* scales,
                               int num_sms, cudaStream_t stream);

// Z2w[t] = bf16(sum_j w_tj Z2[row(t,j)])  [T,r]
cudaError_t launch_z2w(const PlanView& pl, const uint16_t* Z2, const float* topk_w, uint16_t* Z2w, int r,
                       int num_sms, cudaStream_t stream);

// Dp[p] = dy[token], D2p[p] = bf16(s*dyB2[token]), dZ2p[p] = bf16(s*w*dyB2[token]); zero on padding.
cudaError_t launch_gather_bwd(const PlanView& pl, const uint16_t* dy, const uint16_t* dyB2, const float* topk_w,
                              uint16_t* Dp, uint16_t* D2p, uint16_t* dZ2p, int H, int r, float s, int num_sms,
                              cudaStream_t stream);

// out[t] = bf16(base[t] + sum_j w_tj src[row(t,j)])  [T,H]; w = 1 when topk_w is NULL.
cudaError_t launch_combine_rows(const PlanView& pl, const uint16_t* base, const uint16_t* src, const float* topk_w,
                                uint16_t* out, int H, int num_sms, cudaStream_t stream, int slot);

// dw[t*k+j] = sum over n-tiles of part[row(t,j)], 0 for masked routes.
cudaError_t launch_dw(const PlanView& pl, const float* part, int nparts, float* dw, int num_sms,
                      cudaStream_t stream);

// dY13w[t] = bf16(sum_j dY13[row(t,j)])  [T,2r]
cudaError_t launch_dy13w(const PlanView& pl, const float* dY13, uint16_t* dY13w, int r2, int num_sms,
                         cudaStream_t stream);

}  // namespace moelora
