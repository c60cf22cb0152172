// C-ABI entry points of the MoE side-LoRA library (declared in include/moe_lora.h):
// host-side validation (every rejection happens before any launch), workspace
// sizing, TMA tensor-map construction and dispatch to the launch sequences.
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdlib>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "launch.h"
#include "passes.h"
#include "tmap.h"

namespace moelora {

// ------------------------------------------------------------------ tensor maps
static PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
static std::once_flag g_encode_once;

static void load_encode() {
  cudaDriverEntryPointQueryResult q;
  void* fn = nullptr;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
}

static int encode(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
                  const cuuint32_t* box, CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B,
                  CUtensorMapDataType type = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
  std::call_once(g_encode_once, load_encode);
  if (!g_encode) return -1;
  const cuuint32_t es[5] = {1, 1, 1, 1, 1};  // rank <= 5
  const CUresult r = g_encode(m, type, rank, const_cast<void*>(base), dims, strides, box, es,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : (int)r;
}

int tmap_2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint32_t box_inner,
            uint32_t box_outer) {
  const cuuint64_t dims[2] = {inner, outer > 0 ? outer : 1};
  const cuuint64_t strides[1] = {inner * 2};
  const cuuint32_t box[2] = {box_inner, box_outer};
  return encode(m, base, 2, dims, strides, box);
}

int tmap_2d_store32(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer) {
  const cuuint64_t dims[2] = {inner, outer > 0 ? outer : 1};
  const cuuint64_t strides[1] = {inner * 2};
  const cuuint32_t box[2] = {32, 32};
  return encode(m, base, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_64B);
}

int tmap_3d(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint32_t b0, uint32_t b1) {
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {d0 * 2, d0 * d1 * 2};
  const cuuint32_t box[3] = {b0, b1, 1};
  return encode(m, base, 3, dims, strides, box);
}

int tmap_3d_u8(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint32_t b0, uint32_t b1) {
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {d0, d0 * d1};
  const cuuint32_t box[3] = {b0, b1, 1};
  return encode(m, base, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_DATA_TYPE_UINT8);
}

int tmap_mn4(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint64_t d2) {
  const cuuint64_t dims[4] = {64, rows, cols / 64, d2};
  const cuuint64_t strides[3] = {cols * 2, 128, rows * cols * 2};
  const cuuint32_t box[4] = {64, 64, 4, 1};
  return encode(m, base, 4, dims, strides, box);
}

int tmap_mn_k8(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint64_t d2, uint32_t chunks) {
  const cuuint64_t dims[5] = {64, 8, cols / 64, rows / 8, d2};
  const cuuint64_t strides[4] = {cols * 2, 128, cols * 16, rows * cols * 2};
  const cuuint32_t box[5] = {64, 8, chunks, 8, 1};
  return encode(m, base, 5, dims, strides, box);
}

int tmap_2d_b8(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint32_t box_outer) {
  const cuuint64_t dims[2] = {inner, outer > 0 ? outer : 1};
  const cuuint64_t strides[1] = {inner};
  const cuuint32_t box[2] = {128, box_outer};
  return encode(m, base, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_DATA_TYPE_UINT8);
}

int tmap_fp4_unpacked(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint32_t b1) {
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {d0 / 2, d0 / 2 * d1};
  const cuuint32_t box[3] = {128, b1, 1};
  return encode(m, base, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B);
}

// ------------------------------------------------------------------ device
// Requires the current device to be an sm_103 GPU; returns its SM count (or the
// MOELORA_NUM_SMS override, for running beside other work).
static int device_sms(int* sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_LORA_ERR_DEVICE;
  int major = 0, minor = 0, n = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return MOE_LORA_ERR_DEVICE;
  if (major != 10 || minor != 3) return MOE_LORA_ERR_DEVICE;
  if (const char* env = std::getenv("MOELORA_NUM_SMS")) {
    const int v = std::atoi(env);
    if (v > 0 && v < n) n = v;
  }
  *sms = n;
  return MOE_LORA_OK;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static int check_ptr(const void* p) {
  if (!p) return MOE_LORA_ERR_NULL;
  if (!aligned16(p)) return MOE_LORA_ERR_ALIGN;
  return MOE_LORA_OK;
}

static int check_weights(const moe_lora_dims* d, const moe_lora_weights* w) {
  if (!w) return MOE_LORA_ERR_NULL;
  const void* ps[] = {w->W1, w->W3, w->W2, w->A1, w->A3, w->B1, w->B3, w->A2, w->B2};
  for (const void* p : ps) {
    const int rc = check_ptr(p);
    if (rc) return rc;
  }
  if (fmt_mx(d)) {
    const void* sc[] = {w->S1, w->S3, w->S2};
    for (const void* p : sc) {
      const int rc = check_ptr(p);
      if (rc) return rc;
    }
  }
  // the native forward's FP4 tensor maps read W1/W3/W2 with 32-byte alignment
  if (fmt_native(d) && ((reinterpret_cast<uintptr_t>(w->W1) | reinterpret_cast<uintptr_t>(w->W3) |
                         reinterpret_cast<uintptr_t>(w->W2)) & 31u))
    return MOE_LORA_ERR_ALIGN;
  return MOE_LORA_OK;
}

}  // namespace moelora

using namespace moelora;

extern "C" {

size_t moe_lora_workspace_bytes(const moe_lora_dims* d, int which) {
  if (check_dims(d) != MOE_LORA_OK) return 0;
  switch (which) {
    case MOE_LORA_WS_PLAN: return plan_layout(d).total;
    case MOE_LORA_WS_SAVED: return saved_layout(d).total;
    case MOE_LORA_WS_FWD_SCRATCH: return fwd_layout(d).total;
    case MOE_LORA_WS_BWD_SCRATCH: return bwd_layout(d).total;
    case MOE_LORA_WS_ROUTER_SCRATCH: return check_router_dims(d) == MOE_LORA_OK ? router_layout(d).total : 0;
    default: return 0;
  }
}

int moe_lora_plan(const moe_lora_dims* d, const int32_t* topk_ids, const int64_t* adapter_offsets, void* plan_ws,
                  size_t plan_bytes, void* stream) {
  int rc = check_dims(d);
  if (rc) return rc;
  if ((rc = check_ptr(plan_ws))) return rc;
  if (d->T > 0 && !topk_ids) return MOE_LORA_ERR_NULL;
  if (plan_bytes < plan_layout(d).total) return MOE_LORA_ERR_WORKSPACE;
  AdapterTable at;
  if ((rc = make_adapter_table(d, adapter_offsets, &at))) return rc;
  int sms;
  if ((rc = device_sms(&sms))) return rc;
  int* chunk_base = reinterpret_cast<int*>(static_cast<char*>(plan_ws) + plan_layout(d).chunk_base);
  return launch_plan(d, topk_ids, at, plan_ws, chunk_base, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? MOE_LORA_OK
             : MOE_LORA_ERR_CUDA;
}

int moe_lora_forward(const moe_lora_dims* d, const void* plan_ws, const uint16_t* x, const float* topk_w,
                     const moe_lora_weights* w, uint16_t* y, void* saved, size_t saved_bytes, void* scratch,
                     size_t scratch_bytes, void* stream) {
  int rc = check_dims(d);
  if (rc) return rc;
  if ((rc = check_ptr(plan_ws)) || (rc = check_weights(d, w)) || (rc = check_ptr(saved)) ||
      (rc = check_ptr(scratch)))
    return rc;
  if (saved_bytes < saved_layout(d).total || scratch_bytes < fwd_layout(d).total) return MOE_LORA_ERR_WORKSPACE;
  if (d->T == 0) return MOE_LORA_OK;
  if ((rc = check_ptr(x)) || (rc = check_ptr(y))) return rc;
  if (!topk_w) return MOE_LORA_ERR_NULL;
  int sms;
  if ((rc = device_sms(&sms))) return rc;
  return run_forward(d, plan_ws, x, topk_w, w, y, saved, scratch, sms, static_cast<cudaStream_t>(stream));
}

int moe_lora_backward(const moe_lora_dims* d, const void* plan_ws, const void* saved, const uint16_t* x,
                      const float* topk_w, const uint16_t* dy, const moe_lora_weights* w, uint16_t* dx, float* dw,
                      const moe_lora_grads* g, void* scratch, size_t scratch_bytes, void* stream) {
  int rc = check_dims(d);
  if (rc) return rc;
  if ((rc = check_ptr(plan_ws)) || (rc = check_weights(d, w)) || (rc = check_ptr(saved)) ||
      (rc = check_ptr(scratch)))
    return rc;
  if (!g) return MOE_LORA_ERR_NULL;
  const void* gp[] = {g->dA1, g->dA3, g->dB1, g->dB3, g->dA2, g->dB2};
  for (const void* p : gp)
    if ((rc = check_ptr(p))) return rc;
  if (scratch_bytes < bwd_layout(d).total) return MOE_LORA_ERR_WORKSPACE;
  int sms;
  if ((rc = device_sms(&sms))) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (d->T == 0) {  // sums over no token: every adapter gradient is zero
    const size_t A = d->A, E = d->E, H = d->H, I = d->I, r = d->r;
    const size_t n[] = {A * r * H, A * r * H, A * E * I * r, A * E * I * r, A * E * r * I, A * H * r};
    float* p[] = {g->dA1, g->dA3, g->dB1, g->dB3, g->dA2, g->dB2};
    for (int i = 0; i < 6; ++i)
      if (cudaMemsetAsync(p[i], 0, n[i] * sizeof(float), s) != cudaSuccess) return MOE_LORA_ERR_CUDA;
    return MOE_LORA_OK;
  }
  if ((rc = check_ptr(x)) || (rc = check_ptr(dy)) || (rc = check_ptr(dx))) return rc;
  if (!topk_w || !dw) return MOE_LORA_ERR_NULL;
  return run_backward(d, plan_ws, saved, x, topk_w, dy, w, dx, dw, g, scratch, sms, s);
}

int moe_lora_router_forward(const moe_lora_dims* d, const uint16_t* x, const uint16_t* Wr,
                            const int64_t* adapter_offsets, int32_t* topk_ids, float* topk_w, float* logits,
                            void* scratch, size_t scratch_bytes, void* stream) {
  int rc = check_router_dims(d);
  if (rc) return rc;
  AdapterTable at;
  if ((rc = make_adapter_table(d, adapter_offsets, &at))) return rc;
  if ((rc = check_ptr(scratch))) return rc;
  if (scratch_bytes < router_layout(d).total) return MOE_LORA_ERR_WORKSPACE;
  if ((rc = check_ptr(Wr))) return rc;
  if (logits && !aligned16(logits)) return MOE_LORA_ERR_ALIGN;
  if (d->T > 0) {
    const void* ps[] = {x, topk_ids, topk_w};
    for (const void* p : ps)
      if ((rc = check_ptr(p))) return rc;
  }
  int sms;
  if ((rc = device_sms(&sms))) return rc;
  return run_router_forward(d, at, x, Wr, topk_ids, topk_w, logits, scratch, sms, static_cast<cudaStream_t>(stream));
}

int moe_lora_router_backward(const moe_lora_dims* d, const uint16_t* x, const uint16_t* Wr,
                             const int64_t* adapter_offsets, const int32_t* topk_ids, const float* topk_w,
                             const float* dw, float* dlogits, float* dWr, uint16_t* dx, void* scratch,
                             size_t scratch_bytes, void* stream) {
  int rc = check_router_dims(d);
  if (rc) return rc;
  AdapterTable at;
  if ((rc = make_adapter_table(d, adapter_offsets, &at))) return rc;
  if ((rc = check_ptr(scratch))) return rc;
  if (scratch_bytes < router_layout(d).total) return MOE_LORA_ERR_WORKSPACE;
  if ((rc = check_ptr(Wr)) || (rc = check_ptr(dWr))) return rc;
  if (dlogits && !aligned16(dlogits)) return MOE_LORA_ERR_ALIGN;
  if (d->T > 0) {
    const void* ps[] = {x, topk_ids, topk_w, dw, dx};
    for (const void* p : ps)
      if ((rc = check_ptr(p))) return rc;
  }
  int sms;
  if ((rc = device_sms(&sms))) return rc;
  return run_router_backward(d, at, x, Wr, topk_ids, topk_w, dw, dlogits, dWr, dx, scratch, sms,
                             static_cast<cudaStream_t>(stream));
}

int moe_lora_router_get_error(const void* scratch, void* stream) {
  if (!scratch) return MOE_LORA_ERR_NULL;
  int v = 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(&v, scratch, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return MOE_LORA_ERR_CUDA;
  return v;
}

int moe_lora_get_error(const moe_lora_dims* d, const void* plan_ws, void* stream) {
  if (check_dims(d) != MOE_LORA_OK) return MOE_LORA_ERR_DIMS;
  if (!plan_ws) return MOE_LORA_ERR_NULL;
  const PlanLayout L = plan_layout(d);
  int v = 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(&v, static_cast<const char*>(plan_ws) + L.err, sizeof(int), cudaMemcpyDeviceToHost, s) !=
          cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return MOE_LORA_ERR_CUDA;
  return v;
}

int moe_lora_plan_readback(const moe_lora_dims* d, const void* plan_ws, int32_t* counts, int32_t* offsets,
                           int32_t* row_of_route, int32_t* route_of_row, int64_t cap, void* stream) {
  if (check_dims(d) != MOE_LORA_OK) return MOE_LORA_ERR_DIMS;
  if (!plan_ws || !counts || !offsets || (d->T > 0 && !row_of_route)) return MOE_LORA_ERR_NULL;
  const PlanLayout L = plan_layout(d);
  const char* b = static_cast<const char*>(plan_ws);
  const size_t G = (size_t)d->A * d->E;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(counts, b + L.counts, G * 4, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaMemcpyAsync(offsets, b + L.offsets, (G + 1) * 4, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      (d->T > 0 && cudaMemcpyAsync(row_of_route, b + L.row_of_route, (size_t)(d->T * d->k) * 4,
                                   cudaMemcpyDeviceToHost, s) != cudaSuccess) ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return MOE_LORA_ERR_CUDA;
  const int64_t P = offsets[G];
  if (route_of_row && cap > 0) {
    if (cap < P) return MOE_LORA_ERR_WORKSPACE;
    if (P > 0 && (cudaMemcpyAsync(route_of_row, b + L.route_of_row, (size_t)P * 4, cudaMemcpyDeviceToHost, s) !=
                      cudaSuccess ||
                  cudaStreamSynchronize(s) != cudaSuccess))
      return MOE_LORA_ERR_CUDA;
  }
  return MOE_LORA_OK;
}

const char* moe_lora_strerror(int code) {
  switch (code) {
    case MOE_LORA_OK: return "ok";
    case MOE_LORA_ERR_NULL: return "a required pointer is NULL";
    case MOE_LORA_ERR_DIMS: return "unsupported or inconsistent sizes";
    case MOE_LORA_ERR_ALIGN: return "a pointer is not 16-byte aligned";
    case MOE_LORA_ERR_WORKSPACE: return "a workspace is smaller than required";
    case MOE_LORA_ERR_UNSUPPORTED: return "unsupported activation or base format";
    case MOE_LORA_ERR_CUDA: return "a CUDA call or kernel launch failed";
    case MOE_LORA_ERR_DEVICE: return "the current device is not an sm_103 GPU";
    case MOE_LORA_ERR_SCRATCH_LIMIT: return "sizes exceed the fixed scratch of moe_lora_plan_noalloc";
    default: return "unknown error";
  }
}

}  // extern "C"

// ------------------------------------------------------------------ engine self-test
static __device__ int g_selftest_err;

static int selftest(int32_t M, int32_t N, int32_t K, const uint16_t* A, int32_t a_mn, const uint16_t* B,
                    int32_t b_mn, float* C, int pair, int starve, void* stream) {
  if (M <= 0 || M % 128 || K <= 0 || K % 64 || N <= 0) return MOE_LORA_ERR_DIMS;
  if (!(N % 256 == 0 || (N <= 256 && N % 16 == 0))) return MOE_LORA_ERR_DIMS;
  int rc;
  if ((rc = check_ptr(A)) || (rc = check_ptr(B)) || (rc = check_ptr(C))) return rc;
  int sms;
  if ((rc = device_sms(&sms))) return rc;
  int* err = nullptr;
  if (cudaGetSymbolAddress(reinterpret_cast<void**>(&err), g_selftest_err) != cudaSuccess) return MOE_LORA_ERR_CUDA;
  return run_plain_gemm(M, N, K, A, a_mn, B, b_mn, C, err, sms, pair, starve, static_cast<cudaStream_t>(stream));
}

extern "C" int moe_lora_mxfp4_decode(const uint8_t* packed, const uint8_t* scales, uint16_t* out, int64_t elems,
                                     void* stream) {
  if (elems < 0 || elems % 32) return MOE_LORA_ERR_DIMS;
  if (elems == 0) return MOE_LORA_OK;
  int rc;
  if ((rc = check_ptr(packed)) || (rc = check_ptr(out))) return rc;
  if (!scales) return MOE_LORA_ERR_NULL;
  int sms = 0;
  if ((rc = device_sms(&sms))) return rc;
  return launch_dequant_mxfp4(packed, scales, out, elems, sms, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? MOE_LORA_OK
             : MOE_LORA_ERR_CUDA;
}

extern "C" int moe_lora_gemm_selftest(int32_t M, int32_t N, int32_t K, const uint16_t* A, int32_t a_mn,
                                      const uint16_t* B, int32_t b_mn, float* C, void* stream) {
  return selftest(M, N, K, A, a_mn, B, b_mn, C, 0, 0, stream);
}

extern "C" int moe_lora_gemm_pair_selftest(int32_t M, int32_t N, int32_t K, const uint16_t* A, int32_t a_mn,
                                           const uint16_t* B, int32_t b_mn, float* C, void* stream) {
  return selftest(M, N, K, A, a_mn, B, b_mn, C, 1, 0, stream);
}

extern "C" int moe_lora_gemm_starved_selftest(int32_t M, int32_t N, int32_t K, const uint16_t* A, int32_t a_mn,
                                              const uint16_t* B, int32_t b_mn, float* C, int32_t pair,
                                              void* stream) {
  return selftest(M, N, K, A, a_mn, B, b_mn, C, pair ? 1 : 0, 1, stream);
}

extern "C" int moe_lora_native_selftest(int32_t M, int32_t N, int32_t K, const uint8_t* Aq, const uint8_t* As,
                                        const uint8_t* Bq, const uint8_t* Bs, float* C, int32_t layout,
                                        void* stream) {
  if (M <= 0 || M % 128 || N <= 0 || N % 256 || K <= 0 || K % 128) return MOE_LORA_ERR_DIMS;
  if (layout < 0 || layout > 2) return MOE_LORA_ERR_UNSUPPORTED;
  int rc;
  if ((rc = check_ptr(Aq)) || (rc = check_ptr(As)) || (rc = check_ptr(Bq)) || (rc = check_ptr(Bs)) ||
      (rc = check_ptr(C)))
    return rc;
  if (reinterpret_cast<uintptr_t>(Bq) % 32) return MOE_LORA_ERR_ALIGN;
  int sms;
  if ((rc = device_sms(&sms))) return rc;
  int* err = nullptr;
  if (cudaGetSymbolAddress(reinterpret_cast<void**>(&err), g_selftest_err) != cudaSuccess) return MOE_LORA_ERR_CUDA;
  return run_plain_native(M, N, K, Aq, As, Bq, Bs, C, layout, err, sms, static_cast<cudaStream_t>(stream));
}

extern "C" int moe_lora_mxfp8_quantize(const uint16_t* x, int64_t rows, int32_t n, uint8_t* codes, uint8_t* scales,
                                       void* stream) {
  if (rows < 0 || n <= 0 || n % 32) return MOE_LORA_ERR_DIMS;
  if (rows == 0) return MOE_LORA_OK;
  int rc;
  if ((rc = check_ptr(x)) || (rc = check_ptr(codes))) return rc;
  if (!scales) return MOE_LORA_ERR_NULL;
  int sms = 0;
  if ((rc = device_sms(&sms))) return rc;
  return launch_quant_mxfp8(x, rows, n, codes, scales, sms, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? MOE_LORA_OK
             : MOE_LORA_ERR_CUDA;
}

extern "C" int moe_lora_gemm_selftest_error(void* stream) {
  int* err = nullptr;
  if (cudaGetSymbolAddress(reinterpret_cast<void**>(&err), g_selftest_err) != cudaSuccess) return MOE_LORA_ERR_CUDA;
  int v = 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(&v, err, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaMemsetAsync(err, 0, sizeof(int), s) != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess)
    return MOE_LORA_ERR_CUDA;
  return v;
}
