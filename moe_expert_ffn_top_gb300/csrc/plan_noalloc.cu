// Routing plan for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc, or any allocator, at the point where they
// route tokens: code that runs while a CUDA stream is being captured into a
// graph (an allocation there breaks the capture), memory-planned serving
// runtimes that hand out only pre-reserved buffers, and plain C hosts without an
// allocator binding.  They still own the plan buffer itself (the output), but
// cannot provide the extra temporary space that moe_lora_plan() keeps at the
// end of its workspace for per-chunk expert histograms.
//
// moe_lora_plan_noalloc() therefore takes that temporary space from a fixed
// file-scope device array instead.  The array is part of the library image: every
// GPU on which the library is loaded holds it (4 MiB) until the process exits.
// Nothing here calls cudaMalloc, cudaFree or any allocating library routine.
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>

#include "common.cuh"
#include "launch.h"
#include "plan_kernels.h"

namespace moelora {

// Per-chunk histograms of the plan: (adapters * experts) x ceil(T*k / 1024) ints.
constexpr int64_t kNoallocScratchInts = int64_t(1) << 20;  // 4 MiB
static __device__ __align__(256) int g_plan_scratch[kNoallocScratchInts];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_mu;
int* g_scratch_addr[kMaxDevices] = {};  // device address of g_plan_scratch, per device

// In host code `g_plan_scratch` names a host-side stand-in, not device memory, so
// the device address is looked up once per device (with that device current).
int scratch_for_current_device(int** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_LORA_ERR_DEVICE;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_plan_scratch) != cudaSuccess || !p) return MOE_LORA_ERR_CUDA;
    g_scratch_addr[dev] = static_cast<int*>(p);
  }
  *out = g_scratch_addr[dev];
  return MOE_LORA_OK;
}
}  // namespace

}  // namespace moelora

using namespace moelora;

extern "C" int moe_lora_plan_noalloc(const moe_lora_dims* d, const int32_t* topk_ids, const int64_t* adapter_offsets,
                                     void* plan_ws, size_t plan_bytes, void* stream) {
  int rc = check_dims(d);
  if (rc) return rc;
  if (!plan_ws) return MOE_LORA_ERR_NULL;
  if (reinterpret_cast<uintptr_t>(plan_ws) & 15u) return MOE_LORA_ERR_ALIGN;
  if (d->T > 0 && !topk_ids) return MOE_LORA_ERR_NULL;
  const int G = d->A * d->E;
  const int64_t nchunks = plan_chunks(d);
  if ((int64_t)G * (nchunks > 0 ? nchunks : 1) > kNoallocScratchInts) return MOE_LORA_ERR_SCRATCH_LIMIT;
  const PlanLayout L = plan_layout(d);
  if (plan_bytes < L.chunk_base) return MOE_LORA_ERR_WORKSPACE;  // the plan itself, without the histograms
  AdapterTable at;
  if ((rc = make_adapter_table(d, adapter_offsets, &at))) return rc;
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess || major != 10 ||
      minor != 3)
    return MOE_LORA_ERR_DEVICE;
  int* chunk_base = nullptr;
  if ((rc = scratch_for_current_device(&chunk_base))) return rc;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* b = static_cast<char*>(plan_ws);
  int* err = (int*)(b + L.err);
  int* counts = (int*)(b + L.counts);
  int* offsets = (int*)(b + L.offsets);
  int* row_of_route = (int*)(b + L.row_of_route);
  int* route_of_row = (int*)(b + L.route_of_row);
  int* tile_group = (int*)(b + L.tile_group);
  int2* tile_span = (int2*)(b + L.tile_span);
  int* tok_off = (int*)(b + L.tok_off);
  int* tok_tile = (int*)(b + L.tok_tile);
  int* wtile_off = (int*)(b + L.wtile_off);
  int4* wtile = (int4*)(b + L.wtile);
  const int64_t TK = d->T * d->k;
  const int nch = (int)nchunks;
  if (cudaMemsetAsync(err, 0, 16, s) != cudaSuccess) return MOE_LORA_ERR_CUDA;
  const size_t hist_bytes = sizeof(int) * (size_t)G;
  if (hist_bytes > 48 * 1024) {
    if (cudaFuncSetAttribute(plan_count, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)hist_bytes) !=
            cudaSuccess ||
        cudaFuncSetAttribute(plan_scatter, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)hist_bytes) !=
            cudaSuccess)
      return MOE_LORA_ERR_CUDA;
  }
  // The shared array keeps the previous call's histograms.  plan_count rewrites
  // every entry this call reads; with no routes at all, the G entries read by
  // plan_scan are cleared here.
  if (nch > 0) {
    plan_count<<<nch, 32, hist_bytes, s>>>(topk_ids, TK, d->k, d->E, G, at, chunk_base, nch, err);
  } else if (cudaMemsetAsync(chunk_base, 0, sizeof(int) * (size_t)G, s) != cudaSuccess) {
    return MOE_LORA_ERR_CUDA;
  }
  plan_scan<<<1, 1024, 0, s>>>(chunk_base, nch > 0 ? nch : 1, G, counts, offsets);
  if (nch > 0)
    plan_scatter<<<nch, 32, hist_bytes, s>>>(topk_ids, TK, d->k, d->E, G, at, chunk_base, offsets, nch, row_of_route,
                                             route_of_row, err);
  plan_finish<<<G < 1024 ? G : 1024, 128, 0, s>>>(G, d->E, counts, offsets, route_of_row, tile_group, tile_span,
                                                  at, tok_off, tok_tile);
  plan_wide<<<1, 1024, 0, s>>>(G, d->A, d->E, offsets, wtile_off, wtile);
  return cudaGetLastError() == cudaSuccess ? MOE_LORA_OK : MOE_LORA_ERR_CUDA;
}
