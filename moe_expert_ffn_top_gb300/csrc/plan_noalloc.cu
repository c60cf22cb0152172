// Routing plan for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc, or any allocator, at the point where they
// route tokens: memory-planned serving runtimes that reserve all device memory up
// front and hand out only pre-reserved buffers (an allocation there fails or
// fragments the reserved pool), and plain C hosts that hold device pointers but
// have no allocator binding of their own.  They still own the plan buffer itself
// (the output), but cannot provide the extra temporary space that moe_lora_plan()
// keeps at the end of its workspace for per-chunk expert histograms.
//
// moe_lora_plan_noalloc() therefore takes that temporary space from a fixed
// file-scope device array instead.  The array is part of the library image: every
// GPU on which the library is loaded holds it (4 MiB) until the process exits.
// Nothing here calls cudaMalloc, cudaFree or any allocating library routine; the
// launch sequence is moe_lora_plan()'s own (launch_plan), given the array.
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

#include "common.cuh"
#include "launch.h"

namespace moelora {

// Per-chunk histograms of the plan: (adapters * experts) x ceil(T*k / 1024) ints.
constexpr int64_t kNoallocScratchInts = int64_t(1) << 20;  // 4 MiB
static __device__ __align__(256) int g_plan_scratch[kNoallocScratchInts];

namespace {
// In host code `g_plan_scratch` names a host-side stand-in, not device memory, so
// its device address is looked up with cudaGetSymbolAddress.  A module is loaded
// once per CUDA context (not per device: a driver-API host may create several
// contexts on one device, and cudaDeviceReset replaces the primary context), so
// the address is cached per context, keyed by the driver's unique context id.
struct ScratchEntry {
  unsigned long long ctx_id;
  int* addr;
};
constexpr int kMaxContexts = 64;
std::mutex g_mu;
ScratchEntry g_cache[kMaxContexts];
int g_cached = 0;

PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
PFN_cuCtxGetId_v12000 g_ctx_id = nullptr;
std::once_flag g_ctx_once;

void load_ctx_entry_points() {
  cudaDriverEntryPointQueryResult q;
  void* fn = nullptr;
  if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
  fn = nullptr;
  if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    g_ctx_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(fn);
}

// Device address of g_plan_scratch in the current context.
int scratch_for_current_context(int** out) {
  std::call_once(g_ctx_once, load_ctx_entry_points);
  if (!g_ctx_current || !g_ctx_id) return MOE_LORA_ERR_CUDA;
  CUcontext ctx = nullptr;
  if (g_ctx_current(&ctx) != CUDA_SUCCESS) return MOE_LORA_ERR_CUDA;
  void* fresh = nullptr;
  if (!ctx) {
    // No context is current yet: the runtime's symbol lookup makes the current
    // device's primary context current (as any runtime call would).
    if (cudaGetSymbolAddress(&fresh, g_plan_scratch) != cudaSuccess || !fresh) return MOE_LORA_ERR_CUDA;
    if (g_ctx_current(&ctx) != CUDA_SUCCESS || !ctx) return MOE_LORA_ERR_CUDA;
  }
  unsigned long long id = 0;
  if (g_ctx_id(ctx, &id) != CUDA_SUCCESS) return MOE_LORA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  for (int i = 0; i < g_cached; ++i)
    if (g_cache[i].ctx_id == id) {
      *out = g_cache[i].addr;
      return MOE_LORA_OK;
    }
  if (!fresh && (cudaGetSymbolAddress(&fresh, g_plan_scratch) != cudaSuccess || !fresh)) return MOE_LORA_ERR_CUDA;
  // Context ids are never reused within a process; a full table keeps the oldest
  // entries and looks the address up again on every call from a newer context.
  if (g_cached < kMaxContexts) g_cache[g_cached++] = ScratchEntry{id, static_cast<int*>(fresh)};
  *out = static_cast<int*>(fresh);
  return MOE_LORA_OK;
}

bool device_ok() {
  int dev = 0, major = 0, minor = 0;
  return cudaGetDevice(&dev) == cudaSuccess &&
         cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) == cudaSuccess &&
         cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) == cudaSuccess && major == 10 &&
         minor == 3;
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
  const int64_t nchunks = plan_chunks(d);
  if ((int64_t)d->A * d->E * (nchunks > 0 ? nchunks : 1) > kNoallocScratchInts) return MOE_LORA_ERR_SCRATCH_LIMIT;
  if (plan_bytes < plan_layout(d).chunk_base) return MOE_LORA_ERR_WORKSPACE;  // the plan, without the histograms
  AdapterTable at;
  if ((rc = make_adapter_table(d, adapter_offsets, &at))) return rc;
  if (!device_ok()) return MOE_LORA_ERR_DEVICE;
  int* chunk_base = nullptr;
  if ((rc = scratch_for_current_context(&chunk_base))) return rc;
  // The array keeps the previous call's histograms; launch_plan rewrites (or, with
  // no routes, clears) every entry it reads before reading it.
  return launch_plan(d, topk_ids, at, plan_ws, chunk_base, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? MOE_LORA_OK
             : MOE_LORA_ERR_CUDA;
}
