// Event-based per-kernel timing (see prof.h).  Event pairs come from a pool that
// grows on demand and is recycled after each read; nothing is allocated on the
// device and nothing runs when timing is off except an atomic launch counter.
#include <atomic>
#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/moe_lora.h"
#include "prof.h"

namespace moelora {

namespace {
struct Rec {
  int slot;
  cudaEvent_t a, b;
};
std::mutex g_mu;
std::atomic<bool> g_on{false};
std::atomic<int> g_only{-1};        // >= 0: time only launches of this slot
std::atomic<long long> g_launches{0};
std::vector<Rec> g_pending;         // recorded, not yet read
std::vector<cudaEvent_t> g_free;    // recycled events
thread_local int t_slot = -1;
thread_local cudaEvent_t t_start = nullptr;

cudaEvent_t take_event() {
  if (!g_free.empty()) {
    cudaEvent_t e = g_free.back();
    g_free.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}
}  // namespace

const char* prof_name(int slot) {
  static const char* names[K_NUM_SLOTS] = {
      "plan_count", "plan_scan", "plan_scatter", "plan_finish", "plan_wide",
      "shrink_x_A13", "gather_fwd", "w13_lora_swiglu", "w2_a2", "z2_combine", "b2_expand", "combine_y",
      "dy_b2", "dB2", "gather_bwd", "w2_dgrad_swiglu_bwd", "dw_reduce", "dA2", "w13_dgrad_b13", "dB13",
      "dy13_combine", "a13_expand", "combine_dx", "dA13", "dequant_mxfp4", "split_reduce", "selftest_gemm",
      "router_topk", "router_dlogits", "router_dx", "router_dWr", "w13_native", "w2_native", "dw_native"};
  return (slot >= 0 && slot < K_NUM_SLOTS) ? names[slot] : "?";
}

void prof_begin(int slot, cudaStream_t s) {
  t_slot = -1;
  if (!g_on.load(std::memory_order_relaxed)) return;
  const int only = g_only.load(std::memory_order_relaxed);
  if (only >= 0 && only != slot) return;
  std::lock_guard<std::mutex> lk(g_mu);
  t_start = take_event();
  if (!t_start) return;
  cudaEventRecord(t_start, s);
  t_slot = slot;
}

void prof_end(int slot, cudaStream_t s) {
  g_launches.fetch_add(1, std::memory_order_relaxed);
  if (t_slot != slot || !t_start) return;
  std::lock_guard<std::mutex> lk(g_mu);
  cudaEvent_t b = take_event();
  if (!b) return;
  cudaEventRecord(b, s);
  g_pending.push_back(Rec{slot, t_start, b});
  t_slot = -1;
  t_start = nullptr;
}

}  // namespace moelora

using namespace moelora;

extern "C" {

int moe_lora_profile_enable(int on) {
  g_on.store(on != 0);
  return MOE_LORA_OK;
}

int moe_lora_profile_select(const char* kernel) {
  if (!kernel) {
    g_only.store(-1);
    return MOE_LORA_OK;
  }
  for (int s = 0; s < K_NUM_SLOTS; ++s)
    if (std::strcmp(prof_name(s), kernel) == 0) {
      g_only.store(s);
      return MOE_LORA_OK;
    }
  return MOE_LORA_ERR_DIMS;
}

int moe_lora_profile_read(const char** names, double* total_ms, int64_t* launches, int cap) {
  std::lock_guard<std::mutex> lk(g_mu);
  double tot[K_NUM_SLOTS] = {};
  long long cnt[K_NUM_SLOTS] = {};
  int rc = MOE_LORA_OK;
  for (const Rec& r : g_pending) {
    if (cudaEventSynchronize(r.b) != cudaSuccess) rc = MOE_LORA_ERR_CUDA;
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, r.a, r.b) == cudaSuccess) {
      tot[r.slot] += ms;
      cnt[r.slot] += 1;
    }
    g_free.push_back(r.a);
    g_free.push_back(r.b);
  }
  g_pending.clear();
  if (rc) return rc;
  int n = 0;
  for (int s = 0; s < K_NUM_SLOTS && n < cap; ++s) {
    if (!cnt[s]) continue;
    if (names) names[n] = prof_name(s);
    if (total_ms) total_ms[n] = tot[s];
    if (launches) launches[n] = cnt[s];
    ++n;
  }
  return n;
}

int64_t moe_lora_launch_count(int reset) {
  return reset ? g_launches.exchange(0) : g_launches.load();
}

}  // extern "C"
