// Per-kernel timing of the library's own launches: when enabled, a CUDA event
// pair is recorded on the launch stream around every kernel; totals are read
// (and reset) through the C ABI.  Launches are always counted.
#pragma once
#include <cuda_runtime.h>

namespace moelora {

enum ProfSlot {
  K_PLAN_COUNT, K_PLAN_SCAN, K_PLAN_SCATTER, K_PLAN_FINISH, K_PLAN_WIDE,
  K_SHRINK, K_GATHER_FWD, K_W13, K_W2, K_Z2W, K_B2_EXPAND, K_COMBINE_Y,
  K_DYB2, K_DB2, K_GATHER_BWD, K_W2_DGRAD, K_DW, K_DA2, K_W13_DGRAD, K_DB13, K_DY13W, K_A13_EXPAND, K_COMBINE_DX, K_DA13,
  K_DEQUANT, K_SPLIT_REDUCE, K_SELFTEST,
  K_ROUTER_FWD, K_ROUTER_DL, K_ROUTER_DX, K_ROUTER_DW,
  K_W13_NV, K_W2_NV, K_DW_NV,  // native FP4 forward
  K_NUM_SLOTS
};

const char* prof_name(int slot);
void prof_begin(int slot, cudaStream_t s);
void prof_end(int slot, cudaStream_t s);

}  // namespace moelora
