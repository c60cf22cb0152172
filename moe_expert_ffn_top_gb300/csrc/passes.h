// Forward / backward launch sequences (forward.cu, backward.cu) and the plain
// engine GEMM used by the self-test entry point (selftest.cu).
#pragma once
#include <cuda_runtime.h>

#include "../../include/moe_lora.h"
#include "launch.h"

namespace moelora {

int run_forward(const moe_lora_dims* d, const void* plan_ws, const uint16_t* x, const float* topk_w,
                const moe_lora_weights* w, uint16_t* y, void* saved, void* scratch, int num_sms,
                cudaStream_t stream);

int run_backward(const moe_lora_dims* d, const void* plan_ws, const void* saved, const uint16_t* x,
                 const float* topk_w, const uint16_t* dy, const moe_lora_weights* w, uint16_t* dx, float* dw,
                 const moe_lora_grads* gr, void* scratch, int num_sms, cudaStream_t stream);

// Router step (router.cu): softmax top-k forward; logit gradient, grad-x update
// and W_r gradient backward.
int run_router_forward(const moe_lora_dims* d, const AdapterTable& at, const uint16_t* x, const uint16_t* Wr,
                       int32_t* ids, float* w, float* logits, void* scratch, int num_sms, cudaStream_t stream);
int run_router_backward(const moe_lora_dims* d, const AdapterTable& at, const uint16_t* x, const uint16_t* Wr,
                        const int32_t* ids, const float* w, const float* dw, float* dlogits, float* dWr, uint16_t* dx,
                        void* scratch, int num_sms, cudaStream_t stream);

// pair != 0: on the two-SM (cta_group::2) engine; starve != 0: no operand copy is
// issued, so the pipeline's bounded waits expire (error-path self-test).
int run_plain_gemm(int M, int N, int K, const uint16_t* A, int a_mn, const uint16_t* B, int b_mn, float* C,
                   int* err, int num_sms, int pair, int starve, cudaStream_t stream);
// Block-scaled plain GEMM through the native FP4 engine path (see ProbPlainNv).
int run_plain_native(int M, int N, int K, const uint8_t* Aq, const uint8_t* As, const uint8_t* Bq, const uint8_t* Bs,
                     float* C, int layout, int* err, int num_sms, cudaStream_t stream);

}  // namespace moelora
