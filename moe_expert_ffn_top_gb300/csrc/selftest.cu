// Plain GEMM through the same tcgen05/TMA engine as the MoE path, for the
// engine self-test entry point (all four operand-majorness combinations).
#include "gemm_problems.cuh"
#include "passes.h"
#include "tmap.h"

namespace moelora {

template <bool AMN, bool BMN>
static int plain(int M, int N, int K, const uint16_t* A, const uint16_t* B, float* C, int* err, int num_sms,
                 cudaStream_t stream) {
  ProbPlain<AMN, BMN> p;
  const uint32_t tn = N < 256 ? (uint32_t)N : 256u;
  if (AMN) {
    if (tmap_2d(&p.mA, A, (uint64_t)M, (uint64_t)K, 64, 64)) return MOE_LORA_ERR_CUDA;
  } else {
    if (tmap_2d(&p.mA, A, (uint64_t)K, (uint64_t)M, 64, 128)) return MOE_LORA_ERR_CUDA;
  }
  if (BMN) {
    if (tmap_2d(&p.mB, B, (uint64_t)N, (uint64_t)K, 64, 64)) return MOE_LORA_ERR_CUDA;
  } else {
    if (tmap_2d(&p.mB, B, (uint64_t)K, (uint64_t)N, 64, tn)) return MOE_LORA_ERR_CUDA;
  }
  p.err = err;
  p.C = C;
  p.M = M;
  p.N = N;
  p.K = K;
  const int tiles = M / 128 * ((N + 255) / 256);
  return launch_gemm(p, tiles, num_sms, stream, K_SELFTEST) == cudaSuccess ? MOE_LORA_OK : MOE_LORA_ERR_CUDA;
}

int run_plain_gemm(int M, int N, int K, const uint16_t* A, int a_mn, const uint16_t* B, int b_mn, float* C,
                   int* err, int num_sms, cudaStream_t stream) {
  if (a_mn && b_mn) return plain<true, true>(M, N, K, A, B, C, err, num_sms, stream);
  if (a_mn) return plain<true, false>(M, N, K, A, B, C, err, num_sms, stream);
  if (b_mn) return plain<false, true>(M, N, K, A, B, C, err, num_sms, stream);
  return plain<false, false>(M, N, K, A, B, C, err, num_sms, stream);
}

}  // namespace moelora
