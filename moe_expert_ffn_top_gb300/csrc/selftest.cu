// Plain GEMM through the same tcgen05/TMA engines as the MoE path, for the
// engine self-test entry points (all four operand-majorness combinations, on
// the one-SM engine and on the two-SM cta_group::2 engine).
#include "gemm_pair.cuh"
#include "gemm_problems.cuh"
#include "passes.h"
#include "tmap.h"

namespace moelora {

template <class Prob, bool AMN, bool BMN>
static int plain_maps(Prob& p, int M, int N, int K, const uint16_t* A, const uint16_t* B, uint32_t b_rows) {
  if (AMN) {
    if (tmap_2d(&p.mA, A, (uint64_t)M, (uint64_t)K, 64, 64)) return MOE_LORA_ERR_CUDA;
  } else {
    if (tmap_2d(&p.mA, A, (uint64_t)K, (uint64_t)M, 64, 128)) return MOE_LORA_ERR_CUDA;
  }
  if (BMN) {
    if (tmap_2d(&p.mB, B, (uint64_t)N, (uint64_t)K, 64, 64)) return MOE_LORA_ERR_CUDA;
  } else {
    if (tmap_2d(&p.mB, B, (uint64_t)K, (uint64_t)N, 64, b_rows)) return MOE_LORA_ERR_CUDA;
  }
  return MOE_LORA_OK;
}

template <bool AMN, bool BMN, bool CB>
static int plain_pair(int M, int N, int K, const uint16_t* A, const uint16_t* B, float* C, int* err, int num_sms,
                      int starve, cudaStream_t stream) {
  using Prob = ProbPlainPair<AMN, BMN, CB>;
  const uint32_t tn = N < 256 ? (uint32_t)N : 256u;
  Prob p;
  int rc;
  if ((rc = plain_maps<Prob, AMN, BMN>(p, M, N, K, A, B, ((tn + 31) & ~31u) / 2))) return rc;
  if (Prob::kBmnCompact && tmap_mn_k8(&p.mB5, B, (uint64_t)N, (uint64_t)K, 1, 2)) return MOE_LORA_ERR_CUDA;
  p.err = err;
  p.C = C;
  p.M = M;
  p.N = N;
  p.K = K;
  p.starve = starve;
  return launch_gemm_pair(p, (M + 255) / 256 * ((N + 255) / 256), num_sms, stream, K_SELFTEST) == cudaSuccess
             ? MOE_LORA_OK
             : MOE_LORA_ERR_CUDA;
}

template <bool AMN, bool BMN>
static int plain(int M, int N, int K, const uint16_t* A, const uint16_t* B, float* C, int* err, int num_sms,
                 bool pair, int starve, cudaStream_t stream) {
  if (pair)  // MN-major B in whole 256-column tiles: the chunk-pair layout
    return BMN && N % 256 == 0 ? plain_pair<AMN, BMN, true>(M, N, K, A, B, C, err, num_sms, starve, stream)
                               : plain_pair<AMN, BMN, false>(M, N, K, A, B, C, err, num_sms, starve, stream);
  const uint32_t tn = N < 256 ? (uint32_t)N : 256u;
  ProbPlain<AMN, BMN> p;
  int rc;
  if ((rc = plain_maps<ProbPlain<AMN, BMN>, AMN, BMN>(p, M, N, K, A, B, tn))) return rc;
  p.err = err;
  p.C = C;
  p.M = M;
  p.N = N;
  p.K = K;
  p.starve = starve;
  return launch_gemm(p, M / 128 * ((N + 255) / 256), num_sms, stream, K_SELFTEST) == cudaSuccess
             ? MOE_LORA_OK
             : MOE_LORA_ERR_CUDA;
}

int run_plain_gemm(int M, int N, int K, const uint16_t* A, int a_mn, const uint16_t* B, int b_mn, float* C,
                   int* err, int num_sms, int pair, int starve, cudaStream_t stream) {
  const bool pr = pair != 0;
  if (a_mn && b_mn) return plain<true, true>(M, N, K, A, B, C, err, num_sms, pr, starve, stream);
  if (a_mn) return plain<true, false>(M, N, K, A, B, C, err, num_sms, pr, starve, stream);
  if (b_mn) return plain<false, true>(M, N, K, A, B, C, err, num_sms, pr, starve, stream);
  return plain<false, false>(M, N, K, A, B, C, err, num_sms, pr, starve, stream);
}

template <int L>
static int plain_native(int M, int N, int K, const uint8_t* Aq, const uint8_t* As, const uint8_t* Bq,
                        const uint8_t* Bs, float* C, int* err, int num_sms, cudaStream_t stream) {
  ProbPlainNv<L> p;
  if (tmap_2d_b8(&p.mA, Aq, (uint64_t)K, (uint64_t)M, 128) ||
      tmap_fp4_unpacked(&p.mB, Bq, (uint64_t)K, (uint64_t)N, 1, 256))
    return MOE_LORA_ERR_CUDA;
  p.As = As;
  p.Bs = Bs;
  p.err = err;
  p.C = C;
  p.M = M;
  p.N = N;
  p.K = K;
  return launch_gemm(p, M / 128 * (N / 256), num_sms, stream, K_SELFTEST) == cudaSuccess ? MOE_LORA_OK
                                                                                       : MOE_LORA_ERR_CUDA;
}

int run_plain_native(int M, int N, int K, const uint8_t* Aq, const uint8_t* As, const uint8_t* Bq, const uint8_t* Bs,
                     float* C, int layout, int* err, int num_sms, cudaStream_t stream) {
  if (layout == kNvLayoutRows) return plain_native<kNvLayoutRows>(M, N, K, Aq, As, Bq, Bs, C, err, num_sms, stream);
  if (layout == kNvLayoutCopy) return plain_native<kNvLayoutCopy>(M, N, K, Aq, As, Bq, Bs, C, err, num_sms, stream);
  return plain_native<kNvLayoutGroups>(M, N, K, Aq, As, Bq, Bs, C, err, num_sms, stream);
}

}  // namespace moelora

