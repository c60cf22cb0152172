/*
 * moe_lora.h -- C ABI of the GB300 (sm_103a) routed MoE SwiGLU expert FFN with
 * rank-r side-LoRA adapters, forward and backward, BF16 with FP32 accumulation.
 *
 * The operation ("feat(mega): add fused shared side-LoRA kernels", DeepGEMM PR #9,
 * Summary): each token goes to its top-k experts; expert e computes
 *     gate = x W1_e^T + s (x A1^T) B1_e^T,   up = x W3_e^T + s (x A3^T) B3_e^T,
 *     h = silu(gate) * up,                    down = h W2_e^T + s (h A2_e^T) B2^T,
 * and the routing-weighted sum of the k down rows is the output.  A1/A3 [r,H]
 * and B2 [H,r] are shared by all experts; B1_e/B3_e [I,r] and A2_e [r,I] are
 * expert-local (the shared-factor contract of that Summary).
 * The frozen W1/W2/W3 receive no gradient; the backward returns grad-x, the
 * router-weight gradient and the six adapter gradients (same PR, Summary).
 *
 * Conventions for every entry point
 *   - All tensors are row-major, contiguous, in DEVICE memory unless stated.
 *     bf16 tensors are passed as uint16_t* holding bf16 bit patterns.
 *   - Every device pointer must be 16-byte aligned.
 *   - The caller owns and allocates every buffer; the library never allocates,
 *     frees or synchronises the stream.  Inputs are read only.  Outputs are fully
 *     overwritten (never accumulated into), so buffers may be reused across calls
 *     (PR #9, Correctness coverage, lists buffer reuse among the tested cases).
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  All work of a
 *     call is enqueued on it; nothing returns to the host in between.
 *   - Return value: 0 on success.  A negative code means the call was rejected on
 *     the host BEFORE any launch (bad shape, NULL or misaligned pointer, short
 *     workspace, unsupported option), in the spirit of PR #9's fail-fast checks
 *     (Summary: unsupported placements and short scratch are refused before any
 *     kernel starts).  MOE_LORA_ERR_CUDA means a launch failed.  Problems
 *     only the device can see (an expert id out of range, a pipeline wait that
 *     timed out) set bits in a sticky device error word read by
 *     moe_lora_get_error().
 */
#ifndef MOE_LORA_H_
#define MOE_LORA_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_LORA_API __attribute__((visibility("default")))
#else
#define MOE_LORA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* ---- return codes ---- */
#define MOE_LORA_OK 0
#define MOE_LORA_ERR_NULL (-1)        /* a required pointer is NULL */
#define MOE_LORA_ERR_DIMS (-2)        /* unsupported or inconsistent sizes */
#define MOE_LORA_ERR_ALIGN (-3)       /* a pointer is not 16-byte aligned */
#define MOE_LORA_ERR_WORKSPACE (-4)   /* a workspace is smaller than required */
#define MOE_LORA_ERR_UNSUPPORTED (-5) /* activation / base format not supported */
#define MOE_LORA_ERR_CUDA (-6)        /* a CUDA call or kernel launch failed */
#define MOE_LORA_ERR_DEVICE (-7)      /* current device is not an sm_103 GPU */
#define MOE_LORA_ERR_SCRATCH_LIMIT (-8) /* sizes exceed moe_lora_plan_noalloc's fixed scratch */

/* ---- device error word bits (moe_lora_get_error) ---- */
#define MOE_LORA_DEV_BAD_ID 1         /* an id >= E or < -1 was seen and dropped */
#define MOE_LORA_DEV_TIMEOUT 2        /* a bounded pipeline wait expired */

/* ---- workspaces ---- */
#define MOE_LORA_WS_PLAN 0        /* routing plan; written by moe_lora_plan */
#define MOE_LORA_WS_SAVED 1       /* forward activations kept for the backward */
#define MOE_LORA_WS_FWD_SCRATCH 2 /* forward temporaries */
#define MOE_LORA_WS_BWD_SCRATCH 3 /* backward temporaries */
#define MOE_LORA_WS_ROUTER_SCRATCH 4 /* router error word and backward temporaries */

/* Problem sizes.  H and I must be multiples of 64 (the 64-element K step of every
 * contraction; the 128- and 256-wide output tiles need not divide them: loads past
 * a tensor's edge read zeros and nothing is stored there); r a multiple of 8 in [8,128];
 * 1 <= k <= 32; 1 <= E; A >= 1 adapters; block_m must be 128 (the plan pads
 * every (adapter, expert) group to a multiple of it).
 * Gated activation h = act(cl(gate)) * cl(up): act 0 = SwiGLU (silu), 1 = GeGLU
 * (exact erf GELU); cl clamps to [-act_clamp, act_clamp] when act_clamp > 0 (the
 * gradient passes on the closed interval), no clamp when act_clamp = 0.  The pages
 * thread SwiGLU/GeGLU and an activation clamp through every kernel (PR #9,
 * Summary); which pre-activations the clamp applies to is not stated there, and
 * this library clamps both gate and up.
 * base_fmt 0: bf16 base weights.  base_fmt 1 or 2: MXFP4 base weights (see
 * moe_lora_weights), decoded exactly to bf16 and fed to the same BF16 tensor-core
 * contractions -- 1: inside the expert GEMMs, tile by tile in shared memory, so
 * the base occupies only its packed bytes and scales (no bf16 copy anywhere);
 * 2: once per forward into the saved workspace (3 * E*I*H bf16 more), which the
 * backward reuses -- faster on GB300 today, since the in-GEMM decode is repeated
 * by every row tile of an expert.  base_fmt 3 or 4: the native FP4 forward -- both
 * base products of the forward run on block-scaled FP4 tensor cores (tcgen05
 * kind::mxf8f6f4) with their activations quantised to MXFP8 (E4M3 codes, one UE8M0
 * scale per 32 consecutive values; the rule of moe_lora_mxfp8_quantize): the routed
 * rows of x against the MXFP4 W1/W3 as stored, the bf16 activation against the MXFP4
 * W2, so their results carry that quantisation ("FP8/FP4/FP8 forwards", PR #9, Fresh
 * validation).  The side paths stay bf16; the backward (straight through the
 * quantisation) runs as base_fmt 1 (3) or 2 (4), and the router-weight gradient is
 * taken from the forward's routed down rows, which these modes keep in `saved`
 * (3.5 GB more at 65,536 tokens, H4096).  H and I must be multiples of 128 and
 * W1/W3/W2 32-byte aligned.
 * T may be 0 (every call is a no-op). */
typedef struct moe_lora_dims {
  int64_t T;        /* tokens */
  int32_t H;        /* hidden size */
  int32_t I;        /* expert intermediate size */
  int32_t E;        /* experts */
  int32_t k;        /* experts per token (top-k) */
  int32_t r;        /* side-LoRA rank */
  int32_t A;        /* adapters sharing the layer (1 = one adapter) */
  int32_t block_m;  /* plan padding unit, 128 */
  float scale;      /* side-LoRA scale s */
  int32_t act;      /* 0 = SwiGLU, 1 = GeGLU */
  int32_t base_fmt; /* 0 = bf16, 1 = MXFP4 decoded in the GEMMs, 2 = MXFP4 decoded once,
                       3 / 4 = native FP4 forward, the rest as 1 / 2 */
  float act_clamp;  /* activation clamp (0 = none) */
} moe_lora_dims;

/* Frozen base and adapter weights (device).
 *   W1, W3 [E,I,H]; W2 [E,H,I]: bf16 bits when base_fmt = 0.  When base_fmt = 1..4
 *     (MXFP4) they hold E2M1 element codes, two per byte (low nibble = lower index
 *     along the last axis), and S1, S3 [E,I,H/32], S2 [E,H,I/32] hold one UE8M0
 *     scale byte (value 2^(b-127); 255 decodes to NaN) per 32 consecutive elements
 *     of that axis: the OCP MX encoding, read from the pages' "E2M1 values with a
 *     UE8M0 scale per 32 elements".  The base is decoded exactly to bf16 and the
 *     BF16 tensor-core path runs on it (except the native gate/up products of
 *     base_fmt 3 and 4, which read it as stored); the adapters stay bf16.
 *     S1/S3/S2 are ignored (may be NULL) when base_fmt = 0.
 *   A1, A3 [A,r,H] (shared by experts); B1, B3 [A,E,I,r] (expert-local);
 *   A2 [A,E,r,I] (expert-local); B2 [A,H,r] (shared), bf16 bits. */
typedef struct moe_lora_weights {
  const void* W1;
  const void* W3;
  const void* W2;
  const uint16_t* A1;
  const uint16_t* A3;
  const uint16_t* B1;
  const uint16_t* B3;
  const uint16_t* A2;
  const uint16_t* B2;
  const uint8_t* S1;
  const uint8_t* S3;
  const uint8_t* S2;
} moe_lora_weights;

/* Adapter gradients (device, fp32), same shapes as the factors they belong to. */
typedef struct moe_lora_grads {
  float* dA1;
  float* dA3;
  float* dB1;
  float* dB3;
  float* dA2;
  float* dB2;
} moe_lora_grads;

/* Bytes of workspace `which` (MOE_LORA_WS_*) for these sizes; 0 for bad sizes.
 * Sizes depend only on dims (the routed row count is bounded on the host by
 * T*k + A*E*(block_m-1)), so no device value is ever read back. */
MOE_LORA_API size_t moe_lora_workspace_bytes(const moe_lora_dims* dims, int which);

/* Routing plan (PR #9 leaves plan construction out of its timed scope).  A stable counting sort of the live routes by
 * (expert, adapter, token, slot) -- the adapters routed to one expert sit side by
 * side, so their tiles share that expert's base weights in L2 -- with group slot
 * q = e*A + a (q = e for one adapter); each group's rows are padded to a multiple of
 * block_m and padding rows map to no route; every group starts at its own padded
 * offset, never rounded into a neighbouring expert (PR #9, Implementation).
 *   topk_ids         [T,k] int32, device.  -1 = masked route (not dispatched).
 *                    Ids >= E or < -1 are dropped and flagged MOE_LORA_DEV_BAD_ID.
 *   adapter_offsets  [A+1] int64, HOST.  Tokens of adapter a are
 *                    [off[a], off[a+1]); off[0] = 0, off[A] = T, non-decreasing,
 *                    and every off[a] with a < A a multiple of 128 when A > 1.
 *                    May be NULL when A == 1.
 *   plan_ws          device buffer of moe_lora_workspace_bytes(.., MOE_LORA_WS_PLAN).
 * Also clears the device error word. */
MOE_LORA_API int moe_lora_plan(const moe_lora_dims* dims, const int32_t* topk_ids, const int64_t* adapter_offsets,
                  void* plan_ws, size_t plan_bytes, void* stream);

/* Routing plan for callers that cannot allocate device memory.  The pages have no
 * counterpart to this entry point.  It exists for callers that may not call
 * cudaMalloc (or any allocator) when they route tokens: memory-planned serving
 * runtimes that reserve all device memory up front and hand out only
 * pre-reserved buffers, and C hosts that hold device pointers but have no
 * allocator binding of their own.
 * It writes exactly the plan moe_lora_plan() writes, with the same launch
 * sequence, but the per-chunk expert histograms it needs as temporary space live
 * in a fixed 4 MiB array inside the library (a file-scope __device__ array that
 * every GPU loading the library holds until the process exits), so the caller
 * passes only the plan buffer itself:
 *   plan_bytes >= moe_lora_workspace_bytes(dims, MOE_LORA_WS_PLAN)
 *                 - 256 * ceil(4 * A * E * max(1, ceil(T*k / 1024)) / 256)
 * (a full MOE_LORA_WS_PLAN buffer also works).  Sizes with
 * A * E * max(1, ceil(T*k / 1024)) > 1,048,576 are rejected with
 * MOE_LORA_ERR_SCRATCH_LIMIT before any launch.  Nothing is allocated or freed.
 * The first call in each CUDA context (for runtime-API callers: on each device,
 * in its primary context) looks up the array's device address with that context
 * current and caches it; make that first call before any stream capture begins.
 * All calls share the one array and every call overwrites it: calls whose work
 * overlaps on the GPU (other streams, other host threads) race on it and must be
 * serialised by the caller.
 * Other arguments, checks and errors are those of moe_lora_plan(). */
MOE_LORA_API int moe_lora_plan_noalloc(const moe_lora_dims* dims, const int32_t* topk_ids,
                                       const int64_t* adapter_offsets, void* plan_ws, size_t plan_bytes,
                                       void* stream);

/* Forward.  x [T,H] bf16; topk_w [T,k] fp32 routing weights (masked slots are
 * ignored); y [T,H] bf16 output.  `saved` receives what the backward needs
 * (opaque; size MOE_LORA_WS_SAVED); `scratch` is temporary (MOE_LORA_WS_FWD_SCRATCH).
 * Requires a plan built by moe_lora_plan for the same dims. */
MOE_LORA_API int moe_lora_forward(const moe_lora_dims* dims, const void* plan_ws, const uint16_t* x, const float* topk_w,
                     const moe_lora_weights* w, uint16_t* y, void* saved, size_t saved_bytes, void* scratch,
                     size_t scratch_bytes, void* stream);

/* Backward of the forward above, given dy [T,H] bf16.
 * Outputs: dx [T,H] bf16; dw [T,k] fp32 (0 at masked slots); the six adapter
 * gradients in fp32.  No gradient is produced for W1/W2/W3.  `saved` must come
 * from moe_lora_forward with the same plan, inputs and weights. */
MOE_LORA_API int moe_lora_backward(const moe_lora_dims* dims, const void* plan_ws, const void* saved, const uint16_t* x,
                      const float* topk_w, const uint16_t* dy, const moe_lora_weights* w, uint16_t* dx, float* dw,
                      const moe_lora_grads* grads, void* scratch, size_t scratch_bytes, void* stream);

/* Reads the sticky device error word of a plan workspace (MOE_LORA_DEV_* bits,
 * 0 = none).  Synchronises `stream`.  Returns a negative MOE_LORA_ERR_* code if
 * the read itself failed. */
MOE_LORA_API int moe_lora_get_error(const moe_lora_dims* dims, const void* plan_ws, void* stream);

/* Copies a plan to HOST arrays for inspection (tests, debugging); synchronises
 * `stream`.  counts [A*E] and offsets [A*E+1], both by group slot q = e*A + a
 * (offsets[A*E] = P, the padded routed row count), row_of_route [T*k] (-1 = not
 * dispatched), route_of_row [P] (t*k+j, or -1 on a padding row; pass cap >= P, or
 * NULL/0 to skip). */
MOE_LORA_API int moe_lora_plan_readback(const moe_lora_dims* dims, const void* plan_ws, int32_t* counts,
                                        int32_t* offsets, int32_t* row_of_route, int32_t* route_of_row,
                                        int64_t route_of_row_cap, void* stream);

/* Decodes an MXFP4 tensor (the frozen-base format of moe_lora_dims.base_fmt = 1 and 2) to
 * bf16, exactly, on `stream`: elems E2M1 codes (two per byte, the lower index in the
 * low nibble; bit 3 = sign, magnitudes {0, 0.5, 1, 1.5, 2, 3, 4, 6}) with one UE8M0
 * scale byte per 32 consecutive elements (b -> 2^(b-127); b = 0 gives 2^-127, b = 255
 * NaN).  Every decoded value is a bf16 value (no rounding), overflowing to +-inf at
 * the largest scales.  The forward runs the same decode on W1, W3 and W2 (PR #9:
 * "MXFP4-dequantized BF16" base).
 *   packed [elems/2] uint8 and out [elems] bf16, device, 16-byte aligned; scales
 *   [elems/32] uint8, device.  elems % 32 == 0 (MOE_LORA_ERR_DIMS otherwise). */
MOE_LORA_API int moe_lora_mxfp4_decode(const uint8_t* packed, const uint8_t* scales, uint16_t* out, int64_t elems,
                                       void* stream);

/* Per-kernel timing of this library's own launches, for profiling and the
 * benchmark's roofline figures (off by default).  When on, every kernel launch is
 * bracketed by a CUDA event pair recorded on its launch stream. */
MOE_LORA_API int moe_lora_profile_enable(int on);
/* Restricts the timing to the launches of one kernel (by the name that
 * moe_lora_profile_read reports), so that the event pairs around every other
 * launch do not slow the step down; NULL times every kernel again.  Returns
 * MOE_LORA_ERR_DIMS for an unknown name. */
MOE_LORA_API int moe_lora_profile_select(const char* kernel);
/* Reads and resets the per-kernel totals since the last read: for each kernel
 * that ran (at most cap), its static name, total milliseconds and launch count.
 * Waits for the recorded events.  Returns how many entries were written, or a
 * negative MOE_LORA_ERR_* code. */
MOE_LORA_API int moe_lora_profile_read(const char** names, double* total_ms, int64_t* launches, int cap);
/* Kernel launches issued by this library since the last reset (always counted);
 * reset != 0 returns the count and sets it to zero. */
MOE_LORA_API int64_t moe_lora_launch_count(int reset);

/* ---- router: the routing step ahead of the expert path ----
 * PR #9 takes the routes as inputs and returns their weight gradient (its
 * "grad-route", Correctness coverage).  These two calls add the step that makes
 * the routes and carry that gradient back to the router, read as the usual
 * softmax top-k gate:
 *     l_t = W_r x_t  (fp32 accumulation),   p_t = softmax(l_t) over all E,
 *     the k experts of largest p_t, largest first, equal values to the lower id
 *     (selected on l_t in fp32: softmax keeps the order),
 *     w_tj = p_t[e_j] / sum_j' p_t[e_j']   (renormalised to sum 1).
 * Backward, for the selection made in the forward: since w_t is the softmax of
 * the selected logits alone, dl_te = w_tj (dw_tj - sum_j' w_tj' dw_tj') at
 * e = e_j and 0 elsewhere; dW_r = sum_t dl_t^T x_t; grad-x gains dl_t W_r.
 * Several adapters (OpenPipe/ART PR #1139, Behavior: each adapter routes with its
 * own router) own contiguous token ranges given by adapter_offsets [A+1] int64,
 * HOST, with the rules of moe_lora_plan (NULL allowed when A == 1); adapter a's
 * tokens use W_r[a] and contribute to dW_r[a] only, and every adapter's results
 * equal its standalone run with the same tokens bit for bit.
 * Requirements beyond moe_lora_dims' rules: 16 <= E <= 256 with E % 16 == 0,
 * k <= E (else MOE_LORA_ERR_UNSUPPORTED / MOE_LORA_ERR_DIMS).
 * `scratch` is a device buffer of moe_lora_workspace_bytes(.., MOE_LORA_WS_ROUTER_SCRATCH);
 * its first word is the device error word both calls clear and
 * moe_lora_router_get_error() reads. */

/* x [T,H] bf16, W_r [A,E,H] bf16.  Writes topk_ids [T,k] int32 (largest first) and
 * topk_w [T,k] fp32; logits [T,E] fp32 as well when non-NULL.  One launch. */
MOE_LORA_API int moe_lora_router_forward(const moe_lora_dims* dims, const uint16_t* x, const uint16_t* Wr,
                                         const int64_t* adapter_offsets, int32_t* topk_ids, float* topk_w,
                                         float* logits, void* scratch, size_t scratch_bytes, void* stream);

/* topk_ids / topk_w as written by moe_lora_router_forward (slots with an id
 * outside [0, E) are skipped), dw [T,k] fp32 (e.g. moe_lora_backward's dw), the
 * same adapter_offsets as the forward.  Writes dWr [A,E,H] fp32 and, when
 * non-NULL, dlogits [T,E] fp32.  dx [T,H] bf16
 * is READ AND UPDATED in place, dx <- bf16(dx + dl W_r), so that the expert
 * path's grad-x and the router's share one buffer (the one exception to
 * "outputs are overwritten"; pass a zeroed dx for the router's part alone). */
MOE_LORA_API int moe_lora_router_backward(const moe_lora_dims* dims, const uint16_t* x, const uint16_t* Wr,
                                          const int64_t* adapter_offsets, const int32_t* topk_ids,
                                          const float* topk_w, const float* dw, float* dlogits, float* dWr,
                                          uint16_t* dx, void* scratch, size_t scratch_bytes, void* stream);

/* Reads (and keeps) the device error word of a router scratch buffer
 * (MOE_LORA_DEV_* bits); synchronises `stream`. */
MOE_LORA_API int moe_lora_router_get_error(const void* scratch, void* stream);

/* Static description of a return code. */
MOE_LORA_API const char* moe_lora_strerror(int code);

/* Engine self-test: C[M,N] (fp32, device) = sum_k A(m,k) B(n,k) on the same
 * tcgen05/TMA GEMM engine that runs the MoE contractions.  A is [M,K] row-major
 * (a_mn = 0, K-major) or [K,M] (a_mn = 1, MN-major); B is [N,K] (b_mn = 0) or
 * [K,N] (b_mn = 1); bf16 bits, 16-byte aligned.  M % 128 == 0, K % 64 == 0, and
 * N % 256 == 0 or (N <= 256 and N % 16 == 0).  Not part of the MoE method; it
 * exists to check and time the engine in isolation.  Device-side wait timeouts
 * are reported through moe_lora_gemm_selftest_error(). */
MOE_LORA_API int moe_lora_gemm_selftest(int32_t M, int32_t N, int32_t K, const uint16_t* A, int32_t a_mn, const uint16_t* B,
                           int32_t b_mn, float* C, void* stream);
/* The same plain GEMM on the two-SM engine (the forward W2 expert GEMM's alternative
 * form): clusters of two CTAs sharing each 256-row tile through
 * tcgen05.mma.cta_group::2 (an odd last 128-row tile runs on one CTA of the pair).
 * An MN-major B with N a multiple of 256 is copied as 8-row groups of each CTA's two
 * 64-column chunks; other shapes as whole 64-column chunks.  Same arguments, rules and
 * error reporting as moe_lora_gemm_selftest. */
MOE_LORA_API int moe_lora_gemm_pair_selftest(int32_t M, int32_t N, int32_t K, const uint16_t* A, int32_t a_mn,
                                             const uint16_t* B, int32_t b_mn, float* C, void* stream);
/* Error-path self-test of the bounded pipeline waits: the same plain GEMM (pair = 0:
 * one-SM engine, 1: two-SM engine) with every operand copy withheld, as if a copy
 * had been lost.  No wait in the engines is unbounded, so the kernel's waits give
 * up (after about 2 s), set MOE_LORA_DEV_TIMEOUT in the self-test error word, and
 * the kernel ends without writing C; the context stays usable.  Same argument
 * rules as moe_lora_gemm_selftest; the check is the error word, not C. */
MOE_LORA_API int moe_lora_gemm_starved_selftest(int32_t M, int32_t N, int32_t K, const uint16_t* A, int32_t a_mn,
                                                const uint16_t* B, int32_t b_mn, float* C, int32_t pair,
                                                void* stream);
/* Self-test of the block-scaled FP4 tensor-core path (kind::mxf8f6f4) that the
 * native FP4 forward (base_fmt 3 and 4) runs its gate/up and down base products on:
 *   C[M,N] (fp32) = sum_k (Aq[m,k] 2^(As[m,k/32]-127)) (Bq[n,k] 2^(Bs[n,k/32]-127))
 * Aq [M,K]: E4M3 codes, one per byte.  Bq [N,K/2]: E2M1 codes, two per byte, the low
 * nibble holding the lower k; 32-byte aligned.  As, Bs: the UE8M0 scale bytes of A
 * and B (one per 32 consecutive k of a row) in the tile-major layout
 * [rows/128][K/128][32][4][4]: one 4-byte word per (row, 128-wide k step), byte j
 * scaling that row's k elements 32j..32j+31 of the step, and the 128 words of a row
 * block for one k step 512 bytes with row i's word at position 4 (i % 32) + i / 32.
 * M % 128 == 0, N % 256 == 0, K % 128 == 0.  layout selects how the scale words
 * reach tensor memory: 0, written by the epilogue warps (tcgen05.st) in the layout
 * the MMA reads; 2, the same layout copied by the MMA-issuing thread (tcgen05.cp);
 * 1, one row per lane, a comparison case that gives a wrong C.  Bad sizes:
 * MOE_LORA_ERR_DIMS; layout out of range: MOE_LORA_ERR_UNSUPPORTED; Bq not 32-byte
 * aligned: MOE_LORA_ERR_ALIGN.  Device-side wait timeouts are reported through
 * moe_lora_gemm_selftest_error().  Not part of the MoE method. */
MOE_LORA_API int moe_lora_native_selftest(int32_t M, int32_t N, int32_t K, const uint8_t* Aq, const uint8_t* As,
                                          const uint8_t* Bq, const uint8_t* Bs, float* C, int32_t layout,
                                          void* stream);
/* The MXFP8 quantiser of the native FP4 forward, standalone: for x [rows, n] bf16
 * (device, n % 32 == 0), codes [rows, n] E4M3 and scales [rows, n/32] UE8M0 bytes,
 * per 32 consecutive elements of a row -- the OCP MX format: shared scale 2^X with
 * X = floor(log2 max|v|) - 8 (8 = the exponent of E4M3's largest power of two; X = 0
 * for an all-zero block; X clamped to [-127, 127]), each element v / 2^X rounded to
 * nearest even on the E4M3 grid and saturated at +-448.  The pages name the native
 * forward's formats only ("FP8/FP4/FP8 forwards", PR #9, Fresh validation); this is
 * the plainest reading.  Returns MOE_LORA_ERR_DIMS for bad sizes; rows = 0 is a no-op. */
MOE_LORA_API int moe_lora_mxfp8_quantize(const uint16_t* x, int64_t rows, int32_t n, uint8_t* codes,
                                         uint8_t* scales, void* stream);
/* Device error word of the self-test GEMMs (MOE_LORA_DEV_* bits); synchronises
 * the stream and clears the word. */
MOE_LORA_API int moe_lora_gemm_selftest_error(void* stream);

#ifdef __cplusplus
}
#endif
#endif /* MOE_LORA_H_ */
