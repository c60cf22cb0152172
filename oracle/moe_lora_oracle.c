/*
 * Plain CPU oracle for the routed MoE SwiGLU expert FFN with rank-r side-LoRA,
 * forward and backward.  TEST INFRASTRUCTURE ONLY: it is called from tests/,
 * from the package smoke check and from the benchmark's CPU-baseline leg, never
 * from the product path.  It shares no code with the CUDA library.
 *
 * What it computes (the method of "feat(mega): add fused shared side-LoRA kernels",
 * DeepGEMM PR #9, Summary: the down-projection factors A1/A3 of the gate and up
 * projections and the up-projection factor B2 of the down projection are common to
 * all experts, while B1, B3 and A2 belong to each expert; the base weights W1/W2/W3
 * are frozen), per token t and per unmasked slot j with expert e = ids[t,j] and
 * adapter a = adapter(t):
 *
 *   y1 = rb(A1_a x_t)            y3 = rb(A3_a x_t)                       [r]
 *   g  = W1_e x_t + s B1_{a,e} y1      u = W3_e x_t + s B3_{a,e} y3      [I]
 *   h  = rb(act(cl(g)) * cl(u))                                          [I]
 *        act = silu(z) = z / (1 + exp(-z))  (SwiGLU, the default), or
 *        act = gelu(z) = z/2 (1 + erf(z / sqrt 2))  (GeGLU);
 *        cl(v) = min(max(v, -c), c) with the activation clamp c (none when c = 0);
 *        the pages thread "SwiGLU/GeGLU" and an activation clamp through every
 *        kernel (PR #9, Summary; the production runs used clamp 10).
 *   z2 = rb(A2_{a,e} h)                                                  [r]
 *   o  = W2_e h + s B2_a z2                                              [H]
 *   y_t = rb( sum_j w_tj o_j )   (slot order; masked slots contribute nothing)
 *
 * rb() rounds to bf16 (round to nearest even) at the points where a BF16
 * tensor-core implementation forms an operand or an output; it is the identity
 * when rounding is switched off (the FP64 build used for finite differences).
 * The backward is the exact reverse-mode derivative of the above with rb treated
 * as the identity: grad-x, the router-weight gradient dL/dw_tj = <dy_t, o_j>
 * (the "grad-route" of PR #9, Correctness coverage) and the six adapter gradients
 * dA1, dA3, dB1, dB3, dA2, dB2 (PR #9, Summary: the backward yields the input
 * gradient, the routing-weight gradient and all six factor gradients, and nothing
 * for the frozen base weights).  Adapter gradients are summed in (token, slot) order.
 *
 * The routing plan is a stable counting sort of the live routes by
 * (expert, adapter, token, slot) -- group slot q = e*A + a, so q = e for one
 * adapter -- each group padded to a multiple of BLOCK_M rows
 * (pool padding of PR #9, Implementation: each expert's rows start at its own
 * padded offset, never rounded into a neighbour).
 *
 * MXFP4 base weights: E2M1 element codes (1 sign, 2 exponent with bias 1,
 * 1 mantissa bit) with one UE8M0 scale 2^(b-127) per 32 contiguous elements along
 * the contraction axis; low nibble = lower index.  Decoded here from the bit fields.
 *
 * Native FP4 forward (act_quant = 1): both base products of the forward take their
 * activations as MXFP8, so that both operands are block-scaled low-precision values
 * ("FP8/FP4/FP8 forwards" in the PR's Fresh validation; block-scaled FP4 against
 * dequantise-to-BF16 in its Performance notes):
 *   g = W1_e q8(x_t) + s B1 y1,   u = W3_e q8(x_t) + s B3 y3,   o = W2_e q8(h) + s B2 z2
 * with everything else unchanged (y1/y3 use x_t, z2 = rb(A2 h) uses h).  q8 is the OCP MX FP8
 * format with E4M3 elements: per 32 contiguous values one shared scale 2^X,
 * X = floor(log2 max|v|) - 8 (8 = the exponent of E4M3's largest power of two),
 * and each element v / 2^X rounded to nearest even on the E4M3 grid, saturating at
 * +-448; q8(h) takes the blocks along I.  The backward treats q8 as the identity, like
 * rb; the router-weight gradient stays <dy_t, o_j> with this o.
 *
 * Build: real = float (default) or double (-DORACLE_DOUBLE).  Compile with
 * -ffp-contract=off so x86 and Arm hosts give identical results.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#define NTHREADS(d) ((d)->nthreads > 0 ? (d)->nthreads : omp_get_max_threads())
#define NTHREADS_N(n) ((n) > 0 ? (n) : omp_get_max_threads())
#else
#define NTHREADS(d) 1
#define NTHREADS_N(n) 1
#endif

#ifdef ORACLE_DOUBLE
typedef double real;
#define REXP exp
#else
typedef float real;
#define REXP expf
#endif

enum { DT_BF16 = 0, DT_REAL = 1, DT_MXFP4 = 2 };

typedef struct {
  const void* p;          /* element storage */
  const uint8_t* scales;  /* MXFP4: one UE8M0 byte per 32 elements; else NULL */
  int32_t dtype;          /* DT_* */
  int32_t pad_;
} otensor;

typedef struct {
  int64_t T;
  int32_t H, I, E, k, r, A, block_m;
  double scale;           /* side-LoRA scale s */
  int32_t round_bf16;     /* 1: bf16 rounding points on; 0: off */
  int32_t nthreads;       /* OpenMP threads (0 = runtime default) */
  int32_t act;            /* 0: SwiGLU, 1: GeGLU */
  int32_t act_quant;      /* 1: q8(x) and q8(h) in the base products (native FP4 forward) */
  double clamp;           /* activation clamp c (0 = none) */
} odims;

typedef struct {
  const int32_t* ids;              /* [T,k], -1 = masked route */
  const int64_t* adapter_offsets;  /* [A+1] tokens of adapter a are [off[a], off[a+1]) */
  otensor w;                       /* topk weights [T,k] */
  otensor x;                       /* [T,H] */
  otensor dy;                      /* [T,H] (backward only) */
  otensor W1, W3, W2;              /* [E,I,H], [E,I,H], [E,H,I] */
  otensor A1, A3;                  /* [A,r,H] */
  otensor B1, B3;                  /* [A,E,I,r] */
  otensor A2;                      /* [A,E,r,I] */
  otensor B2;                      /* [A,H,r] */
} oinputs;

/* ---------------- scalar helpers ---------------- */

static real bf16_bits_to_real(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (real)f;
}

/* round to the nearest bf16 value (8 significant bits), ties to even */
static real round_bf16(real v) {
  if (!(v == v) || v == 0 || isinf((double)v)) return v;
  int ex;
  double m = frexp((double)v, &ex);          /* v = m * 2^ex, 0.5 <= |m| < 1 */
  double q = nearbyint(ldexp(m, 8));         /* 8 significant bits, RNE */
  return (real)ldexp(q, ex - 8);
}

/* E2M1 code -> value, from the bit fields */
static double e2m1_value(int code) {
  int sign = (code >> 3) & 1, ebits = (code >> 1) & 3, mbit = code & 1;
  double mag = (ebits == 0) ? 0.5 * mbit : ldexp(1.0 + 0.5 * mbit, ebits - 1);
  return sign ? -mag : mag;
}

static double ue8m0_value(uint8_t b) { return b == 255 ? NAN : ldexp(1.0, (int)b - 127); }

/* E4M3 code -> value, from the bit fields: 1 sign, 4 exponent bits with bias 7,
 * 3 mantissa bits; exponent field 0 is subnormal (m/8 * 2^-6); S.1111.111 is NaN
 * (no infinities, so S.1111.110 = 448 is the largest finite magnitude). */
static double e4m3_value(int code) {
  int sign = (code >> 7) & 1, ebits = (code >> 3) & 15, m = code & 7;
  if (ebits == 15 && m == 7) return NAN;
  double mag = ebits == 0 ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, ebits - 7);
  return sign ? -mag : mag;
}

/* v rounded to the nearest E4M3 value (ties to even), saturating at +-448.  On
 * [2^e, 2^(e+1)) the grid spacing is 2^(e-3); below 2^-6 it is the subnormal 2^-9. */
static double e4m3_round(double v) {
  double a = fabs(v);
  if (a == 0) return v;
  int ex;
  frexp(a, &ex); /* a in [2^(ex-1), 2^ex) */
  int e = ex - 1 < -6 ? -6 : ex - 1;
  double q = ldexp(1.0, e - 3);
  double r = nearbyint(a / q) * q;
  if (r > 448) r = 448;
  return signbit(v) ? -r : r;
}

/* E4M3 code of a value already on the grid (the sign taken from v, also for 0). */
static int e4m3_code(double v) {
  int sign = signbit(v) ? 0x80 : 0;
  double a = fabs(v);
  for (int c = 0; c < 127; ++c)
    if (e4m3_value(c) == a) return sign | c;
  return -1;
}

/* One MXFP8 block of n <= 32 values: the scale byte (X + 127; X = 0 for an all-zero
 * block, clamped to the byte range otherwise) and each value's q8 in deq[].  The
 * division by 2^X is exact. */
static uint8_t mxfp8_block(const real* v, int n, double* deq) {
  double amax = 0;
  for (int i = 0; i < n; ++i) amax = fabs((double)v[i]) > amax ? fabs((double)v[i]) : amax;
  int X = 0;
  if (amax > 0) {
    int ex;
    frexp(amax, &ex); /* floor(log2 amax) = ex - 1 */
    X = ex - 1 - 8;
    if (X < -127) X = -127;
    if (X > 127) X = 127;
  }
  for (int i = 0; i < n; ++i) deq[i] = ldexp(e4m3_round(ldexp((double)v[i], -X)), X);
  return (uint8_t)(X + 127);
}

/* q8 of a row of n values in blocks of 32 from its start */
static void mxfp8_row(const real* v, int64_t n, real* out) {
  double deq[32];
  for (int64_t b = 0; b < n; b += 32) {
    int m = n - b < 32 ? (int)(n - b) : 32;
    mxfp8_block(v + b, m, deq);
    for (int i = 0; i < m; ++i) out[b + i] = (real)deq[i];
  }
}

static real ld(const otensor* t, int64_t i) {
  switch (t->dtype) {
    case DT_BF16: return bf16_bits_to_real(((const uint16_t*)t->p)[i]);
    case DT_REAL: return ((const real*)t->p)[i];
    default: {
      uint8_t byte = ((const uint8_t*)t->p)[i >> 1];
      int code = (i & 1) ? (byte >> 4) : (byte & 15);
      return (real)(e2m1_value(code) * ue8m0_value(t->scales[i >> 5]));
    }
  }
}

static void ld_row(const otensor* t, int64_t base, int64_t n, real* dst) {
  for (int64_t i = 0; i < n; ++i) dst[i] = ld(t, base + i);
}

static real rb(const odims* d, real v) { return d->round_bf16 ? round_bf16(v) : v; }

static real silu(real z) { return z / ((real)1 + REXP(-z)); }
static real sigmoid(real z) { return (real)1 / ((real)1 + REXP(-z)); }

#ifdef ORACLE_DOUBLE
#define RERF erf
#else
#define RERF erff
#endif
static const double kInvSqrt2 = 0.70710678118654752440;
static const double kInvSqrt2Pi = 0.39894228040143267794;
static real gelu(real z) { return (real)0.5 * z * ((real)1 + RERF(z * (real)kInvSqrt2)); }
/* d gelu / dz = Phi(z) + z phi(z) */
static real gelu_grad(real z) {
  return (real)0.5 * ((real)1 + RERF(z * (real)kInvSqrt2)) + z * (real)kInvSqrt2Pi * REXP((real)-0.5 * z * z);
}
static real act_f(const odims* d, real z) { return d->act == 1 ? gelu(z) : silu(z); }
static real act_grad(const odims* d, real z) {
  if (d->act == 1) return gelu_grad(z);
  const real sg = sigmoid(z);
  return sg * ((real)1 + z * ((real)1 - sg));
}
static real clampv(const odims* d, real v) {
  if (d->clamp <= 0) return v;
  const real c = (real)d->clamp;
  return v < -c ? -c : (v > c ? c : v);
}
/* derivative of the clamp: 1 on [-c, c] (the ends included), else 0 */
static real clamp_pass(const odims* d, real v) {
  if (d->clamp <= 0) return (real)1;
  const real c = (real)d->clamp;
  return (v >= -c && v <= c) ? (real)1 : (real)0;
}

static int adapter_of(const oinputs* in, int A, int64_t t) {
  for (int a = 0; a < A; ++a)
    if (t >= in->adapter_offsets[a] && t < in->adapter_offsets[a + 1]) return a;
  return -1;
}

/* ---------------- routing plan ---------------- */

/* Stable counting sort of live routes by (expert, adapter, token, slot); counts and
 * offsets are indexed by the group slot q = e*A + a.  The pages fix no row order
 * when several adapters share the layer (OpenPipe/ART PR #1139, Behavior: the
 * dispatched rows only carry adapter ids); expert-major keeps the adapters routed to
 * one expert side by side.  Returns the number of invalid ids (>= E or < -1), which
 * are dropped. */
int oracle_plan(int64_t T, int32_t k, int32_t E, int32_t A, int32_t BM, const int32_t* ids,
                const int64_t* adapter_offsets, int32_t* counts, int32_t* offsets,
                int32_t* row_of_route, int32_t* route_of_row, int64_t row_cap) {
  int64_t G = (int64_t)A * E;
  int bad = 0;
  memset(counts, 0, sizeof(int32_t) * G);
  for (int64_t t = 0; t < T; ++t) {
    int a = 0;
    while (a + 1 < A && t >= adapter_offsets[a + 1]) ++a;
    for (int j = 0; j < k; ++j) {
      int32_t e = ids[t * k + j];
      if (e >= E || e < -1) { ++bad; continue; }
      if (e >= 0) counts[(int64_t)e * A + a]++;
    }
  }
  offsets[0] = 0;
  for (int64_t g = 0; g < G; ++g)
    offsets[g + 1] = offsets[g] + (counts[g] + BM - 1) / BM * BM;
  for (int64_t p = 0; p < row_cap; ++p) route_of_row[p] = -1;
  int32_t* cursor = (int32_t*)malloc(sizeof(int32_t) * G);
  for (int64_t g = 0; g < G; ++g) cursor[g] = offsets[g];
  for (int64_t t = 0; t < T; ++t) {
    int a = 0;
    while (a + 1 < A && t >= adapter_offsets[a + 1]) ++a;
    for (int j = 0; j < k; ++j) {
      int32_t e = ids[t * k + j];
      int64_t rt = t * k + j;
      if (e < 0 || e >= E) { row_of_route[rt] = -1; continue; }
      int32_t row = cursor[(int64_t)e * A + a]++;
      row_of_route[rt] = row;
      if (row < row_cap) route_of_row[row] = (int32_t)rt;
    }
  }
  free(cursor);
  return bad;
}

/* ---------------- per-route forward ---------------- */

typedef struct {
  real *xt, *xq, *y1, *y3, *g, *u, *h, *hq, *z2, *o, *rowbuf;
} fwd_scratch;

static void fwd_alloc(const odims* d, fwd_scratch* s) {
  int64_t H = d->H, I = d->I, r = d->r;
  int64_t n = 2 * H + 2 * r + 4 * I + r + H + (H > I ? H : I);
  real* p = (real*)malloc(sizeof(real) * n);
  s->xt = p; p += H;
  s->xq = p; p += H;
  s->y1 = p; p += r;
  s->y3 = p; p += r;
  s->g = p; p += I;
  s->u = p; p += I;
  s->h = p; p += I;
  s->hq = p; p += I;
  s->z2 = p; p += r;
  s->o = p; p += H;
  s->rowbuf = p;
}

static void fwd_free(fwd_scratch* s) { free(s->xt); }

/* x_t into s->xt, and q8(x_t) into s->xq for the native FP4 forward */
static void load_token(const odims* d, const oinputs* in, int64_t t, fwd_scratch* s) {
  ld_row(&in->x, t * d->H, d->H, s->xt);
  if (d->act_quant) mxfp8_row(s->xt, d->H, s->xq);
}

/* forward of one live route (t, slot with expert e, adapter a); s->xt holds x_t */
static void route_forward(const odims* d, const oinputs* in, int a, int e, fwd_scratch* s) {
  const int64_t H = d->H, I = d->I, r = d->r, E = d->E;
  const real sc = (real)d->scale;
  real* row = s->rowbuf;
  const real* xb = d->act_quant ? s->xq : s->xt; /* x as the gate/up base products see it */
  for (int64_t q = 0; q < r; ++q) {
    real acc1 = 0, acc3 = 0;
    ld_row(&in->A1, ((int64_t)a * r + q) * H, H, row);
    for (int64_t c = 0; c < H; ++c) acc1 += row[c] * s->xt[c];
    ld_row(&in->A3, ((int64_t)a * r + q) * H, H, row);
    for (int64_t c = 0; c < H; ++c) acc3 += row[c] * s->xt[c];
    s->y1[q] = rb(d, acc1);
    s->y3[q] = rb(d, acc3);
  }
  for (int64_t i = 0; i < I; ++i) {
    real gb = 0, ub = 0, gl = 0, ul = 0;
    ld_row(&in->W1, ((int64_t)e * I + i) * H, H, row);
    for (int64_t c = 0; c < H; ++c) gb += row[c] * xb[c];
    ld_row(&in->W3, ((int64_t)e * I + i) * H, H, row);
    for (int64_t c = 0; c < H; ++c) ub += row[c] * xb[c];
    int64_t bbase = (((int64_t)a * E + e) * I + i) * r;
    for (int64_t q = 0; q < r; ++q) gl += ld(&in->B1, bbase + q) * s->y1[q];
    for (int64_t q = 0; q < r; ++q) ul += ld(&in->B3, bbase + q) * s->y3[q];
    s->g[i] = gb + sc * gl;
    s->u[i] = ub + sc * ul;
    s->h[i] = rb(d, act_f(d, clampv(d, s->g[i])) * clampv(d, s->u[i]));
  }
  for (int64_t q = 0; q < r; ++q) {
    real acc = 0;
    ld_row(&in->A2, (((int64_t)a * E + e) * r + q) * I, I, row);
    for (int64_t i = 0; i < I; ++i) acc += row[i] * s->h[i];
    s->z2[q] = rb(d, acc);
  }
  if (d->act_quant) mxfp8_row(s->h, I, s->hq);
  const real* hb = d->act_quant ? s->hq : s->h; /* h as the down base product sees it */
  for (int64_t c = 0; c < H; ++c) {
    real ob = 0, ol = 0;
    ld_row(&in->W2, ((int64_t)e * H + c) * I, I, row);
    for (int64_t i = 0; i < I; ++i) ob += row[i] * hb[i];
    int64_t b2 = ((int64_t)a * H + c) * r;
    for (int64_t q = 0; q < r; ++q) ol += ld(&in->B2, b2 + q) * s->z2[q];
    s->o[c] = ob + sc * ol;
  }
}

/* y for the listed tokens: y[n*H + c] for token tokens[n] (or token n if tokens == NULL). */
int oracle_forward(const odims* d, const oinputs* in, const int64_t* tokens, int64_t ntok, real* y) {
  const int64_t H = d->H, k = d->k;
#pragma omp parallel num_threads(NTHREADS(d))
  {
    fwd_scratch s;
    fwd_alloc(d, &s);
    real* acc = (real*)malloc(sizeof(real) * H);
#pragma omp for schedule(dynamic, 1)
    for (int64_t n = 0; n < ntok; ++n) {
      int64_t t = tokens ? tokens[n] : n;
      int a = adapter_of(in, d->A, t);
      for (int64_t c = 0; c < H; ++c) acc[c] = 0;
      load_token(d, in, t, &s);
      for (int64_t j = 0; j < k; ++j) {
        int32_t e = in->ids[t * k + j];
        if (e < 0 || e >= d->E) continue;
        route_forward(d, in, a, e, &s);
        real wj = ld(&in->w, t * k + j);
        for (int64_t c = 0; c < H; ++c) acc[c] += wj * s.o[c];
      }
      for (int64_t c = 0; c < H; ++c) y[n * H + c] = rb(d, acc[c]);
    }
    free(acc);
    fwd_free(&s);
  }
  return 0;
}

/* ---------------- backward ---------------- */

/* Per-route quantities kept for the adapter-gradient sums. */
typedef struct {
  int64_t t;
  int32_t a, e, live;
  real wj;
} route_meta;

int oracle_backward(const odims* d, const oinputs* in, const int64_t* tokens, int64_t ntok, real* dx,
                    real* dw, real* dA1, real* dA3, real* dB1, real* dB3, real* dA2, real* dB2) {
  const int64_t H = d->H, I = d->I, r = d->r, E = d->E, k = d->k, A = d->A;
  const real sc = (real)d->scale;
  const int64_t nr = ntok * k;
  /* per-route saved vectors */
  real* S_dg = (real*)calloc((size_t)nr * I, sizeof(real));
  real* S_du = (real*)calloc((size_t)nr * I, sizeof(real));
  real* S_h = (real*)calloc((size_t)nr * I, sizeof(real));
  real* S_y1 = (real*)calloc((size_t)nr * r, sizeof(real));
  real* S_y3 = (real*)calloc((size_t)nr * r, sizeof(real));
  real* S_z2 = (real*)calloc((size_t)nr * r, sizeof(real));
  real* S_dz2 = (real*)calloc((size_t)nr * r, sizeof(real));
  real* S_dy1 = (real*)calloc((size_t)nr * r, sizeof(real));
  real* S_dy3 = (real*)calloc((size_t)nr * r, sizeof(real));
  route_meta* M = (route_meta*)calloc((size_t)nr, sizeof(route_meta));
  if (!S_dg || !S_du || !S_h || !S_y1 || !S_y3 || !S_z2 || !S_dz2 || !S_dy1 || !S_dy3 || !M) return -1;

#pragma omp parallel num_threads(NTHREADS(d))
  {
    fwd_scratch s;
    fwd_alloc(d, &s);
    real* dyt = (real*)malloc(sizeof(real) * H);
    real* dyB2 = (real*)malloc(sizeof(real) * r);
    real* dact = (real*)malloc(sizeof(real) * I);
    real* dxa = (real*)malloc(sizeof(real) * H);
    real* row = (real*)malloc(sizeof(real) * (H > I ? H : I));
#pragma omp for schedule(dynamic, 1)
    for (int64_t n = 0; n < ntok; ++n) {
      int64_t t = tokens ? tokens[n] : n;
      int a = adapter_of(in, d->A, t);
      load_token(d, in, t, &s);
      ld_row(&in->dy, t * H, H, dyt);
      for (int64_t c = 0; c < H; ++c) dxa[c] = 0;
      for (int64_t j = 0; j < k; ++j) {
        int64_t ri = n * k + j;
        int32_t e = in->ids[t * k + j];
        M[ri].t = t;
        M[ri].a = a;
        M[ri].e = e;
        M[ri].live = (e >= 0 && e < E);
        if (!M[ri].live) { dw[n * k + j] = 0; continue; }
        real wj = ld(&in->w, t * k + j);
        M[ri].wj = wj;
        route_forward(d, in, a, e, &s);
        /* router-weight gradient */
        real dwj = 0;
        for (int64_t c = 0; c < H; ++c) dwj += dyt[c] * s.o[c];
        dw[n * k + j] = dwj;
        /* B2^T dy */
        for (int64_t q = 0; q < r; ++q) {
          real acc = 0;
          for (int64_t c = 0; c < H; ++c) acc += ld(&in->B2, ((int64_t)a * H + c) * r + q) * dyt[c];
          dyB2[q] = acc;
        }
        /* dL/dh = w (W2_e^T dy + s A2_e^T (B2^T dy)) */
        for (int64_t i = 0; i < I; ++i) dact[i] = 0;
        for (int64_t c = 0; c < H; ++c) {
          ld_row(&in->W2, ((int64_t)e * H + c) * I, I, row);
          for (int64_t i = 0; i < I; ++i) dact[i] += row[i] * dyt[c];
        }
        for (int64_t q = 0; q < r; ++q) {
          ld_row(&in->A2, (((int64_t)a * E + e) * r + q) * I, I, row);
          for (int64_t i = 0; i < I; ++i) dact[i] += sc * row[i] * dyB2[q];
        }
        for (int64_t i = 0; i < I; ++i) dact[i] *= wj;
        for (int64_t q = 0; q < r; ++q) {
          S_dz2[ri * r + q] = sc * wj * dyB2[q];
          S_z2[ri * r + q] = s.z2[q];
          S_y1[ri * r + q] = s.y1[q];
          S_y3[ri * r + q] = s.y3[q];
        }
        /* gated-activation backward (through the clamp) */
        for (int64_t i = 0; i < I; ++i) {
          const real gc = clampv(d, s.g[i]), uc = clampv(d, s.u[i]);
          S_dg[ri * I + i] = dact[i] * uc * act_grad(d, gc) * clamp_pass(d, s.g[i]);
          S_du[ri * I + i] = dact[i] * act_f(d, gc) * clamp_pass(d, s.u[i]);
          S_h[ri * I + i] = s.h[i];
        }
        const real* dg = S_dg + ri * I;
        const real* du = S_du + ri * I;
        /* side-path gradients w.r.t. y1, y3 */
        for (int64_t q = 0; q < r; ++q) {
          real a1 = 0, a3 = 0;
          int64_t bb = (((int64_t)a * E + e) * I) * r + q;
          for (int64_t i = 0; i < I; ++i) {
            a1 += ld(&in->B1, bb + i * r) * dg[i];
            a3 += ld(&in->B3, bb + i * r) * du[i];
          }
          S_dy1[ri * r + q] = sc * a1;
          S_dy3[ri * r + q] = sc * a3;
        }
        /* grad-x: W1_e^T dg + W3_e^T du + A1^T dy1 + A3^T dy3 */
        for (int64_t i = 0; i < I; ++i) {
          ld_row(&in->W1, ((int64_t)e * I + i) * H, H, row);
          for (int64_t c = 0; c < H; ++c) dxa[c] += row[c] * dg[i];
          ld_row(&in->W3, ((int64_t)e * I + i) * H, H, row);
          for (int64_t c = 0; c < H; ++c) dxa[c] += row[c] * du[i];
        }
        for (int64_t q = 0; q < r; ++q) {
          ld_row(&in->A1, ((int64_t)a * r + q) * H, H, row);
          for (int64_t c = 0; c < H; ++c) dxa[c] += row[c] * S_dy1[ri * r + q];
          ld_row(&in->A3, ((int64_t)a * r + q) * H, H, row);
          for (int64_t c = 0; c < H; ++c) dxa[c] += row[c] * S_dy3[ri * r + q];
        }
      }
      for (int64_t c = 0; c < H; ++c) dx[n * H + c] = rb(d, dxa[c]);
    }
    free(dyt); free(dyB2); free(dact); free(dxa); free(row);
    fwd_free(&s);
  }

  /* adapter gradients: sums over live routes in (token, slot) order.
   * Routes of each (adapter, expert) group are listed in that order first. */
  const int64_t G = A * E;
  int64_t* gstart = (int64_t*)calloc((size_t)G + 1, sizeof(int64_t));
  int64_t* gorder = (int64_t*)malloc(sizeof(int64_t) * (nr > 0 ? nr : 1));
  for (int64_t ri = 0; ri < nr; ++ri)
    if (M[ri].live) gstart[(int64_t)M[ri].a * E + M[ri].e + 1]++;
  for (int64_t g = 0; g < G; ++g) gstart[g + 1] += gstart[g];
  {
    int64_t* cur = (int64_t*)malloc(sizeof(int64_t) * (G > 0 ? G : 1));
    for (int64_t g = 0; g < G; ++g) cur[g] = gstart[g];
    for (int64_t ri = 0; ri < nr; ++ri)
      if (M[ri].live) gorder[cur[(int64_t)M[ri].a * E + M[ri].e]++] = ri;
    free(cur);
  }
#pragma omp parallel for schedule(dynamic, 4) num_threads(NTHREADS(d))
  for (int64_t gi = 0; gi < G * I; ++gi) {
    int64_t g = gi / I, i = gi % I;
    int64_t a = g / E, e = g % E;
    real* o1 = dB1 + gi * r;
    real* o3 = dB3 + gi * r;
    for (int64_t q = 0; q < r; ++q) o1[q] = o3[q] = 0;
    (void)a; (void)e;
    for (int64_t n = gstart[g]; n < gstart[g + 1]; ++n) {
      int64_t ri = gorder[n];
      real g1 = S_dg[ri * I + i], g3 = S_du[ri * I + i];
      for (int64_t q = 0; q < r; ++q) {
        o1[q] += sc * g1 * S_y1[ri * r + q];
        o3[q] += sc * g3 * S_y3[ri * r + q];
      }
    }
  }
#pragma omp parallel for schedule(dynamic, 4) num_threads(NTHREADS(d))
  for (int64_t gq = 0; gq < G * r; ++gq) {
    int64_t g = gq / r, q = gq % r;
    int64_t a = g / E, e = g % E;
    real* o = dA2 + gq * I;
    for (int64_t i = 0; i < I; ++i) o[i] = 0;
    (void)a; (void)e;
    for (int64_t n = gstart[g]; n < gstart[g + 1]; ++n) {
      int64_t ri = gorder[n];
      real z = S_dz2[ri * r + q];
      for (int64_t i = 0; i < I; ++i) o[i] += z * S_h[ri * I + i];
    }
  }
#pragma omp parallel for schedule(dynamic, 4) num_threads(NTHREADS(d))
  for (int64_t ac = 0; ac < A * H; ++ac) {
    int64_t a = ac / H, c = ac % H;
    real* o = dB2 + ac * r;
    for (int64_t q = 0; q < r; ++q) o[q] = 0;
    for (int64_t ri = 0; ri < nr; ++ri) {
      if (!M[ri].live || M[ri].a != a) continue;
      real dyc = ld(&in->dy, M[ri].t * H + c);
      for (int64_t q = 0; q < r; ++q) o[q] += sc * M[ri].wj * dyc * S_z2[ri * r + q];
    }
  }
#pragma omp parallel for schedule(dynamic, 1) num_threads(NTHREADS(d))
  for (int64_t aq = 0; aq < A * r; ++aq) {
    int64_t a = aq / r, q = aq % r;
    real* o1 = dA1 + aq * H;
    real* o3 = dA3 + aq * H;
    for (int64_t c = 0; c < H; ++c) o1[c] = o3[c] = 0;
    for (int64_t ri = 0; ri < nr; ++ri) {
      if (!M[ri].live || M[ri].a != a) continue;
      real v1 = S_dy1[ri * r + q], v3 = S_dy3[ri * r + q];
      int64_t xb = M[ri].t * H;
      for (int64_t c = 0; c < H; ++c) {
        real xc = ld(&in->x, xb + c);
        o1[c] += v1 * xc;
        o3[c] += v3 * xc;
      }
    }
  }
  free(S_dg); free(S_du); free(S_h); free(S_y1); free(S_y3); free(S_z2); free(S_dz2);
  free(S_dy1); free(S_dy3); free(M); free(gstart); free(gorder);
  return 0;
}

/* ---------------- router (the routing step ahead of the expert path) ----------------
 *
 * The pages take the routes as given and return the routing-weight gradient
 * ("grad-route", PR #9, Correctness coverage); the router itself follows the usual
 * softmax top-k gate, read here as:
 *   l_t = W_r x_t                         logits [E]
 *   p_t = softmax(l_t) over all E experts
 *   the k experts of largest p_t, in descending order, equal values to the lower
 *   expert id (softmax is strictly increasing in each logit, so the selection is
 *   made on l_t, which is the same order without exp/division rounding)
 *   w_tj = p_t[e_j] / sum_j' p_t[e_j']    (the k weights renormalised to sum 1)
 * The backward is the reverse-mode derivative of this map for a fixed selection:
 *   dp_i = [i selected] (dw_i / S - sum_j dw_j p_j / S^2),  S = sum of selected p
 *   dl   = p (dp - <p, dp>)                 (softmax backward)
 *   dW_r = sum_t dl_t x_t^T,   dx_t = W_r^T dl_t
 * Slots whose id is outside [0, E) are left out of the selection. */

static void router_logits(int64_t H, int64_t E, const otensor* x, const otensor* Wr, int64_t t, real* xt,
                          real* l) {
  ld_row(x, t * H, H, xt);
  for (int64_t e = 0; e < E; ++e) {
    real acc = 0;
    for (int64_t c = 0; c < H; ++c) acc += ld(Wr, e * H + c) * xt[c];
    l[e] = acc;
  }
}

static void softmax_all(int64_t E, const real* l, real* p) {
  real m = l[0];
  for (int64_t e = 1; e < E; ++e) m = l[e] > m ? l[e] : m;
  real z = 0;
  for (int64_t e = 0; e < E; ++e) z += REXP(l[e] - m);
  for (int64_t e = 0; e < E; ++e) p[e] = REXP(l[e] - m) / z;
}

int oracle_router_forward(int64_t T, int32_t H, int32_t E, int32_t k, int32_t nthreads, const otensor* x,
                          const otensor* Wr, real* logits, int32_t* ids, real* w) {
  if (k > E) return -1;
#pragma omp parallel num_threads(NTHREADS_N(nthreads))
  {
    real* xt = (real*)malloc(sizeof(real) * H);
    real* l = (real*)malloc(sizeof(real) * E);
    real* p = (real*)malloc(sizeof(real) * E);
    char* taken = (char*)malloc((size_t)E);
#pragma omp for schedule(dynamic, 8)
    for (int64_t t = 0; t < T; ++t) {
      router_logits(H, E, x, Wr, t, xt, l);
      if (logits)
        for (int64_t e = 0; e < E; ++e) logits[t * E + e] = l[e];
      softmax_all(E, l, p);
      memset(taken, 0, (size_t)E);
      real S = 0;
      for (int j = 0; j < k; ++j) {
        int best = -1;
        for (int e = 0; e < E; ++e)
          if (!taken[e] && (best < 0 || l[e] > l[best])) best = e;  /* strict: ties keep the lower id */
        taken[best] = 1;
        ids[t * k + j] = best;
        S += p[best];
      }
      for (int j = 0; j < k; ++j) w[t * k + j] = p[ids[t * k + j]] / S;
    }
    free(xt); free(l); free(p); free(taken);
  }
  return 0;
}

/* dlogits [T,E] (may be NULL), dWr [E,H], dx [T,H]: the router's part of the input
 * gradient alone. */
int oracle_router_backward(int64_t T, int32_t H, int32_t E, int32_t k, int32_t nthreads, const otensor* x,
                           const otensor* Wr, const int32_t* ids, const real* dw, real* dlogits, real* dWr,
                           real* dx) {
  real* dl_all = (real*)calloc((size_t)(T > 0 ? T : 1) * E, sizeof(real));
  if (!dl_all) return -1;
#pragma omp parallel num_threads(NTHREADS_N(nthreads))
  {
    real* xt = (real*)malloc(sizeof(real) * H);
    real* l = (real*)malloc(sizeof(real) * E);
    real* p = (real*)malloc(sizeof(real) * E);
    real* dp = (real*)malloc(sizeof(real) * E);
#pragma omp for schedule(dynamic, 8)
    for (int64_t t = 0; t < T; ++t) {
      router_logits(H, E, x, Wr, t, xt, l);
      softmax_all(E, l, p);
      real S = 0, num = 0;
      for (int j = 0; j < k; ++j) {
        int e = ids[t * k + j];
        if (e < 0 || e >= E) continue;
        S += p[e];
        num += dw[t * k + j] * p[e];
      }
      for (int64_t e = 0; e < E; ++e) dp[e] = 0;
      for (int j = 0; j < k; ++j) {
        int e = ids[t * k + j];
        if (e < 0 || e >= E) continue;
        dp[e] += dw[t * k + j] / S - num / (S * S);
      }
      real pdp = 0;
      for (int64_t e = 0; e < E; ++e) pdp += p[e] * dp[e];
      real* dl = dl_all + t * E;
      for (int64_t e = 0; e < E; ++e) dl[e] = p[e] * (dp[e] - pdp);
      if (dlogits)
        for (int64_t e = 0; e < E; ++e) dlogits[t * E + e] = dl[e];
      for (int64_t c = 0; c < H; ++c) {
        real acc = 0;
        for (int64_t e = 0; e < E; ++e) acc += dl[e] * ld(Wr, e * H + c);
        dx[t * H + c] = acc;
      }
    }
    free(xt); free(l); free(p); free(dp);
  }
#pragma omp parallel for schedule(dynamic, 1) num_threads(NTHREADS_N(nthreads))
  for (int64_t e = 0; e < E; ++e) {
    real* o = dWr + e * H;
    for (int64_t c = 0; c < H; ++c) o[c] = 0;
    for (int64_t t = 0; t < T; ++t) {
      const real g = dl_all[t * E + e];
      if (g == 0) continue;
      for (int64_t c = 0; c < H; ++c) o[c] += g * ld(x, t * H + c);
    }
  }
  free(dl_all);
  return 0;
}

/* decoders exposed for the format pins */
double oracle_e2m1_value(int code) { return e2m1_value(code); }
double oracle_e4m3_value(int code) { return e4m3_value(code); }
double oracle_e4m3_round(double v) { return e4m3_round(v); }

/* MXFP8 of n values (blocks of 32 from the start): E4M3 codes[n], scale bytes
 * [ceil(n/32)], and the dequantised values deq[n].  Returns the number of values
 * whose q8 is not an E4M3 value times the block scale (0 when consistent). */
int oracle_mxfp8_quantize(const double* v, int64_t n, uint8_t* codes, uint8_t* scales, double* deq) {
  real blk[32];
  double dq[32];
  int bad = 0;
  for (int64_t b = 0; b < n; b += 32) {
    int m = n - b < 32 ? (int)(n - b) : 32;
    for (int i = 0; i < m; ++i) blk[i] = (real)v[b + i];
    uint8_t sb = mxfp8_block(blk, m, dq);
    scales[b / 32] = sb;
    for (int i = 0; i < m; ++i) {
      deq[b + i] = dq[i];
      int c = e4m3_code(ldexp(dq[i], 127 - (int)sb));
      if (c < 0) ++bad;
      codes[b + i] = (uint8_t)(c < 0 ? 0x7F : c);
    }
  }
  return bad;
}
double oracle_ue8m0_value(int b) { return ue8m0_value((uint8_t)b); }
double oracle_round_bf16(double v) { return (double)round_bf16((real)v); }
int oracle_real_bytes(void) { return (int)sizeof(real); }
