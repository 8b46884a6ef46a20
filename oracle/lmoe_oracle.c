/*
 * CPU oracle for the latent mixture-of-experts layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call this code:
 * only the tests, the package smoke check and the benchmark's CPU-baseline
 * leg load it.  It shares no code with the CUDA library.
 *
 * What it computes follows the pages, stage by stage, in plain loops:
 *
 *  - "Muse Spark Open on Gaudi 2", section "What was built": the router is
 *    fp32, 256 experts, top 8; experts run W4A16 (bf16 activations, MXFP4
 *    weights), not W4A4.
 *  - same page, "Why it needed a port": the MXFP4 checkpoint is read as packed
 *    E2M1 nibbles plus E8M0 scale bytes.  The code table, the 32-element block
 *    along K and the nibble order (low nibble = even element) are those of the
 *    OCP Microscaling Formats (MX) v1.0 specification.
 *  - same page, "The latent MoE: A' with a per-expert norm": every (token,
 *    route) pair is its own row; post_expert_norm is applied to each row, the
 *    rows are multiplied by the router weights and summed in fp32, then the
 *    result is unpooled 4096 -> 8192.
 *  - same page, "Correctness": the CPU reference keeps bf16 values with fp32
 *    accumulation and dequantises MXFP4 exactly.
 *  - "Soporte de dia 0 para Muse Spark Open en vLLM", section "MoE latente":
 *    pooler (8192 -> 4096) and unpooler (4096 -> 8192) are learned
 *    projections shared by all experts of the layer; experts work at 4096.
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *  - router probabilities: softmax over all E logits, then the selected top-k
 *    are renormalised to sum to one;
 *  - top-k order: descending logit, ties to the lower expert index;
 *  - router logit: the dot product is accumulated in fp64 and rounded once to
 *    fp32 (the correctly rounded fp32 logit), then the optional bias is added
 *    in fp32;
 *  - expert MLP: rows 0..I-1 of W13 are the gate, rows I..2I-1 the up
 *    projection, h = bf16(silu(gate) * up), y = h . W2^T, no bias or clamp;
 *  - post_expert_norm: RMSNorm over the latent width with eps inside the
 *    square root and a per-expert bf16 gain;
 *  - bf16 round-to-nearest-even at x_lat, h, z (before the unpooler) and out;
 *  - every weight matrix is stored [N_out][K_in], K contiguous.
 *
 * Sums run sequentially in index order in fp32 (compiled with
 * -ffp-contract=off), so a result does not depend on the thread count.
 * oracle_set_acc64(1) switches every such sum (projections, experts, norms,
 * the weighted sum) to fp64, rounded where the fp32 sum is: the difference
 * between the two runs is the oracle's own fp32 accumulation error.
 *
 * LMOE_ORACLE_PLANT (tests only): building with -DLMOE_ORACLE_PLANT=n plants
 * one plausible mistake so the pin tests can show that they catch it.  The
 * default build defines nothing and contains none of them.
 *   1 nibble order swapped          2 gate and up swapped
 *   3 W2 read transposed            4 block scale off by one
 *   5 weights not renormalised      6 ties go to the higher index
 *   7 norm applied to the sum       8 norm gain dropped
 *   9 row RMSNorm drops its gain    10 block drops the residual
 *  11 NVFP4 blocks of 32           12 NVFP4 global scale dropped
 *
 * NVFP4 expert weights ("Muse Spark Open on Gaudi 2" and the vLLM page name
 * the NVFP4 checkpoint; they give no layout).  The format follows NVIDIA's
 * public NVFP4 description: E2M1 elements as in MXFP4 (two per byte, low
 * nibble = even element), one FP8 E4M3 scale per 16 consecutive elements
 * along K (the OCP 8-bit floating point E4M3 encoding: bias 7, no infinity,
 * S.1111.111 = NaN), and one fp32 scale per expert matrix:
 *   w[n][c] = (E2M1(nibble) * E4M3(scale[n][c/16])) * global[e].
 * E2M1 * E4M3 has at most 6 significant bits, exact in fp32 (and bf16); the
 * product with the fp32 global scale is rounded once.
 *
 * The transformer block around the layer ("Soporte de dia 0 para Muse Spark
 * Open en vLLM", section "Normalizacion en sandwich": one norm before the
 * block and one after it, y = x + post_norm(F(norm(x)))), with the router fed
 * by the fp32 output of the pre-norm (same page, section "Nvidia"):
 *  - each norm is an RMSNorm over the hidden width, eps inside the square
 *    root, a bf16 gain per column, multiply order (x * rinv) * g, as for
 *    post_expert_norm;
 *  - the router reads the pre-norm's fp32 output; the pooler reads it
 *    rounded to bf16 (the layer's activations are bf16);
 *  - the residual sum x + post_norm(out) is formed in fp32 and rounded once
 *    to bf16.
 */
#ifndef LMOE_ORACLE_PLANT
#define LMOE_ORACLE_PLANT 0
#endif
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
  int32_t T, H, L, I, E, k;
  float eps;
} or_dims;

/* ------------------------------------------------------------------------ */
/* number formats                                                           */
/* ------------------------------------------------------------------------ */

static float bits_to_f32(uint32_t u) {
  float f;
  memcpy(&f, &u, 4);
  return f;
}

static uint32_t f32_to_bits(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  return u;
}

/* bf16 -> fp32 is exact: the bf16 pattern is the top half of the fp32 one. */
static float bf16_val(uint16_t b) { return bits_to_f32((uint32_t)b << 16); }

/* fp32 -> bf16, round to nearest, ties to even; NaN stays a quiet NaN. */
uint16_t oracle_bf16_rne(float f) {
  uint32_t u = f32_to_bits(f);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0)
    return (uint16_t)((u >> 16) | 0x0040u);
  uint32_t lower = u & 0xFFFFu;
  uint32_t upper = u >> 16;
  if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1;
  return (uint16_t)upper;
}

/* E2M1 (OCP MX v1.0): bit 3 sign, bits 2..1 exponent (bias 1), bit 0 mantissa.
 * Exponent field 0 is subnormal: value = mantissa * 0.5. */
static float e2m1_value(unsigned code) {
  unsigned s = (code >> 3) & 1u, e = (code >> 1) & 3u, m = code & 1u;
  float mag = (e == 0) ? 0.5f * (float)m : ldexpf(1.0f + 0.5f * (float)m, (int)e - 1);
  return s ? -mag : mag;
}

/* E8M0: 2^(s-127); 255 is NaN (never produced by the generator). */
static float e8m0_value(unsigned s) {
  if (s == 255u) return NAN;
  return ldexpf(1.0f, (int)s - 127 + (LMOE_ORACLE_PLANT == 4));
}

/* OCP FP8 E4M3: bit 7 sign, bits 6..3 exponent (bias 7), bits 2..0 mantissa;
 * exponent 0 is subnormal (m/8 * 2^-6); S.1111.111 is NaN; no infinity. */
float oracle_e4m3_value(unsigned b) {
  unsigned s = (b >> 7) & 1u, e = (b >> 3) & 15u, m = b & 7u;
  float mag;
  if (e == 15u && m == 7u) return NAN;
  if (e == 0u)
    mag = ldexpf((float)m / 8.0f, -6);
  else
    mag = ldexpf(1.0f + (float)m / 8.0f, (int)e - 7);
  return s ? -mag : mag;
}

/* E2M1 code times an E4M3 scale byte (the NVFP4 block value before the global scale). */
float oracle_nvfp4_value(unsigned code, unsigned scale_byte) {
  return e2m1_value(code & 15u) * oracle_e4m3_value(scale_byte & 255u);
}

/* One dequantised MXFP4 element: value of code `code` under block scale `s`.
 * Exact in fp32 for s <= 252 (the product has at most 2 significant bits). */
float oracle_mxfp4_value(unsigned code, unsigned s) { return e2m1_value(code & 15u) * e8m0_value(s); }

/* Lookup tables filled from the two functions above (speed only: every
 * entry is exactly the function's value). */
static float g_e2m1_tab[16];
static float g_e8m0_tab[256];
static float g_e4m3_tab[256];
static pthread_once_t g_tab_once = PTHREAD_ONCE_INIT;
static void fill_tables(void) {
  for (unsigned c = 0; c < 16; ++c) g_e2m1_tab[c] = e2m1_value(c);
  for (unsigned s = 0; s < 256; ++s) g_e8m0_tab[s] = e8m0_value(s);
  for (unsigned s = 0; s < 256; ++s) g_e4m3_tab[s] = oracle_e4m3_value(s);
}

/* Element c of row n of a packed [N][K/2] code matrix with [N][K/32] scales. */
static inline float mx_elem(const uint8_t* q, const uint8_t* sc, int64_t n, int64_t K, int64_t c) {
  uint8_t byte = q[n * (K / 2) + c / 2];
  unsigned code = ((c & 1) ^ (LMOE_ORACLE_PLANT == 1)) ? (byte >> 4) : (byte & 15u);
  return g_e2m1_tab[code] * g_e8m0_tab[sc[n * (K / 32) + c / 32]];
}

/* NVFP4 element c of row n: [N][K/2] codes, [N][K/16] E4M3 scales, the
 * matrix's global scale gs. */
#define NV_BLOCK (LMOE_ORACLE_PLANT == 11 ? 32 : 16)
static inline float nv_elem(const uint8_t* q, const uint8_t* sc, int64_t n, int64_t K, int64_t c, float gs) {
  uint8_t byte = q[n * (K / 2) + c / 2];
  unsigned code = (c & 1) ? (byte >> 4) : (byte & 15u);
  float v = g_e2m1_tab[code] * g_e4m3_tab[sc[n * (K / 16) + c / NV_BLOCK]];
#if LMOE_ORACLE_PLANT == 12
  (void)gs;
  return v;
#else
  return v * gs;
#endif
}

/* ------------------------------------------------------------------------ */
/* parallel for over an outer index: each index is computed by exactly one   */
/* thread with the same sequential inner loops, so bits do not depend on the  */
/* thread count                                                               */
/* ------------------------------------------------------------------------ */

static int g_threads = 1;
void oracle_set_threads(int n) { g_threads = n < 1 ? 1 : (n > 256 ? 256 : n); }

static int g_acc64 = 0; /* 1: sums in fp64 (diagnostic), rounded at the same points */
void oracle_set_acc64(int on) { g_acc64 = on ? 1 : 0; }
int oracle_get_acc64(void) { return g_acc64; }
int oracle_get_threads(void) { return g_threads; }

typedef void (*body_fn)(void* ctx, int64_t i);
typedef struct {
  body_fn fn;
  void* ctx;
  int64_t n;
  int tid, nth;
} pf_job;

static void* pf_run(void* arg) {
  pf_job* j = (pf_job*)arg;
  for (int64_t i = j->tid; i < j->n; i += j->nth) j->fn(j->ctx, i);
  return NULL;
}

static void parallel_for(int64_t n, body_fn fn, void* ctx) {
  int nth = g_threads;
  if (nth > n) nth = (int)(n > 0 ? n : 1);
  pthread_t th[256];
  pf_job jobs[256];
  for (int t = 0; t < nth; ++t) jobs[t] = (pf_job){fn, ctx, n, t, nth};
  for (int t = 1; t < nth; ++t) pthread_create(&th[t], NULL, pf_run, &jobs[t]);
  pf_run(&jobs[0]);
  for (int t = 1; t < nth; ++t) pthread_join(th[t], NULL);
}

/* ------------------------------------------------------------------------ */
/* step 1: router logits (fp32 router, "What was built")                    */
/* ------------------------------------------------------------------------ */

typedef struct {
  const or_dims* d;
  const uint16_t* x;
  const float* wr;
  const float* bias;
  float* logits;
  double* absdot;
} router_ctx;

static void router_body(void* p, int64_t i) {
  router_ctx* c = (router_ctx*)p;
  int64_t t = i / c->d->E, e = i % c->d->E, H = c->d->H;
  double acc = 0.0, mag = 0.0;
  for (int64_t h = 0; h < H; ++h) {
    double prod = (double)bf16_val(c->x[t * H + h]) * (double)c->wr[e * H + h];
    acc += prod;
    mag += fabs(prod);
  }
  float lg = (float)acc;
  if (c->bias) lg = lg + c->bias[e];
  c->logits[t * c->d->E + e] = lg;
  if (c->absdot) c->absdot[t * c->d->E + e] = mag;
}

/* logits[t][e] = fp32(sum_h x[t][h] * Wr[e][h]) (+ bias[e]); absdot (optional)
 * gets sum_h |x * Wr|, the scale of the rounding error of any fp32 sum. */
void oracle_router_logits(const or_dims* d, const uint16_t* x, const float* router_w,
                          const float* router_bias, float* logits, double* absdot) {
  router_ctx c = {d, x, router_w, router_bias, logits, absdot};
  parallel_for((int64_t)d->T * d->E, router_body, &c);
}

/* The same logits for an fp32 input row (the sandwich block's pre-norm
 * output): every product of two fp32 values is exact in fp64, so the fp64 sum
 * rounded once is again the correctly rounded fp32 logit. */
typedef struct {
  const or_dims* d;
  const float* x;
  const float* wr;
  const float* bias;
  float* logits;
  double* absdot;
} router_f32_ctx;

static void router_f32_body(void* p, int64_t i) {
  router_f32_ctx* c = (router_f32_ctx*)p;
  int64_t t = i / c->d->E, e = i % c->d->E, H = c->d->H;
  double acc = 0.0, mag = 0.0;
  for (int64_t h = 0; h < H; ++h) {
    double prod = (double)c->x[t * H + h] * (double)c->wr[e * H + h];
    acc += prod;
    mag += fabs(prod);
  }
  float lg = (float)acc;
  if (c->bias) lg = lg + c->bias[e];
  c->logits[t * c->d->E + e] = lg;
  if (c->absdot) c->absdot[t * c->d->E + e] = mag;
}

void oracle_router_logits_f32(const or_dims* d, const float* x, const float* router_w, const float* router_bias,
                              float* logits, double* absdot) {
  router_f32_ctx c = {d, x, router_w, router_bias, logits, absdot};
  parallel_for((int64_t)d->T * d->E, router_f32_body, &c);
}

/* ------------------------------------------------------------------------ */
/* step 2: top-k selection and softmax-renormalised weights                 */
/* ------------------------------------------------------------------------ */

/* For each token: the k largest logits in descending order (ties: lower
 * index first), p = softmax over all E logits (fp64), w_j = p_j / sum_sel p. */
void oracle_topk(const or_dims* d, const float* logits, int32_t* topk_idx, float* topk_w) {
  int E = d->E, k = d->k;
  char* taken = (char*)malloc((size_t)E);
  double* p = (double*)malloc(sizeof(double) * (size_t)E);
  for (int t = 0; t < d->T; ++t) {
    const float* lg = logits + (int64_t)t * E;
    memset(taken, 0, (size_t)E);
    for (int j = 0; j < k; ++j) {
      int best = -1;
      for (int e = 0; e < E; ++e) {
        if (taken[e]) continue;
#if LMOE_ORACLE_PLANT == 6
        if (best < 0 || lg[e] >= lg[best]) best = e;
#else
        if (best < 0 || lg[e] > lg[best]) best = e; /* strict '>' keeps the lower index on ties */
#endif
      }
      taken[best] = 1;
      topk_idx[t * k + j] = best;
    }
    double mx = lg[0];
    for (int e = 1; e < E; ++e)
      if (lg[e] > mx) mx = lg[e];
    double den = 0.0;
    for (int e = 0; e < E; ++e) {
      p[e] = exp((double)lg[e] - mx);
      den += p[e];
    }
    for (int e = 0; e < E; ++e) p[e] /= den;
    double sel = 0.0;
    for (int j = 0; j < k; ++j) sel += p[topk_idx[t * k + j]];
    if (LMOE_ORACLE_PLANT == 5) sel = 1.0;
    for (int j = 0; j < k; ++j) topk_w[t * k + j] = (float)(p[topk_idx[t * k + j]] / sel);
  }
  free(taken);
  free(p);
}

/* ------------------------------------------------------------------------ */
/* step 3: routing table: the (token, route) rows grouped by expert          */
/* ("The latent MoE ...": each (token, route) pair is its own row)          */
/* ------------------------------------------------------------------------ */

/* Row id r = t*k + j.  offsets = exclusive scan of per-expert counts
 * (E+1 entries); sorted_rows lists row ids by expert, ascending r within an
 * expert; row_pos is the inverse permutation. */
void oracle_table(const or_dims* d, const int32_t* topk_idx, int32_t* offsets,
                  int32_t* sorted_rows, int32_t* row_pos) {
  int E = d->E;
  int64_t R = (int64_t)d->T * d->k;
  int32_t* fill = (int32_t*)calloc((size_t)E, sizeof(int32_t));
  for (int e = 0; e <= E; ++e) offsets[e] = 0;
  for (int64_t r = 0; r < R; ++r) offsets[topk_idx[r] + 1] += 1;
  for (int e = 0; e < E; ++e) offsets[e + 1] += offsets[e];
  for (int64_t r = 0; r < R; ++r) {
    int e = topk_idx[r];
    int32_t pos = offsets[e] + fill[e]++;
    sorted_rows[pos] = (int32_t)r;
    row_pos[r] = pos;
  }
  free(fill);
}

/* ------------------------------------------------------------------------ */
/* step 4: pooler, x_lat = bf16(x . P^T)  ("MoE latente")                    */
/* ------------------------------------------------------------------------ */

typedef struct {
  const or_dims* d;
  const uint16_t* x;
  const uint16_t* P;
  uint16_t* x_lat;
} pool_ctx;

static void pool_body(void* p, int64_t i) {
  pool_ctx* c = (pool_ctx*)p;
  int64_t t = i / c->d->L, l = i % c->d->L, H = c->d->H;
  float acc = 0.0f;
  if (g_acc64) {
    double a = 0.0;
    for (int64_t h = 0; h < H; ++h) a += (double)bf16_val(c->x[t * H + h]) * (double)bf16_val(c->P[l * H + h]);
    acc = (float)a;
  } else {
    for (int64_t h = 0; h < H; ++h) acc += bf16_val(c->x[t * H + h]) * bf16_val(c->P[l * H + h]);
  }
  c->x_lat[t * c->d->L + l] = oracle_bf16_rne(acc);
}

void oracle_pool(const or_dims* d, const uint16_t* x, const uint16_t* pooler_w, uint16_t* x_lat) {
  pool_ctx c = {d, x, pooler_w, x_lat};
  parallel_for((int64_t)d->T * d->L, pool_body, &c);
}

/* ------------------------------------------------------------------------ */
/* step 5: routed experts, W4A16 SwiGLU, one output row per (token, route)  */
/* ------------------------------------------------------------------------ */

typedef struct {
  const or_dims* d;
  const uint16_t* x_lat;
  const int32_t* idx;
  const uint8_t *w13q, *w13s, *w2q, *w2s;
  uint16_t* h;  /* [R][I] bf16, required scratch */
  float* gu;    /* [R][2I] optional pre-activation gate/up */
  float* y;     /* [R][L] */
  const float *w13gs, *w2gs; /* NVFP4 global scales [E] (both NULL: MXFP4) */
} exp_ctx;

/* element c of row n of W13 / W2 in the context's format */
static inline float w13_elem(const exp_ctx* c, int64_t e, int64_t n, int64_t col) {
  int64_t L = c->d->L;
  return c->w13gs ? nv_elem(c->w13q, c->w13s, n, L, col, c->w13gs[e]) : mx_elem(c->w13q, c->w13s, n, L, col);
}
static inline float w2_elem(const exp_ctx* c, int64_t e, int64_t n, int64_t col) {
  int64_t I = c->d->I;
  return c->w2gs ? nv_elem(c->w2q, c->w2s, n, I, col, c->w2gs[e]) : mx_elem(c->w2q, c->w2s, n, I, col);
}

/* phase 1 body: one (row, feature) pair -> gate, up, h */
static void gateup_body(void* p, int64_t i) {
  exp_ctx* c = (exp_ctx*)p;
  int64_t I = c->d->I, L = c->d->L;
  int64_t r = i / I, f = i % I;
  int64_t t = r / c->d->k, e = c->idx[r];
  const uint16_t* xr = c->x_lat + t * L;
  int64_t gate_row = e * 2 * I + f, up_row = e * 2 * I + I + f;
#if LMOE_ORACLE_PLANT == 2
  { int64_t tmp = gate_row; gate_row = up_row; up_row = tmp; }
#endif
  float g = 0.0f, u = 0.0f;
  if (g_acc64) {
    double gd = 0.0, ud = 0.0;
    for (int64_t l = 0; l < L; ++l) gd += (double)bf16_val(xr[l]) * (double)w13_elem(c, e, gate_row, l);
    for (int64_t l = 0; l < L; ++l) ud += (double)bf16_val(xr[l]) * (double)w13_elem(c, e, up_row, l);
    g = (float)gd;
    u = (float)ud;
  } else {
    for (int64_t l = 0; l < L; ++l) g += bf16_val(xr[l]) * w13_elem(c, e, gate_row, l);
    for (int64_t l = 0; l < L; ++l) u += bf16_val(xr[l]) * w13_elem(c, e, up_row, l);
  }
  float silu = g / (1.0f + expf(-g));
  c->h[r * I + f] = oracle_bf16_rne(silu * u);
  if (c->gu) {
    c->gu[r * 2 * I + f] = g;
    c->gu[r * 2 * I + I + f] = u;
  }
}

/* phase 2 body: one (row, latent column) pair -> y */
static void down_body(void* p, int64_t i) {
  exp_ctx* c = (exp_ctx*)p;
  int64_t I = c->d->I, L = c->d->L;
  int64_t r = i / L, l = i % L;
  int64_t e = c->idx[r];
  const uint16_t* hr = c->h + r * I;
  float acc = 0.0f;
  double accd = 0.0;
#if LMOE_ORACLE_PLANT == 3
  for (int64_t f = 0; f < I; ++f) {
    if (g_acc64) accd += (double)bf16_val(hr[f]) * (double)w2_elem(c, e, e * L + f, l);
    else acc += bf16_val(hr[f]) * w2_elem(c, e, e * L + f, l);
  }
#else
  for (int64_t f = 0; f < I; ++f) {
    if (g_acc64) accd += (double)bf16_val(hr[f]) * (double)w2_elem(c, e, e * L + l, f);
    else acc += bf16_val(hr[f]) * w2_elem(c, e, e * L + l, f);
  }
#endif
  c->y[r * L + l] = g_acc64 ? (float)accd : acc;
}

/* y[r][:] for every route row r = t*k + j with expert e = topk_idx[r].
 * h_out (optional, [R][I] bf16) and gu_out (optional, [R][2I] fp32) expose
 * the intermediate values. */
void oracle_experts(const or_dims* d, const uint16_t* x_lat, const int32_t* topk_idx,
                    const uint8_t* w13_q, const uint8_t* w13_s, const uint8_t* w2_q,
                    const uint8_t* w2_s, uint16_t* h_out, float* gu_out, float* y) {
  int64_t R = (int64_t)d->T * d->k;
  pthread_once(&g_tab_once, fill_tables);
  uint16_t* h = h_out ? h_out : (uint16_t*)malloc(sizeof(uint16_t) * (size_t)(R * d->I));
  exp_ctx c = {d, x_lat, topk_idx, w13_q, w13_s, w2_q, w2_s, h, gu_out, y, NULL, NULL};
  parallel_for(R * d->I, gateup_body, &c);
  parallel_for(R * d->L, down_body, &c);
  if (!h_out) free(h);
}

/* The same experts on NVFP4 weights: w13_s [E][2I][L/16] and w2_s [E][L][I/16]
 * E4M3 bytes, w13_gs and w2_gs the fp32 global scale of each expert's matrix. */
void oracle_experts_nvfp4(const or_dims* d, const uint16_t* x_lat, const int32_t* topk_idx, const uint8_t* w13_q,
                          const uint8_t* w13_s, const float* w13_gs, const uint8_t* w2_q, const uint8_t* w2_s,
                          const float* w2_gs, uint16_t* h_out, float* gu_out, float* y) {
  int64_t R = (int64_t)d->T * d->k;
  pthread_once(&g_tab_once, fill_tables);
  uint16_t* h = h_out ? h_out : (uint16_t*)malloc(sizeof(uint16_t) * (size_t)(R * d->I));
  exp_ctx c = {d, x_lat, topk_idx, w13_q, w13_s, w2_q, w2_s, h, gu_out, y, w13_gs, w2_gs};
  parallel_for(R * d->I, gateup_body, &c);
  parallel_for(R * d->L, down_body, &c);
  if (!h_out) free(h);
}

/* ------------------------------------------------------------------------ */
/* steps 6-7: post_expert_norm on each route row, then the fp32 weighted sum */
/* ------------------------------------------------------------------------ */

/* For each route row r (expert e): ms = sum_l y^2 / L, rinv = 1/sqrt(ms+eps),
 * yhat[l] = (y[l] * rinv) * g[e][l].  z[t][l] = sum_j w[t][j] * yhat[t*k+j][l]
 * in j order.  yhat_out (optional, [R][L]) exposes the normed rows. */
void oracle_norm_combine(const or_dims* d, const float* y, const int32_t* topk_idx,
                         const float* topk_w, const uint16_t* norm_g, float* yhat_out, float* z) {
  int64_t L = d->L, k = d->k;
  float* yh = (float*)malloc(sizeof(float) * (size_t)L);
  double* zd = (double*)malloc(sizeof(double) * (size_t)L); /* fp64 sums (acc64) */
  for (int64_t t = 0; t < d->T; ++t) {
    for (int64_t l = 0; l < L; ++l) z[t * L + l] = 0.0f;
    for (int64_t l = 0; l < L; ++l) zd[l] = 0.0;
    for (int64_t j = 0; j < k; ++j) {
      int64_t r = t * k + j, e = topk_idx[r];
      const float* yr = y + r * L;
      float ss = 0.0f;
      if (g_acc64) {
        double sd = 0.0;
        for (int64_t l = 0; l < L; ++l) sd += (double)yr[l] * (double)yr[l];
        ss = (float)sd;
      } else {
        for (int64_t l = 0; l < L; ++l) ss += yr[l] * yr[l];
      }
      float ms = ss / (float)L;
      float rinv = 1.0f / sqrtf(ms + d->eps);
#if LMOE_ORACLE_PLANT == 7
      rinv = 1.0f;
#endif
#if LMOE_ORACLE_PLANT == 8
      for (int64_t l = 0; l < L; ++l) yh[l] = yr[l] * rinv;
#else
      for (int64_t l = 0; l < L; ++l) yh[l] = (yr[l] * rinv) * bf16_val(norm_g[e * L + l]);
#endif
      if (yhat_out) memcpy(yhat_out + r * L, yh, sizeof(float) * (size_t)L);
      float w = topk_w[r];
      if (g_acc64) {
        for (int64_t l = 0; l < L; ++l) zd[l] += (double)(w * yh[l]);
      } else {
        for (int64_t l = 0; l < L; ++l) z[t * L + l] += w * yh[l];
      }
    }
    if (g_acc64)
      for (int64_t l = 0; l < L; ++l) z[t * L + l] = (float)zd[l];
#if LMOE_ORACLE_PLANT == 7
    {
      float ss = 0.0f;
      for (int64_t l = 0; l < L; ++l) ss += z[t * L + l] * z[t * L + l];
      float rinv = 1.0f / sqrtf(ss / (float)L + d->eps);
      for (int64_t l = 0; l < L; ++l) z[t * L + l] *= rinv;
    }
#endif
  }
  free(yh);
  free(zd);
}

/* ------------------------------------------------------------------------ */
/* step 8: unpooler, out = bf16(bf16(z) . U^T)                              */
/* ------------------------------------------------------------------------ */

typedef struct {
  const or_dims* d;
  const uint16_t* zb;
  const uint16_t* U;
  uint16_t* out;
} unpool_ctx;

static void unpool_body(void* p, int64_t i) {
  unpool_ctx* c = (unpool_ctx*)p;
  int64_t t = i / c->d->H, o = i % c->d->H, L = c->d->L;
  float acc = 0.0f;
  if (g_acc64) {
    double a = 0.0;
    for (int64_t l = 0; l < L; ++l) a += (double)bf16_val(c->zb[t * L + l]) * (double)bf16_val(c->U[o * L + l]);
    acc = (float)a;
  } else {
    for (int64_t l = 0; l < L; ++l) acc += bf16_val(c->zb[t * L + l]) * bf16_val(c->U[o * L + l]);
  }
  c->out[t * c->d->H + o] = oracle_bf16_rne(acc);
}

void oracle_unpool(const or_dims* d, const float* z, const uint16_t* unpooler_w, uint16_t* out) {
  int64_t n = (int64_t)d->T * d->L;
  uint16_t* zb = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)n);
  for (int64_t i = 0; i < n; ++i) zb[i] = oracle_bf16_rne(z[i]);
  unpool_ctx c = {d, zb, unpooler_w, out};
  parallel_for((int64_t)d->T * d->H, unpool_body, &c);
  free(zb);
}

/* ------------------------------------------------------------------------ */
/* whole layer                                                              */
/* ------------------------------------------------------------------------ */

/* Runs every step.  The optional outputs (any may be NULL) expose the
 * intermediate results so each GPU call can be checked on its own. */
void oracle_forward(const or_dims* d, const uint16_t* x, const float* router_w,
                    const float* router_bias, const uint16_t* pooler_w, const uint8_t* w13_q,
                    const uint8_t* w13_s, const uint8_t* w2_q, const uint8_t* w2_s,
                    const uint16_t* norm_g, const uint16_t* unpooler_w, uint16_t* out,
                    int32_t* topk_idx, float* topk_w, uint16_t* x_lat_out, float* y_out,
                    float* z_out) {
  int64_t T = d->T, R = T * d->k;
  float* logits = (float*)malloc(sizeof(float) * (size_t)(T * d->E));
  int32_t* idx = topk_idx ? topk_idx : (int32_t*)malloc(sizeof(int32_t) * (size_t)R);
  float* w = topk_w ? topk_w : (float*)malloc(sizeof(float) * (size_t)R);
  uint16_t* x_lat = x_lat_out ? x_lat_out : (uint16_t*)malloc(sizeof(uint16_t) * (size_t)(T * d->L));
  float* y = y_out ? y_out : (float*)malloc(sizeof(float) * (size_t)(R * d->L));
  float* z = z_out ? z_out : (float*)malloc(sizeof(float) * (size_t)(T * d->L));
  oracle_router_logits(d, x, router_w, router_bias, logits, NULL);
  oracle_topk(d, logits, idx, w);
  oracle_pool(d, x, pooler_w, x_lat);
  oracle_experts(d, x_lat, idx, w13_q, w13_s, w2_q, w2_s, NULL, NULL, y);
  oracle_norm_combine(d, y, idx, w, norm_g, NULL, z);
  oracle_unpool(d, z, unpooler_w, out);
  free(logits);
  if (!topk_idx) free(idx);
  if (!topk_w) free(w);
  if (!x_lat_out) free(x_lat);
  if (!y_out) free(y);
  if (!z_out) free(z);
}

/* ------------------------------------------------------------------------ */
/* sandwich block around the layer                                          */
/* ------------------------------------------------------------------------ */

/* RMSNorm of each of `rows` bf16 rows of width W: ss = sum x^2 (fp32,
 * sequential), rinv = 1/sqrt(ss/W + eps), out = (x * rinv) * g in fp32. */
void oracle_rmsnorm_rows(int64_t rows, int64_t W, const uint16_t* x, const uint16_t* g, float eps, float* out) {
  for (int64_t r = 0; r < rows; ++r) {
    const uint16_t* xr = x + r * W;
    float ss = 0.0f;
    if (g_acc64) {
      double sd = 0.0;
      for (int64_t c = 0; c < W; ++c) sd += (double)bf16_val(xr[c]) * (double)bf16_val(xr[c]);
      ss = (float)sd;
    } else {
      for (int64_t c = 0; c < W; ++c) ss += bf16_val(xr[c]) * bf16_val(xr[c]);
    }
    float rinv = 1.0f / sqrtf(ss / (float)W + eps);
    for (int64_t c = 0; c < W; ++c) {
#if LMOE_ORACLE_PLANT == 9
      out[r * W + c] = bf16_val(xr[c]) * rinv;
#else
      out[r * W + c] = (bf16_val(xr[c]) * rinv) * bf16_val(g[c]);
#endif
    }
  }
}

/* bf16 round-to-nearest-even of n fp32 values. */
void oracle_bf16_round(int64_t n, const float* a, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_bf16_rne(a[i]);
}

/* out = bf16(x + p): the residual sum in fp32, rounded once. */
void oracle_residual_add(int64_t n, const uint16_t* x, const float* p, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) {
#if LMOE_ORACLE_PLANT == 10
    out[i] = oracle_bf16_rne(p[i]);
#else
    out[i] = oracle_bf16_rne(bf16_val(x[i]) + p[i]);
#endif
  }
}
