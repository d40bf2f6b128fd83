/*
 * moe_oracle.c -- plain, slow fp64 CPU oracle of the W4A16 MoE expert layer.
 *
 * TEST INFRASTRUCTURE ONLY.  This file defines what "correct" means for the
 * GPU library; it is linked only by the tests, by the package smoke check and
 * by the CPU-baseline leg of the benchmark.  It shares no code, header, table
 * or helper with the CUDA path (which lives in the package's csrc/ directory)
 * and must never be called by the product path.
 *
 * Sources (web pages; section names as printed on them):
 *   [MC]  "srswti/axe-diffusion-ksl-xe" model card:
 *           "what the model is"      -- 128-expert MoE, top-8 routing per token
 *           "the kernels we built"   -- asymmetric uint4, fp16 scale and zero-point
 *                                       per group, packed nibbles dequantised inline;
 *                                       activation folded into the first GEMM;
 *                                       fixed-order weighted combine (no index_add_)
 *           "requirements"           -- format dg-w4a16-v1: two nibbles per byte,
 *                                       gate_up_proj groups of 128 along the
 *                                       contraction dim, down_proj groups of 64
 *   [TF]  "ashhart/TensorFold pull 802", paragraph "FP64 reference": an int4 GEMM
 *         is compared with an FP64 evaluation of the same dequantised weights.
 *
 * Readings where the pages are silent (each one is listed in the design notes):
 *   - gating: softmax over the k selected logits only (no temperature, no bias);
 *   - ties between equal logits go to the lower expert index; logits compare as
 *     fp32 values, so -0 and +0 tie;
 *   - nibble order: byte b of a row holds k = 2b in its low nibble and k = 2b+1
 *     in its high nibble;
 *   - fused gate_up_proj: rows [0, f) are the gate projection, rows [f, 2f) the
 *     up projection; h = act(gate) * up;
 *   - act: GELU, tanh form by default, erf form selectable;
 *   - optional per-layer RMSNorm of the combined output: gamma * u / sqrt(mean(u^2) + eps);
 *   - the MoE block around the layer (pre-norm, router projection, residual): see
 *     oracle_block_front below.
 *
 * Everything below is the plain definition: weights are dequantised into a dense
 * fp64 matrix, the FFN is two fp64 matrix-vector products, and the combine is a
 * sum over router ranks in rank order.  No blocking, fusion or reordering.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_ERR_SHAPE 1
#define ORACLE_ERR_NONFINITE 2
#define ORACLE_ERR_ALLOC 3

/* ---------------------------------------------------------------- fp16 ---- */

/* IEEE-754 binary16 -> double, written out from the format: 1 sign bit,
 * 5 exponent bits (bias 15), 10 fraction bits; exponent 0 is subnormal. */
double oracle_half_to_double(uint16_t h) {
  int sign = (h >> 15) & 1;
  int expo = (h >> 10) & 0x1f;
  int frac = h & 0x3ff;
  double v;
  if (expo == 0) {
    v = ldexp((double)frac, -24); /* 2^-14 * frac / 2^10 */
  } else if (expo == 31) {
    v = frac ? NAN : INFINITY;
  } else {
    v = ldexp(1.0 + (double)frac / 1024.0, expo - 15);
  }
  return sign ? -v : v;
}

/* double -> binary16, round to nearest, ties to even (diagnostic mode only). */
uint16_t oracle_double_to_half(double v) {
  uint16_t sign = 0;
  if (signbit(v)) { sign = 0x8000; v = -v; }
  if (isnan(v)) return 0x7e00;
  if (v >= 65520.0) return (uint16_t)(sign | 0x7c00); /* rounds to infinity */
  /* subnormal grid below 2^-14 is spaced 2^-24 */
  int e;
  double m = frexp(v, &e);          /* v = m * 2^e, m in [0.5, 1) */
  if (v == 0.0) return sign;
  int expo = e - 1;                 /* v = (2m) * 2^(e-1), 2m in [1,2) */
  double quantum = expo < -14 ? ldexp(1.0, -24) : ldexp(1.0, expo - 10);
  double q = v / quantum;           /* exact: scaling by a power of two */
  double r = floor(q);
  double rem = q - r;
  if (rem > 0.5 || (rem == 0.5 && fmod(r, 2.0) != 0.0)) r += 1.0;
  double rv = r * quantum;
  /* re-derive the bit pattern from the rounded value */
  if (rv == 0.0) return sign;
  if (rv < ldexp(1.0, -14)) return (uint16_t)(sign | (uint16_t)(rv / ldexp(1.0, -24)));
  int e2;
  double m2 = frexp(rv, &e2);
  int ex = e2 - 1 + 15;
  if (ex >= 31) return (uint16_t)(sign | 0x7c00);
  uint16_t frac = (uint16_t)((2.0 * m2 - 1.0) * 1024.0);
  return (uint16_t)(sign | (ex << 10) | frac);
}

/* ------------------------------------------------------------- routing ---- */

typedef struct { float logit; int e; } oracle_cand;

/* Router order: larger logit first; equal logits (compared as fp32 values, so
 * -0 == +0) go to the lower expert index.  [MC "what the model is": top-8 of
 * 128 experts per token; tie rule is this library's stated reading.] */
static int cand_cmp(const void* pa, const void* pb) {
  const oracle_cand* a = (const oracle_cand*)pa;
  const oracle_cand* b = (const oracle_cand*)pb;
  if (a->logit > b->logit) return -1;
  if (a->logit < b->logit) return 1;
  return (a->e < b->e) ? -1 : (a->e > b->e) ? 1 : 0;
}

/* Top-k and gating for every token.
 *   logits   [T][E] fp32
 *   topk_idx [T][k] expert ids in router-rank order (rank 0 = largest logit)
 *   topk_w   [T][k] softmax over the k selected logits, in fp64:
 *            w_r = exp(l_r - l_0) / sum_j exp(l_j - l_0), summed in rank order.
 * Returns ORACLE_ERR_NONFINITE if any logit is NaN or infinite. */
int oracle_route(int T, int E, int k, const float* logits, int32_t* topk_idx, double* topk_w) {
  if (T < 0 || E < 1 || k < 1 || k > E) return ORACLE_ERR_SHAPE;
  oracle_cand* c = (oracle_cand*)malloc(sizeof(oracle_cand) * (size_t)E);
  if (!c) return ORACLE_ERR_ALLOC;
  for (int t = 0; t < T; ++t) {
    for (int e = 0; e < E; ++e) {
      float v = logits[(size_t)t * E + e];
      if (!isfinite(v)) { free(c); return ORACLE_ERR_NONFINITE; }
      c[e].logit = v;
      c[e].e = e;
    }
    qsort(c, (size_t)E, sizeof(oracle_cand), cand_cmp);
    double m = (double)c[0].logit;
    double denom = 0.0;
    for (int r = 0; r < k; ++r) denom += exp((double)c[r].logit - m);
    for (int r = 0; r < k; ++r) {
      topk_idx[(size_t)t * k + r] = c[r].e;
      topk_w[(size_t)t * k + r] = exp((double)c[r].logit - m) / denom;
    }
  }
  free(c);
  return ORACLE_OK;
}

/* Per-expert row lists.  For every expert e (ascending), the pairs p = t*k + r
 * with topk_idx[t][r] == e, listed with p ascending (hence token ascending).
 *   offsets   [E+1]: pairs of expert e are pair_list[offsets[e] .. offsets[e+1])
 *   pair_list [T*k]
 * [MC "the kernels we built": one launch covers all 128 experts, so the pairs
 * are grouped by expert; the in-expert order is this library's stated reading.] */
int oracle_permute(int T, int E, int k, const int32_t* topk_idx, int32_t* offsets, int32_t* pair_list) {
  if (T < 0 || E < 1 || k < 1) return ORACLE_ERR_SHAPE;
  int64_t P = (int64_t)T * k;
  int32_t n = 0;
  for (int e = 0; e < E; ++e) {
    offsets[e] = n;
    for (int64_t p = 0; p < P; ++p)
      if (topk_idx[p] == e) pair_list[n++] = (int32_t)p;
  }
  offsets[E] = n;
  return (n == P) ? ORACLE_OK : ORACLE_ERR_SHAPE; /* an id outside [0, E) */
}

/* ------------------------------------------------------- weight format ---- */

/* The code at column kk of a packed row: two nibbles per byte, low nibble =
 * even kk, high nibble = odd kk.  [MC "requirements"] */
int oracle_code(const uint8_t* packed_row, int64_t kk) {
  uint8_t b = packed_row[kk >> 1];
  return (kk & 1) ? (b >> 4) : (b & 15);
}

/* w = (q - z) * s with z and s the fp16 zero-point and scale of the group.
 * [MC "the kernels we built": asymmetric uint4, fp16 scale and zero per group] */
double oracle_dequant(int q, uint16_t zero_bits, uint16_t scale_bits) {
  return ((double)q - oracle_half_to_double(zero_bits)) * oracle_half_to_double(scale_bits);
}

/* The three checkpoint formats, each with one fp16 scale s and one fp16 second
 * value per group ([TF] "Summary": symmetric GPTQ 4/128 and MLX affine 4/64 next
 * to the model card's asymmetric uint4):
 *   format 0  asymmetric zero-point   w = (q - z) s      (second value z)
 *   format 1  affine bias (MLX)       w = q s + b        (second value b)
 *   format 2  symmetric (GPTQ)        w = (q - 8) s      (second value unused) */
double oracle_dequant_format(int q, uint16_t second_bits, uint16_t scale_bits, int format) {
  const double s = oracle_half_to_double(scale_bits);
  if (format == 1) return (double)q * s + oracle_half_to_double(second_bits);
  if (format == 2) return ((double)q - 8.0) * s;
  return ((double)q - oracle_half_to_double(second_bits)) * s;
}

/* Dense fp64 copy of one quantised matrix W [rows][K]:
 *   packed [rows][K/2] bytes, scale/zero [rows][K/g] fp16 bits. */
static void dequant_matrix(int64_t rows, int64_t K, int g, const uint8_t* packed, const uint16_t* scale,
                           const uint16_t* zero, int format, int round_fp16, double* W) {
  int64_t ng = K / g;
  for (int64_t n = 0; n < rows; ++n) {
    for (int64_t kk = 0; kk < K; ++kk) {
      int q = oracle_code(packed + n * (K / 2), kk);
      double w = oracle_dequant_format(q, zero[n * ng + kk / g], scale[n * ng + kk / g], format);
      if (round_fp16) w = oracle_half_to_double(oracle_double_to_half(w));
      W[n * K + kk] = w;
    }
  }
}

/* ----------------------------------------------------------- activation ---- */

/* GELU.  act = 0: tanh form 0.5 a (1 + tanh(sqrt(2/pi) (a + 0.044715 a^3)));
 *        act = 1: erf form  0.5 a (1 + erf(a / sqrt(2))).
 * The pages call the activation "gated" without naming the GELU variant. */
double oracle_gelu(double a, int act) {
  if (act == 1) return 0.5 * a * (1.0 + erf(a / sqrt(2.0)));
  const double c = sqrt(2.0 / M_PI);
  return 0.5 * a * (1.0 + tanh(c * (a + 0.044715 * a * a * a)));
}

/* ------------------------------------------------------------ the layer ---- */

typedef struct {
  int32_t tokens, hidden, inter, experts, top_k, group_gate_up, group_down, activation;
  int32_t format; /* 0 asymmetric zero-point, 1 affine bias, 2 symmetric (see oracle_dequant_format) */
} oracle_shape;

typedef struct {
  const uint8_t* gate_up_q;      /* [E][2f][d/2]   canonical packed nibbles */
  const uint16_t* gate_up_scale; /* [E][2f][d/g1]  fp16 bits */
  const uint16_t* gate_up_zero;  /* [E][2f][d/g1]  fp16 bits */
  const uint8_t* down_q;         /* [E][d][f/2] */
  const uint16_t* down_scale;    /* [E][d][f/g2] */
  const uint16_t* down_zero;     /* [E][d][f/g2] */
} oracle_weights;

static int shape_ok(const oracle_shape* s) {
  if (s->tokens < 0 || s->hidden < 2 || s->inter < 1 || s->experts < 1 || s->top_k < 1 ||
      s->top_k > s->experts)
    return 0;
  if (s->group_gate_up < 2 || s->group_down < 2) return 0;
  if (s->hidden % s->group_gate_up || s->inter % s->group_down) return 0;
  if (s->group_gate_up % 2 || s->group_down % 2) return 0;
  if (s->format < 0 || s->format > 2) return 0;
  return s->activation == 0 || s->activation == 1;
}

/* One expert's gated FFN on an fp64 input row:
 *   a = Wgu x (2f outputs), h_j = act(a_j) * a_{f+j}, y = Wd h.
 * [MC "the kernels we built": activation folded into the first GEMM's epilogue] */
static void expert_ffn(const oracle_shape* s, const double* Wgu, const double* Wd, const double* x,
                       int round_fp16, double* a, double* h, double* y) {
  int64_t d = s->hidden, f = s->inter;
  for (int64_t n = 0; n < 2 * f; ++n) {
    double acc = 0.0;
    for (int64_t kk = 0; kk < d; ++kk) acc += Wgu[n * d + kk] * x[kk];
    a[n] = acc;
  }
  for (int64_t j = 0; j < f; ++j) {
    double hj = oracle_gelu(a[j], s->activation) * a[f + j];
    h[j] = round_fp16 ? oracle_half_to_double(oracle_double_to_half(hj)) : hj;
  }
  for (int64_t i = 0; i < d; ++i) {
    double acc = 0.0;
    for (int64_t j = 0; j < f; ++j) acc += Wd[i * f + j] * h[j];
    y[i] = acc;
  }
}

typedef struct {
  const oracle_shape* s;
  const oracle_weights* w;
  const uint16_t* x;         /* [T][d] fp16 bits */
  const int32_t* topk_idx;   /* [T][k] */
  const uint8_t* token_sel;  /* [T] nonzero = compute this token; NULL = all */
  double* ypair;             /* [T*k][d] */
  int round_fp16;
  int e_begin, e_step;
  int status;
} expert_job;

/* Computes y_pair for every (token, rank) routed to the experts of this job. */
static void* expert_worker(void* arg) {
  expert_job* j = (expert_job*)arg;
  const oracle_shape* s = j->s;
  int64_t d = s->hidden, f = s->inter, T = s->tokens, k = s->top_k;
  double* Wgu = (double*)malloc(sizeof(double) * (size_t)(2 * f * d));
  double* Wd = (double*)malloc(sizeof(double) * (size_t)(d * f));
  double* xd = (double*)malloc(sizeof(double) * (size_t)d);
  double* a = (double*)malloc(sizeof(double) * (size_t)(2 * f));
  double* h = (double*)malloc(sizeof(double) * (size_t)f);
  if (!Wgu || !Wd || !xd || !a || !h) { j->status = ORACLE_ERR_ALLOC; goto done; }
  for (int e = j->e_begin; e < s->experts; e += j->e_step) {
    int used = 0;
    for (int64_t p = 0; p < T * k && !used; ++p)
      used = j->topk_idx[p] == e && (!j->token_sel || j->token_sel[p / k]);
    if (!used) continue;
    int64_t ng1 = d / s->group_gate_up, ng2 = f / s->group_down;
    dequant_matrix(2 * f, d, s->group_gate_up, j->w->gate_up_q + (int64_t)e * 2 * f * (d / 2),
                   j->w->gate_up_scale + (int64_t)e * 2 * f * ng1, j->w->gate_up_zero + (int64_t)e * 2 * f * ng1,
                   s->format, j->round_fp16, Wgu);
    dequant_matrix(d, f, s->group_down, j->w->down_q + (int64_t)e * d * (f / 2),
                   j->w->down_scale + (int64_t)e * d * ng2, j->w->down_zero + (int64_t)e * d * ng2,
                   s->format, j->round_fp16, Wd);
    for (int64_t p = 0; p < T * k; ++p) {
      if (j->topk_idx[p] != e) continue;
      int64_t t = p / k;
      if (j->token_sel && !j->token_sel[t]) continue;
      for (int64_t i = 0; i < d; ++i) xd[i] = oracle_half_to_double(j->x[t * d + i]);
      expert_ffn(s, Wgu, Wd, xd, j->round_fp16, a, h, j->ypair + p * d);
    }
  }
done:
  free(Wgu); free(Wd); free(xd); free(a); free(h);
  return NULL;
}

/* RMSNorm of one fp64 row: out_i = gamma_i * u_i / sqrt(mean(u^2) + eps). */
void oracle_rmsnorm(int64_t d, const double* u, const float* gamma, double eps, double* out) {
  double ss = 0.0;
  for (int64_t i = 0; i < d; ++i) ss += u[i] * u[i];
  double inv = 1.0 / sqrt(ss / (double)d + eps);
  for (int64_t i = 0; i < d; ++i) out[i] = (double)gamma[i] * u[i] * inv;
}

/* The layer, sparse form:  out[t] = sum_{r=0..k-1} w[t][r] * FFN_{idx[t][r]}(x[t]),
 * the sum taken over router ranks in rank order.  [MC "the kernels we built":
 * fixed-order weighted combine]  If gamma is non-NULL the combined row is
 * RMS-normalised (fp64) before it is returned.
 *   x          [T][d] fp16 bits
 *   topk_idx   [T][k], topk_w [T][k] fp64 (from oracle_route, or any weights)
 *   token_sel  [T] or NULL; tokens not selected are left untouched in out
 *   out        [T][d] fp64, unrounded
 *   nthreads   worker threads; experts are dealt to them round-robin
 *   round_fp16 diagnostic mode: dequantised weights and h rounded to fp16 */
int oracle_moe_forward(const oracle_shape* s, const uint16_t* x, const int32_t* topk_idx, const double* topk_w,
                       const oracle_weights* w, const float* gamma, double eps, const uint8_t* token_sel,
                       int nthreads, int round_fp16, double* out) {
  if (!shape_ok(s)) return ORACLE_ERR_SHAPE;
  int64_t T = s->tokens, d = s->hidden, k = s->top_k;
  if (T == 0) return ORACLE_OK;
  for (int64_t p = 0; p < T * k; ++p)
    if (topk_idx[p] < 0 || topk_idx[p] >= s->experts) return ORACLE_ERR_SHAPE;
  double* ypair = (double*)calloc((size_t)(T * k * d), sizeof(double));
  if (!ypair) return ORACLE_ERR_ALLOC;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > s->experts) nthreads = s->experts;
  expert_job* jobs = (expert_job*)calloc((size_t)nthreads, sizeof(expert_job));
  pthread_t* th = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
  if (!jobs || !th) { free(ypair); free(jobs); free(th); return ORACLE_ERR_ALLOC; }
  for (int i = 0; i < nthreads; ++i) {
    jobs[i] = (expert_job){s, w, x, topk_idx, token_sel, ypair, round_fp16, i, nthreads, ORACLE_OK};
    if (i > 0) pthread_create(&th[i], NULL, expert_worker, &jobs[i]);
  }
  expert_worker(&jobs[0]);
  int status = jobs[0].status;
  for (int i = 1; i < nthreads; ++i) {
    pthread_join(th[i], NULL);
    if (jobs[i].status != ORACLE_OK) status = jobs[i].status;
  }
  if (status == ORACLE_OK) {
    double* u = (double*)malloc(sizeof(double) * (size_t)d);
    if (!u) status = ORACLE_ERR_ALLOC;
    for (int64_t t = 0; t < T && u; ++t) {
      if (token_sel && !token_sel[t]) continue;
      for (int64_t i = 0; i < d; ++i) u[i] = 0.0;
      for (int64_t r = 0; r < k; ++r) {
        double wr = topk_w[t * k + r];
        const double* y = ypair + (t * k + r) * d;
        for (int64_t i = 0; i < d; ++i) u[i] += wr * y[i];
      }
      if (gamma) oracle_rmsnorm(d, u, gamma, eps, out + t * d);
      else memcpy(out + t * d, u, sizeof(double) * (size_t)d);
    }
    free(u);
  }
  free(ypair); free(jobs); free(th);
  return status;
}

/* The layer, dense form (a second code path used to pin the sparse one):
 *   out[t] = sum_{e=0..E-1} G[t][e] * FFN_e(x[t]),  G[t][e] = w[t][r] if
 *   idx[t][r] == e for some rank r, else 0.  Every expert runs on every token. */
int oracle_moe_forward_dense(const oracle_shape* s, const uint16_t* x, const int32_t* topk_idx,
                             const double* topk_w, const oracle_weights* w, double* out) {
  if (!shape_ok(s)) return ORACLE_ERR_SHAPE;
  int64_t T = s->tokens, d = s->hidden, f = s->inter, k = s->top_k, E = s->experts;
  int64_t ng1 = d / s->group_gate_up, ng2 = f / s->group_down;
  double* Wgu = (double*)malloc(sizeof(double) * (size_t)(2 * f * d));
  double* Wd = (double*)malloc(sizeof(double) * (size_t)(d * f));
  double* G = (double*)calloc((size_t)(T * E + 1), sizeof(double));
  double* xd = (double*)malloc(sizeof(double) * (size_t)d);
  double* a = (double*)malloc(sizeof(double) * (size_t)(2 * f));
  double* h = (double*)malloc(sizeof(double) * (size_t)f);
  double* y = (double*)malloc(sizeof(double) * (size_t)d);
  int status = ORACLE_OK;
  if (!Wgu || !Wd || !G || !xd || !a || !h || !y) { status = ORACLE_ERR_ALLOC; goto done; }
  for (int64_t t = 0; t < T; ++t)
    for (int64_t r = 0; r < k; ++r) {
      int32_t e = topk_idx[t * k + r];
      if (e < 0 || e >= E) { status = ORACLE_ERR_SHAPE; goto done; }
      G[t * E + e] = topk_w[t * k + r];
    }
  for (int64_t i = 0; i < T * d; ++i) out[i] = 0.0;
  for (int64_t e = 0; e < E; ++e) {
    dequant_matrix(2 * f, d, s->group_gate_up, w->gate_up_q + e * 2 * f * (d / 2), w->gate_up_scale + e * 2 * f * ng1,
                   w->gate_up_zero + e * 2 * f * ng1, s->format, 0, Wgu);
    dequant_matrix(d, f, s->group_down, w->down_q + e * d * (f / 2), w->down_scale + e * d * ng2,
                   w->down_zero + e * d * ng2, s->format, 0, Wd);
    for (int64_t t = 0; t < T; ++t) {
      for (int64_t i = 0; i < d; ++i) xd[i] = oracle_half_to_double(x[t * d + i]);
      expert_ffn(s, Wgu, Wd, xd, 0, a, h, y);
      for (int64_t i = 0; i < d; ++i) out[t * d + i] += G[t * E + e] * y[i];
    }
  }
done:
  free(Wgu); free(Wd); free(G); free(xd); free(a); free(h); free(y);
  return status;
}

/* ------------------------------------------------------------- MoE block ---- */

/* The block around the expert layer.  [MC] "the kernels we built": RMSNorm in one
 * launch (180 of them per forward); "what the model is": a router sends each token
 * to its top-8 of 128 experts.  The pages print no formula for the block; the
 * reading taken here (listed in the design notes) is the pre-norm residual block
 *   block(x) = x + layer(u),  u = fp16(gamma * (x * r)),  r = 1 / sqrt(ss / d + eps),
 *   ss = sum_k x_k^2,  logits[t][e] = sum_k u[t][k] * Wr[e][k]  (Wr fp16 [E][d]),
 * with the layer's fp32 output added to x before the one rounding to fp16.
 *
 * The logits decide the routing, an integer result, so ss and the logits are
 * defined in fp32 with one fixed order of operations, which the GPU reproduces
 * bit for bit: the d columns are dealt to 32 lanes in 8-column chunks (lane l
 * takes chunks l, l + 32, l + 64, ... in that order) and each lane accumulates
 * fmaf(a_k, b_k, acc) column by column from acc = 0; the 32 lane sums are then
 * combined by a butterfly: for off = 16, 8, 4, 2, 1 every lane l adds the sum of
 * lane l ^ off, and all lanes end with the same value.  d must be a multiple of
 * 256.  r, v = x_k * r and gamma_k * v are single fp32 operations (IEEE division
 * and square root), u rounds to nearest even. */

static float lane_butterfly_sum(float p[32]) {
  for (int off = 16; off >= 1; off >>= 1) {
    float q[32];
    for (int l = 0; l < 32; ++l) q[l] = p[l] + p[l ^ off];
    memcpy(p, q, sizeof(q));
  }
  return p[0];
}

static float dot_lanes(int64_t d, const float* a, const float* b) {
  float p[32];
  for (int l = 0; l < 32; ++l) {
    float acc = 0.0f;
    for (int64_t c = l; c < d / 8; c += 32)
      for (int i = 0; i < 8; ++i) acc = fmaf(a[8 * c + i], b[8 * c + i], acc);
    p[l] = acc;
  }
  return lane_butterfly_sum(p);
}

/* x fp16 bits [T][d], gamma fp32 [d], wr fp16 bits [E][d] -> u fp16 bits [T][d],
 * logits fp32 [T][E].  Non-finite inputs give ORACLE_ERR_NONFINITE. */
int oracle_block_front(int T, int d, int E, const uint16_t* x, const float* gamma, float eps, const uint16_t* wr,
                       uint16_t* u_out, float* logits) {
  if (T < 0 || d <= 0 || d % 256 != 0 || E < 1) return ORACLE_ERR_SHAPE;
  float* xf = (float*)malloc(sizeof(float) * (size_t)d);
  float* uf = (float*)malloc(sizeof(float) * (size_t)d);
  float* wf = (float*)malloc(sizeof(float) * (size_t)E * (size_t)d);
  if (!xf || !uf || !wf) {
    free(xf);
    free(uf);
    free(wf);
    return ORACLE_ERR_ALLOC;
  }
  int st = ORACLE_OK;
  for (int64_t i = 0; i < (int64_t)E * d; ++i) wf[i] = (float)oracle_half_to_double(wr[i]);
  for (int t = 0; t < T && st == ORACLE_OK; ++t) {
    for (int k = 0; k < d; ++k) {
      xf[k] = (float)oracle_half_to_double(x[(int64_t)t * d + k]);
      if (!isfinite(xf[k]) || !isfinite(gamma[k])) st = ORACLE_ERR_NONFINITE;
    }
    const float ss = dot_lanes(d, xf, xf);
    const float r = 1.0f / sqrtf(ss / (float)d + eps);
    for (int k = 0; k < d; ++k) {
      const float v = xf[k] * r;
      const float w = gamma[k] * v;
      const uint16_t h = oracle_double_to_half((double)w);
      u_out[(int64_t)t * d + k] = h;
      uf[k] = (float)oracle_half_to_double(h);
    }
    for (int e = 0; e < E; ++e) logits[(int64_t)t * E + e] = dot_lanes(d, uf, wf + (int64_t)e * d);
  }
  free(xf);
  free(uf);
  free(wf);
  return st;
}
