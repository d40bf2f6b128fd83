/*
 * sampler_oracle.c -- plain CPU oracle of the per-step sampler of a block-diffusion
 * denoising step: per canvas position the entropy of the softmax over the vocabulary,
 * one Gumbel-max sample, and the acceptance of positions.
 *
 * TEST INFRASTRUCTURE ONLY.  Like moe_oracle.c, this file defines what "correct"
 * means for the GPU library; it is linked only by the tests, the package smoke check
 * and the CPU-baseline leg of the benchmark, shares no code, header, table or helper
 * with the CUDA path, and must never be called by the product path.
 *
 * Sources (web pages; section names as printed on them):
 *   [MC]  "srswti/axe-diffusion-ksl-xe" model card, "the kernels we built": the
 *         sampler computes the entropy once per denoising step in one streaming pass
 *         over the logits and replaces softmax + multinomial with one Gumbel-max
 *         kernel; "requirements": the fp32 logits of one step are 268 MB.
 *   [ML]  "lablup/mlxcel block-diffusion docs", "Samplers": entropy-bound acceptance
 *         (positions sorted by ascending entropy, the mlx-vlm rule
 *         (cumsum - cummax) <= bound, at least one position accepted) and the
 *         confidence-threshold rule (top-1 probability above a threshold among the
 *         positions not yet revealed, else the most confident such position).
 *   Philox4x32-10: J. K. Salmon, M. A. Moraes, R. O. Dror, D. E. Shaw, "Parallel
 *         random numbers: as easy as 1, 2, 3", SC'11: the counter-based generator the
 *         Gumbel noise is drawn from (multipliers 0xD2511F53 and 0xCD9E8D57, key
 *         increments 0x9E3779B9 and 0xBB67AE85, ten rounds).
 *
 * Readings where the pages are silent (each one is listed in the design notes):
 *   - the sampled distribution is softmax(t), t_v = logit_v * inv_temp, and the
 *     entropy is that distribution's, H = -sum_v p_v ln p_v (natural log); the
 *     confidence of a position is max_v p_v;
 *   - Gumbel-max: token = argmax_v (t_v + G_v), G_v = -ln(-ln U_v), ties to the lower
 *     index; U_v = ((x & 0x7fffff) + 1/2) 2^-23 from the low 23 bits of the 32-bit
 *     word x that Philox4x32-10
 *     gives for element v: counter (v / 4, position, step, 0), key (seed low, seed
 *     high), word v % 4;
 *   - the key t_v + G_v decides an integer, so it is defined in fp32 with one IEEE
 *     rounding per operation (log_f32 below, then fmaf(logit, inv_temp, G)); any
 *     implementation that follows these steps gets the same bits;
 *   - both acceptance rules consider only positions not yet revealed; the
 *     entropy-bound rule evaluates the mlx-vlm formula elementwise in fp32 over the
 *     sorted entropies (ties: lower position first).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define SAMPLER_OK 0
#define SAMPLER_ERR_SHAPE 1
#define SAMPLER_ERR_NONFINITE 2
#define SAMPLER_ERR_ALLOC 3

/* ------------------------------------------------------------- Philox ---- */

/* Philox4x32 with ten rounds (Salmon et al., SC'11): each round multiplies words 0
 * and 2 by the two constants into 64-bit products and forms
 * (hi(M1 c2) ^ c1 ^ k0, lo(M1 c2), hi(M0 c0) ^ c3 ^ k1, lo(M0 c0)); the key grows by
 * the two Weyl increments before every round but the first. */
void oracle_philox4x32_10(const uint32_t* ctr, const uint32_t* key, uint32_t* out) {
  uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
  uint32_t k0 = key[0], k1 = key[1];
  for (int r = 0; r < 10; ++r) {
    if (r > 0) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    const uint64_t p0 = (uint64_t)0xD2511F53u * c0;
    const uint64_t p1 = (uint64_t)0xCD9E8D57u * c2;
    const uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0;
    const uint32_t n1 = (uint32_t)p1;
    const uint32_t n2 = (uint32_t)(p0 >> 32) ^ c3 ^ k1;
    const uint32_t n3 = (uint32_t)p0;
    c0 = n0;
    c1 = n1;
    c2 = n2;
    c3 = n3;
  }
  out[0] = c0;
  out[1] = c1;
  out[2] = c2;
  out[3] = c3;
}

/* --------------------------------------------------------- fp32 log ---- */

/* Natural logarithm of a positive, finite, normal fp32 value, defined as a
 * sequence of IEEE fp32 operations (this file is compiled without contraction;
 * fused steps are explicit fmaf):
 *   x = 2^e m with m in [1, 2); if m > 1.41421354 (bits 0x3fb504f3) then m = m / 2,
 *   e = e + 1 (exact);
 *   f = m - 1 (exact);  s = f / (m + 1);  z = s * s;
 *   P = ((((1/11 z + 1/9) z + 1/7) z + 1/5) z + 1/3) z + 1   (Horner, fmaf;
 *       the coefficients are the fp32 quotients 1.0f / 11.0f, ...);
 *   ln m = (2 s) P   -- the atanh series ln m = 2 atanh(s) = 2 sum s^(2j+1) / (2j+1),
 *                       |s| <= 0.1716, so the first omitted term is below 2^-26 of it;
 *   ln x = fmaf(e, LN2_HI, fmaf(e, LN2_LO, ln m)), LN2_HI = 0.693145751953125 (ln 2
 *       to 16 bits, so e LN2_HI is exact) and LN2_LO = 1.42860677e-06f (the rest). */
float oracle_log_f32(float x) {
  uint32_t b;
  memcpy(&b, &x, 4);
  int e = (int)(b >> 23) - 127;
  uint32_t mb = (b & 0x007fffffu) | 0x3f800000u;
  if (mb > 0x3fb504f3u) {
    mb -= 0x00800000u;
    e += 1;
  }
  float m;
  memcpy(&m, &mb, 4);
  const float f = m - 1.0f;
  const float s = f / (m + 1.0f);
  const float z = s * s;
  float p = 1.0f / 11.0f;
  p = fmaf(p, z, 1.0f / 9.0f);
  p = fmaf(p, z, 1.0f / 7.0f);
  p = fmaf(p, z, 1.0f / 5.0f);
  p = fmaf(p, z, 1.0f / 3.0f);
  p = fmaf(p, z, 1.0f);
  const float lnm = (2.0f * s) * p;
  const float ef = (float)e;
  return fmaf(ef, 0.693145751953125f, fmaf(ef, 1.42860677e-06f, lnm));
}

/* The Gumbel-max key of one element: U from the word's low 23 bits (exact),
 * E = -ln U, G = -ln E, key = fmaf(logit, inv_temp, G). */
float oracle_gumbel_key(float logit, float inv_temp, uint32_t word) {
  const float u = ((float)(word & 0x007fffffu) + 0.5f) * 0x1p-23f;
  const float e = -oracle_log_f32(u);
  const float g = -oracle_log_f32(e);
  return fmaf(logit, inv_temp, g);
}

/* ---------------------------------------------------------- sampling ---- */

typedef struct {
  int p0, p1;
  int64_t V;
  const float* logits;
  float inv_temp;
  uint32_t key[2];
  uint32_t step;
  int32_t* token;
  double* entropy;
  double* pmax;
} sample_job;

/* Positions [p0, p1): the fp64 entropy and top-1 probability of softmax(t), and the
 * Gumbel-max token (element by element in vocabulary order, a strictly larger key
 * replaces the best, so ties keep the lower index). */
static void* sample_worker(void* arg) {
  const sample_job* j = (const sample_job*)arg;
  for (int p = j->p0; p < j->p1; ++p) {
    const float* l = j->logits + (int64_t)p * j->V;
    double m = -INFINITY;
    for (int64_t v = 0; v < j->V; ++v) {
      const double t = (double)l[v] * (double)j->inv_temp;
      if (t > m) m = t;
    }
    double Z = 0.0, S1 = 0.0;
    for (int64_t v = 0; v < j->V; ++v) {
      const double d = (double)l[v] * (double)j->inv_temp - m;
      const double w = exp(d);
      Z += w;
      S1 += w * d;
    }
    j->entropy[p] = log(Z) - S1 / Z; /* -sum p ln p with p = e^d / Z */
    j->pmax[p] = 1.0 / Z;
    float best = -INFINITY;
    int32_t tok = 0;
    for (int64_t g = 0; g < j->V / 4; ++g) {
      const uint32_t ctr[4] = {(uint32_t)g, (uint32_t)p, j->step, 0u};
      uint32_t words[4];
      oracle_philox4x32_10(ctr, j->key, words);
      for (int i = 0; i < 4; ++i) {
        const int64_t v = 4 * g + i;
        const float k = oracle_gumbel_key(l[v], j->inv_temp, words[i]);
        if (k > best) {
          best = k;
          tok = (int32_t)v;
        }
      }
    }
    j->token[p] = tok;
  }
  return NULL;
}

/* logits fp32 [P][V] (V a multiple of 4, all finite), inv_temp > 0 and finite.
 * Outputs token [P], entropy [P] and pmax [P] (fp64). */
int oracle_sample(int P, int64_t V, const float* logits, float inv_temp, uint64_t seed, uint32_t step,
                  int nthreads, int32_t* token, double* entropy, double* pmax) {
  if (P < 1 || V < 4 || V % 4 != 0 || V > ((int64_t)1 << 32)) return SAMPLER_ERR_SHAPE;
  if (!(inv_temp > 0.0f) || !isfinite(inv_temp)) return SAMPLER_ERR_SHAPE;
  for (int64_t i = 0; i < (int64_t)P * V; ++i)
    if (!isfinite(logits[i])) return SAMPLER_ERR_NONFINITE;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > P) nthreads = P;
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
  sample_job* jobs = (sample_job*)malloc(sizeof(sample_job) * (size_t)nthreads);
  if (!th || !jobs) {
    free(th);
    free(jobs);
    return SAMPLER_ERR_ALLOC;
  }
  for (int t = 0; t < nthreads; ++t) {
    sample_job* j = &jobs[t];
    j->p0 = (int)((int64_t)P * t / nthreads);
    j->p1 = (int)((int64_t)P * (t + 1) / nthreads);
    j->V = V;
    j->logits = logits;
    j->inv_temp = inv_temp;
    j->key[0] = (uint32_t)seed;
    j->key[1] = (uint32_t)(seed >> 32);
    j->step = step;
    j->token = token;
    j->entropy = entropy;
    j->pmax = pmax;
  }
  for (int t = 1; t < nthreads; ++t) pthread_create(&th[t], NULL, sample_worker, &jobs[t]);
  sample_worker(&jobs[0]);
  for (int t = 1; t < nthreads; ++t) pthread_join(th[t], NULL);
  free(th);
  free(jobs);
  return SAMPLER_OK;
}

/* -------------------------------------------------------- acceptance ---- */

/* Entropy-bound rule ([ML] "Samplers"): the positions not yet revealed, sorted by
 * ascending entropy (ties: lower position first); with c_i the running fp32 sum of
 * the sorted entropies and x_i their running maximum, sorted position i is accepted
 * iff fl(c_i - x_i) <= bound, and the first sorted position always.  entropy holds
 * fp32 values (the precision the rule is decided in). */
typedef struct {
  float h;
  int p;
} ent_pos;

static int ent_cmp(const void* pa, const void* pb) {
  const ent_pos* a = (const ent_pos*)pa;
  const ent_pos* b = (const ent_pos*)pb;
  if (a->h < b->h) return -1;
  if (a->h > b->h) return 1;
  return (a->p > b->p) - (a->p < b->p);
}

int oracle_accept_entropy(int P, const float* entropy, const uint8_t* revealed, float bound, uint8_t* accept) {
  if (P < 1) return SAMPLER_ERR_SHAPE;
  ent_pos* s = (ent_pos*)malloc(sizeof(ent_pos) * (size_t)P);
  if (!s) return SAMPLER_ERR_ALLOC;
  int n = 0;
  for (int p = 0; p < P; ++p) {
    if (!isfinite(entropy[p])) {
      free(s);
      return SAMPLER_ERR_NONFINITE;
    }
    accept[p] = 0;
    if (!revealed[p]) {
      s[n].h = entropy[p];
      s[n].p = p;
      ++n;
    }
  }
  qsort(s, (size_t)n, sizeof(ent_pos), ent_cmp);
  float c = 0.0f, x = -INFINITY;
  for (int i = 0; i < n; ++i) {
    c = c + s[i].h;
    if (s[i].h > x) x = s[i].h;
    const float d = c - x;
    if (i == 0 || d <= bound) accept[s[i].p] = 1;
  }
  free(s);
  return SAMPLER_OK;
}

/* Confidence-threshold rule ([ML] "Samplers"): every position not yet revealed
 * whose top-1 probability exceeds the threshold; if there is none, the most
 * confident such position (ties: lower position).  pmax holds fp32 values. */
int oracle_accept_confidence(int P, const float* pmax, const uint8_t* revealed, float threshold, uint8_t* accept) {
  if (P < 1) return SAMPLER_ERR_SHAPE;
  int any = 0, best = -1;
  for (int p = 0; p < P; ++p) {
    if (!isfinite(pmax[p])) return SAMPLER_ERR_NONFINITE;
    accept[p] = 0;
    if (revealed[p]) continue;
    if (pmax[p] > threshold) {
      accept[p] = 1;
      any = 1;
    }
    if (best < 0 || pmax[p] > pmax[best]) best = p;
  }
  if (!any && best >= 0) accept[best] = 1;
  return SAMPLER_OK;
}
