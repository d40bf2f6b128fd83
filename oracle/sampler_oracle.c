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
 *   - Gumbel-max, two forms selected by `noise` (both sample softmax(t) exactly in
 *     real arithmetic; [MC] fixes the distribution and the Gumbel-max method, not how
 *     the noise is laid over the vocabulary):
 *     noise 1 (one Gumbel per token): token = argmax_v (t_v + G_v), G_v = -ln(-ln U_v),
 *       ties to the lower index; U_v = ((x & 0x7fffff) + 1/2) 2^-23 from the low 23
 *       bits of the 32-bit word x that Philox4x32-10 gives for element v: counter
 *       (v / 4, position, step, 0), key (seed low, seed high), word v % 4;
 *     noise 0 (one Gumbel per group of four, the default): the vocabulary is cut into
 *       groups g of four consecutive entries (4g .. 4g+3).  The largest of four
 *       independent Gumbel keys t_i + G_i is itself Gumbel-distributed around
 *       LSE_g = ln sum_i e^(t_i), and which of the four attains it is independent of
 *       that value and distributed as softmax over the group (the max-stability of the
 *       Gumbel law, the top-down construction of a Gumbel process).  So the group's
 *       key is LSE_g + G_g with one Gumbel G_g, the token's group is the argmax of
 *       the group keys (ties to the lower group), and the token inside it is drawn by
 *       inverse CDF from a second uniform U'_g: the first i whose running sum of
 *       e^(t_i - m) exceeds U'_g times the group's sum.  U_g comes from Philox word
 *       r / 256 of counter (256 (g / 1024) + r % 256, position, step, 0), r = g % 1024
 *       (the 1,024 groups of each 4,096-entry block share 256 counters), and U'_g from
 *       the same word of the counter with fourth word 1.  This mapping was chosen to
 *       suit the GPU pass, whose threads own float4s 256 apart; any bijection would do;
 *   - each key decides an integer, so it is defined in fp32 with one IEEE rounding per
 *     operation (log_f32 and exp_f32 below; the per-token key is
 *     fmaf(logit, inv_temp, G), the group key fl(fl(m + ln S) + G) with
 *     t_i = fl(l_i inv_temp), m = max t_i, S = ((e_0 + e_1) + e_2) + e_3,
 *     e_i = exp_f32(fl(t_i - m))); any implementation that follows these steps gets
 *     the same bits;
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

/* --------------------------------------------------------- fp32 exp ---- */

/* e^x for x <= 0, defined as a sequence of IEEE fp32 operations:
 *   below -87 (where 2^n would leave the normal range) the result is 0;
 *   n = rint(fl(x * LOG2E)), LOG2E = fp32 log2(e) = 0x1.715476p+0;
 *   r = fmaf(-n, LN2_LO, fmaf(-n, LN2_HI, x))  (the split of ln 2 used by log_f32);
 *   P = 1 + r(1 + r(1/2 + r(1/6 + r(1/24 + r(1/120 + r(1/720 + r/5040))))))
 *       (the Taylor series of e^r to r^7, Horner with fmaf, coefficients the fp32
 *       quotients 1.0f / 5040.0f, ...; |r| <= 0.35, so the first omitted term is below
 *       2^-27 of the result);
 *   e^x = fl(P * 2^n), 2^n built from its exponent bits. */
float oracle_exp_f32(float x) {
  if (!(x >= -87.0f)) return 0.0f;
  const float n = rintf(x * 0x1.715476p+0f);
  float r = fmaf(-n, 0.693145751953125f, x);
  r = fmaf(-n, 1.42860677e-06f, r);
  float p = 1.0f / 5040.0f;
  p = fmaf(p, r, 1.0f / 720.0f);
  p = fmaf(p, r, 1.0f / 120.0f);
  p = fmaf(p, r, 1.0f / 24.0f);
  p = fmaf(p, r, 1.0f / 6.0f);
  p = fmaf(p, r, 0.5f);
  p = fmaf(p, r, 1.0f);
  p = fmaf(p, r, 1.0f);
  const uint32_t sb = (uint32_t)((int)n + 127) << 23;
  float sc;
  memcpy(&sc, &sb, 4);
  return p * sc;
}

/* ------------------------------------------------- groups of four ---- */

/* The Philox counter (first word) and the word index of group g. */
uint32_t oracle_group_counter(uint32_t g) { return ((g >> 10) << 8) | (g & 255u); }
int oracle_group_word(uint32_t g) { return (int)((g >> 8) & 3u); }

/* t_i = fl(l_i inv_temp), m = max t_i, e_i = exp_f32(fl(t_i - m)), S = ((e_0 + e_1) + e_2) + e_3. */
static float group_exp(const float* l, float inv_temp, float* e) {
  float t[4];
  for (int i = 0; i < 4; ++i) t[i] = l[i] * inv_temp;
  const float m = fmaxf(fmaxf(t[0], t[1]), fmaxf(t[2], t[3]));
  for (int i = 0; i < 4; ++i) e[i] = oracle_exp_f32(t[i] - m);
  return m;
}

/* The key of a group of four logits: LSE = fl(m + ln S), G = -ln(-ln U) from the
 * word's low 23 bits, key = fl(LSE + G). */
float oracle_group_key(const float* l, float inv_temp, uint32_t word) {
  float e[4];
  const float m = group_exp(l, inv_temp, e);
  const float S = ((e[0] + e[1]) + e[2]) + e[3];
  const float lse = m + oracle_log_f32(S);
  const float u = ((float)(word & 0x007fffffu) + 0.5f) * 0x1p-23f;
  const float g = -oracle_log_f32(-oracle_log_f32(u));
  return lse + g;
}

/* The token inside a group (0 .. 3) by inverse CDF: U' from the word's low 23 bits,
 * T = fl(U' S); the first i with fl(..fl(e_0 + e_1).. + e_i) > T; if none (T rounded up
 * to S), the last i with e_i > 0. */
int oracle_group_pick(const float* l, float inv_temp, uint32_t word) {
  float e[4];
  group_exp(l, inv_temp, e);
  const float S = ((e[0] + e[1]) + e[2]) + e[3];
  const float u = ((float)(word & 0x007fffffu) + 0.5f) * 0x1p-23f;
  const float T = u * S;
  float c = 0.0f;
  for (int i = 0; i < 4; ++i) {
    c = i == 0 ? e[0] : c + e[i];
    if (c > T) return i;
  }
  int last = 0;
  for (int i = 0; i < 4; ++i)
    if (e[i] > 0.0f) last = i;
  return last;
}

/* ---------------------------------------------------------- sampling ---- */

typedef struct {
  int p0, p1;
  int64_t V;
  const float* logits;
  float inv_temp;
  uint32_t key[2];
  uint32_t step;
  int noise;
  int32_t* token;
  double* entropy;
  double* pmax;
} sample_job;

/* Positions [p0, p1): the fp64 entropy and top-1 probability of softmax(t), and the
 * Gumbel-max token (keys in vocabulary order, per token or per group; a strictly larger
 * key replaces the best, so ties keep the lower index). */
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
    if (j->noise == 1) {
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
    } else {
      uint32_t bg = 0;
      for (int64_t g = 0; g < j->V / 4; ++g) {
        const uint32_t ctr[4] = {oracle_group_counter((uint32_t)g), (uint32_t)p, j->step, 0u};
        uint32_t words[4];
        oracle_philox4x32_10(ctr, j->key, words);
        const float k = oracle_group_key(l + 4 * g, j->inv_temp, words[oracle_group_word((uint32_t)g)]);
        if (k > best) {
          best = k;
          bg = (uint32_t)g;
        }
      }
      const uint32_t ctr[4] = {oracle_group_counter(bg), (uint32_t)p, j->step, 1u};
      uint32_t words[4];
      oracle_philox4x32_10(ctr, j->key, words);
      tok = (int32_t)(4 * bg) + oracle_group_pick(l + 4 * (int64_t)bg, j->inv_temp, words[oracle_group_word(bg)]);
    }
    j->token[p] = tok;
  }
  return NULL;
}

/* logits fp32 [P][V] (V a multiple of 4, all finite), inv_temp > 0 and finite,
 * noise 0 (one Gumbel per group of four) or 1 (one per token).
 * Outputs token [P], entropy [P] and pmax [P] (fp64). */
int oracle_sample(int P, int64_t V, const float* logits, float inv_temp, uint64_t seed, uint32_t step,
                  int noise, int nthreads, int32_t* token, double* entropy, double* pmax) {
  if (P < 1 || V < 4 || V % 4 != 0 || V > ((int64_t)1 << 32)) return SAMPLER_ERR_SHAPE;
  if (noise != 0 && noise != 1) return SAMPLER_ERR_SHAPE;
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
    j->noise = noise;
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
