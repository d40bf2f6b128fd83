// sampler.cu -- the per-step sampler of a denoising step: per canvas position
// the entropy of softmax(logits * inv_temp), one Gumbel-max token and the
// top-1 probability, in one streaming pass over the fp32 logits; then the
// acceptance of positions.
//
// Model card "srswti/axe-diffusion-ksl-xe", "the kernels we built": the entropy
// is computed once per denoising step in a single streaming pass, and one
// Gumbel-max kernel replaces softmax + multinomial ("requirements": the logits of
// a step are 268 MB of fp32).  "lablup/mlxcel block-diffusion docs", "Samplers":
// entropy-bound acceptance (positions by ascending entropy, the mlx-vlm rule
// (cumsum - cummax) <= bound, at least one) or confidence-threshold acceptance.
//
// Gumbel-max, two forms (both sample softmax(t), t_v = logit_v * inv_temp):
//   noise 1, one Gumbel per token: token = argmax_v (t_v + G_v), G_v = -ln(-ln U_v),
//     U_v = ((x & 0x7fffff) + 1/2) 2^-23 from word v % 4 of Philox4x32-10 (Salmon et al.,
//     SC'11) at counter (v / 4, position, step, 0) under key (seed low, seed high); ties to
//     the lower index; key = fma(logit, inv_temp, G).
//   noise 0, one Gumbel per group of four entries (the default): the largest of four
//     independent Gumbel keys is Gumbel around the group's log-sum-exp, and where it
//     falls is softmax within the group (max-stability of the Gumbel law), so group
//     g = entries 4g .. 4g+3 gets the key LSE_g + G_g, the winning group is the argmax
//     (ties to the lower group) and the token inside it is drawn by inverse CDF from a
//     second uniform.  U_g is word r / 256 of counter (256 (g / 1024) + r % 256,
//     position, step, 0), r = g % 1024, so that one Philox call serves the four groups a
//     thread holds (float4s 256 apart); U'_g the same word with fourth counter word 1.
// Every key decides an integer, so it is computed with one IEEE fp32 rounding per
// operation (ln_f32 and exp_f32 below): any implementation that takes these steps gets
// the same token.
//
// Pass kernel (grid: vocabulary splits x positions, 256 threads): each thread
// streams float4s of its position's logits and keeps, in base 2, the running
// maximum m2 of t2 = t log2(e), Z = sum 2^(t2 - m2) and S1 = sum 2^(t2 - m2)(t2 - m2).
// Exact keys cost logarithms (and, per group, four exponentials), so a cheap
// necessary condition screens them: with K the best exact key the CTA has found so
// far, a token (group) can reach K only if w = 1 - U <= e^(t - K) (the group's sum of
// e^(t_i - K)), because -ln U >= 1 - U and G = -ln(-ln U); the test is made with a
// margin that covers every rounding involved (fast exponentials included) and reuses
// 2^(t2 - m2) of the softmax sum; only the few that pass get their exact key.  Per
// token, an element costs one Philox quarter, one exp2 and about eight other
// instructions; per group, a Philox call serves sixteen elements and the screen runs
// once per four, so the pass streams at memory speed.  Loads are streaming 16-byte
// loads into registers, issued one to two iterations ahead; nothing waits on shared
// memory or a barrier.  Per group, the CTA reduction carries the best group's four
// logits and thread 0 draws the token inside it (inverse CDF); each CTA writes its
// partial (m2, Z, S1, best key, token).
//
// Final kernel (one CTA, one thread per position): merges each position's
// partials in split order, writes entropy H = ln Z - (S1 / Z) ln 2, top-1
// probability 1 / Z and the token, then applies the acceptance rule to those fp32
// values (entropy rule: a bitonic sort by (H, position), then one thread runs the
// fp32 cumulative sum in sorted order and every thread decides its own entry).
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kPassThreads = 256;
constexpr int kFinalThreads = 1024;  // positions per call at most

struct __align__(16) Partial {
  float m2, z, s1, key;
  int32_t v;
  int32_t pad[3];
};

// Round keys of Philox4x32-10: round r uses (k0 + r 0x9E3779B9, k1 + r 0xBB67AE85).
struct PhiloxKeys {
  uint32_t k0[10], k1[10];
};
__device__ __forceinline__ PhiloxKeys philox_keys(uint32_t k0, uint32_t k1) {
  PhiloxKeys k;
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    k.k0[r] = k0 + static_cast<uint32_t>(r) * 0x9E3779B9u;
    k.k1[r] = k1 + static_cast<uint32_t>(r) * 0xBB67AE85u;
  }
  return k;
}

__device__ __forceinline__ void philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                              const PhiloxKeys& k, uint32_t (&o)[4]) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    // the two 32 x 32 -> 64-bit products of the round, each one wide multiply
    uint32_t h0, l0, h1, l1;
    asm("{\n .reg .u64 t;\n mul.wide.u32 t, %2, %3;\n mov.b64 {%0, %1}, t;\n}" : "=r"(l0), "=r"(h0)
        : "r"(0xD2511F53u), "r"(c0));
    asm("{\n .reg .u64 t;\n mul.wide.u32 t, %2, %3;\n mov.b64 {%0, %1}, t;\n}" : "=r"(l1), "=r"(h1)
        : "r"(0xCD9E8D57u), "r"(c2));
    const uint32_t n0 = h1 ^ c1 ^ k.k0[r];
    const uint32_t n2 = h0 ^ c3 ^ k.k1[r];
    c1 = l1;
    c3 = l0;
    c0 = n0;
    c2 = n2;
  }
  o[0] = c0;
  o[1] = c1;
  o[2] = c2;
  o[3] = c3;
}

// Natural log of a positive normal fp32 value as a fixed sequence of IEEE fp32
// operations: x = 2^e m, m in [1, 2), halved (e + 1) when above 0x3fb504f3;
// s = (m - 1) / (m + 1); ln m = 2 s (1 + z/3 + z^2/5 + z^3/7 + z^4/9 + z^5/11), z = s^2
// (the atanh series, Horner with fused multiply-adds, coefficients the fp32
// quotients 1/3 ... 1/11); ln x = e ln2_hi + (e ln2_lo + ln m) with ln2_hi = ln 2 to
// 16 bits (e ln2_hi exact).  Explicit _rn intrinsics: nothing is contracted or
// approximated, so the result is the same on any IEEE machine that takes the steps.
__device__ __forceinline__ float ln_f32(float x) {
  const uint32_t b = __float_as_uint(x);
  int e = static_cast<int>(b >> 23) - 127;
  uint32_t mb = (b & 0x007fffffu) | 0x3f800000u;
  if (mb > 0x3fb504f3u) {
    mb -= 0x00800000u;
    e += 1;
  }
  const float m = __uint_as_float(mb);
  const float f = __fadd_rn(m, -1.0f);
  const float s = __fdiv_rn(f, __fadd_rn(m, 1.0f));
  const float z = __fmul_rn(s, s);
  float p = 0x1.745d18p-4f;              // 1/11
  p = __fmaf_rn(p, z, 0x1.c71c72p-4f);   // 1/9
  p = __fmaf_rn(p, z, 0x1.24924ap-3f);   // 1/7
  p = __fmaf_rn(p, z, 0x1.99999ap-3f);   // 1/5
  p = __fmaf_rn(p, z, 0x1.555556p-2f);   // 1/3
  p = __fmaf_rn(p, z, 1.0f);
  const float lnm = __fmul_rn(__fmul_rn(2.0f, s), p);
  const float ef = static_cast<float>(e);
  return __fmaf_rn(ef, 0x1.62e4p-1f, __fmaf_rn(ef, 0x1.7f7d1cp-20f, lnm));
}

__device__ __forceinline__ float gumbel_key(float logit, float inv_temp, uint32_t word) {
  const float u = __fmul_rn(__fadd_rn(static_cast<float>(word & 0x007fffffu), 0.5f), 0x1p-23f);
  const float e = -ln_f32(u);
  const float g = -ln_f32(e);
  return __fmaf_rn(logit, inv_temp, g);
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Order-preserving encoding of fp32 keys as unsigned integers (for atomicMax).
__device__ __forceinline__ uint32_t key_enc(float k) {
  const uint32_t b = __float_as_uint(k);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_dec(uint32_t u) {
  return __uint_as_float((u & 0x80000000u) ? (u & 0x7fffffffu) : ~u);
}

// (key, index) order of the token choice: larger key, then lower index.
__device__ __forceinline__ bool better(float k, int32_t v, float bk, int32_t bv) {
  return k > bk || (k == bk && v < bv);
}

// Merge of two partial softmax sums in base 2 (empty sums have z == 0).
__device__ __forceinline__ void merge_sums(float& m2, float& z, float& s1, float om2, float oz, float os1) {
  if (oz == 0.f) return;
  if (z == 0.f) {
    m2 = om2;
    z = oz;
    s1 = os1;
    return;
  }
  const float m = fmaxf(m2, om2);
  const float da = m2 - m, db = om2 - m;
  const float ra = exp2f(da), rb = exp2f(db);
  s1 = ra * fmaf(da, z, s1) + rb * fmaf(db, oz, os1);
  z = ra * z + rb * oz;
  m2 = m;
}

// e^x for x <= 0 as a fixed sequence of IEEE fp32 operations: n = rint(x log2 e),
// r = (x - n ln2_hi) - n ln2_lo (ln2_hi = ln 2 to 16 bits, so n ln2_hi is exact),
// e^r by its Taylor series to r^7 (Horner with fused multiply-adds, coefficients
// the fp32 quotients 1/5040 ... 1/2), times 2^n built from exponent bits.  Below
// -87 the result is defined as 0 (2^n would leave the normal range).
__device__ __forceinline__ float exp_f32(float x) {
  if (!(x >= -87.f)) return 0.f;
  const float n = rintf(__fmul_rn(x, 0x1.715476p+0f));
  float r = __fmaf_rn(-n, 0x1.62e4p-1f, x);
  r = __fmaf_rn(-n, 0x1.7f7d1cp-20f, r);
  float p = 0x1.a01a02p-13f;             // 1/5040
  p = __fmaf_rn(p, r, 0x1.6c16c2p-10f);  // 1/720
  p = __fmaf_rn(p, r, 0x1.111112p-7f);   // 1/120
  p = __fmaf_rn(p, r, 0x1.555556p-5f);   // 1/24
  p = __fmaf_rn(p, r, 0x1.555556p-3f);   // 1/6
  p = __fmaf_rn(p, r, 0.5f);
  p = __fmaf_rn(p, r, 1.0f);
  p = __fmaf_rn(p, r, 1.0f);
  return __fmul_rn(p, __uint_as_float(static_cast<uint32_t>(static_cast<int>(n) + 127) << 23));
}

// A group of four logits (one float4, vocabulary entries 4g .. 4g+3) in fp32 operations:
// t_i = fl(l_i inv_temp), m = max t_i, e_i = e^(t_i - m) (exp_f32), S = ((e_0 + e_1) + e_2) + e_3.
struct GroupExp {
  float m, e[4], s;
};
__device__ __forceinline__ GroupExp group_exp(float4 l, float inv_temp) {
  GroupExp g;
  const float t[4] = {__fmul_rn(l.x, inv_temp), __fmul_rn(l.y, inv_temp), __fmul_rn(l.z, inv_temp),
                      __fmul_rn(l.w, inv_temp)};
  g.m = fmaxf(fmaxf(t[0], t[1]), fmaxf(t[2], t[3]));
#pragma unroll
  for (int i = 0; i < 4; ++i) g.e[i] = exp_f32(__fsub_rn(t[i], g.m));
  g.s = __fadd_rn(__fadd_rn(__fadd_rn(g.e[0], g.e[1]), g.e[2]), g.e[3]);
  return g;
}

// Exact key of a group: fl(fl(m + ln S) + G), G = -ln(-ln U) of its Philox word.
__device__ __forceinline__ float group_key(float4 l, float inv_temp, uint32_t word) {
  const GroupExp g = group_exp(l, inv_temp);
  const float u = __fmul_rn(__fadd_rn(static_cast<float>(word & 0x007fffffu), 0.5f), 0x1p-23f);
  const float gum = -ln_f32(-ln_f32(u));
  return __fadd_rn(__fadd_rn(g.m, ln_f32(g.s)), gum);
}

// The token inside a group (0 .. 3) by inverse CDF: T = fl(U' S) with U' from the
// word, the first i whose running sum fl(..fl(e_0 + e_1).. + e_i) exceeds T; if none
// does (T rounded up to S), the last i with e_i > 0.
__device__ __forceinline__ int group_pick(float4 l, float inv_temp, uint32_t word) {
  const GroupExp ge = group_exp(l, inv_temp);
  const float u = __fmul_rn(__fadd_rn(static_cast<float>(word & 0x007fffffu), 0.5f), 0x1p-23f);
  const float T = __fmul_rn(u, ge.s);
  int pick = -1, last = 0;
  float c = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    c = i == 0 ? ge.e[0] : __fadd_rn(c, ge.e[i]);
    if (pick < 0 && c > T) pick = i;
    if (ge.e[i] > 0.f) last = i;
  }
  return pick < 0 ? last : pick;
}

// Philox counter word 0 of group g (float4 index in the position's row): the groups of
// each 4,096-entry block share 256 counters, group r of the block taking word r / 256
// of counter 256 * block + r % 256.
__device__ __forceinline__ uint32_t group_counter(uint32_t g) { return ((g >> 10) << 8) | (g & 255u); }
__device__ __forceinline__ int group_word(uint32_t g) { return static_cast<int>((g >> 8) & 3u); }

// Running state of one pass thread.
struct PassState {
  float m2, z, s1;     // base-2 online softmax sums
  float bk;            // best exact key so far, and its token (per group: its group)
  int32_t bv;
  float c2, c_K, c_m2;  // screening factor and the (K, m2) it was made for
  float4 bl;            // per group: the best group's four logits
};

// Eight elements of one thread: float4s j and j + 256 of the CTA's range (ids
// v0 + 4 j ...).  With kGuard, float4s at or past n4 take no part (the last
// iteration of a range that is not a multiple of 512 float4s).
template <bool kGuard>
__device__ __forceinline__ void pass_iter(PassState& S, const float4 (&x)[2], int j, int n4, int64_t v0, uint32_t g0,
                                          uint32_t p, uint32_t step, const PhiloxKeys& pk, float c2e, float inv_temp,
                                          volatile uint32_t* vbest, uint32_t* cta_best) {
  uint32_t w[2][4];
  philox4x32_10(g0 + static_cast<uint32_t>(j), p, step, 0u, pk, w[0]);
  philox4x32_10(g0 + static_cast<uint32_t>(j + kPassThreads), p, step, 0u, pk, w[1]);
  const bool act[2] = {!kGuard || j < n4, !kGuard || j + kPassThreads < n4};
  const float l[8] = {x[0].x, x[0].y, x[0].z, x[0].w, x[1].x, x[1].y, x[1].z, x[1].w};
  float mx;
  if (kGuard) {
    mx = -INFINITY;
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (act[i / 4]) mx = fmaxf(mx, l[i]);
  } else {
    mx = fmaxf(fmaxf(fmaxf(l[0], l[1]), fmaxf(l[2], l[3])), fmaxf(fmaxf(l[4], l[5]), fmaxf(l[6], l[7])));
  }
  mx *= c2e;
  if (mx > S.m2) {
    if (S.z != 0.f) {
      const float dm = S.m2 - mx;
      const float r = fast_exp2(dm);
      S.s1 = r * fmaf(dm, S.z, S.s1);
      S.z *= r;
    }
    S.m2 = mx;
  }
  // screen: element v needs w_v <= 2^(t2_v - K2 + slack) = 2^(t2_v - m2) c2 with
  // c2 = 2^(m2 - K2 + slack); the slack (base-2 units) and the factor 1.01 cover
  // the roundings of t2, K2 and the approximate exp2.  Before the CTA has a key,
  // c2 is huge: every element whose 2^(t2 - m2) does not underflow is screened in
  // (one that underflows cannot beat its thread's own maximum, which is screened in)
  const float K = key_dec(*vbest);
  if (K != S.c_K || S.m2 != S.c_m2) {
    S.c_K = K;
    S.c_m2 = S.m2;
    S.c2 = 3e38f;
    if (K != -INFINITY) {
      const float K2 = K * 1.44269504088896341f;
      const float slack = 0x1p-8f + (fabsf(S.m2) + fabsf(K2)) * 0x1p-14f;
      S.c2 = fminf(fast_exp2(S.m2 - K2 + slack) * 1.01f, 3e38f);
    }
  }
  // the largest f + e c2 of the eight: element i is screened in iff its own value is at
  // least 2 - 2^-23 (implied by w <= e c2, since fl(2 - 2^-24) = 2)
  float qmax = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    if (!act[i / 4]) continue;
    const float d = fmaf(l[i], c2e, -S.m2);
    const float e = fast_exp2(d);
    S.z += e;
    S.s1 = fmaf(e, d, S.s1);
    const float f = __uint_as_float(0x3f800000u | (w[i / 4][i % 4] & 0x007fffffu));
    qmax = fmaxf(qmax, fmaf(e, S.c2, f));
  }
  const bool any = qmax >= 0x1.fffffep+0f;
  if (__any_sync(0xffffffffu, any)) {
    if (any) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if (!act[i / 4]) continue;
        const float e = fast_exp2(fmaf(l[i], c2e, -S.m2));
        const float f = __uint_as_float(0x3f800000u | (w[i / 4][i % 4] & 0x007fffffu));
        if (!(fmaf(e, S.c2, f) >= 0x1.fffffep+0f)) continue;
        const float k = gumbel_key(l[i], inv_temp, w[i / 4][i % 4]);
        const int32_t v = static_cast<int32_t>(v0 + 4 * static_cast<int64_t>(j + (i / 4) * kPassThreads) + i % 4);
        if (better(k, v, S.bk, S.bv)) {
          S.bk = k;
          S.bv = v;
        }
      }
      atomicMax(cta_best, key_enc(S.bk));
    }
  }
}

// Sixteen logits of one thread: float4s j + 256 q (q = 0..3) of a 4,096-entry block, the
// four groups of Philox counter cnt (group q takes word q).  With kGuard, float4s at or
// past n4 take no part (the range's last, partial block).
template <bool kGuard>
__device__ __forceinline__ void pass_block(PassState& S, const float4 (&x)[4], int j, int n4, uint32_t gbase,
                                           uint32_t cnt, uint32_t p, uint32_t step, const PhiloxKeys& pk, float c2e,
                                           float inv_temp, volatile uint32_t* vbest, uint32_t* cta_best) {
  uint32_t w[4];
  philox4x32_10(cnt, p, step, 0u, pk, w);
  bool act[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) act[q] = !kGuard || j + q * kPassThreads < n4;
  float mx = -INFINITY;
#pragma unroll
  for (int q = 0; q < 4; ++q)
    if (act[q]) mx = fmaxf(mx, fmaxf(fmaxf(x[q].x, x[q].y), fmaxf(x[q].z, x[q].w)));
  mx *= c2e;
  if (mx > S.m2) {
    if (S.z != 0.f) {
      const float dm = S.m2 - mx;
      const float r = fast_exp2(dm);
      S.s1 = r * fmaf(dm, S.z, S.s1);
      S.z *= r;
    }
    S.m2 = mx;
  }
  // screen: group g can reach the best key K only if w_g = 1 - U_g <= sum_i e^(t_i - K)
  // (its key is ln sum_i e^(t_i) - ln(-ln U_g) and -ln U >= 1 - U), tested as
  // w_g <= zg c2 with zg = sum_i 2^(t2_i - m2) and c2 = 2^(m2 - K2 + slack) 1.01; the slack
  // covers the roundings of t2, K2, the group's exact sum and logarithm, and the fast exp2
  const float K = key_dec(*vbest);
  if (K != S.c_K || S.m2 != S.c_m2) {
    S.c_K = K;
    S.c_m2 = S.m2;
    S.c2 = 3e38f;
    if (K != -INFINITY) {
      const float K2 = K * 1.44269504088896341f;
      const float slack = 0x1p-8f + (fabsf(S.m2) + fabsf(K2)) * 0x1p-14f;
      S.c2 = fminf(fast_exp2(S.m2 - K2 + slack) * 1.01f, 3e38f);
    }
  }
  // f_g + zg c2 >= 2 - 2^-23 with f_g = 1 + (x & 0x7fffff) 2^-23 is implied by w_g <= zg c2
  float qmax = 0.f;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    if (!act[q]) continue;
    const float l[4] = {x[q].x, x[q].y, x[q].z, x[q].w};
    float e[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float d = fmaf(l[i], c2e, -S.m2);
      e[i] = fast_exp2(d);
      S.s1 = fmaf(e[i], d, S.s1);
    }
    const float zg = (e[0] + e[1]) + (e[2] + e[3]);
    S.z += zg;
    const float f = __uint_as_float(0x3f800000u | (w[q] & 0x007fffffu));
    qmax = fmaxf(qmax, fmaf(zg, S.c2, f));
  }
  const bool any = qmax >= 0x1.fffffep+0f;
  if (__any_sync(0xffffffffu, any)) {
    if (any) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        if (!act[q]) continue;
        const float l[4] = {x[q].x, x[q].y, x[q].z, x[q].w};
        float zg = 0.f;
        {
          float e[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) e[i] = fast_exp2(fmaf(l[i], c2e, -S.m2));
          zg = (e[0] + e[1]) + (e[2] + e[3]);
        }
        const float f = __uint_as_float(0x3f800000u | (w[q] & 0x007fffffu));
        if (!(fmaf(zg, S.c2, f) >= 0x1.fffffep+0f)) continue;
        const float k = group_key(x[q], inv_temp, w[q]);
        const int32_t g = static_cast<int32_t>(gbase + static_cast<uint32_t>(j + q * kPassThreads));
        if (better(k, g, S.bk, S.bv)) {
          S.bk = k;
          S.bv = g;
          S.bl = x[q];
        }
      }
      atomicMax(cta_best, key_enc(S.bk));
    }
  }
}

// The per-token pass over float4s [0, n4) of the CTA's range: iteration it covers
// float4s it * 512 + tid and + 256; the loads run two iterations ahead over three
// register buffers, streaming (evict-first), from addresses clamped into the range
// (a load past its end is never used).
__device__ __forceinline__ void run_tokens(PassState& S, const float4* src, int n4, int64_t v0, uint32_t p,
                                           uint32_t step, const PhiloxKeys& pk, float c2e, float inv_temp,
                                           uint32_t* cta_best) {
  const int tid = threadIdx.x;
  const uint32_t g0 = static_cast<uint32_t>(v0 / 4);
  constexpr int kStep = 2 * kPassThreads;
  const int n_full = n4 / kStep, n_iter = (n4 + kStep - 1) / kStep;
  const int last4 = max(n4 - 1, 0);
  auto load = [&](int j) { return __ldcs(src + min(j, last4)); };
  float4 cur[2] = {load(tid), load(tid + kPassThreads)};
  float4 nxt[2] = {load(kStep + tid), load(kStep + tid + kPassThreads)};
  {
    // a first threshold for the screen: the exact key of each thread's largest logit
    // among its first eight (any element's exact key is a valid threshold; without
    // one, every element of the first iteration would need its exact key)
    const float l[8] = {cur[0].x, cur[0].y, cur[0].z, cur[0].w, cur[1].x, cur[1].y, cur[1].z, cur[1].w};
    int ib = -1;
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (tid + (i / 4) * kPassThreads < n4 && (ib < 0 || l[i] > l[ib])) ib = i;
    if (ib >= 0) {
      const int j = tid + (ib / 4) * kPassThreads;
      uint32_t w[4];
      philox4x32_10(g0 + static_cast<uint32_t>(j), p, step, 0u, pk, w);
      const float lmax = ib == 0 ? l[0] : ib == 1 ? l[1] : ib == 2 ? l[2] : ib == 3 ? l[3]
                       : ib == 4 ? l[4] : ib == 5 ? l[5] : ib == 6 ? l[6] : l[7];
      const uint32_t wb = (ib & 3) == 0 ? w[0] : (ib & 3) == 1 ? w[1] : (ib & 3) == 2 ? w[2] : w[3];
      S.bk = gumbel_key(lmax, inv_temp, wb);
      S.bv = static_cast<int32_t>(v0 + 4 * static_cast<int64_t>(j) + (ib & 3));
      atomicMax(cta_best, key_enc(S.bk));
    }
    __syncthreads();
  }
  int it = 0;
  // three iterations per trip over three buffers in turn (cur, nxt, third), each refilled two
  // iterations ahead, so that no float4 is moved between registers
  float4 third[2];
  for (; it + 3 <= n_full; it += 3) {  // uniform trip count
    const int j = it * kStep + tid;
    third[0] = load(j + 2 * kStep);
    third[1] = load(j + 2 * kStep + kPassThreads);
    pass_iter<false>(S, cur, j, n4, v0, g0, p, step, pk, c2e, inv_temp, cta_best, cta_best);
    cur[0] = load(j + 3 * kStep);
    cur[1] = load(j + 3 * kStep + kPassThreads);
    pass_iter<false>(S, nxt, j + kStep, n4, v0, g0, p, step, pk, c2e, inv_temp, cta_best, cta_best);
    nxt[0] = load(j + 4 * kStep);
    nxt[1] = load(j + 4 * kStep + kPassThreads);
    pass_iter<false>(S, third, j + 2 * kStep, n4, v0, g0, p, step, pk, c2e, inv_temp, cta_best, cta_best);
  }
  for (; it < n_full; ++it) {  // the last full iterations, one at a time
    const int j = it * kStep + tid;
    const float4 pf0 = load(j + 2 * kStep), pf1 = load(j + 2 * kStep + kPassThreads);
    pass_iter<false>(S, cur, j, n4, v0, g0, p, step, pk, c2e, inv_temp, cta_best, cta_best);
    cur[0] = nxt[0];
    cur[1] = nxt[1];
    nxt[0] = pf0;
    nxt[1] = pf1;
  }
  if (it < n_iter)  // the range's last, partial iteration
    pass_iter<true>(S, cur, it * kStep + tid, n4, v0, g0, p, step, pk, c2e, inv_temp, cta_best, cta_best);
}

// The per-group pass over float4s [0, n4) of the CTA's range (v0 a multiple of 4,096):
// block b covers float4s b * 1024 + tid + 256 q (q = 0..3), the four groups of one
// Philox counter; the loads run one block ahead over two register buffers.
__device__ __forceinline__ void run_groups(PassState& S, const float4* src, int n4, int64_t v0, uint32_t p,
                                           uint32_t step, const PhiloxKeys& pk, float c2e, float inv_temp,
                                           uint32_t* cta_best) {
  const int tid = threadIdx.x;
  const uint32_t gbase = static_cast<uint32_t>(v0 / 4);
  const uint32_t cnt0 = ((gbase >> 10) << 8) | static_cast<uint32_t>(tid);  // counter of the thread's first block
  constexpr int kBlk = 4 * kPassThreads;
  const int n_full = n4 / kBlk, n_blk = (n4 + kBlk - 1) / kBlk;
  const int last4 = max(n4 - 1, 0);
  auto load = [&](int j) { return __ldcs(src + min(j, last4)); };
  float4 A[4], B[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) A[q] = load(tid + q * kPassThreads);
#pragma unroll
  for (int q = 0; q < 4; ++q) B[q] = load(kBlk + tid + q * kPassThreads);
  {
    // a first threshold for the screen: the exact key of the thread's first group with
    // the largest logit (any group's exact key is a valid threshold)
    int qb = -1;
    float lb = -INFINITY;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float mq = fmaxf(fmaxf(A[q].x, A[q].y), fmaxf(A[q].z, A[q].w));
      if (tid + q * kPassThreads < n4 && (qb < 0 || mq > lb)) {
        qb = q;
        lb = mq;
      }
    }
    if (qb >= 0) {
      uint32_t w[4];
      philox4x32_10(cnt0, p, step, 0u, pk, w);
      const float4 xb = qb == 0 ? A[0] : qb == 1 ? A[1] : qb == 2 ? A[2] : A[3];
      const uint32_t wb = qb == 0 ? w[0] : qb == 1 ? w[1] : qb == 2 ? w[2] : w[3];
      S.bk = group_key(xb, inv_temp, wb);
      S.bv = static_cast<int32_t>(gbase + static_cast<uint32_t>(tid + qb * kPassThreads));
      S.bl = xb;
      atomicMax(cta_best, key_enc(S.bk));
    }
    __syncthreads();
  }
  int b = 0;
  for (; b + 2 <= n_full; b += 2) {  // uniform trip count; two blocks per trip over two buffers
    const int j = b * kBlk + tid;
    pass_block<false>(S, A, j, n4, gbase, cnt0 + (static_cast<uint32_t>(b) << 8), p, step, pk, c2e, inv_temp,
                      cta_best, cta_best);
#pragma unroll
    for (int q = 0; q < 4; ++q) A[q] = load(j + 2 * kBlk + q * kPassThreads);
    pass_block<false>(S, B, j + kBlk, n4, gbase, cnt0 + (static_cast<uint32_t>(b + 1) << 8), p, step, pk, c2e,
                      inv_temp, cta_best, cta_best);
#pragma unroll
    for (int q = 0; q < 4; ++q) B[q] = load(j + 3 * kBlk + q * kPassThreads);
  }
  if (b < n_full) {  // an odd last full block
    pass_block<false>(S, A, b * kBlk + tid, n4, gbase, cnt0 + (static_cast<uint32_t>(b) << 8), p, step, pk, c2e,
                      inv_temp, cta_best, cta_best);
#pragma unroll
    for (int q = 0; q < 4; ++q) A[q] = B[q];
    ++b;
  }
  if (b < n_blk)  // the range's last, partial block
    pass_block<true>(S, A, b * kBlk + tid, n4, gbase, cnt0 + (static_cast<uint32_t>(b) << 8), p, step, pk, c2e,
                     inv_temp, cta_best, cta_best);
}

template <int kNoise>
__global__ void __launch_bounds__(kPassThreads, 3)
    sample_pass_kernel(const float* __restrict__ logits, int64_t V, int chunk, float inv_temp, uint32_t k0,
                       uint32_t k1, uint32_t step, Partial* __restrict__ part) {
  __shared__ uint32_t cta_best;  // encoded best exact key of the CTA so far
  __shared__ float red_f[kPassThreads / 32][4];
  __shared__ int32_t red_v[kPassThreads / 32];
  __shared__ float4 red_l[kPassThreads / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int s = blockIdx.x, p = blockIdx.y;
  if (tid == 0) cta_best = key_enc(-INFINITY);
  grid_dependents_launch();  // the final launch may set up meanwhile; it waits for this one
  grid_dependency_wait();    // the logits of the launch before
  __syncthreads();
  const int64_t v0 = static_cast<int64_t>(s) * chunk;
  const int n4 = static_cast<int>((min(V, v0 + chunk) - v0) / 4);
  const float4* src = reinterpret_cast<const float4*>(logits + static_cast<int64_t>(p) * V + v0);
  const float c2e = inv_temp * 1.44269504088896341f;  // screening only
  const PhiloxKeys pk = philox_keys(k0, k1);
  PassState S{-INFINITY, 0.f, 0.f, -INFINITY, 0x7fffffff, 3e38f, NAN, NAN, make_float4(0.f, 0.f, 0.f, 0.f)};
  if (kNoise == 0)
    run_groups(S, src, n4, v0, static_cast<uint32_t>(p), step, pk, c2e, inv_temp, &cta_best);
  else
    run_tokens(S, src, n4, v0, static_cast<uint32_t>(p), step, pk, c2e, inv_temp, &cta_best);
  float m2 = S.m2, z = S.z, s1 = S.s1, bk = S.bk;
  int32_t bv = S.bv;
  float4 bl = S.bl;
  // reduce: sums and the best (key, token or group), lanes then warps in a fixed order
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float om2 = __shfl_down_sync(0xffffffffu, m2, off);
    const float oz = __shfl_down_sync(0xffffffffu, z, off);
    const float os1 = __shfl_down_sync(0xffffffffu, s1, off);
    const float ok = __shfl_down_sync(0xffffffffu, bk, off);
    const int32_t ov = __shfl_down_sync(0xffffffffu, bv, off);
    float4 ol;
    if (kNoise == 0) {
      ol.x = __shfl_down_sync(0xffffffffu, bl.x, off);
      ol.y = __shfl_down_sync(0xffffffffu, bl.y, off);
      ol.z = __shfl_down_sync(0xffffffffu, bl.z, off);
      ol.w = __shfl_down_sync(0xffffffffu, bl.w, off);
    }
    merge_sums(m2, z, s1, om2, oz, os1);
    if (better(ok, ov, bk, bv)) {
      bk = ok;
      bv = ov;
      if (kNoise == 0) bl = ol;
    }
  }
  if (lane == 0) {
    red_f[warp][0] = m2;
    red_f[warp][1] = z;
    red_f[warp][2] = s1;
    red_f[warp][3] = bk;
    red_v[warp] = bv;
    red_l[warp] = bl;
  }
  __syncthreads();
  if (tid == 0) {
    for (int q = 1; q < kPassThreads / 32; ++q) {
      merge_sums(m2, z, s1, red_f[q][0], red_f[q][1], red_f[q][2]);
      if (better(red_f[q][3], red_v[q], bk, bv)) {
        bk = red_f[q][3];
        bv = red_v[q];
        bl = red_l[q];
      }
    }
    if (kNoise == 0) {
      // the token inside the CTA's best group: groups of different CTAs are disjoint and
      // the tokens of a lower group are lower, so (key, token) orders the partials as
      // (key, group) did
      const uint32_t g = static_cast<uint32_t>(bv);
      uint32_t w[4];
      philox4x32_10(group_counter(g), static_cast<uint32_t>(p), step, 1u, pk, w);
      const uint32_t x = group_word(g) == 0 ? w[0] : group_word(g) == 1 ? w[1] : group_word(g) == 2 ? w[2] : w[3];
      bv = static_cast<int32_t>(4 * g) + group_pick(bl, inv_temp, x);
    }
    Partial o;
    o.m2 = m2;
    o.z = z;
    o.s1 = s1;
    o.key = bk;
    o.v = bv;
    o.pad[0] = o.pad[1] = o.pad[2] = 0;
    part[static_cast<int64_t>(p) * gridDim.x + s] = o;
  }
}

// Order-preserving encoding of an entropy for the ascending sort (-0 as +0, so
// that equal values tie and fall back to the position, as fp32 comparison does).
__device__ __forceinline__ uint32_t asc_enc(float h) {
  const uint32_t b = __float_as_uint(h == 0.f ? 0.f : h);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float asc_dec(uint32_t u) {
  return __uint_as_float((u & 0x80000000u) ? (u & 0x7fffffffu) : ~u);
}

__global__ void __launch_bounds__(kFinalThreads)
    sample_final_kernel(const Partial* __restrict__ part, int P, int S, int rule, float bound,
                        const uint8_t* __restrict__ revealed, int32_t* __restrict__ token, float* __restrict__ entropy,
                        float* __restrict__ pmax, uint8_t* __restrict__ accept) {
  __shared__ unsigned long long keys[kFinalThreads];  // rule 0: (entropy, position), sorted ascending
  __shared__ float red_pm[kFinalThreads / 32];
  __shared__ int red_q[kFinalThreads / 32];
  __shared__ uint8_t sh_acc[kFinalThreads];
  __shared__ __align__(16) float hs[kFinalThreads];  // rule 0: the sorted entropies
  __shared__ __align__(16) float cs[kFinalThreads];  // and their running fp32 sums
  grid_dependents_launch();  // the next call's pass may set up; it waits for this launch to finish
  grid_dependency_wait();    // the pass launch's partials
  const int p = threadIdx.x, lane = p & 31, warp = p >> 5;
  float h = INFINITY, pm = 0.f;
  bool rev = true;  // positions past P take part as revealed
  if (p < P) {
    // merge the position's partials in split order (loads four at a time ahead of the merges)
    const float4* q = reinterpret_cast<const float4*>(part + static_cast<int64_t>(p) * S);
    float m2 = -INFINITY, z = 0.f, s1 = 0.f, bk = -INFINITY;
    int32_t bv = 0x7fffffff;
    for (int i0 = 0; i0 < S; i0 += 4) {
      float4 a[4];
      int32_t v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (i0 + u < S) {
          a[u] = __ldg(q + 2 * (i0 + u));
          v[u] = __float_as_int(__ldg(q + 2 * (i0 + u) + 1).x);
        }
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (i0 + u < S) {
          merge_sums(m2, z, s1, a[u].x, a[u].y, a[u].z);
          if (better(a[u].w, v[u], bk, bv)) {
            bk = a[u].w;
            bv = v[u];
          }
        }
    }
    h = logf(z) - (s1 / z) * 0.693147180559945309f;
    pm = 1.f / z;
    rev = revealed[p] != 0;
    token[p] = bv;
    entropy[p] = h;
    pmax[p] = pm;
  }
  sh_acc[p] = 0;
  if (rule == 1) {
    // confidence: every unrevealed position above the threshold; if none, the
    // unrevealed one with the largest pmax (ties to the lower position)
    const bool acc = !rev && pm > bound;
    const int any = __syncthreads_or(acc);
    if (any) {
      if (p < P) accept[p] = acc;
      return;
    }
    float bpm = rev ? -1.f : pm;
    int bq = rev ? 0x7fffffff : p;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float opm = __shfl_xor_sync(0xffffffffu, bpm, off);
      const int oq = __shfl_xor_sync(0xffffffffu, bq, off);
      if (opm > bpm || (opm == bpm && oq < bq)) {
        bpm = opm;
        bq = oq;
      }
    }
    if (lane == 0) {
      red_pm[warp] = bpm;
      red_q[warp] = bq;
    }
    __syncthreads();
    if (p == 0) {
      for (int w = 1; w < kFinalThreads / 32; ++w)
        if (red_pm[w] > red_pm[0] || (red_pm[w] == red_pm[0] && red_q[w] < red_q[0])) {
          red_pm[0] = red_pm[w];
          red_q[0] = red_q[w];
        }
      if (red_q[0] < P) sh_acc[red_q[0]] = 1;
    }
  } else {
    // entropy bound: sort the unrevealed positions by (entropy, position) (bitonic, over
    // the next power of two >= P), then one thread applies the rule in sorted order with
    // one fp32 rounding per step
    int n2 = 32;
    while (n2 < P) n2 <<= 1;
    unsigned long long key =
        rev ? ~0ull : (static_cast<unsigned long long>(asc_enc(h)) << 32) | static_cast<uint32_t>(p);
    const int n = __syncthreads_count(!rev);
    // thread p < n2 holds entry p; a stage pairs p with p ^ j, and the lower one of the
    // pair keeps the smaller key where the k-block sorts ascending.  Pairs inside a warp
    // (j < 32) swap through shuffles; the others through shared memory, ordered by a
    // barrier of the n2 sorting threads alone (the warps past n2 hold no entries)
    if (p < n2) {
      for (int k = 2; k <= n2; k <<= 1)
        for (int j = k >> 1; j > 0; j >>= 1) {
          unsigned long long other;
          if (j < 32) {
            other = __shfl_xor_sync(0xffffffffu, key, j);
          } else {
            keys[p] = key;
            asm volatile("bar.sync 1, %0;" ::"r"(n2) : "memory");
            other = keys[p ^ j];
            asm volatile("bar.sync 1, %0;" ::"r"(n2) : "memory");
          }
          const bool keep_min = ((p & k) == 0) == ((p & j) == 0);
          key = keep_min ? (other < key ? other : key) : (other > key ? other : key);
        }
    }
    // the rule in sorted order: c_i = fl(c_(i-1) + h_i) is the one sequential part (the
    // order of the fp32 roundings is the rule's); the running maximum of ascending
    // entropies is h_i itself.  Every thread decodes its entry, one thread runs the sums
    // four entries at a time, then every thread decides its own entry
    hs[p] = p < n ? asc_dec(static_cast<uint32_t>(key >> 32)) : 0.f;
    __syncthreads();
    if (p == 0) {
      // four entries per trip, the next four loaded ahead (hs is zero past n)
      float c = 0.f;
      float4 h4 = *reinterpret_cast<const float4*>(hs);
      for (int i0 = 0; i0 < n; i0 += 4) {
        const float4 nx = *reinterpret_cast<const float4*>(hs + min(i0 + 4, kFinalThreads - 4));
        const float c0 = __fadd_rn(c, h4.x);
        const float c1 = __fadd_rn(c0, h4.y);
        const float c2 = __fadd_rn(c1, h4.z);
        c = __fadd_rn(c2, h4.w);
        *reinterpret_cast<float4*>(cs + i0) = make_float4(c0, c1, c2, c);
        h4 = nx;
      }
    }
    __syncthreads();
    if (p < n && (p == 0 || __fsub_rn(cs[p], hs[p]) <= bound)) sh_acc[static_cast<uint32_t>(key)] = 1;
  }
  __syncthreads();
  if (p < P) accept[p] = sh_acc[p];
}

}  // namespace


cudaError_t launch_sample(int P, int64_t V, float inv_temp, uint64_t seed, uint32_t step, int rule, float bound,
                          int noise, const float* logits, const uint8_t* revealed, int32_t* token, float* entropy, float* pmax,
                          uint8_t* accept, void* workspace, cudaStream_t st) {
  const int S = sampler_splits(P, V);
  const int chunk = static_cast<int>(sampler_chunk(P, V));
  auto* part = static_cast<Partial*>(workspace);
  const uint32_t k0 = static_cast<uint32_t>(seed), k1 = static_cast<uint32_t>(seed >> 32);
  cudaError_t e = noise == 0 ? launch_pdl(sample_pass_kernel<0>, dim3(S, P), dim3(kPassThreads), 0, st, logits, V,
                                          chunk, inv_temp, k0, k1, step, part)
                             : launch_pdl(sample_pass_kernel<1>, dim3(S, P), dim3(kPassThreads), 0, st, logits, V,
                                          chunk, inv_temp, k0, k1, step, part);
  if (e != cudaSuccess) return e;
  return launch_pdl(sample_final_kernel, dim3(1), dim3(kFinalThreads), 0, st, static_cast<const Partial*>(part), P, S,
                    rule, bound, revealed, token, entropy, pmax, accept);
}

}  // namespace moe
