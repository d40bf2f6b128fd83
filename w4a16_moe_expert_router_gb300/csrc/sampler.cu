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
// Gumbel-max: token = argmax_v (t_v + G_v), t_v = logit_v * inv_temp,
// G_v = -ln(-ln U_v), U_v = ((x & 0x7fffff) + 1/2) 2^-23 from word v % 4 of
// Philox4x32-10 (Salmon et al., SC'11) at counter (v / 4, position, step, 0) under
// key (seed low, seed high); ties to the lower index.  The key decides an
// integer, so it is computed with one IEEE fp32 rounding per operation (ln_f32
// below, then fma(logit, inv_temp, G)): any implementation that takes these
// steps gets the same token.
//
// Pass kernel (grid: vocabulary splits x positions, 256 threads): each thread
// streams float4s of its position's logits and keeps, in base 2, the running
// maximum m2 of t2 = t log2(e), Z = sum 2^(t2 - m2) and S1 = sum 2^(t2 - m2)(t2 - m2).
// Computing the exact key of every element would cost two logarithms each and
// make the pass arithmetic-bound, so a cheap necessary condition screens them:
// with K the best exact key the CTA has found so far, element v can reach K only
// if w_v = 1 - U_v <= e^(t_v - K) (because -ln U >= 1 - U, and G = -ln(-ln U));
// the test is made with a margin that covers every rounding involved (fast
// exponentials included), and only the elements that pass it (a few per warp
// over the pass) get their exact key.  The test reuses 2^(t2 - m2) of the
// softmax sum, so an element costs one Philox quarter, one exp2 and about eight
// other instructions.  The logits stream through an 8-stage cp.async ring in
// shared memory (each thread copies and later reads its own float4 of every
// stage, so the only wait is cp.async.wait_group on the thread's own copies and
// no barrier is needed); seven 16-byte copies per thread are in flight.  Each CTA
// writes its partial (m2, Z, S1, best key, index).
//
// Final kernel (one CTA, one thread per position): merges each position's
// partials in split order, writes token, entropy H = ln Z - (S1 / Z) ln 2 and
// top-1 probability 1 / Z, then applies the acceptance rule to those fp32
// values (entropy rule: rank by (H, position), then one thread runs the fp32
// cumulative sum and maximum in sorted order).
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"

namespace moe {
namespace {

constexpr int kPassThreads = 256;
constexpr int kStages = 8;  // cp.async stages per thread: one float4 each, up to seven in flight
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
    const uint64_t p0 = static_cast<uint64_t>(0xD2511F53u) * c0;
    const uint64_t p1 = static_cast<uint64_t>(0xCD9E8D57u) * c2;
    const uint32_t n0 = static_cast<uint32_t>(p1 >> 32) ^ c1 ^ k.k0[r];
    const uint32_t n2 = static_cast<uint32_t>(p0 >> 32) ^ c3 ^ k.k1[r];
    c1 = static_cast<uint32_t>(p1);
    c3 = static_cast<uint32_t>(p0);
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

__global__ void __launch_bounds__(kPassThreads, 4)
    sample_pass_kernel(const float* __restrict__ logits, int64_t V, int chunk, float inv_temp, uint32_t k0,
                       uint32_t k1, uint32_t step, Partial* __restrict__ part) {
  __shared__ uint32_t cta_best;  // encoded best exact key of the CTA so far
  __shared__ float red_f[kPassThreads / 32][4];
  __shared__ int32_t red_v[kPassThreads / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int s = blockIdx.x, p = blockIdx.y;
  if (tid == 0) cta_best = key_enc(-INFINITY);
  __syncthreads();
  const int64_t v0 = static_cast<int64_t>(s) * chunk;
  const int64_t n4 = (min(V, v0 + chunk) - v0) / 4;
  const float4* src = reinterpret_cast<const float4*>(logits + static_cast<int64_t>(p) * V + v0);
  const uint32_t g0 = static_cast<uint32_t>(v0 / 4);
  const float c2e = inv_temp * 1.44269504088896341f;  // screening only
  volatile uint32_t* vbest = &cta_best;
  float m2 = -INFINITY, z = 0.f, s1 = 0.f;
  float bk = -INFINITY;
  int32_t bv = 0x7fffffff;
  __shared__ float4 ring[kStages][kPassThreads];
  const PhiloxKeys pk = philox_keys(k0, k1);
  const int n_iter = static_cast<int>((n4 + kPassThreads - 1) / kPassThreads);
  // copy of float4 (it * 256 + tid) into slot it % kStages; one commit group per iteration
  auto issue = [&](int it) {
    const int64_t j = static_cast<int64_t>(it) * kPassThreads + tid;
    if (it < n_iter && j < n4) {
      const uint32_t dst = static_cast<uint32_t>(__cvta_generic_to_shared(&ring[it % kStages][tid]));
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src + j) : "memory");
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };
#pragma unroll
  for (int it = 0; it < kStages - 1; ++it) issue(it);
  float c2 = 3e38f, c_K = NAN, c_m2 = NAN;  // screening factor and the (K, m2) it was made for
  for (int it = 0; it < n_iter; ++it) {  // uniform trip count
    issue(it + kStages - 1);
    asm volatile("cp.async.wait_group %0;" ::"n"(kStages - 1) : "memory");  // this thread's copy of `it` landed
    const int64_t j = static_cast<int64_t>(it) * kPassThreads + tid;
    const bool active = j < n4;
    float4 l4 = make_float4(0.f, 0.f, 0.f, 0.f);
    if (active) l4 = ring[it % kStages][tid];
    uint32_t w[4];
    philox4x32_10(g0 + static_cast<uint32_t>(j), static_cast<uint32_t>(p), step, 0u, pk, w);
    const float l[4] = {l4.x, l4.y, l4.z, l4.w};
    bool cand[4] = {false, false, false, false};
    if (active) {
      const float mx = fmaxf(fmaxf(l[0], l[1]), fmaxf(l[2], l[3])) * c2e;
      if (mx > m2) {
        if (z != 0.f) {
          const float dm = m2 - mx;
          const float r = fast_exp2(dm);
          s1 = r * fmaf(dm, z, s1);
          z *= r;
        }
        m2 = mx;
      }
      // screen: element v needs w_v <= 2^(t2_v - K2 + slack) = 2^(t2_v - m2) c2 with
      // c2 = 2^(m2 - K2 + slack); the slack (base-2 units) and the factor 1.01 cover
      // the roundings of t2, K2 and the approximate exp2.  Before the CTA has a key,
      // c2 is huge: every element whose 2^(t2 - m2) does not underflow is screened in
      // (one that underflows cannot beat its thread's own maximum, which is screened in)
      const float K = key_dec(*vbest);
      if (K != c_K || m2 != c_m2) {
        c_K = K;
        c_m2 = m2;
        c2 = 3e38f;
        if (K != -INFINITY) {
          const float K2 = K * 1.44269504088896341f;
          const float slack = 0x1p-8f + (fabsf(m2) + fabsf(K2)) * 0x1p-14f;
          c2 = fminf(fast_exp2(m2 - K2 + slack) * 1.01f, 3e38f);
        }
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float d = fmaf(l[i], c2e, -m2);
        const float e = fast_exp2(d);
        z += e;
        s1 = fmaf(e, d, s1);
        // with f = 1 + (x & 0x7fffff) 2^-23, w = 1 - U = 2 - 2^-24 - f exactly, so
        // w <= e c2  <=>  f >= 2 - 2^-24 - e c2, implied by f >= fl(2 - 2^-23 - e c2)
        const float f = __uint_as_float(0x3f800000u | (w[i] & 0x007fffffu));
        cand[i] = f >= fmaf(-e, c2, 0x1.fffffep+0f);
      }
    }
    const bool any = cand[0] || cand[1] || cand[2] || cand[3];
    if (__any_sync(0xffffffffu, any)) {
      if (any) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          if (!cand[i]) continue;
          const float k = gumbel_key(l[i], inv_temp, w[i]);
          const int32_t v = static_cast<int32_t>(v0 + 4 * j + i);
          if (better(k, v, bk, bv)) {
            bk = k;
            bv = v;
          }
        }
        atomicMax(&cta_best, key_enc(bk));
      }
    }
  }
  asm volatile("cp.async.wait_all;" ::: "memory");
  // reduce: sums and the best (key, index), lanes then warps in a fixed order
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float om2 = __shfl_down_sync(0xffffffffu, m2, off);
    const float oz = __shfl_down_sync(0xffffffffu, z, off);
    const float os1 = __shfl_down_sync(0xffffffffu, s1, off);
    const float ok = __shfl_down_sync(0xffffffffu, bk, off);
    const int32_t ov = __shfl_down_sync(0xffffffffu, bv, off);
    merge_sums(m2, z, s1, om2, oz, os1);
    if (better(ok, ov, bk, bv)) {
      bk = ok;
      bv = ov;
    }
  }
  if (lane == 0) {
    red_f[warp][0] = m2;
    red_f[warp][1] = z;
    red_f[warp][2] = s1;
    red_f[warp][3] = bk;
    red_v[warp] = bv;
  }
  __syncthreads();
  if (tid == 0) {
    for (int q = 1; q < kPassThreads / 32; ++q) {
      merge_sums(m2, z, s1, red_f[q][0], red_f[q][1], red_f[q][2]);
      if (better(red_f[q][3], red_v[q], bk, bv)) {
        bk = red_f[q][3];
        bv = red_v[q];
      }
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

__global__ void __launch_bounds__(kFinalThreads)
    sample_final_kernel(const Partial* __restrict__ part, int P, int S, int rule, float bound,
                        const uint8_t* __restrict__ revealed, int32_t* __restrict__ token, float* __restrict__ entropy,
                        float* __restrict__ pmax, uint8_t* __restrict__ accept) {
  __shared__ __align__(16) float sh_h[kFinalThreads];
  __shared__ __align__(16) float sh_pm[kFinalThreads];
  __shared__ __align__(16) float sorted_h[kFinalThreads];
  __shared__ __align__(16) int sorted_p[kFinalThreads];
  __shared__ __align__(16) uint8_t sh_rev[kFinalThreads];
  __shared__ uint8_t sh_acc[kFinalThreads];
  const int p = threadIdx.x;
  // positions past P take part as revealed, with an entropy that ranks last
  float h = INFINITY, pm = 0.f;
  uint8_t rev = 1;
  if (p < P) {
    const float4* q = reinterpret_cast<const float4*>(part + static_cast<int64_t>(p) * S);
    float4 a = __ldg(q);
    float m2 = a.x, z = a.y, s1 = a.z, bk = a.w;
    int32_t bv = __float_as_int(__ldg(q + 1).x);
    for (int i = 1; i < S; ++i) {
      const float4 b = __ldg(q + 2 * i);
      const int32_t v = __float_as_int(__ldg(q + 2 * i + 1).x);
      merge_sums(m2, z, s1, b.x, b.y, b.z);
      if (better(b.w, v, bk, bv)) {
        bk = b.w;
        bv = v;
      }
    }
    h = logf(z) - (s1 / z) * 0.693147180559945309f;
    pm = 1.f / z;
    rev = revealed[p] != 0;
    token[p] = bv;
    entropy[p] = h;
    pmax[p] = pm;
  }
  sh_h[p] = h;
  sh_pm[p] = pm;
  sh_rev[p] = rev;
  sh_acc[p] = 0;
  const int n = __syncthreads_count(!rev);  // unrevealed positions
  const int P4 = (P + 3) & ~3;              // rank over whole float4s: padded slots are revealed
  if (rule == 0) {
    // rank of each unrevealed position by (entropy, position)
    if (!rev) {
      int r = 0;
      for (int q = 0; q < P4; q += 4) {
        const float4 hq = *reinterpret_cast<const float4*>(&sh_h[q]);
        const uchar4 rq = *reinterpret_cast<const uchar4*>(&sh_rev[q]);
        r += !rq.x && (hq.x < h || (hq.x == h && q < p));
        r += !rq.y && (hq.y < h || (hq.y == h && q + 1 < p));
        r += !rq.z && (hq.z < h || (hq.z == h && q + 2 < p));
        r += !rq.w && (hq.w < h || (hq.w == h && q + 3 < p));
      }
      sorted_h[r] = h;
      sorted_p[r] = p;
    }
    __syncthreads();
    if (p == 0) {
      // the mlx-vlm rule in sorted order, one fp32 rounding per step, in sequence
      float c = 0.f, x = -INFINITY;
      int i = 0;
      for (; i + 4 <= n; i += 4) {
        const float4 hv = *reinterpret_cast<const float4*>(&sorted_h[i]);
        const int4 pv = *reinterpret_cast<const int4*>(&sorted_p[i]);
        const float hh[4] = {hv.x, hv.y, hv.z, hv.w};
        const int pp[4] = {pv.x, pv.y, pv.z, pv.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          c = __fadd_rn(c, hh[u]);
          x = fmaxf(x, hh[u]);
          if (i + u == 0 || __fsub_rn(c, x) <= bound) sh_acc[pp[u]] = 1;
        }
      }
      for (; i < n; ++i) {
        c = __fadd_rn(c, sorted_h[i]);
        x = fmaxf(x, sorted_h[i]);
        if (i == 0 || __fsub_rn(c, x) <= bound) sh_acc[sorted_p[i]] = 1;
      }
    }
  } else if (p == 0) {
    int best = -1;
    bool any = false;
    for (int q = 0; q < P; ++q) {
      if (sh_rev[q]) continue;
      if (sh_pm[q] > bound) {
        sh_acc[q] = 1;
        any = true;
      }
      if (best < 0 || sh_pm[q] > sh_pm[best]) best = q;
    }
    if (!any && best >= 0) sh_acc[best] = 1;
  }
  __syncthreads();
  if (p < P) accept[p] = sh_acc[p];
}

}  // namespace

int sampler_splits(int64_t vocab) { return static_cast<int>((vocab + kSamplerChunk - 1) / kSamplerChunk); }

cudaError_t launch_sample(int P, int64_t V, float inv_temp, uint64_t seed, uint32_t step, int rule, float bound,
                          const float* logits, const uint8_t* revealed, int32_t* token, float* entropy, float* pmax,
                          uint8_t* accept, void* workspace, cudaStream_t st) {
  const int S = sampler_splits(V);
  auto* part = static_cast<Partial*>(workspace);
  sample_pass_kernel<<<dim3(S, P), kPassThreads, 0, st>>>(logits, V, kSamplerChunk, inv_temp,
                                                          static_cast<uint32_t>(seed),
                                                          static_cast<uint32_t>(seed >> 32), step, part);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  sample_final_kernel<<<1, kFinalThreads, 0, st>>>(part, P, S, rule, bound, revealed, token, entropy, pmax, accept);
  return cudaGetLastError();
}

}  // namespace moe
