// combine.cu -- fixed-order weighted combine of the k expert outputs of each
// token, with an optional fused RMSNorm.
//
// Model card "srswti/axe-diffusion-ksl-xe", "the kernels we built": the weighted
// combine uses a fixed-order reduction instead of index_add_, because a 1-ulp
// difference from atomics can flip a block-diffusion acceptance threshold; and
// RMSNorm collapses into a single launch.  With RMSNorm one CTA owns one token
// row (the norm needs the whole row); without it four 128-thread CTAs share a
// row, a quarter each (more CTAs to spread the reads over the SMs):
//   u[i]   = w[t][0] y[t*k][i] + ... + w[t][k-1] y[t*k+k-1][i]   (fp32, rank order, fused multiply-adds)
//   out[i] = fp16(u[i])                                         without gamma
//   out[i] = fp16(gamma[i] * u[i] / sqrt(mean(u^2) + eps))       with gamma
// The sum of squares uses a fixed tree (per-thread in index order, butterfly
// inside each warp, then the warps in order), so the result is bit-identical
// from run to run.
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kThreads = 512;
constexpr int kMaxVec = 4;  // float4 per thread: d <= 8192

template <bool kNorm>
__global__ void __launch_bounds__(kThreads) combine_kernel(const float* __restrict__ topk_w,
                                                           const float* __restrict__ y, int d, int k,
                                                           const float* __restrict__ gamma, float eps,
                                                           uint16_t* __restrict__ out) {
  __shared__ float warp_ss[kThreads / 32];
  grid_dependents_launch();
  grid_dependency_wait();  // the expert outputs y of the launch before
  const int t = blockIdx.x, tid = threadIdx.x;
  const int n4 = d >> 2;
  float wr[kMaxTopK];
#pragma unroll
  for (int r = 0; r < kMaxTopK; ++r) wr[r] = r < k ? topk_w[static_cast<size_t>(t) * k + r] : 0.f;
  const float4* y4 = reinterpret_cast<const float4*>(y) + static_cast<size_t>(t) * k * n4;
  float4 u[kMaxVec];
  float ss = 0.f;
#pragma unroll
  for (int j = 0; j < kMaxVec; ++j) {
    const int i4 = tid + kThreads * j;
    if (i4 < n4) {
      // all k rows' values are requested before the first is used
      float4 v[kMaxTopK];
#pragma unroll
      for (int r = 0; r < kMaxTopK; ++r)
        if (r < k) v[r] = y4[static_cast<size_t>(r) * n4 + i4];
      float4 acc = make_float4(wr[0] * v[0].x, wr[0] * v[0].y, wr[0] * v[0].z, wr[0] * v[0].w);
#pragma unroll
      for (int r = 1; r < kMaxTopK; ++r) {
        if (r < k) {
          acc.x = fmaf(wr[r], v[r].x, acc.x);
          acc.y = fmaf(wr[r], v[r].y, acc.y);
          acc.z = fmaf(wr[r], v[r].z, acc.z);
          acc.w = fmaf(wr[r], v[r].w, acc.w);
        }
      }
      u[j] = acc;
      if (kNorm) {
        ss = fmaf(acc.x, acc.x, ss);
        ss = fmaf(acc.y, acc.y, ss);
        ss = fmaf(acc.z, acc.z, ss);
        ss = fmaf(acc.w, acc.w, ss);
      }
    }
  }
  float scale = 1.f;
  if (kNorm) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    if ((tid & 31) == 0) warp_ss[tid >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) tot += warp_ss[w];
    scale = 1.f / sqrtf(tot / static_cast<float>(d) + eps);
  }
  uint2* o2 = reinterpret_cast<uint2*>(out + static_cast<size_t>(t) * d);
  const float4* g4 = reinterpret_cast<const float4*>(gamma);
#pragma unroll
  for (int j = 0; j < kMaxVec; ++j) {
    const int i4 = tid + kThreads * j;
    if (i4 < n4) {
      float4 v = u[j];
      if (kNorm) {
        const float4 g = g4[i4];
        v = make_float4(g.x * (v.x * scale), g.y * (v.y * scale), g.z * (v.z * scale), g.w * (v.w * scale));
      }
      const __half2 lo = __floats2half2_rn(v.x, v.y);
      const __half2 hi = __floats2half2_rn(v.z, v.w);
      o2[i4] = make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
    }
  }
}

// Without RMSNorm: one 128-thread CTA per quarter of a token row (d / 4 columns,
// one float4 per thread and row), the same arithmetic in the same order; with a
// residual x, out = fp16(x + u) (one fp32 addition after the rank-order sum).
__global__ void __launch_bounds__(128) combine_quarter_kernel(const float* __restrict__ topk_w,
                                                             const float* __restrict__ y, int d, int k,
                                                             const uint16_t* residual,  // may equal out
                                                             uint16_t* out) {
  grid_dependents_launch();
  grid_dependency_wait();
  const int t = blockIdx.x >> 2, q = blockIdx.x & 3;
  const int n4 = d >> 2;
  const float4* y4 = reinterpret_cast<const float4*>(y) + static_cast<size_t>(t) * k * n4;
  uint2* o2 = reinterpret_cast<uint2*>(out + static_cast<size_t>(t) * d);
  for (int i4 = q * (n4 >> 2) + threadIdx.x; i4 < (q + 1) * (n4 >> 2); i4 += 128) {
    float wr[kMaxTopK];
    float4 v[kMaxTopK];
#pragma unroll
    for (int r = 0; r < kMaxTopK; ++r)
      if (r < k) {
        wr[r] = topk_w[static_cast<size_t>(t) * k + r];
        v[r] = y4[static_cast<size_t>(r) * n4 + i4];
      }
    float4 acc = make_float4(wr[0] * v[0].x, wr[0] * v[0].y, wr[0] * v[0].z, wr[0] * v[0].w);
#pragma unroll
    for (int r = 1; r < kMaxTopK; ++r)
      if (r < k) {
        acc.x = fmaf(wr[r], v[r].x, acc.x);
        acc.y = fmaf(wr[r], v[r].y, acc.y);
        acc.z = fmaf(wr[r], v[r].z, acc.z);
        acc.w = fmaf(wr[r], v[r].w, acc.w);
      }
    if (residual) {
      const uint2 xr = reinterpret_cast<const uint2*>(residual + static_cast<size_t>(t) * d)[i4];
      const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&xr.x));
      const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&xr.y));
      acc = make_float4(__fadd_rn(a.x, acc.x), __fadd_rn(a.y, acc.y), __fadd_rn(b.x, acc.z), __fadd_rn(b.y, acc.w));
    }
    const __half2 lo = __floats2half2_rn(acc.x, acc.y);
    const __half2 hi = __floats2half2_rn(acc.z, acc.w);
    o2[i4] = make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
  }
}

}  // namespace

cudaError_t launch_combine(const Dims& s, const float* topk_w, const float* y, const float* gamma, float eps,
                           const uint16_t* residual, uint16_t* out, cudaStream_t st) {
  if (gamma && residual) return cudaErrorInvalidValue;
  if (gamma) return launch_pdl(combine_kernel<true>, dim3(s.T), dim3(kThreads), 0, st, topk_w, y, s.d, s.k, gamma, eps, out);
  return launch_pdl(combine_quarter_kernel, dim3(4 * s.T), dim3(128), 0, st, topk_w, y, s.d, s.k, residual, out);
}

}  // namespace moe
