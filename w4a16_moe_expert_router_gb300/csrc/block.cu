// block.cu -- the front of the MoE block around the expert layer: the pre-norm
// and the router projection.
//
// Model card "srswti/axe-diffusion-ksl-xe", "the kernels we built": the RMSNorm of
// a block runs as one launch; "what the model is": a router sends each token to
// its top-8 of 128 experts.  The block is read as a pre-norm residual block:
//   u = fp16(gamma * (x * r)),  r = 1 / sqrt(ss / d + eps),  ss = sum_k x_k^2
//   logits[t][e] = sum_k u[t][k] * Wr[e][k]      (Wr fp16 [E][d])
//   out = fp16(x + layer(u))                      (the residual, in the combine)
// The logits decide the routing, an integer result, so ss and the logits follow
// one fixed order of fp32 operations that is part of the definition: the d
// columns are dealt to the 32 lanes of a warp in 8-column chunks (lane l takes
// chunks l, l + 32, ... in that order), each lane accumulates fmaf(a_k, b_k, acc)
// column by column from 0, and the lane sums meet in an xor butterfly (offsets
// 16, 8, 4, 2, 1).  r, x_k * r and gamma_k * (x_k * r) are single IEEE fp32
// operations and u rounds to nearest even, so u and the logits are reproducible
// bit for bit off the GPU.
//
// One CTA per 8 tokens and 32 experts: warp w normalises token w into shared
// memory (the CTAs of the first expert column also write u out), then each warp
// forms the logits of four experts for the 8 tokens in one pass over its lanes'
// columns: a lane converts each 8-column chunk of u once and of each router row
// once, and feeds all 32 (expert, token) sums from them.
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kFrontTokens = 8;    // tokens per CTA (one warp each for the norm)
constexpr int kFrontExperts = 32;  // experts per CTA (four per warp for the router)
constexpr int kWarpExperts = 4;
constexpr int kFrontThreads = 256;

__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 p = __half22float2(bits_h2(w[i]));
    f[2 * i] = p.x;
    f[2 * i + 1] = p.y;
  }
}

// Sum of one value per lane in the butterfly order (every lane ends with the total).
__device__ __forceinline__ float lane_butterfly_sum(float v) {
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, off));
  return v;
}

__global__ void __launch_bounds__(kFrontThreads) block_front_kernel(const uint16_t* __restrict__ x,
                                                                     const float* __restrict__ gamma, float eps,
                                                                     const uint16_t* __restrict__ wr, int T, int d,
                                                                     int E, uint16_t* __restrict__ u_out,
                                                                     float* __restrict__ logits) {
  extern __shared__ uint4 su[];  // [kFrontTokens][d / 8]: the CTA's rows of u
  grid_dependents_launch();
  grid_dependency_wait();  // x may be the output of the launch before
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = blockIdx.x * kFrontTokens, e0 = blockIdx.y * kFrontExperts;
  const int nch = d / 8;
  // the router rows of the warp's four experts; their first two chunks are loaded now, so
  // that the loads overlap the pre-norm (rows past E read row E - 1 and are not written)
  const int eb = e0 + kWarpExperts * warp;
  const uint4* wrow[kWarpExperts];
  uint4 wnext[kWarpExperts], wnext2[kWarpExperts];  // chunks c and c + 32 of the rows
#pragma unroll
  for (int j = 0; j < kWarpExperts; ++j) {
    wrow[j] = reinterpret_cast<const uint4*>(wr + static_cast<size_t>(min(eb + j, E - 1)) * d);
    wnext[j] = wrow[j][lane];
    wnext2[j] = wrow[j][min(lane + 32, nch - 1)];
  }
  {
    // ---- pre-norm of token t0 + warp
    const int t = t0 + warp;
    uint4* srow = su + warp * nch;
    if (t < T) {
      const uint4* xr = reinterpret_cast<const uint4*>(x + static_cast<size_t>(t) * d);
      float ss = 0.f;
#pragma unroll 8
      for (int c = lane; c < nch; c += 32) {
        const uint4 v = xr[c];
        srow[c] = v;
        float f[8];
        unpack8(v, f);
#pragma unroll
        for (int i = 0; i < 8; ++i) ss = fmaf(f[i], f[i], ss);
      }
      ss = lane_butterfly_sum(ss);
      const float r = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, static_cast<float>(d)), eps)));
      uint4* urow = reinterpret_cast<uint4*>(u_out + static_cast<size_t>(t) * d);
      const float4* g4 = reinterpret_cast<const float4*>(gamma);
#pragma unroll 8
      for (int c = lane; c < nch; c += 32) {
        float f[8];
        unpack8(srow[c], f);
        const float4 ga = g4[2 * c], gb = g4[2 * c + 1];
        const float g[8] = {ga.x, ga.y, ga.z, ga.w, gb.x, gb.y, gb.z, gb.w};
        uint32_t h[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
          h[i] = h2_bits(__halves2half2(__float2half_rn(__fmul_rn(g[2 * i], __fmul_rn(f[2 * i], r))),
                                        __float2half_rn(__fmul_rn(g[2 * i + 1], __fmul_rn(f[2 * i + 1], r)))));
        const uint4 uv = make_uint4(h[0], h[1], h[2], h[3]);
        srow[c] = uv;
        if (blockIdx.y == 0) urow[c] = uv;
      }
    }
  }
  __syncthreads();
  // ---- router logits of experts e0 + 4 warp + j (j < 4) for the CTA's tokens; each
  // trip loads the chunk two ahead of the four rows before it uses the current one
  float acc[kWarpExperts][kFrontTokens];
#pragma unroll
  for (int j = 0; j < kWarpExperts; ++j)
#pragma unroll
    for (int tt = 0; tt < kFrontTokens; ++tt) acc[j][tt] = 0.f;
  for (int c = lane; c < nch; c += 32) {
    float w[kWarpExperts][8];
#pragma unroll
    for (int j = 0; j < kWarpExperts; ++j) {
      unpack8(wnext[j], w[j]);
      wnext[j] = wnext2[j];
      if (c + 64 < nch) wnext2[j] = wrow[j][c + 64];
    }
#pragma unroll
    for (int tt = 0; tt < kFrontTokens; ++tt) {
      float uf[8];
      unpack8(su[tt * nch + c], uf);
#pragma unroll
      for (int j = 0; j < kWarpExperts; ++j)
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[j][tt] = fmaf(uf[i], w[j][i], acc[j][tt]);
    }
  }
#pragma unroll
  for (int j = 0; j < kWarpExperts; ++j)
#pragma unroll
    for (int tt = 0; tt < kFrontTokens; ++tt) {
      const float v = lane_butterfly_sum(acc[j][tt]);
      if (lane == 0 && eb + j < E && t0 + tt < T) logits[static_cast<size_t>(t0 + tt) * E + eb + j] = v;
    }
}

}  // namespace

cudaError_t init_block_kernels() {
  return cudaFuncSetAttribute(block_front_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kFrontTokens * kMaxHidden * 2);
}

cudaError_t launch_block_front(const Dims& s, const uint16_t* x, const float* gamma, float eps, const uint16_t* wr,
                               uint16_t* u, float* logits, cudaStream_t st) {
  const dim3 grid((s.T + kFrontTokens - 1) / kFrontTokens, (s.E + kFrontExperts - 1) / kFrontExperts);
  return launch_pdl(block_front_kernel, grid, dim3(kFrontThreads), size_t(kFrontTokens) * s.d * 2, st, x, gamma, eps,
                    wr, s.T, s.d, s.E, u, logits);
}

}  // namespace moe
