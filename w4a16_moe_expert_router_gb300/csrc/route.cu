// route.cu -- routing of a canvas: top-k experts per token, softmax over the
// selected logits, and the per-expert pair lists.
//
// Model card "srswti/axe-diffusion-ksl-xe", "what the model is": every token is
// routed to its top-8 of 128 experts.  "The kernels we built": one launch then
// serves all experts, so pairs are grouped by expert here; the grouping is a
// stable counting sort (pair id ascending inside an expert) with no atomics on
// positions, so the lists are identical from run to run.
#include <cfloat>
#include <climits>

#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kRouteWarps = 8;    // tokens per CTA of the top-k kernel
constexpr int kPermThreads = 1024;
constexpr int kPermWarps = kPermThreads / 32;

// Router order: larger logit first; equal logits (fp32 compare, so -0 == +0)
// go to the lower expert index.  An id of INT_MAX marks "no candidate".
__device__ __forceinline__ bool ranks_before(float a, int ea, float b, int eb) {
  if (ea == INT_MAX) return false;
  if (eb == INT_MAX) return true;
  return a > b || (a == b && ea < eb);
}

// One warp per token.  Lane j holds logits of experts j, j+32, ... (E <= 256).
__global__ void __launch_bounds__(kRouteWarps * 32) topk_softmax_kernel(const float* __restrict__ logits, int T,
                                                                         int E, int k, int32_t* __restrict__ topk_idx,
                                                                         float* __restrict__ topk_w) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * kRouteWarps + (threadIdx.x >> 5);
  if (t >= T) return;
  const float* row = logits + static_cast<size_t>(t) * E;
  float v[kMaxExperts / 32];
  uint32_t avail = 0;
#pragma unroll
  for (int j = 0; j < kMaxExperts / 32; ++j) {
    const int e = lane + 32 * j;
    v[j] = 0.f;
    if (e < E) {
      v[j] = row[e];
      avail |= 1u << j;
    }
  }
  float sel_v[kMaxTopK];
  int sel_e[kMaxTopK];
#pragma unroll
  for (int r = 0; r < kMaxTopK; ++r) {
    sel_v[r] = 0.f;
    sel_e[r] = 0;
    if (r < k) {
      float bv = 0.f;
      int be = INT_MAX;
#pragma unroll
      for (int j = 0; j < kMaxExperts / 32; ++j)
        if (((avail >> j) & 1u) && ranks_before(v[j], lane + 32 * j, bv, be)) {
          bv = v[j];
          be = lane + 32 * j;
        }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
        const int oe = __shfl_xor_sync(0xffffffffu, be, off);
        if (ranks_before(ov, oe, bv, be)) {
          bv = ov;
          be = oe;
        }
      }
      // every lane now holds the same winner (the order is total)
      if ((be & 31) == lane) avail &= ~(1u << (be >> 5));
      sel_v[r] = bv;
      sel_e[r] = be;
    }
  }
  // softmax over the k selected logits, summed in rank order
  const float m = sel_v[0];
  float den = 0.f;
#pragma unroll
  for (int r = 0; r < kMaxTopK; ++r)
    if (r < k) den += expf(sel_v[r] - m);
#pragma unroll
  for (int r = 0; r < kMaxTopK; ++r)
    if (r < k && r == lane) {
      topk_idx[static_cast<size_t>(t) * k + r] = sel_e[r];
      topk_w[static_cast<size_t>(t) * k + r] = expf(sel_v[r] - m) / den;
    }
}

// Single CTA: expert_offsets and pair_list from topk_idx.  Pairs are visited
// in rounds of kPermThreads in pair order; a pair's slot is its expert's base
// plus the number of earlier pairs (same round, lower warp or lower lane) with
// the same expert, so the result is the stable order by construction.
__global__ void __launch_bounds__(kPermThreads) permute_kernel(const int32_t* __restrict__ topk_idx, int P, int E,
                                                               int32_t* __restrict__ expert_offsets,
                                                               int32_t* __restrict__ pair_list) {
  __shared__ int cnt[kMaxExperts];
  __shared__ int base[kMaxExperts];
  __shared__ int wcnt[kPermWarps][kMaxExperts];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int e = tid; e < kMaxExperts; e += kPermThreads) cnt[e] = 0;
  for (int i = tid; i < kPermWarps * kMaxExperts; i += kPermThreads) (&wcnt[0][0])[i] = 0;
  __syncthreads();
  for (int p = tid; p < P; p += kPermThreads) {
    const int e = topk_idx[p];
    if (static_cast<unsigned>(e) < static_cast<unsigned>(E)) atomicAdd(&cnt[e], 1);  // integer count
  }
  __syncthreads();
  if (warp == 0) {  // exclusive scan of cnt[0..E) : lane owns 8 consecutive experts
    int local[8], sum = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int e = lane * 8 + j;
      local[j] = sum;
      sum += (e < E) ? cnt[e] : 0;
    }
    int incl = sum;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += o;
    }
    const int excl = incl - sum;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int e = lane * 8 + j;
      if (e < E) {
        base[e] = excl + local[j];
        expert_offsets[e] = excl + local[j];
      }
    }
    if (lane == 31) expert_offsets[E] = incl;
  }
  __syncthreads();
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int r0 = 0; r0 < P; r0 += kPermThreads) {
    const int p = r0 + tid;
    int e = (p < P) ? topk_idx[p] : -1;
    if (static_cast<unsigned>(e) >= static_cast<unsigned>(E)) e = -1;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & lt_mask);
    if (e >= 0 && rank == 0) wcnt[warp][e] = __popc(peers);
    __syncthreads();
    if (e >= 0) {
      int before = 0;
      for (int w = 0; w < warp; ++w) before += wcnt[w][e];
      pair_list[base[e] + before + rank] = p;
    }
    __syncthreads();
    for (int ee = tid; ee < E; ee += kPermThreads) {
      int tot = 0;
      for (int w = 0; w < kPermWarps; ++w) {
        tot += wcnt[w][ee];
        wcnt[w][ee] = 0;
      }
      base[ee] += tot;
    }
    __syncthreads();
  }
}

}  // namespace

cudaError_t launch_route(const Dims& s, const float* logits, int32_t* topk_idx, float* topk_w,
                         int32_t* expert_offsets, int32_t* pair_list, WsHeader* /*hdr*/, cudaStream_t st) {
  const int grid = (s.T + kRouteWarps - 1) / kRouteWarps;
  topk_softmax_kernel<<<grid, kRouteWarps * 32, 0, st>>>(logits, s.T, s.E, s.k, topk_idx, topk_w);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  permute_kernel<<<1, kPermThreads, 0, st>>>(topk_idx, static_cast<int>(s.pairs()), s.E, expert_offsets,
                                             pair_list);
  return cudaGetLastError();
}

}  // namespace moe
