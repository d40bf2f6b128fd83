// route.cu -- routing of a canvas: top-k experts per token, softmax over the
// selected logits, and the per-expert pair lists.
//
// Model card "srswti/axe-diffusion-ksl-xe", "what the model is": every token is
// routed to its top-8 of 128 experts.  "The kernels we built": one launch then
// serves all experts, so pairs are grouped by expert here; the grouping is a
// stable counting sort (pair id ascending inside an expert) with no atomics on
// positions, so the lists are identical from run to run.
//
// Two launches.  The first ranks the experts of every token (one warp per
// token, eight tokens per CTA, so even a 256-token canvas spreads over 32 SMs)
// and, per CTA, counts its pairs per expert and ranks each pair among the
// CTA's earlier pairs of the same expert.  The second, one CTA launched with
// programmatic dependent launch, turns the per-CTA counts into positions
// (exclusive scans over CTAs, then over experts) and places every pair.
#include <cfloat>
#include <climits>

#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kTopkWarps = 8;        // tokens per CTA of the top-k launch
constexpr int kGroupThreads = 1024;  // the grouping CTA
constexpr int kScanSplit = kGroupThreads / kMaxExperts;  // threads per expert in the scan over CTAs

// Router order as one unsigned key: a larger logit gives a larger key, -0 and
// +0 give the same key (they compare equal as fp32 values); NaN ranks below
// every number.  Equal keys go to the lower expert index.
__device__ __forceinline__ uint32_t order_key(float v) {
  if (v != v) return 1u;
  if (v == 0.f) v = 0.f;
  const uint32_t b = __float_as_uint(v);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Top-k of one token's E logits by one warp (lane j holds experts j, j+32, ...;
// E <= 256), then the softmax over the k selected logits, summed in rank order.
// Each round takes the largest key over the warp (one reduction) and, among the
// lanes holding it, the lowest expert index (a second reduction).
__device__ __forceinline__ void topk_softmax_warp(const float* __restrict__ row, int E, int k, int lane,
                                                  int32_t* __restrict__ idx_out, float* __restrict__ w_out,
                                                  int* __restrict__ sel_out) {
  float v[kMaxExperts / 32];
  uint32_t key[kMaxExperts / 32];
  uint32_t avail = 0;
#pragma unroll
  for (int j = 0; j < kMaxExperts / 32; ++j) {
    const int e = lane + 32 * j;
    v[j] = 0.f;
    key[j] = 0u;
    if (e < E) {
      v[j] = row[e];
      key[j] = order_key(v[j]);
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
      // this lane's best remaining candidate: largest key, then lowest index
      uint32_t bk = 0u;
      int bj = -1;
      float bv = 0.f;
#pragma unroll
      for (int j = 0; j < kMaxExperts / 32; ++j)
        if (((avail >> j) & 1u) && (bj < 0 || key[j] > bk)) {
          bk = key[j];
          bj = j;
          bv = v[j];
        }
      const uint32_t kmax = __reduce_max_sync(0xffffffffu, bj >= 0 ? bk : 0u);
      const uint32_t cand = (bj >= 0 && bk == kmax) ? static_cast<uint32_t>(lane + 32 * bj) : 0xffffffffu;
      const uint32_t win = __reduce_min_sync(0xffffffffu, cand);
      if (static_cast<int>(win & 31u) == lane) avail &= ~(1u << (win >> 5));
      sel_e[r] = static_cast<int>(win);
      sel_v[r] = __shfl_sync(0xffffffffu, bv, static_cast<int>(win & 31u));
    }
  }
  const float m = sel_v[0];
  float den = 0.f;
#pragma unroll
  for (int r = 0; r < kMaxTopK; ++r)
    if (r < k) den += expf(sel_v[r] - m);
#pragma unroll
  for (int r = 0; r < kMaxTopK; ++r)
    if (r < k && r == lane) {
      idx_out[r] = sel_e[r];
      w_out[r] = expf(sel_v[r] - m) / den;
      sel_out[r] = sel_e[r];
    }
}

// Top-k of 8 tokens per CTA, then the CTA's pairs (p = t*k + r, in order) counted
// per expert (cta_hist[cta][e]) and ranked among the CTA's earlier pairs of the
// same expert (local_rank[p]).
__global__ void __launch_bounds__(kTopkWarps * 32) topk_kernel(const float* __restrict__ logits, int T, int E, int k,
                                                                int32_t* __restrict__ topk_idx,
                                                                float* __restrict__ topk_w,
                                                                int32_t* __restrict__ cta_hist,
                                                                int32_t* __restrict__ local_rank) {
  __shared__ int sel[kTopkWarps * kMaxTopK];
  __shared__ int hist[kMaxExperts];
  grid_dependents_launch();  // the grouping launch may set up meanwhile; it waits for this one
  grid_dependency_wait();    // logits, and the routing arrays an earlier launch may still read
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int e = tid; e < E; e += kTopkWarps * 32) hist[e] = 0;
  const int t = blockIdx.x * kTopkWarps + warp;
  if (t < T) {
    topk_softmax_warp(logits + static_cast<size_t>(t) * E, E, k, lane, topk_idx + static_cast<size_t>(t) * k,
                      topk_w + static_cast<size_t>(t) * k, sel + warp * k);
  } else if (lane < k) {
    sel[warp * k + lane] = -1;
  }
  __syncthreads();
  const int npairs = kTopkWarps * k;  // <= 64
  if (warp == 0) {
    // the CTA's pairs in rounds of 32, in pair order: a pair's rank is the count of its expert
    // in earlier rounds plus the lower lanes of its round with the same expert
    const unsigned lt_mask = (1u << lane) - 1u;
    for (int r0 = 0; r0 < npairs; r0 += 32) {
      const int i = r0 + lane;
      int e = i < npairs ? sel[i] : -1;
      if (static_cast<unsigned>(e) >= static_cast<unsigned>(E)) e = -1;
      const unsigned peers = __match_any_sync(0xffffffffu, e);
      if (e >= 0) local_rank[static_cast<size_t>(blockIdx.x) * npairs + i] = hist[e] + __popc(peers & lt_mask);
      __syncwarp();
      if (e >= 0 && (peers & lt_mask) == 0) hist[e] += __popc(peers);
      __syncwarp();
    }
  }
  __syncthreads();
  for (int e = tid; e < E; e += kTopkWarps * 32) cta_hist[static_cast<size_t>(blockIdx.x) * E + e] = hist[e];
}

// One CTA: per expert, the exclusive scan of the per-CTA counts over the CTAs
// (written back in place), the expert offsets (exclusive scan over experts), and
// every pair placed at offset + earlier CTAs' count + its rank in its CTA.
__global__ void __launch_bounds__(kGroupThreads) group_kernel(const int32_t* __restrict__ topk_idx, int P, int E,
                                                              int k, int nctas, int32_t* __restrict__ cta_hist,
                                                              const int32_t* __restrict__ local_rank,
                                                              int32_t* __restrict__ expert_offsets,
                                                              int32_t* __restrict__ pair_list) {
  __shared__ int base[kMaxExperts];
  __shared__ int tot[kMaxExperts];
  grid_dependents_launch();
  grid_dependency_wait();  // the top-k launch's outputs
  __shared__ int part[kMaxExperts][kScanSplit];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // per expert, kScanSplit threads each own a contiguous range of CTAs: their sums, an
  // exclusive scan of those sums, then each range's prefixes written back in place
  const int e_s = tid / kScanSplit, sub = tid % kScanSplit;
  const int per = (nctas + kScanSplit - 1) / kScanSplit;
  const int c_lo = sub * per, c_hi = min(nctas, c_lo + per);
  if (e_s < E) {
    int sum = 0;
#pragma unroll 8
    for (int c = c_lo; c < c_hi; ++c) sum += cta_hist[static_cast<size_t>(c) * E + e_s];
    part[e_s][sub] = sum;
  }
  __syncthreads();
  if (e_s < E) {
    int run = 0;
    for (int j = 0; j < sub; ++j) run += part[e_s][j];
    if (sub == kScanSplit - 1) tot[e_s] = run + part[e_s][sub];
#pragma unroll 8
    for (int c = c_lo; c < c_hi; ++c) {
      const int h = cta_hist[static_cast<size_t>(c) * E + e_s];
      cta_hist[static_cast<size_t>(c) * E + e_s] = run;
      run += h;
    }
  }
  __syncthreads();
  if (warp == 0) {  // exclusive scan of the expert totals: lane owns 8 consecutive experts
    int local[8], sum = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int e = lane * 8 + j;
      local[j] = sum;
      sum += e < E ? tot[e] : 0;
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
  const int pairs_per_cta = kTopkWarps * k;
  constexpr int kU = 4;  // pairs per thread per round, their loads issued together
  for (int p0 = tid; p0 < P; p0 += kU * kGroupThreads) {
    int e[kU], lr[kU], h[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int p = p0 + u * kGroupThreads;
      e[u] = p < P ? topk_idx[p] : -1;
      lr[u] = p < P ? local_rank[p] : 0;
      if (static_cast<unsigned>(e[u]) >= static_cast<unsigned>(E)) e[u] = -1;
    }
#pragma unroll
    for (int u = 0; u < kU; ++u)
      h[u] = e[u] >= 0 ? cta_hist[static_cast<size_t>((p0 + u * kGroupThreads) / pairs_per_cta) * E + e[u]] : 0;
#pragma unroll
    for (int u = 0; u < kU; ++u)
      if (e[u] >= 0) pair_list[base[e[u]] + h[u] + lr[u]] = p0 + u * kGroupThreads;
  }
}

}  // namespace

cudaError_t launch_route(const Dims& s, const float* logits, int32_t* topk_idx, float* topk_w,
                         int32_t* expert_offsets, int32_t* pair_list, void* workspace, cudaStream_t st) {
  const int nctas = (s.T + kTopkWarps - 1) / kTopkWarps;
  auto* base = static_cast<uint8_t*>(workspace);
  auto* cta_hist = reinterpret_cast<int32_t*>(base + ws_route_offset(s));
  auto* local_rank = reinterpret_cast<int32_t*>(base + ws_route_offset(s) + ws_route_hist_bytes(s));
  cudaError_t err = launch_pdl(topk_kernel, dim3(nctas), dim3(kTopkWarps * 32), 0, st, logits, s.T, s.E, s.k,
                               topk_idx, topk_w, cta_hist, local_rank);
  if (err != cudaSuccess) return err;
  return launch_pdl(group_kernel, dim3(1), dim3(kGroupThreads), 0, st, static_cast<const int32_t*>(topk_idx),
                    static_cast<int>(s.pairs()), s.E, s.k, nctas, cta_hist,
                    static_cast<const int32_t*>(local_rank), expert_offsets, pair_list);
}

}  // namespace moe
