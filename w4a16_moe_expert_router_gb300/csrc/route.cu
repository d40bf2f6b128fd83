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
// CTA's earlier pairs of the same expert.  The second, launched with
// programmatic dependent launch, has one CTA per CTA of the first: each reads
// the whole table of per-CTA counts (one parallel round of loads), forms the
// expert totals, their exclusive scan (the expert offsets) and its own CTA's
// prefix per expert, and places that CTA's pairs.
#include <cfloat>
#include <climits>

#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kTopkWarps = 8;        // tokens per CTA of the top-k launch
constexpr int kGroupThreads = 256;   // a grouping CTA: one thread per expert (E <= 256)

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
// same expert (local_rank[p]).  A token selects an expert at most once, so the
// rank of pair (t, e) is the number of earlier tokens of the CTA that selected e:
// one bit per token (warp) in a per-expert mask, set with an order-independent
// atomicOr, then popcounts.
__global__ void __launch_bounds__(kTopkWarps * 32) topk_kernel(const float* __restrict__ logits, int T, int E, int k,
                                                                int32_t* __restrict__ topk_idx,
                                                                float* __restrict__ topk_w,
                                                                int32_t* __restrict__ cta_hist,
                                                                int32_t* __restrict__ local_rank) {
  __shared__ int sel[kTopkWarps * kMaxTopK];
  __shared__ unsigned emask[kMaxExperts];
  grid_dependents_launch();  // the grouping launch may set up meanwhile; it waits for this one
  grid_dependency_wait();    // logits, and the routing arrays an earlier launch may still read
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int e = tid; e < E; e += kTopkWarps * 32) emask[e] = 0u;
  __syncthreads();
  const int t = blockIdx.x * kTopkWarps + warp;
  if (t < T) {
    topk_softmax_warp(logits + static_cast<size_t>(t) * E, E, k, lane, topk_idx + static_cast<size_t>(t) * k,
                      topk_w + static_cast<size_t>(t) * k, sel + warp * k);
    __syncwarp();
    if (lane < k) {
      const int e = sel[warp * k + lane];
      if (static_cast<unsigned>(e) < static_cast<unsigned>(E)) atomicOr(&emask[e], 1u << warp);
    }
  }
  __syncthreads();
  if (t < T && lane < k) {
    const int e = sel[warp * k + lane];
    if (static_cast<unsigned>(e) < static_cast<unsigned>(E))
      local_rank[static_cast<size_t>(t) * k + lane] = __popc(emask[e] & ((1u << warp) - 1u));
  }
  for (int e = tid; e < E; e += kTopkWarps * 32) cta_hist[static_cast<size_t>(blockIdx.x) * E + e] = __popc(emask[e]);
}

// Grouping CTA c (one per top-k CTA): thread e sums the counts of expert e over
// all top-k CTAs (its total) and over CTAs before c (its prefix for CTA c); the
// exclusive scan of the totals gives the expert offsets; then CTA c places its
// own pairs at offset + prefix + rank in the CTA.  CTA 0 also writes the offsets.
__global__ void __launch_bounds__(kGroupThreads) group_kernel(const int32_t* __restrict__ topk_idx, int P, int E,
                                                              int k, int nctas, const int32_t* __restrict__ cta_hist,
                                                              const int32_t* __restrict__ local_rank,
                                                              int32_t* __restrict__ expert_offsets,
                                                              int32_t* __restrict__ pair_list) {
  __shared__ int pos_base[kMaxExperts];  // offset of expert e + the count of e in CTAs before this one
  __shared__ int warp_tot[kGroupThreads / 32];
  grid_dependents_launch();
  grid_dependency_wait();  // the top-k launch's outputs
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, c = blockIdx.x;
  const int e = tid;
  int tot = 0, pre = 0;
  if (e < E) {
#pragma unroll 16
    for (int cc = 0; cc < nctas; ++cc) {
      const int h = cta_hist[static_cast<size_t>(cc) * E + e];
      tot += h;
      pre += cc < c ? h : 0;
    }
  }
  // exclusive scan of the totals over the experts (thread e holds expert e)
  int incl = tot;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  int before = 0;
#pragma unroll
  for (int w = 0; w < kGroupThreads / 32; ++w) before += w < warp ? warp_tot[w] : 0;
  const int offset = before + incl - tot;
  if (e < E) {
    pos_base[e] = offset + pre;
    if (c == 0) expert_offsets[e] = offset;
  }
  if (c == 0 && e == E - 1) expert_offsets[E] = offset + tot;
  __syncthreads();
  // this CTA's pairs: p = c * (tokens per top-k CTA * k) + i
  const int pairs_per_cta = kTopkWarps * k;  // <= 64
  const int p = c * pairs_per_cta + tid;
  if (tid < pairs_per_cta && p < P) {
    const int ep = topk_idx[p];
    if (static_cast<unsigned>(ep) < static_cast<unsigned>(E)) pair_list[pos_base[ep] + local_rank[p]] = p;
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
  return launch_pdl(group_kernel, dim3(nctas), dim3(kGroupThreads), 0, st, static_cast<const int32_t*>(topk_idx),
                    static_cast<int>(s.pairs()), s.E, s.k, nctas, static_cast<const int32_t*>(cta_hist),
                    static_cast<const int32_t*>(local_rank), expert_offsets, pair_list);
}

}  // namespace moe
