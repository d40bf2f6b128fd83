// route.cu -- routing of a canvas: top-k experts per token, softmax over the
// selected logits, and the per-expert pair lists.
//
// Model card "srswti/axe-diffusion-ksl-xe", "what the model is": every token is
// routed to its top-8 of 128 experts.  "The kernels we built": one launch then
// serves all experts, so pairs are grouped by expert here; the grouping is a
// stable counting sort (pair id ascending inside an expert) with no atomics on
// positions, so the lists are identical from run to run.
//
// Top-k step (one warp per token, eight tokens per CTA, so even a 256-token canvas
// spreads over 32 SMs): each CTA ranks the experts of its tokens, counts its pairs
// per expert (hist[c][e]) and ranks each pair among the CTA's earlier pairs of the
// same expert.  A pair's place in the lists is then
//   offset[e] + sum_{c' < c} hist[c'][e] + its rank in CTA c.
// Up to 64 top-k CTAs (512 tokens) a grouping launch follows, one CTA per top-k
// CTA, each summing the count table's column of every expert itself (one parallel
// round of loads).  Above that, the work of that launch would grow with the square
// of the CTA count, so two launches take its place, each linear in the input: the
// prefix over CTAs of each expert's counts, in place, with the expert totals; then
// the placement, one CTA per top-k CTA.  Launches are chained by programmatic
// dependent launch.
#include <cfloat>
#include <climits>

#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kTopkWarps = 8;        // tokens per top-k CTA
constexpr int kRouteThreads = 256;   // threads of a routing CTA: one per expert (E <= 256) when grouping
constexpr int kGroupMaxCtas = 64;    // the one-launch grouping up to 64 top-k CTAs (512 tokens)
static_assert(kTopkWarps * 32 == kRouteThreads && kMaxExperts <= kRouteThreads, "one thread per expert");

// Router order as one unsigned key: a larger logit gives a larger key, -0 and
// +0 give the same key (they compare equal as fp32 values); NaN ranks below
// every number.  Equal keys go to the lower expert index.
__device__ __forceinline__ uint32_t order_key(float v) {
  if (v != v) return 1u;
  if (v == 0.f) v = 0.f;
  const uint32_t b = __float_as_uint(v);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Compare-exchange of two candidates of a lane: afterwards slot a holds the one
// that ranks first (larger key, then lower slot, i.e. lower expert index).
__device__ __forceinline__ void cx(uint32_t& ka, int& ja, float& va, uint32_t& kb, int& jb, float& vb) {
  const bool swap = kb > ka || (kb == ka && jb < ja);
  if (swap) {
    const uint32_t tk = ka;
    const int tj = ja;
    const float tv = va;
    ka = kb;
    ja = jb;
    va = vb;
    kb = tk;
    jb = tj;
    vb = tv;
  }
}

// Top-k of one token's E logits by one warp, then the softmax over the k selected
// logits, summed in rank order.  Lane l holds experts l + 32 j (j < NS, NS = 4 for
// E <= 128, else 8) and sorts them once by (key descending, index ascending) with a
// sorting network (5 or 19 compare-exchanges), so its head is its best remaining
// candidate.  Each round takes the largest head key over the warp (one reduction);
// if one lane holds it (one ballot) that lane wins, otherwise the lowest expert
// index among the tied heads does (a second reduction); the winning lane drops its
// head.
template <int NS>
__device__ __forceinline__ void topk_softmax_warp(const float* __restrict__ row, int E, int k, int lane,
                                                  int32_t* __restrict__ idx_out, float* __restrict__ w_out,
                                                  int* __restrict__ sel_out) {
  float v[NS];
  uint32_t key[NS];
  int js[NS];
#pragma unroll
  for (int j = 0; j < NS; ++j) {
    const int e = lane + 32 * j;
    v[j] = 0.f;
    key[j] = 0u;  // below every real key (order_key >= 1)
    js[j] = j;
    if (e < E) {
      v[j] = row[e];
      key[j] = order_key(v[j]);
    }
  }
  if constexpr (NS == 4) {
    constexpr int net[5][2] = {{0, 1}, {2, 3}, {0, 2}, {1, 3}, {1, 2}};
#pragma unroll
    for (int c = 0; c < 5; ++c) {
      const int a = net[c][0], b = net[c][1];
      cx(key[a], js[a], v[a], key[b], js[b], v[b]);
    }
  } else {
    constexpr int net[19][2] = {{0, 2}, {1, 3}, {4, 6}, {5, 7}, {0, 4}, {1, 5}, {2, 6}, {3, 7}, {0, 1}, {2, 3},
                                {4, 5}, {6, 7}, {2, 4}, {3, 5}, {1, 4}, {3, 6}, {1, 2}, {3, 4}, {5, 6}};
#pragma unroll
    for (int c = 0; c < 19; ++c) {
      const int a = net[c][0], b = net[c][1];
      cx(key[a], js[a], v[a], key[b], js[b], v[b]);
    }
  }
  float sel_v[kMaxTopK];
  int sel_e[kMaxTopK];
#pragma unroll
  for (int r = 0; r < kMaxTopK; ++r) {
    sel_v[r] = 0.f;
    sel_e[r] = 0;
    if (r < k) {
      const uint32_t kmax = __reduce_max_sync(0xffffffffu, key[0]);
      const bool mine = key[0] == kmax;
      const unsigned tied = __ballot_sync(0xffffffffu, mine);
      int wl;  // winning lane
      if ((tied & (tied - 1u)) == 0u) {
        wl = __ffs(tied) - 1;
      } else {
        const uint32_t cand = mine ? static_cast<uint32_t>(lane + 32 * js[0]) : 0xffffffffu;
        wl = static_cast<int>(__reduce_min_sync(0xffffffffu, cand) & 31u);
      }
      sel_e[r] = __shfl_sync(0xffffffffu, lane + 32 * js[0], wl);
      sel_v[r] = __shfl_sync(0xffffffffu, v[0], wl);
      if (lane == wl) {
#pragma unroll
        for (int j = 0; j + 1 < NS; ++j) {
          key[j] = key[j + 1];
          js[j] = js[j + 1];
          v[j] = v[j + 1];
        }
        key[NS - 1] = 0u;
      }
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

// Top-k of the CTA's 8 tokens, then the CTA's pairs (p = t*k + r, in order)
// counted per expert (hist[c][e]) and ranked among the CTA's earlier pairs of the
// same expert (local_rank[p]).  A token selects an expert at most once, so the
// rank of pair (t, e) is the number of earlier tokens of the CTA that selected e:
// one bit per token (warp) in a per-expert mask, set with an order-independent
// atomicOr, then popcounts.
__device__ __forceinline__ void topk_cta(const float* __restrict__ logits, int T, int E, int k,
                                         int32_t* __restrict__ topk_idx, float* __restrict__ topk_w,
                                         int32_t* __restrict__ cta_hist, int32_t* __restrict__ local_rank, int* sel,
                                         unsigned* emask) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int e = tid; e < E; e += kRouteThreads) emask[e] = 0u;
  __syncthreads();
  const int t = blockIdx.x * kTopkWarps + warp;
  if (t < T) {
    if (E <= 128)
      topk_softmax_warp<4>(logits + static_cast<size_t>(t) * E, E, k, lane, topk_idx + static_cast<size_t>(t) * k,
                           topk_w + static_cast<size_t>(t) * k, sel + warp * k);
    else
      topk_softmax_warp<8>(logits + static_cast<size_t>(t) * E, E, k, lane, topk_idx + static_cast<size_t>(t) * k,
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
  for (int e = tid; e < E; e += kRouteThreads) cta_hist[static_cast<size_t>(blockIdx.x) * E + e] = __popc(emask[e]);
}

// Exclusive scan of one value per thread over the CTA's 256 threads (thread e holds
// expert e); returns the thread's prefix.  Uses warp_tot[8]; starts and ends with a
// barrier.
__device__ __forceinline__ int cta_exclusive_scan(int v, int* warp_tot) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  __syncthreads();
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  int before = 0;
#pragma unroll
  for (int w = 0; w < kRouteThreads / 32; ++w) before += w < warp ? warp_tot[w] : 0;
  __syncthreads();
  return before + incl - v;
}

// Grouping CTA c (one per top-k CTA, at most kGroupMaxCtas): thread e sums the
// counts of expert e over all top-k CTAs (its total) and over CTAs before c (its
// prefix for CTA c); the exclusive scan of the totals gives the expert offsets;
// then CTA c places its own pairs.  CTA 0 also writes the offsets.
__global__ void __launch_bounds__(kRouteThreads) group_kernel(const int32_t* __restrict__ topk_idx, int P, int E,
                                                              int k, int nctas, const int32_t* __restrict__ cta_hist,
                                                              const int32_t* __restrict__ local_rank,
                                                              int32_t* __restrict__ expert_offsets,
                                                              int32_t* __restrict__ pair_list) {
  __shared__ int pos_base[kMaxExperts];
  __shared__ int warp_tot[kRouteThreads / 32];
  grid_dependents_launch();
  grid_dependency_wait();  // the top-k launch's outputs
  const int tid = threadIdx.x, c = blockIdx.x, e = tid;
  int tot = 0, pre = 0;
  if (e < E) {
#pragma unroll 16
    for (int cc = 0; cc < nctas; ++cc) {
      const int h = cta_hist[static_cast<size_t>(cc) * E + e];
      tot += h;
      pre += cc < c ? h : 0;
    }
  }
  const int offset = cta_exclusive_scan(tot, warp_tot);
  if (e < E) {
    pos_base[e] = offset + pre;
    if (c == 0) expert_offsets[e] = offset;
  }
  if (c == 0 && e == E - 1) expert_offsets[E] = offset + tot;
  __syncthreads();
  const int per_cta = kTopkWarps * k;  // <= 64
  const int p = c * per_cta + tid;
  if (tid < per_cta && p < P) {
    const int ep = topk_idx[p];
    if (static_cast<unsigned>(ep) < static_cast<unsigned>(E)) pair_list[pos_base[ep] + local_rank[p]] = p;
  }
}

// Top-k step.
__global__ void __launch_bounds__(kRouteThreads) topk_kernel(const float* __restrict__ logits, int T, int E, int k,
                                                              int32_t* __restrict__ topk_idx,
                                                              float* __restrict__ topk_w,
                                                              int32_t* __restrict__ cta_hist,
                                                              int32_t* __restrict__ local_rank) {
  __shared__ int sel[kTopkWarps * kMaxTopK];
  __shared__ unsigned emask[kMaxExperts];
  grid_dependents_launch();  // the next launch may set up meanwhile; it waits for this one
  grid_dependency_wait();    // logits, and the routing arrays an earlier launch may still read
  topk_cta(logits, T, E, k, topk_idx, topk_w, cta_hist, local_rank, sel, emask);
}

// Prefix step: for 32 experts per CTA (lane = expert), hist[c][e] is replaced in
// place by sum_{c' < c} hist[c'][e], and tot[e] receives the expert's total.  Warp w
// takes a contiguous segment of the CTAs: segment sums, their exclusive scan over
// the warps, then a second pass that writes the prefixes.
__global__ void __launch_bounds__(1024) prefix_kernel(int32_t* __restrict__ cta_hist, int nctas, int E,
                                                      int32_t* __restrict__ tot) {
  __shared__ int seg_sum[32][33];
  grid_dependents_launch();
  grid_dependency_wait();  // the top-k launch's counts
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int e = blockIdx.x * 32 + lane;
  const int seg = (nctas + 31) / 32;
  const int c0 = min(nctas, warp * seg), c1 = min(nctas, c0 + seg);
  int s = 0;
  if (e < E) {
#pragma unroll 8
    for (int c = c0; c < c1; ++c) s += cta_hist[static_cast<size_t>(c) * E + e];
  }
  seg_sum[warp][lane] = s;
  __syncthreads();
  int run = 0;
  for (int w = 0; w < warp; ++w) run += seg_sum[w][lane];
  if (warp == 31 && e < E) tot[e] = run + s;
  if (e < E) {
    for (int c = c0; c < c1; ++c) {
      int32_t* h = cta_hist + static_cast<size_t>(c) * E + e;
      const int v = *h;
      *h = run;
      run += v;
    }
  }
}

// Placement step, CTA c per top-k CTA: the expert offsets from the totals (CTA 0
// also writes them), then CTA c's pairs at offset + prefix + rank.
__global__ void __launch_bounds__(kRouteThreads) place_kernel(const int32_t* __restrict__ topk_idx, int P, int E,
                                                               int k, const int32_t* __restrict__ cta_pre,
                                                               const int32_t* __restrict__ local_rank,
                                                               const int32_t* __restrict__ tot,
                                                               int32_t* __restrict__ expert_offsets,
                                                               int32_t* __restrict__ pair_list) {
  __shared__ int pos_base[kMaxExperts];
  __shared__ int warp_tot[kRouteThreads / 32];
  grid_dependents_launch();
  grid_dependency_wait();  // the prefix launch's outputs (and, through it, the top-k launch's)
  const int tid = threadIdx.x, c = blockIdx.x, e = tid;
  const int t = e < E ? tot[e] : 0;
  const int offset = cta_exclusive_scan(t, warp_tot);
  if (e < E) {
    pos_base[e] = offset + cta_pre[static_cast<size_t>(c) * E + e];
    if (c == 0) expert_offsets[e] = offset;
  }
  if (c == 0 && e == E - 1) expert_offsets[E] = offset + t;
  __syncthreads();
  const int per_cta = kTopkWarps * k;  // <= 64
  const int p = c * per_cta + tid;
  if (tid < per_cta && p < P) {
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
  auto* tot = local_rank + s.pairs();
  cudaError_t err = launch_pdl(topk_kernel, dim3(nctas), dim3(kRouteThreads), 0, st, logits, s.T, s.E, s.k,
                               topk_idx, topk_w, cta_hist, local_rank);
  if (err != cudaSuccess) return err;
  if (nctas <= kGroupMaxCtas)
    return launch_pdl(group_kernel, dim3(nctas), dim3(kRouteThreads), 0, st, static_cast<const int32_t*>(topk_idx),
                      static_cast<int>(s.pairs()), s.E, s.k, nctas, static_cast<const int32_t*>(cta_hist),
                      static_cast<const int32_t*>(local_rank), expert_offsets, pair_list);
  err = launch_pdl(prefix_kernel, dim3((s.E + 31) / 32), dim3(1024), 0, st, cta_hist, nctas, s.E, tot);
  if (err != cudaSuccess) return err;
  return launch_pdl(place_kernel, dim3(nctas), dim3(kRouteThreads), 0, st, static_cast<const int32_t*>(topk_idx),
                    static_cast<int>(s.pairs()), s.E, s.k, static_cast<const int32_t*>(cta_hist),
                    static_cast<const int32_t*>(local_rank), static_cast<const int32_t*>(tot), expert_offsets,
                    pair_list);
}

}  // namespace moe
