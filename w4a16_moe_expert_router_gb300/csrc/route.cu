// route.cu -- routing of a canvas in one launch: top-k experts per token,
// softmax over the selected logits, and the per-expert pair lists.
//
// Model card "srswti/axe-diffusion-ksl-xe", "what the model is": every token is
// routed to its top-8 of 128 experts.  "The kernels we built": one launch then
// serves all experts, so pairs are grouped by expert here; the grouping is a
// stable counting sort (pair id ascending inside an expert) with no atomics on
// positions, so the lists are identical from run to run.
//
// Every CTA ranks the experts of 32 tokens (one warp per token).  The CTA that
// finishes last -- it learns so from a ticket counter in the workspace header,
// taken after its top-k results are fenced -- then groups all pairs by expert.
// No CTA waits for another, so the launch cannot stall however its CTAs are
// scheduled.
#include <cfloat>
#include <climits>

#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kRouteThreads = 1024;
constexpr int kRouteWarps = kRouteThreads / 32;  // tokens per CTA

// Router order: larger logit first; equal logits (fp32 compare, so -0 == +0)
// go to the lower expert index.  An id of INT_MAX marks "no candidate".
__device__ __forceinline__ bool ranks_before(float a, int ea, float b, int eb) {
  if (ea == INT_MAX) return false;
  if (eb == INT_MAX) return true;
  return a > b || (a == b && ea < eb);
}

// Top-k of one token's E logits by one warp (lane j holds experts j, j+32, ...;
// E <= 256), then the softmax over the k selected logits, summed in rank order.
__device__ __forceinline__ void topk_softmax_warp(const float* __restrict__ row, int E, int k, int lane,
                                                  int32_t* __restrict__ idx_out, float* __restrict__ w_out) {
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
    }
}

// Stable grouping of the P pairs by expert, by one CTA of kRouteThreads.  Warp w
// owns the contiguous pair range [w*chunk, (w+1)*chunk); pass 1 counts each
// warp's pairs per expert, a scan over (expert, warp) turns the counts into
// first positions, pass 2 places every pair at its warp's running position for
// its expert.  Within a warp, pairs go in rounds of 32 in pair order and a pair's
// rank among equal experts of its round is the number of lower lanes with the
// same expert, so the order inside an expert is the pair order.
__device__ __forceinline__ void group_pairs_block(const int32_t* __restrict__ topk_idx, int P, int E,
                                                  int32_t* __restrict__ expert_offsets,
                                                  int32_t* __restrict__ pair_list) {
  __shared__ int cnt[kRouteWarps][kMaxExperts];  // per warp and expert: count, then next position
  __shared__ int base[kMaxExperts + 1];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int i = tid; i < kRouteWarps * kMaxExperts; i += kRouteThreads) (&cnt[0][0])[i] = 0;
  __syncthreads();
  const int chunk = (P + kRouteWarps - 1) / kRouteWarps;
  const int p_lo = warp * chunk, p_hi = min(P, p_lo + chunk);
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int r0 = p_lo; r0 < p_hi; r0 += 32) {
    const int p = r0 + lane;
    int e = p < p_hi ? __ldcg(topk_idx + p) : -1;
    if (static_cast<unsigned>(e) >= static_cast<unsigned>(E)) e = -1;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    if (e >= 0 && __popc(peers & lt_mask) == 0) cnt[warp][e] += __popc(peers);
    __syncwarp();
  }
  __syncthreads();
  if (tid < E) {  // per expert: exclusive scan over the warps, total in tot
    int run = 0;
    for (int w = 0; w < kRouteWarps; ++w) {
      const int c = cnt[w][tid];
      cnt[w][tid] = run;
      run += c;
    }
    base[tid] = run;
  }
  __syncthreads();
  if (warp == 0) {  // exclusive scan of the expert totals: lane owns 8 consecutive experts
    int local[8], sum = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int e = lane * 8 + j;
      local[j] = sum;
      sum += e < E ? base[e] : 0;
    }
    int incl = sum;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += o;
    }
    const int excl = incl - sum;
    __syncwarp();
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
  for (int r0 = p_lo; r0 < p_hi; r0 += 32) {
    const int p = r0 + lane;
    int e = p < p_hi ? __ldcg(topk_idx + p) : -1;
    if (static_cast<unsigned>(e) >= static_cast<unsigned>(E)) e = -1;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & lt_mask);
    if (e >= 0) pair_list[base[e] + cnt[warp][e] + rank] = p;
    __syncwarp();
    if (e >= 0 && rank == 0) cnt[warp][e] += __popc(peers);
    __syncwarp();
  }
}

__global__ void __launch_bounds__(kRouteThreads) route_kernel(const float* __restrict__ logits, int T, int E, int k,
                                                              int32_t* __restrict__ topk_idx,
                                                              float* __restrict__ topk_w,
                                                              int32_t* __restrict__ expert_offsets,
                                                              int32_t* __restrict__ pair_list,
                                                              uint32_t* __restrict__ ticket) {
  __shared__ int is_last;
  grid_dependents_launch();  // the next launch may set up meanwhile; it waits for this one
  grid_dependency_wait();    // logits, and the routing arrays an earlier launch may still read
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * kRouteWarps + (threadIdx.x >> 5);
  if (t < T)
    topk_softmax_warp(logits + static_cast<size_t>(t) * E, E, k, lane, topk_idx + static_cast<size_t>(t) * k,
                      topk_w + static_cast<size_t>(t) * k);
  __threadfence();  // this CTA's results are visible device-wide before its ticket is taken
  __syncthreads();
  if (threadIdx.x == 0) is_last = atomicAdd(ticket, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  group_pairs_block(topk_idx, T * k, E, expert_offsets, pair_list);
  if (threadIdx.x == 0) *ticket = 0;  // ready for the next launch on this workspace
}

}  // namespace

cudaError_t launch_route(const Dims& s, const float* logits, int32_t* topk_idx, float* topk_w,
                         int32_t* expert_offsets, int32_t* pair_list, WsHeader* hdr, cudaStream_t st) {
  const int grid = (s.T + kRouteWarps - 1) / kRouteWarps;
  return launch_pdl(route_kernel, dim3(grid), dim3(kRouteThreads), 0, st, logits, s.T, s.E, s.k, topk_idx, topk_w,
                    expert_offsets, pair_list, &hdr->route_ticket);
}

}  // namespace moe
