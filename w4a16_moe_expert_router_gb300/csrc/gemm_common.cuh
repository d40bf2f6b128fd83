// gemm_common.cuh -- device helpers of the expert GEMM launch: the work list of
// (projection, expert, 128-row block, token chunk) items, the launch arguments,
// bounded waits, and the 2-D TMA load of token rows.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace gemm {

struct Proj {
  const uint8_t* w;         // prepared stream of the projection, all experts
  int64_t expert_bytes;     // stream bytes per expert
  int64_t block_bytes;      // stream bytes per 128-row block
  int nblocks;              // blocks per expert
  int K;                    // contraction length (multiple of 64)
  int g;                    // quantisation group along K (32, 64 or 128)
};

struct Args {
  Proj p[2];                // 0: gate_up, 1: down
  int first, last;          // projections in this launch's work list (0 <= first <= last <= 1)
  const int32_t* offsets;   // [E+1]
  const int32_t* pair_list; // [T*k]
  int E;
  uint16_t* h;              // gate_up output, down input [T*k][f] (expert-sorted rows)
  float* y_out;             // down output [T*k][d]
  int f, d, act;
  int32_t* err;
  int32_t* counter;         // work counter of this launch
  int32_t* done_ctas;       // CTAs that have finished; the last one resets both counters
  int32_t* gu_done;         // [E] gate_up epilogue warps finished per expert
};

// Fills the launch arguments of one expert-GEMM launch (which: kGemmGateUp and/or kGemmDown).
inline bool make_args(Args& a, int which, const Dims& s, const int32_t* expert_offsets, const int32_t* pair_list,
                      const uint8_t* w_gate_up, const uint8_t* w_down, const GemmWorkspace& ws) {
  a = Args{};
  const int K[2] = {s.d, s.f}, g[2] = {s.g1, s.g2}, nb[2] = {s.f / 64, s.d / kBlockRows};
  const uint8_t* w[2] = {w_gate_up, w_down};
  for (int pj = 0; pj < 2; ++pj) {
    a.p[pj].w = w[pj];
    a.p[pj].K = K[pj];
    a.p[pj].g = g[pj];
    a.p[pj].nblocks = nb[pj];
    a.p[pj].block_bytes = int64_t(kBlockRows) * K[pj] / 2 + int64_t(kBlockRows) * (K[pj] / g[pj]) * 4;
    a.p[pj].expert_bytes = a.p[pj].block_bytes * nb[pj];
  }
  a.first = (which & kGemmGateUp) ? 0 : 1;
  a.last = (which & kGemmDown) ? 1 : 0;
  if (which == 0 || a.first > a.last) return false;
  a.offsets = expert_offsets;
  a.pair_list = pair_list;
  a.E = s.E;
  a.f = s.f;
  a.d = s.d;
  a.act = s.act;
  a.err = &ws.hdr->error;
  a.h = ws.h;
  a.y_out = ws.y;
  // gate_up launches (alone or fused) and down-only launches keep separate counters
  const int c = a.first == 0 ? 0 : 1;
  a.counter = &ws.hdr->next_item[c];
  a.done_ctas = &ws.hdr->done_ctas[c];
  a.gu_done = ws.gu_done;
  return true;
}

__device__ __forceinline__ int expert_of(int item, const int* prefix, int E) {
  int lo = 0, hi = E - 1;
  while (lo < hi) {  // largest e with prefix[e] <= item
    const int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= item) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// Work item of one projection -> (expert, 128-row block, token chunk); the chunk
// varies fastest, so concurrent items of a busy expert share weight blocks in L2.
__device__ __forceinline__ void decode_item(int item, const int* prefix, const int* offs, int E, int chunk,
                                            int& expert, int& blk, int& n_cnt, int& pos0) {
  const int e = expert_of(item, prefix, E);
  const int n_e = offs[e + 1] - offs[e];
  const int nch = (n_e + chunk - 1) / chunk;
  const int r = item - prefix[e];
  const int c = r % nch;
  expert = e;
  blk = r / nch;
  n_cnt = min(chunk, n_e - chunk * c);
  pos0 = offs[e] + chunk * c;
}

// Items per expert = blocks * ceil(n_e / chunk), exclusive scans into prefix[pj][e]
// (one warp, 8 experts per lane), and the expert offsets copied to shared memory.
__device__ __forceinline__ void scan_items(const Args& a, int chunk, int lane, int (*prefix)[kMaxExperts + 1],
                                           int* offs) {
  for (int pj = 0; pj < 2; ++pj) {
    const int nb = a.p[pj].nblocks;
    int loc[8], sum = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int e = lane * 8 + j;
      loc[j] = sum;
      if (e < a.E) sum += nb * ((a.offsets[e + 1] - a.offsets[e] + chunk - 1) / chunk);
    }
    int incl = sum;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += o;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (lane * 8 + j < a.E) prefix[pj][lane * 8 + j] = incl - sum + loc[j];
    if (lane == 31) prefix[pj][a.E] = incl;
  }
  for (int e = lane; e <= a.E; e += 32) offs[e] = a.offsets[e];
}

constexpr uint64_t kDepWaitNs = 2000000000ull;  // bound of the wait for an expert's gate_up outputs

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(map), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// GELU; the tanh form as a * sigmoid(2 y) = a / (1 + e^(-2 y)), y = sqrt(2/pi) (a + 0.044715 a^3),
// which equals 0.5 a (1 + tanh y) (relative error a few 1e-6 at most, below the fp16 rounding of h)
__device__ __forceinline__ float gelu(float a, int act) {
  if (act == 1) return 0.5f * a * (1.f + erff(a * 0.70710678118654752f));
  const float y2 = -1.59576912160573071f * a * fmaf(0.044715f * a, a, 1.f);
  return __fdividef(a, 1.f + __expf(y2));
}

// Warp-uniform bounded wait: every lane polls the barrier (so each acquires the
// phase), the warp leaves together once all lanes have seen it complete, and the
// decision to give up is lane 0's, broadcast.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, int32_t* err, volatile int* abort,
                                          uint64_t limit_ns = kWaitLimitNs) {
  if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    if (__all_sync(0xffffffffu, mbar_try_wait_sleep(bar, parity, kSuspendNs))) return true;
    int give_up = 0;
    if ((threadIdx.x & 31) == 0) {
      give_up = *abort != 0;
      if (!give_up && global_timer_ns() - t0 > limit_ns) {
        atomicExch(err, kStatusTimeout);
        *abort = 1;
        give_up = 1;
      }
    }
    if (__shfl_sync(0xffffffffu, give_up, 0)) return false;
  }
}

// Bounded wait by one thread until a device-scope counter written by other CTAs
// reaches need (acquire: their writes released before the count are visible).
__device__ __forceinline__ bool wait_count(const int32_t* ctr, int need, int32_t* err, volatile int* abort,
                                           uint64_t limit_ns) {
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
    if (v >= need) return true;
    if (*abort || global_timer_ns() - t0 > limit_ns) {
      atomicExch(err, kStatusTimeout);
      *abort = 1;
      return false;
    }
    __nanosleep(256);
  }
}

}  // namespace gemm
}  // namespace moe
