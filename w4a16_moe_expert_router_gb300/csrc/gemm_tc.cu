// gemm_tc.cu -- grouped W4A16 expert GEMMs with inline dequantisation on the
// 5th-generation tensor cores (tcgen05, accumulators in tensor memory).
//
// Model card "srswti/axe-diffusion-ksl-xe", "the kernels we built": the GEMM
// reads packed nibbles and dequantises inline, so HBM carries real 4-bit
// traffic; one launch covers all experts; the activation is folded into the
// first GEMM's epilogue.  One persistent launch runs both projections:
//   gate_up:  a[p][n] = sum_k Wgu[e][n][k] x[t(p)][k]  (64 gate + 64 up rows per item)
//             h[pos(p)][j] = gelu(a[p][j]) * a[p][f+j]  -> fp16, rows in expert-sorted order
//   down:     y[p][i] = sum_j Wd[e][i][j] h[pos(p)][j]   -> fp32, rows by pair id p = t*k + r
// The work list holds every gate_up item followed by every down item.  A down
// item of expert e starts once all gate_up items of e have written their h rows
// (a per-expert counter, bounded wait), so CTAs that run out of gate_up work go
// straight on with down work instead of idling until the slowest CTA finishes.
// The same kernel also runs one projection alone (the separate C entry points).
//
// Arithmetic: the zero-point is split into its nearest integer zr and the rest
// zf = z - zr, and each weight is formed as w = fp16((q - zr) * s - fp16(zf * s)):
// q - zr is exact in fp16, the fused multiply-add rounds once, and the rounding of
// zf * s (|zf| <= 1/2) adds at most a few 1e-6.  The tensor core multiplies w with
// the fp16 activations into an fp32 accumulator that stays in tensor memory for
// the whole contraction.
//
// Roles of the persistent CTA (two per SM, 256 tensor-memory columns each; work
// items = (expert, 128-row block, chunk of <= 32 tokens) taken from a global
// counter, each item self-contained so results do not depend on which CTA ran
// it; the CTA's stages are numbered t = 0, 1, ... across its items):
//   warp 0      producer: claims items one ahead of use; per 64-column stage it
//               writes the decoded item (projection, stage, tokens, block, first
//               row, expert) into the slot header and issues one 1-D bulk copy of the block's
//               stream segment (scale/zero pairs + codes) and one 2-D TMA load
//               (128-byte swizzle, 32 token rows) of the activations into a ring
//               of eight shared-memory slots (mbarrier complete_tx);
//   warps 1-2   MMA issuers (warp 1 also allocates tensor memory): one lane
//               each; issuer i issues the tcgen05.mma of k16 steps 2i and 2i+1 of
//               every stage into its own fp32 accumulator (A = dequantised
//               weights in TMEM, B = activations in SMEM, M = 128 rows, N =
//               tokens rounded up to 16).  Issuing an MMA of this skinny shape
//               occupies the issuing thread for ~50-90 cycles whatever N is, so
//               two issuers share that cost; each commits once per stage
//               (releasing the slot and the TMEM stage) and once per item;
//   warps 3-14  three dequant groups of four warps, one warp per TMEM lane
//               quadrant; group G takes the stages t = G mod 3: each thread owns
//               one GEMM row and writes the row's 64 weights of the stage into
//               the stage's TMEM buffer (two tcgen05.st of 16 columns).  The
//               group that gets an item's last stage reads the row's two
//               accumulators (tcgen05.ld, added in a fixed order) and runs the
//               epilogue -- the gated GELU through a shared-memory exchange of
//               the up rows, or the fp32 row stores of the down projection --
//               while the other group carries on with the next item.
// Every wait is bounded: on expiry the CTA records MOE_W4A16_ERR_TIMEOUT in the
// workspace and all roles leave their loops, drain what is in flight and free
// tensor memory.  No split-K and no atomics on data.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kGroups = 3;                     // dequant groups (four warps each, one per lane quadrant)
constexpr int kDqWarps = 4 * kGroups;
constexpr int kIssuers = 2;                    // MMA issuers: k16 steps {0,1} and {2,3} of every stage
constexpr int kFirstDqWarp = 1 + kIssuers;
constexpr int kThreads = (kFirstDqWarp + kDqWarps) * 32;  // 224
constexpr int kCtasPerSm = 2;
constexpr int kAStages = 4;                    // TMEM stages of dequantised weights
constexpr int kSlots = 8;                      // shared-memory stages in flight per CTA
constexpr int kDBufs = 2;                      // accumulator sets (items alternate)
constexpr int kNMax = kChunkN;                 // 32 tokens per item
constexpr int kACols = 32;                     // 128 rows x 64 fp16 = 32 columns
constexpr int kDCols = kIssuers * kNMax;       // the issuers' fp32 accumulators of one item
constexpr int kDCol0 = kAStages * kACols;      // first accumulator column
constexpr int kTmemCols = 256;
static_assert(kDCol0 + kDBufs * kDCols <= kTmemCols, "TMEM budget");
static_assert(kNMax == 32, "the dequant warps hold 32 accumulator columns");
static_assert(kSlots % kAStages == 0, "stage t uses slot t % kSlots and TMEM stage t % kAStages");
constexpr int kBBoxRows = 32;                  // TMA box: 64 columns x 32 rows = 4 KiB
constexpr int kBBytes = kNMax * 128;           // 4 KiB, 128B-swizzled K-major
constexpr int kSzBytes = kBlockRows * 4;       // 512: (scale, zero) of 128 rows for one group
constexpr int kCodeBytes = kBlockRows * kStageK / 2;  // 4096
constexpr int kCodeOff = kBBytes + 2 * kSzBytes;      // codes always land here
constexpr int kSlotBytes = 10240;                     // multiple of 1024
static_assert(kCodeOff + kCodeBytes <= kSlotBytes && kSlotBytes % 1024 == 0, "slot layout");
constexpr int kXchStride = kNMax + 4;          // floats per exchanged row (bank-conflict padding)
constexpr int kXchBytes = kDBufs * 64 * kXchStride * 4;   // one exchange area per accumulator set
constexpr int kHeaderBytes = 4096;
constexpr int kRingOff = (kHeaderBytes + kXchBytes + 1023) / 1024 * 1024;
constexpr int kSmemBytes = 1024 + kRingOff + kSlots * kSlotBytes;  // +1024 for alignment

struct Proj {
  const uint8_t* w;         // prepared stream of the projection, all experts
  int64_t expert_bytes;     // stream bytes per expert
  int64_t block_bytes;      // stream bytes per 128-row block
  int nblocks;              // blocks per expert
  int K;                    // contraction length (multiple of 64)
  int g;                    // quantisation group along K (32, 64 or 128)
};

struct TcArgs {
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
  int32_t* gu_done;         // [E] gate_up epilogues finished per expert (two per item)
};

// Shared-memory header (at the 1024-aligned base of dynamic shared memory).
struct __align__(8) TcHeader {
  uint64_t slot_full[kSlots];
  uint64_t slot_empty[kSlots];
  uint64_t a_full[kAStages];    // a TMEM stage is written (4 warps)
  uint64_t d_full[kDBufs];      // an item's accumulators are final (one commit per issuer)
  uint64_t d_free[kDBufs];      // the epilogue has read them (4 warps)
  uint64_t drain;
  uint64_t xch_ready[kDBufs];   // the 2 up-row warps of an item have written their rows
  uint64_t xch_done[kDBufs];    // the 2 gate-row warps of an item have read them
  int slot_desc[kSlots];        // stage | tokens << 8 | block << 16 | proj << 24 | last << 25, or -1 at the end
  int slot_pos0[kSlots];        // first expert-sorted row of the item's tokens | expert << 22
  int slot_seq[kSlots];         // the item's sequence number within this CTA
  uint32_t tmem_base;
  int abort;
  int prefix[2][kMaxExperts + 1];  // items of each projection before expert e
  int offs[kMaxExperts + 1];    // expert_offsets, copied once
};
static_assert(sizeof(TcHeader) <= kHeaderBytes, "header fits");

// Groups whose first column lies in stage s (g is 32, 64 or 128).
__device__ __forceinline__ int groups_in_stage(int s, int g) {
  return g == 32 ? 2 : (((s * kStageK) & (g - 1)) == 0 ? 1 : 0);
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
__device__ __forceinline__ void decode_item(int item, const int* prefix, const int* offs, int E, int& expert,
                                            int& blk, int& n_cnt, int& pos0) {
  const int e = expert_of(item, prefix, E);
  const int n_e = offs[e + 1] - offs[e];
  const int nch = (n_e + kChunkN - 1) / kChunkN;
  const int r = item - prefix[e];
  const int c = r % nch;
  expert = e;
  blk = r / nch;
  n_cnt = min(kChunkN, n_e - kChunkN * c);
  pos0 = offs[e] + kChunkN * c;
}

constexpr uint64_t kDepWaitNs = 2000000000ull;  // bound of the wait for an expert's gate_up outputs

// --- tcgen05 wrappers ---------------------------------------------------------

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem desc]^T, kind::f16 (fp16 inputs, fp32 accumulate)
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void tc_st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}

__device__ __forceinline__ void tc_ld16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]),
        "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(taddr));
}

__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row atoms 1024 B apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) | (static_cast<uint64_t>(1) << 16) |
         (static_cast<uint64_t>(1024 >> 4) << 32) | (static_cast<uint64_t>(1) << 46) | (static_cast<uint64_t>(2) << 61);
}

// Instruction descriptor of kind::f16: fp16 A and B (K-major), fp32 D, M = 128, N = n.
__device__ __forceinline__ uint32_t f16_idesc(int n) {
  return (1u << 4) | (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(kBlockRows >> 4) << 24);
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(map), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// Per-(row, group) constants of the dequantiser: the zero-point split into its
// nearest integer zr and the rest zf = z - zr (exact in fp16), so that
// (q - z) * s = (q - zr) * s - zf * s.
struct DqGroup {
  __half2 zb1024;  // 1024 + zr (exact)
  __half2 zb64;    // 64 + zr (exact)
  __half2 s;       // scale
  __half2 c;       // -fp16(zf * s)
};
__device__ __forceinline__ DqGroup dq_group(__half2 s, __half2 z) {
  const __half2 zr = h2rint(z);
  const __half2 zf = __hsub2(z, zr);
  DqGroup g;
  g.zb1024 = __hadd2(zr, bits_h2(0x64006400u));
  g.zb64 = __hadd2(zr, bits_h2(0x54005400u));
  g.s = s;
  g.c = __hneg2(__hmul2(zf, s));
  return g;
}

// 8 codes of one row (nibbles in column order 0,2,4,6,1,3,5,7) -> four f16x2 weights
// w = fp16((q - zr) * s - fp16(zf * s)) for columns (k, k+1), (k+2, k+3), (k+4, k+5),
// (k+6, k+7).  (1024 + q) and (64 + q) come from OR-ing exponent bits onto the
// nibbles; one fp16 subtract of (1024 + zr) or (64 + zr) gives q - zr exactly (both
// operands are integers in fp16), and one fused multiply-add rounds the weight once.
__device__ __forceinline__ void dequant_row8(uint32_t w, const DqGroup& g, uint32_t* out) {
  const uint32_t w8 = w >> 8;
  out[0] = h2_bits(__hfma2(__hsub2(bits_h2(and_or(w, 0x000f000fu, 0x64006400u)), g.zb1024), g.s, g.c));
  out[1] = h2_bits(__hfma2(__hsub2(bits_h2(and_or(w, 0x00f000f0u, 0x54005400u)), g.zb64), g.s, g.c));
  out[2] = h2_bits(__hfma2(__hsub2(bits_h2(and_or(w8, 0x000f000fu, 0x64006400u)), g.zb1024), g.s, g.c));
  out[3] = h2_bits(__hfma2(__hsub2(bits_h2(and_or(w8, 0x00f000f0u, 0x54005400u)), g.zb64), g.s, g.c));
}

__device__ __forceinline__ float gelu(float a, int act) {
  if (act == 1) return 0.5f * a * (1.f + erff(a * 0.70710678118654752f));
  return 0.5f * a * (1.f + tanhf(0.79788456080286536f * (a + 0.044715f * a * a * a)));
}

// Bounded wait by one thread that also gives up once another role of this CTA has.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, const TcArgs& a, volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait_sleep(bar, parity, kSuspendNs)) {
    if (*abort) return false;
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      atomicExch(a.err, kStatusTimeout);
      *abort = 1;
      return false;
    }
  }
  return true;
}

// Warp-uniform bounded wait: every lane polls the barrier (so each acquires the
// phase), the warp leaves together once all lanes have seen it complete, and the
// decision to give up is lane 0's, broadcast, so a warp never splits before a
// warp-collective instruction.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const TcArgs& a, volatile int* abort) {
  if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    if (__all_sync(0xffffffffu, mbar_try_wait_sleep(bar, parity, kSuspendNs))) return true;
    int give_up = 0;
    if ((threadIdx.x & 31) == 0) {
      give_up = *abort != 0;
      if (!give_up && global_timer_ns() - t0 > kWaitLimitNs) {
        atomicExch(a.err, kStatusTimeout);
        *abort = 1;
        give_up = 1;
      }
    }
    if (__shfl_sync(0xffffffffu, give_up, 0)) return false;
  }
}

__global__ void __launch_bounds__(kThreads, kCtasPerSm)
    expert_gemm_tc_kernel(const TcArgs a, const __grid_constant__ CUtensorMap map_x,
                          const __grid_constant__ CUtensorMap map_h) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  TcHeader& H = *reinterpret_cast<TcHeader*>(smem);
  float* xch_all = reinterpret_cast<float*>(smem + kHeaderBytes);
  uint8_t* ring = smem + kRingOff;
  volatile int* abort = &H.abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(smem_addr(&H.slot_full[i]), 1);
      mbar_init(smem_addr(&H.slot_empty[i]), 4 + kIssuers);  // the stage's 4 dequant warps + 2 commits
    }
    for (int i = 0; i < kAStages; ++i) mbar_init(smem_addr(&H.a_full[i]), 4);
    for (int i = 0; i < kDBufs; ++i) {
      mbar_init(smem_addr(&H.xch_ready[i]), 2);
      mbar_init(smem_addr(&H.xch_done[i]), 2);
    }
    for (int i = 0; i < kDBufs; ++i) {
      mbar_init(smem_addr(&H.d_full[i]), kIssuers);
      mbar_init(smem_addr(&H.d_free[i]), 4);
    }
    mbar_init(smem_addr(&H.drain), kIssuers);
    H.abort = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(&H.tmem_base)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  // everything above is set-up; the routing arrays, the row copy and h come from earlier launches
  grid_dependents_launch();
  grid_dependency_wait();
  if (warp == 2) {  // items per expert = blocks * ceil(n_e / 32); exclusive scans, 8 experts per lane
    for (int pj = 0; pj < 2; ++pj) {
      const int nb = a.p[pj].nblocks;
      int loc[8], sum = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int e = lane * 8 + j;
        loc[j] = sum;
        if (e < a.E) sum += nb * ((a.offsets[e + 1] - a.offsets[e] + kChunkN - 1) / kChunkN);
      }
      int incl = sum;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
      }
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (lane * 8 + j < a.E) H.prefix[pj][lane * 8 + j] = incl - sum + loc[j];
      if (lane == 31) H.prefix[pj][a.E] = incl;
    }
    for (int e = lane; e <= a.E; e += 32) H.offs[e] = a.offsets[e];
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = H.tmem_base;
  // the launch's work list: [gate_up items][down items], restricted to projections first..last
  const int total0 = a.first == 0 ? H.prefix[0][a.E] : 0;
  const int total = total0 + (a.last == 1 ? H.prefix[1][a.E] : 0);

  if (warp == 0) {
    // ------------------------------------------------------------------ producer
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(&map_x) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(&map_h) : "memory");
    }
    int t = 0, seq = 0, sentinels = 0;
    // every weight byte is read once: it leaves L2 first, so that h, y and the token rows stay
    const uint64_t w_policy = l2_evict_first_policy();
    uint32_t issued_mask = 0;   // slots whose last phase carried copies
    uint32_t issued_par = 0;    // parity of that phase, one bit per slot
    bool ok = true;
    // the next item is claimed one item ahead, so the atomic's latency hides behind this item's stages
    int next = 0;
    if (lane == 0) next = atomicAdd(a.counter, 1);
    while (ok && sentinels < kGroups) {
      const int item = __shfl_sync(0xffffffffu, next, 0);
      const bool done = item >= total;
      if (lane == 0 && !done) next = atomicAdd(a.counter, 1);
      const int pj = (a.first == 0 && item < total0) ? 0 : 1;
      const Proj& P = a.p[pj];
      int e = 0, blk = 0, n_cnt = 0, pos0 = 0;
      if (!done) decode_item(pj == 0 ? item : item - total0, H.prefix[pj], H.offs, a.E, e, blk, n_cnt, pos0);
      const int nst = P.K / kStageK;
      if (!done && pj == 1 && a.first == 0 && lane == 0) {
        // a down item reads the h rows of its expert: wait until every gate_up item of the
        // expert has written them (two epilogue warps per item report)
        const int need = 2 * a.p[0].nblocks * ((H.offs[e + 1] - H.offs[e] + kChunkN - 1) / kChunkN);
        const uint64_t t0 = global_timer_ns();
        for (;;) {
          int v;
          asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(a.gu_done + e) : "memory");
          if (v >= need) break;
          if (*abort || global_timer_ns() - t0 > kDepWaitNs) {
            atomicExch(a.err, kStatusTimeout);
            *abort = 1;
            ok = false;
            break;
          }
          __nanosleep(256);
        }
        // the TMA loads below read those rows through the async proxy
        asm volatile("fence.proxy.async.global;" ::: "memory");
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok) break;
      const CUtensorMap* bmap = pj == 0 ? &map_x : &map_h;
      const uint8_t* wsrc =
          P.w + static_cast<int64_t>(e) * P.expert_bytes + static_cast<int64_t>(blk) * P.block_bytes;
      const uint8_t* sz_src = wsrc;  // (scale, zero) segment of the group in progress
      // the end of the work list is one sentinel stage per group
      const int stages = done ? kGroups : nst;
      for (int s = 0; s < stages && ok; ++s, ++t) {
        const int slot = t % kSlots;
        const uint32_t par = static_cast<uint32_t>(t / kSlots) & 1u;
        const uint32_t full = smem_addr(&H.slot_full[slot]);
        ok = warp_wait(smem_addr(&H.slot_empty[slot]), par ^ 1u, a, abort);
        if (!ok) break;
        if (lane == 0) {
          H.slot_desc[slot] =
              done ? -1 : (s | (n_cnt << 8) | (blk << 16) | (pj << 24) | ((s == nst - 1 ? 1 : 0) << 25));
          H.slot_pos0[slot] = pos0 | (e << 22);
          H.slot_seq[slot] = seq;
          if (done) {
            issued_mask &= ~(1u << slot);  // this phase carries no copies
            mbar_arrive(full);
            ++sentinels;
          } else {
            const int ngrp = groups_in_stage(s, P.g);
            const uint32_t seg = kCodeBytes + kSzBytes * ngrp;
            const uint32_t dst = smem_addr(ring + slot * kSlotBytes);
            if (ngrp > 0) {
              mbar_arrive_expect_tx(full, seg + kBBoxRows * 128);
              bulk_g2s_hint(dst + kCodeOff - kSzBytes * ngrp, wsrc, seg, full, w_policy);
              sz_src = wsrc;
            } else {
              // a stage inside a group (groups of 128) gets a copy of the group's (scale, zero)
              // pairs (from L2) so that every slot is self-contained
              mbar_arrive_expect_tx(full, kSzBytes + seg + kBBoxRows * 128);
              bulk_g2s(dst + kCodeOff - kSzBytes, sz_src, kSzBytes, full);
              bulk_g2s_hint(dst + kCodeOff, wsrc, seg, full, w_policy);
            }
            tma_load_2d(dst, bmap, s * kStageK, pos0, full);
            wsrc += seg;
            issued_mask |= 1u << slot;
            issued_par = (issued_par & ~(1u << slot)) | (par << slot);
          }
        }
        sentinels = __shfl_sync(0xffffffffu, sentinels, 0);
        __syncwarp();
      }
      ++seq;
    }
    // drain: every bulk copy this warp issued has landed before the CTA can exit
    if (lane == 0)
      for (int i = 0; i < kSlots; ++i)
        if ((issued_mask >> i) & 1u) mbar_wait(smem_addr(&H.slot_full[i]), (issued_par >> i) & 1u, a.err);
  } else if (warp <= kIssuers) {
    // ------------------------------------------------------------------ MMA issuers
    if (lane == 0) {
      const int r = warp - 1;                              // issuer 0..1
      const int k0 = 2 * r;                                // its two k16 steps of every stage
      // descriptor of slot 0's activation tile; slot i adds i * kSlotBytes / 16, k16 step kk adds 2 * kk
      const uint64_t desc0 = sw128_desc(smem_addr(ring)) + 2 * k0;
      uint32_t idesc = f16_idesc(16);
      bool ok = true;
      int t = 0;
      while (ok) {
        // first stage of an item (or the end of the work list): its header gives the item
        {
          const int ast = t % kAStages;
          ok = wait_or_abort(smem_addr(&H.a_full[ast]), static_cast<uint32_t>(t / kAStages) & 1u, a, abort);
          if (!ok) break;
        }
        const int desc = H.slot_desc[t % kSlots];
        if (desc < 0) break;  // the end of the work list
        const int seq = H.slot_seq[t % kSlots];
        const int nst = a.p[(desc >> 24) & 1].K / kStageK;
        const int b = seq & 1;
        const uint32_t dcol = tmem + kDCol0 + b * kDCols + r * kNMax;
        idesc = f16_idesc((((desc >> 8) & 0xff) + 15) & ~15);
        // the accumulators are free once the epilogue two items back has read them
        ok = wait_or_abort(smem_addr(&H.d_free[b]), (static_cast<uint32_t>(seq >> 1) & 1u) ^ 1u, a, abort);
        for (int s = 0; s < nst && ok; ++s, ++t) {
          const int ast = t % kAStages, slot = t % kSlots;
          // the stage is in TMEM (the first stage's wait is above)
          if (s > 0) {
            ok = wait_or_abort(smem_addr(&H.a_full[ast]), static_cast<uint32_t>(t / kAStages) & 1u, a, abort);
            if (!ok) break;
          }
          tc_fence_after();
          const uint64_t bdesc = desc0 + static_cast<uint64_t>(slot * (kSlotBytes >> 4));
          const uint32_t acol = tmem + ast * kACols + 8 * k0;
          tc_mma(dcol, acol, bdesc, idesc, s > 0 ? 1u : 0u);
          tc_mma(dcol, acol + 8, bdesc + 2, idesc, 1u);
          tc_commit(smem_addr(&H.slot_empty[slot]));  // slot and (for the group) TMEM stage reusable
        }
        if (ok) tc_commit(smem_addr(&H.d_full[b]));
      }
      // every MMA issued has completed before tensor memory is freed
      tc_commit(smem_addr(&H.drain));
      mbar_wait(smem_addr(&H.drain), 0, a.err);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ dequant groups
    const int grp = (warp - kFirstDqWarp) >> 2;
    const int q = warp & 3;              // TMEM lane quadrant (rows 32q .. 32q+31)
    const int m = 32 * q + lane;         // GEMM row within the 128-row block
    const uint32_t lane_bits = static_cast<uint32_t>(32 * q) << 16;
    DqGroup g0, g1;  // the dequantiser constants of the stage's group(s) for row m
    int n_cnt = 0, pos0 = 0, blk = 0;
    bool ok = true;
    // A gate warp of a launch that also holds down items reports each finished item
    // to its expert's counter (a device-scope release after its h stores), but one
    // stage late, when those stores have long completed and the fence costs little;
    // or at once when the next stage is not there yet, since the producer may be
    // waiting for exactly this count before it issues more.
    int sig_e = -1;
    auto signal = [&]() {
      __threadfence();
      __syncwarp();
      if (lane == 0) asm volatile("red.release.gpu.global.add.s32 [%0], 1;" ::"l"(a.gu_done + sig_e) : "memory");
      sig_e = -1;
    };
    for (int t = grp; ok; t += kGroups) {
      const int slot = t % kSlots;
      const uint32_t full = smem_addr(&H.slot_full[slot]);
      const uint32_t fpar = static_cast<uint32_t>(t / kSlots) & 1u;
      if (sig_e >= 0 && !__all_sync(0xffffffffu, mbar_test_wait(full, fpar))) signal();
      ok = warp_wait(full, fpar, a, abort);
      if (!ok) break;
      const int desc = H.slot_desc[slot];
      const int seq = H.slot_seq[slot];
      if (desc < 0) {  // end of the work list: pass it on to the issuers, which learn of stages via a_full
        if (sig_e >= 0) signal();
        // (only after the stage that last used this TMEM stage was consumed, so a_full never runs a
        // phase ahead)
        if (t >= kAStages) {
          const int tp = t - kAStages;
          ok = warp_wait(smem_addr(&H.slot_empty[tp % kSlots]), static_cast<uint32_t>(tp / kSlots) & 1u, a, abort);
          if (!ok) break;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&H.a_full[t % kAStages]));
        break;
      }
      const int s = desc & 0xff;
      n_cnt = (desc >> 8) & 0xff;
      blk = (desc >> 16) & 0xff;
      const int pj = (desc >> 24) & 1;
      const int aux = H.slot_pos0[slot];
      pos0 = aux & ((1 << 22) - 1);
      const int e = aux >> 22;
      const uint8_t* st = ring + slot * kSlotBytes;
      // (scale, zero) of row m for the group(s) of this stage (every slot carries them)
      const int ngrp = max(groups_in_stage(s, a.p[pj].g), 1);
      const uint32_t* sz = reinterpret_cast<const uint32_t*>(st + kCodeOff - kSzBytes * ngrp);
      // this row's 64 codes: two 16-byte halves, [half][row][16 B]; with groups of 32
      // the second half belongs to the stage's second group
      const uint4 c0 = *reinterpret_cast<const uint4*>(st + kCodeOff + m * 16);
      const uint4 c1 = *reinterpret_cast<const uint4*>(st + kCodeOff + kBlockRows * 16 + m * 16);
      {
        const __half2 v0 = bits_h2(sz[m]);
        g0 = dq_group(__low2half2(v0), __high2half2(v0));
        if (ngrp > 1) {
          const __half2 v1 = bits_h2(sz[kBlockRows + m]);
          g1 = dq_group(__low2half2(v1), __high2half2(v1));
        } else {
          g1 = g0;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&H.slot_empty[slot]));  // codes and scales are in registers
      const int ast = t % kAStages;
      uint32_t w[16];
      dequant_row8(c0.x, g0, w + 0);
      dequant_row8(c0.y, g0, w + 4);
      dequant_row8(c0.z, g0, w + 8);
      dequant_row8(c0.w, g0, w + 12);
      if (t >= kAStages) {
        // the TMEM stage is free once the MMAs of the stage that used it last (t - kAStages)
        // have completed: that stage's slot is released by the issuers' commits (and our arrivals)
        const int tp = t - kAStages;
        ok = warp_wait(smem_addr(&H.slot_empty[tp % kSlots]), static_cast<uint32_t>(tp / kSlots) & 1u, a, abort);
        if (!ok) break;
      }
      tc_fence_after();
      tc_st16(tmem + lane_bits + ast * kACols, w);
      dequant_row8(c1.x, g1, w + 0);
      dequant_row8(c1.y, g1, w + 4);
      dequant_row8(c1.z, g1, w + 8);
      dequant_row8(c1.w, g1, w + 12);
      tc_st16(tmem + lane_bits + ast * kACols + 16, w);
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&H.a_full[ast]));
      if (sig_e >= 0) signal();
      if ((desc >> 25) & 1) {  // the item's last stage
        // ------------------------------------------------------------ accumulators
        const int b = seq & 1;
        ok = warp_wait(smem_addr(&H.d_full[b]), static_cast<uint32_t>(seq >> 1) & 1u, a, abort);
        if (!ok) break;
        tc_fence_after();
        const uint32_t dcol = tmem + lane_bits + kDCol0 + b * kDCols;
        // the accumulators in halves of 16 token columns (a half past the item's tokens is
        // skipped: the MMA did not write it); each column is the accumulator of k16 steps
        // 0-1 plus that of steps 2-3, in this order
        if (pj == 0) {
          // rows 0..63 gate j = 64*blk + m, rows 64..127 up j = 64*blk + m - 64; the up rows
          // reach the gate rows' threads through the exchange area of the item's accumulator
          // set (bounded mbarriers, not a named barrier, so a timed-out warp cannot strand the
          // others).  A CTA's gate_up items come first in its sequence, so item seq is the
          // (seq >> 1)-th user of area seq & 1.
          float* xch = xch_all + b * 64 * kXchStride;
          const uint32_t xphase = static_cast<uint32_t>(seq >> 1) & 1u;
          ok = q >= 2 ? warp_wait(smem_addr(&H.xch_done[b]), xphase ^ 1u, a, abort)  // previous reads finished
                      : warp_wait(smem_addr(&H.xch_ready[b]), xphase, a, abort);
          if (!ok) break;
          const int j = 64 * blk + m;
          for (int c = 0; c < kNMax && c < n_cnt; c += 16) {
            uint32_t v0[16], v1[16];
            tc_ld16(dcol + c, v0);
            tc_ld16(dcol + kNMax + c, v1);
            tc_wait_ld();
            if (q >= 2) {
              float4* dst = reinterpret_cast<float4*>(xch + (m - 64) * kXchStride + c);
#pragma unroll
              for (int i = 0; i < 4; ++i)
                dst[i] = make_float4(__uint_as_float(v0[4 * i]) + __uint_as_float(v1[4 * i]),
                                     __uint_as_float(v0[4 * i + 1]) + __uint_as_float(v1[4 * i + 1]),
                                     __uint_as_float(v0[4 * i + 2]) + __uint_as_float(v1[4 * i + 2]),
                                     __uint_as_float(v0[4 * i + 3]) + __uint_as_float(v1[4 * i + 3]));
            } else {
              const float4* up4 = reinterpret_cast<const float4*>(xch + m * kXchStride + c);
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const float4 u = up4[i];
                const float up[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                  const int n = c + 4 * i + cc;
                  const float g = __uint_as_float(v0[4 * i + cc]) + __uint_as_float(v1[4 * i + cc]);
                  if (n < n_cnt)
                    a.h[static_cast<size_t>(pos0 + n) * a.f + j] =
                        __half_as_ushort(__float2half_rn(gelu(g, a.act) * up[cc]));
                }
              }
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(smem_addr(&H.d_free[b]));  // the item after next may accumulate here
            mbar_arrive(smem_addr(q >= 2 ? &H.xch_ready[b] : &H.xch_done[b]));
          }
          if (q < 2 && a.last == 1) sig_e = e;  // reported one stage later (see signal above)
        } else {
          const int i_row = kBlockRows * blk + m;
          for (int c = 0; c < kNMax && c < n_cnt; c += 16) {
            uint32_t v0[16], v1[16];
            tc_ld16(dcol + c, v0);
            tc_ld16(dcol + kNMax + c, v1);
            tc_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i)
              if (c + i < n_cnt)
                a.y_out[static_cast<size_t>(a.pair_list[pos0 + c + i]) * a.d + i_row] =
                    __uint_as_float(v0[i]) + __uint_as_float(v1[i]);
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_addr(&H.d_free[b]));  // the item after next may accumulate here
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
  }
  // The last CTA to finish clears the work counter for the next launch on this
  // workspace: by then every CTA has seen the list exhausted and claims no more.
  if (tid == 0 && atomicAdd(a.done_ctas, 1) == static_cast<int>(gridDim.x) - 1) {
    *a.counter = 0;
    *a.done_ctas = 0;
  }
}

// Token rows of every (token, expert) pair, copied in expert-sorted order:
// xs[pos] = x[pair_list[pos] / k].  One warp per row, 16-byte accesses.  Also
// clears the per-expert gate_up counters that the GEMM launch after it counts up.
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint16_t* __restrict__ x,
                                                          const int32_t* __restrict__ pair_list, int P, int k, int d,
                                                          uint16_t* __restrict__ xs, int32_t* __restrict__ gu_done,
                                                          int E) {
  grid_dependents_launch();
  grid_dependency_wait();  // pair_list of the routing launch
  if (blockIdx.x == 0)
    for (int e = threadIdx.x; e < E; e += blockDim.x) gu_done[e] = 0;
  const int pos = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (pos >= P) return;
  const int t = pair_list[pos] / k;
  const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<size_t>(t) * d);
  uint4* dst = reinterpret_cast<uint4*>(xs + static_cast<size_t>(pos) * d);
  // up to 8 loads in flight per lane before the first store (d <= 8192: 32 per lane)
  for (int i0 = 0; i0 < d / 8; i0 += 32 * 8) {
    uint4 v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int i = i0 + j * 32 + lane;
      if (i < d / 8) v[j] = src[i];
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int i = i0 + j * 32 + lane;
      if (i < d / 8) dst[i] = v[j];
    }
  }
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

// 2-D tensor map over rows x cols fp16 (row-major), box 64 columns x 32 rows, 128B swizzle.
bool make_row_map(CUtensorMap* map, const void* base, int64_t rows, int64_t cols) {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (!g_encode) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
  const cuuint32_t box[2] = {kStageK, kBBoxRows};
  const cuuint32_t estr[2] = {1, 1};
  return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t init_gemm_kernels(int* blocks_per_sm) {
  const void* fn = reinterpret_cast<const void*>(expert_gemm_tc_kernel);
  cudaError_t err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (err != cudaSuccess) return err;
  err = cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  if (err != cudaSuccess) return err;
  // Two CTAs per SM: shared memory, registers (launch bounds) and tensor memory
  // (2 x 256 of 512 columns) all allow exactly two.
  *blocks_per_sm = kCtasPerSm;
  return cudaSuccess;
}

cudaError_t launch_expert_gemm(int which, const Dims& s, const uint16_t* x, const int32_t* expert_offsets,
                               const int32_t* pair_list, const uint8_t* w_gate_up, const uint8_t* w_down,
                               const GemmWorkspace& ws, int grid, cudaStream_t st) {
  const int P = static_cast<int>(s.pairs());
  TcArgs a{};
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
  if (which == 0 || a.first > a.last) return cudaErrorInvalidValue;
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
  if (which & kGemmGateUp) {
    // the token rows are first copied in expert order
    cudaError_t err = launch_pdl(gather_rows_kernel, dim3((P + 7) / 8), dim3(256), 0, st, x, pair_list, P, s.k, s.d,
                                 ws.xs, ws.gu_done, s.E);
    if (err != cudaSuccess) return err;
  }
  CUtensorMap map_x, map_h;
  if (!make_row_map(&map_x, ws.xs, P, s.d) || !make_row_map(&map_h, ws.h, P, s.f)) return cudaErrorInvalidValue;
  return launch_pdl(expert_gemm_tc_kernel, dim3(grid), dim3(kThreads), kSmemBytes, st, a, map_x, map_h);
}

}  // namespace moe
