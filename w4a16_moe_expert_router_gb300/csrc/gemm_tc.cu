// gemm_tc.cu -- grouped W4A16 expert GEMMs on the 5th-generation tensor cores:
// CUDA-core warps dequantise the weights straight into tensor memory, and
// tcgen05.mma multiplies them with token tiles that TMA brings into shared memory.
//
// Model card "srswti/axe-diffusion-ksl-xe", "the kernels we built": the GEMM
// reads packed nibbles and dequantises inline, so HBM carries real 4-bit
// traffic; one launch covers all experts; the activation is folded into the
// first GEMM's epilogue.  One persistent launch runs both projections:
//   gate_up:  a[p][n] = sum_k Wgu[e][n][k] x[t(p)][k]  (64 gate + 64 up rows per item)
//             h[pos(p)][j] = gelu(a[p][j]) * a[p][f+j]  -> fp16, rows in expert-sorted order
//   down:     y[p][i] = sum_j Wd[e][i][j] h[pos(p)][j]   -> fp32, rows by pair id p = t*k + r
// Work items are (projection, expert, 128-row block, chunk of <= 32 tokens) over
// the whole contraction, gate_up items first; a down item of expert e starts once
// all gate_up items of e have written their h rows (a per-expert counter, bounded
// wait).  Items are self-contained (no split-K, no atomics on data), so results do
// not depend on which CTA ran which item.
//
// Shape of the work on GB300.  An expert sees ~16 tokens of a 256-token canvas,
// so the MMA is M = 128 weight rows by N = 16 or 32 tokens by K = 16.  Measured on
// this GPU: a warp can issue such a tcgen05.mma only every ~70-150 cycles (its
// tensor work takes ~10-20) and a tcgen05.commit costs about as much, while
// several issuing warps overlap; an mbarrier wait or arrive costs a thread ~100
// cycles even when it does not block, and a single thread issuing every bulk
// copy of the SM cannot keep up with the dequantisers; the fp16 dequant arithmetic
// runs at half the FMA rate.  So the work is cut into three independent pipes:
// stage t of the CTA's stage sequence (128 contraction columns of one item) is
// loaded by producer t % 3, dequantised by team t % 3 and multiplied by issuer
// t % 3 into that issuer's fp32 accumulator.  Each class of an item's stages
// (s = c, c + 3, ...) thus accumulates in one accumulator in stage order, and the
// epilogue sums the three classes in a fixed order, so the result does not depend
// on which CTA ran the item or where it fell in the CTA's sequence.  The
// dequantised weights (the A operand, 128 rows x 128 fp16 per stage) go to tensor
// memory, not shared memory: the MMA would otherwise spend more shared-memory
// bandwidth reading A than the CUDA cores spend writing it.
//
// Arithmetic: the zero-point is split into its nearest integer zr and the rest
// zf = z - zr, and each weight is formed as w = fp16((q - zr) * s - fp16(zf * s)):
// (1024 + q) and (64 + q) come from OR-ing exponent bits onto the nibbles, one fp16
// subtract of (1024 + zr) or (64 + zr) gives q - zr exactly, one fused multiply-add
// rounds the weight once.  The affine format (w = q s + b) uses the bare offsets
// and b in place of -fp16(zf s).  The tensor core accumulates w x in fp32.
//
// Roles of the persistent CTA (one per SM: its tensor memory holds six A stages,
// two per pipe, and the three accumulators):
//   warps 0-2   producers: producer j fills the slots of the stages t = j, j + 3,
//               ... (four slots per pipe): one bulk copy of the stage's weight segment
//               ((scale, second) pairs of its groups, then 128 rows x 128 codes)
//               and two 2-D TMA loads of the token tile (32 rows x 64 fp16 each,
//               128-byte swizzle).  Producer 0 also claims the work items and
//               keeps a queue of them filled ahead;
//   warps 3-5   MMA issuers: issuer r takes the stages t = r, r + 3, ... (eight
//               MMAs of 16 columns into its accumulator, then one commit that
//               frees the A stage and one that frees the token tile), and commits
//               once more at the end of each item;
//   warps 6-9   epilogue, one per lane quarter: once the item's MMAs are done it
//               sums the accumulators for its 32 rows, frees them for the next
//               item, and writes h (the gated GELU: gate rows sit in lanes 0-15
//               of a quarter and their up rows in lanes 16-31) or the fp32 rows
//               of y;
//   warps 10-21 dequantisers, three teams of one warp per lane quarter; team j
//               takes the stages t = j, j + 3, ...: each thread owns one weight
//               row of the stage, turns sixteen words of codes into 128 fp16
//               weights and stores them to tensor memory (four tcgen05.st).
// Every wait is bounded: on expiry the CTA records MOE_W4A16_ERR_TIMEOUT in the
// workspace, all roles leave their loops, the issuers wait for their MMAs, the
// copies in flight are drained and tensor memory is freed.
#include <cuda.h>
#include <cuda_fp16.h>

#include "gemm_common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

using gemm::Args;

constexpr int kCols = 128;                              // contraction columns per stage (the last may have 64)
constexpr int kPipes = 3;                               // stage t: producer, dequant team and issuer t % 3
constexpr int kSlots = 12;                              // shared-memory stages in flight (4 per pipe)
constexpr int kAStages = 6;                             // tensor-memory stages of dequantised weights (2 per pipe)
// Every ring is a multiple of the pipe count, so a slot or an A stage is only ever
// reused by its own pipe, in stage order: a wait on its barrier is never more than
// one phase behind, which the parity test of an mbarrier needs.
static_assert(kSlots % kPipes == 0 && kAStages % kPipes == 0, "rings are per-pipe");
constexpr int kEpiWarps = 4;                            // epilogue warps, one per lane quarter
constexpr int kDqWarps = 4 * kPipes;                    // a dequant team per pipe, one warp per lane quarter
constexpr int kFirstIssuer = kPipes;                    // warps 0-2 producers (warp 0 also fills the item queue)
constexpr int kFirstEpi = kFirstIssuer + kPipes;        // 6
constexpr int kFirstDq = kFirstEpi + kEpiWarps;         // 10
constexpr int kThreads = (kFirstDq + kDqWarps) * 32;    // 704
constexpr int kCtasPerSm = 1;
constexpr int kQueue = 4;                               // item descriptors in flight per CTA
constexpr int kConsumers = kPipes + kPipes + kEpiWarps + kDqWarps;  // warps that read each queue entry
constexpr int kNMax = kChunkN;                          // tokens per item; the MMA's N is 16 or 32
constexpr int kACols = kCols / 2;                       // tensor-memory columns of one A stage: 64
constexpr int kAccCol0 = kAStages * kACols;             // 384: the issuers' accumulators, kNMax columns each
constexpr int kTmemCols = 512;                          // the whole tensor memory of the SM
static_assert(kAccCol0 + kPipes * kNMax <= kTmemCols && kCtasPerSm == 1, "one CTA per SM holds tensor memory");
static_assert(kNMax == 32 && kRowBoxRows == kNMax, "items of at most 32 tokens, one token box per 64 columns");
constexpr int kBoxBytes = kRowBoxRows * 128;            // token box: 32 rows x 64 fp16 (4 KiB)
constexpr int kBBytes = 2 * kBoxBytes;                  // a stage's token tile
constexpr int kSzRowBytes = kBlockRows * 4;             // (scale, second) pairs of 128 rows, one group
constexpr int kCodeOff = kBBytes + 4 * kSzRowBytes;     // the codes always land here (up to 4 groups before)
constexpr int kCodeBytes = kBlockRows * kCols / 2;      // 8192
constexpr int kSlotBytes = kCodeOff + kCodeBytes;       // 18432, a multiple of 1024 (token tiles stay aligned)
static_assert(kSlotBytes % 1024 == 0, "slot alignment");
constexpr int kHeaderBytes = 4096;
constexpr int kSmemBytes = 1024 + kHeaderBytes + kSlots * kSlotBytes;  // +1024 for alignment

struct __align__(8) TcHeader {
  uint64_t slot_full[kSlots];    // the stage's weight segment and token tile landed (transaction bytes)
  uint64_t codes_empty[kSlots];  // the 4 dequant warps of the stage's team have read its weight segment
  uint64_t slot_free[kSlots];    // the stage's MMAs completed: its token tile may be overwritten (commit)
  uint64_t a_full[kAStages];     // the 4 dequant warps of the stage's team wrote the A stage
  uint64_t a_empty[kAStages];    // the MMAs that read the A stage completed (commit)
  uint64_t acc_full;             // every issuer's MMAs of the item completed (one commit each)
  uint64_t acc_free;             // the 4 epilogue warps have read the accumulators
  uint64_t drain[kPipes];        // per issuer: every MMA it issued completed
  uint64_t item_full[kQueue];    // queue entry written
  uint64_t item_empty[kQueue];   // every consumer warp is done with the item
  int item_desc[kQueue][3];      // {proj | tokens << 8 | block << 16 (or -1 at the end), expert, first row}
  uint32_t tmem_base;
  int abort;
  int slot_t[kSlots];            // the last stage whose copies went into each slot (-1: none)
  int prefix[2][kMaxExperts + 1];  // items of each projection before expert e
  int offs[kMaxExperts + 1];       // expert_offsets, copied once
};
static_assert(sizeof(TcHeader) <= kHeaderBytes, "header fits");

// Stages of a contraction of K columns and the stream bytes of one full stage.
__device__ __forceinline__ int num_stages(int K) { return (K + kCols - 1) / kCols; }
__device__ __forceinline__ int groups_per_stage(int width, int g) { return width >= g ? width / g : 1; }
__device__ __forceinline__ int64_t full_stage_bytes(int g) { return kCodeBytes + groups_per_stage(kCols, g) * kSzRowBytes; }

// Dequantiser constants of one row and group, each in both halves of an f16x2.
struct Dq {
  __half2 zb1;   // 1024 + zr (exact)
  __half2 zb64;  // 64 + zr (exact)
  __half2 s;     // scale
  __half2 c;     // -fp16(zf * s) (asymmetric) or the bias b (affine)
};
// v = (scale, second value) as an fp16 pair (scale in the low half).  For 0 <= z <= 16,
// fp16(z + 1024) is 1024 + zr with zr = z rounded to the nearest integer (ties to
// even): fp16 has unit spacing in [1024, 2048).
template <bool AF>
__device__ __forceinline__ Dq dq_const(uint32_t v) {
  const __half2 s = __low2half2(bits_h2(v)), z = __high2half2(bits_h2(v));
  Dq k;
  k.s = s;
  if (AF) {
    k.zb1 = bits_h2(0x64006400u);
    k.zb64 = bits_h2(0x54005400u);
    k.c = z;
  } else {
    k.zb1 = __hadd2(z, bits_h2(0x64006400u));
    const __half2 zr = __hsub2(k.zb1, bits_h2(0x64006400u));
    k.c = __hmul2(__hsub2(zr, z), s);                 // (zr - z) s = -(zf s), rounded once
    k.zb64 = __hsub2(k.zb1, bits_h2(0x63806380u));    // (1024 + zr) - 960
  }
  return k;
}

// One word of codes -> the fp16 weights of 8 consecutive columns of the row, as four
// f16x2 (columns (0,1), (2,3), (4,5), (6,7)).  Nibble i of the word (bits 4i..4i+3)
// holds column 0, 2, 4, 6, 1, 3, 5, 7 for i = 0..7: the masks pick nibbles (0,4),
// (1,5), then, after a shift by 8, (2,6) and (3,7), each pair already in column order.
__device__ __forceinline__ void dequant8(uint32_t w, const Dq& k, uint32_t* o) {
  const uint32_t w8 = w >> 8;
  o[0] = h2_bits(__hfma2(__hsub2(bits_h2(and_or(w, 0x000f000fu, 0x64006400u)), k.zb1), k.s, k.c));
  o[1] = h2_bits(__hfma2(__hsub2(bits_h2(and_or(w, 0x00f000f0u, 0x54005400u)), k.zb64), k.s, k.c));
  o[2] = h2_bits(__hfma2(__hsub2(bits_h2(and_or(w8, 0x000f000fu, 0x64006400u)), k.zb1), k.s, k.c));
  o[3] = h2_bits(__hfma2(__hsub2(bits_h2(and_or(w8, 0x00f000f0u, 0x54005400u)), k.zb64), k.s, k.c));
}

// Adds columns c .. c+7 of accumulators taddr0 and taddr1 (the thread's lane) into
// v, in that order.
__device__ __forceinline__ void add_acc8x2(uint32_t taddr0, uint32_t taddr1, float* v) {
  uint32_t r0[8], r1[8];
  tmem_ld8(taddr0, r0);
  tmem_ld8(taddr1, r1);
  tmem_wait_ld();
#pragma unroll
  for (int j = 0; j < 8; ++j) v[j] = (v[j] + __uint_as_float(r0[j])) + __uint_as_float(r1[j]);
}
__device__ __forceinline__ void add_acc8(uint32_t taddr, float* v) {
  uint32_t r[8];
  tmem_ld8(taddr, r);
  tmem_wait_ld();
#pragma unroll
  for (int j = 0; j < 8; ++j) v[j] += __uint_as_float(r[j]);
}

// GELU of the gate value: the tanh form as a * sigmoid(2u) = a / (1 + e^(-2u)), an
// identity of 0.5 a (1 + tanh(u)), u = sqrt(2/pi) (a + 0.044715 a^3); or the erf form.
__device__ __forceinline__ float gelu_fast(float a, int act) {
  if (act == 1) return 0.5f * a * (1.f + erff(a * 0.70710678118654752f));
  const float u = 0.79788456080286536f * fmaf(0.044715f * a, a * a, a);
  return __fdividef(a, 1.f + __expf(-2.f * u));
}

// First stage s of an item (its stages t0 .. t0 + nst - 1) with (t0 + s) % kPipes == pipe.
__device__ __forceinline__ int first_stage(int t0, int pipe) { return (pipe - t0 % kPipes + kPipes) % kPipes; }

// Item queue, producer 0's side: publishes item n (claimed beforehand into `next`) once
// its queue entry is free.  A down item of the fused launch is published only after
// every gate_up epilogue warp of its expert has written the expert's h rows.  With
// `block` false it returns at once (false) when the entry is still in use.
struct Dispatch {
  int next;        // the claimed item after the published ones (lane 0)
  int published;   // items published so far (the end of the list counts as one)
  bool ended;
};
__device__ __forceinline__ bool publish_one(TcHeader& H, Dispatch& D, const Args& a, int total0, int total,
                                            volatile int* abort, int lane, bool block, bool& ok) {
  const int n = D.published;
  const uint32_t bar = smem_addr(&H.item_empty[n % kQueue]);
  const uint32_t par = ((n / kQueue) & 1) ^ 1;
  if (!block) {
    if (!__all_sync(0xffffffffu, mbar_test_wait(bar, par))) return false;
  } else if (!gemm::warp_wait(bar, par, a.err, abort)) {
    ok = false;
    return false;
  }
  const int item = __shfl_sync(0xffffffffu, D.next, 0);
  const bool done = item >= total;
  const int pj = (a.first == 0 && item < total0) ? 0 : 1;
  int e = 0, blk = 0, n_cnt = 0, pos0 = 0;
  if (!done) gemm::decode_item(pj == 0 ? item : item - total0, H.prefix[pj], H.offs, a.E, kNMax, e, blk, n_cnt, pos0);
  if (!done && pj == 1 && a.first == 0) {
    // a down item reads the h rows of its expert: it is published only once every gate_up
    // epilogue warp of the expert has written them (acquire).  Looking ahead, a count not yet
    // reached leaves the item claimed but unpublished (this CTA may itself still owe some of
    // those h rows); when the item is needed now, the wait is bounded.
    const int need = kEpiWarps * a.p[0].nblocks * ((H.offs[e + 1] - H.offs[e] + kNMax - 1) / kNMax);
    int ready = 0;
    if (lane == 0) {
      if (block) {
        ok = gemm::wait_count(a.gu_done + e, need, a.err, abort, gemm::kDepWaitNs);
        ready = ok;
      } else {
        int v;
        asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(a.gu_done + e) : "memory");
        ready = v >= need;
      }
    }
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    if (!ok || !__shfl_sync(0xffffffffu, ready, 0)) return false;
  }
  if (lane == 0 && !done) D.next = atomicAdd(a.counter, 1);  // the next one, claimed ahead
  if (lane == 0) {
    H.item_desc[n % kQueue][0] = done ? -1 : (pj | (n_cnt << 8) | (blk << 16));
    H.item_desc[n % kQueue][1] = e;
    H.item_desc[n % kQueue][2] = pos0;
    mbar_arrive(smem_addr(&H.item_full[n % kQueue]));  // release: the entry is visible to its waiters
  }
  __syncwarp();
  ++D.published;
  D.ended = done;
  return true;
}

template <bool AF>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
    expert_gemm_tc_kernel(const Args a, const __grid_constant__ CUtensorMap map_x,
                          const __grid_constant__ CUtensorMap map_h) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  TcHeader& H = *reinterpret_cast<TcHeader*>(smem);
  uint8_t* ring = smem + kHeaderBytes;
  volatile int* abort = &H.abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int i = 0; i < kSlots; ++i) {
      H.slot_t[i] = -1;
      mbar_init(smem_addr(&H.slot_full[i]), 1);
      mbar_init(smem_addr(&H.codes_empty[i]), 4);
      mbar_init(smem_addr(&H.slot_free[i]), 1);
    }
    for (int i = 0; i < kAStages; ++i) {
      mbar_init(smem_addr(&H.a_full[i]), 4);
      mbar_init(smem_addr(&H.a_empty[i]), 1);
    }
    mbar_init(smem_addr(&H.acc_full), kPipes);
    mbar_init(smem_addr(&H.acc_free), kEpiWarps);
    for (int i = 0; i < kPipes; ++i) mbar_init(smem_addr(&H.drain[i]), 1);
    for (int i = 0; i < kQueue; ++i) {
      mbar_init(smem_addr(&H.item_full[i]), 1);
      mbar_init(smem_addr(&H.item_empty[i]), kConsumers);
    }
    H.abort = 0;
    fence_barrier_init();
  }
  if (warp == kFirstIssuer) tmem_alloc(smem_addr(&H.tmem_base), kTmemCols);
  // everything above is set-up; the routing arrays, the row copy and h come from earlier launches
  grid_dependents_launch();
  grid_dependency_wait();
  if (warp == kFirstDq) gemm::scan_items(a, kNMax, lane, H.prefix, H.offs);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = H.tmem_base;
  const uint32_t ring_s = smem_addr(ring);
  // the launch's work list: [gate_up items][down items], restricted to projections first..last
  const int total0 = a.first == 0 ? H.prefix[0][a.E] : 0;
  const int total = total0 + (a.last == 1 ? H.prefix[1][a.E] : 0);

  if (warp < kFirstIssuer) {
    // ------------------------------------------------------------------ producers
    // producer j fills the slots of the stages t = j, j + 3, ...; producer 0 also claims the
    // work items and keeps the queue filled ahead (the whole warp waits, lane 0 issues)
    const int pipe = warp;
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(&map_x) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(&map_h) : "memory");
    }
    // every weight byte is read once: it leaves L2 first, so that h, y and the token rows stay
    const uint64_t w_policy = l2_evict_first_policy();
    bool ok = true;
    Dispatch D{0, 0, false};
    if (pipe == 0 && lane == 0) D.next = atomicAdd(a.counter, 1);
    int t0 = 0;
    for (int i = 0; ok; ++i) {
      if (pipe == 0) {
        // publish item i (blocking) and up to kQueue - 1 more if their entries are free
        while (ok && D.published <= i && publish_one(H, D, a, total0, total, abort, lane, true, ok)) {
        }
        while (ok && !D.ended && D.published < i + kQueue && publish_one(H, D, a, total0, total, abort, lane, false, ok)) {
        }
        if (!ok) break;
      }
      if (!gemm::warp_wait(smem_addr(&H.item_full[i % kQueue]), (i / kQueue) & 1, a.err, abort)) break;
      const int d0 = H.item_desc[i % kQueue][0];
      if (d0 < 0) break;
      const int pj = d0 & 1, blk = d0 >> 16;
      const int e = H.item_desc[i % kQueue][1], pos0 = H.item_desc[i % kQueue][2];
      // the h rows of a down item were released to producer 0 (acquire); the TMA loads below
      // read them through the async proxy
      if (pj == 1 && a.first == 0) asm volatile("fence.proxy.async.global;" ::: "memory");
      const gemm::Proj& P = a.p[pj];
      const CUtensorMap* bmap = pj == 0 ? &map_x : &map_h;
      const int nst = num_stages(P.K);
      const uint8_t* wblk = P.w + static_cast<int64_t>(e) * P.expert_bytes + static_cast<int64_t>(blk) * P.block_bytes;
      for (int s = first_stage(t0, pipe); s < nst && ok; s += kPipes) {
        const int t = t0 + s, slot = t % kSlots;
        const uint32_t par = static_cast<uint32_t>(t / kSlots) & 1u;
        // the slot's previous stage: its codes read by the dequantisers, its MMAs (token tile) done
        ok = gemm::warp_wait(smem_addr(&H.codes_empty[slot]), par ^ 1u, a.err, abort) &&
             gemm::warp_wait(smem_addr(&H.slot_free[slot]), par ^ 1u, a.err, abort);
        if (!ok) break;
        const int width = min(kCols, P.K - s * kCols);
        const uint32_t wbytes = width * (kBlockRows / 2) + groups_per_stage(width, P.g) * kSzRowBytes;
        if (lane == 0) {
          const uint32_t full = smem_addr(&H.slot_full[slot]);
          const uint32_t dst = ring_s + slot * kSlotBytes;
          H.slot_t[slot] = t;
          mbar_arrive_expect_tx(full, (width / 64) * kBoxBytes + wbytes);
          bulk_g2s_hint(dst + kCodeOff + width * (kBlockRows / 2) - wbytes, wblk + s * full_stage_bytes(P.g), wbytes,
                        full, w_policy);
          gemm::tma_load_2d(dst, bmap, s * kCols, pos0, full);
          if (width > 64) gemm::tma_load_2d(dst + kBoxBytes, bmap, s * kCols + 64, pos0, full);
        }
        __syncwarp();
      }
      if (!ok) break;
      t0 += nst;
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&H.item_empty[i % kQueue]));
    }
  } else if (warp < kFirstEpi) {
    // ------------------------------------------------------------------ MMA issuers
    const int r = warp - kFirstIssuer;                   // this issuer's stages: t = r, r + 3, ...
    const uint32_t d_col = tmem + kAccCol0 + kNMax * r;  // its accumulator
    bool ok = true;
    int t0 = 0;  // global index of the item's first stage
    for (int i = 0;; ++i) {
      if (!gemm::warp_wait(smem_addr(&H.item_full[i % kQueue]), (i / kQueue) & 1, a.err, abort)) {
        ok = false;
        break;
      }
      const int d0 = H.item_desc[i % kQueue][0];
      if (d0 < 0) break;
      const int pj = d0 & 1, n_cnt = (d0 >> 8) & 0xff;
      const int K = a.p[pj].K, nst = num_stages(K);
      const uint32_t idesc = f16_idesc_m128(n_cnt <= 16 ? 16 : 32);
      if (lane == 0) {
        const int s0 = first_stage(t0, r);
        // the accumulator is free once the epilogue warps have read the previous item's (waited
        // for every item, even one without stages of this issuer, so that the wait is never more
        // than one phase behind)
        ok = gemm::thread_wait(smem_addr(&H.acc_free), (i & 1) ^ 1, a.err, abort);
        for (int s = s0; s < nst && ok; s += kPipes) {
          const int t = t0 + s, slot = t % kSlots, as = t % kAStages;
          ok = gemm::thread_wait(smem_addr(&H.a_full[as]), (t / kAStages) & 1, a.err, abort) &&
               gemm::thread_wait(smem_addr(&H.slot_full[slot]), (t / kSlots) & 1, a.err, abort);
          if (!ok) break;
          tc_fence_after();
          const uint64_t bdesc = sw128_desc(ring_s + slot * kSlotBytes);
          const uint32_t acol = tmem + as * kACols;
          const int ksteps = min(kCols, K - s * kCols) / 16;
          for (int kk = 0; kk < ksteps; ++kk)  // 16 columns: 8 A columns (fp16 pairs), 32 bytes of a token box
            tc_mma_ts(d_col, acol + 8 * kk, bdesc + (kk >> 2) * (kBoxBytes >> 4) + 2 * (kk & 3), idesc,
                      (s > s0 || kk > 0) ? 1u : 0u);
          tc_commit(smem_addr(&H.a_empty[as]));      // the A stage may be rewritten
          tc_commit(smem_addr(&H.slot_free[slot]));  // the token tile may be overwritten
        }
        if (ok) tc_commit(smem_addr(&H.acc_full));  // every issuer, once per item
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok) break;
      t0 += nst;
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&H.item_empty[i % kQueue]));
    }
    // every MMA this thread issued has completed before tensor memory is freed
    (void)ok;
    if (lane == 0) {
      tc_commit(smem_addr(&H.drain[r]));
      mbar_wait(smem_addr(&H.drain[r]), 0, a.err);
    }
    __syncwarp();
  } else if (warp < kFirstDq) {
    // ------------------------------------------------------------------ epilogue (32 rows of the block)
    const int q = warp & 3;
    const uint32_t acc = tmem + (static_cast<uint32_t>(32 * q) << 16) + kAccCol0;
    int t0 = 0;
    for (int i = 0;; ++i) {
      if (!gemm::warp_wait(smem_addr(&H.item_full[i % kQueue]), (i / kQueue) & 1, a.err, abort)) break;
      const int d0 = H.item_desc[i % kQueue][0];
      if (d0 < 0) break;
      const int pj = d0 & 1, n_cnt = (d0 >> 8) & 0xff, blk = d0 >> 16;
      const int e = H.item_desc[i % kQueue][1], pos0 = H.item_desc[i % kQueue][2];
      const int nst = num_stages(a.p[pj].K);
      if (!gemm::warp_wait(smem_addr(&H.acc_full), i & 1, a.err, abort)) break;
      tc_fence_after();
      // the thread's row of the item: class c of the item's stages (s = c, c + 3, ...) sits in
      // the accumulator of issuer (t0 + c) % 3; the classes are summed in the fixed order
      // (C0 + C1) + C2, so the result does not depend on where the item fell in this CTA's
      // stage sequence
      const int ncls = min(kPipes, nst);
      float v[kNMax];
#pragma unroll
      for (int n = 0; n < kNMax; ++n) v[n] = 0.f;
      for (int c = 0; c < (n_cnt > 16 ? 32 : 16); c += 8) {
        int cl = 0;
        for (; cl + 1 < ncls; cl += 2)
          add_acc8x2(acc + kNMax * ((t0 + cl) % kPipes) + c, acc + kNMax * ((t0 + cl + 1) % kPipes) + c, v + c);
        if (cl < ncls) add_acc8(acc + kNMax * ((t0 + cl) % kPipes) + c, v + c);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&H.acc_free));  // the issuers may overwrite the accumulators
      if (pj == 0) {
        // lanes 0-15 of the quarter hold gate rows j = 64 blk + 16 q + (0..15), lanes 16-31 the
        // matching up rows; lane l < 16 then forms tokens 0-15 and lane l + 16 tokens 16-31 of row j
        const bool lo = lane < 16;
        const int jcol = 64 * blk + 16 * q + (lane & 15);
#pragma unroll
        for (int n = 0; n < 16; ++n) {
          const float other = __shfl_xor_sync(0xffffffffu, lo ? v[16 + n] : v[n], 16);
          const float gate = lo ? v[n] : other, up = lo ? other : v[16 + n];
          const int nt = lo ? n : 16 + n;
          if (nt < n_cnt)
            a.h[static_cast<size_t>(pos0 + nt) * a.f + jcol] = __half_as_ushort(__float2half_rn(gelu_fast(gate, a.act) * up));
        }
        if (a.last == 1) {
          // report the h rows to the expert's counter: __syncwarp orders the lanes' stores before
          // lane 0's release, which is cumulative at device scope
          __syncwarp();
          if (lane == 0) asm volatile("red.release.gpu.global.add.s32 [%0], 1;" ::"l"(a.gu_done + e) : "memory");
        }
      } else {
        const int i_row = kBlockRows * blk + 32 * q + lane;
        const int my_p = lane < n_cnt ? a.pair_list[pos0 + lane] : 0;  // pair id of token `lane` of the item
#pragma unroll
        for (int n = 0; n < kNMax; ++n) {
          const int p = __shfl_sync(0xffffffffu, my_p, n);
          if (n < n_cnt) a.y_out[static_cast<size_t>(p) * a.d + i_row] = v[n];
        }
      }
      t0 += nst;
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&H.item_empty[i % kQueue]));
    }
  } else {
    // ------------------------------------------------------------------ dequantisers
    const int q = warp & 3;                        // lane quarter: rows 32 q .. 32 q + 31 of the block
    const int team = (warp - kFirstDq) >> 2;       // this warp's stages: t = team, team + 3, ...
    const int m = 32 * q + lane;                   // the thread's weight row (tensor-memory lane)
    const uint32_t a_dst = tmem + (static_cast<uint32_t>(32 * q) << 16);
    int t0 = 0;                                    // global index of the item's first stage
    for (int i = 0;; ++i) {
      if (!gemm::warp_wait(smem_addr(&H.item_full[i % kQueue]), (i / kQueue) & 1, a.err, abort)) break;
      const int d0 = H.item_desc[i % kQueue][0];
      if (d0 < 0) break;
      const int pj = d0 & 1;
      const int g = a.p[pj].g, K = a.p[pj].K, nst = num_stages(K);
      bool ok = true;
      for (int s = first_stage(t0, team); s < nst; s += kPipes) {
        const int t = t0 + s, slot = t % kSlots, as = t % kAStages;
        const int nch = min(kCols, K - s * kCols) / 32;  // 32-column chunks: 4, or 2 in a last stage of 64
        ok = gemm::warp_wait(smem_addr(&H.slot_full[slot]), (t / kSlots) & 1, a.err, abort);
        if (!ok) break;
        const uint32_t sl = ring_s + slot * kSlotBytes;
        // the stage's codes of this row (chunk c: 32 columns) and the (scale, second) pair of each chunk's group
        uint32_t w[4][4], v[4];
        const int ng = groups_per_stage(nch * 32, g);
        const uint32_t sz = sl + kCodeOff - ng * kSzRowBytes + m * 4;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          if (c < nch) {
            asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                         : "=r"(w[c][0]), "=r"(w[c][1]), "=r"(w[c][2]), "=r"(w[c][3])
                         : "r"(sl + kCodeOff + ((q * nch + c) * 32 + lane) * 16));
            const int grp = (32 * c) / g;  // 0 for g = 128, c / 2 for 64, c for 32
            if (grp * g == 32 * c)  // the chunk starts a group
              asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v[c]) : "r"(sz + grp * kSzRowBytes));
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&H.codes_empty[slot]));  // codes and constants are in registers
        Dq k;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          if (c < nch) {
            if (((32 * c) / g) * g == 32 * c) k = dq_const<AF>(v[c]);
            uint32_t o[16];
            dequant8(w[c][0], k, o);
            dequant8(w[c][1], k, o + 4);
            dequant8(w[c][2], k, o + 8);
            dequant8(w[c][3], k, o + 12);
            if (c == 0) {
              // the A stage is free once the MMAs of the stage that used it last (t - kAStages,
              // this pipe's) completed
              ok = gemm::warp_wait(smem_addr(&H.a_empty[as]), ((t / kAStages) & 1) ^ 1, a.err, abort);
              if (!ok) break;
              tc_fence_after();
            }
            tmem_st16(a_dst + as * kACols + 16 * c, o);
          }
        }
        if (!ok) break;
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&H.a_full[as]));
      }
      if (!ok) break;
      t0 += nst;
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&H.item_empty[i % kQueue]));
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kFirstIssuer) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  // drain: the last copies into every slot have landed before the CTA exits (no copy is
  // issued any more; after a timed-out wait some may still be in flight)
  if (tid == 0)
    for (int i = 0; i < kSlots; ++i)
      if (H.slot_t[i] >= 0) mbar_wait(smem_addr(&H.slot_full[i]), (H.slot_t[i] / kSlots) & 1, a.err);
  // The last CTA to finish clears the work counter for the next launch on this
  // workspace: by then every CTA has seen the list exhausted and claims no more.
  if (tid == 0 && atomicAdd(a.done_ctas, 1) == static_cast<int>(gridDim.x) - 1) {
    *a.counter = 0;
    *a.done_ctas = 0;
  }
}

}  // namespace

cudaError_t init_gemm_tc_kernels() {
  for (const void* fn : {reinterpret_cast<const void*>(expert_gemm_tc_kernel<false>),
                         reinterpret_cast<const void*>(expert_gemm_tc_kernel<true>)}) {
    cudaError_t err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (err != cudaSuccess) return err;
    err = cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (err != cudaSuccess) return err;
  }
  return cudaSuccess;
}

cudaError_t launch_expert_gemm_tc(const gemm::Args& a, const CUtensorMap& map_x, const CUtensorMap& map_h, bool affine,
                                  int num_sms, cudaStream_t st) {
  auto* kern = affine ? expert_gemm_tc_kernel<true> : expert_gemm_tc_kernel<false>;
  return launch_pdl(kern, dim3(num_sms * kCtasPerSm), dim3(kThreads), kSmemBytes, st, a, map_x, map_h);
}

}  // namespace moe
