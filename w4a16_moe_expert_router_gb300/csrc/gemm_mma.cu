// gemm_mma.cu -- grouped W4A16 expert GEMMs with the weights dequantised in
// registers and multiplied on the warp-level tensor-core path.
//
// Model card "srswti/axe-diffusion-ksl-xe", "the kernels we built": the GEMM
// reads packed nibbles and dequantises inline, so HBM carries real 4-bit
// traffic; one launch covers all experts; the activation is folded into the
// first GEMM's epilogue.  One persistent launch runs both projections:
//   gate_up:  a[p][n] = sum_k Wgu[e][n][k] x[t(p)][k]
//             h[pos(p)][j] = gelu(a[p][j]) * a[p][f+j]  -> fp16, rows in expert-sorted order
//   down:     y[p][i] = sum_j Wd[e][i][j] h[pos(p)][j]   -> fp32, rows by pair id p = t*k + r
// The work list holds every gate_up item followed by every down item; an item
// is (projection, expert, 128-row block, chunk of <= 32 tokens) over the whole
// contraction.  A down item of expert e starts once all gate_up items of e have
// written their h rows (a per-expert counter, bounded wait).
//
// Why registers and mma.sync: a canvas gives an expert ~16 tokens, so each
// weight is used by few MACs and the work is the dequantisation, not the
// multiply.  A thread turns one 32-bit word of codes into exactly the four f16x2
// registers of an m16n8k16 A fragment and hands them to the MMA itself; no
// weight tile is written to shared or tensor memory and no other warp has to be
// told that it is ready.  The tokens (the B operand) are shared by the CTA's
// four compute warps through a TMA-filled shared-memory ring.
//
// Arithmetic: the zero-point is split into its nearest integer zr and the rest
// zf = z - zr, and each weight is formed as w = fp16((q - zr) * s - fp16(zf * s)):
// q - zr is exact in fp16 and the fused multiply-add rounds once.  The MMA
// multiplies w with the fp16 activations into fp32 accumulators (16-column
// steps in contraction order).  A second instantiation of the kernel takes the
// group-factorised order instead (shape field reduction = 1; see run_stage_gf):
// codes as fp16 subnormals straight into the MMA, per-group fp32 partial sums,
// scale and zero-point applied per group, items of at most 16 tokens.
//
// Roles of the persistent CTA (three per SM; a stage is 128 contraction columns,
// the last one 64 when the contraction is an odd multiple of 64):
//   warp 0      producer: claims items one ahead of use, publishes each in a
//               small queue in shared memory, and per stage issues one bulk
//               copy of the stage's weight segment (codes and (scale, zero)
//               pairs of all eight 16-row strips, contiguous in the stream) and
//               two 2-D TMA loads (64 columns x 32 token rows each, 128-byte
//               swizzle) of the activations into the same slot of a ring of
//               three;
//   warps 1-4   compute: warp w owns strips 2w and 2w+1, 32 GEMM rows of the
//               block (a gate_up strip holds 8 gate rows and the 8 matching up
//               rows, so the gated GELU needs nothing from another warp).  Per
//               stage each reads its strips' codes (16-byte vectors, 512
//               contiguous bytes per strip and load) and (scale, zero) pairs
//               from the slot, dequantises them into A fragments, reads each
//               token fragment once with ldmatrix for both strips and issues
//               the MMAs; an item's accumulators stay in registers.  Two
//               strips per warp share the token fragments, the waits and the
//               address work, and give each warp twice the independent work.
//               The kernel is specialised per item on the token tiles (1-4
//               tiles of 8) and the group size, so a stage has no data-dependent
//               branches.
// Every wait is bounded: on expiry the CTA records MOE_W4A16_ERR_TIMEOUT in the
// workspace and all roles leave their loops; the producer drains its copies.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "gemm_common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kStrips = kBlockRows / kStripRows;   // 16-row strips per block
constexpr int kMmaWarps = kStrips / 2;             // compute warps, two strips each
constexpr int kThreads = (1 + kMmaWarps) * 32;     // 160
constexpr int kCtasPerSm = 3;
constexpr int kSlots = 3;                          // stages in flight per CTA (three CTAs per SM share 227 KiB)
constexpr int kQueue = 4;                          // item descriptors in flight per CTA
constexpr int kChunkGf = 16;                       // tokens per work item in the group-factorised order
constexpr int kBBoxRows = 32;                      // TMA box: 64 columns x 32 token rows
constexpr int kBoxBytes = kBBoxRows * 128;         // 4 KiB, 128-byte swizzle
constexpr int kBBytes = 2 * kBoxBytes;             // a stage's token tile: two boxes
constexpr int kSzBytesW = 64;                      // one warp's (scale, zero) pairs of one group
constexpr int kWMaxBytes = kStrips * (1024 + 4 * kSzBytesW);  // a stage's weights, at most 10 KiB
constexpr int kSlotBytes = 18432;                  // [tokens 8 KiB][weights <= 10 KiB], a multiple of 1024
static_assert(kBBytes + kWMaxBytes <= kSlotBytes && kSlotBytes % 1024 == 0, "slot layout");
constexpr int kHeaderBytes = 4096;
constexpr int kSmemBytes = 1024 + kHeaderBytes + kSlots * kSlotBytes;  // +1024 for alignment



using MmArgs = gemm::Args;
using gemm::decode_item;
using gemm::gelu;
using gemm::kDepWaitNs;
using gemm::tma_load_2d;
using gemm::wait_count;

// Shared-memory header (at the 1024-aligned base of dynamic shared memory).
struct __align__(8) MmHeader {
  uint64_t slot_full[kSlots];   // the stage's tokens and weights landed
  uint64_t slot_empty[kSlots];  // the compute warps have read the stage
  uint64_t item_full[kQueue];   // queue entry written
  uint64_t item_empty[kQueue];  // the compute warps are done with the item
  int item_desc[kQueue][3];     // {proj | tokens << 8 | block << 16 (or -1 at the end), expert, first row}
  int abort;
  int prefix[2][kMaxExperts + 1];  // items of each projection before expert e
  int offs[kMaxExperts + 1];    // expert_offsets, copied once
};
static_assert(sizeof(MmHeader) <= kHeaderBytes, "header fits");

// Weight bytes of one stage of kk16 16-column steps (all eight warps) with groups of g.
__device__ __forceinline__ uint32_t stage_weight_bytes(int kk16, int g) {
  const int ng = (16 * kk16) / min(g, 16 * kk16);
  return static_cast<uint32_t>(kStrips * (kk16 * 128 + kSzBytesW * ng));
}





// Dequantiser constants of one thread's two rows (g and g+8 of its warp's 16)
// for one group, each broadcast to both halves of an f16x2: the zero-point split
// into its nearest integer zr and the rest zf = z - zr, so that
// (q - zr) * s - zf * s = (q - z) * s.
struct DqRows {
  __half2 zb_lo;  // 1024 + zr of row g (exact)
  __half2 s_lo;
  __half2 c_lo;   // -fp16(zf * s) of row g
  __half2 zb_hi;  // 64 + zr of row g + 8 (exact)
  __half2 s_hi;
  __half2 c_hi;
};
// v.x = (scale, zero) of row g, v.y = those of row g + 8 (fp16 pairs).  For
// 0 <= z <= 16, fp16(z + 1024) is 1024 + zr with zr = z rounded to the nearest
// integer (ties to even): fp16 has unit spacing in [1024, 2048).
__device__ __forceinline__ DqRows dq_rows(uint32_t vx, uint32_t vy) {
  const uint32_t zz = __byte_perm(vx, vy, 0x7632), ss = __byte_perm(vx, vy, 0x5410);
  const __half2 z = bits_h2(zz), s = bits_h2(ss);
  const __half2 zb1 = __hadd2(z, bits_h2(0x64006400u));            // 1024 + zr, both rows
  const __half2 zr = __hsub2(zb1, bits_h2(0x64006400u));
  const __half2 c = __hneg2(__hmul2(__hsub2(z, zr), s));
  const __half2 zb = __hsub2(zb1, bits_h2(0x63800000u));           // (1024 + zr_g, 64 + zr_g8)
  DqRows k;
  k.zb_lo = __low2half2(zb);
  k.s_lo = __low2half2(s);
  k.c_lo = __low2half2(c);
  k.zb_hi = __high2half2(zb);
  k.s_hi = __high2half2(s);
  k.c_hi = __high2half2(c);
  return k;
}

// The same constants for the affine format (w = q s + b, the second value of the
// group is the bias b): the offset is the bare 1024 / 64, so the subtract gives q
// exactly, and the fused multiply-add forms fp16(q s + b) with one rounding.
__device__ __forceinline__ DqRows dq_rows_affine(uint32_t vx, uint32_t vy) {
  const uint32_t bb = __byte_perm(vx, vy, 0x7632), ss = __byte_perm(vx, vy, 0x5410);
  const __half2 b = bits_h2(bb), s = bits_h2(ss);
  DqRows k;
  k.zb_lo = bits_h2(0x64006400u);
  k.s_lo = __low2half2(s);
  k.c_lo = __low2half2(b);
  k.zb_hi = bits_h2(0x54005400u);
  k.s_hi = __high2half2(s);
  k.c_hi = __high2half2(b);
  return k;
}

// One word of codes -> the m16n8k16 A fragment of the thread: nibbles (0,4) are
// row g columns (2t, 2t+1), (1,5) row g+8 columns (2t, 2t+1), (2,6) row g
// columns (2t+8, 2t+9), (3,7) row g+8 columns (2t+8, 2t+9).  (1024 + q) and
// (64 + q) come from OR-ing exponent bits onto the nibbles; one fp16 subtract of
// (1024 + zr) or (64 + zr) gives q - zr exactly, and one fused multiply-add
// rounds the weight once.
__device__ __forceinline__ void dequant_frag(uint32_t w, const DqRows& k, uint32_t (&a)[4]) {
  const uint32_t w8 = w >> 8;
  a[0] = h2_bits(__hfma2(__hsub2(bits_h2(and_or(w, 0x000f000fu, 0x64006400u)), k.zb_lo), k.s_lo, k.c_lo));
  a[1] = h2_bits(__hfma2(__hsub2(bits_h2(and_or(w, 0x00f000f0u, 0x54005400u)), k.zb_hi), k.s_hi, k.c_hi));
  a[2] = h2_bits(__hfma2(__hsub2(bits_h2(and_or(w8, 0x000f000fu, 0x64006400u)), k.zb_lo), k.s_lo, k.c_lo));
  a[3] = h2_bits(__hfma2(__hsub2(bits_h2(and_or(w8, 0x00f000f0u, 0x54005400u)), k.zb_hi), k.s_hi, k.c_hi));
}

// Group-factorised order ("ashhart/TensorFold pull 802", section "Contracts":
// partial sums per group, then the scale, then the bias): the codes go to the MMA
// as they are, as fp16 subnormals, and each group's scale and zero-point are
// applied once per group to fp32 partial sums:
//   sum_k x_k (q_k - z) s = s * sum_k x_k q_k - s z * sum_k x_k   (k over one group).
// One word of codes -> the A fragment by masks alone: rows g hold q * 2^-24, rows
// g + 8 hold 16 q * 2^-24 (their nibbles sit four bits higher and stay there).
// Products of fp16 values are exact in the fp32 accumulators.
__device__ __forceinline__ void code_frag(uint32_t w, uint32_t (&a)[4]) {
  const uint32_t w8 = w >> 8;
  a[0] = w & 0x000f000fu;
  a[1] = w & 0x00f000f0u;
  a[2] = w8 & 0x000f000fu;
  a[3] = w8 & 0x00f000f0u;
}

// Per-group fp32 constants of one thread's rows g and g + 8 (v.x, v.y as in dq_rows),
// in the units of the partial sums: s for rows g, s / 16 for rows g + 8, and -s z
// for the sum of the activations (products of two fp16 values: exact).
struct GfRows {
  float s_lo, z_lo, s_hi, z_hi;
};
__device__ __forceinline__ GfRows gf_rows(uint32_t vx, uint32_t vy) {
  const float2 a = __half22float2(bits_h2(vx)), b = __half22float2(bits_h2(vy));
  GfRows k;
  k.s_lo = a.x;
  k.z_lo = -a.x * a.y;
  k.s_hi = b.x * 0.0625f;
  k.z_hi = -b.x * b.y;
  return k;
}
// Affine format: the term of the activation sum is the bias itself (b sum(x)).
__device__ __forceinline__ GfRows gf_rows_affine(uint32_t vx, uint32_t vy) {
  const float2 a = __half22float2(bits_h2(vx)), b = __half22float2(bits_h2(vy));
  GfRows k;
  k.s_lo = a.x;
  k.z_lo = a.y;
  k.s_hi = b.x * 0.0625f;
  k.z_hi = b.y;
  return k;
}

// D = A * B + (Z ? 0 : D)
template <bool Z>
__device__ __forceinline__ void mma_acc(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  if (Z) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%10,%10,%10};\n"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(0.f));
  } else {
    mma_f16_16816(d, a, b0, b1);
  }
}


__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const MmArgs& a, volatile int* abort) {
  return gemm::warp_wait(bar, parity, a.err, abort);
}


// Work item as the compute warps read it from the queue.
struct ItemView {
  int pj, n_cnt, blk, e, pos0, g;
};

__device__ __forceinline__ bool read_item(const MmHeader& H, int i, const MmArgs& a, ItemView& v) {
  const int d0 = H.item_desc[i % kQueue][0];
  if (d0 < 0) return false;
  v.pj = d0 & 1;
  v.n_cnt = (d0 >> 8) & 0xff;
  v.blk = d0 >> 16;
  v.e = H.item_desc[i % kQueue][1];
  v.pos0 = H.item_desc[i % kQueue][2];
  v.g = a.p[v.pj].g;
  return true;
}

// One stage of one compute warp: KK 16-column steps, NT tiles of 8 tokens, groups of G,
// for the warp's two strips 2 sw and 2 sw + 1 (one token fragment serves both).
template <int NT, int G, int KK, bool AF>
__device__ __forceinline__ bool run_stage(const MmArgs& a, MmHeader& H, volatile int* abort,
                                          float (&acc)[2][NT][4], int& slot, uint32_t& phase, uint32_t ring_s,
                                          const uint32_t (&loff)[4], int sw, int lane) {
  constexpr int NG = (16 * KK) / (G < 16 * KK ? G : 16 * KK);  // groups in the stage
  constexpr int kStepsPerGroup = KK / NG;
  constexpr int kStripBytes = KK * 128 + kSzBytesW * NG;
  if (!warp_wait(smem_addr(&H.slot_full[slot]), phase, a, abort)) return false;
  const uint32_t sl = ring_s + slot * kSlotBytes;
  // the warp's strips of the stage's weights: [(scale, zero) x NG][codes], one after the other
  const uint32_t wseg = sl + kBBytes + 2 * sw * kStripBytes;
  const uint32_t caddr = wseg + kSzBytesW * NG + lane * 16;
  uint32_t szw[2][2 * NG];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint32_t szaddr = wseg + h * kStripBytes + (lane >> 2) * (8 * NG);
    if (NG == 1) {
      asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(szw[h][0]), "=r"(szw[h][1]) : "r"(szaddr));
    } else {
#pragma unroll
      for (int q = 0; q < NG / 2; ++q)
        asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(szw[h][4 * q]), "=r"(szw[h][4 * q + 1]), "=r"(szw[h][4 * q + 2]), "=r"(szw[h][4 * q + 3])
                     : "r"(szaddr + 16 * q));
    }
  }
  DqRows k[2];
  uint32_t words[2][4];
#pragma unroll
  for (int kk = 0; kk < KK; ++kk) {
    if (kk % 4 == 0)
#pragma unroll
      for (int h = 0; h < 2; ++h)
        asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(words[h][0]), "=r"(words[h][1]), "=r"(words[h][2]), "=r"(words[h][3])
                     : "r"(caddr + h * kStripBytes + (kk / 4) * 512));
    if (kk % kStepsPerGroup == 0)
#pragma unroll
      for (int h = 0; h < 2; ++h)
        k[h] = AF ? dq_rows_affine(szw[h][2 * (kk / kStepsPerGroup)], szw[h][2 * (kk / kStepsPerGroup) + 1])
                  : dq_rows(szw[h][2 * (kk / kStepsPerGroup)], szw[h][2 * (kk / kStepsPerGroup) + 1]);
    uint32_t af[2][4];
    dequant_frag(words[0][kk % 4], k[0], af[0]);
    dequant_frag(words[1][kk % 4], k[1], af[1]);
    const uint32_t baddr = sl + (kk / 4) * kBoxBytes + loff[kk % 4];
    {
      uint32_t b0, b1, b2, b3;
      ldmatrix_x4(baddr, b0, b1, b2, b3);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        mma_f16_16816(acc[h][0], af[h], b0, b1);
        if (NT > 1) mma_f16_16816(acc[h][NT > 1 ? 1 : 0], af[h], b2, b3);
      }
    }
    if (NT > 2) {
      uint32_t b0, b1, b2, b3;
      ldmatrix_x4(baddr + 16 * 128, b0, b1, b2, b3);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        mma_f16_16816(acc[h][NT > 2 ? 2 : 0], af[h], b0, b1);
        if (NT > 3) mma_f16_16816(acc[h][NT > 3 ? 3 : 0], af[h], b2, b3);
      }
    }
  }
  __syncwarp();
  if (lane == 0) mbar_arrive(smem_addr(&H.slot_empty[slot]));  // shared-memory reads of the stage done
  if (++slot == kSlots) {
    slot = 0;
    phase ^= 1u;
  }
  return true;
}

// One stage in the group-factorised form (items of at most two token tiles): per
// group, the MMAs of both strips into partial sums that start at zero, and the
// activation sums of the item's 16 token rows, then
// tot += s * partial - s z * sum (two fused multiply-adds per accumulator).  tot is
// in units of 2^-24.  The sums take one more MMA per 16-column step with the roles
// swapped: the token fragments the step already holds (tokens 0-7 and 8-15 at its
// two 8-column halves) form the m16k16 A fragment {b0, b2, b1, b3}, times a B
// fragment of 2^-24, so that row m of the result is token m's sum; four shuffles
// move those into the accumulators' token columns.
template <int NT, int G, int KK, bool AF>
__device__ __forceinline__ bool run_stage_gf(const MmArgs& a, MmHeader& H, volatile int* abort,
                                             float (&tot)[2][NT][4], int& slot, uint32_t& phase, uint32_t ring_s,
                                             const uint32_t (&loff)[4], int sw, int lane) {
  static_assert(NT == 1 || NT == 2, "group-factorised items have at most 16 tokens");
  constexpr int NG = (16 * KK) / (G < 16 * KK ? G : 16 * KK);
  constexpr int kStepsPerGroup = KK / NG;
  constexpr int kStripBytes = KK * 128 + kSzBytesW * NG;
  constexpr uint32_t kUnit = 0x00010001u;  // 2^-24 in both halves
  if (!warp_wait(smem_addr(&H.slot_full[slot]), phase, a, abort)) return false;
  const uint32_t sl = ring_s + slot * kSlotBytes;
  const uint32_t wseg = sl + kBBytes + 2 * sw * kStripBytes;
  const uint32_t caddr = wseg + kSzBytesW * NG + lane * 16;
  uint32_t szw[2][2 * NG];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint32_t szaddr = wseg + h * kStripBytes + (lane >> 2) * (8 * NG);
    if (NG == 1) {
      asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(szw[h][0]), "=r"(szw[h][1]) : "r"(szaddr));
    } else {
#pragma unroll
      for (int q = 0; q < NG / 2; ++q)
        asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(szw[h][4 * q]), "=r"(szw[h][4 * q + 1]), "=r"(szw[h][4 * q + 2]), "=r"(szw[h][4 * q + 3])
                     : "r"(szaddr + 16 * q));
    }
  }
  uint32_t words[2][4];
#pragma unroll
  for (int j = 0; j < NG; ++j) {
    float part[2][NT][4], rs[4];  // rs: sums of token rows g (0, 1) and g + 8 (2, 3)
#pragma unroll
    for (int st = 0; st < kStepsPerGroup; ++st) {
      const int kk = j * kStepsPerGroup + st;
      if (kk % 4 == 0)
#pragma unroll
        for (int h = 0; h < 2; ++h)
          asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                       : "=r"(words[h][0]), "=r"(words[h][1]), "=r"(words[h][2]), "=r"(words[h][3])
                       : "r"(caddr + h * kStripBytes + (kk / 4) * 512));
      uint32_t af[2][4];
      code_frag(words[0][kk % 4], af[0]);
      code_frag(words[1][kk % 4], af[1]);
      uint32_t b0, b1, b2, b3;
      ldmatrix_x4(sl + (kk / 4) * kBoxBytes + loff[kk % 4], b0, b1, b2, b3);
      const uint32_t tok[4] = {b0, b2, b1, b3};
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        if (st == 0) {
          mma_acc<true>(part[h][0], af[h], b0, b1);
          if (NT > 1) mma_acc<true>(part[h][NT - 1], af[h], b2, b3);
        } else {
          mma_acc<false>(part[h][0], af[h], b0, b1);
          if (NT > 1) mma_acc<false>(part[h][NT - 1], af[h], b2, b3);
        }
      }
      if (st == 0) mma_acc<true>(rs, tok, kUnit, kUnit);
      else mma_acc<false>(rs, tok, kUnit, kUnit);
    }
    // token column n of tile u is row 8 u + n of rs, held by lanes 4 n .. 4 n + 3
    const int src = 8 * (lane & 3);
    float xs[NT][2];
    xs[0][0] = __shfl_sync(0xffffffffu, rs[0], src);
    xs[0][1] = __shfl_sync(0xffffffffu, rs[0], src + 4);
    if (NT > 1) {
      xs[NT - 1][0] = __shfl_sync(0xffffffffu, rs[2], src);
      xs[NT - 1][1] = __shfl_sync(0xffffffffu, rs[2], src + 4);
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const GfRows k = AF ? gf_rows_affine(szw[h][2 * j], szw[h][2 * j + 1]) : gf_rows(szw[h][2 * j], szw[h][2 * j + 1]);
#pragma unroll
      for (int u = 0; u < NT; ++u) {
        float(&t)[4] = tot[h][u];
        t[0] = fmaf(k.s_lo, part[h][u][0], fmaf(k.z_lo, xs[u][0], t[0]));
        t[1] = fmaf(k.s_lo, part[h][u][1], fmaf(k.z_lo, xs[u][1], t[1]));
        t[2] = fmaf(k.s_hi, part[h][u][2], fmaf(k.z_hi, xs[u][0], t[2]));
        t[3] = fmaf(k.s_hi, part[h][u][3], fmaf(k.z_hi, xs[u][1], t[3]));
      }
    }
  }
  __syncwarp();
  if (lane == 0) mbar_arrive(smem_addr(&H.slot_empty[slot]));
  if (++slot == kSlots) {
    slot = 0;
    phase ^= 1u;
  }
  return true;
}

// One item of one compute warp: every stage of the contraction, then the epilogue.
// Returns false if a wait gave up.
template <int NT, int G, bool GF, bool AF>
__device__ __forceinline__ bool run_item(const MmArgs& a, MmHeader& H, volatile int* abort, const ItemView& v,
                                         int& slot, uint32_t& phase, uint32_t ring_s, const uint32_t (&loff)[4],
                                         int sw, int lane) {
  const int gq = lane >> 2, tq = lane & 3;
  float acc[2][NT][4];
#pragma unroll
  for (int h = 0; h < 2; ++h)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[h][nt][j] = 0.f;
  const int K = a.p[v.pj].K;
  constexpr int G4 = G < 64 ? G : 64;  // groups of the last 64 columns
  if constexpr (GF) {
    for (int c0 = 0; c0 + kStageCols <= K; c0 += kStageCols)
      if (!run_stage_gf<NT, G, 8, AF>(a, H, abort, acc, slot, phase, ring_s, loff, sw, lane)) return false;
    if (G < 128 && (K % kStageCols) != 0)
      if (!run_stage_gf<NT, G4, 4, AF>(a, H, abort, acc, slot, phase, ring_s, loff, sw, lane)) return false;
  } else {
    for (int c0 = 0; c0 + kStageCols <= K; c0 += kStageCols)
      if (!run_stage<NT, G, 8, AF>(a, H, abort, acc, slot, phase, ring_s, loff, sw, lane)) return false;
    if (G < 128 && (K % kStageCols) != 0)  // the last 64 columns
      if (!run_stage<NT, G4, 4, AF>(a, H, abort, acc, slot, phase, ring_s, loff, sw, lane)) return false;
  }
  if constexpr (GF) {
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[h][nt][j] *= 16777216.f;  // 2^24: back from the partial sums' units
  }
  // ------------------------------------------------------------------ epilogue
  if (v.pj == 0) {
    // strip s: rows gq gate j, gq + 8 up j, with j = 64 * blk + 8 * s + gq
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int j = 64 * v.blk + 8 * (2 * sw + h) + gq;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int n = 8 * nt + 2 * tq;
        if (n < v.n_cnt)
          a.h[static_cast<size_t>(v.pos0 + n) * a.f + j] =
              __half_as_ushort(__float2half_rn(gelu(acc[h][nt][0], a.act) * acc[h][nt][2]));
        if (n + 1 < v.n_cnt)
          a.h[static_cast<size_t>(v.pos0 + n + 1) * a.f + j] =
              __half_as_ushort(__float2half_rn(gelu(acc[h][nt][1], a.act) * acc[h][nt][3]));
      }
    }
    if (a.last == 1) {
      // report the h rows to the expert's counter: __syncwarp orders the lanes' stores before
      // lane 0's release, which is cumulative at device scope
      __syncwarp();
      if (lane == 0) asm volatile("red.release.gpu.global.add.s32 [%0], 1;" ::"l"(a.gu_done + v.e) : "memory");
    }
  } else {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int n = 8 * nt + 2 * tq;
      const int p0 = n < v.n_cnt ? a.pair_list[v.pos0 + n] : 0;
      const int p1 = n + 1 < v.n_cnt ? a.pair_list[v.pos0 + n + 1] : 0;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int i_row = kBlockRows * v.blk + 16 * (2 * sw + h) + gq;
        if (n < v.n_cnt) {
          float* yr = a.y_out + static_cast<size_t>(p0) * a.d + i_row;
          yr[0] = acc[h][nt][0];
          yr[8] = acc[h][nt][2];
        }
        if (n + 1 < v.n_cnt) {
          float* yr = a.y_out + static_cast<size_t>(p1) * a.d + i_row;
          yr[0] = acc[h][nt][1];
          yr[8] = acc[h][nt][3];
        }
      }
    }
  }
  return true;
}

template <int G, bool GF, bool AF>
__device__ __forceinline__ bool run_item_g(const MmArgs& a, MmHeader& H, volatile int* abort, const ItemView& v,
                                           int& slot, uint32_t& phase, uint32_t ring_s, const uint32_t (&loff)[4],
                                           int sw, int lane) {
  const int nt = (v.n_cnt + 7) / 8;
  if constexpr (GF)  // items of at most kChunkGf tokens
    return nt == 1 ? run_item<1, G, true, AF>(a, H, abort, v, slot, phase, ring_s, loff, sw, lane)
                   : run_item<2, G, true, AF>(a, H, abort, v, slot, phase, ring_s, loff, sw, lane);
  switch (nt) {
    case 1: return run_item<1, G, false, AF>(a, H, abort, v, slot, phase, ring_s, loff, sw, lane);
    case 2: return run_item<2, G, false, AF>(a, H, abort, v, slot, phase, ring_s, loff, sw, lane);
    case 3: return run_item<3, G, false, AF>(a, H, abort, v, slot, phase, ring_s, loff, sw, lane);
    default: return run_item<4, G, false, AF>(a, H, abort, v, slot, phase, ring_s, loff, sw, lane);
  }
}

// GF: the group-factorised reduction order; AF: the affine weight format (its own
// instantiations, so that each gets its own register allocation; the symmetric
// format is the asymmetric one with every zero-point 8).
template <bool GF, bool AF>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
    expert_gemm_mma_kernel(const MmArgs a, const __grid_constant__ CUtensorMap map_x,
                           const __grid_constant__ CUtensorMap map_h) {
  constexpr int kChunk = GF ? kChunkGf : kChunkN;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  MmHeader& H = *reinterpret_cast<MmHeader*>(smem);
  uint8_t* ring = smem + kHeaderBytes;
  volatile int* abort = &H.abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(smem_addr(&H.slot_full[i]), 1);
      mbar_init(smem_addr(&H.slot_empty[i]), kMmaWarps);
    }
    for (int i = 0; i < kQueue; ++i) {
      mbar_init(smem_addr(&H.item_full[i]), 1);
      mbar_init(smem_addr(&H.item_empty[i]), kMmaWarps);
    }
    H.abort = 0;
    fence_barrier_init();
  }
  // everything above is set-up; the routing arrays, the row copy and h come from earlier launches
  grid_dependents_launch();
  grid_dependency_wait();
  if (warp == 1) gemm::scan_items(a, kChunk, lane, H.prefix, H.offs);
  __syncthreads();
  // the launch's work list: [gate_up items][down items], restricted to projections first..last
  const int total0 = a.first == 0 ? H.prefix[0][a.E] : 0;
  const int total = total0 + (a.last == 1 ? H.prefix[1][a.E] : 0);

  if (warp == 0) {
    // ------------------------------------------------------------------ producer
    // (the whole warp waits, lane 0 writes and issues)
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(&map_x) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(&map_h) : "memory");
    }
    // every weight byte is read once: it leaves L2 first, so that h, y and the token rows stay
    const uint64_t w_policy = l2_evict_first_policy();
    uint32_t issued_mask = 0;  // slots whose last phase carried copies
    uint32_t issued_par = 0;   // parity of that phase, one bit per slot
    bool ok = true;
    int t = 0;
    int next = 0;
    if (lane == 0) next = atomicAdd(a.counter, 1);  // claimed one item ahead
    for (int i = 0; ok; ++i) {
      const int item = __shfl_sync(0xffffffffu, next, 0);
      const bool done = item >= total;
      if (lane == 0 && !done) next = atomicAdd(a.counter, 1);
      const int pj = (a.first == 0 && item < total0) ? 0 : 1;
      int e = 0, blk = 0, n_cnt = 0, pos0 = 0;
      if (!done) decode_item(pj == 0 ? item : item - total0, H.prefix[pj], H.offs, a.E, kChunk, e, blk, n_cnt, pos0);
      ok = warp_wait(smem_addr(&H.item_empty[i % kQueue]), ((i / kQueue) & 1) ^ 1, a, abort);
      if (!ok) break;
      if (lane == 0) {
        H.item_desc[i % kQueue][0] = done ? -1 : (pj | (n_cnt << 8) | (blk << 16));
        H.item_desc[i % kQueue][1] = e;
        H.item_desc[i % kQueue][2] = pos0;
        mbar_arrive(smem_addr(&H.item_full[i % kQueue]));  // release: the entry is visible to its waiters
      }
      __syncwarp();
      if (done) break;
      if (pj == 1 && a.first == 0) {
        // a down item reads the h rows of its expert: wait until every gate_up warp of the
        // expert has written them
        if (lane == 0) {
          const int need = kMmaWarps * a.p[0].nblocks * ((H.offs[e + 1] - H.offs[e] + kChunk - 1) / kChunk);
          ok = wait_count(a.gu_done + e, need, a.err, abort, kDepWaitNs);
          // the TMA loads below read those rows through the async proxy
          asm volatile("fence.proxy.async.global;" ::: "memory");
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok) break;
      }
      const gemm::Proj& P = a.p[pj];
      const CUtensorMap* bmap = pj == 0 ? &map_x : &map_h;
      const uint8_t* wsrc = P.w + static_cast<int64_t>(e) * P.expert_bytes + static_cast<int64_t>(blk) * P.block_bytes;
      for (int c0 = 0; c0 < P.K; c0 += kStageCols, ++t) {
        const int slot = t % kSlots;
        const uint32_t par = static_cast<uint32_t>(t / kSlots) & 1u;
        ok = warp_wait(smem_addr(&H.slot_empty[slot]), par ^ 1u, a, abort);
        if (!ok) break;
        const int kk16 = min(kStageCols, P.K - c0) / 16;  // 8, or 4 for a last 64-column stage
        const uint32_t wbytes = stage_weight_bytes(kk16, P.g);
        if (lane == 0) {
          const uint32_t full = smem_addr(&H.slot_full[slot]);
          const uint32_t dst = smem_addr(ring + slot * kSlotBytes);
          mbar_arrive_expect_tx(full, (kk16 / 4) * kBoxBytes + wbytes);
          bulk_g2s_hint(dst + kBBytes, wsrc, wbytes, full, w_policy);
          tma_load_2d(dst, bmap, c0, pos0, full);
          if (kk16 == 8) tma_load_2d(dst + kBoxBytes, bmap, c0 + 64, pos0, full);
        }
        __syncwarp();
        wsrc += wbytes;
        issued_mask |= 1u << slot;
        issued_par = (issued_par & ~(1u << slot)) | (par << slot);
      }
    }
    // drain: every copy issued has landed before the CTA can exit
    if (lane == 0)
      for (int i = 0; i < kSlots; ++i)
        if ((issued_mask >> i) & 1u) mbar_wait(smem_addr(&H.slot_full[i]), (issued_par >> i) & 1u, a.err);
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ compute warps
    const int sw = warp - 1;  // the warp's strips 2 sw and 2 sw + 1 of the block
    // ldmatrix: lanes 0-7 / 8-15 / 16-23 / 24-31 address token rows 0-7 / 0-7 / 8-15 / 8-15 at the
    // step's first / second / first / second 8 columns; the token tile is 128-byte swizzled (the
    // 16-byte chunk c of token row n sits at chunk c ^ (n & 7))
    uint32_t loff[4];
    {
      const int lrow = ((lane >> 4) << 3) + (lane & 7), lhi = (lane >> 3) & 1;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) loff[kk] = lrow * 128 + ((((2 * kk + lhi) ^ (lrow & 7))) << 4);
    }
    const uint32_t ring_s = smem_addr(ring);
    int slot = 0;
    uint32_t phase = 0;
    for (int i = 0;; ++i) {
      if (!warp_wait(smem_addr(&H.item_full[i % kQueue]), (i / kQueue) & 1, a, abort)) break;
      ItemView v;
      if (!read_item(H, i, a, v)) break;
      const bool ok = v.g == 32   ? run_item_g<32, GF, AF>(a, H, abort, v, slot, phase, ring_s, loff, sw, lane)
                      : v.g == 64 ? run_item_g<64, GF, AF>(a, H, abort, v, slot, phase, ring_s, loff, sw, lane)
                                  : run_item_g<128, GF, AF>(a, H, abort, v, slot, phase, ring_s, loff, sw, lane);
      if (!ok) break;
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&H.item_empty[i % kQueue]));
    }
  }
  __syncthreads();
  // The last CTA to finish clears the work counter for the next launch on this
  // workspace: by then every CTA has seen the list exhausted and claims no more.
  if (tid == 0 && atomicAdd(a.done_ctas, 1) == static_cast<int>(gridDim.x) - 1) {
    *a.counter = 0;
    *a.done_ctas = 0;
  }
}

// Self-test of the bounded waits above: one warp waits, with the given bound, on
// an mbarrier phase that nothing completes and then on a counter that nothing
// raises (flag, left at 0); each wait gives up, records MOE_W4A16_ERR_TIMEOUT in
// *err and the kernel returns.  Nothing is in flight when it returns.
__global__ void __launch_bounds__(32) wait_selftest_kernel(int32_t* err, const int32_t* flag, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort;
  if (threadIdx.x == 0) {
    mbar_init(smem_addr(&bar), 1);  // one arrival that never comes
    abort = 0;
    fence_barrier_init();
  }
  __syncwarp();
  volatile int* ab = &abort;
  gemm::warp_wait(smem_addr(&bar), 0, err, ab, limit_ns);
  __syncwarp();
  if (threadIdx.x == 0) {
    *ab = 0;  // the counter wait is timed on its own
    wait_count(flag, 1, err, ab, limit_ns);
  }
}

}  // namespace

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

namespace {
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
}  // namespace

// 2-D tensor map over rows x cols fp16 (row-major), box 64 columns x 32 rows, 128-byte swizzle.
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
  const cuuint32_t box[2] = {kBoxCols, kRowBoxRows};
  const cuuint32_t estr[2] = {1, 1};
  return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_gather_rows(const Dims& s, const uint16_t* x, const int32_t* pair_list, const GemmWorkspace& ws,
                               cudaStream_t st) {
  const int P = static_cast<int>(s.pairs());
  return launch_pdl(gather_rows_kernel, dim3((P + 7) / 8), dim3(256), 0, st, x, pair_list, P, s.k, s.d, ws.xs,
                    ws.gu_done, s.E);
}

cudaError_t init_gemm_kernels() {
  for (const void* fn : {reinterpret_cast<const void*>(expert_gemm_mma_kernel<false, false>),
                         reinterpret_cast<const void*>(expert_gemm_mma_kernel<true, false>),
                         reinterpret_cast<const void*>(expert_gemm_mma_kernel<false, true>),
                         reinterpret_cast<const void*>(expert_gemm_mma_kernel<true, true>)}) {
    cudaError_t err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (err != cudaSuccess) return err;
    err = cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (err != cudaSuccess) return err;
  }
  return cudaSuccess;
}

cudaError_t launch_wait_selftest(int32_t* err, const int32_t* flag, uint64_t limit_ns, cudaStream_t st) {
  wait_selftest_kernel<<<1, 32, 0, st>>>(err, flag, limit_ns);
  return cudaGetLastError();
}

cudaError_t launch_expert_gemm(int which, const Dims& s, const uint16_t* x, const int32_t* expert_offsets,
                               const int32_t* pair_list, const uint8_t* w_gate_up, const uint8_t* w_down,
                               const GemmWorkspace& ws, int num_sms, cudaStream_t st) {
  MmArgs a;
  if (!gemm::make_args(a, which, s, expert_offsets, pair_list, w_gate_up, w_down, ws)) return cudaErrorInvalidValue;
  if (which & kGemmGateUp) {
    // the token rows are first copied in expert order
    const cudaError_t err = launch_gather_rows(s, x, pair_list, ws, st);
    if (err != cudaSuccess) return err;
  }
  const int P = static_cast<int>(s.pairs());
  CUtensorMap map_x, map_h;
  if (!make_row_map(&map_x, ws.xs, P, s.d) || !make_row_map(&map_h, ws.h, P, s.f)) return cudaErrorInvalidValue;
  auto* kern = s.fmt == 1 ? (s.red ? expert_gemm_mma_kernel<true, true> : expert_gemm_mma_kernel<false, true>)
                          : (s.red ? expert_gemm_mma_kernel<true, false> : expert_gemm_mma_kernel<false, false>);
  return launch_pdl(kern, dim3(num_sms * kCtasPerSm), dim3(kThreads), kSmemBytes, st, a, map_x, map_h);
}

}  // namespace moe
