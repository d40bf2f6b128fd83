// gemm_mma.cu -- grouped W4A16 expert GEMMs with inline dequantisation
// (warp-level tensor-core MMA variant).
//
// Model card "srswti/axe-diffusion-ksl-xe", "the kernels we built": the GEMM
// reads packed nibbles and dequantises inline, so HBM carries real 4-bit
// traffic; one launch covers all experts; the activation is folded into the
// first GEMM's epilogue.  Two launches of one kernel template do the work:
//   gate_up:  a[p][n] = sum_k Wgu[e][n][k] x[t(p)][k]   (n over 64 gate + 64 up rows per item)
//             h[pos(p)][j] = gelu(a[p][j]) * a[p][f+j]  -> fp16, rows in expert-sorted order
//   down:     y[p][i] = sum_j Wd[e][i][j] h[pos(p)][j]   -> fp32, rows by pair id p = t*k + r
// with W = (q - z) * s rebuilt in registers from the prepared stream.
//
// Structure (per CTA, persistent, work items taken from a global counter):
//   warp 4      producer: 1-D bulk copies of each 64-column stage of the item's
//               weight stream (codes + scale/zero) and of the 64 activation
//               columns of every token row of the item, into a ring of
//               kStages shared-memory slots guarded by mbarriers;
//   warps 0..3  consumers: each owns two 16-row MMA tiles of the 128-row block,
//               dequantises its codes straight into MMA A fragments and runs
//               m16n8k16 MMAs against activation fragments read by ldmatrix.
// Weights are the M side ("swap AB"): an expert sees ~16 tokens per canvas, so
// tokens are the narrow N side (up to 64 per item, in 8-wide tiles).
//
// Arithmetic, in the group-factorised order of the "ashhart/TensorFold pull 802"
// thread (partial sums per group, then the scale): for each quantisation group
// the MMA runs on the fp16 value (q - z), exact except when |q - z| >= 8 needs a
// 12th significand bit, into fresh fp32 partial sums P; the group's scale is
// then applied in fp32, acc += s * P.  Per 32-bit word (8 codes) the dequantiser
// spends 13 instructions:
//   low nibble  -> 1024 + q by OR-ing exponent bits 0x6400 (q in the low mantissa bits),
//   high nibble -> 64 + q   by OR-ing exponent bits 0x5400 over bits 4..7,
//   then one fp16 add removes the offset (exactly) and one fp16 subtract forms q - z.
// No split-K and no atomics on data: each output element is produced by one
// thread in a fixed K order, so results do not depend on scheduling.
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kStages = 4;
constexpr int kCodeBytes = kBlockRows * kStageK / 2;        // 4096: codes of one stage
constexpr int kSzBytes = kBlockRows * 4;                    // 512: (scale, zero) of one group
constexpr int kABytes = kCodeBytes + 2 * kSzBytes;          // up to two groups start in a stage (g = 32)
constexpr int kBRowBytes = kStageK * 2 + 16;                // 144: 128 B of activations + 16 B pad (no bank conflicts)
constexpr int kSlotBytes = kABytes + kChunkN * kBRowBytes;  // 14336
constexpr int kHeaderBytes = 2048;
constexpr int kSmemBytes = kHeaderBytes + kStages * kSlotBytes;
static_assert(kSlotBytes % 128 == 0, "slots stay 128-byte aligned");
static_assert(16 * kStages + 8 * kStages + 4 * (kMaxExperts + 1) <= kHeaderBytes, "header fits");

struct GemmArgs {
  const uint8_t* w;           // prepared stream of the projection, all experts
  int64_t expert_bytes;       // stream bytes per expert
  int64_t block_bytes;        // stream bytes per 128-row block
  int nblocks;                // blocks per expert
  int K;                      // contraction length (multiple of 64)
  int g;                      // quantisation group along K
  const int32_t* offsets;     // [E+1]
  const int32_t* pair_list;   // [T*k]
  int E, topk;
  const uint16_t* bsrc;       // gate_up: x [T][d]; down: h [T*k][f] (expert-sorted rows)
  int bsrc_ld;                // elements per bsrc row
  uint16_t* h_out;            // gate_up output [T*k][f]
  float* y_out;               // down output [T*k][d]
  int f, d, act;
  int32_t* err;
  int32_t* counter;           // this launch's work counter (starts at 0)
  int32_t* counter_to_reset;  // the other launch's counter, zeroed for the next call
};

__device__ __forceinline__ int groups_in_stage(int s, int g) {
  return g <= kStageK ? kStageK / g : ((s * kStageK) % g == 0 ? 1 : 0);
}

// Work item -> (expert, 128-row block, token chunk).  Items are ordered by
// expert, then block, then chunk, and the chunk varies fastest so concurrent
// items of a busy expert share weight blocks in L2.
__device__ __forceinline__ void decode_item(int item, const int* prefix, const GemmArgs& a, int& blk, int& n_cnt,
                                            int& pos0, int& expert) {
  int lo = 0, hi = a.E - 1;
  while (lo < hi) {  // largest e with prefix[e] <= item
    const int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= item) lo = mid;
    else hi = mid - 1;
  }
  const int e = lo;
  const int n_e = a.offsets[e + 1] - a.offsets[e];
  const int nch = (n_e + kChunkN - 1) / kChunkN;
  const int r = item - prefix[e];
  const int c = r % nch;
  blk = r / nch;
  n_cnt = min(kChunkN, n_e - kChunkN * c);
  pos0 = a.offsets[e] + kChunkN * c;
  expert = e;
}

// 8 codes -> (q - z) in the four f16x2 registers of an m16n8k16 A fragment.
// zz[0] = (z, z) of row g, zz[1] = (z, z) of row g+8.
__device__ __forceinline__ void dequant8(uint32_t w, const uint32_t (&zz)[2], uint32_t (&af)[4]) {
  const uint32_t w8 = w >> 8;
  const __half2 r0 = bits_h2(and_or(w, 0x000f000fu, 0x64006400u));   // row g,   cols 2t, 2t+1   : 1024 + q
  const __half2 r1 = bits_h2(and_or(w, 0x00f000f0u, 0x54005400u));   // row g+8, cols 2t, 2t+1   : 64 + q
  const __half2 r2 = bits_h2(and_or(w8, 0x000f000fu, 0x64006400u));  // row g,   cols 2t+8, 2t+9
  const __half2 r3 = bits_h2(and_or(w8, 0x00f000f0u, 0x54005400u));  // row g+8, cols 2t+8, 2t+9
  const __half2 m1024 = bits_h2(0xe400e400u), m64 = bits_h2(0xd400d400u);  // -1024, -64
  af[0] = h2_bits(__hsub2(__hadd2(r0, m1024), bits_h2(zz[0])));
  af[1] = h2_bits(__hsub2(__hadd2(r1, m64), bits_h2(zz[1])));
  af[2] = h2_bits(__hsub2(__hadd2(r2, m1024), bits_h2(zz[0])));
  af[3] = h2_bits(__hsub2(__hadd2(r3, m64), bits_h2(zz[1])));
}

__device__ __forceinline__ float gelu(float a, int act) {
  if (act == 1) return 0.5f * a * (1.f + erff(a * 0.70710678118654752f));
  return 0.5f * a * (1.f + tanhf(0.79788456080286536f * (a + 0.044715f * a * a * a)));
}

template <int kEpi>  // 0: gate_up with GeGLU epilogue, 1: down projection
__global__ void __launch_bounds__(kThreads, 2) expert_gemm_kernel(const GemmArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + kStages;
  int* slot_item = reinterpret_cast<int*>(empty + kStages);
  int* slot_stage = slot_item + kStages;
  int* prefix = slot_stage + kStages;  // [E+1] work-item prefix per expert
  uint8_t* ring = smem + kHeaderBytes;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (blockIdx.x == 0 && tid == 0) *a.counter_to_reset = 0;
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_addr(&full[s]), 1);
      mbar_init(smem_addr(&empty[s]), kConsumerWarps);
    }
    fence_barrier_init();
  }
  if (warp == 0) {  // items per expert = blocks * ceil(n_e / 64); exclusive scan, 8 experts per lane
    int loc[8], sum = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int e = lane * 8 + j;
      loc[j] = sum;
      if (e < a.E) {
        const int n_e = a.offsets[e + 1] - a.offsets[e];
        sum += a.nblocks * ((n_e + kChunkN - 1) / kChunkN);
      }
    }
    int incl = sum;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += o;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (lane * 8 + j < a.E) prefix[lane * 8 + j] = incl - sum + loc[j];
    if (lane == 31) prefix[a.E] = incl;
  }
  __syncthreads();
  const int total = prefix[a.E];
  const int nst = a.K / kStageK;

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    int slot = 0;
    uint32_t phase = 0;
    for (;;) {
      int item = 0;
      if (lane == 0) item = atomicAdd(a.counter, 1);
      item = __shfl_sync(0xffffffffu, item, 0);
      const bool done = item >= total;
      int blk = 0, n_cnt = 0, pos0 = 0, e = 0;
      if (!done) decode_item(item, prefix, a, blk, n_cnt, pos0, e);
      const uint16_t* src0 = nullptr;
      const uint16_t* src1 = nullptr;
      if (lane < n_cnt) {
        const int pos = pos0 + lane;
        const int row = kEpi == 0 ? a.pair_list[pos] / a.topk : pos;
        src0 = a.bsrc + static_cast<size_t>(row) * a.bsrc_ld;
      }
      if (lane + 32 < n_cnt) {
        const int pos = pos0 + lane + 32;
        const int row = kEpi == 0 ? a.pair_list[pos] / a.topk : pos;
        src1 = a.bsrc + static_cast<size_t>(row) * a.bsrc_ld;
      }
      const uint8_t* wsrc = a.w + static_cast<int64_t>(e) * a.expert_bytes + static_cast<int64_t>(blk) * a.block_bytes;
      const int stages = done ? 1 : nst;
      for (int s = 0; s < stages; ++s) {
        const uint32_t full_bar = smem_addr(&full[slot]);
        if (!mbar_wait(smem_addr(&empty[slot]), phase ^ 1u, a.err)) return;
        const uint32_t a_bytes = kCodeBytes + kSzBytes * groups_in_stage(s, a.g);
        if (lane == 0) {
          slot_item[slot] = done ? -1 : item;
          slot_stage[slot] = s;
          if (done) mbar_arrive(full_bar);
          else mbar_arrive_expect_tx(full_bar, a_bytes + static_cast<uint32_t>(n_cnt) * (kStageK * 2));
        }
        __syncwarp();
        if (!done) {
          const uint32_t dst = smem_addr(ring + slot * kSlotBytes);
          if (lane == 0) bulk_g2s(dst, wsrc, a_bytes, full_bar);
          if (src0) bulk_g2s(dst + kABytes + lane * kBRowBytes, src0 + s * kStageK, kStageK * 2, full_bar);
          if (src1) bulk_g2s(dst + kABytes + (lane + 32) * kBRowBytes, src1 + s * kStageK, kStageK * 2, full_bar);
          wsrc += a_bytes;
        }
        if (++slot == kStages) {
          slot = 0;
          phase ^= 1u;
        }
      }
      if (done) break;
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int g8 = lane >> 2, t4 = lane & 3;
  float acc[2][8][4];
  float sc[2][2];     // scale of rows g and g+8 of each m-tile
  uint32_t zz[2][2];  // (z, z) of rows g and g+8 of each m-tile
#pragma unroll
  for (int mt = 0; mt < 2; ++mt) {
    sc[mt][0] = sc[mt][1] = 0.f;
    zz[mt][0] = zz[mt][1] = 0u;
  }
  int slot = 0;
  uint32_t phase = 0;
  int n_tiles = 0, n_cnt = 0, pos0 = 0, blk = 0, e = 0;
  // ldmatrix.x4 row address of this lane: matrices {k16 step j: cols 0-7, 8-15; step j+1: cols 0-7, 8-15}
  // of one 8-token tile, rows = tokens
  const uint32_t lm_off = static_cast<uint32_t>((lane & 7) * kBRowBytes + (lane >> 3) * 16);
  for (;;) {
    if (!mbar_wait(smem_addr(&full[slot]), phase, a.err)) return;
    const int item = slot_item[slot];
    const int s = slot_stage[slot];
    if (item < 0) break;
    if (s == 0) {
      decode_item(item, prefix, a, blk, n_cnt, pos0, e);
      n_tiles = (n_cnt + 7) >> 3;
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
          for (int i = 0; i < 4; ++i) acc[mt][nt][i] = 0.f;
    }
    const uint8_t* st = ring + slot * kSlotBytes;
    const int ngrp = groups_in_stage(s, a.g);
    const uint4* words = reinterpret_cast<const uint4*>(st + kSzBytes * ngrp);
    uint4 wv[2];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) wv[mt] = words[(2 * warp + mt) * 32 + lane];
    const uint32_t bbase = smem_addr(st + kABytes) + lm_off;
    // two halves of 32 columns; a group boundary can only fall at a half (g >= 32)
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const bool new_group = ((s * kStageK + half * 32) % a.g) == 0;
      if (new_group) {
        const int j = (a.g == 32) ? half : 0;
        const uint32_t* sz = reinterpret_cast<const uint32_t*>(st + j * kSzBytes);
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
#pragma unroll
          for (int hi = 0; hi < 2; ++hi) {
            const __half2 v = bits_h2(sz[16 * (2 * warp + mt) + g8 + 8 * hi]);  // (scale, zero)
            sc[mt][hi] = __low2float(v);
            zz[mt][hi] = h2_bits(__high2half2(v));
          }
        }
      }
      uint32_t af[2][2][4];  // [k16 step][m-tile][reg]
#pragma unroll
      for (int kq = 0; kq < 2; ++kq) {
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
          const int kk = half * 2 + kq;
          const uint32_t wd = kk == 0 ? wv[mt].x : kk == 1 ? wv[mt].y : kk == 2 ? wv[mt].z : wv[mt].w;
          dequant8(wd, zz[mt], af[kq][mt]);
        }
      }
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        if (nt >= n_tiles) continue;
        uint32_t b[4];
        ldmatrix_x4(bbase + nt * 8 * kBRowBytes + half * 64, b[0], b[1], b[2], b[3]);
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
          float p[4] = {0.f, 0.f, 0.f, 0.f};
          mma_f16_16816(p, af[0][mt], b[0], b[1]);
          mma_f16_16816(p, af[1][mt], b[2], b[3]);
          acc[mt][nt][0] = fmaf(sc[mt][0], p[0], acc[mt][nt][0]);
          acc[mt][nt][1] = fmaf(sc[mt][0], p[1], acc[mt][nt][1]);
          acc[mt][nt][2] = fmaf(sc[mt][1], p[2], acc[mt][nt][2]);
          acc[mt][nt][3] = fmaf(sc[mt][1], p[3], acc[mt][nt][3]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_addr(&empty[slot]));
    if (s == nst - 1) {
      // ------------------------------------------------------------ epilogue
#pragma unroll
      for (int mt = 0; mt < 2; ++mt) {
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
          if (nt >= n_tiles) continue;
          const int n0 = nt * 8 + 2 * t4;
          if (kEpi == 0) {
            const int j = 64 * blk + 8 * (2 * warp + mt) + g8;  // rows g = gate j, g+8 = up j
            if (n0 < n_cnt)
              a.h_out[static_cast<size_t>(pos0 + n0) * a.f + j] =
                  __half_as_ushort(__float2half_rn(gelu(acc[mt][nt][0], a.act) * acc[mt][nt][2]));
            if (n0 + 1 < n_cnt)
              a.h_out[static_cast<size_t>(pos0 + n0 + 1) * a.f + j] =
                  __half_as_ushort(__float2half_rn(gelu(acc[mt][nt][1], a.act) * acc[mt][nt][3]));
          } else {
            const int i = kBlockRows * blk + 16 * (2 * warp + mt) + g8;
            if (n0 < n_cnt) {
              float* yr = a.y_out + static_cast<size_t>(a.pair_list[pos0 + n0]) * a.d;
              yr[i] = acc[mt][nt][0];
              yr[i + 8] = acc[mt][nt][2];
            }
            if (n0 + 1 < n_cnt) {
              float* yr = a.y_out + static_cast<size_t>(a.pair_list[pos0 + n0 + 1]) * a.d;
              yr[i] = acc[mt][nt][1];
              yr[i + 8] = acc[mt][nt][3];
            }
          }
        }
      }
    }
    if (++slot == kStages) {
      slot = 0;
      phase ^= 1u;
    }
  }
}

}  // namespace

cudaError_t init_gemm_kernels(int* blocks_per_sm) {
  cudaError_t err = cudaFuncSetAttribute(expert_gemm_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (err != cudaSuccess) return err;
  err = cudaFuncSetAttribute(expert_gemm_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (err != cudaSuccess) return err;
  int bps = 0;
  err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&bps, expert_gemm_kernel<0>, kThreads, kSmemBytes);
  if (err != cudaSuccess) return err;
  *blocks_per_sm = bps > 0 ? bps : 1;
  return cudaSuccess;
}

cudaError_t launch_expert_gemm(int which, const Dims& s, const uint16_t* x, const int32_t* expert_offsets,
                               const int32_t* pair_list, const uint8_t* w, uint16_t* h, float* y, WsHeader* hdr,
                               int grid, cudaStream_t st) {
  GemmArgs a{};
  a.w = w;
  a.offsets = expert_offsets;
  a.pair_list = pair_list;
  a.E = s.E;
  a.topk = s.k;
  a.f = s.f;
  a.d = s.d;
  a.act = s.act;
  a.err = &hdr->error;
  a.h_out = h;
  a.y_out = y;
  if (which == 0) {  // gate_up: rows 2f in f/64 blocks of 64 gate + 64 up rows, K = d
    a.K = s.d;
    a.g = s.g1;
    a.nblocks = s.f / 64;
    a.bsrc = x;
    a.bsrc_ld = s.d;
    a.counter = &hdr->next_item[0];
    a.counter_to_reset = &hdr->next_item[1];
  } else {           // down: rows d in d/128 blocks, K = f
    a.K = s.f;
    a.g = s.g2;
    a.nblocks = s.d / kBlockRows;
    a.bsrc = h;
    a.bsrc_ld = s.f;
    a.counter = &hdr->next_item[1];
    a.counter_to_reset = &hdr->next_item[0];
  }
  a.block_bytes = int64_t(kBlockRows) * a.K / 2 + int64_t(kBlockRows) * (a.K / a.g) * 4;
  a.expert_bytes = a.block_bytes * a.nblocks;
  if (which == 0) expert_gemm_kernel<0><<<grid, kThreads, kSmemBytes, st>>>(a);
  else expert_gemm_kernel<1><<<grid, kThreads, kSmemBytes, st>>>(a);
  return cudaGetLastError();
}

}  // namespace moe
