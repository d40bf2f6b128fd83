// internal.h -- declarations shared by the library's translation units (host side).
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda.h>
#include <cuda_runtime.h>

#include <utility>

#include "moe_w4a16.h"

namespace moe {

// Tiling of the grouped dequant GEMMs (gate_up and down share it).
constexpr int kBlockRows = 128;   // GEMM rows per work item (gate_up: 64 gate + 64 up rows)
constexpr int kStripRows = 16;    // GEMM rows per compute warp (one m16n8k16 row tile)
constexpr int kStageCols = 128;   // contraction columns per pipeline stage (the last may have 64)
constexpr int kBoxCols = 64;      // contraction columns per TMA box of token rows (128 bytes)
constexpr int kRowBoxRows = 32;   // token rows per TMA box
constexpr int kChunkN = 32;       // tokens (pairs) per work item
constexpr int kMaxExperts = 256;
constexpr int kMaxHidden = 8192;
constexpr int kMaxTopK = 8;
constexpr int64_t kMaxPairs = int64_t(1) << 22;

// Workspace header (bytes at the start of the workspace).
struct WsHeader {
  int32_t error;          // sticky moe_w4a16_status of device-side failures
  int32_t next_item[2];   // work counters of GEMM launches with gate_up items (0) and of down-only launches (1)
  int32_t done_ctas[2];   // CTAs of such a launch that have finished (the last resets both)
  int32_t never_set;      // stays 0: the counter the wait self-test waits on
  int32_t pad[58];
};
static_assert(sizeof(WsHeader) == 256, "header is 256 bytes");

struct Dims {
  int T, d, f, E, k, g1, g2, act, red, fmt;
  int64_t pairs() const { return int64_t(T) * k; }
};

// Host-side validation of a layer shape (the rules of moe_w4a16_shape); fills *out
// when the shape is valid.
moe_w4a16_status check_shape(const moe_w4a16_shape* sh, Dims* out);

// The whole forward pass (gate_up + down in one launch, then the combine) on the
// given workspace, with the checks and launch sequence of moe_w4a16_forward; when
// clear_header is set the workspace header (error word, work counters) is cleared
// on the stream after the checks pass and before the first launch.
moe_w4a16_status forward_all_steps(const moe_w4a16_shape* shape, const uint16_t* x, const moe_w4a16_routing* routing,
                                   const moe_w4a16_weights* weights, const float* norm_gamma, float norm_eps,
                                   uint16_t* out, void* workspace, size_t workspace_bytes, void* stream,
                                   bool clear_header);

// Workspace carve-up: header | per-expert gate_up counters | h | xs | y | routing scratch.
inline size_t ws_cnt_offset() { return sizeof(WsHeader); }
inline size_t ws_h_offset() { return ws_cnt_offset() + size_t(kMaxExperts) * 4; }
inline size_t ws_h_bytes(const Dims& s) { return size_t(s.pairs()) * s.f * 2; }
inline size_t ws_xs_offset(const Dims& s) { return (ws_h_offset() + ws_h_bytes(s) + 255) / 256 * 256; }
inline size_t ws_xs_bytes(const Dims& s) { return size_t(s.pairs()) * s.d * 2; }
inline size_t ws_y_offset(const Dims& s) { return (ws_xs_offset(s) + ws_xs_bytes(s) + 255) / 256 * 256; }
inline size_t ws_y_bytes(const Dims& s) { return size_t(s.pairs()) * s.d * 4; }
// routing scratch: per-CTA expert counts of the top-k step (8 tokens per CTA), the pairs'
// ranks, then the expert totals
inline size_t ws_route_offset(const Dims& s) { return (ws_y_offset(s) + ws_y_bytes(s) + 255) / 256 * 256; }
inline size_t ws_route_hist_bytes(const Dims& s) {  // rounded to 16 bytes: the ranks are read as vectors
  return (size_t((s.T + 7) / 8) * s.E * 4 + 15) / 16 * 16;
}
inline size_t ws_route_bytes(const Dims& s) {
  return ws_route_hist_bytes(s) + size_t(s.pairs()) * 4 + size_t(kMaxExperts) * 4;
}
// the MoE block's normalised input u (fp16 [T][d]) and router logits (fp32 [T][E])
inline size_t ws_u_offset(const Dims& s) { return (ws_route_offset(s) + ws_route_bytes(s) + 255) / 256 * 256; }
inline size_t ws_u_bytes(const Dims& s) { return size_t(s.T) * s.d * 2; }
inline size_t ws_logits_offset(const Dims& s) { return (ws_u_offset(s) + ws_u_bytes(s) + 255) / 256 * 256; }
inline size_t ws_total(const Dims& s) { return ws_logits_offset(s) + size_t(s.T) * s.E * 4; }

// Device pointers of one workspace's parts.
struct GemmWorkspace {
  WsHeader* hdr;
  int32_t* gu_done;  // [kMaxExperts]
  uint16_t* h;       // [T*k][f]
  uint16_t* xs;      // [T*k][d]
  float* y;          // [T*k][d]
};
inline GemmWorkspace carve_workspace(void* ws, const Dims& s) {
  auto* base = static_cast<uint8_t*>(ws);
  return GemmWorkspace{static_cast<WsHeader*>(ws), reinterpret_cast<int32_t*>(base + ws_cnt_offset()),
                       reinterpret_cast<uint16_t*>(base + ws_h_offset()),
                       reinterpret_cast<uint16_t*>(base + ws_xs_offset(s)),
                       reinterpret_cast<float*>(base + ws_y_offset(s))};
}

// Launches kernel<<<grid, block, smem, st>>>(args...) allowing programmatic
// dependent launch: the kernel may start while the previous kernel on the
// stream finishes, and waits for it (griddepcontrol.wait) before it touches
// anything that kernel writes.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args&&... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Kernel launchers (defined in the .cu files).  Each returns the launch status.
cudaError_t launch_route(const Dims& s, const float* logits, int32_t* topk_idx, float* topk_w,
                         int32_t* expert_offsets, int32_t* pair_list, void* workspace, cudaStream_t st);

// Sets the GEMM kernels' attributes on the current device.  Called once per
// device before the first launch there.
cudaError_t init_gemm_kernels();

// Expert GEMMs.  which is a mask: kGemmGateUp (x -> h, with the copy of the
// token rows in expert order), kGemmDown (h -> y), or both in one launch (down
// items wait for their expert's gate_up items).  A persistent grid sized from
// the device's SM count.
constexpr int kGemmGateUp = 1, kGemmDown = 2;
cudaError_t launch_expert_gemm(int which, const Dims& s, const uint16_t* x, const int32_t* expert_offsets,
                               const int32_t* pair_list, const uint8_t* w_gate_up, const uint8_t* w_down,
                               const GemmWorkspace& ws, int num_sms, cudaStream_t st);

// The expert-order copy of the token rows (the gate_up items' TMA source), which
// also clears the per-expert gate_up counters.
cudaError_t launch_gather_rows(const Dims& s, const uint16_t* x, const int32_t* pair_list, const GemmWorkspace& ws,
                               cudaStream_t st);

// 2-D tensor map over a rows x cols fp16 row-major matrix: boxes of 64 columns x
// 32 rows, 128-byte swizzle.
bool make_row_map(CUtensorMap* map, const void* base, int64_t rows, int64_t cols);


// Combine (and optional RMSNorm, or optional residual add out = fp16(x + u); not both).
cudaError_t launch_combine(const Dims& s, const float* topk_w, const float* y, const float* gamma, float eps,
                           const uint16_t* residual, uint16_t* out, cudaStream_t st);

// The MoE block's pre-norm and router projection (block.cu): u fp16 [T][d] and the
// router logits fp32 [T][E] from the residual stream x.  d a multiple of 256.
cudaError_t init_block_kernels();
cudaError_t launch_block_front(const Dims& s, const uint16_t* x, const float* gamma, float eps, const uint16_t* wr,
                               uint16_t* u, float* logits, cudaStream_t st);

// Per-step sampler (sampler.cu): one streaming pass over the logits (grid of
// vocabulary splits x positions) writing 32-byte partials to the workspace, then
// one CTA that merges them and applies the acceptance rule.
constexpr int kSamplerMaxPositions = 1024;  // one thread per position in the final CTA
// Vocabulary elements per CTA of the pass: the vocabulary is cut into about
// ceil(912 / positions) splits (912 CTAs: two waves of three 256-thread CTAs on
// each of 152 SMs), each a multiple of 4,096 elements (a block of the per-group pass,
// whose 1,024 groups share 256 Philox counters; two iterations of the per-token pass).
// Fewer, longer CTAs amortise each CTA's start and final reduction.
inline int64_t sampler_chunk(int positions, int64_t vocab) {
  const int64_t want = (912 + positions - 1) / positions;
  const int64_t per = (vocab + want - 1) / want;
  return (per + 4095) / 4096 * 4096;
}
inline int sampler_splits(int positions, int64_t vocab) {
  return static_cast<int>((vocab + sampler_chunk(positions, vocab) - 1) / sampler_chunk(positions, vocab));
}
inline size_t sampler_ws_bytes(int positions, int64_t vocab) {
  return size_t(positions) * size_t(sampler_splits(positions, vocab)) * 32;
}
cudaError_t launch_sample(int P, int64_t V, float inv_temp, uint64_t seed, uint32_t step, int rule, float bound,
                          int noise, const float* logits, const uint8_t* revealed, int32_t* token, float* entropy, float* pmax,
                          uint8_t* accept, void* workspace, cudaStream_t st);

// Self-test of the expert launch's bounded waits: waits that cannot complete (an
// mbarrier phase, then the counter *flag, which must stay 0) give up after limit_ns
// each and record MOE_W4A16_ERR_TIMEOUT in *err.
cudaError_t launch_wait_selftest(int32_t* err, const int32_t* flag, uint64_t limit_ns, cudaStream_t st);

}  // namespace moe
