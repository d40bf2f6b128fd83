// internal.h -- declarations shared by the library's translation units (host side).
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "moe_w4a16.h"

namespace moe {

// Tiling of the grouped dequant GEMMs (gate_up and down share it).
constexpr int kBlockRows = 128;   // GEMM rows per work item (gate_up: 64 gate + 64 up rows)
constexpr int kStageK = 64;       // contraction columns per pipeline stage
constexpr int kChunkN = 32;       // tokens (pairs) per work item
constexpr int kMaxExperts = 256;
constexpr int kMaxTopK = 8;
constexpr int64_t kMaxPairs = int64_t(1) << 22;

// Workspace header (bytes at the start of the workspace).
struct WsHeader {
  int32_t error;          // sticky moe_w4a16_status of device-side failures
  int32_t next_item[2];   // dynamic work counters of the gate_up (0) and down (1) kernels
  uint32_t route_ticket;  // CTAs of the routing launch that have finished their top-k (reset by the last)
  int32_t pad[60];
};
static_assert(sizeof(WsHeader) == 256, "header is 256 bytes");

struct Dims {
  int T, d, f, E, k, g1, g2, act;
  int64_t pairs() const { return int64_t(T) * k; }
};

// Workspace carve-up.
inline size_t ws_h_offset() { return sizeof(WsHeader); }
inline size_t ws_h_bytes(const Dims& s) { return size_t(s.pairs()) * s.f * 2; }
inline size_t ws_y_offset(const Dims& s) { return (ws_h_offset() + ws_h_bytes(s) + 255) / 256 * 256; }
inline size_t ws_y_bytes(const Dims& s) { return size_t(s.pairs()) * s.d * 4; }
inline size_t ws_total(const Dims& s) { return ws_y_offset(s) + ws_y_bytes(s); }

// Kernel launchers (defined in the .cu files).  Each returns the launch status.
cudaError_t launch_route(const Dims& s, const float* logits, int32_t* topk_idx, float* topk_w,
                         int32_t* expert_offsets, int32_t* pair_list, WsHeader* hdr, cudaStream_t st);

// Sets the kernels' attributes on the current device and reports how many GEMM
// CTAs fit on one SM.  Called once per device before the first launch there.
cudaError_t init_gemm_kernels(int* blocks_per_sm);

// which = 0: gate_up GEMM (x -> h), which = 1: down GEMM (h -> y).
cudaError_t launch_expert_gemm(int which, const Dims& s, const uint16_t* x, const int32_t* expert_offsets,
                               const int32_t* pair_list, const uint8_t* w, uint16_t* h, float* y, WsHeader* hdr,
                               int grid, cudaStream_t st);

cudaError_t launch_combine(const Dims& s, const float* topk_w, const float* y, const float* gamma, float eps,
                           uint16_t* out, cudaStream_t st);

}  // namespace moe
