// api.cpp -- the C ABI: host-side validation, workspace carve-up and the launch
// sequence of route and forward.  Nothing here reads device data, allocates
// device memory or synchronises the host (except moe_w4a16_read_error).
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda_runtime.h>

#include "internal.h"
#include "moe_w4a16.h"

namespace moe {

moe_w4a16_status check_shape(const moe_w4a16_shape* sh, Dims* out) {
  const auto pow2_group = [](int g) { return g == 32 || g == 64 || g == 128; };
  if (!sh) return MOE_W4A16_ERR_NULL;
  const Dims s{sh->tokens, sh->hidden, sh->inter, sh->experts, sh->top_k, sh->group_gate_up, sh->group_down,
               sh->activation, sh->reduction, sh->format};
  if (s.T < 0) return MOE_W4A16_ERR_SHAPE;
  if (s.d < 128 || s.d % 128 != 0 || s.d > 8192) return MOE_W4A16_ERR_SHAPE;
  if (s.f < 64 || s.f % 64 != 0 || s.f > 16384) return MOE_W4A16_ERR_SHAPE;
  if (s.E < 1 || s.E > moe::kMaxExperts) return MOE_W4A16_ERR_SHAPE;
  if (s.k < 1 || s.k > moe::kMaxTopK || s.k > s.E) return MOE_W4A16_ERR_SHAPE;
  if (!pow2_group(s.g1) || s.d % s.g1 != 0) return MOE_W4A16_ERR_SHAPE;
  if (!pow2_group(s.g2) || s.f % s.g2 != 0) return MOE_W4A16_ERR_SHAPE;
  if (s.act != 0 && s.act != 1) return MOE_W4A16_ERR_SHAPE;
  if (s.red != 0 && s.red != 1) return MOE_W4A16_ERR_SHAPE;
  if (s.fmt < 0 || s.fmt > 2) return MOE_W4A16_ERR_SHAPE;
  if (s.pairs() > moe::kMaxPairs) return MOE_W4A16_ERR_SHAPE;
  if (out) *out = s;
  return MOE_W4A16_OK;
}

}  // namespace moe

namespace {

using moe::check_shape;
using moe::Dims;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Per-device state: checked compute capability, kernel attributes, SM count.
struct DeviceState {
  bool ready = false;
  moe_w4a16_status status = MOE_W4A16_OK;
  int num_sms = 0;
};
constexpr int kMaxDevices = 64;
DeviceState g_dev[kMaxDevices];
std::mutex g_dev_mutex;

moe_w4a16_status device_state(const DeviceState** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_W4A16_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_dev_mutex);
  DeviceState& st = g_dev[dev];
  if (!st.ready) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      return MOE_W4A16_ERR_CUDA;
    }
    if (major != 10 || minor != 3) {
      st.status = MOE_W4A16_ERR_DEVICE;
    } else {
      st.num_sms = sms;
      st.status = (moe::init_gemm_kernels() == cudaSuccess && moe::init_block_kernels() == cudaSuccess)
                      ? MOE_W4A16_OK
                      : MOE_W4A16_ERR_CUDA;
    }
    st.ready = true;
  }
  *out = &st;
  return st.status;
}

moe_w4a16_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_W4A16_OK : MOE_W4A16_ERR_CUDA; }

}  // namespace

extern "C" {

size_t moe_w4a16_workspace_bytes(const moe_w4a16_shape* shape) {
  Dims s;
  if (check_shape(shape, &s) != MOE_W4A16_OK) return 0;
  return moe::ws_total(s);
}

moe_w4a16_status moe_w4a16_workspace_init(void* workspace, size_t workspace_bytes, void* stream) {
  if (!workspace) return MOE_W4A16_ERR_NULL;
  if (!aligned16(workspace)) return MOE_W4A16_ERR_ALIGN;
  if (workspace_bytes < sizeof(moe::WsHeader)) return MOE_W4A16_ERR_WORKSPACE;
  return cuda_status(cudaMemsetAsync(workspace, 0, sizeof(moe::WsHeader), static_cast<cudaStream_t>(stream)));
}

moe_w4a16_status moe_w4a16_selftest_wait_timeout(void* workspace, size_t workspace_bytes, uint64_t limit_ns,
                                                void* stream) {
  if (!workspace) return MOE_W4A16_ERR_NULL;
  if (!aligned16(workspace)) return MOE_W4A16_ERR_ALIGN;
  if (workspace_bytes < sizeof(moe::WsHeader)) return MOE_W4A16_ERR_WORKSPACE;
  if (limit_ns == 0 || limit_ns > 2000000000ull) return MOE_W4A16_ERR_VALUE;
  moe_w4a16_status st;
  const DeviceState* dev = nullptr;
  if ((st = device_state(&dev)) != MOE_W4A16_OK) return st;
  auto* hdr = static_cast<moe::WsHeader*>(workspace);
  return cuda_status(moe::launch_wait_selftest(&hdr->error, &hdr->never_set, limit_ns, static_cast<cudaStream_t>(stream)));
}

namespace {
bool sampler_ok(const moe_w4a16_sampler* c) {
  return c->positions >= 1 && c->positions <= moe::kSamplerMaxPositions && c->vocab >= 4 && c->vocab % 4 == 0 &&
         c->vocab <= (1 << 30) && c->inv_temperature > 0.f && c->inv_temperature <= 3.4e38f &&
         (c->rule == 0 || c->rule == 1) && c->bound >= -3.4e38f && c->bound <= 3.4e38f &&
         (c->noise == 0 || c->noise == 1);
}
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }
}  // namespace

size_t moe_w4a16_sampler_workspace_bytes(const moe_w4a16_sampler* cfg) {
  if (!cfg || !sampler_ok(cfg)) return 0;
  return moe::sampler_ws_bytes(cfg->positions, cfg->vocab);
}

moe_w4a16_status moe_w4a16_sample(const moe_w4a16_sampler* cfg, const float* logits, const uint8_t* revealed,
                                  int32_t* token, float* entropy, float* pmax, uint8_t* accept, void* workspace,
                                  size_t workspace_bytes, void* stream) {
  if (!cfg) return MOE_W4A16_ERR_NULL;
  if (!sampler_ok(cfg)) return MOE_W4A16_ERR_SHAPE;
  if (!logits || !revealed || !token || !entropy || !pmax || !accept || !workspace) return MOE_W4A16_ERR_NULL;
  if (!aligned16(logits) || !aligned16(workspace) || !aligned4(token) || !aligned4(entropy) || !aligned4(pmax))
    return MOE_W4A16_ERR_ALIGN;
  if (workspace_bytes < moe::sampler_ws_bytes(cfg->positions, cfg->vocab)) return MOE_W4A16_ERR_WORKSPACE;
  moe_w4a16_status st;
  const DeviceState* dev = nullptr;
  if ((st = device_state(&dev)) != MOE_W4A16_OK) return st;
  return cuda_status(moe::launch_sample(cfg->positions, cfg->vocab, cfg->inv_temperature, cfg->seed, cfg->step,
                                        cfg->rule, cfg->bound, cfg->noise, logits, revealed, token, entropy, pmax,
                                        accept, workspace, static_cast<cudaStream_t>(stream)));
}

moe_w4a16_status moe_w4a16_route(const moe_w4a16_shape* shape, const float* logits, const moe_w4a16_routing* out,
                                 void* workspace, size_t workspace_bytes, void* stream) {
  Dims s;
  moe_w4a16_status st = check_shape(shape, &s);
  if (st != MOE_W4A16_OK) return st;
  if (!out) return MOE_W4A16_ERR_NULL;
  if (s.T == 0) return MOE_W4A16_OK;
  if (!logits || !out->topk_idx || !out->topk_w || !out->expert_offsets || !out->pair_list || !workspace)
    return MOE_W4A16_ERR_NULL;
  if (!aligned16(logits) || !aligned16(out->topk_idx) || !aligned16(out->topk_w) ||
      !aligned16(out->expert_offsets) || !aligned16(out->pair_list) || !aligned16(workspace))
    return MOE_W4A16_ERR_ALIGN;
  if (workspace_bytes < moe::ws_total(s)) return MOE_W4A16_ERR_WORKSPACE;
  const DeviceState* dev = nullptr;
  if ((st = device_state(&dev)) != MOE_W4A16_OK) return st;
  return cuda_status(moe::launch_route(s, logits, out->topk_idx, out->topk_w, out->expert_offsets, out->pair_list,
                                       workspace, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

namespace {

// Steps of the forward pass (bit mask).
constexpr int kGateUp = 1, kDown = 2, kCombine = 4;

struct FwdArgs {
  const uint16_t* x;
  const moe_w4a16_routing* routing;
  const moe_w4a16_weights* weights;
  const float* gamma;
  float eps;
  uint16_t* out;
  void* ws;
  size_t ws_bytes;
  void* stream;
  bool clear_header;  // clear the workspace header (error word, work counters) before the launches
  const uint16_t* residual = nullptr;  // combine: out = fp16(residual + u) (the MoE block)
};

// Validates what the requested steps read and write, then launches them in order.
moe_w4a16_status run_forward_steps(const moe_w4a16_shape* shape, int steps, const FwdArgs& a) {
  Dims s;
  moe_w4a16_status st = check_shape(shape, &s);
  if (st != MOE_W4A16_OK) return st;
  if (!a.routing || ((steps & (kGateUp | kDown)) && !a.weights)) return MOE_W4A16_ERR_NULL;
  if (s.T == 0) return MOE_W4A16_OK;
  const moe_w4a16_routing& r = *a.routing;
  if (!a.ws) return MOE_W4A16_ERR_NULL;
  if ((steps & (kGateUp | kDown)) && (!r.expert_offsets || !r.pair_list)) return MOE_W4A16_ERR_NULL;
  if ((steps & kGateUp) && (!a.x || !a.weights->gate_up)) return MOE_W4A16_ERR_NULL;
  if ((steps & kDown) && !a.weights->down) return MOE_W4A16_ERR_NULL;
  if ((steps & kCombine) && (!r.topk_w || !a.out)) return MOE_W4A16_ERR_NULL;
  if (!aligned16(a.ws)) return MOE_W4A16_ERR_ALIGN;
  if ((steps & (kGateUp | kDown)) && (!aligned16(r.expert_offsets) || !aligned16(r.pair_list)))
    return MOE_W4A16_ERR_ALIGN;
  if ((steps & kGateUp) && (!aligned16(a.x) || !aligned16(a.weights->gate_up))) return MOE_W4A16_ERR_ALIGN;
  if ((steps & kDown) && !aligned16(a.weights->down)) return MOE_W4A16_ERR_ALIGN;
  if ((steps & kCombine) && (!aligned16(r.topk_w) || !aligned16(a.out) || (a.gamma && !aligned16(a.gamma))))
    return MOE_W4A16_ERR_ALIGN;
  if (a.ws_bytes < moe::ws_total(s)) return MOE_W4A16_ERR_WORKSPACE;
  if ((steps & kCombine) && !(a.eps >= 0.f)) return MOE_W4A16_ERR_VALUE;
  const DeviceState* dev = nullptr;
  if ((st = device_state(&dev)) != MOE_W4A16_OK) return st;
  const moe::GemmWorkspace ws = moe::carve_workspace(a.ws, s);
  const auto cs = static_cast<cudaStream_t>(a.stream);
  if (a.clear_header && cudaMemsetAsync(ws.hdr, 0, sizeof(moe::WsHeader), cs) != cudaSuccess)
    return MOE_W4A16_ERR_CUDA;
  // gate_up and down together run as one launch (down items wait for their expert's h rows)
  const int gemm = ((steps & kGateUp) ? moe::kGemmGateUp : 0) | ((steps & kDown) ? moe::kGemmDown : 0);
  if (gemm && moe::launch_expert_gemm(gemm, s, a.x, r.expert_offsets, r.pair_list,
                                      (steps & kGateUp) ? a.weights->gate_up : nullptr,
                                      (steps & kDown) ? a.weights->down : nullptr, ws, dev->num_sms, cs) != cudaSuccess)
    return MOE_W4A16_ERR_CUDA;
  if ((steps & kCombine) &&
      moe::launch_combine(s, r.topk_w, ws.y, a.gamma, a.eps, a.residual, a.out, cs) != cudaSuccess)
    return MOE_W4A16_ERR_CUDA;
  return MOE_W4A16_OK;
}

}  // namespace

moe_w4a16_status moe::forward_all_steps(const moe_w4a16_shape* shape, const uint16_t* x,
                                        const moe_w4a16_routing* routing, const moe_w4a16_weights* weights,
                                        const float* norm_gamma, float norm_eps, uint16_t* out, void* workspace,
                                        size_t workspace_bytes, void* stream, bool clear_header) {
  return run_forward_steps(shape, kGateUp | kDown | kCombine,
                           FwdArgs{x, routing, weights, norm_gamma, norm_eps, out, workspace, workspace_bytes, stream,
                                   clear_header});
}

extern "C" {

moe_w4a16_status moe_w4a16_forward(const moe_w4a16_shape* shape, const uint16_t* x, const moe_w4a16_routing* routing,
                                   const moe_w4a16_weights* weights, const float* norm_gamma, float norm_eps,
                                   uint16_t* out, void* workspace, size_t workspace_bytes, void* stream) {
  return run_forward_steps(shape, kGateUp | kDown | kCombine,
                           FwdArgs{x, routing, weights, norm_gamma, norm_eps, out, workspace, workspace_bytes, stream, false});
}

moe_w4a16_status moe_w4a16_experts(const moe_w4a16_shape* shape, const uint16_t* x, const moe_w4a16_routing* routing,
                                   const moe_w4a16_weights* weights, void* workspace, size_t workspace_bytes,
                                   void* stream) {
  return run_forward_steps(shape, kGateUp | kDown,
                           FwdArgs{x, routing, weights, nullptr, 0.f, nullptr, workspace, workspace_bytes, stream, false});
}

moe_w4a16_status moe_w4a16_gate_up(const moe_w4a16_shape* shape, const uint16_t* x, const moe_w4a16_routing* routing,
                                   const moe_w4a16_weights* weights, void* workspace, size_t workspace_bytes,
                                   void* stream) {
  return run_forward_steps(shape, kGateUp,
                           FwdArgs{x, routing, weights, nullptr, 0.f, nullptr, workspace, workspace_bytes, stream, false});
}

moe_w4a16_status moe_w4a16_down(const moe_w4a16_shape* shape, const moe_w4a16_routing* routing,
                                const moe_w4a16_weights* weights, void* workspace, size_t workspace_bytes,
                                void* stream) {
  return run_forward_steps(shape, kDown,
                           FwdArgs{nullptr, routing, weights, nullptr, 0.f, nullptr, workspace, workspace_bytes, stream, false});
}

moe_w4a16_status moe_w4a16_combine(const moe_w4a16_shape* shape, const moe_w4a16_routing* routing,
                                   const float* norm_gamma, float norm_eps, uint16_t* out, void* workspace,
                                   size_t workspace_bytes, void* stream) {
  return run_forward_steps(shape, kCombine, FwdArgs{nullptr, routing, nullptr, norm_gamma, norm_eps, out, workspace,
                                                    workspace_bytes, stream, false});
}

moe_w4a16_status moe_w4a16_block_front(const moe_w4a16_shape* shape, const uint16_t* x, const float* norm_gamma,
                                       float norm_eps, const uint16_t* router_w, uint16_t* u, float* logits,
                                       void* stream) {
  Dims s;
  moe_w4a16_status st = check_shape(shape, &s);
  if (st != MOE_W4A16_OK) return st;
  if (s.d % 256 != 0) return MOE_W4A16_ERR_SHAPE;
  if (s.T == 0) return MOE_W4A16_OK;
  if (!x || !norm_gamma || !router_w || !u || !logits) return MOE_W4A16_ERR_NULL;
  if (!aligned16(x) || !aligned16(norm_gamma) || !aligned16(router_w) || !aligned16(u) || !aligned16(logits))
    return MOE_W4A16_ERR_ALIGN;
  if (!(norm_eps >= 0.f) || !(norm_eps <= 3.4e38f)) return MOE_W4A16_ERR_VALUE;
  const DeviceState* dev = nullptr;
  if ((st = device_state(&dev)) != MOE_W4A16_OK) return st;
  return cuda_status(moe::launch_block_front(s, x, norm_gamma, norm_eps, router_w, u, logits,
                                             static_cast<cudaStream_t>(stream)));
}

moe_w4a16_status moe_w4a16_block(const moe_w4a16_shape* shape, const uint16_t* x, const float* norm_gamma,
                                 float norm_eps, const uint16_t* router_w, const moe_w4a16_routing* routing,
                                 const moe_w4a16_weights* weights, uint16_t* out, void* workspace,
                                 size_t workspace_bytes, void* stream) {
  Dims s;
  moe_w4a16_status st = check_shape(shape, &s);
  if (st != MOE_W4A16_OK) return st;
  if (s.d % 256 != 0) return MOE_W4A16_ERR_SHAPE;
  if (!routing || !weights) return MOE_W4A16_ERR_NULL;
  if (s.T == 0) return MOE_W4A16_OK;
  const moe_w4a16_routing& r = *routing;
  if (!x || !norm_gamma || !router_w || !out || !workspace || !weights->gate_up || !weights->down || !r.topk_idx ||
      !r.topk_w || !r.expert_offsets || !r.pair_list)
    return MOE_W4A16_ERR_NULL;
  if (!aligned16(x) || !aligned16(norm_gamma) || !aligned16(router_w) || !aligned16(out) || !aligned16(workspace) ||
      !aligned16(weights->gate_up) || !aligned16(weights->down) || !aligned16(r.topk_idx) || !aligned16(r.topk_w) ||
      !aligned16(r.expert_offsets) || !aligned16(r.pair_list))
    return MOE_W4A16_ERR_ALIGN;
  if (workspace_bytes < moe::ws_total(s)) return MOE_W4A16_ERR_WORKSPACE;
  if (!(norm_eps >= 0.f) || !(norm_eps <= 3.4e38f)) return MOE_W4A16_ERR_VALUE;
  const DeviceState* dev = nullptr;
  if ((st = device_state(&dev)) != MOE_W4A16_OK) return st;
  auto* base = static_cast<uint8_t*>(workspace);
  auto* u = reinterpret_cast<uint16_t*>(base + moe::ws_u_offset(s));
  auto* logits = reinterpret_cast<float*>(base + moe::ws_logits_offset(s));
  const auto cs = static_cast<cudaStream_t>(stream);
  if (moe::launch_block_front(s, x, norm_gamma, norm_eps, router_w, u, logits, cs) != cudaSuccess ||
      moe::launch_route(s, logits, r.topk_idx, r.topk_w, r.expert_offsets, r.pair_list, workspace, cs) != cudaSuccess)
    return MOE_W4A16_ERR_CUDA;
  FwdArgs fa{u, routing, weights, nullptr, 0.f, out, workspace, workspace_bytes, stream, false};
  fa.residual = x;
  return run_forward_steps(shape, kGateUp | kDown | kCombine, fa);
}

moe_w4a16_status moe_w4a16_read_error(const void* workspace, size_t workspace_bytes, void* stream,
                                      moe_w4a16_status* device_status) {
  if (!workspace || !device_status) return MOE_W4A16_ERR_NULL;
  if (workspace_bytes < sizeof(moe::WsHeader)) return MOE_W4A16_ERR_WORKSPACE;
  int32_t code = 0;
  const auto cs = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(&code, workspace, sizeof(code), cudaMemcpyDeviceToHost, cs) != cudaSuccess ||
      cudaStreamSynchronize(cs) != cudaSuccess)
    return MOE_W4A16_ERR_CUDA;
  *device_status = static_cast<moe_w4a16_status>(code);
  return MOE_W4A16_OK;
}

const char* moe_w4a16_status_string(moe_w4a16_status status) {
  switch (status) {
    case MOE_W4A16_OK: return "ok";
    case MOE_W4A16_ERR_NULL: return "a required pointer is NULL";
    case MOE_W4A16_ERR_SHAPE: return "shape outside the supported set";
    case MOE_W4A16_ERR_ALIGN: return "a device pointer is not 16-byte aligned";
    case MOE_W4A16_ERR_WORKSPACE: return "workspace smaller than moe_w4a16_workspace_bytes()";
    case MOE_W4A16_ERR_CUDA: return "a CUDA runtime call or kernel launch failed";
    case MOE_W4A16_ERR_DEVICE: return "current device is not a compute capability 10.3 GPU";
    case MOE_W4A16_ERR_TIMEOUT: return "a device-side wait ran out";
    case MOE_W4A16_ERR_VALUE: return "value out of range";
  }
  return "unknown status";
}

}  // extern "C"
