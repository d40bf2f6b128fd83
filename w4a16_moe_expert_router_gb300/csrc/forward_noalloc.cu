// forward_noalloc.cu -- moe_w4a16_forward_noalloc: the forward pass (gate_up,
// down, combine) with its scratch memory in a fixed static device array, for
// callers that cannot allocate device memory themselves.
//
// The scratch (work counters and error word, the fp16 activations h and the
// fp32 per-pair outputs) lives in g_scratch below.  Every GPU that loads this
// library holds the array until the process exits.  All calls on a device share
// it, so calls whose work overlaps on the GPU race; the header part (counters,
// error word) is cleared at the start of every call, the rest is fully written
// before it is read.
#include <mutex>

#include <cuda_runtime.h>

#include "internal.h"
#include "moe_w4a16.h"

namespace {

constexpr size_t kScratchBytes = MOE_W4A16_NOALLOC_SCRATCH_BYTES;
static_assert(kScratchBytes % 256 == 0, "scratch size keeps the 256-byte alignment of its parts");

static __device__ __align__(256) uint8_t g_scratch[kScratchBytes];

struct NoallocDevice {
  bool ready = false;
  moe_w4a16_status status = MOE_W4A16_OK;
  uint8_t* scratch = nullptr;  // device address of g_scratch on this device
  int grid = 0;                // persistent GEMM grid
};
constexpr int kMaxDevices = 64;
NoallocDevice g_devices[kMaxDevices];
std::mutex g_mutex;

// One-time set-up per device, done by the first call on that device with the
// device current: resolve the device address of g_scratch (in host code the
// symbol's name is only a host-side stand-in) and set the GEMM kernels' attributes.
moe_w4a16_status device_setup(const NoallocDevice** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_W4A16_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mutex);
  NoallocDevice& st = g_devices[dev];
  if (!st.ready) {
    int major = 0, minor = 0, sms = 0, bps = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return MOE_W4A16_ERR_CUDA;
    if (major != 10 || minor != 3) {
      st.status = MOE_W4A16_ERR_DEVICE;
    } else {
      void* ptr = nullptr;
      if (cudaGetSymbolAddress(&ptr, g_scratch) != cudaSuccess || ptr == nullptr ||
          moe::init_gemm_kernels(&bps) != cudaSuccess) {
        return MOE_W4A16_ERR_CUDA;  // not marked ready: the next call retries
      }
      st.scratch = static_cast<uint8_t*>(ptr);
      st.grid = sms * bps;
      st.status = MOE_W4A16_OK;
    }
    st.ready = true;
  }
  *out = &st;
  return st.status;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" moe_w4a16_status moe_w4a16_forward_noalloc(const moe_w4a16_shape* shape, const uint16_t* x,
                                                      const moe_w4a16_routing* routing,
                                                      const moe_w4a16_weights* weights, const float* norm_gamma,
                                                      float norm_eps, uint16_t* out, void* stream) {
  if (!shape) return MOE_W4A16_ERR_NULL;
  const size_t need = moe_w4a16_workspace_bytes(shape);  // 0 for a shape outside the supported set
  if (need == 0) return MOE_W4A16_ERR_SHAPE;
  if (need > kScratchBytes) return MOE_W4A16_ERR_WORKSPACE;
  if (!routing || !weights) return MOE_W4A16_ERR_NULL;
  const moe::Dims s{shape->tokens, shape->hidden, shape->inter, shape->experts, shape->top_k, shape->group_gate_up,
                    shape->group_down, shape->activation};
  if (s.T == 0) return MOE_W4A16_OK;
  const moe_w4a16_routing& r = *routing;
  if (!x || !r.topk_w || !r.expert_offsets || !r.pair_list || !weights->gate_up || !weights->down || !out)
    return MOE_W4A16_ERR_NULL;
  if (!aligned16(x) || !aligned16(r.topk_w) || !aligned16(r.expert_offsets) || !aligned16(r.pair_list) ||
      !aligned16(weights->gate_up) || !aligned16(weights->down) || !aligned16(out) ||
      (norm_gamma && !aligned16(norm_gamma)))
    return MOE_W4A16_ERR_ALIGN;
  if (!(norm_eps >= 0.f)) return MOE_W4A16_ERR_VALUE;
  const NoallocDevice* dev = nullptr;
  moe_w4a16_status st = device_setup(&dev);
  if (st != MOE_W4A16_OK) return st;
  const auto cs = static_cast<cudaStream_t>(stream);
  const moe::GemmWorkspace ws = moe::carve_workspace(dev->scratch, s);
  if (cudaMemsetAsync(ws.hdr, 0, sizeof(moe::WsHeader), cs) != cudaSuccess) return MOE_W4A16_ERR_CUDA;
  if (moe::launch_expert_gemm(moe::kGemmGateUp | moe::kGemmDown, s, x, r.expert_offsets, r.pair_list,
                              weights->gate_up, weights->down, ws, dev->grid, cs) != cudaSuccess)
    return MOE_W4A16_ERR_CUDA;
  if (moe::launch_combine(s, r.topk_w, ws.y, norm_gamma, norm_eps, out, cs) != cudaSuccess) return MOE_W4A16_ERR_CUDA;
  return MOE_W4A16_OK;
}
