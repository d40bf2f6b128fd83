// forward_noalloc.cu -- moe_w4a16_forward_noalloc: the forward pass (gate_up,
// down, combine) with its scratch memory in a fixed static device array, for
// callers that cannot allocate device memory themselves.
//
// The scratch (work counters and error word, the fp16 activations h, the token
// rows in expert order and the fp32 per-pair outputs) lives in g_scratch below.
// Every GPU that loads this library holds the array until the process exits.
// All calls on a device share it, so calls whose work overlaps on the GPU race;
// the header part (counters, error word) is cleared at the start of every call,
// the rest is fully written before it is read.  Apart from where the scratch
// lives, a call runs exactly the checks and launches of moe_w4a16_forward (same
// shape rules, same kernel instantiation for the shape's reduction order and
// weight format), so its output is bit-identical to that call's.
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
  void* scratch = nullptr;  // device address of g_scratch on this device
};
constexpr int kMaxDevices = 64;
NoallocDevice g_devices[kMaxDevices];
std::mutex g_mutex;

// One-time set-up per device, done by the first call on that device with the
// device current: resolve the device address of g_scratch (in host code the
// symbol's name is only a host-side stand-in, never a device address).
moe_w4a16_status device_setup(void** scratch) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_W4A16_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mutex);
  NoallocDevice& st = g_devices[dev];
  if (!st.ready) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return MOE_W4A16_ERR_CUDA;
    if (major != 10 || minor != 3) {
      st.status = MOE_W4A16_ERR_DEVICE;
    } else {
      void* ptr = nullptr;
      if (cudaGetSymbolAddress(&ptr, g_scratch) != cudaSuccess || ptr == nullptr)
        return MOE_W4A16_ERR_CUDA;  // not marked ready: the next call retries
      st.scratch = ptr;
      st.status = MOE_W4A16_OK;
    }
    st.ready = true;
  }
  *scratch = st.scratch;
  return st.status;
}

}  // namespace

extern "C" moe_w4a16_status moe_w4a16_forward_noalloc(const moe_w4a16_shape* shape, const uint16_t* x,
                                                      const moe_w4a16_routing* routing,
                                                      const moe_w4a16_weights* weights, const float* norm_gamma,
                                                      float norm_eps, uint16_t* out, void* stream) {
  moe::Dims s;
  moe_w4a16_status st = moe::check_shape(shape, &s);
  if (st != MOE_W4A16_OK) return st;
  if (moe::ws_total(s) > kScratchBytes) return MOE_W4A16_ERR_WORKSPACE;
  void* scratch = nullptr;
  if ((st = device_setup(&scratch)) != MOE_W4A16_OK) return st;
  return moe::forward_all_steps(shape, x, routing, weights, norm_gamma, norm_eps, out, scratch, kScratchBytes, stream,
                                true);
}

// The sticky error word at the start of this device's static array: the status of
// device-side failures of the last moe_w4a16_forward_noalloc call on the device
// (each call clears it when it starts).  Synchronises the stream.
extern "C" moe_w4a16_status moe_w4a16_noalloc_read_error(void* stream, moe_w4a16_status* device_status) {
  if (!device_status) return MOE_W4A16_ERR_NULL;
  void* scratch = nullptr;
  moe_w4a16_status st = device_setup(&scratch);
  if (st != MOE_W4A16_OK) return st;
  int32_t code = 0;
  const auto cs = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(&code, scratch, sizeof(code), cudaMemcpyDeviceToHost, cs) != cudaSuccess ||
      cudaStreamSynchronize(cs) != cudaSuccess)
    return MOE_W4A16_ERR_CUDA;
  *device_status = static_cast<moe_w4a16_status>(code);
  return MOE_W4A16_OK;
}
