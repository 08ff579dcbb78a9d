// cbr_forward_train_noalloc: the training forward for callers that cannot allocate device
// memory.  Its scratch lives in a fixed array compiled into the library instead of a
// caller-supplied workspace; see the declaration in include/cbr.h.
#include <mutex>

#include "../../include/cbr.h"
#include "cbr_internal.h"

namespace cbr {
namespace {

// Upper bound on the scratch this entry point can use.  With the conv output kept by the
// caller (z_saved), the forward needs 256 bytes of arrival counters, 2*Cout floats of apply
// coefficients and 2*Cout + 4 floats of partial statistics per CTA (at most kMaxCtas CTAs):
// about 261 KiB for Cout = 128.  Every GPU that loads the library holds this array until exit.
constexpr size_t kNoAllocScratchBytes = 320 * 1024;
static_assert(kNoAllocScratchBytes >= forward_scratch_bytes(128),
              "the fixed scratch must hold the largest supported forward (Cout = 128, kMaxCtas CTAs)");
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices];  // device address of the array, per device

// One-time set-up per device, done with that device current: in host code the array's name
// is only a stand-in, so its device address is looked up and cached.
int scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return CBR_ERR_DEVICE;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return CBR_ERR_CUDA;
    }
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return CBR_OK;
}

}  // namespace
}  // namespace cbr

extern "C" cbr_status_t cbr_forward_train_noalloc(
    const cbr_desc_t* desc, const void* x, const void* w, const float* gamma, const float* beta,
    float* running_mean, float* running_var, float momentum, float eps, void* y,
    uint32_t* relu_mask, void* z_saved, float* saved_mean, float* saved_inv_var,
    cbr_stream_t stream) {
  // Every argument and the device are checked before the scratch is touched, so a rejected call
  // enqueues nothing (in particular not the counter reset below, which could otherwise clear the
  // counters of an earlier call still running on the shared array).
  size_t need = 0;
  int st = cbr::check_forward_train(desc, x, w, gamma, beta, running_mean, running_var, momentum, eps,
                                    y, relu_mask, z_saved, saved_mean, saved_inv_var, &need);
  if (st) return (cbr_status_t)st;
  if (!z_saved) return CBR_ERR_INVALID_ARG;  // the conv output cannot live in the fixed scratch
  if (need > cbr::kNoAllocScratchBytes) return CBR_ERR_WORKSPACE;
  if ((st = cbr::check_device())) return (cbr_status_t)st;
  void* scratch = nullptr;
  if ((st = cbr::scratch_address(&scratch))) return (cbr_status_t)st;
  // The arrival counters must start at zero; the array keeps whatever the last call left.
  if (cudaMemsetAsync(scratch, 0, cbr::kWsHeaderBytes, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return CBR_ERR_CUDA;
  }
  return cbr_forward_train(desc, x, w, gamma, beta, running_mean, running_var, momentum, eps, y,
                           relu_mask, z_saved, saved_mean, saved_inv_var, scratch,
                           cbr::kNoAllocScratchBytes, stream);
}
