// Forward entry point that allocates nothing: its workspace is a fixed array in device memory
// that belongs to the library (see lce_forward_static_scratch in include/lce.h).
//
// Who needs it: code that is handed a stream but may not allocate device memory itself -- a
// plugin inside an inference or training engine that owns every byte of device memory through
// its own pool and only lends its plugins the buffers it planned; a service that fixes its device
// memory budget at start-up and must not grow it per request; latency-critical paths that cannot
// take the cost of cudaMalloc or the device-wide synchronisation of a cudaFree.  Such a caller
// still passes its inputs and outputs; only the scratch comes from here.
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "lce.h"
#include "lce_internal.h"

namespace {

// The scratch array.  Every GPU that loads this library holds these bytes until the process exits.
__device__ __align__(256) unsigned char g_static_scratch[LCE_STATIC_SCRATCH_BYTES];

std::atomic<void*> g_scratch_addr[lce::kMaxDevices];

// Device address of the array on the current device.  In host code the array's name is only a
// host-side handle, so the address is asked from the runtime, once per device, with that device
// current.  The device is checked first: a device of another architecture has no image of this
// library, so it is refused as unsupported rather than failing the lookup.
lce_status_t scratch_address(void** out) {
  int num_sms = 0;
  lce_status_t st = lce::check_device(&num_sms);  // also makes the device's context current
  if (st != LCE_OK) return st;
  int dev = 0;
  if (lce::note(cudaGetDevice(&dev)) != cudaSuccess) return LCE_ERR_CUDA;
  void* p = g_scratch_addr[dev].load(std::memory_order_acquire);
  if (p == nullptr) {
    if (lce::note(cudaGetSymbolAddress(&p, g_static_scratch)) != cudaSuccess) return LCE_ERR_CUDA;
    if (p == nullptr) {
      lce::set_error_detail("no device address for the static scratch array");
      return LCE_ERR_CUDA;
    }
    g_scratch_addr[dev].store(p, std::memory_order_release);
  }
  *out = p;
  return LCE_OK;
}

}  // namespace

extern "C" lce_status_t lce_forward_static_scratch(
    const void* H, const void* W, const int64_t* labels, int64_t N, int64_t d, int64_t V,
    int64_t ignore_index, int64_t strip_V, lce_reduction_t reduction, lce_dtype_t dtype,
    float* loss, float* lse, int64_t* n_valid, uint32_t* device_error_flags, void* stream) {
  const size_t need = lce_workspace_size(N, d, V, strip_V, dtype);
  if (need == 0) return LCE_ERR_UNSUPPORTED_SHAPE;
  if (need > LCE_STATIC_SCRATCH_BYTES) return LCE_ERR_WORKSPACE_TOO_SMALL;
  void* scratch = nullptr;
  lce_status_t st = scratch_address(&scratch);
  if (st != LCE_OK) return st;
  // lce_forward clears the error flags at the head of the scratch and initialises every other
  // part it reads, so nothing left by an earlier call leaks into this one.
  st = lce_forward(H, W, labels, N, d, V, ignore_index, strip_V, reduction, dtype, loss, lse,
                   n_valid, scratch, LCE_STATIC_SCRATCH_BYTES, stream);
  if (st != LCE_OK) return st;
  if (device_error_flags != nullptr &&
      lce::note(cudaMemcpyAsync(device_error_flags, scratch, sizeof(uint32_t),
                                cudaMemcpyDeviceToDevice, static_cast<cudaStream_t>(stream))) !=
          cudaSuccess)
    return LCE_ERR_CUDA;
  return LCE_OK;
}
