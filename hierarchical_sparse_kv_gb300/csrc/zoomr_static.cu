// zr_decode_attend_static: the decode step with its scratch in a static device
// array, for callers that cannot allocate device memory themselves.
//
// Who needs it: code that is handed only its input and output buffers by a
// host engine that owns every device allocation (a plugin inside an inference
// runtime with its own memory pool, for example) and offers no way to request
// or size a scratch buffer; and loops that must never call cudaMalloc because
// it can synchronize the whole device and stall work already queued. Such a
// caller creates the plan once at start-up and then calls this entry point with
// nothing but its tensors.
//
// The scratch is kStaticScratchBytes (16 MiB) of device memory that every GPU
// which loads this library holds until the process exits. Host code never uses
// the array's name as an address (in host code it is only a stand-in): the
// device address is fetched with cudaGetSymbolAddress once per device, the
// first time the entry point runs on that device, with that device current, and
// kept for the life of the process. A device reset (cudaDeviceReset) reloads the
// module at another address, so the entry point must not be used across one.

#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "zoomr_internal.h"

namespace {

constexpr size_t kStaticScratchBytes = size_t(16) << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_zr_scratch[kStaticScratchBytes];

std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch on the current device (set up on first use).
zr_status scratch_on_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return ZR_ECUDA;
  }
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_zr_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return ZR_ECUDA;
    }
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return ZR_OK;
}

}  // namespace

extern "C" {

zr_status zr_decode_attend_static(zr_plan_t plan, const void* q, const void* k_pool, const void* v_pool,
                                  const int32_t* block_tables, const void* sum_k, const void* sum_v, float* out,
                                  void* stream) {
  // Every check comes before the first enqueued operation: an error return leaves the stream untouched.
  zr_status st = zr::check_decode_args(plan, q, k_pool, v_pool, block_tables, sum_k, sum_v, out);
  if (st != ZR_OK) return st;
  if (plan->p.ws.total > kStaticScratchBytes) return ZR_EUNSUPPORTED;
  // The plan's metadata, kernel attributes and grid size belong to its device: that device must be current
  // (the scratch is looked up on the current device).
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return ZR_ECUDA;
  }
  if (dev != plan->p.device) return ZR_EINVAL;
  void* ws = nullptr;
  st = scratch_on_current_device(&ws);
  if (st != ZR_OK) return st;
  // The array keeps the previous call's contents; only the error word must start at zero.
  if (cudaMemsetAsync(static_cast<char*>(ws) + plan->p.ws.err, 0, sizeof(int32_t),
                      static_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return ZR_ECUDA;
  }
  return zr::decode_into(plan, ws, q, k_pool, v_pool, block_tables, sum_k, sum_v, out, nullptr, nullptr, nullptr,
                         stream, nullptr, nullptr);
}

}  // extern "C"
