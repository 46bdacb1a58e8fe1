// Fixed device-resident counter block for mk_decode_step_static.
//
// The decode step's counters, queue claim heads and error words normally live
// in memory the handle allocates at creation.  mk_decode_step_static runs the
// same persistent kernel with them placed in this file-scope array instead,
// so the call itself needs no allocation.  The array is looked up once per
// device (cudaGetSymbolAddress) and the address cached.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/mk.h"

namespace mk {

// MK_STATIC_COUNTER_WORDS x 4 bytes = 256 KB per device
static __device__ __align__(256) uint32_t g_static_counters[MK_STATIC_COUNTER_WORDS];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_lock;
uint32_t* g_addr[kMaxDevices] = {};
}  // namespace

// Device address of the counter block on `device` (the current device).
// MK_OK, MK_ERR_BAD_ARG (device index out of range) or MK_ERR_CUDA.
int static_counters(int device, uint32_t** out) {
  if (device < 0 || device >= kMaxDevices || !out) return MK_ERR_BAD_ARG;
  std::lock_guard<std::mutex> guard(g_lock);
  if (!g_addr[device]) {
    uint32_t* ptr = nullptr;
    if (cudaGetSymbolAddress((void**)&ptr, g_static_counters) != cudaSuccess || !ptr) {
      cudaGetLastError();
      return MK_ERR_CUDA;
    }
    g_addr[device] = ptr;
  }
  *out = g_addr[device];
  return MK_OK;
}

}  // namespace mk
