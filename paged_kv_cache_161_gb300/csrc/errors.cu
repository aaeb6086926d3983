// The per-device error word that kernels set when they skip an out-of-range index or
// give up a wait (bits PA_DEVERR_* of pa.h).
#include <cuda_runtime.h>

#include <mutex>

#include "launch.h"

namespace pa {

static __device__ unsigned int g_error_word;

unsigned int* device_error_word(cudaError_t* err) {
  // One address per device; the lookup runs with that device current.
  static std::mutex mu;
  static unsigned int* cached[64] = {};
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= 64) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!cached[dev]) {
    void* p = nullptr;
    *err = cudaGetSymbolAddress(&p, g_error_word);
    if (*err != cudaSuccess) return nullptr;
    cached[dev] = static_cast<unsigned int*>(p);
  }
  return cached[dev];
}

}  // namespace pa
