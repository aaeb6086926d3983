// The per-device error word that kernels set when they skip an out-of-range index or
// give up a wait (bits PA_DEVERR_* of pa.h), and the per-device side stream on which the
// decode kernels of a mixed batch run beside the prefill kernel.
#include <cuda_runtime.h>

#include <mutex>

#include "launch.h"

namespace pa {

static __device__ unsigned int g_error_word;

bool side_stream(SideStream* out, cudaError_t* err) {
  static std::mutex mu;
  static std::mutex call_mu[64];
  static SideStream cached[64] = {};
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return false;
  if (dev < 0 || dev >= 64) {
    *err = cudaErrorInvalidDevice;
    return false;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!cached[dev].stream) {
    int least = 0, greatest = 0;  // greatest priority = numerically lowest value
    *err = cudaDeviceGetStreamPriorityRange(&least, &greatest);
    if (*err != cudaSuccess) return false;
    SideStream s = {nullptr, nullptr, nullptr, &call_mu[dev]};
    *err = cudaStreamCreateWithPriority(&s.stream, cudaStreamNonBlocking, greatest);
    if (*err == cudaSuccess) *err = cudaEventCreateWithFlags(&s.fork, cudaEventDisableTiming);
    if (*err == cudaSuccess) *err = cudaEventCreateWithFlags(&s.join, cudaEventDisableTiming);
    if (*err != cudaSuccess) {  // release what was created; a later call tries again
      if (s.fork) cudaEventDestroy(s.fork);
      if (s.stream) cudaStreamDestroy(s.stream);
      return false;
    }
    cached[dev] = s;
  }
  *out = cached[dev];
  return true;
}

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
