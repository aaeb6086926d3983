// Device helpers shared by the sm_103a kernels: element traits, mbarrier and bulk-copy
// (TMA engine) wrappers with bounded waits, warp reductions.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>
#include <utility>

#include "pa.h"

namespace pa {

// ---------------------------------------------------------------- element types
template <typename T>
struct Elem;

template <>
struct Elem<float> {
  static constexpr int kBytes = 4;
  // Four consecutive floats of a 16-byte vector.
  static __device__ __forceinline__ void unpack(const uint4& u, float* f) {
    f[0] = __uint_as_float(u.x);
    f[1] = __uint_as_float(u.y);
    f[2] = __uint_as_float(u.z);
    f[3] = __uint_as_float(u.w);
  }
  static __device__ __forceinline__ uint4 pack(const float* f) {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                      __float_as_uint(f[3]));
  }
};

template <>
struct Elem<__nv_bfloat16> {
  static constexpr int kBytes = 2;
  // Eight bf16 of a 16-byte vector -> fp32 (exact: a bf16 is the top half of a binary32).
  static __device__ __forceinline__ void unpack(const uint4& u, float* f) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
  // fp32 -> bf16, round to nearest even (the CUDA intrinsic).
  static __device__ __forceinline__ uint4 pack(const float* f) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
      w[i] = *reinterpret_cast<uint32_t*>(&h);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
};

// FP8 E4M3 cache element (1 sign, 4 exponent bits with bias 7, 3 mantissa bits; no
// infinities, largest finite 448). Stored values stand for E4M3 value * scale.
struct Fp8E4M3 {
  uint8_t bits;
};

// Two E4M3 codes (low byte first) -> two floats, exactly (through the f16x2 hardware
// conversion, which is exact: every E4M3 value is an f16 value).
__device__ __forceinline__ float2 fp8x2_to_float2(uint32_t two_codes) {
  uint32_t h2;
  asm("{\n\t.reg .b16 c;\n\tcvt.u16.u32 c, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, c;\n\t}" : "=r"(h2) : "r"(two_codes));
  const __half2 h = *reinterpret_cast<const __half2*>(&h2);
  return __half22float2(h);
}

// Two floats -> two E4M3 codes (lo -> low byte): round to nearest even, magnitudes beyond
// 448 saturate to 448.
__device__ __forceinline__ uint32_t float2_to_fp8x2(float lo, float hi) {
  uint16_t c;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(c) : "f"(hi), "f"(lo));
  return c;
}

template <>
struct Elem<Fp8E4M3> {
  static constexpr int kBytes = 1;
  // Sixteen E4M3 codes of a 16-byte vector -> fp32 (exact).
  static __device__ __forceinline__ void unpack(const uint4& u, float* f) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 a = fp8x2_to_float2(w[i] & 0xffffu), b = fp8x2_to_float2(w[i] >> 16);
      f[4 * i] = a.x;
      f[4 * i + 1] = a.y;
      f[4 * i + 2] = b.x;
      f[4 * i + 3] = b.y;
    }
  }
};

// ---------------------------------------------------------------- error word
__device__ __forceinline__ void raise_error(unsigned int* err, unsigned int bit) {
  if (err) atomicOr(err, bit);
}

// ---------------------------------------------------------------- shared-memory addresses
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// A wait that gives up after `kWaitTimeoutNs` of wall time. Every pipeline wait in this
// library goes through here so that no kernel can spin forever.
constexpr uint64_t kWaitTimeoutNs = 200ull * 1000ull * 1000ull;  // 200 ms

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > kWaitTimeoutNs) return false;
  }
}

// ---------------------------------------------------------------- bulk copies (TMA engine)
// global -> shared, completion counted in bytes on `bar`. dst, src, bytes: multiples of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// ---------------------------------------------------------------- packed fp32 FMA
// d.x += a.x * b.x; d.y += a.y * b.y in one instruction (sm_100 family).
__device__ __forceinline__ void ffma2(float2& d, const float2 a, const float2 b) {
  unsigned long long dd = (static_cast<unsigned long long>(__float_as_uint(d.y)) << 32) |
                          __float_as_uint(d.x);
  const unsigned long long aa = (static_cast<unsigned long long>(__float_as_uint(a.y)) << 32) |
                                __float_as_uint(a.x);
  const unsigned long long bb = (static_cast<unsigned long long>(__float_as_uint(b.y)) << 32) |
                                __float_as_uint(b.x);
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(dd) : "l"(aa), "l"(bb));
  d.x = __uint_as_float(static_cast<uint32_t>(dd));
  d.y = __uint_as_float(static_cast<uint32_t>(dd >> 32));
}

// Packed fp32 add (sm_100 family): (a.x + b.x, a.y + b.y).
__device__ __forceinline__ float2 fadd2(const float2 a, const float2 b) {
  unsigned long long d;
  const unsigned long long aa = (static_cast<unsigned long long>(__float_as_uint(a.y)) << 32) | __float_as_uint(a.x);
  const unsigned long long bb = (static_cast<unsigned long long>(__float_as_uint(b.y)) << 32) | __float_as_uint(b.x);
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(aa), "l"(bb));
  return make_float2(__uint_as_float(static_cast<uint32_t>(d)), __uint_as_float(static_cast<uint32_t>(d >> 32)));
}

// Packed fp32 fused multiply-add: (a.x * b.x + c.x, a.y * b.y + c.y).
__device__ __forceinline__ float2 ffma2v(const float2 a, const float2 b, const float2 c) {
  unsigned long long d;
  const unsigned long long aa = (static_cast<unsigned long long>(__float_as_uint(a.y)) << 32) | __float_as_uint(a.x);
  const unsigned long long bb = (static_cast<unsigned long long>(__float_as_uint(b.y)) << 32) | __float_as_uint(b.x);
  const unsigned long long cc = (static_cast<unsigned long long>(__float_as_uint(c.y)) << 32) | __float_as_uint(c.x);
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(aa), "l"(bb), "l"(cc));
  return make_float2(__uint_as_float(static_cast<uint32_t>(d)), __uint_as_float(static_cast<uint32_t>(d >> 32)));
}

// Three-input maximum (sm_100 family).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// 2^x with the hardware approximation (subnormal results flushed to zero).
__device__ __forceinline__ float ex2_ftz(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---------------------------------------------------------------- programmatic dependent launch
// Wait until the preceding grid in the stream has completed and its writes are visible
// (returns at once when the kernel was launched without the PDL attribute).
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Allow the next grid in the stream (launched with the PDL attribute) to be scheduled.
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Raises kernel Kern's dynamic shared-memory limit to at least `bytes` on the current
// device, once per device (later calls only read a table). Host threads launching the same
// kernel concurrently therefore never set its attribute while another thread launches it.
template <auto Kern>
static cudaError_t ensure_smem(size_t bytes) {
  static std::mutex mu;
  static size_t done[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (done[dev] >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(Kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(bytes));
  if (e == cudaSuccess) done[dev] = bytes;
  return e;
}

// Launch with programmatic stream serialisation allowed: the kernel may start while the
// previous kernel in the stream finishes; it must call griddep_wait() before touching
// anything that kernel may write.
template <typename... KArgs, typename... Args>
static cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace pa
