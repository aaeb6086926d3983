// pa_kv_write: scatter each new token's K and V rows into the cache slot named by
// slot_mapping ("vLLM" docs page, PagedAttention algorithm flow: store the KV of each
// new token in its physical block; vLLM 0.10.0 flow page, 3.3 KV Manager: slot =
// block * block_size + offset, so the cache is [num_blocks * block_size] rows).
//
// A row is num_kv_heads * head_dim elements (2 KiB for 8 bf16 heads of 128). The kernel
// moves 16-byte vectors: consecutive threads take consecutive vectors of one row, so
// every warp reads 512 contiguous bytes and writes 512 contiguous bytes of one slot.
// HBM-bound; algorithmic bytes = 2 * num_tokens * row_bytes read + the same written.
#include "common.cuh"
#include "launch.h"

namespace pa {

__global__ void __launch_bounds__(256) kv_write_kernel(const uint4* __restrict__ k,
                                                       const uint4* __restrict__ v,
                                                       uint4* __restrict__ k_cache,
                                                       uint4* __restrict__ v_cache,
                                                       const int64_t* __restrict__ slot_mapping,
                                                       int64_t num_tokens, int64_t num_slots,
                                                       int vec_per_row, unsigned int* err) {
  griddep_launch_dependents();  // a following attention launch may be scheduled early
  const int64_t per_token = 2 * static_cast<int64_t>(vec_per_row);
  const int64_t total = num_tokens * per_token;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += stride) {
    const int64_t t = i / per_token;
    const int rem = static_cast<int>(i - t * per_token);
    const int64_t slot = __ldg(slot_mapping + t);
    if (slot < 0) continue;  // padding token
    if (slot >= num_slots) {
      if (rem == 0) raise_error(err, PA_DEVERR_SLOT_RANGE);
      continue;
    }
    const bool is_v = rem >= vec_per_row;
    const int e = is_v ? rem - vec_per_row : rem;
    const uint4 val = __ldg((is_v ? v : k) + t * vec_per_row + e);
    (is_v ? v_cache : k_cache)[slot * vec_per_row + e] = val;
  }
}

cudaError_t launch_kv_write(const void* k, const void* v, void* k_cache, void* v_cache,
                            const int64_t* slot_mapping, int64_t num_tokens, int64_t num_slots,
                            int64_t row_bytes, unsigned int* err, cudaStream_t stream) {
  if (num_tokens == 0) return cudaSuccess;
  const int vec_per_row = static_cast<int>(row_bytes / 16);
  const int64_t total = num_tokens * 2 * vec_per_row;
  const int threads = 256;
  int64_t blocks = (total + threads - 1) / threads;
  if (blocks > 152 * 16) blocks = 152 * 16;  // grid-stride beyond 16 CTAs per SM
  kv_write_kernel<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(
      static_cast<const uint4*>(k), static_cast<const uint4*>(v), static_cast<uint4*>(k_cache),
      static_cast<uint4*>(v_cache), slot_mapping, num_tokens, num_slots, vec_per_row, err);
  return cudaGetLastError();
}

// FP8 E4M3 cache ("vLLM" docs page, quantisation support: FP8, 8-bit, 2x smaller than
// 16-bit): each element of a new token's K (V) row is stored as E4M3(x / k_scale): x
// widened to binary32, one correctly rounded binary32 division, then round to nearest
// even with saturation at +-448. A thread handles 16 consecutive elements of one row
// (16 bytes of cache). HBM-bound: algorithmic bytes per token = 2 * row elements * (input
// bytes + 1).
template <typename TIn>
__global__ void __launch_bounds__(256) kv_write_fp8_kernel(const TIn* __restrict__ k, const TIn* __restrict__ v,
                                                           uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                                                           const int64_t* __restrict__ slot_mapping,
                                                           int64_t num_tokens, int64_t num_slots, int chunks_per_row,
                                                           float k_scale, float v_scale, unsigned int* err) {
  griddep_launch_dependents();
  const int64_t per_token = 2 * static_cast<int64_t>(chunks_per_row);
  const int64_t total = num_tokens * per_token;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  constexpr int kInVec = 16 / sizeof(TIn);  // inputs per 16-byte load
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += stride) {
    const int64_t t = i / per_token;
    const int rem = static_cast<int>(i - t * per_token);
    const int64_t slot = __ldg(slot_mapping + t);
    if (slot < 0) continue;
    if (slot >= num_slots) {
      if (rem == 0) raise_error(err, PA_DEVERR_SLOT_RANGE);
      continue;
    }
    const bool is_v = rem >= chunks_per_row;
    const int c = is_v ? rem - chunks_per_row : rem;
    const float sc = is_v ? v_scale : k_scale;
    const uint4* src = reinterpret_cast<const uint4*>((is_v ? v : k) + (t * chunks_per_row + c) * 16);
    float f[16];
#pragma unroll
    for (int j = 0; j < 16 / kInVec; ++j) Elem<TIn>::unpack(__ldg(src + j), f + j * kInVec);
    uint32_t w[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t lo = float2_to_fp8x2(__fdiv_rn(f[4 * j], sc), __fdiv_rn(f[4 * j + 1], sc));
      const uint32_t hi = float2_to_fp8x2(__fdiv_rn(f[4 * j + 2], sc), __fdiv_rn(f[4 * j + 3], sc));
      w[j] = lo | (hi << 16);
    }
    (is_v ? v_cache : k_cache)[slot * chunks_per_row + c] = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

cudaError_t launch_kv_write_fp8(const void* k, const void* v, pa_dtype in_dtype, void* k_cache, void* v_cache,
                                const int64_t* slot_mapping, int64_t num_tokens, int64_t num_slots,
                                int64_t row_elems, float k_scale, float v_scale, unsigned int* err,
                                cudaStream_t stream) {
  if (num_tokens == 0) return cudaSuccess;
  const int chunks_per_row = static_cast<int>(row_elems / 16);
  const int64_t total = num_tokens * 2 * chunks_per_row;
  const int threads = 256;
  int64_t blocks = (total + threads - 1) / threads;
  if (blocks > 152 * 16) blocks = 152 * 16;
  if (in_dtype == PA_BF16) {
    kv_write_fp8_kernel<__nv_bfloat16><<<static_cast<unsigned>(blocks), threads, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(k), static_cast<const __nv_bfloat16*>(v), static_cast<uint4*>(k_cache),
        static_cast<uint4*>(v_cache), slot_mapping, num_tokens, num_slots, chunks_per_row, k_scale, v_scale, err);
  } else {
    kv_write_fp8_kernel<float><<<static_cast<unsigned>(blocks), threads, 0, stream>>>(
        static_cast<const float*>(k), static_cast<const float*>(v), static_cast<uint4*>(k_cache),
        static_cast<uint4*>(v_cache), slot_mapping, num_tokens, num_slots, chunks_per_row, k_scale, v_scale, err);
  }
  return cudaGetLastError();
}

}  // namespace pa
