// pa_attention_fixed_scratch: pa_attention for callers that cannot allocate device memory.
//
// Some callers have no way to obtain a workspace: a serving loop that reserved all of the
// GPU's memory for its KV pool at start-up and must not call cudaMalloc afterwards (the call
// synchronises the device and can fail once the pool owns the memory), a plugin running
// inside a host framework whose allocator it cannot reach, or a foreign-language binding
// with no device allocator at all. This entry point takes the same inputs and outputs as
// pa_attention but uses, as its split-K scratch, a fixed array that lives in the library
// itself and is held by every GPU that loads the library until the process exits.
//
// The scratch holds the decode kernel's per-CTA partial results and their merge indices.
// No part of it needs to start at zero: in every call the split-K kernel writes each
// partial and index before the merge kernel of the same call reads it.
#include <cuda_runtime.h>

#include <mutex>

#include "launch.h"
#include "pa.h"

namespace {

constexpr size_t kFixedScratchBytes = size_t(16) << 20;  // 16 MiB per device

static __device__ __align__(256) unsigned char g_fixed_scratch[kFixedScratchBytes];

// Device address of g_fixed_scratch on the current device, looked up once per device.
// (In host code the array's name is only a host-side stand-in for the device symbol.)
void* fixed_scratch_address(cudaError_t* err) {
  static std::mutex mu;
  static void* addr[64] = {};
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= 64) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    *err = cudaGetSymbolAddress(&p, g_fixed_scratch);
    if (*err != cudaSuccess) return nullptr;
    addr[dev] = p;
  }
  return addr[dev];
}

}  // namespace

extern "C" int pa_attention_fixed_scratch(void* out, const void* q, const void* k_cache,
                                          const void* v_cache, const int32_t* block_table,
                                          int max_blocks_per_seq, const int32_t* seq_lens,
                                          const int32_t* query_start_loc, int num_seqs,
                                          int num_tokens, int max_query_len, int max_seq_len,
                                          int num_heads, int num_kv_heads, int head_dim,
                                          int block_size, int64_t num_blocks, float scale,
                                          pa_dtype dtype, pa_stream_t stream) {
  size_t need = 0;
  const int st = pa_attention_workspace_size(num_seqs, num_heads, num_kv_heads, head_dim, &need);
  if (st != PA_OK) return st;
  if (need > kFixedScratchBytes) return PA_ERR_WORKSPACE;  // batch too large for the fixed scratch
  cudaError_t e;
  void* scratch = fixed_scratch_address(&e);
  if (!scratch) return PA_ERR_CUDA;
  return pa::attention_entry(out, q, k_cache, v_cache, block_table, max_blocks_per_seq, seq_lens,
                             query_start_loc, num_seqs, num_tokens, max_query_len, max_seq_len, num_heads,
                             num_kv_heads, head_dim, block_size, num_blocks, scale, dtype, scratch,
                             kFixedScratchBytes, stream, false);
}
