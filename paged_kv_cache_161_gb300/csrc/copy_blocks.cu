// pa_copy_blocks: the copy step of copy-on-write ("vLLM" docs page, Copy-on-Write:
// allocate a new block and copy the old block's content into it before the divergent
// write; code-reading page 5.2.1: A1's logical block 1 moves from physical 1 to 3).
//
// One CTA per (pair, K or V) copies one whole physical block (block_size * num_kv_heads
// * head_dim elements, 32 KiB for 16 x 8 x 128 bf16) with 16-byte vectors, four
// independent loads in flight per thread. HBM-bound; algorithmic bytes per pair =
// 2 * block_bytes read + 2 * block_bytes written.
#include "common.cuh"
#include "launch.h"

namespace pa {

__global__ void __launch_bounds__(256) copy_blocks_kernel(uint4* __restrict__ k_cache,
                                                          uint4* __restrict__ v_cache,
                                                          const int64_t* __restrict__ mapping,
                                                          int64_t num_blocks, int vec_per_block,
                                                          unsigned int* err) {
  const int64_t pair = blockIdx.x;
  const int64_t src = __ldg(mapping + 2 * pair);
  const int64_t dst = __ldg(mapping + 2 * pair + 1);
  if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
    if (threadIdx.x == 0 && blockIdx.y == 0) raise_error(err, PA_DEVERR_BLOCK_RANGE);
    return;
  }
  uint4* cache = blockIdx.y ? v_cache : k_cache;
  const uint4* s = cache + src * vec_per_block;
  uint4* d = cache + dst * vec_per_block;
  constexpr int kUnroll = 4;
  int i = threadIdx.x;
  for (; i + (kUnroll - 1) * 256 < vec_per_block; i += kUnroll * 256) {
    uint4 r[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) r[u] = __ldg(s + i + u * 256);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) d[i + u * 256] = r[u];
  }
  for (; i < vec_per_block; i += 256) d[i] = __ldg(s + i);
}

cudaError_t launch_copy_blocks(void* k_cache, void* v_cache, const int64_t* block_mapping,
                               int64_t num_pairs, int64_t num_blocks, int64_t block_bytes,
                               unsigned int* err, cudaStream_t stream) {
  if (num_pairs == 0) return cudaSuccess;
  dim3 grid(static_cast<unsigned>(num_pairs), 2);
  copy_blocks_kernel<<<grid, 256, 0, stream>>>(static_cast<uint4*>(k_cache),
                                                static_cast<uint4*>(v_cache), block_mapping,
                                                num_blocks, static_cast<int>(block_bytes / 16),
                                                err);
  return cudaGetLastError();
}

// pa_swap_blocks: whole blocks from one pool to another (code-reading page 6.2.1: a
// preempted group's KV blocks are swapped out to CPU memory and back in later). Either pool
// may be pinned host memory, which the kernel reads or writes directly through unified
// addressing over the CPU-GPU link, so a whole swap is one launch however many blocks it
// moves. One CTA per (pair, K or V), 16-byte vectors, four loads in flight per thread.
__global__ void __launch_bounds__(256) swap_blocks_kernel(const uint4* __restrict__ src_k,
                                                          const uint4* __restrict__ src_v,
                                                          uint4* __restrict__ dst_k, uint4* __restrict__ dst_v,
                                                          const int64_t* __restrict__ mapping, int64_t src_blocks,
                                                          int64_t dst_blocks, int vec_per_block, unsigned int* err) {
  const int64_t pair = blockIdx.x;
  const int64_t src = mapping[2 * pair];
  const int64_t dst = mapping[2 * pair + 1];
  if (src < 0 || src >= src_blocks || dst < 0 || dst >= dst_blocks) {
    if (threadIdx.x == 0 && blockIdx.y == 0) raise_error(err, PA_DEVERR_BLOCK_RANGE);
    return;
  }
  const uint4* s = (blockIdx.y ? src_v : src_k) + src * vec_per_block;
  uint4* d = (blockIdx.y ? dst_v : dst_k) + dst * vec_per_block;
  constexpr int kUnroll = 4;
  int i = threadIdx.x;
  for (; i + (kUnroll - 1) * 256 < vec_per_block; i += kUnroll * 256) {
    uint4 r[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) r[u] = s[i + u * 256];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) d[i + u * 256] = r[u];
  }
  for (; i < vec_per_block; i += 256) d[i] = s[i];
}

cudaError_t launch_swap_blocks(const void* src_k, const void* src_v, void* dst_k, void* dst_v,
                               const int64_t* block_mapping, int64_t num_pairs, int64_t src_blocks,
                               int64_t dst_blocks, int64_t block_bytes, unsigned int* err, cudaStream_t stream) {
  if (num_pairs == 0) return cudaSuccess;
  dim3 grid(static_cast<unsigned>(num_pairs), 2);
  swap_blocks_kernel<<<grid, 256, 0, stream>>>(static_cast<const uint4*>(src_k), static_cast<const uint4*>(src_v),
                                               static_cast<uint4*>(dst_k), static_cast<uint4*>(dst_v), block_mapping,
                                               src_blocks, dst_blocks, static_cast<int>(block_bytes / 16), err);
  return cudaGetLastError();
}

}  // namespace pa
