// Internal launchers behind the C ABI (include/pa.h). Arguments are validated by the
// caller (api.cpp); these only pick a kernel instantiation and enqueue it.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <mutex>

#include "pa.h"

namespace pa {

// Bytes of an attention workspace after the decode kernels' part: the tensor-core prefill
// kernel's pair counter (16-byte aligned, like the parts before it).
constexpr size_t kPrefillSchedBytes = 16;

// A second stream of the current device, of the highest priority, with a fork and a join
// event, on which the decode kernels of a mixed batch run beside the prefill kernel (which
// stays on the caller's stream); created on first use, kept until exit. `mu` serialises
// the fork, the launches and the join of one call against other host threads (the events
// are shared).
struct SideStream {
  cudaStream_t stream;
  cudaEvent_t fork, join;
  std::mutex* mu;
};
bool side_stream(SideStream* out, cudaError_t* err);

// pa_attention's body; `concurrent` false keeps every kernel on the caller's stream
// (no side stream: for callers that must not create CUDA resources).
int attention_entry(void* out, const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
                    int max_blocks_per_seq, const int32_t* seq_lens, const int32_t* query_start_loc, int num_seqs,
                    int num_tokens, int max_query_len, int max_seq_len, int num_heads, int num_kv_heads,
                    int head_dim, int block_size, int64_t num_blocks, float scale, pa_dtype dtype, void* workspace,
                    size_t workspace_bytes, pa_stream_t stream, bool concurrent);

// Device address of the per-device error word (set up once per device).
unsigned int* device_error_word(cudaError_t* err);

cudaError_t launch_kv_write(const void* k, const void* v, void* k_cache, void* v_cache,
                            const int64_t* slot_mapping, int64_t num_tokens, int64_t num_slots,
                            int64_t row_bytes, unsigned int* err, cudaStream_t stream);

// E4M3 cache write: row_elems = num_kv_heads * head_dim (a multiple of 16).
cudaError_t launch_kv_write_fp8(const void* k, const void* v, pa_dtype in_dtype, void* k_cache, void* v_cache,
                                const int64_t* slot_mapping, int64_t num_tokens, int64_t num_slots,
                                int64_t row_elems, float k_scale, float v_scale, unsigned int* err,
                                cudaStream_t stream);

cudaError_t launch_copy_blocks(void* k_cache, void* v_cache, const int64_t* block_mapping,
                               int64_t num_pairs, int64_t num_blocks, int64_t block_bytes,
                               unsigned int* err, cudaStream_t stream);

cudaError_t launch_swap_blocks(const void* src_k, const void* src_v, void* dst_k, void* dst_v,
                               const int64_t* block_mapping, int64_t num_pairs, int64_t src_blocks,
                               int64_t dst_blocks, int64_t block_bytes, unsigned int* err, cudaStream_t stream);

struct AttnArgs {
  void* out;
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_table;
  const int32_t* seq_lens;
  const int32_t* query_start_loc;
  int max_blocks_per_seq;
  int num_seqs;
  int num_tokens;
  int max_query_len;
  int num_heads;
  int num_kv_heads;
  int head_dim;
  int block_size;
  int64_t num_blocks;
  float scale;
  pa_dtype dtype;  // of q and out (and of the caches unless cache_dtype says otherwise)
  void* workspace;
  unsigned int* err;
  // The tensor-core prefill kernel's pair counter: kPrefillSchedBytes at the end of the
  // caller's workspace (after the decode kernels' part); reset by the launch itself.
  int* prefill_sched = nullptr;
  // false: the decode merge kernel is launched in plain stream order (see launch_merge)
  bool merge_pdl = true;
  // false: never run the prefill kernel on the side stream (callers that must not create
  // CUDA resources)
  bool concurrent = true;
  // q (and k_new / v_new) are page-locked host memory: the decode kernel reads them with
  // plain loads over the CPU-GPU link (never with bulk copies into shared memory)
  bool host_inputs = false;
  // Fused KV write (decode requests only; all three null otherwise): row t of k_new / v_new
  // [num_tokens, num_kv_heads, head_dim] goes to cache slot slot_mapping[t].
  const void* k_new = nullptr;
  const void* v_new = nullptr;
  const int64_t* slot_mapping = nullptr;
  // FP8 E4M3 caches: cache_dtype = PA_FP8_E4M3, values = code * k_scale (v_scale).
  pa_dtype cache_dtype = PA_BF16;
  float k_scale = 1.f;
  float v_scale = 1.f;
  // Shared-prefix groups of a decode batch (tensor-core kernel only; see pa_attention_grouped)
  const int32_t* seq_group = nullptr;
  const int32_t* group_start = nullptr;
  const int32_t* shared_len = nullptr;
  int num_groups = 0;
};

// Decode (q_len == 1 requests): workspace bytes needed, and the launch (split-K + merge).
size_t decode_workspace_bytes(int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                              int num_ctas, pa_dtype dtype);
int decode_num_ctas(int device, cudaError_t* err);
bool decode_supported(pa_dtype dtype, int head_dim, int group);
// KV heads per CTA of the decode kernels for this cache type and shape (0: unsupported).
int decode_hg(pa_dtype cache_dtype, int head_dim, int group, int num_kv_heads);
cudaError_t launch_decode(const AttnArgs& a, int num_ctas, cudaStream_t stream);
// The tensor-core decode kernel (bf16 queries; bf16 caches with head_dim 64 / 128, with or
// without the fused write, or E4M3 caches with head_dim 128; block size 8 or a multiple of
// 16), with the
// CUDA-core kernel's head grouping `hg` so the workspace layout is the same.
bool decode_mma_supported(const AttnArgs& a, int hg);
cudaError_t launch_decode_mma(const AttnArgs& a, int hg, int num_ctas, cudaStream_t stream);
// Workspace of a grouped decode call (the pieces carry 16 rows per KV head).
size_t decode_grouped_workspace_bytes(int num_seqs, int num_groups, int num_kv_heads, int head_dim, int hg,
                                      int num_ctas);

// Prefill (q_len >= 2 requests): the tcgen05 tensor-core kernel where it applies (bf16,
// block size 8..128 dividing 128, <= 4096 requests), else the CUDA-core tile kernel.
bool prefill_supported(pa_dtype dtype, int head_dim, int group);
cudaError_t launch_prefill(const AttnArgs& a, cudaStream_t stream);
bool prefill_tc_supported(const AttnArgs& a);
// How one launch of the tensor-core prefill kernel takes its pairs: a call's first launch
// starts CTA c on pair c (first_static) after zeroing the pair counter (zero_counter); a
// second launch of the same call takes tickets only. ticket_base = the first launch's grid.
struct PrefillLaunch {
  bool first_static;
  int ticket_base;
  bool zero_counter;
};
// The host-side steps of a call's tensor-core prefill launches that can fail (the Q, K and
// V tensor maps, the kernel's shared-memory attribute), done once per call before anything
// of it is enqueued; every launch of the call then uses the plan.
struct PrefillTcPlan {
  CUtensorMap qm, km, vm;
};
cudaError_t prepare_prefill_tc(const AttnArgs& a, PrefillTcPlan* plan);
cudaError_t launch_prefill_tc(const AttnArgs& a, const PrefillTcPlan& plan, int num_ctas, cudaStream_t stream,
                              const PrefillLaunch& how);

}  // namespace pa
