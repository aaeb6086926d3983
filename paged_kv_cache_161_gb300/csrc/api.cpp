// C ABI of include/pa.h: argument validation, then dispatch to the kernel launchers.
// Nothing here allocates device memory or synchronises (except pa_read_device_errors).
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "launch.h"
#include "pa.h"

namespace {

thread_local int g_last_cuda_error = 0;

int cuda_fail(cudaError_t e) {
  g_last_cuda_error = static_cast<int>(e);
  return PA_ERR_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int elem_bytes(pa_dtype dt) {
  switch (dt) {
    case PA_F32: return 4;
    case PA_BF16: return 2;
    case PA_FP8_E4M3: return 1;
  }
  return 0;
}

bool pow2_le8(int g) { return g == 1 || g == 2 || g == 4 || g == 8; }

// Cache geometry shared by the three device entry points.
int check_cache(const void* k_cache, const void* v_cache, int64_t num_blocks, int block_size,
                int num_kv_heads, int head_dim, pa_dtype dtype) {
  if (!k_cache || !v_cache) return PA_ERR_INVALID_ARG;
  if (!aligned16(k_cache) || !aligned16(v_cache)) return PA_ERR_INVALID_ARG;
  if (num_blocks < 1 || block_size < 1 || num_kv_heads < 1 || head_dim < 1) return PA_ERR_INVALID_ARG;
  if (elem_bytes(dtype) == 0) return PA_ERR_INVALID_ARG;
  if ((int64_t(num_kv_heads) * head_dim * elem_bytes(dtype)) % 16 != 0) return PA_ERR_UNSUPPORTED;
  return PA_OK;
}

}  // namespace

extern "C" {

const char* pa_status_string(int status) {
  switch (status) {
    case PA_OK: return "ok";
    case PA_ERR_INVALID_ARG: return "invalid argument";
    case PA_ERR_UNSUPPORTED: return "unsupported shape or type";
    case PA_ERR_WORKSPACE: return "workspace missing or too small";
    case PA_ERR_CUDA: return "CUDA error";
    case PA_ERR_NO_BLOCKS: return "not enough free blocks";
    case PA_ERR_TOO_LARGE: return "sequence larger than the block pool";
    case PA_ERR_NOT_FOUND: return "unknown or duplicate sequence id";
  }
  return "unknown status";
}

int pa_last_cuda_error(void) { return g_last_cuda_error; }

int pa_read_device_errors(unsigned int* flags_out, int clear) {
  if (!flags_out) return PA_ERR_INVALID_ARG;
  cudaError_t e;
  unsigned int* w = pa::device_error_word(&e);
  if (!w) return cuda_fail(e);
  e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e);
  e = cudaMemcpy(flags_out, w, sizeof(unsigned int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e);
  if (clear) {
    e = cudaMemset(w, 0, sizeof(unsigned int));
    if (e != cudaSuccess) return cuda_fail(e);
    e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e);
  }
  return PA_OK;
}

int pa_kv_write(const void* k, const void* v, void* k_cache, void* v_cache,
                const int64_t* slot_mapping, int64_t num_tokens, int64_t num_blocks,
                int block_size, int num_kv_heads, int head_dim, pa_dtype dtype,
                pa_stream_t stream) {
  int st = check_cache(k_cache, v_cache, num_blocks, block_size, num_kv_heads, head_dim, dtype);
  if (st != PA_OK) return st;
  if (num_tokens < 0) return PA_ERR_INVALID_ARG;
  if (num_tokens == 0) return PA_OK;
  if (!k || !v || !slot_mapping || !aligned16(k) || !aligned16(v)) return PA_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(slot_mapping) % 8 != 0) return PA_ERR_INVALID_ARG;
  cudaError_t e;
  unsigned int* err = pa::device_error_word(&e);
  if (!err) return cuda_fail(e);
  const int64_t row_bytes = int64_t(num_kv_heads) * head_dim * elem_bytes(dtype);
  e = pa::launch_kv_write(k, v, k_cache, v_cache, slot_mapping, num_tokens, num_blocks * block_size,
                          row_bytes, err, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

int pa_copy_blocks(void* k_cache, void* v_cache, const int64_t* block_mapping, int64_t num_pairs,
                   int64_t num_blocks, int block_size, int num_kv_heads, int head_dim,
                   pa_dtype dtype, pa_stream_t stream) {
  int st = check_cache(k_cache, v_cache, num_blocks, block_size, num_kv_heads, head_dim, dtype);
  if (st != PA_OK) return st;
  if (num_pairs < 0 || num_pairs > 0x7fffffff) return PA_ERR_INVALID_ARG;
  if (num_pairs == 0) return PA_OK;
  if (!block_mapping || reinterpret_cast<uintptr_t>(block_mapping) % 8 != 0) return PA_ERR_INVALID_ARG;
  cudaError_t e;
  unsigned int* err = pa::device_error_word(&e);
  if (!err) return cuda_fail(e);
  const int64_t block_bytes = int64_t(block_size) * num_kv_heads * head_dim * elem_bytes(dtype);
  e = pa::launch_copy_blocks(k_cache, v_cache, block_mapping, num_pairs, num_blocks, block_bytes, err,
                             reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

int pa_attention_workspace_size(int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                                size_t* bytes_out) {
  if (!bytes_out || num_seqs < 0 || num_heads < 1 || num_kv_heads < 1) return PA_ERR_INVALID_ARG;
  if (num_heads % num_kv_heads != 0) return PA_ERR_INVALID_ARG;
  if (!pa::decode_supported(PA_BF16, head_dim, num_heads / num_kv_heads)) return PA_ERR_UNSUPPORTED;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  const int ctas = pa::decode_num_ctas(dev, &e);
  if (e != cudaSuccess) return cuda_fail(e);
  // The largest of the element types' layouts, so one size serves them all.
  size_t need = 0;
  for (pa_dtype dt : {PA_BF16, PA_F32, PA_FP8_E4M3}) {
    const size_t n = pa::decode_workspace_bytes(num_seqs, num_heads, num_kv_heads, head_dim, ctas, dt);
    need = n > need ? n : need;
  }
  *bytes_out = need + pa::kPrefillSchedBytes;
  return PA_OK;
}

}  // extern "C"

namespace {

// Where a row input of an attention call lives: 0 device memory (or managed) of the current
// device, 1 page-locked host memory mapped at its own address, -1 anything else (pageable
// host memory, another device's memory), which no kernel may dereference.
int input_home(const void* p, int dev) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();  // reset the error state the failed query set
    return -1;
  }
  switch (at.type) {
    case cudaMemoryTypeDevice: return at.device == dev ? 0 : -1;
    case cudaMemoryTypeManaged: return 0;
    case cudaMemoryTypeHost: return at.devicePointer == p ? 1 : -1;
    default: return -1;
  }
}

// Validation and argument packing shared by pa_attention and pa_write_attention; nothing
// is launched. On success `a` and `ctas` are ready for run_attention.
int prepare_attention(void* out, const void* q, const void* k_cache, const void* v_cache,
                      const int32_t* block_table, int max_blocks_per_seq, const int32_t* seq_lens,
                      const int32_t* query_start_loc, int num_seqs, int num_tokens, int max_query_len,
                      int max_seq_len, int num_heads, int num_kv_heads, int head_dim, int block_size,
                      int64_t num_blocks, float scale, pa_dtype dtype, void* workspace,
                      size_t workspace_bytes, pa::AttnArgs& a, int& ctas, bool& nothing,
                      pa_dtype cache_dtype) {
  nothing = false;
  int st = check_cache(k_cache, v_cache, num_blocks, block_size, num_kv_heads, head_dim, cache_dtype);
  if (st != PA_OK) return st;
  if (num_seqs < 0 || num_tokens < 0 || max_query_len < 0 || max_seq_len < 0) return PA_ERR_INVALID_ARG;
  if (num_heads < 1 || num_heads % num_kv_heads != 0) return PA_ERR_INVALID_ARG;
  if (!(scale > 0.f) || scale != scale) return PA_ERR_INVALID_ARG;
  if (num_seqs == 0 || num_tokens == 0) {
    nothing = true;
    return PA_OK;
  }
  if (!out || !q || !block_table || !seq_lens || !query_start_loc) return PA_ERR_INVALID_ARG;
  if (!aligned16(out) || !aligned16(q)) return PA_ERR_INVALID_ARG;
  if (max_blocks_per_seq < 1) return PA_ERR_INVALID_ARG;
  if (int64_t(max_blocks_per_seq) * block_size > 0x7fffffff) return PA_ERR_INVALID_ARG;
  if (int64_t(max_blocks_per_seq) * block_size < max_seq_len) return PA_ERR_INVALID_ARG;
  if (max_query_len > max_seq_len) return PA_ERR_INVALID_ARG;
  const int G = num_heads / num_kv_heads;
  if (!pow2_le8(G) || (head_dim != 64 && head_dim != 128)) return PA_ERR_UNSUPPORTED;
  if (!(16 % block_size == 0 || block_size % 16 == 0)) return PA_ERR_UNSUPPORTED;
  if (!pa::decode_supported(dtype, head_dim, G) || !pa::prefill_supported(dtype, head_dim, G))
    return PA_ERR_UNSUPPORTED;
  if (num_seqs > 0x7fffffff / 8) return PA_ERR_INVALID_ARG;
  if (num_kv_heads > 65535 || (max_query_len + 7) / 8 > 65535) return PA_ERR_UNSUPPORTED;  // prefill grid

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  // Make the device's primary context current on this thread: the tensor maps are encoded
  // by a driver call before any other CUDA call of the attention path, and in a thread that
  // has made no CUDA call yet no context is current (the encoding then fails).
  e = cudaSetDevice(dev);
  if (e != cudaSuccess) return cuda_fail(e);
  ctas = pa::decode_num_ctas(dev, &e);
  if (e != cudaSuccess) return cuda_fail(e);
  const size_t dneed = pa::decode_workspace_bytes(num_seqs, num_heads, num_kv_heads, head_dim, ctas, cache_dtype);
  const size_t need = dneed + pa::kPrefillSchedBytes;
  if (!workspace || workspace_bytes < need || !aligned16(workspace)) return PA_ERR_WORKSPACE;
  unsigned int* err = pa::device_error_word(&e);
  if (!err) return cuda_fail(e);

  a.out = out;
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.block_table = block_table;
  a.seq_lens = seq_lens;
  a.query_start_loc = query_start_loc;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.num_seqs = num_seqs;
  a.num_tokens = num_tokens;
  a.max_query_len = max_query_len;
  a.num_heads = num_heads;
  a.num_kv_heads = num_kv_heads;
  a.head_dim = head_dim;
  a.block_size = block_size;
  a.num_blocks = num_blocks;
  a.scale = scale;
  a.dtype = dtype;
  a.cache_dtype = cache_dtype;
  a.workspace = workspace;
  a.prefill_sched = reinterpret_cast<int*>(static_cast<unsigned char*>(workspace) + dneed);
  a.err = err;
  const int qh = input_home(q, dev);
  if (qh < 0) return PA_ERR_INVALID_ARG;
  a.host_inputs = qh == 1;
  return PA_OK;
}

// Host-memory row inputs are read by the tensor-core decode kernel only (plain loads over
// the CPU-GPU link): decode-only batches on that kernel.
int check_host_inputs(const pa::AttnArgs& a) {
  if (!a.host_inputs) return PA_OK;
  if (a.max_query_len >= 2) return PA_ERR_INVALID_ARG;
  const int hg = pa::decode_hg(a.cache_dtype, a.head_dim, a.num_heads / a.num_kv_heads, a.num_kv_heads);
  return pa::decode_mma_supported(a, hg) ? PA_OK : PA_ERR_UNSUPPORTED;
}

// Whether `s` is being captured into a CUDA graph (an error of the query counts as yes).
bool stream_capturing(cudaStream_t s) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) {
    cudaGetLastError();  // reset the error state the failed query set
    return true;
  }
  return cs != cudaStreamCaptureStatusNone;
}

// A cache write to enqueue ahead of the attention kernels (pa_write_attention with prefill
// rows), after the attention's own host-side preparation.
struct KvWriteStep {
  const void* k;
  const void* v;
  const int64_t* slot_mapping;
  int64_t row_bytes;
};

int run_attention(const pa::AttnArgs& a, int ctas, cudaStream_t s, const KvWriteStep* write = nullptr) {
  const bool prefill = a.max_query_len >= 2;
  const bool tc = prefill && pa::prefill_tc_supported(a);
  pa::PrefillTcPlan plan;
  if (tc) {  // every host-side step of the prefill launches that can fail, before any launch
    const cudaError_t e = pa::prepare_prefill_tc(a, &plan);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  if (write) {
    const cudaError_t e = pa::launch_kv_write(write->k, write->v, const_cast<void*>(a.k_cache),
                                              const_cast<void*>(a.v_cache), write->slot_mapping, a.num_tokens,
                                              a.num_blocks * a.block_size, write->row_bytes, a.err, s);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  const int hg = pa::decode_hg(a.cache_dtype, a.head_dim, a.num_heads / a.num_kv_heads, a.num_kv_heads);
  // Side by side only with the tensor-core decode kernel (its CTAs and the prefill kernel's
  // cannot share an SM, which keeps the SM split below), and never while `s` is captured
  // into a graph: the internal stream is shared by every caller of the device, and a
  // capture would hold it until the capture ends.
  if (tc && a.concurrent && pa::decode_mma_supported(a, hg) && !stream_capturing(s)) {
    // A batch with prefill rows: the decode kernels (HBM-bound) run on 3/5 of the SMs (1/2
    // over an E4M3 cache, whose prefill steps cost more: the best of 1/2 .. 3/4 measured on
    // the mixed chunked-prefill batch for each cache type), on a side stream of the
    // highest priority, beside a first prefill launch (tensor-bound) of as many CTAs as
    // the other SMs on the caller's stream, so neither can take the other's
    // SMs whichever is dispatched first. A second prefill launch queued behind the decode
    // merge on the side stream takes the SMs the decode kernel leaves; both launches draw
    // the remaining pairs from one counter, zeroed before the fork. The caller's stream
    // then waits for the side stream -- on the error path too, once the fork is recorded,
    // so nothing the call queued is left unordered against the caller's later work.
    pa::SideStream side;
    cudaError_t e;
    if (!pa::side_stream(&side, &e)) return cuda_fail(e);
    pa::AttnArgs ad = a;
    ad.merge_pdl = false;  // the merge's CTAs must not hold SMs while the decode kernel runs
    const int dctas = ctas > 1 ? (a.cache_dtype == PA_FP8_E4M3 ? ctas / 2 : ctas * 3 / 5) : 1;
    const int pctas = ctas - dctas > 0 ? ctas - dctas : 1;
    std::lock_guard<std::mutex> lock(*side.mu);
    e = cudaMemsetAsync(a.prefill_sched, 0, sizeof(int), s);
    if (e == cudaSuccess) e = cudaEventRecord(side.fork, s);
    if (e != cudaSuccess) return cuda_fail(e);
    e = cudaStreamWaitEvent(side.stream, side.fork, 0);
    if (e == cudaSuccess) e = pa::launch_decode(ad, dctas, side.stream);
    if (e == cudaSuccess) e = pa::launch_prefill_tc(a, plan, pctas, s, pa::PrefillLaunch{true, pctas, false});
    if (e == cudaSuccess) e = pa::launch_prefill_tc(a, plan, ctas, side.stream, pa::PrefillLaunch{false, pctas, false});
    cudaError_t j = cudaEventRecord(side.join, side.stream);
    if (j == cudaSuccess) j = cudaStreamWaitEvent(s, side.join, 0);
    if (e == cudaSuccess) e = j;
    return e == cudaSuccess ? PA_OK : cuda_fail(e);
  }
  cudaError_t e = pa::launch_decode(a, ctas, s);
  if (e != cudaSuccess) return cuda_fail(e);
  if (prefill) {
    e = tc ? pa::launch_prefill_tc(a, plan, ctas, s, pa::PrefillLaunch{true, ctas, true}) : pa::launch_prefill(a, s);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  return PA_OK;
}

}  // namespace

namespace pa {

int attention_entry(void* out, const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
                    int max_blocks_per_seq, const int32_t* seq_lens, const int32_t* query_start_loc, int num_seqs,
                    int num_tokens, int max_query_len, int max_seq_len, int num_heads, int num_kv_heads,
                    int head_dim, int block_size, int64_t num_blocks, float scale, pa_dtype dtype, void* workspace,
                    size_t workspace_bytes, pa_stream_t stream, bool concurrent) {
  AttnArgs a;
  int ctas = 0;
  bool nothing = false;
  const int st = prepare_attention(out, q, k_cache, v_cache, block_table, max_blocks_per_seq, seq_lens,
                                   query_start_loc, num_seqs, num_tokens, max_query_len, max_seq_len, num_heads,
                                   num_kv_heads, head_dim, block_size, num_blocks, scale, dtype, workspace,
                                   workspace_bytes, a, ctas, nothing, dtype);
  if (st != PA_OK || nothing) return st;
  a.concurrent = concurrent;
  const int hs = check_host_inputs(a);
  if (hs != PA_OK) return hs;
  return run_attention(a, ctas, reinterpret_cast<cudaStream_t>(stream));
}

}  // namespace pa

extern "C" {

int pa_attention(void* out, const void* q, const void* k_cache, const void* v_cache,
                 const int32_t* block_table, int max_blocks_per_seq, const int32_t* seq_lens,
                 const int32_t* query_start_loc, int num_seqs, int num_tokens, int max_query_len,
                 int max_seq_len, int num_heads, int num_kv_heads, int head_dim, int block_size,
                 int64_t num_blocks, float scale, pa_dtype dtype, void* workspace,
                 size_t workspace_bytes, pa_stream_t stream) {
  return pa::attention_entry(out, q, k_cache, v_cache, block_table, max_blocks_per_seq, seq_lens, query_start_loc,
                             num_seqs, num_tokens, max_query_len, max_seq_len, num_heads, num_kv_heads, head_dim,
                             block_size, num_blocks, scale, dtype, workspace, workspace_bytes, stream, true);
}

int pa_write_attention(void* out, const void* q, const void* k_new, const void* v_new,
                       const int64_t* slot_mapping, void* k_cache, void* v_cache,
                       const int32_t* block_table, int max_blocks_per_seq, const int32_t* seq_lens,
                       const int32_t* query_start_loc, int num_seqs, int num_tokens, int max_query_len,
                       int max_seq_len, int num_heads, int num_kv_heads, int head_dim, int block_size,
                       int64_t num_blocks, float scale, pa_dtype dtype, void* workspace,
                       size_t workspace_bytes, pa_stream_t stream) {
  if (num_seqs > 0 && num_tokens > 0) {
    if (!k_new || !v_new || !slot_mapping || !aligned16(k_new) || !aligned16(v_new)) return PA_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(slot_mapping) % 8 != 0) return PA_ERR_INVALID_ARG;
  }
  pa::AttnArgs a;
  int ctas = 0;
  bool nothing = false;
  const int st = prepare_attention(out, q, k_cache, v_cache, block_table, max_blocks_per_seq, seq_lens,
                                   query_start_loc, num_seqs, num_tokens, max_query_len, max_seq_len, num_heads,
                                   num_kv_heads, head_dim, block_size, num_blocks, scale, dtype, workspace,
                                   workspace_bytes, a, ctas, nothing, dtype);
  if (st != PA_OK || nothing) return st;
  {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cuda_fail(cudaGetLastError());
    const int kh = input_home(k_new, dev), vh = input_home(v_new, dev);
    if (kh < 0 || vh < 0) return PA_ERR_INVALID_ARG;
    a.host_inputs = a.host_inputs || kh == 1 || vh == 1;
    const int hs = check_host_inputs(a);
    if (hs != PA_OK) return hs;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (max_query_len >= 2) {
    // prefill rows read their own new tokens from the cache through many CTAs: write every
    // new token first, then attend
    const KvWriteStep w{k_new, v_new, slot_mapping, int64_t(num_kv_heads) * head_dim * elem_bytes(dtype)};
    return run_attention(a, ctas, s, &w);
  }
  a.k_new = k_new;  // a decode-only batch: the decode kernel writes each new token itself
  a.v_new = v_new;
  a.slot_mapping = slot_mapping;
  return run_attention(a, ctas, s);
}

int pa_kv_write_fp8(const void* k, const void* v, pa_dtype in_dtype, void* k_cache, void* v_cache,
                    const int64_t* slot_mapping, int64_t num_tokens, int64_t num_blocks, int block_size,
                    int num_kv_heads, int head_dim, float k_scale, float v_scale, pa_stream_t stream) {
  int st = check_cache(k_cache, v_cache, num_blocks, block_size, num_kv_heads, head_dim, PA_FP8_E4M3);
  if (st != PA_OK) return st;
  if (in_dtype != PA_BF16 && in_dtype != PA_F32) return PA_ERR_INVALID_ARG;
  if (!(k_scale > 0.f) || !(v_scale > 0.f) || k_scale == INFINITY || v_scale == INFINITY) return PA_ERR_INVALID_ARG;
  if ((int64_t(num_kv_heads) * head_dim) % 16 != 0) return PA_ERR_UNSUPPORTED;
  if (num_tokens < 0) return PA_ERR_INVALID_ARG;
  if (num_tokens == 0) return PA_OK;
  if (!k || !v || !slot_mapping || !aligned16(k) || !aligned16(v)) return PA_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(slot_mapping) % 8 != 0) return PA_ERR_INVALID_ARG;
  cudaError_t e;
  unsigned int* err = pa::device_error_word(&e);
  if (!err) return cuda_fail(e);
  e = pa::launch_kv_write_fp8(k, v, in_dtype, k_cache, v_cache, slot_mapping, num_tokens, num_blocks * block_size,
                              int64_t(num_kv_heads) * head_dim, k_scale, v_scale, err,
                              reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

int pa_attention_fp8(void* out, const void* q, const void* k_cache, const void* v_cache,
                     const int32_t* block_table, int max_blocks_per_seq, const int32_t* seq_lens,
                     const int32_t* query_start_loc, int num_seqs, int num_tokens, int max_query_len,
                     int max_seq_len, int num_heads, int num_kv_heads, int head_dim, int block_size,
                     int64_t num_blocks, float scale, float k_scale, float v_scale, void* workspace,
                     size_t workspace_bytes, pa_stream_t stream) {
  if (!(k_scale > 0.f) || !(v_scale > 0.f) || k_scale == INFINITY || v_scale == INFINITY) return PA_ERR_INVALID_ARG;
  pa::AttnArgs a;
  int ctas = 0;
  bool nothing = false;
  const int st = prepare_attention(out, q, k_cache, v_cache, block_table, max_blocks_per_seq, seq_lens,
                                   query_start_loc, num_seqs, num_tokens, max_query_len, max_seq_len, num_heads,
                                   num_kv_heads, head_dim, block_size, num_blocks, scale, PA_BF16, workspace,
                                   workspace_bytes, a, ctas, nothing, PA_FP8_E4M3);
  if (st != PA_OK || nothing) return st;
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  const int hs = check_host_inputs(a);
  if (hs != PA_OK) return hs;
  return run_attention(a, ctas, reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"

namespace {

// A pool pointer the kernels may dereference: device memory of the current device, managed
// memory, or pinned host memory mapped at the same address (unified addressing).
int check_kernel_visible(const void* p, int dev) {
  cudaPointerAttributes at;
  cudaError_t e = cudaPointerGetAttributes(&at, p);
  if (e != cudaSuccess) {
    cudaGetLastError();  // reset the error state the failed query set
    return PA_ERR_INVALID_ARG;
  }
  switch (at.type) {
    case cudaMemoryTypeDevice: return at.device == dev ? PA_OK : PA_ERR_INVALID_ARG;
    case cudaMemoryTypeManaged: return PA_OK;
    case cudaMemoryTypeHost: return at.devicePointer == p ? PA_OK : PA_ERR_INVALID_ARG;
    default: return PA_ERR_INVALID_ARG;  // pageable host memory
  }
}

}  // namespace

extern "C" {

int pa_swap_blocks(const void* src_k, const void* src_v, void* dst_k, void* dst_v, const int64_t* block_mapping,
                   int64_t num_pairs, int64_t src_num_blocks, int64_t dst_num_blocks, int block_size,
                   int num_kv_heads, int head_dim, pa_dtype dtype, pa_stream_t stream) {
  if (!src_k || !src_v || !dst_k || !dst_v) return PA_ERR_INVALID_ARG;
  if (!aligned16(src_k) || !aligned16(src_v) || !aligned16(dst_k) || !aligned16(dst_v)) return PA_ERR_INVALID_ARG;
  if (src_num_blocks < 1 || dst_num_blocks < 1 || block_size < 1 || num_kv_heads < 1 || head_dim < 1)
    return PA_ERR_INVALID_ARG;
  if (elem_bytes(dtype) == 0) return PA_ERR_INVALID_ARG;
  const int64_t block_bytes = int64_t(block_size) * num_kv_heads * head_dim * elem_bytes(dtype);
  if (block_bytes % 16 != 0) return PA_ERR_UNSUPPORTED;
  if (block_bytes / 16 > 0x7fffffff) return PA_ERR_UNSUPPORTED;
  if (num_pairs < 0 || num_pairs > 0x7fffffff) return PA_ERR_INVALID_ARG;
  if (num_pairs == 0) return PA_OK;
  if (!block_mapping || reinterpret_cast<uintptr_t>(block_mapping) % 8 != 0) return PA_ERR_INVALID_ARG;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  for (const void* p : {src_k, src_v, static_cast<const void*>(dst_k), static_cast<const void*>(dst_v),
                        static_cast<const void*>(block_mapping)}) {
    const int st = check_kernel_visible(p, dev);
    if (st != PA_OK) return st;
  }
  unsigned int* err = pa::device_error_word(&e);
  if (!err) return cuda_fail(e);
  e = pa::launch_swap_blocks(src_k, src_v, dst_k, dst_v, block_mapping, num_pairs, src_num_blocks, dst_num_blocks,
                             block_bytes, err, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

int pa_attention_grouped_workspace_size(int num_seqs, int num_groups, int num_heads, int num_kv_heads, int head_dim,
                                        size_t* bytes_out) {
  if (!bytes_out || num_seqs < 0 || num_groups < 0 || num_heads < 1 || num_kv_heads < 1) return PA_ERR_INVALID_ARG;
  if (num_heads % num_kv_heads != 0) return PA_ERR_INVALID_ARG;
  size_t plain = 0;
  const int st = pa_attention_workspace_size(num_seqs, num_heads, num_kv_heads, head_dim, &plain);
  if (st != PA_OK) return st;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  const int ctas = pa::decode_num_ctas(dev, &e);
  if (e != cudaSuccess) return cuda_fail(e);
  const int G = num_heads / num_kv_heads;
  size_t need = plain;
  for (pa_dtype dt : {PA_BF16, PA_FP8_E4M3}) {
    const int hg = pa::decode_hg(dt, head_dim, G, num_kv_heads);
    const size_t n = pa::decode_grouped_workspace_bytes(num_seqs, num_groups, num_kv_heads, head_dim, hg, ctas);
    need = n > need ? n : need;
  }
  *bytes_out = need;
  return PA_OK;
}

int pa_attention_grouped(void* out, const void* q, const void* k_cache, const void* v_cache,
                         const int32_t* block_table, int max_blocks_per_seq, const int32_t* seq_lens,
                         const int32_t* query_start_loc, int num_seqs, int num_tokens, int max_seq_len,
                         int num_heads, int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                         float scale, pa_dtype dtype, const int32_t* seq_group, const int32_t* group_range,
                         const int32_t* shared_len, int num_groups, void* workspace, size_t workspace_bytes,
                         pa_stream_t stream) {
  if (num_groups < 0) return PA_ERR_INVALID_ARG;
  if (num_groups > 0 && (!seq_group || !group_range || !shared_len)) return PA_ERR_INVALID_ARG;
  pa::AttnArgs a;
  int ctas = 0;
  bool nothing = false;
  int st = prepare_attention(out, q, k_cache, v_cache, block_table, max_blocks_per_seq, seq_lens, query_start_loc,
                             num_seqs, num_tokens, 1, max_seq_len, num_heads, num_kv_heads, head_dim, block_size,
                             num_blocks, scale, dtype, workspace, workspace_bytes, a, ctas, nothing, dtype);
  if (st != PA_OK || nothing) return st;
  if (num_tokens != num_seqs) return PA_ERR_INVALID_ARG;  // a decode batch: one query per request
  const int hg = pa::decode_hg(dtype, head_dim, num_heads / num_kv_heads, num_kv_heads);
  a.seq_group = seq_group;
  a.group_start = group_range;
  a.shared_len = shared_len;
  a.num_groups = num_groups;
  if (!pa::decode_mma_supported(a, hg)) return PA_ERR_UNSUPPORTED;
  const int hs = check_host_inputs(a);
  if (hs != PA_OK) return hs;
  const size_t need = pa::decode_grouped_workspace_bytes(num_seqs, num_groups, num_kv_heads, head_dim, hg, ctas);
  if (!workspace || workspace_bytes < need || !aligned16(workspace)) return PA_ERR_WORKSPACE;
  const cudaError_t e = pa::launch_decode_mma(a, hg, ctas, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

}  // extern "C"
