/*
 * pa.h -- C ABI of the GB300 (sm_103a) paged-KV-cache hot path.
 *
 * Device operations and a host block manager:
 *   pa_kv_write     scatter new tokens' K/V into physical cache blocks through slot_mapping
 *   pa_attention    paged decode and chunked-prefill attention through block_table
 *   pa_write_attention  the two above in one call (the write fused into decode)
 *   pa_kv_write_fp8 / pa_attention_fp8  the same over FP8 (E4M3) caches
 *   pa_attention_grouped  decode attention reading a shared prefix once per group
 *   pa_copy_blocks  copy whole physical blocks (the copy step of copy-on-write)
 *   pa_swap_blocks  move whole blocks between the GPU pool and a CPU pool (preemption)
 *   pa_bm_*         host-side block accounting: free queue, block tables, ref counts, CoW
 *
 * Conventions shared by every entry point:
 *  - Cache layout: k_cache and v_cache are each [num_blocks, block_size, num_kv_heads,
 *    head_dim], row-major and contiguous, element type `dtype`. A "slot" is one token
 *    position in the pool: slot = block * block_size + offset, i.e. the row index of
 *    the cache viewed as [num_blocks * block_size, num_kv_heads * head_dim].
 *  - Pointers marked "device" must point to device memory of the current CUDA device,
 *    owned by the caller and 16-byte aligned; the library never allocates, frees or
 *    synchronises (except pa_read_device_errors, which synchronises by design). Work is
 *    enqueued on `stream` (0 = legacy default stream) and the call returns before it runs.
 *  - Return value: a pa_status. Argument checks happen before anything is launched; a
 *    call that returns an error has enqueued nothing. PA_ERR_CUDA means a launch
 *    failed; pa_last_cuda_error() gives the cudaError_t of the calling thread's last one.
 *  - Index values inside device arrays (slots, block ids, lengths) cannot be checked on
 *    the host. Kernels check them against the sizes passed in and skip any access that
 *    would leave the buffers; such a skip sets a bit in a per-device error word that
 *    pa_read_device_errors() returns. Results are then unspecified but no memory outside
 *    the arguments is touched.
 *  - Per-device state: the library looks up a few device addresses (the error word, the
 *    fixed scratch of pa_attention_fixed_scratch) and creates a side stream with two
 *    events once per device, on first use, and keeps them until exit. A process that
 *    resets a device (cudaDeviceReset) or otherwise destroys its primary context must not
 *    call the library for that device afterwards: the kept addresses and handles would be
 *    stale.
 *
 * Sources (the pages this library restates):
 *  [docs]  "vLLM", docs.acceleratez.fun/llm/model-inference/vllm.html -- PagedAttention
 *          (blocks, block table, algorithm flow), memory-utilisation arithmetic,
 *          Copy-on-Write (reference counting, copy before a divergent write).
 *  [flow]  vLLM 0.10.0 flow analysis, ascendai.csdn.net/69ac14cf54b52172bc5fa372.html --
 *          3.2 Scheduler (prefill compute-bound, decode memory-bound, chunked prefill
 *          mixed with decodes), 3.3 KV Manager (slot, block, pool, slot_mapping),
 *          3.5 Attention (q is the flattened token batch; metadata block_table,
 *          slot_mapping, query_start_loc).
 *  [read]  vLLM code reading, sourceaix.com/community/post/7301643446391930880 --
 *          5.1.1 single request (logical vs physical blocks, '# filled'),
 *          5.2.1 parallel sampling (shared blocks, ref count, copy-on-write).
 *  [intro] VLLM overview, dn008.com.cn/news/553482 -- 2.1 KV cache (causal mask); 4
 *          scheduler (waiting / running / swapped queues, swap phase).
 */
#ifndef PA_H_
#define PA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* pa_stream_t;

typedef enum { PA_F32 = 0, PA_BF16 = 1, PA_FP8_E4M3 = 2 /* caches only: see pa_kv_write_fp8 */ } pa_dtype;

typedef enum {
  PA_OK = 0,
  PA_ERR_INVALID_ARG = 1,  /* null pointer, negative size, misaligned pointer, bad shape */
  PA_ERR_UNSUPPORTED = 2,  /* a valid shape the library has no kernel for */
  PA_ERR_WORKSPACE = 3,    /* workspace missing or smaller than pa_attention_workspace_size */
  PA_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed */
  PA_ERR_NO_BLOCKS = 5,    /* block manager: not enough free blocks now */
  PA_ERR_TOO_LARGE = 6,    /* block manager: the sequence can never fit the pool */
  PA_ERR_NOT_FOUND = 7,    /* block manager: unknown sequence id, or id already in use */
} pa_status;

/* Bits of the per-device error word (see pa_read_device_errors). */
#define PA_DEVERR_SLOT_RANGE   0x1u  /* a slot >= num_blocks * block_size was skipped */
#define PA_DEVERR_BLOCK_RANGE  0x2u  /* a block id outside [0, num_blocks) was skipped */
#define PA_DEVERR_SEQ_RANGE    0x4u  /* seq_len > max_blocks_per_seq * block_size, or q_len > seq_len */
#define PA_DEVERR_TIMEOUT      0x8u  /* a pipeline wait gave up (the kernel returned early) */
#define PA_DEVERR_SLOT_MISMATCH 0x10u /* pa_write_attention: a decode token's slot is not its position's slot */

const char* pa_status_string(int status);
int pa_last_cuda_error(void);

/* Reads the current device's error word (synchronising the device) and clears it if
 * `clear` is non-zero. Returns PA_OK or PA_ERR_CUDA. */
int pa_read_device_errors(unsigned int* flags_out, int clear);

/* ------------------------------------------------------------------------------
 * pa_kv_write -- [docs] PagedAttention, algorithm flow (prefill step c, decode step d:
 * store each new token's KV in its physical block); [flow] 3.3 KV Manager (the model
 * runner builds slot_mapping; attention finds each token's KV through it).
 *
 * For every t in [0, num_tokens) with s = slot_mapping[t] >= 0:
 *     k_cache[s / block_size, s % block_size, :, :] = k[t, :, :]   (same for v)
 * A negative slot marks a padding token: nothing is written for it.
 *
 * k, v          device, [num_tokens, num_kv_heads, head_dim], contiguous, `dtype`
 * k_cache, ...  device, cache layout above (written in place)
 * slot_mapping  device, int64 [num_tokens]; slots must be distinct (no two tokens
 *               written to one slot in a call -- which one would win is unspecified)
 * num_tokens    >= 0 (0 enqueues nothing)
 * Byte-exact copy; no arithmetic on the values.
 * --------------------------------------------------------------------------- */
int pa_kv_write(const void* k, const void* v, void* k_cache, void* v_cache,
                const int64_t* slot_mapping, int64_t num_tokens, int64_t num_blocks,
                int block_size, int num_kv_heads, int head_dim, pa_dtype dtype,
                pa_stream_t stream);

/* ------------------------------------------------------------------------------
 * pa_copy_blocks -- [docs] Copy-on-Write (copy the old block's content into the newly
 * allocated block before the divergent write); [read] 5.2.1 (A1's block 1 copied to 3).
 *
 * For each i in [0, num_pairs): src = block_mapping[2i], dst = block_mapping[2i+1]:
 *     k_cache[dst] = k_cache[src]; v_cache[dst] = v_cache[src]   (all block_size slots)
 * block_mapping  device, int64 [num_pairs, 2]
 * Pairs are applied concurrently: no dst may repeat or appear as another pair's src
 * (pairs emitted by the block manager below always satisfy this: every dst is a block
 * just taken from the free queue and every src is a block still held by others).
 * Byte-exact copy.
 * --------------------------------------------------------------------------- */
int pa_copy_blocks(void* k_cache, void* v_cache, const int64_t* block_mapping,
                   int64_t num_pairs, int64_t num_blocks, int block_size, int num_kv_heads,
                   int head_dim, pa_dtype dtype, pa_stream_t stream);

/* ------------------------------------------------------------------------------
 * pa_attention -- [flow] 3.5 Attention (q = flattened tokens of the batch, requests
 * delimited by query_start_loc; K/V read from the whole cache through block_table);
 * [docs] PagedAttention (block table: logical block -> physical block); [read] 5.1.1
 * (attention runs over the logical blocks, as if contiguous); [intro] 2.1 (causal);
 * [flow] 3.2 (chunked prefill mixed with decodes in one batch).
 *
 * For request s with q_len = query_start_loc[s+1] - query_start_loc[s] and
 * L = seq_lens[s] (keys, including the request's new tokens), query row j (token
 * t = query_start_loc[s] + j) sits at position p = L - q_len + j and, for each query
 * head h with KV head g = h / (num_heads / num_kv_heads):
 *     K_i = k_cache[block_table[s, i / block_size], i % block_size, g, :]   (V alike)
 *     out[t, h, :] = sum_{i<=p} softmax_i(scale * <q[t, h, :], K_i>) * V_i
 * Softmax and accumulation in fp32; out is written in `dtype` (bf16 rounded to nearest
 * even). Requests with q_len == 1 run the split-K decode kernel; q_len >= 2 the prefill
 * kernel; q_len == 0 produces no rows. Requires q_len <= L.
 * With rows of both kinds (max_query_len >= 2) and the tensor-core kernels for both (see
 * "Prefill kernels" below; block size 8, 16, 32, 64 or 128) the two kernels run side by
 * side: the call forks an internal stream of the highest priority off `stream` (event
 * record and wait), runs the decode kernels there on 3/5 of the SMs (1/2 with E4M3
 * caches) and joins it back before returning -- also when a launch fails after the fork --
 * so later work on `stream` is ordered after the whole call, as for one stream. The first such call
 * on a device creates that stream and two events (kept until exit). While `stream` is
 * being captured into a CUDA graph the call keeps every kernel on `stream` instead (the
 * internal stream is shared by all callers of the device and must not join a capture).
 * The decode rows' bits differ between the two ways (a split over fewer CTAs beside the
 * prefill kernel; same tolerance).
 * Prefill kernels: the tensor-core kernel takes bf16 q and out over bf16 caches (head_dim
 * 64 / 128) or E4M3 caches (head_dim 128; see pa_attention_fp8), at most 4096 requests,
 * block size 8, 16, 32, 64 or 128; other prefill batches (fp32, block sizes 1, 2, 4 or
 * above 128, more than 4096 requests) run a CUDA-core kernel with the same result within
 * the tolerance, many times slower.
 * The result does not depend on which physical blocks hold the tokens: the reduction
 * order is fixed by positions only, so relabelling block ids gives identical bits.
 *
 * out           device, [num_tokens, num_heads, head_dim], `dtype` (written, never read);
 *               may also be page-locked host memory mapped into the unified address
 *               space: the kernels then store the rows over the CPU-GPU link and the host
 *               sees them once the stream has been synchronised
 * q             device, [num_tokens, num_heads, head_dim], `dtype`; for a decode-only
 *               batch (max_query_len <= 1) on the tensor-core decode kernel it may also be
 *               page-locked host memory mapped into the unified address space: the kernel
 *               then reads the rows over the CPU-GPU link (plain loads, no copy). q is
 *               checked with cudaPointerGetAttributes: pageable host memory or another
 *               device's memory gives PA_ERR_INVALID_ARG; host memory with prefill rows gives
 *               PA_ERR_INVALID_ARG, and on a shape the tensor-core decode kernel does not take
 *               PA_ERR_UNSUPPORTED (all before anything is enqueued)
 * block_table   device, int32 [num_seqs, max_blocks_per_seq] (entries past a request's
 *               ceil(L / block_size) blocks are never read)
 * seq_lens      device, int32 [num_seqs]
 * query_start_loc device, int32 [num_seqs + 1], non-decreasing, [0] = 0, [num_seqs] =
 *               num_tokens
 * max_query_len host: an upper bound of every q_len (sizes the prefill grid)
 * max_seq_len   host: an upper bound of every L (validated against the table width)
 * workspace     device scratch of at least pa_attention_workspace_size() bytes (at least
 *               16: its last part holds the prefill kernel's work counter, which the call
 *               zeroes on its stream before that kernel); no initial contents needed; must
 *               not be used by another call that may run concurrently.
 * Supported: dtype PA_F32 / PA_BF16; head_dim 64 / 128; num_heads / num_kv_heads in
 * {1, 2, 4, 8}; block_size a divisor of 16 (1, 2, 4, 8, 16) or a multiple of 16.
 * --------------------------------------------------------------------------- */
int pa_attention_workspace_size(int num_seqs, int num_heads, int num_kv_heads,
                                int head_dim, size_t* bytes_out);

int pa_attention(void* out, const void* q, const void* k_cache, const void* v_cache,
                 const int32_t* block_table, int max_blocks_per_seq, const int32_t* seq_lens,
                 const int32_t* query_start_loc, int num_seqs, int num_tokens,
                 int max_query_len, int max_seq_len, int num_heads, int num_kv_heads,
                 int head_dim, int block_size, int64_t num_blocks, float scale,
                 pa_dtype dtype, void* workspace, size_t workspace_bytes, pa_stream_t stream);

/* ------------------------------------------------------------------------------
 * pa_write_attention -- pa_kv_write followed by pa_attention, in one call:
 * [docs] PagedAttention algorithm flow (decode step d stores the new token's KV in its
 * block, then attends over all of the request's blocks); [flow] 3.3 / 3.5 (slot_mapping
 * feeds the cache write that precedes attention in the same forward pass).
 *
 * Result (cache and out) identical to pa_kv_write(k_new, v_new, ..., slot_mapping,
 * num_tokens, ...) then pa_attention(...) on one stream, under one extra contract: for
 * a request with q_len == 1 at length L, slot_mapping of its token is the slot of
 * position L - 1, block_table[s, (L-1) / block_size] * block_size + (L-1) % block_size
 * (or negative: a padding token, nothing written). A token breaking this sets
 * PA_DEVERR_SLOT_MISMATCH; its KV is still written, its request's output is then
 * unspecified.
 *  - max_query_len <= 1 (a decode-only batch): one launch pair. The split-K CTA that
 *    streams a request's last 16 positions for a KV-head group first copies that group's
 *    slice of the new K/V row into the cache, then reads it back with the rest, so the
 *    new token costs one write and no separate kernel.
 *  - max_query_len >= 2: the cache write is a separate kernel ahead of the attention
 *    kernels (prefill rows read their new tokens through many CTAs).
 * k_new, v_new  device, [num_tokens, num_kv_heads, head_dim], `dtype`, 16-byte aligned;
 *               like q, page-locked host memory for decode-only batches (read over the link)
 * slot_mapping  device, int64 [num_tokens], distinct non-negative slots
 * Other arguments, validation, workspace and errors as pa_kv_write and pa_attention;
 * validation happens before anything is enqueued.
 * --------------------------------------------------------------------------- */
int pa_write_attention(void* out, const void* q, const void* k_new, const void* v_new,
                       const int64_t* slot_mapping, void* k_cache, void* v_cache,
                       const int32_t* block_table, int max_blocks_per_seq, const int32_t* seq_lens,
                       const int32_t* query_start_loc, int num_seqs, int num_tokens,
                       int max_query_len, int max_seq_len, int num_heads, int num_kv_heads,
                       int head_dim, int block_size, int64_t num_blocks, float scale,
                       pa_dtype dtype, void* workspace, size_t workspace_bytes, pa_stream_t stream);

/* ------------------------------------------------------------------------------
 * pa_attention_grouped -- pa_attention for a decode batch (one query per request) whose
 * requests come in groups sharing a prefix of physical blocks: [read] 5.2.1 (samples of one
 * prompt share its blocks), [docs] Copy-on-Write (shared blocks, reference counts).
 *
 * Same result as pa_attention. The grouping only changes how the work is done: for group
 * g the first shared_len[g] positions are read once and multiplied against the queries of
 * all its members together (the members' query heads become one set of matrix rows), and
 * each member's remaining positions run on their own; the pieces are merged per request.
 *  seq_group     device int32 [num_seqs]: the request's group, or -1
 *  group_range   device int32 [num_groups, 2]: group g's members are the consecutive
 *                requests [group_range[2g], group_range[2g+1])
 *  shared_len    device int32 [num_groups]: positions [0, shared_len[g]) of every member
 *                are the same physical slots (same block ids in their tables); the library
 *                reads them through the first member's table
 * The kernel uses whole 16-token chunks below shared_len and every member's length, and
 * runs a group ungrouped when members x (num_heads / num_kv_heads) > 16 or it has fewer
 * than 2 members; a request whose seq_group does not match group_range runs ungrouped.
 * bf16 only (q, out, caches); head_dim 64 / 128; block size 8 or a multiple of 16;
 * num_heads / num_kv_heads <= 8. Workspace from pa_attention_grouped_workspace_size.
 * pa_bm_batch_groups builds the three arrays from the block manager's tables.
 * --------------------------------------------------------------------------- */
int pa_attention_grouped_workspace_size(int num_seqs, int num_groups, int num_heads, int num_kv_heads,
                                        int head_dim, size_t* bytes_out);

int pa_attention_grouped(void* out, const void* q, const void* k_cache, const void* v_cache,
                         const int32_t* block_table, int max_blocks_per_seq, const int32_t* seq_lens,
                         const int32_t* query_start_loc, int num_seqs, int num_tokens, int max_seq_len,
                         int num_heads, int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                         float scale, pa_dtype dtype, const int32_t* seq_group, const int32_t* group_range,
                         const int32_t* shared_len, int num_groups, void* workspace, size_t workspace_bytes,
                         pa_stream_t stream);

/* ------------------------------------------------------------------------------
 * FP8 KV cache -- [docs] quantisation support (FP8: 8-bit, 2x smaller than 16-bit storage).
 *
 * k_cache / v_cache hold one E4M3 code per element (PA_FP8_E4M3: 1 sign bit, 4 exponent
 * bits with bias 7, 3 mantissa bits, no infinities, largest finite 448), same layout as
 * above with 1-byte elements. A code c of the K (V) cache stands for value(c) * k_scale
 * (v_scale): one positive scale per cache, chosen by the caller (e.g. max |K| / 448).
 *
 * pa_kv_write_fp8: for every t with s = slot_mapping[t] >= 0,
 *     k_cache[s / B, s % B, :, :] = E4M3(k[t, :, :] / k_scale)      (same for v)
 * where x is widened to binary32, divided once (binary32, round to nearest even), then
 * rounded to E4M3 (nearest, ties to even; magnitudes beyond 448 saturate to 448).
 * k, v are [num_tokens, num_kv_heads, head_dim] in `in_dtype` (PA_BF16 or PA_F32).
 * num_kv_heads * head_dim must be a multiple of 16. Other rules as pa_kv_write.
 *
 * pa_attention_fp8: pa_attention over E4M3 caches with bf16 q and out: K and V are
 * read as value(code) * scale (exact in fp32 up to the scale product), the rest is
 * pa_attention's arithmetic. The split-K decode kernel reads the 1-byte cache directly
 * (half the bytes of bf16). Requests with q_len >= 2 run the tensor-core prefill kernel
 * when head_dim is 128 and the block size is 8, 16, 32, 64 or 128 (at most 4096 requests):
 * it converts each K/V tile of codes to f16 in shared memory (exact) and the pair's queries
 * from bf16 to f16, so q must lie within f16's range (|q| < 65520; magnitudes below 2^-24
 * become 0) and P is rounded to f16; other prefill shapes run the CUDA-core kernel.
 * Workspace from pa_attention_workspace_size. pa_copy_blocks takes PA_FP8_E4M3 caches
 * (byte copy), and pa_kv_write with dtype PA_FP8_E4M3 copies already-encoded rows.
 * --------------------------------------------------------------------------- */
int pa_kv_write_fp8(const void* k, const void* v, pa_dtype in_dtype, void* k_cache, void* v_cache,
                    const int64_t* slot_mapping, int64_t num_tokens, int64_t num_blocks, int block_size,
                    int num_kv_heads, int head_dim, float k_scale, float v_scale, pa_stream_t stream);

int pa_attention_fp8(void* out, const void* q, const void* k_cache, const void* v_cache,
                     const int32_t* block_table, int max_blocks_per_seq, const int32_t* seq_lens,
                     const int32_t* query_start_loc, int num_seqs, int num_tokens, int max_query_len,
                     int max_seq_len, int num_heads, int num_kv_heads, int head_dim, int block_size,
                     int64_t num_blocks, float scale, float k_scale, float v_scale, void* workspace,
                     size_t workspace_bytes, pa_stream_t stream);

/* ------------------------------------------------------------------------------
 * pa_swap_blocks -- [read] 6.2.1 (a preempted sequence group's KV blocks are swapped out
 * to the CPU, and swapped back in when GPU resources return); [intro] 4, scheduling flow,
 * swap phase (the swapped queue lives in CPU memory).
 *
 * For each i in [0, num_pairs): s = block_mapping[2i], d = block_mapping[2i+1]:
 *     dst_k[d] = src_k[s]; dst_v[d] = src_v[s]     (whole blocks, byte copy)
 * src_* pools have src_num_blocks blocks, dst_* pools dst_num_blocks, all with the block
 * geometry [block_size, num_kv_heads, head_dim] of `dtype` (PA_F32 / PA_BF16 /
 * PA_FP8_E4M3). Each pool may be device memory or pinned host memory (cudaHostAlloc or
 * cudaHostRegister'ed, used through its unified address): the kernel moves the blocks
 * over the CPU-GPU link itself, one launch per call. block_mapping: int64 [num_pairs, 2],
 * device or pinned host memory. No dst may repeat. Out-of-range ids are skipped and set
 * PA_DEVERR_BLOCK_RANGE. The pairs come from pa_bm_swap_out / pa_bm_swap_in. Every
 * pointer is checked with cudaPointerGetAttributes before the launch: another device's
 * memory, pageable host memory or host memory not mapped at its own address gives
 * PA_ERR_INVALID_ARG.
 * --------------------------------------------------------------------------- */
int pa_swap_blocks(const void* src_k, const void* src_v, void* dst_k, void* dst_v,
                   const int64_t* block_mapping, int64_t num_pairs, int64_t src_num_blocks,
                   int64_t dst_num_blocks, int block_size, int num_kv_heads, int head_dim,
                   pa_dtype dtype, pa_stream_t stream);

/* ------------------------------------------------------------------------------
 * pa_attention_fixed_scratch -- no counterpart in the pages: an addition for callers that
 * cannot allocate device memory, so cannot provide pa_attention's workspace. Examples: a
 * serving loop that reserved the GPU's free memory for its KV pool at start-up and must not
 * call cudaMalloc again (the call synchronises the device and fails once the pool owns the
 * memory); a plugin inside a host framework whose allocator it cannot reach; a binding from
 * a language with no device allocator.
 *
 * Same arguments and result as pa_attention, minus workspace / workspace_bytes, and with
 * every kernel on `stream` (no internal stream, so nothing is created). The split-K
 * scratch is instead a fixed 16 MiB array inside the library, which every GPU that loads
 * the library holds until the process exits. Allocates nothing (no cudaMalloc / cudaFree,
 * no allocating library call).
 *  - Limit: returns PA_ERR_WORKSPACE, enqueuing nothing, when the batch needs more scratch
 *    than 16 MiB (pa_attention_workspace_size gives the need; e.g. up to ~850 requests of
 *    32 query / 8 KV heads at head_dim 128 on a 152-SM GPU).
 *  - The first call on each device looks up the array's device address (once, with that
 *    device current); make that first call before any stream capture.
 *  - All calls on a device share the one array, which keeps the last call's contents; no
 *    part of it needs to start at zero. Calls whose work may overlap on the GPU (different
 *    streams without ordering between them) race on it and give wrong results: order them.
 * --------------------------------------------------------------------------- */
int pa_attention_fixed_scratch(void* out, const void* q, const void* k_cache, const void* v_cache,
                               const int32_t* block_table, int max_blocks_per_seq,
                               const int32_t* seq_lens, const int32_t* query_start_loc,
                               int num_seqs, int num_tokens, int max_query_len, int max_seq_len,
                               int num_heads, int num_kv_heads, int head_dim, int block_size,
                               int64_t num_blocks, float scale, pa_dtype dtype,
                               pa_stream_t stream);

/* ------------------------------------------------------------------------------
 * Host block manager -- [docs] PagedAttention algorithm flow and Copy-on-Write
 * (reference counting); [read] 5.1.1 and 5.2.1; [flow] 3.3 (pool of blocks, slots).
 *
 * Free blocks are handed out first-in first-out, starting from `free_order` (a
 * permutation of [0, num_blocks)); a released block rejoins the tail (the free list is
 * doubly linked so that prefix caching, below, can take a released block back out). Appending a
 * token takes a new block only when the sequence's last block is full (or it has none),
 * so a sequence of n tokens holds ceil(n / block_size) blocks. Writing into a last
 * block whose reference count is > 1 first moves the writer to a fresh block and
 * records a (src, dst) copy pair; the old block's count drops by 1. An append that
 * cannot be satisfied changes nothing. Not thread-safe: one manager per thread.
 * All arrays are host memory.
 * --------------------------------------------------------------------------- */
typedef struct pa_bm pa_bm;

/* NULL on invalid arguments (free_order not a permutation, sizes < 1) or no memory. */
pa_bm* pa_bm_create(int64_t num_blocks, int block_size, const int32_t* free_order);
void pa_bm_destroy(pa_bm* bm);

int pa_bm_add_seq(pa_bm* bm, int64_t seq);               /* PA_ERR_NOT_FOUND if id in use */
/* Appends n >= 0 tokens; writes their n slots to slots_out (may be NULL when n == 0).
 * PA_ERR_NO_BLOCKS: the free queue is too short now; PA_ERR_TOO_LARGE: the sequence
 * would need more blocks than the pool has. */
int pa_bm_append(pa_bm* bm, int64_t seq, int64_t n, int64_t* slots_out);
/* Batched append: for i in [0, n), appends counts[i] >= 0 tokens to seqs[i], in order, writing
 * all slots concatenated to slots_out (capacity >= sum of counts). Stops at the first append
 * that fails and returns its status; *done_out (if not NULL) gets the number of entries fully
 * applied, so those appends stay and the rest are not attempted. */
int pa_bm_append_batch(pa_bm* bm, const int64_t* seqs, const int64_t* counts, int64_t n,
                       int64_t* slots_out, int64_t* done_out);
int pa_bm_fork(pa_bm* bm, int64_t parent, int64_t child); /* child shares parent's blocks */
int pa_bm_free_seq(pa_bm* bm, int64_t seq);               /* counts - 1, release at 0 */
int64_t pa_bm_seq_len(const pa_bm* bm, int64_t seq);      /* -1 if unknown */
int64_t pa_bm_num_seq_blocks(const pa_bm* bm, int64_t seq);/* -1 if unknown */
int pa_bm_ref_count(const pa_bm* bm, int64_t block);      /* -1 if out of range */
int64_t pa_bm_num_free(const pa_bm* bm);
/* Copies the free queue, head first, into out (capacity >= pa_bm_num_free). */
int pa_bm_free_queue(const pa_bm* bm, int32_t* out, int64_t capacity);
/* Copies seq's block table (logical order) into out (capacity >= its block count). */
int pa_bm_block_table(const pa_bm* bm, int64_t seq, int32_t* out, int64_t capacity);
/* Fills a batch's metadata: row i of table_out [n, width] gets seqs[i]'s block table
 * (unused entries 0) and seq_lens_out[i] its length. PA_ERR_INVALID_ARG if a table is
 * wider than `width`. */
int pa_bm_batch_tables(const pa_bm* bm, const int64_t* seqs, int64_t n, int32_t* table_out,
                       int64_t width, int32_t* seq_lens_out);
int64_t pa_bm_num_pending_copies(const pa_bm* bm);
/* Moves up to `capacity` pending (src, dst) pairs, oldest first, into pairs_out
 * [capacity, 2]; returns how many were moved (or -1 on a bad argument). */
int64_t pa_bm_take_copies(pa_bm* bm, int64_t* pairs_out, int64_t capacity);

/* ------------------------------------------------------------------------------
 * Prefix caching -- [docs] Copy-on-Write › shared-prefix detection (hash a prompt's
 * prefix; if its KV is cached, reuse it and raise the blocks' reference counts) and
 * Prefix Caching › mechanism (look up on arrival; a hit reuses the KV and skips that
 * prefill, a miss computes and caches it); [flow] 3.3 (blocks on a doubly linked list,
 * evicted least recently used first).
 *
 * Once enabled, a full block is keyed by its whole token prefix (all token ids of its
 * sequence up to its last slot; a 128-bit hash chain encodes it). A block is registered
 * when its last slot is written, unless its key is registered already (the first block
 * stays registered). A released block keeps its registration at the tail of the free
 * list; the free list hands blocks out from its head, and a registered block handed out
 * loses its registration (eviction, least recently released first). Cached blocks are
 * full, so nothing ever writes into them while they are shared.
 * --------------------------------------------------------------------------- */
/* Turns prefix caching on; only on a fresh manager (no sequence yet). From then on appends
 * need token ids: pa_bm_append / pa_bm_append_batch return PA_ERR_INVALID_ARG. */
int pa_bm_enable_prefix_caching(pa_bm* bm);
/* Starts sequence `seq` from the longest cached prefix of prompt[0, n): whole blocks, walked
 * from the start until the first miss, covering at most max_hit tokens (pass n - 1 so the
 * last prompt token is always computed). The reused blocks' counts go up (a released one
 * leaves the free list). *hit_out = tokens reused (a multiple of block_size); the caller
 * appends prompt[*hit_out, n) next and computes only those rows. */
int pa_bm_add_seq_cached(pa_bm* bm, int64_t seq, const int32_t* prompt, int64_t n, int64_t max_hit,
                         int64_t* hit_out);
/* pa_bm_append with the appended tokens' ids (token_ids[n]; ignored without caching). */
int pa_bm_append_tokens(pa_bm* bm, int64_t seq, const int32_t* token_ids, int64_t n, int64_t* slots_out);
/* pa_bm_append_batch with token ids, concatenated like the slots. */
int pa_bm_append_tokens_batch(pa_bm* bm, const int64_t* seqs, const int64_t* counts, int64_t n,
                              const int32_t* token_ids, int64_t* slots_out, int64_t* done_out);
/* Registered blocks now, blocks reused by lookups so far, registrations evicted so far. */
int pa_bm_prefix_stats(const pa_bm* bm, int64_t* cached_blocks, int64_t* hit_blocks, int64_t* evictions);

/* Groups for pa_attention_grouped over the batch seqs[0, n) (in batch order): runs of
 * consecutive sequences whose block tables start with the same block id, at most
 * max_members each, become groups; shared_len = the number of leading table entries all
 * members have in common x block_size, capped by the shortest member. Writes
 * seq_group_out[n] (-1 outside groups), group_range_out[2 * groups] and
 * shared_len_out[groups] (capacity >= n / 2 groups is always enough) and *num_groups_out. */
int pa_bm_batch_groups(const pa_bm* bm, const int64_t* seqs, int64_t n, int max_members, int32_t* seq_group_out,
                       int32_t* group_range_out, int32_t* shared_len_out, int64_t capacity,
                       int64_t* num_groups_out);

/* ------------------------------------------------------------------------------
 * Swapping -- [read] 6.2.1 SequenceGroup (preempted groups are swapped out to the CPU and
 * swapped back in later); [intro] 4, scheduling flow, swap phase (swapped queue in CPU
 * memory).
 *
 * A CPU pool of num_cpu_blocks blocks with its own FIFO free queue (initial order
 * cpu_free_order) and reference counts. pa_bm_swap_out moves a group of sequences to the
 * CPU: each distinct block of their tables (first met walking seqs in order, each table
 * from its first block) gets one CPU block whose count is the number of group members
 * holding it; the GPU block's count drops by that number and it is released at 0 (a block
 * still held outside the group stays). The (gpu, cpu) pairs to copy go to pairs_out
 * [capacity, 2] and their number to *num_pairs_out; run pa_swap_blocks with them before
 * the released GPU blocks are written again. pa_bm_swap_in is the reverse (new GPU
 * blocks from the free list, (cpu, gpu) pairs; copy them before reading the sequences).
 * Either returns PA_ERR_NO_BLOCKS (changing nothing) when the other pool is short,
 * PA_ERR_INVALID_ARG when capacity is below the number of pairs, a sequence repeats or is
 * already on the other side. A swapped sequence takes no append or fork and cannot be in
 * pa_bm_batch_tables; pa_bm_free_seq releases its CPU blocks.
 * --------------------------------------------------------------------------- */
int pa_bm_enable_swap(pa_bm* bm, int64_t num_cpu_blocks, const int32_t* cpu_free_order);
int pa_bm_swap_out(pa_bm* bm, const int64_t* seqs, int64_t n, int64_t* pairs_out, int64_t capacity,
                   int64_t* num_pairs_out);
int pa_bm_swap_in(pa_bm* bm, const int64_t* seqs, int64_t n, int64_t* pairs_out, int64_t capacity,
                  int64_t* num_pairs_out);
int pa_bm_is_swapped(const pa_bm* bm, int64_t seq);        /* 1, 0, or -1 if unknown */
int64_t pa_bm_num_free_cpu(const pa_bm* bm);               /* -1 without swapping */
int pa_bm_cpu_ref_count(const pa_bm* bm, int64_t block);  /* -1 if out of range */

#ifdef __cplusplus
}
#endif

#endif /* PA_H_ */
