// Shared by the split-K decode kernels (decode_attention.cu: CUDA-core consumers;
// decode_mma.cu: tensor-core consumers): the work unit, the stage descriptor, the
// kernel parameters, the per-CTA plan over the balanced unit partition, and the merge
// kernel that combines the pieces of requests cut between CTAs.
#pragma once

#include <float.h>

#include "common.cuh"
#include "launch.h"

namespace pa {
namespace {
constexpr int kTPS = 16;    // tokens per stage
constexpr int kSmemLimit = 227 * 1024;

enum : int { kFirst = 1, kLast = 2, kSeqStart = 4, kSeqEnd = 8, kBad = 16 };

struct __align__(16) StageDesc {
  int s, hg, j, valid, flags, pad;
  int64_t wslot;  // >= 0: row valid - 1 came from the new token's K/V; store it to this slot
};

struct DecodeParams {
  void* out;
  const void* q;
  const char* k_cache;
  const char* v_cache;
  char* k_cache_w;  // the same caches, for the fused write of new tokens
  char* v_cache_w;
  const char* k_new;  // fused write inputs (null: no write); [num_tokens, Hkv, D]
  const char* v_new;
  const int64_t* slot_mapping;
  const int32_t* block_table;
  const int32_t* seq_lens;
  const int32_t* qsl;
  float* ws_o;
  float* ws_lse;
  int4* ws_meta;  // per (head group, request): first CTA (-1: nothing to merge), last CTA,
                  // units per head group, output row
  unsigned int* err;
  int64_t num_blocks;
  int max_blocks_per_seq;
  int num_seqs;
  int num_heads;
  int num_kv_heads;
  int block_size;
  int hg_size;  // KV heads per CTA (HG)
  int num_hg;   // num_kv_heads / HG
  int group;    // query heads per KV head
  int qg;       // consumer warps per KV head = group / (query heads per warp)
  int num_ctas; // grid of the split-K kernel
  float scale_log2;  // softmax scale * log2(e) (* k_scale for E4M3 caches)
  float v_scale;     // 1, or the E4M3 V scale
  // Shared-prefix groups (tensor-core kernel; num_groups = 0: none): request s belongs to
  // group seq_group[s] (or -1); group g's members are requests [group_start[2g],
  // group_start[2g+1]) and their first shared_len[g] positions are the same physical slots.
  const int32_t* seq_group;
  const int32_t* group_start;
  const int32_t* shared_len;
  int num_groups;
  int rmax;  // workspace rows per KV head of a piece: G, or 16 with groups
  // tensor-core kernel without groups: bytes of a query slot in shared memory (the head
  // group's query rows, and the new K / V rows of a fused write), filled by the producer's
  // bulk copies; 0: consumers read the queries from global memory
  int q_slot;
};

// Keys of request s if it is a decode request (q_len == 1), else 0.
__device__ __forceinline__ int decode_len(const DecodeParams& p, int s) {
  const int q_len = __ldg(p.qsl + s + 1) - __ldg(p.qsl + s);
  if (q_len != 1) return 0;
  int L = __ldg(p.seq_lens + s);
  const int cap = p.max_blocks_per_seq * p.block_size;
  if (L > cap) {
    raise_error(p.err, PA_DEVERR_SEQ_RANGE);
    L = cap;
  }
  return L > 0 ? L : 0;
}

__device__ __forceinline__ int units_of(int L) { return (L + kTPS - 1) / kTPS; }

// ---------------------------------------------------------------- block-wide helpers
__device__ __forceinline__ int warp_sum_i(int x) {
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) x += __shfl_xor_sync(0xffffffffu, x, m);
  return x;
}

// Sum over the block; `red` holds >= 33 ints of shared memory.
__device__ int block_sum(int x, int* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  x = warp_sum_i(x);
  if (lane == 0) red[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int y = lane < nw ? red[lane] : 0;
    y = warp_sum_i(y);
    if (lane == 0) red[32] = y;
  }
  __syncthreads();
  const int r = red[32];
  __syncthreads();
  return r;
}

// Exclusive prefix over the block (thread order); returns it and the block total.
__device__ int block_exclusive_scan(int x, int* red, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int inc = x;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, inc, d);
    if (lane >= d) inc += y;
  }
  if (lane == 31) red[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    const int w = lane < nw ? red[lane] : 0;
    int wi = w;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, wi, d);
      if (lane >= d) wi += y;
    }
    if (lane < nw) red[lane] = wi - w;  // exclusive warp offsets
    if (lane == 31) red[32] = wi;
  }
  __syncthreads();
  const int r = red[warp] + inc - x;
  *total = red[32];
  __syncthreads();
  return r;
}

// ---------------------------------------------------------------- the CTA's range of units
struct Plan {
  int64_t u_begin, u_end;  // this CTA's units [u_begin, u_end) of the request-major numbering
  int start_s, start_hg, start_j;
  int units_per_hg;
};

// Every CTA computes the same numbering: units of (request, head group, 16 positions),
// request-major, split into gridDim.x equal contiguous ranges. CTA 0 also marks the
// requests no CTA touches for the merge kernel and zeroes the output of a decode query
// without keys. Returns false when this CTA's range is empty. `red` holds >= 36 ints.
template <typename T, int D>
__device__ bool plan_range(const DecodeParams& p, int* red, Plan& pl) {
  const int S = p.num_seqs;
  int my_units = 0;
  for (int s = threadIdx.x; s < S; s += blockDim.x) my_units += units_of(decode_len(p, s));
  pl.units_per_hg = block_sum(my_units, red);
  const int64_t U = int64_t(pl.units_per_hg) * p.num_hg;
  const int64_t c = blockIdx.x, C_ = gridDim.x;
  if (c == 0) {
    for (int s = threadIdx.x; s < S; s += blockDim.x) {
      if (units_of(decode_len(p, s)) > 0) continue;
      for (int hg = 0; hg < p.num_hg; ++hg) p.ws_meta[int64_t(s) * p.num_hg + hg] = make_int4(-1, -1, 0, 0);
      const int q0 = __ldg(p.qsl + s);
      if (__ldg(p.qsl + s + 1) - q0 == 1) {
        raise_error(p.err, PA_DEVERR_SEQ_RANGE);
        T* o = reinterpret_cast<T*>(p.out) + int64_t(q0) * p.num_heads * D;
        for (int i = 0; i < p.num_heads * D; ++i) o[i] = T(0.f);
      }
    }
  }
  pl.u_begin = c * U / C_;
  pl.u_end = (c + 1) * U / C_;
  if (pl.u_begin >= pl.u_end) return false;
  const int64_t rem = pl.u_begin;
  int64_t run = 0;
  for (int base = 0; base < S; base += blockDim.x) {
    const int s = base + threadIdx.x;
    const int us = s < S ? units_of(decode_len(p, s)) * p.num_hg : 0;
    int total;
    const int ex = block_exclusive_scan(us, red, &total);
    if (us > 0 && run + ex <= rem && rem < run + ex + us) {
      red[34] = s;
      red[35] = int(rem - (run + ex));
    }
    __syncthreads();
    run += total;
    if (run > rem) break;
  }
  pl.start_s = red[34];
  const int start_us = units_of(decode_len(p, pl.start_s));
  pl.start_hg = red[35] / start_us;
  pl.start_j = red[35] % start_us;
  return true;
}
// ---------------------------------------------------------------- register tile helpers
template <typename T, int VEC>
struct RowVec;

// VEC elements of a row -> fp32, from shared or global memory.
template <int VEC>
struct RowVec<__nv_bfloat16, VEC> {
  static_assert(VEC == 4 || VEC == 8, "bf16 rows move 8 or 16 bytes per lane");
  static __device__ __forceinline__ void load(const __nv_bfloat16* p, float* f) {
    if constexpr (VEC == 8) {
      Elem<__nv_bfloat16>::unpack(*reinterpret_cast<const uint4*>(p), f);
    } else {
      const uint2 u = *reinterpret_cast<const uint2*>(p);
      f[0] = __uint_as_float(u.x << 16);
      f[1] = __uint_as_float(u.x & 0xffff0000u);
      f[2] = __uint_as_float(u.y << 16);
      f[3] = __uint_as_float(u.y & 0xffff0000u);
    }
  }
  static __device__ __forceinline__ void store(__nv_bfloat16* p, const float* f) {
    uint32_t w[VEC / 2];
#pragma unroll
    for (int i = 0; i < VEC / 2; ++i) {
      __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
      w[i] = *reinterpret_cast<uint32_t*>(&h);
    }
    if constexpr (VEC == 8)
      *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
    else
      *reinterpret_cast<uint2*>(p) = make_uint2(w[0], w[1]);
  }
};

// FP8 E4M3 rows: 8 codes (8 bytes) per lane -> fp32, exact.
template <int VEC>
struct RowVec<Fp8E4M3, VEC> {
  static_assert(VEC == 8, "E4M3 rows move 8 bytes per lane");
  static __device__ __forceinline__ void load(const Fp8E4M3* p, float* f) {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    const float2 a = fp8x2_to_float2(u.x & 0xffffu), b = fp8x2_to_float2(u.x >> 16);
    const float2 c = fp8x2_to_float2(u.y & 0xffffu), d = fp8x2_to_float2(u.y >> 16);
    f[0] = a.x, f[1] = a.y, f[2] = b.x, f[3] = b.y, f[4] = c.x, f[5] = c.y, f[6] = d.x, f[7] = d.y;
  }
};

template <int VEC>
struct RowVec<float, VEC> {
  static_assert(VEC == 4, "fp32 rows move 16 bytes per lane");
  static __device__ __forceinline__ void load(const float* p, float* f) {
    const float4 u = *reinterpret_cast<const float4*>(p);
    f[0] = u.x;
    f[1] = u.y;
    f[2] = u.z;
    f[3] = u.w;
  }
  static __device__ __forceinline__ void store(float* p, const float* f) {
    *reinterpret_cast<float4*>(p) = make_float4(f[0], f[1], f[2], f[3]);
  }
};

template <int G>
__device__ __forceinline__ float pick(const float (&a)[G], int g) {
  float r = a[0];
#pragma unroll
  for (int i = 1; i < G; ++i) r = (g == i) ? a[i] : r;
  return r;
}
// ---------------------------------------------------------------- merge of the pieces
// One CTA per (head group, request). It reads the request's descriptor written by the
// split-K kernel and leaves at once unless the request was cut into pieces; then warp w
// merges heads w, w + nwarps, ...: lane i reads piece i's log-sum-exp (32 pieces at a
// time) for the max and the weights, which reach the other lanes by shuffles, and each
// lane accumulates its 4 dims over the pieces four at a time, their loads issued together.
template <typename T, int D>
__global__ void __launch_bounds__(1024) decode_merge_kernel(const __grid_constant__ DecodeParams p, int group) {
  griddep_launch_dependents();  // the next kernel may be scheduled; it still waits for this grid
  griddep_wait();  // the split-K grid's pieces and descriptors must be complete and visible
  const int v = blockIdx.x;
  const int hg = v % p.num_hg;
  const int4 meta = p.ws_meta[v];
  if (meta.x < 0 || meta.x == meta.y) return;  // nothing to merge / one CTA wrote `out` itself
  if (meta.y >= p.num_ctas || meta.x > meta.y || meta.z <= 0) {
    // only if the split-K kernel gave up early: leave `out` alone, report it
    if (threadIdx.x == 0) raise_error(p.err, PA_DEVERR_TIMEOUT);
    return;
  }
  const int HGG = p.hg_size * group;
  const int qrow = meta.w;
  T* out = reinterpret_cast<T*>(p.out);
  constexpr int D4 = D / 4;
  // CTAs whose range is empty (fewer units than CTAs) left no piece: weight 0, not read.
  const int64_t U = int64_t(meta.z) * p.num_hg, C = p.num_ctas;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
  const int npieces = meta.y - meta.x + 1;
  auto lse_of = [&](int i, int head) {  // piece i's log-sum-exp, -inf for an empty range
    const int64_t cc = meta.x + i;
    return (cc * U / C != (cc + 1) * U / C) ? p.ws_lse[(cc + v) * HGG + head] : -INFINITY;
  };
  for (int head = warp; head < HGG; head += nwarps) {
    float l0 = lane < npieces ? lse_of(lane, head) : -INFINITY;  // pieces 0..31, kept
    float M = l0;
    for (int i = 32 + lane; i < npieces; i += 32) M = fmaxf(M, lse_of(i, head));
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, m));
    const float Ms = (M == -INFINITY) ? 0.f : M;
    float a[4] = {0.f, 0.f, 0.f, 0.f}, wsum = 0.f;
    for (int i0 = 0; i0 < npieces; i0 += 32) {
      const float lw = (i0 == 0) ? l0 : (i0 + lane < npieces ? lse_of(i0 + lane, head) : -INFINITY);
      const float wl = exp2f(lw - Ms);  // 0 for an empty range or an empty piece
      const int n = min(32, npieces - i0);
      for (int b = 0; b < n; b += 4) {
        float w[4];
        float4 o[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          w[q] = __shfl_sync(0xffffffffu, wl, b + q);
          if (b + q >= n) w[q] = 0.f;
          o[q] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (lane < D4 && w[q] > 0.f)
            o[q] = *reinterpret_cast<const float4*>(p.ws_o + ((meta.x + i0 + b + q + v) * HGG + head) * D + lane * 4);
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          a[0] += w[q] * o[q].x;
          a[1] += w[q] * o[q].y;
          a[2] += w[q] * o[q].z;
          a[3] += w[q] * o[q].w;
          wsum += w[q];
        }
      }
    }
    if (lane < D4) {
      const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) a[e] *= inv;
      RowVec<T, 4>::store(out + (int64_t(qrow) * p.num_heads + hg * HGG + head) * D + lane * 4, a);
    }
  }
}

// ---------------------------------------------------------------- host side
// Parameters shared by both split-K kernels; hg KV heads per CTA, qg consumer warps per KV
// head. The workspace layout (per-CTA-slot partials, log-sum-exps, per-request
// descriptors) depends only on num_ctas, num_seqs, hg and G.
inline DecodeParams fill_decode_params(const AttnArgs& a, int hg, int qg, int num_ctas, int D) {
  const int G = a.num_heads / a.num_kv_heads;
  DecodeParams p;
  p.out = a.out;
  p.q = a.q;
  p.k_cache = static_cast<const char*>(a.k_cache);
  p.v_cache = static_cast<const char*>(a.v_cache);
  p.k_cache_w = static_cast<char*>(const_cast<void*>(a.k_cache));
  p.v_cache_w = static_cast<char*>(const_cast<void*>(a.v_cache));
  p.k_new = nullptr;
  p.v_new = nullptr;
  p.slot_mapping = nullptr;
  p.block_table = a.block_table;
  p.seq_lens = a.seq_lens;
  p.qsl = a.query_start_loc;
  const int num_hg = a.num_kv_heads / hg;
  const int64_t slots = int64_t(num_ctas) + int64_t(a.num_seqs) * num_hg;
  const int64_t HGG = int64_t(hg) * G;
  char* ws = static_cast<char*>(a.workspace);
  p.ws_o = reinterpret_cast<float*>(ws);
  p.ws_lse = reinterpret_cast<float*>(ws + slots * HGG * D * 4);
  p.ws_meta = reinterpret_cast<int4*>(ws + slots * HGG * D * 4 + ((slots * HGG * 4 + 15) / 16) * 16);
  p.err = a.err;
  p.num_blocks = a.num_blocks;
  p.max_blocks_per_seq = a.max_blocks_per_seq;
  p.num_seqs = a.num_seqs;
  p.num_heads = a.num_heads;
  p.num_kv_heads = a.num_kv_heads;
  p.block_size = a.block_size;
  p.hg_size = hg;
  p.num_hg = num_hg;
  p.group = G;
  p.qg = qg;
  p.num_ctas = num_ctas;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.v_scale = 1.f;
  p.seq_group = nullptr;
  p.group_start = nullptr;
  p.shared_len = nullptr;
  p.num_groups = 0;
  p.rmax = G;
  p.q_slot = 0;
  return p;
}

// The merge of the pieces, after the split-K grid: by programmatic dependent launch, or
// (pdl false) in plain stream order, so that its CTAs take no SM while the split-K grid
// runs (a prefill grid on another stream is then filling the SMs the split-K grid leaves).
template <typename T, int D>
cudaError_t launch_merge(const DecodeParams& p, cudaStream_t stream, bool pdl) {
  const int64_t HGG = int64_t(p.hg_size) * p.group;
  const int merge_threads = 32 * (HGG < 32 ? int(HGG) : 32);
  const dim3 grid(unsigned(int64_t(p.num_seqs) * p.num_hg));
  if (!pdl) {
    decode_merge_kernel<T, D><<<grid, dim3(merge_threads), 0, stream>>>(p, p.group);
    return cudaGetLastError();
  }
  return launch_pdl(decode_merge_kernel<T, D>, grid, dim3(merge_threads), 0, stream, p, p.group);
}

}  // namespace
}  // namespace pa
