// Chunked-prefill attention (requests with q_len >= 2), CUDA-core tile kernel.
//
// What it computes: vLLM 0.10.0 flow page, 3.2 Scheduler (a long prefill is cut into
// chunks that run in the same batch as decodes) and 3.5 Attention (requests delimited
// by query_start_loc, K/V found through block_table); VLLM overview page, 2.1 (causal:
// each token sees only itself and earlier tokens). Query j of a request with q_len
// queries and L keys sits at position L - q_len + j (the chunk's own K/V are already
// in the cache) and sees keys 0..L - q_len + j.
//
// One CTA per (request, KV head, tile of 64 / G queries): its rows are the tile's queries for the
// G query heads that share the KV head, so each K/V tile is read once per KV head.
// K/V tiles of 16 positions are gathered through the block table into shared memory as
// fp32; S = Q.K^T, online softmax and O += P.V run on fp32 CUDA cores.
#include "common.cuh"
#include "launch.h"

namespace pa {
namespace {

constexpr int kRows = 64;  // tile rows = queries per tile x G
constexpr int kKT = 16;    // keys per tile
constexpr int kThreads = 256;

template <int D>
constexpr size_t simple_smem_bytes() {
  return size_t(kRows) * D * 4 + size_t(kKT) * (D + 1) * 4 + size_t(kKT) * D * 4 + size_t(kRows) * kKT * 4;
}

// T: q / out element type; KV: cache element type (T, or Fp8E4M3 with bf16 T).
template <typename T, int D, int G, typename KV>
__global__ void __launch_bounds__(kThreads) prefill_simple_kernel(const __grid_constant__ AttnArgs a) {
  constexpr int kQT = kRows / G;       // queries per tile
  constexpr int R = kRows;             // rows of the tile
  constexpr int TPR = kThreads / R;     // threads per row
  static_assert(TPR >= 1 && kKT % TPR == 0 && D % TPR == 0, "tile mapping");
  constexpr int KPT = kKT / TPR;        // keys per thread in S
  constexpr int DPT = D / TPR;          // output dims per thread
  constexpr int EL = sizeof(T);
  constexpr int VEC = 16 / EL;
  constexpr int KVEC = 16 / int(sizeof(KV));  // cache elements per 16-byte load

  const int s = blockIdx.x, hk = blockIdx.y;
  const int q0 = blockIdx.z * kQT;
  const int qs = __ldg(a.query_start_loc + s);
  const int q_len = __ldg(a.query_start_loc + s + 1) - qs;
  if (q_len < 2 || q0 >= q_len) return;
  int L = __ldg(a.seq_lens + s);
  const int cap = a.max_blocks_per_seq * a.block_size;
  if (L > cap || q_len > L) {
    if (threadIdx.x == 0 && hk == 0 && blockIdx.z == 0) raise_error(a.err, PA_DEVERR_SEQ_RANGE);
    if (L > cap) L = cap;
    if (q_len > L) return;
  }
  const int nq = min(kQT, q_len - q0);
  const int pos0 = L - q_len + q0;  // position of the tile's first query
  const int Hq = a.num_heads, Hkv = a.num_kv_heads, B = a.block_size;

  extern __shared__ __align__(16) float smem_f[];
  float(*Qs)[D] = reinterpret_cast<float(*)[D]>(smem_f);
  float(*Ks)[D + 1] = reinterpret_cast<float(*)[D + 1]>(smem_f + R * D);
  float(*Vs)[D] = reinterpret_cast<float(*)[D]>(smem_f + R * D + kKT * (D + 1));
  float(*Ps)[kKT] = reinterpret_cast<float(*)[kKT]>(smem_f + R * D + kKT * (D + 1) + kKT * D);

  const float scale_log2 = a.scale * 1.4426950408889634f;
  const T* q = static_cast<const T*>(a.q);
  // rows: r = qi * G + g
  for (int i = threadIdx.x; i < R * (D / VEC); i += kThreads) {
    const int rr = i / (D / VEC), d0 = (i % (D / VEC)) * VEC;
    const int qi = rr / G, g = rr % G;
    float f[VEC];
    if (qi < nq) {
      const uint4 u = *reinterpret_cast<const uint4*>(q + (int64_t(qs + q0 + qi) * Hq + hk * G + g) * D + d0);
      Elem<T>::unpack(u, f);
    } else {
#pragma unroll
      for (int e = 0; e < VEC; ++e) f[e] = 0.f;
    }
#pragma unroll
    for (int e = 0; e < VEC; ++e) Qs[rr][d0 + e] = f[e] * scale_log2;
  }

  const int row = threadIdx.x / TPR, sub = threadIdx.x % TPR;
  const int my_pos = pos0 + row / G;
  float o[DPT];
#pragma unroll
  for (int e = 0; e < DPT; ++e) o[e] = 0.f;
  float m = -INFINITY, l = 0.f;

  const int last_key = pos0 + nq - 1;  // highest position any row of the tile sees
  const int32_t* bt = a.block_table + int64_t(s) * a.max_blocks_per_seq;
  const KV* kc = static_cast<const KV*>(a.k_cache);
  const KV* vc = static_cast<const KV*>(a.v_cache);
  for (int k0 = 0; k0 <= last_key; k0 += kKT) {
    __syncthreads();  // previous tile fully used
    for (int i = threadIdx.x; i < kKT * (D / KVEC); i += kThreads) {
      const int t = i / (D / KVEC), d0 = (i % (D / KVEC)) * KVEC;
      const int kp = k0 + t;
      float kf[KVEC], vf[KVEC];
      bool ok = kp <= last_key;
      int64_t blk = 0;
      if (ok) {
        blk = __ldg(bt + kp / B);
        if (blk < 0 || blk >= a.num_blocks) {
          raise_error(a.err, PA_DEVERR_BLOCK_RANGE);
          ok = false;
        }
      }
      if (ok) {
        const int64_t off = ((blk * B + kp % B) * Hkv + hk) * D + d0;
        Elem<KV>::unpack(*reinterpret_cast<const uint4*>(kc + off), kf);
        Elem<KV>::unpack(*reinterpret_cast<const uint4*>(vc + off), vf);
        if constexpr (sizeof(KV) == 1) {  // E4M3 codes -> values
#pragma unroll
          for (int e = 0; e < KVEC; ++e) {
            kf[e] *= a.k_scale;
            vf[e] *= a.v_scale;
          }
        }
      } else {
#pragma unroll
        for (int e = 0; e < KVEC; ++e) kf[e] = vf[e] = 0.f;
      }
#pragma unroll
      for (int e = 0; e < KVEC; ++e) {
        Ks[t][d0 + e] = kf[e];
        Vs[t][d0 + e] = vf[e];
      }
    }
    __syncthreads();
    // S for this thread's keys
    float sc[KPT];
    float mt = -INFINITY;
#pragma unroll
    for (int kk = 0; kk < KPT; ++kk) {
      const int t = sub * KPT + kk;
      float acc = 0.f;
#pragma unroll 8
      for (int d = 0; d < D; ++d) acc = fmaf(Qs[row][d], Ks[t][d], acc);
      sc[kk] = (k0 + t <= my_pos) ? acc : -INFINITY;
      mt = fmaxf(mt, sc[kk]);
    }
#pragma unroll
    for (int msk = 1; msk < TPR; msk <<= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, msk));
    const float mn = fmaxf(m, mt);
    const float ms = (mn == -INFINITY) ? 0.f : mn;
    const float alpha = exp2f(m - ms);
    float ls = 0.f;
#pragma unroll
    for (int kk = 0; kk < KPT; ++kk) {
      const float pv = exp2f(sc[kk] - ms);
      Ps[row][sub * KPT + kk] = pv;
      ls += pv;
    }
#pragma unroll
    for (int msk = 1; msk < TPR; msk <<= 1) ls += __shfl_xor_sync(0xffffffffu, ls, msk);
    l = l * alpha + ls;
    m = mn;
    __syncwarp();
#pragma unroll
    for (int e = 0; e < DPT; ++e) o[e] *= alpha;
#pragma unroll
    for (int t = 0; t < kKT; ++t) {
      const float pv = Ps[row][t];
#pragma unroll
      for (int e = 0; e < DPT; ++e) o[e] = fmaf(pv, Vs[t][sub * DPT + e], o[e]);
    }
  }
  if (row / G < nq) {
    const float inv = l > 0.f ? 1.f / l : 0.f;
    T* out = static_cast<T*>(a.out) + (int64_t(qs + q0 + row / G) * Hq + hk * G + row % G) * D + sub * DPT;
#pragma unroll
    for (int e = 0; e < DPT; e += VEC) {
      float f[VEC];
#pragma unroll
      for (int x = 0; x < VEC; ++x) f[x] = o[e + x] * inv;
      *reinterpret_cast<uint4*>(out + e) = Elem<T>::pack(f);
    }
  }
}

template <typename T, int D, int G, typename KV>
cudaError_t run(const AttnArgs& a, cudaStream_t stream) {
  constexpr int kQT = kRows / G;
  const size_t smem = simple_smem_bytes<D>();
  auto kern = prefill_simple_kernel<T, D, G, KV>;
  cudaError_t e = ensure_smem<prefill_simple_kernel<T, D, G, KV>>(smem);
  if (e != cudaSuccess) return e;
  dim3 grid(a.num_seqs, a.num_kv_heads, (a.max_query_len + kQT - 1) / kQT);
  kern<<<grid, kThreads, smem, stream>>>(a);
  return cudaGetLastError();
}

template <typename T, int D, typename KV = T>
cudaError_t run_g(const AttnArgs& a, int G, cudaStream_t stream) {
  switch (G) {
    case 1: return run<T, D, 1, KV>(a, stream);
    case 2: return run<T, D, 2, KV>(a, stream);
    case 4: return run<T, D, 4, KV>(a, stream);
    case 8: return run<T, D, 8, KV>(a, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

bool prefill_supported(pa_dtype dtype, int head_dim, int group) {
  if (head_dim != 64 && head_dim != 128) return false;
  if (group != 1 && group != 2 && group != 4 && group != 8) return false;
  return dtype == PA_F32 || dtype == PA_BF16;
}

cudaError_t launch_prefill(const AttnArgs& a, cudaStream_t stream) {
  if (a.max_query_len < 2 || a.num_seqs == 0) return cudaSuccess;
  const int G = a.num_heads / a.num_kv_heads;
  if (a.cache_dtype == PA_FP8_E4M3) {  // E4M3 caches: bf16 q and out only
    if (a.dtype != PA_BF16) return cudaErrorInvalidValue;
    if (a.head_dim == 64) return run_g<__nv_bfloat16, 64, Fp8E4M3>(a, G, stream);
    return run_g<__nv_bfloat16, 128, Fp8E4M3>(a, G, stream);
  }
  if (a.dtype == PA_BF16) {
    if (a.head_dim == 64) return run_g<__nv_bfloat16, 64>(a, G, stream);
    return run_g<__nv_bfloat16, 128>(a, G, stream);
  }
  if (a.head_dim == 64) return run_g<float, 64>(a, G, stream);
  return run_g<float, 128>(a, G, stream);
}

}  // namespace pa
