// Paged decode attention (requests with q_len == 1): split-K over a balanced partition of
// all K/V pages, then a log-sum-exp merge of the pieces.
//
// What it computes: vLLM 0.10.0 flow page, 3.5 Attention -- the query of each request
// attends to all of its cached K/V, which attention finds through block_table;
// "vLLM" docs page, PagedAttention -- logical block i of a request lives in physical
// block block_table[s, i]; code-reading page 5.1.1 -- the computation runs over the
// logical blocks as if the tokens were contiguous. Decode is memory-bound (flow page,
// 3.2 Scheduler), so the kernel is built around streaming K/V once at HBM speed.
//
// Design (sm_103a):
//  * Work unit = 16 consecutive logical tokens of one request for one group of HG KV
//    heads ("stage"): 16 x HG x D elements of K and the same of V (64 KiB for bf16,
//    HG = 8, D = 128). Units are numbered request-major, then head group, then
//    position; the grid (one CTA per SM) splits that numbering into equal contiguous
//    ranges, so every SM streams the same number of bytes whatever the length mix.
//    A request cut by a range boundary leaves one partial result per CTA; the merge
//    kernel combines them in CTA order. The cut points depend only on seq_lens, so
//    results do not depend on which physical blocks hold the tokens.
//  * One producer warp walks the CTA's units and moves each stage into shared memory
//    with bulk copies (cp.async.bulk, the TMA engine): one copy per physical block
//    when the CTA covers all KV heads (the block's rows are contiguous), one per token
//    row otherwise. A 3-deep ring of stages with full/empty mbarriers keeps two stages
//    in flight while one is consumed. Every wait is bounded (common.cuh).
//  * One consumer warp per KV head (two when it has 8 query heads) takes all 16 tokens
//    of a stage. A lane owns one 16-byte vector of a row (8 bf16 / 4 fp32 dims); q of
//    the warp's query heads sits in registers (fp32, pre-scaled by scale * log2 e). Dot
//    products are packed fp32 FMAs; the per-lane partial dots of (token, head) pairs are
//    summed across the row's lanes by a halving butterfly in which each lane's register
//    slots are pre-permuted by its lane bits, so every step is one shuffle and one add
//    (no selects) and a lane ends with whole logits of its own pairs. Online softmax in
//    fp32 (exp2 domain) with warp-shuffle max/sum; P goes through a small shared buffer
//    to the P.V product, accumulated in fp32 registers.
//  * At a request's last unit in the CTA the warp writes its heads' result to `out`
//    directly when the CTA covered the whole request, else to the workspace as
//    (O / l, m + log2 l).
#include "decode_common.cuh"

namespace pa {
namespace {

// ---------------------------------------------------------------- compile-time layout
// KV is the cache element type. G here is the number of query heads one warp serves (at
// most 4; a KV head with 8 query heads is served by two warps). One warp covers all 16
// tokens of a stage for its heads.
template <typename KV, int D, int G>
struct Cfg {
  static constexpr int EL = sizeof(KV);
  // dims per lane: one 16-byte vector of a 16- or 32-bit row; 8 bytes of an E4M3 row (so
  // the lane layout, and the query / output vectors, match the bf16 case)
  static constexpr int VEC = EL == 1 ? 8 : 16 / EL;
  // stages in the ring: the same bytes in flight for every element size
  static constexpr int STAGES = EL == 1 ? 6 : 3;
  static constexpr int LPR = D / VEC;  // lanes per token row
  static_assert(LPR >= 1 && LPR <= 32 && (32 % LPR) == 0, "row must map onto a warp");
  static constexpr int RPI = 32 / LPR;  // token rows per warp instruction
  static_assert(kTPS % RPI == 0, "a stage must fill whole row groups");
  static constexpr int TPL = kTPS / RPI;  // tokens per lane per stage
  static constexpr int NV = TPL * G;      // partial dots per lane before the reduction
  static constexpr int LOG_LPR = LPR == 1 ? 0 : LPR == 2 ? 1 : LPR == 4 ? 2 : LPR == 8 ? 3 : LPR == 16 ? 4 : 5;
  static constexpr int LOG_NV = NV == 1 ? 0 : NV == 2 ? 1 : NV == 4 ? 2 : NV == 8 ? 3 : NV == 16 ? 4 : NV == 32 ? 5 : NV == 64 ? 6 : 7;
  static_assert((1 << LOG_NV) == NV, "NV must be a power of two");
  static constexpr int LOG_G = G == 1 ? 0 : G == 2 ? 1 : 2;
  static constexpr int NVF = NV > LPR ? NV / LPR : 1;  // whole logits per lane after it
  // Low lane bits that hold duplicates after the reduction (NV < LPR).
  static constexpr int SH = LOG_LPR > LOG_NV ? LOG_LPR - LOG_NV : 0;
  // Lane mask bit b reduces over tokens (not heads, not duplicates)?
  static constexpr __host__ __device__ bool token_bit(int b) {
    return b >= LOG_LPR || (b >= SH && (((1 << (b - SH)) * NVF) % G) == 0);
  }
};

template <typename KV, int D, int G>
struct Smem {
  using C = Cfg<KV, D, G>;
  static constexpr int kStages = C::STAGES;
  // Byte offsets inside the dynamic shared memory of one CTA with HG KV heads served by
  // `warps` consumer warps.
  static __host__ __device__ size_t stage_bytes(int hg) { return size_t(kTPS) * hg * D * C::EL; }
  static __host__ __device__ size_t k_off(int) { return 0; }
  static __host__ __device__ size_t v_off(int hg) { return kStages * stage_bytes(hg); }
  static __host__ __device__ size_t pbuf_off(int hg) { return 2 * kStages * stage_bytes(hg); }
  static __host__ __device__ size_t pbuf_floats_per_warp() { return size_t(C::RPI) * C::NV; }
  static __host__ __device__ size_t desc_off(int hg, int warps) {
    return (pbuf_off(hg) + warps * pbuf_floats_per_warp() * 4 + 15) / 16 * 16;
  }
  static __host__ __device__ size_t bar_off(int hg, int warps) { return desc_off(hg, warps) + kStages * sizeof(StageDesc); }
  // barriers: kStages full, kStages empty
  static __host__ __device__ size_t red_off(int hg, int warps) { return bar_off(hg, warps) + 2 * kStages * 8; }
  static __host__ __device__ size_t total(int hg, int warps) { return red_off(hg, warps) + 40 * 4; }
};

// ---------------------------------------------------------------- the split-K kernel
template <typename T, int D, int G, typename KV>
__global__ void __launch_bounds__(9 * 32, 1) decode_splitk_kernel(const __grid_constant__ DecodeParams p) {
  using C = Cfg<KV, D, G>;
  using SM = Smem<KV, D, G>;
  constexpr int kStages = C::STAGES;
  constexpr int VEC = C::VEC, LPR = C::LPR, RPI = C::RPI, TPL = C::TPL, NV = C::NV, NVF = C::NVF;
  constexpr int SH = C::SH, LOG_G = C::LOG_G;
  const int HG = p.hg_size, QG = p.qg, GF = p.group;
  const int S = p.num_seqs;
  const int num_consumers = HG * QG;

  extern __shared__ __align__(128) unsigned char smem[];
  StageDesc* desc = reinterpret_cast<StageDesc*>(smem + SM::desc_off(HG, num_consumers));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + SM::bar_off(HG, num_consumers));
  int* red = reinterpret_cast<int*>(smem + SM::red_off(HG, num_consumers));
  const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + kStages);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // Programmatic dependent launch: inputs may come from the previous kernel in the stream
  // (e.g. the KV write), so wait for it before reading anything; the merge kernel may be
  // scheduled now and waits for this grid itself.
  griddep_wait();
  griddep_launch_dependents();

  Plan pl;
  if (!plan_range<T, D>(p, red, pl)) return;
  const int64_t u_begin = pl.u_begin, u_end = pl.u_end, c = blockIdx.x;
  const int units_per_hg = pl.units_per_hg;
  const int start_s = pl.start_s, start_hg = pl.start_hg, start_j = pl.start_j;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(full0 + 8 * i, 1);
      mbar_init(empty0 + 8 * i, num_consumers);
    }
    fence_mbar_init();
  }
  __syncthreads();

  const size_t sbytes = SM::stage_bytes(HG);
  const int Hkv = p.num_kv_heads, B = p.block_size;
  const int64_t kv_row_bytes = int64_t(Hkv) * D * C::EL;  // one token, all KV heads

  if (warp == num_consumers) {
    // =========================== producer warp ===========================
    int s = start_s, j = start_j, hg = start_hg;
    int L = decode_len(p, s);
    int units_s = units_of(L);
    int stage = 0;
    uint32_t phase = 0;
    const bool whole_rows = (HG == Hkv);
    const int kv = lane >> 4, idx = lane & 15;
    const char* cache = kv ? p.v_cache : p.k_cache;
    const uint32_t buf0 = smem_u32(smem + (kv ? SM::v_off(HG) : SM::k_off(HG)));
    for (int64_t u = u_begin; u < u_end; ++u) {
      // Fused KV write (decode-only batches): at a request's last unit the new token's row
      // (position L - 1) is taken from k_new / v_new instead of the cache, and the consumer
      // warps store it from shared memory to its slot. Only this CTA reads position L - 1
      // of (request s, head group hg), so nothing reads the slot back within the grid.
      int64_t wslot = -1;
      int qrow_new = 0;
      if (p.k_new && j == units_s - 1) {
        qrow_new = __ldg(p.qsl + s);
        const int64_t slot = __ldg(p.slot_mapping + qrow_new);
        const int64_t at =
            int64_t(__ldg(p.block_table + int64_t(s) * p.max_blocks_per_seq + (L - 1) / B)) * B + (L - 1) % B;
        if (slot >= 0 && slot == at && slot < p.num_blocks * B) {
          wslot = slot;
        } else if (slot >= 0) {
          // not the slot of position L - 1 (or out of range): flag it, and write the row
          // where slot_mapping says (as pa_kv_write would); position L - 1 is read from
          // the cache as it stands
          if (lane == 0 && slot != at) raise_error(p.err, PA_DEVERR_SLOT_MISMATCH);
          if (slot < p.num_blocks * B) {
            const int64_t slice = int64_t(HG) * D * C::EL;
            const int64_t src_off = int64_t(qrow_new) * kv_row_bytes + hg * slice;
            const int64_t dst_off = slot * kv_row_bytes + hg * slice;
            for (int64_t o = int64_t(lane) * 16; o < slice; o += 32 * 16) {
              const uint4 kx = __ldg(reinterpret_cast<const uint4*>(p.k_new + src_off + o));
              const uint4 vx = __ldg(reinterpret_cast<const uint4*>(p.v_new + src_off + o));
              *reinterpret_cast<uint4*>(p.k_cache_w + dst_off + o) = kx;
              *reinterpret_cast<uint4*>(p.v_cache_w + dst_off + o) = vx;
            }
          } else if (lane == 0) {
            raise_error(p.err, PA_DEVERR_SLOT_RANGE);
          }
        }
      }
      const int64_t u0 = u - j, u1 = u0 + units_s;
      int flags = 0;
      if (u == u_begin || j == 0) flags |= kFirst;
      if (u == u_end - 1 || j == units_s - 1) flags |= kLast;
      if (u0 >= u_begin) flags |= kSeqStart;
      if (u1 <= u_end) flags |= kSeqEnd;
      const int valid = min(kTPS, L - j * kTPS);
      // ---- this lane's copy (at most one per lane: 16 for K, 16 for V)
      const int32_t* bt = p.block_table + int64_t(s) * p.max_blocks_per_seq;
      const int pos0 = j * kTPS;
      bool have = false, bad = false, have2 = false;
      const char* src = nullptr;
      const char* src2 = nullptr;
      uint32_t dst = 0, bytes = 0, dst2 = 0;
      const char* fresh = (kv ? p.v_new : p.k_new) + int64_t(qrow_new) * kv_row_bytes;  // used iff wslot >= 0
      if (whole_rows) {
        // the lane whose copy ends at row valid - 1 leaves that row to a second copy from
        // the new token's K/V when the write is fused
        if (B >= kTPS) {
          if (idx == 0) {
            const int64_t blk = __ldg(bt + pos0 / B);
            bad = blk < 0 || blk >= p.num_blocks;
            const int rows = valid - (wslot >= 0 ? 1 : 0);
            have = !bad && rows > 0;
            src = cache + (blk * B + pos0 % B) * kv_row_bytes;
            bytes = uint32_t(rows * kv_row_bytes);
            dst = buf0 + stage * sbytes;
          }
        } else {
          const int nblk = (valid + B - 1) / B;
          if (idx < nblk) {
            const int64_t blk = __ldg(bt + pos0 / B + idx);
            bad = blk < 0 || blk >= p.num_blocks;
            const int rows = min(B, valid - idx * B) - ((wslot >= 0 && idx == nblk - 1) ? 1 : 0);
            have = !bad && rows > 0;
            src = cache + blk * B * kv_row_bytes;
            bytes = uint32_t(rows * kv_row_bytes);
            dst = buf0 + stage * sbytes + uint32_t(idx * B * kv_row_bytes);
          }
          if (wslot >= 0 && idx == nblk - 1) {
            have2 = true;
            src2 = fresh;
            dst2 = buf0 + stage * sbytes + uint32_t((valid - 1) * kv_row_bytes);
          }
        }
        if (B >= kTPS && wslot >= 0 && idx == 1) {
          have2 = true;
          src2 = fresh;
          dst2 = buf0 + stage * sbytes + uint32_t((valid - 1) * kv_row_bytes);
        }
      } else if (idx < valid) {
        const int pos = pos0 + idx;
        const int64_t hg_row = int64_t(HG) * D * C::EL;
        if (wslot >= 0 && idx == valid - 1) {
          have = true;
          src = fresh + hg * hg_row;
        } else {
          const int64_t blk = __ldg(bt + pos / B);
          bad = blk < 0 || blk >= p.num_blocks;
          have = !bad;
          src = cache + (blk * B + pos % B) * kv_row_bytes + hg * hg_row;
        }
        bytes = uint32_t(hg_row);
        dst = buf0 + stage * sbytes + uint32_t(idx * hg_row);
      }
      const int total_bytes = warp_sum_i((have ? int(bytes) : 0) + (have2 ? int(kv_row_bytes) : 0));
      const bool any_bad = __any_sync(0xffffffffu, bad);
      if (any_bad) flags |= kBad;
      int ok = 1;
      if (lane == 0) ok = mbar_wait(empty0 + 8 * stage, phase ^ 1) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) {
        raise_error(p.err, PA_DEVERR_TIMEOUT);
        break;
      }
      if (lane == 0) {
        if (any_bad) raise_error(p.err, PA_DEVERR_BLOCK_RANGE);
        StageDesc d;
        d.s = s;
        d.hg = hg;
        d.j = j;
        d.valid = valid;
        d.flags = flags;
        d.pad = 0;
        d.wslot = wslot;
        desc[stage] = d;
        mbar_arrive_expect_tx(full0 + 8 * stage, uint32_t(total_bytes));
      }
      __syncwarp();
      if (have) bulk_g2s(dst, src, bytes, full0 + 8 * stage);
      if (have2) bulk_g2s(dst2, src2, uint32_t(kv_row_bytes), full0 + 8 * stage);
      if (++stage == kStages) {
        stage = 0;
        phase ^= 1;
      }
      if (++j == units_s && u + 1 < u_end) {
        j = 0;
        if (++hg == p.num_hg) {
          hg = 0;
          do {
            if (++s >= S) break;  // cannot happen: the plan counted these units
            L = decode_len(p, s);
            units_s = units_of(L);
          } while (units_s == 0);
          if (s >= S) {
            raise_error(p.err, PA_DEVERR_TIMEOUT);
            break;
          }
        }
      }
    }
    return;
  }

  // =========================== consumer warps ===========================
  // warp -> (KV head hk within the CTA's group, query-head group qg); lane -> (row group
  // r, lane-in-row lir owning dims [lir * VEC, lir * VEC + VEC)).
  const int hk = warp / QG, qg = warp % QG;
  const int lir = lane & (LPR - 1), r = lane / LPR;
  const int Hq = p.num_heads;
  float* pbuf = reinterpret_cast<float*>(smem + SM::pbuf_off(HG)) + warp * SM::pbuf_floats_per_warp();
  const KV* kbase = reinterpret_cast<const KV*>(smem + SM::k_off(HG));
  const KV* vbase = reinterpret_cast<const KV*>(smem + SM::v_off(HG));
  const size_t stage_elems = sbytes / C::EL;

  // Butterfly without selects: slot s of this lane holds the partial dot of value
  // (s ^ P), value = token * G + head, where P collects the lane bits the halving steps
  // test. Each step then keeps the low half of the slots and adds the partner's high half.
  int P = 0;
#pragma unroll
  for (int k = 1; k <= C::LOG_LPR; ++k)
    if ((NV >> k) >= 1 && (lir & (LPR >> k))) P |= (NV >> k);
  const int Pt = P >> LOG_G;        // token part of the permutation
  const int Pg = P & (G - 1);       // head part
  // After the reduction slot i (< NVF) holds value (lir >> SH) * NVF + i.
  int my_g[NVF], my_ti[NVF];
#pragma unroll
  for (int i = 0; i < NVF; ++i) {
    const int id = (lir >> SH) * NVF + i;
    my_g[i] = id % G;
    my_ti[i] = id / G;
  }
  const bool p_writer = (lir & ((1 << SH) - 1)) == 0;

  float2 qf[G][VEC / 2];   // q of head (g ^ Pg), scaled to the log2 domain
  float2 acc[G][VEC / 2];  // unnormalised O of head g, this lane's dims, this row group
  float mrun[G];
  float lpart[NVF];
  const KV* kw = kbase + hk * D + lir * VEC;  // this lane's column in every K / V row
  const KV* vw = vbase + hk * D + lir * VEC;
  const int row_stride = HG * D;

  int stage = 0;
  uint32_t phase = 0;
  for (int64_t u = u_begin; u < u_end; ++u) {
    if (!mbar_wait(full0 + 8 * stage, phase)) {
      raise_error(p.err, PA_DEVERR_TIMEOUT);
      return;
    }
    const StageDesc d = desc[stage];
    if (d.flags & kFirst) {
      const int qrow = __ldg(p.qsl + d.s);
      const T* qb = reinterpret_cast<const T*>(p.q) + (int64_t(qrow) * Hq + (d.hg * HG + hk) * GF + qg * G) * D +
                    lir * VEC;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float f[VEC];
        RowVec<T, VEC>::load(qb + (g ^ Pg) * D, f);
#pragma unroll
        for (int e = 0; e < VEC / 2; ++e) {
          qf[g][e] = make_float2(f[2 * e] * p.scale_log2, f[2 * e + 1] * p.scale_log2);
          acc[g][e] = make_float2(0.f, 0.f);
        }
        mrun[g] = -INFINITY;
      }
#pragma unroll
      for (int i = 0; i < NVF; ++i) lpart[i] = 0.f;
    }
    const int valid = (d.flags & kBad) ? 0 : d.valid;
    const KV* ks = kw + stage * stage_elems;
    if constexpr (sizeof(KV) == sizeof(T)) {  // the fused write exists for 16/32-bit caches only
      if (d.wslot >= 0 && qg == 0 && r == (d.valid - 1) % RPI) {
        // fused KV write: this warp's KV head of the new token's row, shared -> cache
        const int64_t off = d.wslot * kv_row_bytes + (int64_t(d.hg * HG + hk) * D + lir * VEC) * C::EL;
        const int t = d.valid - 1;
        *reinterpret_cast<uint4*>(p.k_cache_w + off) = *reinterpret_cast<const uint4*>(ks + t * row_stride);
        *reinterpret_cast<uint4*>(p.v_cache_w + off) =
            *reinterpret_cast<const uint4*>(vw + stage * stage_elems + t * row_stride);
      }
    }

    // ---- S = q . K: slot (tj, gj) holds token r + RPI * (tj ^ Pt), head gj ^ Pg
    float sv[NV];
#pragma unroll
    for (int tj = 0; tj < TPL; ++tj) {
      const int t = r + RPI * (tj ^ Pt);
      float kf[VEC];
      RowVec<KV, VEC>::load(ks + t * row_stride, kf);
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float2 a = make_float2(0.f, 0.f);
#pragma unroll
        for (int e = 0; e < VEC / 2; ++e) ffma2(a, qf[g][e], make_float2(kf[2 * e], kf[2 * e + 1]));
        sv[tj * G + g] = a.x + a.y;
      }
    }
    // ---- butterfly across the row's lanes
#pragma unroll
    for (int k = 1; k <= C::LOG_LPR; ++k) {
      const int m = LPR >> k;
      if ((NV >> k) >= 1) {
#pragma unroll
        for (int i = 0; i < NV / 2; ++i)
          if (i < (NV >> k)) sv[i] += __shfl_xor_sync(0xffffffffu, sv[i + (NV >> k)], m);
      } else {
        sv[0] += __shfl_xor_sync(0xffffffffu, sv[0], m);
      }
    }
    // ---- online softmax (log2 domain)
    float x[NVF], bm[NVF];
#pragma unroll
    for (int i = 0; i < NVF; ++i) {
      const int t = r + RPI * my_ti[i];
      x[i] = (t < valid) ? sv[i] : -INFINITY;
      bm[i] = x[i];
    }
#pragma unroll
    for (int b = 0; b < 5; ++b) {
      if (C::token_bit(b)) {
#pragma unroll
        for (int i = 0; i < NVF; ++i) bm[i] = fmaxf(bm[i], __shfl_xor_sync(0xffffffffu, bm[i], 1 << b));
      }
    }
    float mnew[G], msafe[G], alpha[G];
    bool rescale = false;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float mb = __shfl_sync(0xffffffffu, bm[g % NVF], (g / NVF) << SH);
      mnew[g] = fmaxf(mrun[g], mb);
      msafe[g] = (mnew[g] == -INFINITY) ? 0.f : mnew[g];
      alpha[g] = exp2f(mrun[g] - msafe[g]);
      rescale |= (alpha[g] != 1.f);
    }
    if (rescale) {
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int e = 0; e < VEC / 2; ++e) {
          acc[g][e].x *= alpha[g];
          acc[g][e].y *= alpha[g];
        }
#pragma unroll
      for (int i = 0; i < NVF; ++i) lpart[i] *= pick(alpha, my_g[i]);
    }
#pragma unroll
    for (int i = 0; i < NVF; ++i) {
      const float pv = exp2f(x[i] - pick(msafe, my_g[i]));
      lpart[i] += pv;
      if (p_writer) pbuf[r * NV + (lir >> SH) * NVF + i] = pv;
    }
#pragma unroll
    for (int g = 0; g < G; ++g) mrun[g] = mnew[g];
    __syncwarp();

    // ---- O += P . V over this lane's tokens r + RPI * ti
    const KV* vs = vw + stage * stage_elems;
    if (valid == kTPS) {
#pragma unroll
      for (int ti = 0; ti < TPL; ++ti) {
        const int t = r + RPI * ti;
        float vf[VEC];
        RowVec<KV, VEC>::load(vs + t * row_stride, vf);
        float pw[G];
#pragma unroll
        for (int g = 0; g < G; ++g) pw[g] = pbuf[r * NV + ti * G + g];
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
          for (int e = 0; e < VEC / 2; ++e)
            ffma2(acc[g][e], make_float2(pw[g], pw[g]), make_float2(vf[2 * e], vf[2 * e + 1]));
      }
    } else {
#pragma unroll
      for (int ti = 0; ti < TPL; ++ti) {
        const int t = r + RPI * ti;
        if (t < valid) {  // rows past the request's end hold stale data: skip, never multiply
          float vf[VEC];
          RowVec<KV, VEC>::load(vs + t * row_stride, vf);
          float pw[G];
#pragma unroll
          for (int g = 0; g < G; ++g) pw[g] = pbuf[r * NV + ti * G + g];
#pragma unroll
          for (int g = 0; g < G; ++g)
#pragma unroll
            for (int e = 0; e < VEC / 2; ++e)
              ffma2(acc[g][e], make_float2(pw[g], pw[g]), make_float2(vf[2 * e], vf[2 * e + 1]));
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * stage);
    if (++stage == kStages) {
      stage = 0;
      phase ^= 1;
    }

    if (!(d.flags & kLast)) continue;

    // ================= finalize this request's piece =================
    float lsum[NVF];
#pragma unroll
    for (int i = 0; i < NVF; ++i) lsum[i] = lpart[i];
#pragma unroll
    for (int b = 0; b < 5; ++b) {
      if (C::token_bit(b)) {
#pragma unroll
        for (int i = 0; i < NVF; ++i) lsum[i] += __shfl_xor_sync(0xffffffffu, lsum[i], 1 << b);
      }
    }
    float lh[G];
#pragma unroll
    for (int g = 0; g < G; ++g) lh[g] = __shfl_sync(0xffffffffu, lsum[g % NVF], (g / NVF) << SH);
    // O partials of the row groups -> every lane
#pragma unroll
    for (int m = LPR; m < 32; m <<= 1)
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int e = 0; e < VEC / 2; ++e) {
          acc[g][e].x += __shfl_xor_sync(0xffffffffu, acc[g][e].x, m);
          acc[g][e].y += __shfl_xor_sync(0xffffffffu, acc[g][e].y, m);
        }
    const bool whole = (d.flags & kSeqStart) && (d.flags & kSeqEnd);
    const int qrow = __ldg(p.qsl + d.s);
    if (r == 0) {
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float inv = lh[g] > 0.f ? p.v_scale / lh[g] : 0.f;  // V codes -> values: * v_scale
        float o[VEC];
#pragma unroll
        for (int e = 0; e < VEC / 2; ++e) {
          o[2 * e] = acc[g][e].x * inv;
          o[2 * e + 1] = acc[g][e].y * inv;
        }
        const int hq = (d.hg * HG + hk) * GF + qg * G + g;
        if (whole) {
          RowVec<T, VEC>::store(reinterpret_cast<T*>(p.out) + (int64_t(qrow) * Hq + hq) * D + lir * VEC, o);
        } else {
          const int64_t slot = c + int64_t(d.s) * p.num_hg + d.hg;
          const int64_t hrow = slot * (HG * GF) + hk * GF + qg * G + g;
          float* dst = p.ws_o + hrow * D + lir * VEC;
#pragma unroll
          for (int e = 0; e < VEC; e += 4)
            *reinterpret_cast<float4*>(dst + e) = make_float4(o[e], o[e + 1], o[e + 2], o[e + 3]);
          if (lir == 0) p.ws_lse[hrow] = (lh[g] > 0.f) ? mrun[g] + __log2f(lh[g]) : -INFINITY;
        }
      }
    }
    if (warp == 0 && lane == 0) {
      const int64_t v = int64_t(d.s) * p.num_hg + d.hg;
      if (d.flags & kSeqStart) {
        p.ws_meta[v].x = int(c);
        p.ws_meta[v].z = units_per_hg;
        p.ws_meta[v].w = qrow;
      }
      if (d.flags & kSeqEnd) p.ws_meta[v].y = int(c);
    }
  }
}

// ---------------------------------------------------------------- host side
// GW = query heads per warp (<= 4), QG = G / GW consumer warps per KV head, HG = KV heads
// per CTA: the largest power of two dividing num_kv_heads with HG * QG <= 8 consumer warps
// whose stages fit in shared memory.
template <typename KV, int D, int GW>
int pick_hg(int num_kv_heads, int qg) {
  for (int hg = 8; hg >= 1; hg >>= 1)
    if (num_kv_heads % hg == 0 && hg * qg <= 8 && Smem<KV, D, GW>::total(hg, hg * qg) <= size_t(kSmemLimit))
      return hg;
  return 0;
}

int gw_of(int G) { return G < 4 ? G : 4; }

int hg_for(pa_dtype dt, int D, int G, int num_kv_heads) {
  const int GW = gw_of(G), QG = G / GW;
#define PA_HG_CASE(TT, DD, WW) \
  if (D == DD && GW == WW) return pick_hg<TT, DD, WW>(num_kv_heads, QG);
  if (dt == PA_FP8_E4M3) {
    PA_HG_CASE(Fp8E4M3, 64, 1) PA_HG_CASE(Fp8E4M3, 64, 2) PA_HG_CASE(Fp8E4M3, 64, 4)
    PA_HG_CASE(Fp8E4M3, 128, 1) PA_HG_CASE(Fp8E4M3, 128, 2) PA_HG_CASE(Fp8E4M3, 128, 4)
  } else if (dt == PA_BF16) {
    PA_HG_CASE(__nv_bfloat16, 64, 1) PA_HG_CASE(__nv_bfloat16, 64, 2) PA_HG_CASE(__nv_bfloat16, 64, 4)
    PA_HG_CASE(__nv_bfloat16, 128, 1) PA_HG_CASE(__nv_bfloat16, 128, 2) PA_HG_CASE(__nv_bfloat16, 128, 4)
  } else {
    PA_HG_CASE(float, 64, 1) PA_HG_CASE(float, 64, 2) PA_HG_CASE(float, 64, 4)
    PA_HG_CASE(float, 128, 1) PA_HG_CASE(float, 128, 2) PA_HG_CASE(float, 128, 4)
  }
#undef PA_HG_CASE
  return 0;
}

template <typename T, int D, int GW, typename KV>
cudaError_t run(const AttnArgs& a, int num_ctas, cudaStream_t stream) {
  using SM = Smem<KV, D, GW>;
  const int G = a.num_heads / a.num_kv_heads;
  const int QG = G / GW;
  const int hg = pick_hg<KV, D, GW>(a.num_kv_heads, QG);
  if (hg == 0) return cudaErrorInvalidValue;
  DecodeParams p = fill_decode_params(a, hg, QG, num_ctas, D);
  const bool fused = sizeof(KV) == sizeof(T) && a.k_new != nullptr;
  p.k_new = fused ? static_cast<const char*>(a.k_new) : nullptr;
  p.v_new = fused ? static_cast<const char*>(a.v_new) : nullptr;
  p.slot_mapping = fused ? a.slot_mapping : nullptr;
  if (sizeof(KV) == 1) p.scale_log2 *= a.k_scale;  // K codes -> values: fold k_scale into q
  p.v_scale = sizeof(KV) == 1 ? a.v_scale : 1.f;
  const int warps = hg * QG;
  const size_t smem = SM::total(hg, warps);
  auto kern = decode_splitk_kernel<T, D, GW, KV>;
  cudaError_t e = ensure_smem<decode_splitk_kernel<T, D, GW, KV>>(smem);
  if (e != cudaSuccess) return e;
  e = launch_pdl(kern, dim3(num_ctas), dim3((warps + 1) * 32), smem, stream, p);
  if (e != cudaSuccess) return e;
  return launch_merge<T, D>(p, stream, a.merge_pdl);
}

template <typename T, int D, typename KV = T>
cudaError_t run_g(const AttnArgs& a, int G, int num_ctas, cudaStream_t stream) {
  switch (gw_of(G)) {
    case 1: return run<T, D, 1, KV>(a, num_ctas, stream);
    case 2: return run<T, D, 2, KV>(a, num_ctas, stream);
    case 4: return run<T, D, 4, KV>(a, num_ctas, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

int decode_hg(pa_dtype cache_dtype, int head_dim, int group, int num_kv_heads) {
  return hg_for(cache_dtype, head_dim, group, num_kv_heads);
}

bool decode_supported(pa_dtype dtype, int head_dim, int group) {
  if (head_dim != 64 && head_dim != 128) return false;
  if (group != 1 && group != 2 && group != 4 && group != 8) return false;
  return dtype == PA_F32 || dtype == PA_BF16;
}

int decode_num_ctas(int device, cudaError_t* err) {
  int sms = 0;
  *err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
  return sms;
}

size_t decode_workspace_bytes(int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                              int num_ctas, pa_dtype dtype) {
  const int G = num_heads / num_kv_heads;
  const int hg = hg_for(dtype, head_dim, G, num_kv_heads);
  if (hg == 0) return 0;
  const int num_hg = num_kv_heads / hg;
  const int64_t slots = int64_t(num_ctas) + int64_t(num_seqs) * num_hg;
  const int64_t HGG = int64_t(hg) * G;
  const int64_t o_bytes = slots * HGG * head_dim * 4;
  const int64_t lse_bytes = ((slots * HGG * 4 + 15) / 16) * 16;
  const int64_t meta_bytes = int64_t(num_seqs) * num_hg * 16;
  return size_t(o_bytes + lse_bytes + meta_bytes);
}

cudaError_t launch_decode(const AttnArgs& a, int num_ctas, cudaStream_t stream) {
  const int G = a.num_heads / a.num_kv_heads;
  if (a.num_seqs == 0) return cudaSuccess;
  const int hg = hg_for(a.cache_dtype, a.head_dim, G, a.num_kv_heads);
  if (decode_mma_supported(a, hg)) return launch_decode_mma(a, hg, num_ctas, stream);
  if (a.cache_dtype == PA_FP8_E4M3) {  // E4M3 caches: bf16 q and out only
    if (a.dtype != PA_BF16) return cudaErrorInvalidValue;
    if (a.head_dim == 64) return run_g<__nv_bfloat16, 64, Fp8E4M3>(a, G, num_ctas, stream);
    return run_g<__nv_bfloat16, 128, Fp8E4M3>(a, G, num_ctas, stream);
  }
  if (a.dtype == PA_BF16) {
    if (a.head_dim == 64) return run_g<__nv_bfloat16, 64>(a, G, num_ctas, stream);
    return run_g<__nv_bfloat16, 128>(a, G, num_ctas, stream);
  }
  if (a.head_dim == 64) return run_g<float, 64>(a, G, num_ctas, stream);
  return run_g<float, 128>(a, G, num_ctas, stream);
}

}  // namespace pa
