// Paged decode attention (requests with q_len == 1) with the dot products on the tensor
// cores: split-K over the balanced partition of all K/V pages (decode_common.cuh), then
// the log-sum-exp merge of the pieces.
//
// What it computes: the same as decode_attention.cu (vLLM 0.10.0 flow page, 3.5 Attention;
// "vLLM" docs page, PagedAttention; code-reading page 5.1.1), for bf16 queries over bf16
// or FP8 (E4M3) caches ("vLLM" docs page, quantisation support).
//
// Why: a decode step is a stream of K/V bytes, but with 16 tokens x 8 KV heads per stage
// the CUDA-core consumers need as long per stage as the stage takes to arrive, and an
// E4M3 cache halves the bytes without halving that work. Here each consumer warp does a
// stage as 16-row matrix products on mma.sync (m16n8k16, fp32 accumulate): rows are the
// G query heads of its KV head, so S = Q K^T (16 tokens) is 16 MMAs for D = 128 and
// O += P V another 16, against ~500 FMA-pipe instructions on CUDA cores. (tcgen05 needs
// M >= 64 rows and a TMEM round trip per stage; with at most 8 query heads per KV head
// the register-file MMA has the shorter dependency chain.)
//
// Layout: the producer warp loads each stage with 3-D TMA tensor copies over the cache
// viewed as (dim, token, KV head): a box of {128 bytes of dims, BT tokens, HG heads} lands
// as [head][token][128 B] with the 128-byte swizzle, so the rows a warp reads for one
// head at one 16-byte column sit in 8 different bank groups (conflict-free ldmatrix /
// loads). The cache is read exactly once per stage.
//
// Precision: bf16 caches multiply in bf16 (Q and K exact), P rounded to bf16 for P V;
// E4M3 caches multiply in f16 (E4M3 codes and bf16 queries of normal range are exact in
// f16; P rounded to f16). Accumulation and softmax in fp32 (exp2 domain).
#include <cudaTypedefs.h>

#include "decode_common.cuh"
#include "tcgen05.cuh"

namespace pa {
namespace {

// ---------------------------------------------------------------- tensor-core wrappers
// D (16 x 8, fp32) += A (16 x 16) B (16 x 8): a0 / a2 rows g, a1 / a3 rows g + 8.
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1, bool f16) {
  if (f16)
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  else
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Four 8x8 16-bit matrices, transposed: thread l gets (row 2(l%4), col l/4) and
// (row 2(l%4)+1, col l/4) of each; lanes 8m..8m+7 give matrix m's row addresses.
__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                              uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr)
               : "memory");
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr)
               : "memory");
  return v;
}

// Two 16x16 byte matrices, transposed: lanes 0-15 address rows 0-15 of the first, lanes
// 16-31 those of the second; lane (g, t) = (l / 4, l % 4) gets rows 4t .. 4t+3 of column g
// (r0) and of column g + 8 (r1) of the first, the same of the second in r2, r3.
__device__ __forceinline__ void ldsm_b8_x2_trans(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                                 uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m16n16.x2.trans.shared.b8 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr)
               : "memory");
}

// Four 8x8 16-bit matrices: thread l gets (row l/4, cols 2(l%4), 2(l%4)+1) of each.
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr)
               : "memory");
}


// two fp32 -> packed bf16x2 / f16x2 (lo in the low half), round to nearest even
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
// two E4M3 codes (low 16 bits, low byte first) -> f16x2, exact
// The four E4M3 codes of x -> f16x2 of codes (0, 1) and of codes (2, 3) (exact).
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t x, uint32_t& c01, uint32_t& c23) {
  asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\tcvt.rn.f16x2.e4m3x2 %0, a;\n\tcvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
      : "=r"(c01), "=r"(c23)
      : "r"(x));
}

// ---------------------------------------------------------------- layout
// KV: __nv_bfloat16 or Fp8E4M3; BT: tokens per TMA box (8 or 16; 16 / BT boxes a stage).
template <typename KV, int D, int BT>
struct MmaCfg {
  static constexpr int EL = sizeof(KV);
  static constexpr bool kF16 = EL == 1;           // E4M3 caches multiply in f16
  static constexpr int INNER = 128 / EL;          // elements of one swizzled 128-byte row
  static constexpr int HALVES = D / INNER;        // boxes along the head dimension
  static_assert(HALVES >= 1 && D % INNER == 0, "head_dim must fill 128-byte rows");
  static constexpr int NBOX = kTPS / BT;          // boxes along the tokens of a stage
  static constexpr int STAGES = EL == 1 ? 6 : 3;  // 192 KiB in flight at HG = 8, D = 128
  static constexpr int KC = D / 16;               // 16-dim chunks (MMA k steps of S)
  static constexpr int NT = D / 8;                // 8-dim tiles of O (MMA n tiles of P V)
  // bytes
  static __host__ __device__ uint32_t box_bytes(int hg) { return uint32_t(hg) * BT * 128; }
  static __host__ __device__ uint32_t half_bytes(int hg) { return NBOX * box_bytes(hg); }
  static __host__ __device__ uint32_t stage_bytes(int hg) { return HALVES * half_bytes(hg); }  // K (or V)
  static __host__ __device__ uint32_t k_off(int hg, int st) { return uint32_t(st) * 2 * stage_bytes(hg); }
  static __host__ __device__ uint32_t v_off(int hg, int st) { return k_off(hg, st) + stage_bytes(hg); }
  static __host__ __device__ uint32_t desc_off(int hg) { return STAGES * 2 * stage_bytes(hg); }
  static __host__ __device__ uint32_t bar_off(int hg) { return desc_off(hg) + STAGES * 48; }  // MmaDesc
  static __host__ __device__ uint32_t red_off(int hg) { return bar_off(hg) + 2 * STAGES * 8; }
  // query slots: 2 mbarriers, then 2 slots of q_slot bytes, 16-byte aligned
  static __host__ __device__ uint32_t qbar_off(int hg) { return red_off(hg) + 40 * 4; }
  static __host__ __device__ uint32_t qslot_off(int hg) { return (qbar_off(hg) + 16 + 15) / 16 * 16; }
  static __host__ __device__ uint32_t total(int hg, uint32_t q_slot) {  // + alignment slack
    return qslot_off(hg) + 2 * q_slot + 1024;
  }
  // Byte offset, inside a stage's K (or V), of 16-byte column `chunk` (of the 128-byte
  // row of dims [half * INNER, half * INNER + INNER)) of token `tok` of head `h`.
  static __device__ __forceinline__ uint32_t at(int hg, int half, int tok, int h, int chunk) {
    const int row = h * BT + (tok % BT);  // row inside its box; box bases are 1024-aligned
    return uint32_t(half) * half_bytes(hg) + uint32_t(tok / BT) * box_bytes(hg) + uint32_t(row) * 128 +
           uint32_t((chunk ^ (row & 7)) * 16);
  }
};

// ---------------------------------------------------------------- segments
// The unit numbering runs over segments. Without groups a segment is a request. With
// shared-prefix groups, segments [0, num_groups) are the groups' shared prefixes (16-token
// chunks every member holds in the same physical slots; the MMA rows are all members'
// query heads, so those K/V bytes are read once for the whole group) and segment
// num_groups + s is request s past its group's shared chunks.
struct MmaDesc {
  int s;      // the request (own segment) or the group's first member (shared segment)
  int hg, j, valid, flags;
  int seg;    // segment index
  int nmem;   // requests whose query heads are the MMA rows (1 for an own segment)
  int pos0;   // position of the stage's first token
  int64_t wslot;
  int64_t pad;  // the own segment's skipped (shared) chunks
};
static_assert(sizeof(MmaDesc) == 48, "the shared-memory layout reserves 48 bytes a descriptor");

// Group g's members: requests [group_start[2g], group_start[2g + 1]) (clamped to the batch).
__device__ __forceinline__ void group_span(const DecodeParams& p, int g, int& a, int& b) {
  a = min(max(__ldg(p.group_start + 2 * g), 0), p.num_seqs);
  b = min(max(__ldg(p.group_start + 2 * g + 1), a), p.num_seqs);
}

// Shared 16-token chunks of group g: whole chunks below shared_len and every member's
// length; 0 for a group that is too small or too large for 16 MMA rows.
__device__ int shared_chunks(const DecodeParams& p, int g) {
  int a, b;
  group_span(p, g, a, b);
  if (b - a < 2 || (b - a) * p.group > 16) return 0;
  int lim = __ldg(p.shared_len + g);
  for (int s = a; s < b; ++s) lim = min(lim, decode_len(p, s));
  return max(lim, 0) / kTPS;
}

// Leading chunks of request s that its group's shared segment covers.
__device__ int own_skip(const DecodeParams& p, int s) {
  if (p.num_groups == 0) return 0;
  const int g = __ldg(p.seq_group + s);
  if (g < 0 || g >= p.num_groups) return 0;
  int a, b;
  group_span(p, g, a, b);
  if (s < a || s >= b) return 0;  // inconsistent membership: the request runs on its own
  return shared_chunks(p, g);
}

__device__ int seg_units(const DecodeParams& p, int k) {
  if (k < p.num_groups) return shared_chunks(p, k);
  const int s = k - p.num_groups;
  return max(units_of(decode_len(p, s)) - own_skip(p, s), 0);
}

// The CTA's range over the segment-major numbering (as plan_range over requests). `cache`
// (`cap` ints of shared memory the pipeline has not started on yet) keeps each segment's
// unit count from the first pass for the later ones (each thread rereads the entries it
// wrote; the start segment's is read after the scan's barriers): a grouped request's count
// is a chain of dependent loads (its group, the group's span, the members' lengths).
template <typename T, int D>
__device__ bool plan_segments(const DecodeParams& p, int* red, Plan& pl, int* cache, int cap) {
  const int S = p.num_seqs, NS = p.num_groups + S;
  int my_units = 0;
  for (int k = threadIdx.x; k < NS; k += blockDim.x) {
    const int n = seg_units(p, k);
    if (k < cap) cache[k] = n;
    my_units += n;
  }
  pl.units_per_hg = block_sum(my_units, red);
  const int64_t U = int64_t(pl.units_per_hg) * p.num_hg;
  const int64_t c = blockIdx.x, C_ = gridDim.x;
  if (c == 0) {
    for (int k = threadIdx.x; k < NS; k += blockDim.x) {
      if ((k < cap ? cache[k] : seg_units(p, k)) > 0) continue;
      for (int hg = 0; hg < p.num_hg; ++hg) p.ws_meta[int64_t(k) * p.num_hg + hg] = make_int4(-1, -1, 0, 0);
      if (k < p.num_groups) continue;
      const int s = k - p.num_groups;
      const int q0 = __ldg(p.qsl + s);
      if (__ldg(p.qsl + s + 1) - q0 == 1 && decode_len(p, s) == 0) {  // a decode query without keys
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
  for (int base = 0; base < NS; base += blockDim.x) {
    const int k = base + threadIdx.x;
    const int us = k < NS ? (k < cap ? cache[k] : seg_units(p, k)) * p.num_hg : 0;
    int total;
    const int ex = block_exclusive_scan(us, red, &total);
    if (us > 0 && run + ex <= rem && rem < run + ex + us) {
      red[34] = k;
      red[35] = int(rem - (run + ex));
    }
    __syncthreads();
    run += total;
    if (run > rem) break;
  }
  pl.start_s = red[34];  // a segment here
  const int start_us = pl.start_s < cap ? cache[pl.start_s] : seg_units(p, pl.start_s);
  pl.start_hg = red[35] / start_us;
  pl.start_j = red[35] % start_us;
  return true;
}

// ---------------------------------------------------------------- the kernel
// GROUPED: shared-prefix segments may put up to 16 query heads (several requests) on the
// MMA rows, so rows 8..15 carry data (A fragments a1 / a3, a second softmax row per lane).
template <typename T, int D, typename KV, int BT, bool GROUPED>
__global__ void __launch_bounds__(9 * 32, 1)
    decode_mma_kernel(const __grid_constant__ DecodeParams p, const __grid_constant__ CUtensorMap kmap,
                      const __grid_constant__ CUtensorMap vmap) {
  using C = MmaCfg<KV, D, BT>;
  constexpr int STAGES = C::STAGES;
  const int HG = p.hg_size, G = p.group;
  const int NG = p.num_groups, NS = NG + p.num_seqs;

  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;  // 128-byte swizzle atoms need 1024-byte alignment
  unsigned char* smem = smem_raw + (base - raw);
  MmaDesc* desc = reinterpret_cast<MmaDesc*>(smem + C::desc_off(HG));
  int* red = reinterpret_cast<int*>(smem + C::red_off(HG));
  const uint32_t full0 = base + C::bar_off(HG), empty0 = full0 + 8 * STAGES;
  // query slots: filled with a segment's first stage in this CTA, released by the consumer
  // warps after its last stage (bf16 caches, when they fit in shared memory: p.q_slot > 0;
  // with groups, for the segments of one request, whose query rows are one token's)
  constexpr bool kQSlots = C::EL == 2;  // compiled in for bf16 caches
  const bool qsm = kQSlots && p.q_slot > 0;
  const uint32_t qbar0 = base + C::qbar_off(HG), qslot0 = base + C::qslot_off(HG);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int num_consumers = HG;  // one warp per KV head of the group

  griddep_wait();
  griddep_launch_dependents();

  Plan pl;
  // the stages' shared memory caches the plan's counts (no copy lands there before the
  // barrier below)
  if (!plan_segments<T, D>(p, red, pl, reinterpret_cast<int*>(smem), int(C::desc_off(HG) / 4))) return;
  const int64_t u_begin = pl.u_begin, u_end = pl.u_end, c = blockIdx.x;

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(full0 + 8 * i, 1);
      mbar_init(empty0 + 8 * i, num_consumers);
    }
    if (kQSlots) {
      mbar_init(qbar0, num_consumers);
      mbar_init(qbar0 + 8, num_consumers);
    }
    fence_mbar_init();
  }
  __syncthreads();

  const int B = p.block_size;

  if (warp == num_consumers) {
    // =========================== producer warp ===========================
    if (lane == 0) {
      tc::prefetch_tensormap(&kmap);
      tc::prefetch_tensormap(&vmap);
    }
    // the segment being walked: its request (or first member), members, first chunk,
    // chunk count and key count
    int k = pl.start_s, j = pl.start_j, hg = pl.start_hg;
    int s, nmem, skip, units_s, L, qrow = 0;
    auto open_segment = [&](int kk) {
      if (kk < NG) {
        int a, b;
        group_span(p, kk, a, b);
        s = a;
        nmem = b - a;
        skip = 0;
        units_s = shared_chunks(p, kk);
        L = units_s * kTPS;
      } else {
        s = kk - NG;
        nmem = 1;
        skip = own_skip(p, s);
        L = decode_len(p, s);
        if (kQSlots) qrow = __ldg(p.qsl + s);
        units_s = max(units_of(L) - skip, 0);
      }
    };
    open_segment(k);
    // block ids come from a window of 32 consecutive entries of the walked request's table
    // row, one entry a lane, refilled when a stage's boxes leave it (once per 32 blocks or
    // segment) instead of one dependent load per stage
    int win_s = -1, win_base = 0;
    int32_t win = -1;
    int stage = 0, qord = 0;  // qord: segments started in this CTA (query slot qord % 2)
    uint32_t phase = 0;
    for (int64_t u = u_begin; u < u_end; ++u) {
      const int64_t u0 = u - j, u1 = u0 + units_s;
      int flags = 0;
      if (u == u_begin || j == 0) flags |= kFirst;
      if (u == u_end - 1 || j == units_s - 1) flags |= kLast;
      if (u0 >= u_begin) flags |= kSeqStart;
      if (u1 <= u_end) flags |= kSeqEnd;
      const int pos0 = (skip + j) * kTPS;
      const int valid = min(kTPS, L - pos0);
      const int32_t* bt = p.block_table + int64_t(s) * p.max_blocks_per_seq;
      // Fused KV write (decode-only batches without groups, 16-bit caches): at a request's
      // last unit the consumers patch the new token's row (position L - 1) into the stage
      // and store it to its slot; a slot that is not that position's is written here.
      int64_t wslot = -1;
      if (!GROUPED && p.k_new && j == units_s - 1) {
        const int qrow = __ldg(p.qsl + s);
        const int64_t slot = __ldg(p.slot_mapping + qrow);
        const int64_t at = int64_t(__ldg(bt + (L - 1) / B)) * B + (L - 1) % B;
        const int64_t row_bytes = int64_t(p.num_kv_heads) * D * C::EL;
        if (slot >= 0 && slot == at && slot < p.num_blocks * B) {
          wslot = slot;
        } else if (slot >= 0) {
          if (lane == 0 && slot != at) raise_error(p.err, PA_DEVERR_SLOT_MISMATCH);
          if (slot < p.num_blocks * B) {
            const int64_t slice = int64_t(HG) * D * C::EL;
            const int64_t src_off = int64_t(qrow) * row_bytes + hg * slice;
            const int64_t dst_off = slot * row_bytes + hg * slice;
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
      // lane b < NBOX: the box of tokens [pos0 + b * BT, pos0 + b * BT + BT) (one block)
      const int bi0 = pos0 / B, bi_last = (pos0 + (C::NBOX - 1) * BT) / B;  // table indices of the boxes
      if (s != win_s || bi0 < win_base || bi_last >= win_base + 32) {  // warp-uniform
        win_s = s;
        win_base = bi0;
        win = win_base + lane < p.max_blocks_per_seq ? __ldg(bt + win_base + lane) : -1;
      }
      const int32_t blk_l = __shfl_sync(0xffffffffu, win, (pos0 + min(lane, C::NBOX - 1) * BT) / B - win_base);
      bool have = false, bad = false;
      int y = 0;
      if (lane < C::NBOX && lane * BT < valid) {
        const int pos = pos0 + lane * BT;
        const int64_t blk = blk_l;
        bad = blk < 0 || blk >= p.num_blocks;
        have = !bad;
        y = int(blk * B + pos % B);
      }
      const int nhave = __popc(__ballot_sync(0xffffffffu, have));
      const bool any_bad = __any_sync(0xffffffffu, bad);
      if (any_bad) flags |= kBad;
      const int qslot = (qsm && (flags & kFirst) && nmem == 1) ? (qord & 1) : -1;
      int ok = 1;
      if (lane == 0) {
        ok = mbar_wait(empty0 + 8 * stage, phase ^ 1) ? 1 : 0;
        if (ok && qslot >= 0) ok = mbar_wait(qbar0 + 8 * qslot, ((qord >> 1) & 1) ^ 1) ? 1 : 0;
      }
      if (qslot >= 0) ++qord;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) {
        raise_error(p.err, PA_DEVERR_TIMEOUT);
        break;
      }
      if (lane == 0) {
        if (any_bad) raise_error(p.err, PA_DEVERR_BLOCK_RANGE);
        MmaDesc d;
        d.s = s;
        d.hg = hg;
        d.j = j;
        d.valid = valid;
        d.flags = flags;
        d.seg = k;
        d.nmem = nmem;
        d.pos0 = pos0;
        d.wslot = wslot;
        d.pad = skip;
        desc[stage] = d;
        uint32_t tx = uint32_t(nhave) * C::HALVES * 2 * C::box_bytes(HG);
        // a segment's first stage here also brings its query rows (heads of this head group
        // of one token: contiguous) and, when the segment ends here with a fused write, the
        // new token's K and V rows of the head group
        const uint32_t qb = uint32_t(HG * G * D) * 2u, nb = uint32_t(HG * D) * 2u;
        const bool with_new = qslot >= 0 && p.k_new && (flags & kSeqEnd);
        if (qslot >= 0) tx += qb + (with_new ? 2u * nb : 0u);
        mbar_arrive_expect_tx(full0 + 8 * stage, tx);
        if (qslot >= 0) {
          const uint32_t dst = qslot0 + uint32_t(qslot) * uint32_t(p.q_slot);
          bulk_g2s(dst, static_cast<const char*>(p.q) + (int64_t(qrow) * p.num_heads + int64_t(hg) * HG * G) * D * 2,
                   qb, full0 + 8 * stage);
          if (with_new) {
            const int64_t off = (int64_t(qrow) * p.num_kv_heads + int64_t(hg) * HG) * D * 2;
            bulk_g2s(dst + qb, p.k_new + off, nb, full0 + 8 * stage);
            bulk_g2s(dst + qb + nb, p.v_new + off, nb, full0 + 8 * stage);
          }
        }
      }
      __syncwarp();
      if (have) {
        const uint32_t kd = base + C::k_off(HG, stage) + uint32_t(lane) * C::box_bytes(HG);
        const uint32_t vd = base + C::v_off(HG, stage) + uint32_t(lane) * C::box_bytes(HG);
#pragma unroll
        for (int h = 0; h < C::HALVES; ++h) {
          tc::tma_load_3d(kd + h * C::half_bytes(HG), &kmap, h * C::INNER, y, hg * HG, full0 + 8 * stage);
          tc::tma_load_3d(vd + h * C::half_bytes(HG), &vmap, h * C::INNER, y, hg * HG, full0 + 8 * stage);
        }
      }
      if (++stage == STAGES) {
        stage = 0;
        phase ^= 1;
      }
      if (++j == units_s && u + 1 < u_end) {
        j = 0;
        if (++hg == p.num_hg) {
          hg = 0;
          do {
            if (++k >= NS) break;  // cannot happen: the plan counted these units
            open_segment(k);
          } while (units_s == 0);
          if (k >= NS) {
            raise_error(p.err, PA_DEVERR_TIMEOUT);
            break;
          }
        }
      }
    }
    return;
  }

  // =========================== consumer warps ===========================
  // warp hk = KV head within the group; MMA rows = the G query heads of its KV head for
  // each of the stage's nmem requests (row r: request r / G, head r % G). Lane (g, t):
  // g = lane / 4 is an MMA row (g and g + 8) / token / dim index, t = lane % 4 a column pair.
  const int hk = warp;
  const int g = lane >> 2, t = lane & 3;
  const int Hq = p.num_heads;
  uint32_t qa0[C::KC], qa2[C::KC];  // A fragments of rows g (and, GROUPED, g + 8: qa1, qa3)
  uint32_t qa1[GROUPED ? C::KC : 1], qa3[GROUPED ? C::KC : 1];
  uint4 knew = make_uint4(0u, 0u, 0u, 0u), vnew = knew;  // fused write: this lane's 16 bytes of the new row
  constexpr int kRowChunks = D * C::EL / 16;               // 16-byte pieces of one head's row
  float o[C::NT][4];
  float mrun0 = -INFINITY, lpart0 = 0.f, mrun1 = -INFINITY, lpart1 = 0.f;
  const float cscale = p.scale_log2;
  const float v_scale = p.v_scale;
  const int rmax = p.rmax;

  // All KC chunks of one MMA row of q -> its A fragments (zero past nrows): the row's
  // token is looked up once, then every chunk's load is issued before any is used.
  auto load_q = [&](int row, int nrows, int s0, int hgi, uint32_t (&lo)[C::KC], uint32_t (&hi)[C::KC]) {
    const bool have = row < nrows;
    const int r = have ? row : 0;
    const int qrow = have ? __ldg(p.qsl + s0 + r / G) : 0;
    const int qh = (hgi * HG + hk) * G + r % G;
    const T* qp = reinterpret_cast<const T*>(p.q) + (int64_t(qrow) * Hq + qh) * D;
    if constexpr (C::kF16) {  // dims 4t .. 4t+3 (see the K fragments); bf16 -> f16, exact in range
      uint2 w[C::KC];
#pragma unroll
      for (int kc = 0; kc < C::KC; ++kc)
        w[kc] = have ? __ldg(reinterpret_cast<const uint2*>(qp + 16 * kc + 4 * t)) : make_uint2(0u, 0u);
#pragma unroll
      for (int kc = 0; kc < C::KC; ++kc) {
        lo[kc] = pack_f16(__uint_as_float(w[kc].x << 16), __uint_as_float(w[kc].x & 0xffff0000u));
        hi[kc] = pack_f16(__uint_as_float(w[kc].y << 16), __uint_as_float(w[kc].y & 0xffff0000u));
      }
    } else {  // dims 2t, 2t+1 and 8 + 2t, 9 + 2t (the standard fragment)
#pragma unroll
      for (int kc = 0; kc < C::KC; ++kc) {
        lo[kc] = have ? __ldg(reinterpret_cast<const uint32_t*>(qp + 16 * kc + 2 * t)) : 0u;
        hi[kc] = have ? __ldg(reinterpret_cast<const uint32_t*>(qp + 16 * kc + 8 + 2 * t)) : 0u;
      }
    }
  };

  // The same fragments from this segment's query slot (row g = query head hk * G + g of
  // the head group; rows past G are zero).
  int qord = 0, qcur = 0;  // segments started in this CTA; the current one's slot
  auto load_q_slot = [&](uint32_t (&lo)[C::KC], uint32_t (&hi)[C::KC]) {
    const bool have = g < G;
    const uint32_t row = qslot0 + uint32_t(qcur) * uint32_t(p.q_slot) + uint32_t((hk * G + (have ? g : 0)) * D * 2);
#pragma unroll
    for (int kc = 0; kc < C::KC; ++kc) {
      if constexpr (C::kF16) {
        const uint2 w = have ? lds64(row + uint32_t(16 * kc + 4 * t) * 2u) : make_uint2(0u, 0u);
        lo[kc] = pack_f16(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xffff0000u));
        hi[kc] = pack_f16(__uint_as_float(w.y << 16), __uint_as_float(w.y & 0xffff0000u));
      } else {
        lo[kc] = have ? lds32(row + uint32_t(16 * kc + 2 * t) * 2u) : 0u;
        hi[kc] = have ? lds32(row + uint32_t(16 * kc + 8 + 2 * t) * 2u) : 0u;
      }
    }
  };

  int stage = 0;
  uint32_t phase = 0;
  for (int64_t u = u_begin; u < u_end; ++u) {
    if (!mbar_wait(full0 + 8 * stage, phase)) {
      raise_error(p.err, PA_DEVERR_TIMEOUT);
      return;
    }
    const MmaDesc d = desc[stage];
    const int nrows = d.nmem * G;
    if (d.flags & kFirst) {
      if (qsm && d.nmem == 1) {
        qcur = qord & 1;
        ++qord;
        load_q_slot(qa0, qa2);
        if (!p.k_new) {  // nothing else is read from the slot: hand it back now
          __syncwarp();
          if (lane == 0) mbar_arrive(qbar0 + 8 * qcur);
        }
      } else {
        load_q(g, nrows, d.s, d.hg, qa0, qa2);
      }
      if constexpr (GROUPED) load_q(g + 8, nrows, d.s, d.hg, qa1, qa3);
#pragma unroll
      for (int i = 0; i < C::NT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
      mrun0 = mrun1 = -INFINITY;
      lpart0 = lpart1 = 0.f;
      if constexpr (!C::kF16 && !GROUPED) {
        if (!qsm && p.k_new && (d.flags & kSeqEnd) && lane < kRowChunks) {  // this CTA ends the request
          const int qrow = __ldg(p.qsl + d.s);
          const int64_t off = (int64_t(qrow) * p.num_kv_heads + d.hg * HG + hk) * D * C::EL + lane * 16;
          knew = __ldg(reinterpret_cast<const uint4*>(p.k_new + off));
          vnew = __ldg(reinterpret_cast<const uint4*>(p.v_new + off));
        }
      }
    }
    const int valid = (d.flags & kBad) ? 0 : d.valid;
    const uint32_t kb = base + C::k_off(HG, stage), vb = base + C::v_off(HG, stage);
    if constexpr (!C::kF16 && !GROUPED) {
      if (d.wslot >= 0) {  // fused write: the new row into the stage (row valid - 1) and its slot
        if (lane < kRowChunks) {
          if (qsm) {  // the rows came with the segment's first stage, after its query rows
            const uint32_t nrow = qslot0 + uint32_t(qcur) * uint32_t(p.q_slot) + uint32_t(HG * G * D * 2) +
                                  uint32_t(hk * D * 2 + lane * 16);
            knew = lds128(nrow);
            vnew = lds128(nrow + uint32_t(HG * D * 2));
          }
          const int half = (lane * 16) / 128, ch = ((lane * 16) % 128) / 16;
          const uint32_t so = C::at(HG, half, d.valid - 1, hk, ch);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(kb + so), "r"(knew.x), "r"(knew.y),
                       "r"(knew.z), "r"(knew.w)
                       : "memory");
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(vb + so), "r"(vnew.x), "r"(vnew.y),
                       "r"(vnew.z), "r"(vnew.w)
                       : "memory");
          const int64_t go = d.wslot * (int64_t(p.num_kv_heads) * D * C::EL) + int64_t(d.hg * HG + hk) * D * C::EL +
                             lane * 16;
          *reinterpret_cast<uint4*>(p.k_cache_w + go) = knew;
          *reinterpret_cast<uint4*>(p.v_cache_w + go) = vnew;
        }
        __syncwarp();
      }
    }

    // ---- S = Q K^T: n tile j = tokens 8j .. 8j + 7, this lane's B column = token 8j + g
    // two accumulators per tile (even / odd k chunks) halve the MMA dependency chain
    float sacc[2][4], sacc2[2][4];
#pragma unroll
    for (int jj = 0; jj < 2; ++jj)
#pragma unroll
      for (int e = 0; e < 4; ++e) sacc[jj][e] = sacc2[jj][e] = 0.f;
    // ldmatrix: lane l addresses row l % 8 (a token) of matrix l / 8; matrices are
    // (tokens 0-7 | 8-15) x (two 16-byte columns), so one x4 load gives B fragments for
    // both token tiles. bf16: a column holds 8 dims, fragments are standard (b0 = dims
    // 2t, 2t+1 of chunk kc, b1 = dims 8 + 2t, 9 + 2t). E4M3: a column holds 16 dims = one
    // chunk; a lane's 4 codes are dims 4t .. 4t+3, so k = 2t + e <-> dim 4t + e and
    // k = 2t + 8 + e <-> dim 4t + 2 + e (Q uses the same map).
    const int lm = lane >> 3, lr = lane & 7;
#pragma unroll
    for (int kc = 0; kc < C::KC; ++kc) {
      const uint32_t a1 = GROUPED ? qa1[GROUPED ? kc : 0] : 0u, a3 = GROUPED ? qa3[GROUPED ? kc : 0] : 0u;
      if constexpr (C::kF16) {
        if ((kc & 1) == 0) {  // chunks kc, kc + 1 of tokens 0-7 and 8-15
          const uint32_t a1n = GROUPED ? qa1[GROUPED ? kc + 1 : 0] : 0u;
          const uint32_t a3n = GROUPED ? qa3[GROUPED ? kc + 1 : 0] : 0u;
          uint32_t r0, r1, r2, r3;
          // token rows: tile 0 = tokens 0, 1, 4, 5, .., tile 1 = 2, 3, 6, 7, ..: the lane's
          // scores then cover tokens 4t .. 4t+3, the order in which P V reads V (below)
          ldsm_x4(kb + C::at(HG, 0, 4 * (lr >> 1) + (lr & 1) + 2 * (lm & 1), hk, kc + (lm >> 1)), r0, r1, r2, r3);
          uint32_t k0l, k0h, k1l, k1h, k2l, k2h, k3l, k3h;
          e4m3x4_to_f16x2x2(r0, k0l, k0h);
          e4m3x4_to_f16x2x2(r1, k1l, k1h);
          e4m3x4_to_f16x2x2(r2, k2l, k2h);
          e4m3x4_to_f16x2x2(r3, k3l, k3h);
          mma_16816(sacc[0], qa0[kc], a1, qa2[kc], a3, k0l, k0h, true);
          mma_16816(sacc[1], qa0[kc], a1, qa2[kc], a3, k1l, k1h, true);
          mma_16816(sacc2[0], qa0[kc + 1], a1n, qa2[kc + 1], a3n, k2l, k2h, true);
          mma_16816(sacc2[1], qa0[kc + 1], a1n, qa2[kc + 1], a3n, k3l, k3h, true);
        }
      } else {  // chunk kc: dims 16kc .. 16kc + 15 = 16-byte columns 2kc % 8, +1 of half 16kc / 64
        const int dim = 16 * kc + (lm >> 1) * 8;
        uint32_t r0, r1, r2, r3;
        ldsm_x4(kb + C::at(HG, dim / C::INNER, (lm & 1) * 8 + lr, hk, (dim % C::INNER) / 8), r0, r1, r2, r3);
        mma_16816((kc & 1) ? sacc2[0] : sacc[0], qa0[kc], a1, qa2[kc], a3, r0, r2, false);
        mma_16816((kc & 1) ? sacc2[1] : sacc[1], qa0[kc], a1, qa2[kc], a3, r1, r3, false);
      }
    }
#pragma unroll
    for (int jj = 0; jj < 2; ++jj)
#pragma unroll
      for (int e = 0; e < 4; ++e) sacc[jj][e] += sacc2[jj][e];

    // ---- online softmax over the stage's 16 tokens, rows g (c0, c1) and, GROUPED, g + 8
    // (c2, c3); the lanes of a quad share a row. Without groups nothing of row g + 8 is
    // computed (its MMA rows are zero padding).
    float x[2][4];
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int jj = 0; jj < 2; ++jj)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const bool in = (C::kF16 ? 4 * t + 2 * jj + e : 8 * jj + 2 * t + e) < valid;  // the token
        x[jj][e] = in ? sacc[jj][e] * cscale : -INFINITY;
        mx0 = fmaxf(mx0, x[jj][e]);
        if constexpr (GROUPED) {
          x[jj][2 + e] = in ? sacc[jj][2 + e] * cscale : -INFINITY;
          mx1 = fmaxf(mx1, x[jj][2 + e]);
        }
      }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    // The reference max moves only when a score exceeds it by more than 8 (log2 units; the
    // first finite score always moves it): numerators stay below 2^8, and O and l are
    // rescaled only on those steps (alpha is exactly 1 otherwise).
    const float mnew0 = (mx0 > mrun0 + 8.f) ? mx0 : mrun0;
    const float ms0 = (mnew0 == -INFINITY) ? 0.f : mnew0;
    const float alpha0 = (mnew0 == mrun0) ? 1.f : ex2_ftz(mrun0 - ms0);
    float alpha1 = 1.f, ms1 = 0.f;
    if constexpr (GROUPED) {
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      const float mnew1 = (mx1 > mrun1 + 8.f) ? mx1 : mrun1;
      ms1 = (mnew1 == -INFINITY) ? 0.f : mnew1;
      alpha1 = (mnew1 == mrun1) ? 1.f : ex2_ftz(mrun1 - ms1);
      mrun1 = mnew1;
    }
    float pv[2][4];
    float psum0 = 0.f, psum1 = 0.f;
#pragma unroll
    for (int jj = 0; jj < 2; ++jj)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        pv[jj][e] = ex2_ftz(x[jj][e] - ms0);
        psum0 += pv[jj][e];
        if constexpr (GROUPED) {
          pv[jj][2 + e] = ex2_ftz(x[jj][2 + e] - ms1);
          psum1 += pv[jj][2 + e];
        }
      }
    lpart0 = lpart0 * alpha0 + psum0;
    mrun0 = mnew0;
    if constexpr (GROUPED) {
      lpart1 = lpart1 * alpha1 + psum1;
      if (__any_sync(0xffffffffu, alpha0 != 1.f || alpha1 != 1.f)) {
#pragma unroll
        for (int i = 0; i < C::NT; ++i) {
          o[i][0] *= alpha0;
          o[i][1] *= alpha0;
          o[i][2] *= alpha1;
          o[i][3] *= alpha1;
        }
      }
    } else {
      if (__any_sync(0xffffffffu, alpha0 != 1.f)) {
#pragma unroll
        for (int i = 0; i < C::NT; ++i) {
          o[i][0] *= alpha0;
          o[i][1] *= alpha0;
        }
      }
    }
    // P as the A operand of P V: row g, k = tokens 2t, 2t+1 (a0) and 8 + 2t, 9 + 2t (a2);
    // row g + 8 likewise (a1, a3)
    uint32_t pa0, pa1 = 0u, pa2, pa3 = 0u;
    if constexpr (C::kF16) {
      pa0 = pack_f16(pv[0][0], pv[0][1]);
      pa2 = pack_f16(pv[1][0], pv[1][1]);
      if constexpr (GROUPED) {
        pa1 = pack_f16(pv[0][2], pv[0][3]);
        pa3 = pack_f16(pv[1][2], pv[1][3]);
      }
    } else {
      pa0 = pack_bf16(pv[0][0], pv[0][1]);
      pa2 = pack_bf16(pv[1][0], pv[1][1]);
      if constexpr (GROUPED) {
        pa1 = pack_bf16(pv[0][2], pv[0][3]);
        pa3 = pack_bf16(pv[1][2], pv[1][3]);
      }
    }

    // ---- O += P V. Rows of V past `valid` hold stale or unwritten data: zero them in
    // the B fragments (P is 0 there, but 0 * NaN would not be).
    const bool partial = valid < kTPS;
    if constexpr (C::kF16) {
      // A 16-byte column c of V is a 16-token x 16-dim byte matrix; transposed, lane (g, t)
      // gets tokens 4t .. 4t+3 of dims 16c + g and 16c + 8 + g. P's k slots 2t, 2t+1 and
      // 2t+8, 2t+9 hold tokens 4t, 4t+1 and 4t+2, 4t+3 (the S token order above), so each
      // register's two halves, converted, are the B fragments of tiles 2c and 2c + 1.
      uint32_t vmask = 0xffffffffu;  // bytes of tokens 4t .. 4t+3 that are valid
      if (partial)
        vmask = (4 * t < valid ? 0x000000ffu : 0u) | (4 * t + 1 < valid ? 0x0000ff00u : 0u) |
                (4 * t + 2 < valid ? 0x00ff0000u : 0u) | (4 * t + 3 < valid ? 0xff000000u : 0u);
#pragma unroll
      for (int c2 = 0; c2 < C::KC / 2; ++c2) {
        uint32_t r0, r1, r2, r3;  // columns 2c2 (r0, r1) and 2c2 + 1 (r2, r3)
        ldsm_b8_x2_trans(vb + C::at(HG, 0, lane & 15, hk, 2 * c2 + (lane >> 4)), r0, r1, r2, r3);
        if (partial) {
          r0 &= vmask;
          r1 &= vmask;
          r2 &= vmask;
          r3 &= vmask;
        }
        uint32_t b00, b01, b10, b11, b20, b21, b30, b31;
        e4m3x4_to_f16x2x2(r0, b00, b01);
        e4m3x4_to_f16x2x2(r1, b10, b11);
        e4m3x4_to_f16x2x2(r2, b20, b21);
        e4m3x4_to_f16x2x2(r3, b30, b31);
        mma_16816(o[4 * c2 + 0], pa0, pa1, pa2, pa3, b00, b01, true);
        mma_16816(o[4 * c2 + 1], pa0, pa1, pa2, pa3, b10, b11, true);
        mma_16816(o[4 * c2 + 2], pa0, pa1, pa2, pa3, b20, b21, true);
        mma_16816(o[4 * c2 + 3], pa0, pa1, pa2, pa3, b30, b31, true);
      }
    } else {
      // bf16: ldmatrix.trans, lane l addressing row l % 8 (a token) of matrix l / 8; the
      // matrices are (tokens 0-7 | 8-15) x (dims 8i | 8i + 8) and give b0, b1 of tiles i,
      // i + 1 with the standard fragment (col g <-> dim 8i + g; tokens 2t, 2t+1 | 8+2t, 9+2t)
      const int mi = lane >> 3, rr = lane & 7;
      const int vtok = (mi & 1) * 8 + rr;
      uint32_t lo_mask = 0xffffffffu, hi_mask = 0xffffffffu;
      if (partial) {
        lo_mask = (2 * t < valid ? 0x0000ffffu : 0u) | (2 * t + 1 < valid ? 0xffff0000u : 0u);
        hi_mask = (8 + 2 * t < valid ? 0x0000ffffu : 0u) | (9 + 2 * t < valid ? 0xffff0000u : 0u);
      }
#pragma unroll
      for (int i2 = 0; i2 < C::NT / 2; ++i2) {
        const int dim = 16 * i2 + (mi >> 1) * 8;
        uint32_t r0, r1, r2, r3;
        ldsm_x4_trans(vb + C::at(HG, dim / C::INNER, vtok, hk, (dim % C::INNER) / 8), r0, r1, r2, r3);
        mma_16816(o[2 * i2], pa0, pa1, pa2, pa3, r0 & lo_mask, r1 & hi_mask, false);
        mma_16816(o[2 * i2 + 1], pa0, pa1, pa2, pa3, r2 & lo_mask, r3 & hi_mask, false);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * stage);
    if (++stage == STAGES) {
      stage = 0;
      phase ^= 1;
    }

    if (!(d.flags & kLast)) continue;
    if (qsm && p.k_new && lane == 0) mbar_arrive(qbar0 + 8 * qcur);  // the new rows are written

    // ================= finalize this segment's piece =================
    float l0 = lpart0, l1 = lpart1;
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    if constexpr (GROUPED) {
      l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
      l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    }
    // `out` directly only when this CTA holds the whole request (no shared part, no cut)
    const bool whole = (d.flags & kSeqStart) && (d.flags & kSeqEnd) && d.seg >= NG && d.pad == 0;
    const int64_t slot = c + int64_t(d.seg) * p.num_hg + d.hg;
#pragma unroll
    for (int half_row = 0; half_row < (GROUPED ? 2 : 1); ++half_row) {
      const int row = g + 8 * half_row;
      if (row < nrows) {
        const float l = half_row ? l1 : l0;
        const float mr = half_row ? mrun1 : mrun0;
        const int qrow = __ldg(p.qsl + d.s + row / G);
        const int hq = (d.hg * HG + hk) * G + row % G;
        const float inv = l > 0.f ? v_scale / l : 0.f;
        const int64_t hrow = (slot * HG + hk) * rmax + row;
        const int e0 = 2 * half_row;  // o[i][e0], o[i][e0 + 1]: this row's two columns
        // lane holds dims 8i + 2t, 8i + 2t + 1 of every tile i
#pragma unroll
        for (int i = 0; i < C::NT; ++i) {
          const int dim = 8 * i + 2 * t;
          const float f0 = o[i][e0] * inv, f1 = o[i][e0 + 1] * inv;
          if (whole) {
            *reinterpret_cast<uint32_t*>(reinterpret_cast<T*>(p.out) + (int64_t(qrow) * Hq + hq) * D + dim) =
                pack_bf16(f0, f1);
          } else {
            *reinterpret_cast<float2*>(p.ws_o + hrow * D + dim) = make_float2(f0, f1);
          }
        }
        if (!whole && t == 0) p.ws_lse[hrow] = (l > 0.f) ? mr + __log2f(l) : -INFINITY;
      }
    }
    __syncwarp();
    if (warp == 0 && lane == 0) {
      const int64_t v = int64_t(d.seg) * p.num_hg + d.hg;
      if (d.flags & kSeqStart) {
        p.ws_meta[v].x = int(c);
        p.ws_meta[v].z = pl.units_per_hg;
        // grouped: the chunks the segment skips (its group's shared ones), for the merge
        p.ws_meta[v].w = GROUPED ? d.pad : __ldg(p.qsl + d.s);
      }
      if (d.flags & kSeqEnd) p.ws_meta[v].y = int(c);
    }
  }
}

// ---------------------------------------------------------------- merge with groups
// Keys of request s as decode_len counts them, without raising errors (the split-K kernel
// has raised them already).
__device__ __forceinline__ int decode_len_quiet(const DecodeParams& p, int s) {
  if (__ldg(p.qsl + s + 1) - __ldg(p.qsl + s) != 1) return 0;
  const int L = min(__ldg(p.seq_lens + s), p.max_blocks_per_seq * p.block_size);
  return L > 0 ? L : 0;
}

// One CTA per (request, head group): the request's own pieces and, when its group's shared
// prefix ran as a segment, that segment's pieces (rows of this member), combined by their
// log-sum-exps. (Without groups the common merge kernel runs instead.) Loads that do not
// depend on one another are issued together -- the request's descriptor, group and length;
// then the group's span and descriptor (the split-K kernel left the skipped chunk count in
// the request's own descriptor; only a request without own chunks reads the members'
// lengths) -- and the pieces are merged as in the common merge kernel.
template <typename T, int D>
__global__ void __launch_bounds__(1024) decode_merge_grouped_kernel(const __grid_constant__ DecodeParams p) {
  griddep_launch_dependents();  // the next kernel may be scheduled; it still waits for this grid
  griddep_wait();
  const int s = blockIdx.x / p.num_hg, hg = blockIdx.x % p.num_hg;
  const int NG = p.num_groups, G = p.group, HG = p.hg_size;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
  const int vo = (NG + s) * p.num_hg + hg;
  const int4 mo = p.ws_meta[vo];
  const int gi = NG > 0 ? __ldg(p.seq_group + s) : -1;
  const int Ls = decode_len_quiet(p, s);
  const int q0 = __ldg(p.qsl + s);
  // the shared segment this request's leading chunks ran in (own_skip of the split-K kernel)
  int skip = 0, member = 0, vs = -1;
  int4 msh = make_int4(-1, -1, 0, 0);
  if (gi >= 0 && gi < NG) {
    int a, b;
    group_span(p, gi, a, b);
    const int4 m = p.ws_meta[gi * p.num_hg + hg];
    if (s >= a && s < b && b - a >= 2 && (b - a) * G <= 16) {  // at most 8 members
      if (mo.x >= 0) {  // the request's own segment ran: its descriptor holds the skip
        skip = mo.w;
      } else {  // no own chunks: the skip from the members' lengths, as the split-K kernel
        const int shl = __ldg(p.shared_len + gi);
        int lim = lane < b - a ? decode_len_quiet(p, a + lane) : INT_MAX;
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) lim = min(lim, __shfl_xor_sync(0xffffffffu, lim, o));
        skip = max(min(lim, shl), 0) / kTPS;
      }
      if (skip > 0) {
        member = s - a;
        vs = gi * p.num_hg + hg;
        msh = m;
      }
    }
  }
  if (skip == 0 && (mo.x < 0 || mo.x == mo.y)) return;  // nothing here / one CTA wrote `out` itself
  if (Ls == 0) return;
  auto bad = [&](const int4& m) { return m.x >= 0 && (m.y >= p.num_ctas || m.x > m.y || m.z <= 0); };
  if (bad(mo) || bad(msh) || (skip > 0 && msh.x < 0)) {
    if (threadIdx.x == 0) raise_error(p.err, PA_DEVERR_TIMEOUT);
    return;
  }
  const int64_t C = p.num_ctas;
  const int units = mo.x >= 0 ? mo.z : msh.z;
  const int64_t U = int64_t(units) * p.num_hg;
  T* out = reinterpret_cast<T*>(p.out);
  constexpr int D4 = D / 4;
  const int n_own = mo.x >= 0 ? mo.y - mo.x + 1 : 0;
  const int n_sh = (skip > 0 && msh.x >= 0) ? msh.y - msh.x + 1 : 0;
  const int npieces = n_own + n_sh;
  // piece i -> its workspace row base, or -1 for a CTA whose range is empty (no piece)
  auto piece_row = [&](int i) -> int64_t {
    const bool own = i < n_own;
    const int64_t cc = own ? mo.x + i : msh.x + (i - n_own);
    if (cc * U / C == (cc + 1) * U / C) return -1;
    return own ? ((cc + vo) * HG) * p.rmax : ((cc + vs) * HG) * p.rmax + member * G;
  };
  for (int head = warp; head < HG * G; head += nwarps) {
    const int hk = head / G, h = head % G, off = hk * p.rmax + h;
    // lane i: piece i's row and log-sum-exp (32 pieces at a time)
    int64_t r0 = lane < npieces ? piece_row(lane) : -1;
    float l0 = r0 >= 0 ? p.ws_lse[r0 + off] : -INFINITY;
    float M = l0;
    for (int i = 32 + lane; i < npieces; i += 32) {
      const int64_t r = piece_row(i);
      if (r >= 0) M = fmaxf(M, p.ws_lse[r + off]);
    }
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, m));
    const float Ms = (M == -INFINITY) ? 0.f : M;
    float acc[4] = {0.f, 0.f, 0.f, 0.f}, wsum = 0.f;
    for (int i0 = 0; i0 < npieces; i0 += 32) {
      int64_t rl = r0;
      float ll = l0;
      if (i0 > 0) {
        rl = i0 + lane < npieces ? piece_row(i0 + lane) : -1;
        ll = rl >= 0 ? p.ws_lse[rl + off] : -INFINITY;
      }
      const float wl = exp2f(ll - Ms);  // 0 for an empty range or an empty piece
      const int n = min(32, npieces - i0);
      for (int b = 0; b < n; b += 4) {
        float w[4];
        float4 ov[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          w[q] = __shfl_sync(0xffffffffu, wl, b + q);
          const int64_t rq = __shfl_sync(0xffffffffu, rl, b + q);
          if (b + q >= n) w[q] = 0.f;
          ov[q] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (lane < D4 && w[q] > 0.f) ov[q] = *reinterpret_cast<const float4*>(p.ws_o + (rq + off) * D + lane * 4);
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          acc[0] += w[q] * ov[q].x;
          acc[1] += w[q] * ov[q].y;
          acc[2] += w[q] * ov[q].z;
          acc[3] += w[q] * ov[q].w;
          wsum += w[q];
        }
      }
    }
    if (lane < D4) {
      const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[e] *= inv;
      RowVec<T, 4>::store(out + (int64_t(q0) * p.num_heads + (hg * HG + hk) * G + h) * D + lane * 4, acc);
    }
  }
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }();
  return fn;
}

// The cache as (dim, token, KV head) -- strides decrease, so a box of {128 bytes of dims,
// bt tokens, hg heads} lands as [head][token][128 B].
bool make_cache_map(CUtensorMap* m, const void* cache, int el, int D, int64_t slots, int hkv, int bt, int hg) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {cuuint64_t(D), cuuint64_t(slots), cuuint64_t(hkv)};
  const cuuint64_t strides[2] = {cuuint64_t(hkv) * D * el, cuuint64_t(D) * el};
  const cuuint32_t box[3] = {cuuint32_t(128 / el), cuuint32_t(bt), cuuint32_t(hg)};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, el == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 3,
            const_cast<void*>(cache), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename KV, int D, int BT, bool GROUPED>
cudaError_t run(const AttnArgs& a, int hg, int num_ctas, cudaStream_t stream) {
  using C = MmaCfg<KV, D, BT>;
  CUtensorMap km, vm;
  const int64_t slots = a.num_blocks * a.block_size;
  if (!make_cache_map(&km, a.k_cache, C::EL, D, slots, a.num_kv_heads, BT, hg) ||
      !make_cache_map(&vm, a.v_cache, C::EL, D, slots, a.num_kv_heads, BT, hg))
    return cudaErrorInvalidValue;
  DecodeParams p = fill_decode_params(a, hg, 1, num_ctas, D);
  if (C::EL == 2 && a.k_new != nullptr && !GROUPED) {
    p.k_new = static_cast<const char*>(a.k_new);
    p.v_new = static_cast<const char*>(a.v_new);
    p.slot_mapping = a.slot_mapping;
  }
  if (C::EL == 1) {
    p.scale_log2 *= a.k_scale;
    p.v_scale = a.v_scale;
  }
  if (GROUPED) {  // pieces of every segment, 16 rows a KV head
    p.seq_group = a.seq_group;
    p.group_start = a.group_start;
    p.shared_len = a.shared_len;
    p.num_groups = a.num_groups;
    p.rmax = 16;
    const int64_t nseg = int64_t(a.num_groups) + a.num_seqs;
    const int64_t pslots = int64_t(num_ctas) + nseg * p.num_hg;
    const int64_t rows = pslots * hg * 16;
    char* ws = static_cast<char*>(a.workspace);
    p.ws_o = reinterpret_cast<float*>(ws);
    p.ws_lse = reinterpret_cast<float*>(ws + rows * D * 4);
    p.ws_meta = reinterpret_cast<int4*>(ws + rows * D * 4 + ((rows * 4 + 15) / 16) * 16);
  }
  // query slots when they fit beside the stages (bf16 caches; with E4M3 caches the slots,
  // which push shared memory to the next carveout, measured slower than global loads)
  uint32_t q_slot = 0;
  if (C::EL == 2 && !a.host_inputs) {
    q_slot = uint32_t(hg * p.group * D * 2) + (p.k_new ? uint32_t(2 * hg * D * 2) : 0u);
    q_slot = (q_slot + 15) / 16 * 16;
    if (C::total(hg, q_slot) > uint32_t(kSmemLimit)) q_slot = 0;
  }
  p.q_slot = int(q_slot);
  const size_t smem = C::total(hg, q_slot);
  auto kern = decode_mma_kernel<__nv_bfloat16, D, KV, BT, GROUPED>;
  cudaError_t e = ensure_smem<decode_mma_kernel<__nv_bfloat16, D, KV, BT, GROUPED>>(smem);
  if (e != cudaSuccess) return e;
  e = launch_pdl(kern, dim3(num_ctas), dim3((hg + 1) * 32), smem, stream, p, km, vm);
  if (e != cudaSuccess) return e;
  if (!GROUPED) return launch_merge<__nv_bfloat16, D>(p, stream, a.merge_pdl);
  // 16 warps (a warp per head, looping): the kernel's 64 registers a thread let two such
  // CTAs share an SM, so every member's merge runs in one wave (1024 threads: two waves;
  // shared-prefix batch 89.0 -> 86.9 us, bit-identical)
  const int threads = 32 * (hg * p.group < 16 ? hg * p.group : 16);
  const dim3 mgrid(unsigned(int64_t(a.num_seqs) * p.num_hg));
  if (!a.merge_pdl) {  // plain stream order, as launch_merge
    decode_merge_grouped_kernel<__nv_bfloat16, D><<<mgrid, dim3(threads), 0, stream>>>(p);
    return cudaGetLastError();
  }
  return launch_pdl(decode_merge_grouped_kernel<__nv_bfloat16, D>, mgrid, dim3(threads), 0, stream, p);
}

template <typename KV, int D, int BT>
cudaError_t run_g(const AttnArgs& a, int hg, int num_ctas, cudaStream_t stream) {
  return a.num_groups > 0 ? run<KV, D, BT, true>(a, hg, num_ctas, stream)
                          : run<KV, D, BT, false>(a, hg, num_ctas, stream);
}

}  // namespace

bool decode_mma_supported(const AttnArgs& a, int hg) {
  const int B = a.block_size, D = a.head_dim;
  const int G = a.num_heads / a.num_kv_heads;
  if (a.dtype != PA_BF16 || hg < 1 || G > 8) return false;
  if (a.k_new != nullptr && a.cache_dtype != PA_BF16) return false;  // no fused write into E4M3
  if (a.k_new != nullptr && a.num_groups > 0) return false;          // nor with groups
  if (!(B == 8 || (B % 16 == 0 && B <= 1024))) return false;
  if (a.num_blocks * B > 0x7fffffff) return false;  // TMA token coordinates are int32
  if (a.cache_dtype == PA_BF16) {
    if (D != 64 && D != 128) return false;
  } else if (a.cache_dtype == PA_FP8_E4M3) {
    if (D != 128) return false;
  } else {
    return false;
  }
  return encode_fn() != nullptr;
}

cudaError_t launch_decode_mma(const AttnArgs& a, int hg, int num_ctas, cudaStream_t stream) {
  const bool bt8 = a.block_size == 8;
  if (a.cache_dtype == PA_FP8_E4M3)
    return bt8 ? run_g<Fp8E4M3, 128, 8>(a, hg, num_ctas, stream) : run_g<Fp8E4M3, 128, 16>(a, hg, num_ctas, stream);
  if (a.head_dim == 64)
    return bt8 ? run_g<__nv_bfloat16, 64, 8>(a, hg, num_ctas, stream)
               : run_g<__nv_bfloat16, 64, 16>(a, hg, num_ctas, stream);
  return bt8 ? run_g<__nv_bfloat16, 128, 8>(a, hg, num_ctas, stream)
             : run_g<__nv_bfloat16, 128, 16>(a, hg, num_ctas, stream);
}

size_t decode_grouped_workspace_bytes(int num_seqs, int num_groups, int num_kv_heads, int head_dim, int hg,
                                      int num_ctas) {
  if (hg < 1) return 0;
  const int64_t num_hg = num_kv_heads / hg;
  const int64_t nseg = int64_t(num_groups) + num_seqs;
  const int64_t rows = (int64_t(num_ctas) + nseg * num_hg) * hg * 16;
  return size_t(rows * head_dim * 4 + ((rows * 4 + 15) / 16) * 16 + nseg * num_hg * 16);
}

}  // namespace pa
