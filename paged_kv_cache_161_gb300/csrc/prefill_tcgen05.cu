// Chunked-prefill attention on the tensor cores (tcgen05, TMEM accumulators, TMA).
//
// What it computes: vLLM 0.10.0 flow page, 3.2 Scheduler (a long prefill is cut into
// chunks that run in one batch with decodes; prefill is compute-bound) and 3.5 Attention
// (requests delimited by query_start_loc, K/V found through block_table); VLLM overview
// page, 2.1 (causal mask). Query j of a request with q_len queries and L keys sits at
// position L - q_len + j and sees keys 0..L - q_len + j; its chunk's own K/V are already
// in the cache (written by pa_kv_write).
//
// Tile: 128 rows = (128 / G) query tokens x the G query heads that share one KV head, so
// each K/V tile feeds all of them. A CTA works on a pair of consecutive tiles of one
// (request, KV head) at a time; both consume the same K/V steps of 128 keys:
//   S_x = Q_x.K^T  (8 x tcgen05.mma 128x128x16, bf16 in, f32 accumulate in TMEM)
//   softmax_x      one thread per row in registers: two passes over S in TMEM (row max,
//                  then p = 2^(s * scale * log2 e - m) with one packed FMA per pair and
//                  ex2.approx.ftz), lazy rescaling of O only when the row max grows by
//                  more than 2^8, P packed to bf16 and written back over S
//   O_x += P_x.V   (8 x tcgen05.mma 128xDx16, A = P from TMEM, B = V as an MN-major
//                  shared-memory operand), O in TMEM; issued in two halves of 4, keys
//                  64..127 as soon as the softmax has stored their P, then keys 0..63
// The two tiles ping-pong: while tile A's softmax runs, the tensor core does tile B's
// P.V and next Q.K, and the other way round. E4M3 caches (head_dim 128) take the same
// path with f16 operands: the producer warps and a converter warp turn each step's codes,
// and the pair's bf16 queries, into f16 tiles in shared memory.
//
// Roles (352 threads, 384 with E4M3 caches; one CTA per SM, persistent: pairs enumerated
// with the requests longest first and each request's last tiles first; CTA c starts with
// pair c and then draws the next unclaimed pair from a grid-wide counter whenever it needs
// one):
//   warps 0-3 / 4-7  softmax + epilogue of tile A / tile B (thread = row = TMEM lane);
//   warp 8           draws the pairs (ring of two slots in shared memory, read by every
//                    other role); TMA: both Q tiles once per pair (3-D box {64 dims, G heads, 128 / G
//                    tokens}, 128-byte swizzle) and K (2-deep ring, one 3-D box per
//                    physical block and 64-dim half, block-table entries read by the
//                    warp's lanes one step ahead);
//   warp 10          TMA: V (2-deep ring) the same way;
//   warp 9           allocates the 512 TMEM columns (S_A, S_B, O_A, O_B) and one thread
//                    issues the MMAs of both tiles, tracking completion with tcgen05.commit
//                    (one thread for both keeps the tiles out of phase: a thread per tile
//                    measured 205 us against 170 us on the mixed batch's prefill part);
//   warp 11          E4M3 caches only: converts the last rows of every K and V step and
//                    tile B's queries (warps 8 and 10 convert the rest of their operand).
// Every wait is bounded; on a timeout the kernel sets an error bit and leaves after its
// copies and MMAs in flight have landed, freeing TMEM.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "launch.h"
#include "tcgen05.cuh"

namespace pa {
namespace {

constexpr int kBM = 128;             // rows per tile
constexpr int kBN = 128;             // keys per step
constexpr int kMaxSeqs = 4096;       // requests per call this kernel accepts
constexpr int kThreads = 11 * 32;    // 8 softmax warps (4 per tile), Q/K TMA, MMA, V TMA
constexpr int kWarpQK = 8, kWarpMMA = 9, kWarpV = 10;
// E4M3 caches: one more warp converts half of each step's codes (and half the queries) to
// f16 beside the two producers (384 threads x 168 registers fit the SM's 65536)
constexpr int kWarpCvt = 11;
// rows [0, kCvtSplitK) of a K step and [0, kCvtSplitV) of a V step: the producer of that
// operand, which also issues its copies and waits for them (the K producer also converts
// tile A's queries); the rest: the converter warp, for both operands. Mixed-batch E4M3
// prefill by split (same box, bit-identical): K/V 48/48: 259.0 us, 56/56: 241.9, 64/64:
// 228.9, 72/72: 230.2, 84/84: 244.0; 64/72: 226.4, 64/76: 230.2, 64/80: 233.2, 68/72:
// 230.4, 56/72: 231.3, 56/64: 235.0.
constexpr int kCvtSplitK = 64, kCvtSplitV = 72;
template <bool F8>
__host__ __device__ constexpr int threads_of() { return F8 ? kThreads + 32 : kThreads; }
constexpr uint32_t kTmemCols = 512;  // S_A, S_B, O_A, O_B: 128 columns each
constexpr uint32_t kHalf = 128 * 128;  // bytes of a 128-row x 64-element bf16 half tile

struct PrefillParams {
  void* out;
  const int32_t* block_table;
  const int32_t* seq_lens;
  const int32_t* qsl;
  unsigned int* err;
  int* sched;  // pair counter, zero before the first launch of the call
  // first_static: CTA c takes pair c first, then tickets; else every pair is a ticket.
  // A ticket is ticket_base + the counter's next value (ticket_base: the grid size of the
  // call's first launch, whose CTAs took pairs 0 .. ticket_base - 1 statically).
  int first_static;
  int ticket_base;
  int64_t num_blocks;
  int max_blocks_per_seq;
  int num_seqs;
  int num_heads;
  int num_kv_heads;
  int block_size;
  float scale_log2;  // softmax scale x log2(e) (x k_scale over an E4M3 cache)
  float out_scale;   // 1, or v_scale over an E4M3 cache
  int out_v8;        // out is 32-byte aligned: the epilogue stores 32 bytes per instruction
};

template <int D>
struct Layout {
  static constexpr int NH = D / 64;  // 64-element halves of the head dim
  static constexpr uint32_t Q = 0;                      // tile A, tile B
  static constexpr uint32_t K = Q + 2 * NH * kHalf;     // 2 stages
  static constexpr uint32_t V = K + 2 * NH * kHalf;     // 2 stages
  static constexpr uint32_t PFX = V + 2 * NH * kHalf;   // int[kMaxSeqs + 8]
  static constexpr uint32_t ORD = PFX + (kMaxSeqs + 8) * 4;  // int[kMaxSeqs + 8], right after PFX
  static constexpr uint32_t BAR = ORD + (kMaxSeqs + 8) * 4;
  static constexpr int NBAR = 28;
  static constexpr uint32_t MISC = BAR + NBAR * 8;       // tmem base, abort flag
  static constexpr uint32_t RING = MISC + 16;            // RingSlot[2]: the next pairs, for every role
  static constexpr uint32_t BYTES = RING + 128;
  static constexpr uint32_t SMEM = BYTES + 1024;         // + alignment slack
};

// barrier indices (X = tile A or B: index + X)
enum : int {
  // K stage s released (both tiles' Q.K on it landed) -- tile B's Q.K is issued last on a
  // stage, so the same completion tells tile B's softmax that S_B is ready and the Q/K
  // producer that the pair's queries are free after its last step; V stage s released
  // (both tiles' P.V landed) -- which also tells that P.V(B) is done. Tile A has its own
  // S-ready and P.V-done barriers. One commit per signal: a commit issued before the
  // previous one has retired stalls the issuing thread.
  bQFull = 0, bKFull0, bKFull1, bKEmpty0, bKEmpty1, bVFull0, bVFull1, bVEmpty0, bVEmpty1,
  bSFullA, bPFull0, bPFull1, bPVDoneA, bOEmpty0, bOEmpty1, bMmaDone,
  bPHalf0, bPHalf1,  // P of keys 64..127 is in TMEM (the first half of P.V may start)
  bRingFull0, bRingFull1, bRingEmpty0, bRingEmpty1,
  // E4M3 caches: the producer has converted the stage's codes (Q: its bf16 values) to f16
  bQReady, bKReady0, bKReady1, bVReady0, bVReady1
};
// roles that take each pair from the ring: the V producer, the MMA thread, 8 softmax warps
// (and, E4M3 caches, the converter warp)
constexpr uint32_t kRingTakers = 10;
static_assert(bVReady1 < Layout<128>::NBAR && bVReady1 < Layout<64>::NBAR,
              "every barrier index needs a slot in the shared-memory layout");

// A pair of consecutive query tiles of one (request, KV head); they share every K/V step.
struct Pair {
  int s, hk, qs, L, leff, nt;
  int q0[2], nq[2], pos0[2];
};

// A pair as the Q/K producer hands it to the other roles (its ticket t, -1 at the end, and
// the pair's geometry, so no taker repeats the lookups).
struct RingSlot {
  int t;
  Pair pr;
};
static_assert(2 * sizeof(RingSlot) <= 128, "two ring slots in the layout's ring bytes");

// Pair t of the enumeration: the prefill requests in the order ord[0..P) (longest first),
// each request's pairs with the KV head fastest and the query tiles from the last one back
// (the last tiles see the most keys).
template <int G>
__device__ __forceinline__ void pair_info(const PrefillParams& p, const int* pfx, int P, int t, Pair& pr) {
  const int* ord = pfx + (kMaxSeqs + 8);  // the order array follows the prefix (Layout::ORD)
  int lo = 0, hi = P;  // find i with pfx[i] <= t < pfx[i + 1]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (pfx[mid] <= t) lo = mid; else hi = mid;
  }
  constexpr int TOK = kBM / G;
  const int s = ord[lo];
  const int r = t - pfx[lo];
  const int Hkv = p.num_kv_heads;
  pr.s = s;
  pr.hk = r % Hkv;
  pr.qs = __ldg(p.qsl + s);
  const int q_len = __ldg(p.qsl + s + 1) - pr.qs;
  const int qp = (q_len + 2 * TOK - 1) / (2 * TOK) - 1 - r / Hkv;
  int L = __ldg(p.seq_lens + s);
  const int cap = p.max_blocks_per_seq * p.block_size;
  if (L > cap) L = cap;
  pr.L = L;
  int leff = 0;
#pragma unroll
  for (int x = 0; x < 2; ++x) {
    pr.q0[x] = (2 * qp + x) * TOK;
    pr.nq[x] = min(TOK, q_len - pr.q0[x]);  // <= 0: tile B past the chunk's end
    pr.pos0[x] = L - q_len + pr.q0[x];
    if (pr.nq[x] > 0) leff = pr.pos0[x] + pr.nq[x];
  }
  pr.leff = leff;  // keys the pair needs: 0 .. leff - 1
  if (q_len > L) raise_error(p.err, PA_DEVERR_SEQ_RANGE);
  pr.nt = (q_len > L || pr.nq[0] <= 0) ? 0 : (leff + kBN - 1) / kBN;
}

// ---- E4M3 caches: the producer warps turn their operands into f16 tiles in shared memory
// (every E4M3 value, and every bf16 query in f16's range, is exact in f16), so the MMAs
// run as kind::f16 with f16 operands exactly as with bf16 caches.
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t x, uint32_t& c01, uint32_t& c23) {
  asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\tcvt.rn.f16x2.e4m3x2 %0, a;\n\tcvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
      : "=r"(c01), "=r"(c23)
      : "r"(x));
}

// Rows [r_begin, r_end) (multiples of 4) of one 128-key step of codes -> the step's f16
// tile, in place. TMA stored key row r's 128 codes (head_dim 128), 128-byte swizzled, in
// the stage's second 64-dim half; dims 0..63 become row r of half 0 and dims 64..127 row r
// of half 1, swizzled the same way. Rows at or past `valid` become zeros (stale rows of V
// must not be NaN: P is 0 there, and 0 * NaN is not 0). Each iteration reads its 4 rows
// (8 lanes a row) before a __syncwarp and stores after it, so a row's half-1 codes are read
// before they are overwritten; no row's codes are written but by the warp converting that
// row, so two warps may convert disjoint row ranges of one stage.
__device__ __forceinline__ void convert_kv_step(unsigned char* stage, int valid, int lane, int r_begin, int r_end) {
  const int rsub = lane >> 3, c = lane & 7;
  const unsigned char* codes = stage + kHalf;
#pragma unroll 4
  for (int r0 = r_begin; r0 < r_end; r0 += 4) {
    const int r = r0 + rsub, sw = r & 7;
    const uint4 v = *reinterpret_cast<const uint4*>(codes + r * 128 + ((c ^ sw) << 4));
    __syncwarp();
    uint32_t h[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
    if (r < valid) {
      e4m3x4_to_f16x2x2(v.x, h[0], h[1]);
      e4m3x4_to_f16x2x2(v.y, h[2], h[3]);
      e4m3x4_to_f16x2x2(v.z, h[4], h[5]);
      e4m3x4_to_f16x2x2(v.w, h[6], h[7]);
    }
    unsigned char* row = stage + (c >> 2) * kHalf + r * 128;
    const int j0 = 2 * (c & 3);  // dims 16c .. 16c + 15 are 16-byte chunks j0, j0 + 1 of the half row
    *reinterpret_cast<uint4*>(row + ((j0 ^ sw) << 4)) = make_uint4(h[0], h[1], h[2], h[3]);
    *reinterpret_cast<uint4*>(row + (((j0 + 1) ^ sw) << 4)) = make_uint4(h[4], h[5], h[6], h[7]);
    __syncwarp();
  }
}

// bf16 -> f16 in place over `bytes` of shared memory (the pair's two query tiles).
__device__ __forceinline__ void convert_q_to_f16(unsigned char* q, uint32_t bytes, int lane) {
  uint4* v = reinterpret_cast<uint4*>(q);
  for (uint32_t i = lane; i < bytes / 16; i += 32) {
    uint4 x = v[i];
    uint32_t* w = reinterpret_cast<uint32_t*>(&x);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[k]));
      const __half2 h = __float22half2_rn(f);
      w[k] = *reinterpret_cast<const uint32_t*>(&h);
    }
    v[i] = x;
  }
}

// F8: E4M3 caches (head_dim 128): q and out bf16, K/V codes converted to f16 tiles by the
// producer warps, MMAs and P in f16.
template <int D, int G, bool F8>
__global__ void __launch_bounds__(threads_of<F8>(), 1) prefill_tc_kernel(const __grid_constant__ PrefillParams p,
                                                                 const __grid_constant__ CUtensorMap qmap,
                                                                 const __grid_constant__ CUtensorMap kmap,
                                                                 const __grid_constant__ CUtensorMap vmap) {
  using LY = Layout<D>;
  constexpr int NH = LY::NH;
  constexpr int TOK = kBM / G;
  static_assert(!F8 || D == 128, "E4M3 tiles: one 128-byte row of codes per key");
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;  // 128-byte swizzle atoms need 1024-byte alignment
  unsigned char* sm = smem_raw + (base - raw);
  int* pfx = reinterpret_cast<int*>(sm + LY::PFX);
  const uint32_t bar0 = base + LY::BAR;
  auto bar = [&](int i) { return bar0 + 8u * uint32_t(i); };
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(sm + LY::MISC);

  griddep_wait();  // inputs (e.g. this step's KV writes) come from earlier kernels

  const int S = p.num_seqs;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- the prefill requests (q_len >= 2), their order and the pair prefix in that order
  // (pairs = ceil(q_len / (2 TOK)) x num_kv_heads). Pairs are claimed in this order by the
  // CTAs as they run out of work, requests longest first (keys, then batch order, when at
  // most one per thread; else batch order): the costliest pairs start first and the cheap
  // ones at the end fill the CTAs that finish early.
  int* ord = reinterpret_cast<int*>(sm + LY::ORD);
  constexpr int NT = threads_of<F8>();
  __shared__ int wsum[NT / 32];
  // Block-wide exclusive scan of x (thread order); returns it, the total in *tot.
  auto block_scan = [&](int x, int* tot) {
    int inc = x;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, inc, d);
      if (lane >= d) inc += y;
    }
    if (lane == 31) wsum[warp] = inc;
    __syncthreads();
    int off = 0, t = 0;
#pragma unroll
    for (int w = 0; w < NT / 32; ++w) {
      if (w < warp) off += wsum[w];
      t += wsum[w];
    }
    __syncthreads();
    *tot = t;
    return off + inc - x;
  };
  const int cap = p.max_blocks_per_seq * p.block_size;
  int P = 0;  // compact: ord[i] = the i-th prefill request, pfx[i] = its length (the key)
  for (int b0 = 0; b0 < S; b0 += NT) {
    const int s = b0 + threadIdx.x;
    const int flag = (s < S && __ldg(p.qsl + s + 1) - __ldg(p.qsl + s) >= 2) ? 1 : 0;
    int tot;
    const int at = P + block_scan(flag, &tot);
    if (flag) {
      ord[at] = s;
      pfx[at] = min(__ldg(p.seq_lens + s), cap);
    }
    P += tot;
  }
  __syncthreads();
  if (P <= NT) {  // rank: longer first, then batch order
    int my_s = 0, my_key = 0, rank = 0;
    if (int(threadIdx.x) < P) {
      my_s = ord[threadIdx.x];
      my_key = pfx[threadIdx.x];
      for (int i = 0; i < P; ++i) {
        const int k = pfx[i];
        rank += (k > my_key || (k == my_key && i < int(threadIdx.x))) ? 1 : 0;
      }
    }
    __syncthreads();
    if (int(threadIdx.x) < P) ord[rank] = my_s;
    __syncthreads();
  }
  int run = 0;  // pfx[i]: pairs of ord[0..i); pfx[P] = total
  for (int b0 = 0; b0 <= P; b0 += NT) {
    const int i = b0 + threadIdx.x;
    int cnt = 0;
    if (i < P) {
      const int s = ord[i];
      const int q_len = __ldg(p.qsl + s + 1) - __ldg(p.qsl + s);
      cnt = ((q_len + 2 * TOK - 1) / (2 * TOK)) * p.num_kv_heads;
    }
    int tot;
    const int ex = block_scan(cnt, &tot);
    if (i <= P) pfx[i] = run + ex;
    run += tot;
  }
  __syncthreads();
  const int total = pfx[P];
  if (p.first_static ? int(blockIdx.x) >= total : p.ticket_base >= total) return;
  // The i-th pair of this CTA: for i = 0 pair blockIdx.x (first_static), after that the
  // next ticket of a counter shared by the grid and by a second launch of the same call
  // (dealt in enumeration order as CTAs run out of work; -1 when none is left). The Q/K
  // producer draws the tickets and passes each pair to the other roles through a two-slot
  // ring in shared memory.
  RingSlot* ring = reinterpret_cast<RingSlot*>(sm + LY::RING);
  auto ring_take = [&](int i, int& t, Pair& pr) -> bool {  // one thread; false on a timeout
    if (!mbar_wait(bar(bRingFull0 + (i & 1)), uint32_t(i >> 1) & 1u)) return false;
    t = ring[i & 1].t;
    if (t >= 0) pr = ring[i & 1].pr;
    mbar_arrive(bar(bRingEmpty0 + (i & 1)));
    return true;
  };
  auto ring_take_warp = [&](int i, int& t, Pair& pr) -> bool {  // a whole warp; each lane reads the slot
    if (!__all_sync(0xffffffffu, mbar_wait(bar(bRingFull0 + (i & 1)), uint32_t(i >> 1) & 1u))) return false;
    t = ring[i & 1].t;
    if (t >= 0) pr = ring[i & 1].pr;
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(bRingEmpty0 + (i & 1)));
    return true;
  };

  if (threadIdx.x == 0) {
    for (int i = 0; i < LY::NBAR; ++i) {
      uint32_t cnt = 1;
      if (i == bPFull0 || i == bPFull1 || i == bOEmpty0 || i == bOEmpty1 || i == bPHalf0 || i == bPHalf1) cnt = 4;
      if (i == bRingEmpty0 || i == bRingEmpty1) cnt = kRingTakers + (F8 ? 1 : 0);
      if (i == bQReady || i == bKReady0 || i == bKReady1 || i == bVReady0 || i == bVReady1) cnt = 2;  // E4M3 only
      mbar_init(bar(i), cnt);
    }
    fence_mbar_init();
  }
  if (warp == kWarpMMA) {
    tc::tmem_alloc(base + LY::MISC, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  auto fail = [&]() { raise_error(p.err, PA_DEVERR_TIMEOUT); };

  if (warp == kWarpQK || warp == kWarpV) {
    // =========================== TMA producers ===========================
    // warp 8: both Q tiles (once per pair) and K (2-deep ring); warp 10: V (2-deep ring).
    // Lane j handles physical block j of a 128-key step: it reads that block-table entry
    // one step ahead and issues the block's boxes itself.
    const bool is_k = (warp == kWarpQK);
    const CUtensorMap* map = is_k ? &kmap : &vmap;
    if (lane == 0) {
      if (is_k) tc::prefetch_tensormap(&qmap);
      tc::prefetch_tensormap(map);
    }
    const int B = p.block_size;
    const int nb = kBN / B;  // physical blocks per step (<= 16)
    int n = 0, tt = 0;
    bool ok = true;
    for (int i = 0; ok; ++i) {
      int t = -1;
      Pair pr;
      if (is_k) {  // draw the CTA's i-th pair and publish it, with its geometry, in ring slot i % 2
        if (lane == 0) {
          if (i == 0 && p.first_static) {
            t = int(blockIdx.x);
          } else {
            t = p.ticket_base + atomicAdd(p.sched, 1);
            if (t >= total) t = -1;
          }
        }
        t = __shfl_sync(0xffffffffu, t, 0);
        if (t >= 0) pair_info<G>(p, pfx, P, t, pr);
        int rok = 1;
        if (lane == 0) {
          rok = mbar_wait(bar(bRingEmpty0 + (i & 1)), (uint32_t(i >> 1) & 1u) ^ 1u) ? 1 : 0;
          if (rok) {
            ring[i & 1].t = t;
            if (t >= 0) ring[i & 1].pr = pr;
            mbar_arrive(bar(bRingFull0 + (i & 1)));
          }
        }
        if (!__shfl_sync(0xffffffffu, rok, 0)) { ok = false; break; }
      } else if (!ring_take_warp(i, t, pr)) {
        ok = false;
        break;
      }
      if (t < 0) break;
      if (pr.nt == 0) continue;
      if (is_k) {
        int qok = 1;
        if (lane == 0) {
          // the previous pair's queries are free once its last Q.K (step n - 1) has landed,
          // which the release of that step's K stage tells
          qok = (tt == 0 || mbar_wait(bar(bKEmpty0 + ((n - 1) & 1)), uint32_t((n - 1) >> 1) & 1u)) ? 1 : 0;
          if (qok) {
            mbar_arrive_expect_tx(bar(bQFull), uint32_t(2 * kBM * D * 2));
#pragma unroll
            for (int x = 0; x < 2; ++x)
#pragma unroll
              for (int h = 0; h < NH; ++h)
                tc::tma_load_3d(base + LY::Q + uint32_t(x * NH + h) * kHalf, &qmap, 64 * h, pr.hk * G,
                                pr.qs + pr.q0[x], bar(bQFull));
          }
        }
        if (!__shfl_sync(0xffffffffu, qok, 0)) { ok = false; break; }
      }
      const int32_t* bt = p.block_table + int64_t(pr.s) * p.max_blocks_per_seq;
      auto entry = [&](int kb) -> int64_t {  // this lane's block of step kb, or -1
        const int key = kb * kBN + lane * B;
        return (lane < nb && key < pr.leff) ? int64_t(__ldg(bt + key / B)) : int64_t(-1);
      };
      int64_t ent_next = entry(0);
      for (int kb = 0; kb < pr.nt; ++kb, ++n) {
        const int64_t ent = ent_next;
        if (kb + 1 < pr.nt) ent_next = entry(kb + 1);  // prefetch one step ahead
        const bool needed = lane < nb && kb * kBN + lane * B < pr.leff;
        const bool good = needed && ent >= 0 && ent < p.num_blocks;
        if (is_k && needed && !good) raise_error(p.err, PA_DEVERR_BLOCK_RANGE);
        const int nload = __popc(__ballot_sync(0xffffffffu, good));
        const int stage = n & 1;
        const uint32_t fb = bar((is_k ? bKFull0 : bVFull0) + stage);
        int wok = 1;
        if (lane == 0) {
          wok = mbar_wait(bar((is_k ? bKEmpty0 : bVEmpty0) + stage), ((n >> 1) & 1) ^ 1) ? 1 : 0;
          if (wok) mbar_arrive_expect_tx(fb, uint32_t(nload * B * 128 * (F8 ? 1 : NH)));
        }
        if (!__shfl_sync(0xffffffffu, wok, 0)) { ok = false; break; }
        const uint32_t sbase = (is_k ? LY::K : LY::V) + uint32_t(stage * NH) * kHalf;
        if (good) {
          const uint32_t dst = base + sbase + uint32_t(lane * B * 128);
          if constexpr (F8) {  // the codes of a key row: one 128-byte box row, in half 1
            tc::tma_load_3d(dst + kHalf, map, 0, pr.hk, int(ent * B), fb);
          } else {
#pragma unroll
            for (int h = 0; h < NH; ++h)
              tc::tma_load_3d(dst + uint32_t(h) * kHalf, map, 64 * h, pr.hk, int(ent * B), fb);
          }
        }
        if constexpr (F8) {
          if (is_k && kb == 0) {  // tile A's queries, bf16 -> f16, while K(0) is in flight
            if (!__all_sync(0xffffffffu, mbar_wait(bar(bQFull), tt & 1))) { ok = false; break; }
            convert_q_to_f16(sm + LY::Q, uint32_t(NH) * kHalf, lane);
            tc::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(bQReady));
          }
          // this step's codes to f16 once they have landed, while the MMAs of the previous
          // step run (converting step n - 1 after issuing step n's copy would wait, through
          // the 2-deep ring, for the MMAs of step n - 2, and serialise conversion and MMA)
          if (!__all_sync(0xffffffffu, mbar_wait(fb, (n >> 1) & 1))) { ok = false; break; }
          convert_kv_step(sm + sbase, min(kBN, pr.leff - kb * kBN), lane, 0, is_k ? kCvtSplitK : kCvtSplitV);  // the converter warp: the rest
          tc::fence_proxy_async_smem();  // generic-proxy stores -> the MMA's operand reads
          __syncwarp();
          if (lane == 0) mbar_arrive(bar((is_k ? bKReady0 : bVReady0) + stage));
        }
      }
      ++tt;
    }
    if (!ok && lane == 0) fail();
  } else if (F8 && warp == kWarpCvt) {
    // =========================== E4M3 converter ===========================
    // Tile B's queries and rows kCvtSplitK..127 of every K step and kCvtSplitV..127 of every
    // V step, beside the producers (which convert tile A's queries and the rows below); the
    // Ready barriers take both arrivals.
    int n = 0, tt = 0;
    bool ok = true;
    auto convert = [&](int full0, int ready0, uint32_t off, int kb, int leff, int r0) -> bool {
      const int stage = n & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(bar(full0 + stage), (n >> 1) & 1))) return false;
      convert_kv_step(sm + off + uint32_t(stage * NH) * kHalf, min(kBN, leff - kb * kBN), lane, r0, kBN);
      tc::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(ready0 + stage));
      return true;
    };
    for (int i = 0; ok; ++i) {
      int t = -1;
      Pair pr;
      if (!ring_take_warp(i, t, pr)) { ok = false; break; }
      if (t < 0) break;
      if (pr.nt == 0) continue;
      if (!__all_sync(0xffffffffu, mbar_wait(bar(bQFull), tt & 1))) { ok = false; break; }
      convert_q_to_f16(sm + LY::Q + uint32_t(NH) * kHalf, uint32_t(NH) * kHalf, lane);
      tc::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(bQReady));
      for (int kb = 0; kb < pr.nt; ++kb, ++n) {
        if (!convert(bKFull0, bKReady0, LY::K, kb, pr.leff, kCvtSplitK) ||
            !convert(bVFull0, bVReady0, LY::V, kb, pr.leff, kCvtSplitV)) {
          ok = false;
          break;
        }
      }
      ++tt;
    }
    if (!ok && lane == 0) fail();
  } else if (warp == kWarpMMA) {
    // =========================== MMA issuer ===========================
    // Per step n, in this order: P.V(A, n); Q.K(A, n + 1) once that P.V has landed (P lives
    // in S's columns); P.V(B, n); Q.K(B, n + 1). Tile A's softmax overlaps tile B's MMAs
    // and the other way round.
    if (lane == 0) {
      constexpr uint32_t idesc_qk = F8 ? tc::idesc_f16_f32(kBM, kBN, 0) : tc::idesc_bf16_f32(kBM, kBN, 0);
      constexpr uint32_t idesc_pv = F8 ? tc::idesc_f16_f32(kBM, D, 1) : tc::idesc_bf16_f32(kBM, D, 1);
      constexpr int kQ = F8 ? bQReady : bQFull, kK0 = F8 ? bKReady0 : bKFull0, kV0 = F8 ? bVReady0 : bVFull0;
      // Descriptors are built once per operand and advanced by the byte offset / 16 (the
      // start-address field counts 16-byte units; shared addresses stay below 256 KB, so
      // the 14-bit field never carries), keeping the issuing thread's work per MMA small.
      const uint64_t dq0 = tc::smem_desc_sw128(base + LY::Q, 16, 1024);
      const uint64_t dk0 = tc::smem_desc_sw128(base + LY::K, 16, 1024);
      const uint64_t dv0 = tc::smem_desc_sw128(base + LY::V, kHalf, 1024);
      auto qk = [&](int x, int nn) {  // S_x = Q_x . K(nn)^T
        const int stage = nn & 1;
        const uint64_t a0 = dq0 + uint64_t((uint32_t(x * NH) * kHalf) >> 4);
        const uint64_t b0 = dk0 + uint64_t((uint32_t(stage * NH) * kHalf) >> 4);
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t koff = uint32_t(k / 4) * kHalf + uint32_t(k % 4) * 32;
          tc::mma_f16(tmem + uint32_t(x * kBN), a0 + (koff >> 4), b0 + (koff >> 4), idesc_qk, k > 0 ? 1u : 0u);
        }
        // tile A: S_A ready; tile B (issued last on this K stage): the stage's release, which
        // is also S_B's ready signal (one commit where two would stall the issuing thread)
        tc::mma_commit(x == 0 ? bar(bSFullA) : bar(bKEmpty0 + stage));
      };
      // O_x += P_x . V(nn) over keys 64 h .. 64 h + 63 (h = 1 first: the softmax stores
      // those first); `first`: the pair's first step, whose first MMA starts O afresh
      auto pv_half = [&](int x, int nn, int h, bool first) {
        const int stage = nn & 1;
        const uint32_t pcol = tmem + uint32_t(x * kBN);
        const uint64_t b0 = dv0 + uint64_t((uint32_t(stage * NH) * kHalf) >> 4);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const int k = 4 * h + kk;
          // P keys 0..63 packed in columns 0..31, keys 64..127 in columns 64..95
          const uint32_t acol = pcol + uint32_t(64 * h + kk * 8);
          tc::mma_f16_ts(tmem + 256u + uint32_t(x * kBN), acol, b0 + uint64_t((uint32_t(k) * 2048) >> 4), idesc_pv,
                         (first && kk == 0) ? 0u : 1u);
        }
      };
      int n = 0, tt = 0;
      bool ok = true;
      for (int i = 0; ok; ++i) {
        int t = -1;
        Pair pr;
        if (!ring_take(i, t, pr)) { ok = false; break; }
        if (t < 0) break;
        if (pr.nt == 0) continue;
        const int n0 = n;
        if (!mbar_wait(bar(kQ), tt & 1)) { ok = false; break; }
        if (!mbar_wait(bar(kK0 + (n0 & 1)), (n0 >> 1) & 1)) { ok = false; break; }
        if (n0 > 0 && (!mbar_wait(bar(bPVDoneA), (n0 - 1) & 1) ||
                       !mbar_wait(bar(bVEmpty0 + ((n0 - 1) & 1)), uint32_t((n0 - 1) >> 1) & 1u))) {
          ok = false;  // the previous pair's last P.V read P out of S
          break;
        }
        tc::fence_after_sync();
        qk(0, n0);
        qk(1, n0);

        for (int kb = 0; kb < pr.nt && ok; ++kb, ++n) {
          const bool more = kb + 1 < pr.nt;
#pragma unroll
          for (int x = 0; x < 2; ++x) {
            if (!mbar_wait(bar(bPHalf0 + x), n & 1)) { ok = false; break; }
            if (kb == 0 && !mbar_wait(bar(bOEmpty0 + x), (tt & 1) ^ 1)) { ok = false; break; }
            if (x == 0 && !mbar_wait(bar(kV0 + (n & 1)), (n >> 1) & 1)) { ok = false; break; }
            tc::fence_after_sync();
            pv_half(x, n, 1, kb == 0);
            if (!mbar_wait(bar(bPFull0 + x), n & 1)) { ok = false; break; }
            tc::fence_after_sync();
            pv_half(x, n, 0, false);
            // tile A: P.V done; tile B (the step's last reader of V): the V stage's release,
            // which also tells that P.V(B) has landed
            tc::mma_commit(x == 0 ? bar(bPVDoneA) : bar(bVEmpty0 + (n & 1)));
            if (more) {
              if (!(x == 0 ? mbar_wait(bar(bPVDoneA), n & 1)
                           : mbar_wait(bar(bVEmpty0 + (n & 1)), uint32_t(n >> 1) & 1u))) { ok = false; break; }
              if (x == 0 && !mbar_wait(bar(kK0 + ((n + 1) & 1)), ((n + 1) >> 1) & 1)) { ok = false; break; }
              tc::fence_after_sync();
              qk(x, n + 1);

            }
          }
        }
        ++tt;
      }
      if (!ok) fail();
      // let every MMA issued by this thread land before TMEM is released
      tc::mma_commit(bar(bMmaDone));
      mbar_wait(bar(bMmaDone), 0);
    }
  } else {
    // =========================== softmax + epilogue ===========================
    // warps 4x .. 4x + 3 serve tile x; thread = row r (TMEM lane), all 128 keys of a step.
    const int x = warp >> 2;
    const int r = (warp & 3) * 32 + lane;
    const uint32_t trow = tmem + (uint32_t((warp & 3) * 32) << 16);
    const uint32_t scol = uint32_t(x * kBN), ocol = 256u + uint32_t(x * kBN);
    const float sc = p.scale_log2;
    int n = 0, tt = 0;
    bool ok = true;
    for (int it = 0; ok; ++it) {
      int t = -1;
      Pair pr;
      if (!ring_take_warp(it, t, pr)) { ok = false; break; }
      if (t < 0) break;
      if (pr.nt == 0) continue;
      const int i = r / G, g = r % G;
      const int nq_x = x ? pr.nq[1] : pr.nq[0];  // selects, not a runtime index into the struct
      const int pos_lo = x ? pr.pos0[1] : pr.pos0[0];
      const int q0_x = x ? pr.q0[1] : pr.q0[0];
      const bool active = i < nq_x;
      const int mypos = active ? pos_lo + i : pr.leff - 1;
      float m_used = -INFINITY, l = 0.f;  // m in raw score units
      for (int kb = 0; kb < pr.nt; ++kb, ++n) {
        if (!(x == 0 ? mbar_wait(bar(bSFullA), n & 1)
                     : mbar_wait(bar(bKEmpty0 + (n & 1)), uint32_t(n >> 1) & 1u))) { ok = false; break; }
        tc::fence_after_sync();
        const int key0 = kb * kBN;
        const bool diag = key0 + kBN - 1 > pos_lo;
        float s[64];
        // pass 1: the row max over both 64-key halves; each 32-column part of the second
        // half is loaded as soon as the part of the first half in its registers is reduced
        auto mask = [&](int c0, int koff) {  // keys past this row's position, for 32 columns
#pragma unroll
          for (int c = c0; c < c0 + 32; ++c) s[c] = (key0 + koff + c <= mypos) ? s[c] : -INFINITY;
        };
        auto max32 = [&](int c0) {
          float m10[10];
#pragma unroll
          for (int c = 0; c < 10; ++c) m10[c] = fmax3(s[c0 + 3 * c], s[c0 + 3 * c + 1], s[c0 + 3 * c + 2]);
          const float a = fmax3(m10[0], m10[1], m10[2]), b = fmax3(m10[3], m10[4], m10[5]);
          const float d = fmax3(m10[6], m10[7], m10[8]);
          return fmax3(fmax3(a, b, d), m10[9], fmaxf(s[c0 + 30], s[c0 + 31]));
        };
        tc::tmem_ld32(trow + scol, *reinterpret_cast<float(*)[32]>(s));
        tc::tmem_ld32(trow + scol + 32u, *reinterpret_cast<float(*)[32]>(s + 32));
        tc::tmem_wait_ld();
        if (diag) {
          mask(0, 0);
          mask(32, 0);
        }
        float mt = max32(0);
        tc::tmem_ld32(trow + scol + 64u, *reinterpret_cast<float(*)[32]>(s));
        mt = fmaxf(mt, max32(32));
        tc::tmem_ld32(trow + scol + 96u, *reinterpret_cast<float(*)[32]>(s + 32));
        tc::tmem_wait_ld();
        if (diag) {
          mask(0, 64);
          mask(32, 64);
        }
        mt = fmax3(mt, max32(0), max32(32));
        const float m_new = fmaxf(m_used, mt);
        const bool grow = (m_new - m_used) * sc > 8.f;  // also true on the first step
        const float m_use = grow ? m_new : m_used;
        const float alpha = exp2f((m_used - m_use) * sc);
        const float2 sc2 = make_float2(sc, sc), bias2 = make_float2(-m_use * sc, -m_use * sc);
        float2 rs[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
        // O rescale (its previous P.V is complete: this step's Q.K was issued after it)
        if (kb > 0 && __any_sync(0xffffffffu, grow)) {
          const float a = grow ? alpha : 1.f;
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            float o[32];
            tc::tmem_ld32(trow + ocol + uint32_t(c * 32), o);
            tc::tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] *= a;
            tc::tmem_st32(trow + ocol + uint32_t(c * 32), o);
          }
        }
        // pass 2: p = 2^(s * scale_log2 - m * scale_log2). Keys 64..127 (still in registers)
        // go to columns 64..95; keys 0..63 are reloaded, the first 32 as soon as their
        // registers are free (the load overlaps the remaining exponentials), and go to 0..31.
        auto exps = [&](float* pk, int c) {
          const float2 xv = ffma2v(make_float2(s[c], s[c + 1]), sc2, bias2);
          const float2 pp = make_float2(ex2_ftz(xv.x), ex2_ftz(xv.y));
          rs[(c >> 1) & 3] = fadd2(rs[(c >> 1) & 3], pp);
          if constexpr (F8) {
            __half2 hh = __floats2half2_rn(pp.x, pp.y);
            pk[c / 2] = __uint_as_float(*reinterpret_cast<uint32_t*>(&hh));
          } else {
            __nv_bfloat162 hh = __floats2bfloat162_rn(pp.x, pp.y);
            pk[c / 2] = __uint_as_float(*reinterpret_cast<uint32_t*>(&hh));
          }
        };
        {
          float pk[32];
#pragma unroll
          for (int c = 0; c < 64; c += 2) {
            exps(pk, c);
            if (c == 30) tc::tmem_ld32(trow + scol, *reinterpret_cast<float(*)[32]>(s));  // s[0..31] are free
          }
          tc::tmem_st32(trow + scol + 64u, pk);
        }
        tc::tmem_ld32(trow + scol + 32u, *reinterpret_cast<float(*)[32]>(s + 32));
        // last step: V rows past the keys the pair needs may hold stale or invalid data;
        // P is 0 there, but 0 * NaN is NaN in the MMA: tile A's threads zero them before
        // any P.V of the step starts (E4M3 caches: the V converter writes zeros there)
        if (!F8 && x == 0 && kb == pr.nt - 1 && pr.leff - key0 < kBN) {
          if (!mbar_wait(bar(bVFull0 + (n & 1)), (n >> 1) & 1)) { ok = false; break; }
          if (r >= pr.leff - key0) {
#pragma unroll
            for (int h = 0; h < NH; ++h)
#pragma unroll
              for (int ch = 0; ch < 8; ++ch)
                *reinterpret_cast<uint4*>(sm + LY::V + uint32_t((n & 1) * NH + h) * kHalf + uint32_t(r) * 128 +
                                          ch * 16) = make_uint4(0, 0, 0, 0);
          }
          tc::fence_proxy_async_smem();
        }
        // keys 64..127 of P are in place: the MMA thread may start on them
        tc::tmem_wait_st();
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(bPHalf0 + x));
        tc::tmem_wait_ld();
        if (diag) {
#pragma unroll
          for (int c = 0; c < 64; ++c) s[c] = (key0 + c <= mypos) ? s[c] : -INFINITY;
        }
        {
          float pk[32];
#pragma unroll
          for (int c = 0; c < 64; c += 2) exps(pk, c);
          tc::tmem_st32(trow + scol, pk);
        }
        const float2 r01 = fadd2(rs[0], rs[1]), r23 = fadd2(rs[2], rs[3]);
        l = l * alpha + ((r01.x + r01.y) + (r23.x + r23.y));
        m_used = m_use;
        tc::tmem_wait_st();
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(bPFull0 + x));
      }
      if (!ok) break;
      // ---- epilogue: O / l -> out
      if (!(x == 0 ? mbar_wait(bar(bPVDoneA), (n - 1) & 1)
                   : mbar_wait(bar(bVEmpty0 + ((n - 1) & 1)), uint32_t((n - 1) >> 1) & 1u))) { ok = false; break; }
      tc::fence_after_sync();
      const float inv = l > 0.f ? p.out_scale / l : 0.f;
      __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out) +
                           (int64_t(pr.qs + q0_x + i) * p.num_heads + pr.hk * G + g) * D;
      // two 32-column loads per wait (the score registers are free here)
      float o2[64];
#pragma unroll
      for (int c = 0; c < D / 32; c += 2) {
        tc::tmem_ld32(trow + ocol + uint32_t(c * 32), *reinterpret_cast<float(*)[32]>(o2));
        tc::tmem_ld32(trow + ocol + uint32_t(c * 32 + 32), *reinterpret_cast<float(*)[32]>(o2 + 32));
        tc::tmem_wait_ld();
        if (active && p.out_v8) {  // 32 bytes (16 dims) per store: half the store instructions
#pragma unroll
          for (int e = 0; e < 64; e += 16) {
            float f[8], h[8];
#pragma unroll
            for (int xx = 0; xx < 8; ++xx) {
              f[xx] = o2[e + xx] * inv;
              h[xx] = o2[e + 8 + xx] * inv;
            }
            const uint4 u = Elem<__nv_bfloat16>::pack(f), w = Elem<__nv_bfloat16>::pack(h);
            asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(out + c * 32 + e),
                         "r"(u.x), "r"(u.y), "r"(u.z), "r"(u.w), "r"(w.x), "r"(w.y), "r"(w.z), "r"(w.w)
                         : "memory");
          }
        } else if (active) {
#pragma unroll
          for (int e = 0; e < 64; e += 8) {
            float f[8];
#pragma unroll
            for (int xx = 0; xx < 8; ++xx) f[xx] = o2[e + xx] * inv;
            *reinterpret_cast<uint4*>(out + c * 32 + e) = Elem<__nv_bfloat16>::pack(f);
          }
        }
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(bOEmpty0 + x));
      ++tt;
    }
    if (!ok) fail();
  }

  // ---- teardown: everyone done with TMEM, then the allocating warp frees it
  tc::fence_before_sync();
  __syncthreads();
  if (warp == kWarpMMA) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
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

// 3-D map over [d2][d1][d0] (d0 contiguous) of bf16 (el 2) or 1-byte codes (el 1), box
// {128 bytes of d0, b1, b2}, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* ptr, int el, uint64_t d0, uint64_t d1, uint64_t d2, uint32_t b1,
              uint32_t b2) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {d0 * el, d0 * d1 * el};
  const cuuint32_t box[3] = {cuuint32_t(128 / el), b1, b2};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, el == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(ptr),
            dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, int G, bool F8>
cudaError_t prepare(const AttnArgs& a, PrefillTcPlan* plan) {
  const int B = a.block_size;
  const int el = F8 ? 1 : 2;
  if (!make_map(&plan->qm, a.q, 2, D, uint64_t(a.num_heads), uint64_t(a.num_tokens), G, kBM / G) ||
      !make_map(&plan->km, a.k_cache, el, D, uint64_t(a.num_kv_heads), uint64_t(a.num_blocks) * B, 1, B) ||
      !make_map(&plan->vm, a.v_cache, el, D, uint64_t(a.num_kv_heads), uint64_t(a.num_blocks) * B, 1, B))
    return cudaErrorInvalidValue;
  if (!a.prefill_sched) return cudaErrorInvalidValue;
  return ensure_smem<prefill_tc_kernel<D, G, F8>>(Layout<D>::SMEM);
}

template <int D, int G, bool F8>
cudaError_t run(const AttnArgs& a, const PrefillTcPlan& plan, int num_ctas, cudaStream_t stream,
                const PrefillLaunch& how) {
  PrefillParams p;
  p.out = a.out;
  p.block_table = a.block_table;
  p.seq_lens = a.seq_lens;
  p.qsl = a.query_start_loc;
  p.err = a.err;
  p.sched = a.prefill_sched;
  p.first_static = how.first_static ? 1 : 0;
  p.ticket_base = how.ticket_base;
  p.num_blocks = a.num_blocks;
  p.max_blocks_per_seq = a.max_blocks_per_seq;
  p.num_seqs = a.num_seqs;
  p.num_heads = a.num_heads;
  p.num_kv_heads = a.num_kv_heads;
  p.block_size = a.block_size;
  // E4M3: a K code stands for value * k_scale (folded into the logit scale), a V code for
  // value * v_scale (folded into the final 1 / l)
  p.scale_log2 = a.scale * 1.4426950408889634f * (F8 ? a.k_scale : 1.f);
  p.out_scale = F8 ? a.v_scale : 1.f;
  p.out_v8 = (reinterpret_cast<uintptr_t>(a.out) % 32 == 0) ? 1 : 0;
  if (!p.sched || how.ticket_base < 0) return cudaErrorInvalidValue;
  if (how.zero_counter) {
    const cudaError_t e = cudaMemsetAsync(p.sched, 0, sizeof(int), stream);  // the pair counter starts at 0
    if (e != cudaSuccess) return e;
  }
  return launch_pdl(prefill_tc_kernel<D, G, F8>, dim3(num_ctas), dim3(threads_of<F8>()), Layout<D>::SMEM, stream, p,
                    plan.qm, plan.km, plan.vm);
}

template <int D, bool F8>
cudaError_t prepare_g(const AttnArgs& a, int G, PrefillTcPlan* plan) {
  switch (G) {
    case 1: return prepare<D, 1, F8>(a, plan);
    case 2: return prepare<D, 2, F8>(a, plan);
    case 4: return prepare<D, 4, F8>(a, plan);
    case 8: return prepare<D, 8, F8>(a, plan);
  }
  return cudaErrorInvalidValue;
}

template <int D, bool F8>
cudaError_t run_g(const AttnArgs& a, const PrefillTcPlan& plan, int G, int num_ctas, cudaStream_t stream,
                  const PrefillLaunch& how) {
  switch (G) {
    case 1: return run<D, 1, F8>(a, plan, num_ctas, stream, how);
    case 2: return run<D, 2, F8>(a, plan, num_ctas, stream, how);
    case 4: return run<D, 4, F8>(a, plan, num_ctas, stream, how);
    case 8: return run<D, 8, F8>(a, plan, num_ctas, stream, how);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

bool prefill_tc_supported(const AttnArgs& a) {
  const int B = a.block_size;
  const bool types = a.dtype == PA_BF16 &&
                     ((a.cache_dtype == PA_BF16 && (a.head_dim == 64 || a.head_dim == 128)) ||
                      (a.cache_dtype == PA_FP8_E4M3 && a.head_dim == 128));
  return types && B >= 8 && B <= kBN && kBN % B == 0 && a.num_seqs <= kMaxSeqs && encode_fn() != nullptr;
}

cudaError_t prepare_prefill_tc(const AttnArgs& a, PrefillTcPlan* plan) {
  const int G = a.num_heads / a.num_kv_heads;
  if (a.cache_dtype == PA_FP8_E4M3) return prepare_g<128, true>(a, G, plan);
  if (a.head_dim == 64) return prepare_g<64, false>(a, G, plan);
  return prepare_g<128, false>(a, G, plan);
}

cudaError_t launch_prefill_tc(const AttnArgs& a, const PrefillTcPlan& plan, int num_ctas, cudaStream_t stream,
                              const PrefillLaunch& how) {
  const int G = a.num_heads / a.num_kv_heads;
  if (a.cache_dtype == PA_FP8_E4M3) return run_g<128, true>(a, plan, G, num_ctas, stream, how);
  if (a.head_dim == 64) return run_g<64, false>(a, plan, G, num_ctas, stream, how);
  return run_g<128, false>(a, plan, G, num_ctas, stream, how);
}

}  // namespace pa
