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
// each K/V tile feeds all of them. Per 128-key tile: S = Q.K^T (8 x tcgen05.mma
// 128x128x16, bf16 in, f32 accumulate in TMEM), online softmax in registers (exp2
// domain, the scale folded into one FMA per score, lazy rescaling of O only when the row
// max grows by more than 2^8), P as bf16 back into TMEM, O += P.V (8 x tcgen05.mma
// 128xDx16, A = P from TMEM, B = V as an MN-major shared-memory operand), O in TMEM.
//
// Roles (352 threads, one CTA per SM, persistent over a static round-robin of tiles):
//   warps 0-7  softmax + epilogue: two threads per row (TMEM lane r), one per 64-key half
//              of S and 64-dim half of O; the row max (and the final sum) cross halves
//              through shared memory on a bounded mbarrier;
//   warps 8/10 TMA producers: Q tile once per tile and K tiles (3-deep ring) on warp 8,
//              V tiles (2-deep ring) on warp 10, 128 keys at a time by physical block
//              through the block table (one 3-D box per block and 64-dim half);
//   warp 9     allocates 512 TMEM columns (S triple buffer 3 x 128, O 128) and one thread
//              issues the MMAs, tracking completion with tcgen05.commit. P is written back
//              into its S buffer as packed bf16 and read from TMEM by the P.V MMA.
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
constexpr int kBN = 128;             // keys per tile
constexpr int kMaxSeqs = 4096;       // requests per call this kernel accepts
constexpr int kSoftmaxWarps = 8;     // two threads per row: column halves
constexpr int kThreads = (kSoftmaxWarps + 3) * 32;  // + K/Q producer, MMA issuer, V producer
constexpr int kKStages = 3;
constexpr int kVStages = 2;
constexpr uint32_t kTmemCols = 512;  // S buffers 3 x 128 columns, O 128 columns
constexpr uint32_t kOCol = 384;
constexpr uint32_t kHalf = 128 * 128;  // bytes of a 128-row x 64-element bf16 half tile

struct PrefillParams {
  void* out;
  const int32_t* block_table;
  const int32_t* seq_lens;
  const int32_t* qsl;
  unsigned int* err;
  int64_t num_blocks;
  int max_blocks_per_seq;
  int num_seqs;
  int num_heads;
  int num_kv_heads;
  int block_size;
  float scale_log2;
};

template <int D>
struct Layout {
  static constexpr int NH = D / 64;  // 64-element halves of the head dim
  static constexpr uint32_t Q = 0;
  static constexpr uint32_t K = Q + NH * kHalf;                  // kKStages stages
  static constexpr uint32_t V = K + kKStages * NH * kHalf;       // kVStages stages
  static constexpr uint32_t PFX = V + kVStages * NH * kHalf;     // int[kMaxSeqs + 8]
  static constexpr uint32_t XCH = PFX + (kMaxSeqs + 8) * 4;  // float[2 slots][2 halves][128 rows]
  static constexpr uint32_t BAR = XCH + 2 * 2 * 128 * 4;     // mbarriers
  static constexpr int NBAR = 26;
  static constexpr uint32_t MISC = BAR + NBAR * 8;           // tmem base, abort flag
  static constexpr uint32_t BYTES = MISC + 16;
  static constexpr uint32_t SMEM = BYTES + 1024;             // + alignment slack
};

// barrier indices
enum : int {
  bQFull = 0, bQEmpty,
  bKFull0, bKFull1, bKFull2, bKEmpty0, bKEmpty1, bKEmpty2,
  bVFull0, bVFull1, bVEmpty0, bVEmpty1,
  bSFull0, bSFull1, bSFull2, bSFree0, bSFree1, bSFree2,
  bPFull, bPVDone, bOEmpty, bXch, bMmaDone
};

struct Tile {
  int s, hk, qs, L, q0, nq, pos0, leff, nt;
};

// Tile t of the batch: binary search of the per-request tile prefix in shared memory.
template <int G>
__device__ __forceinline__ void tile_info(const PrefillParams& p, const int* pfx, int S, int t, Tile& tl) {
  int lo = 0, hi = S;  // find s with pfx[s] <= t < pfx[s + 1]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (pfx[mid] <= t) lo = mid; else hi = mid;
  }
  constexpr int TOK = kBM / G;
  const int s = lo;
  const int r = t - pfx[s];
  const int Hkv = p.num_kv_heads;
  tl.s = s;
  tl.hk = r % Hkv;
  const int qt = r / Hkv;
  tl.qs = __ldg(p.qsl + s);
  const int q_len = __ldg(p.qsl + s + 1) - tl.qs;
  int L = __ldg(p.seq_lens + s);
  const int cap = p.max_blocks_per_seq * p.block_size;
  if (L > cap) L = cap;
  tl.L = L;
  tl.q0 = qt * TOK;
  tl.nq = min(TOK, q_len - tl.q0);
  tl.pos0 = L - q_len + tl.q0;
  tl.leff = tl.pos0 + tl.nq;  // keys this tile needs: 0 .. leff - 1
  if (q_len > L) raise_error(p.err, PA_DEVERR_SEQ_RANGE);
  tl.nt = (q_len > L || tl.nq <= 0) ? 0 : (tl.leff + kBN - 1) / kBN;
}

template <int D, int G>
__global__ void __launch_bounds__(kThreads, 1) prefill_tc_kernel(const __grid_constant__ PrefillParams p,
                                                                 const __grid_constant__ CUtensorMap qmap,
                                                                 const __grid_constant__ CUtensorMap kmap,
                                                                 const __grid_constant__ CUtensorMap vmap) {
  using LY = Layout<D>;
  constexpr int NH = LY::NH;
  constexpr int TOK = kBM / G;
  constexpr int DH = D / 2;  // O dims per softmax thread
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;  // 128-byte swizzle atoms need 1024-byte alignment
  unsigned char* sm = smem_raw + (base - raw);
  int* pfx = reinterpret_cast<int*>(sm + LY::PFX);
  float* xch = reinterpret_cast<float*>(sm + LY::XCH);
  const uint32_t bar0 = base + LY::BAR;
  auto bar = [&](int i) { return bar0 + 8u * uint32_t(i); };
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(sm + LY::MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + LY::MISC + 4);

  griddep_wait();  // inputs (e.g. this step's KV writes) come from earlier kernels

  const int S = p.num_seqs;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- per-request tile prefix (tiles = ceil(q_len / TOK) x num_kv_heads for q_len >= 2)
  int run = 0;
  for (int b0 = 0; b0 <= S; b0 += kThreads) {
    const int s = b0 + threadIdx.x;
    int cnt = 0;
    if (s < S) {
      const int q_len = __ldg(p.qsl + s + 1) - __ldg(p.qsl + s);
      if (q_len >= 2) cnt = ((q_len + TOK - 1) / TOK) * p.num_kv_heads;
    }
    int inc = cnt;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, inc, d);
      if (lane >= d) inc += y;
    }
    __shared__ int wsum[kThreads / 32];
    if (lane == 31) wsum[warp] = inc;
    __syncthreads();
    int off = 0, tot = 0;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) {
      if (w < warp) off += wsum[w];
      tot += wsum[w];
    }
    if (s <= S) pfx[s] = run + off + inc - cnt;  // exclusive prefix; pfx[S] = total
    run += tot;
    __syncthreads();
  }
  const int total = pfx[S];
  if (int(blockIdx.x) >= total) return;

  if (threadIdx.x == 0) {
    for (int i = 0; i < LY::NBAR; ++i) {
      uint32_t cnt = 1;
      if (i == bPFull || i == bOEmpty || i == bXch) cnt = kSoftmaxWarps;
      mbar_init(bar(i), cnt);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kSoftmaxWarps + 1) {
    tc::tmem_alloc(base + LY::MISC, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  auto fail = [&]() {
    raise_error(p.err, PA_DEVERR_TIMEOUT);
    *abort_flag = 1;
  };

  if (warp == kSoftmaxWarps || warp == kSoftmaxWarps + 2) {
    // =========================== TMA producers ===========================
    // warp 8: Q (once per tile) and K (3-deep ring); warp 10: V (2-deep ring). Separate
    // warps so that a K load never queues behind a V stage still in use. Lane j handles
    // physical block j of a 128-key step: it reads that block-table entry one step ahead
    // and issues the block's boxes itself.
    const bool is_k = (warp == kSoftmaxWarps);
    const CUtensorMap* map = is_k ? &kmap : &vmap;
    if (lane == 0) {
      if (is_k) tc::prefetch_tensormap(&qmap);
      tc::prefetch_tensormap(map);
    }
    const int B = p.block_size;
    const int nb = kBN / B;  // physical blocks per step (<= 16)
    const int nst = is_k ? kKStages : kVStages;
    int n = 0, tt = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
      Tile tl;
      tile_info<G>(p, pfx, S, t, tl);
      if (tl.nt == 0) continue;
      if (is_k) {
        int qok = 1;
        if (lane == 0) {
          qok = mbar_wait(bar(bQEmpty), (tt & 1) ^ 1) ? 1 : 0;
          if (qok) {
            mbar_arrive_expect_tx(bar(bQFull), uint32_t(kBM * D * 2));
#pragma unroll
            for (int h = 0; h < NH; ++h)
              tc::tma_load_3d(base + LY::Q + h * kHalf, &qmap, 64 * h, tl.hk * G, tl.qs + tl.q0, bar(bQFull));
          }
        }
        if (!__shfl_sync(0xffffffffu, qok, 0)) { ok = false; break; }
      }
      const int32_t* bt = p.block_table + int64_t(tl.s) * p.max_blocks_per_seq;
      auto entry = [&](int kb) -> int64_t {  // this lane's block of step kb, or -1
        const int key = kb * kBN + lane * B;
        return (lane < nb && key < tl.leff) ? int64_t(__ldg(bt + key / B)) : int64_t(-1);
      };
      int64_t ent_next = entry(0);
      for (int kb = 0; kb < tl.nt; ++kb, ++n) {
        const int64_t ent = ent_next;
        if (kb + 1 < tl.nt) ent_next = entry(kb + 1);  // prefetch one step ahead
        const bool needed = lane < nb && kb * kBN + lane * B < tl.leff;
        const bool good = needed && ent >= 0 && ent < p.num_blocks;
        if (is_k && needed && !good) raise_error(p.err, PA_DEVERR_BLOCK_RANGE);
        const int nload = __popc(__ballot_sync(0xffffffffu, good));
        const int stage = n % nst, use = n / nst;
        const uint32_t fb = bar((is_k ? bKFull0 : bVFull0) + stage);
        int wok = 1;
        if (lane == 0) {
          wok = mbar_wait(bar((is_k ? bKEmpty0 : bVEmpty0) + stage), (use & 1) ^ 1) ? 1 : 0;
          if (wok) mbar_arrive_expect_tx(fb, uint32_t(nload * B * 128 * NH));
        }
        if (!__shfl_sync(0xffffffffu, wok, 0)) { ok = false; break; }
        if (good) {
          const uint32_t dst = base + (is_k ? LY::K : LY::V) + uint32_t(stage * NH) * kHalf + uint32_t(lane * B * 128);
#pragma unroll
          for (int h = 0; h < NH; ++h)
            tc::tma_load_3d(dst + uint32_t(h) * kHalf, map, 64 * h, tl.hk, int(ent * B), fb);
        }
      }
      ++tt;
    }
    if (!ok && lane == 0) fail();
  } else if (warp == kSoftmaxWarps + 1) {
    // =========================== MMA issuer ===========================
    if (lane == 0) {
      constexpr uint32_t idesc_qk = tc::idesc_bf16_f32(kBM, kBN, 0);
      constexpr uint32_t idesc_pv = tc::idesc_bf16_f32(kBM, D, 1);
      int n = 0, tt = 0;
      // S(nn) = Q . K(nn)^T into S buffer nn % 3
      auto issue_qk = [&](int nn) -> bool {
        const int stage = nn % kKStages, sb = nn % 3;
        if (!mbar_wait(bar(bKFull0 + stage), (nn / kKStages) & 1)) return false;
        if (!mbar_wait(bar(bSFree0 + sb), ((nn / 3) & 1) ^ 1)) return false;
        tc::fence_after_sync();
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t koff = uint32_t(k / 4) * kHalf + uint32_t(k % 4) * 32;
          const uint64_t a = tc::smem_desc_sw128(base + LY::Q + koff, 16, 1024);
          const uint64_t b = tc::smem_desc_sw128(base + LY::K + uint32_t(stage * NH) * kHalf + koff, 16, 1024);
          tc::mma_f16(tmem + uint32_t(sb * kBN), a, b, idesc_qk, k > 0 ? 1u : 0u);
        }
        tc::mma_commit(bar(bKEmpty0 + stage));
        tc::mma_commit(bar(bSFull0 + sb));
        return true;
      };
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        Tile tl;
        tile_info<G>(p, pfx, S, t, tl);
        if (tl.nt == 0) continue;
        if (!mbar_wait(bar(bQFull), tt & 1)) { ok = false; break; }
        tc::fence_after_sync();
        const int n0 = n;
        for (int i = 0; i < 2 && i < tl.nt; ++i)
          if (!issue_qk(n0 + i)) { ok = false; break; }
        if (!ok) break;
        if (tl.nt <= 2) tc::mma_commit(bar(bQEmpty));  // every QK of the tile is issued
        for (int kb = 0; kb < tl.nt; ++kb, ++n) {
          if (!mbar_wait(bar(bPFull), n & 1)) { ok = false; break; }
          if (kb == 0 && !mbar_wait(bar(bOEmpty), (tt & 1) ^ 1)) { ok = false; break; }
          const int stage = n % kVStages;
          if (!mbar_wait(bar(bVFull0 + stage), (n / kVStages) & 1)) { ok = false; break; }
          tc::fence_after_sync();
          const uint32_t pcol = tmem + uint32_t((n % 3) * kBN);  // P (bf16 pairs) over S's first 64 columns
#pragma unroll
          for (int k = 0; k < kBN / 16; ++k) {
            const uint64_t b = tc::smem_desc_sw128(base + LY::V + uint32_t(stage * NH) * kHalf + uint32_t(k) * 2048,
                                                   kHalf, 1024);
            tc::mma_f16_ts(tmem + kOCol, pcol + uint32_t(k * 8), b, idesc_pv, (kb > 0 || k > 0) ? 1u : 0u);
          }
          tc::mma_commit(bar(bVEmpty0 + stage));
          tc::mma_commit(bar(bSFree0 + n % 3));
          tc::mma_commit(bar(bPVDone));
          if (kb + 2 < tl.nt) {
            if (!issue_qk(n + 2)) { ok = false; break; }
            if (kb + 3 == tl.nt) tc::mma_commit(bar(bQEmpty));
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
    // warp w: rows 32 (w % 4) .. + 31 (its TMEM lane quarter), column half h = w / 4 of S
    // (keys 64h .. 64h + 63 of each tile) and of O (dims DH h .. DH h + DH - 1).
    const int h = warp >> 2;
    const int r = (warp & 3) * 32 + lane;  // tile row == TMEM lane
    const uint32_t trow = tmem + (uint32_t((warp & 3) * 32) << 16);
    const float sc = p.scale_log2;
    int n = 0, xph = 0;
    bool ok = true;
    // exchange a per-row value with the thread holding the other column half (bounded)
    auto exchange = [&](float v, float& other) -> bool {
      float* slot = xch + (xph & 1) * 256;
      slot[h * 128 + r] = v;
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(bXch));
      const bool done = mbar_wait(bar(bXch), xph & 1);
      other = slot[(1 - h) * 128 + r];
      ++xph;
      return done;
    };
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
      Tile tl;
      tile_info<G>(p, pfx, S, t, tl);
      if (tl.nt == 0) continue;
      const int i = r / G, g = r % G;
      const bool active = i < tl.nq;
      const int mypos = tl.pos0 + (active ? i : tl.nq - 1);
      float m_used = -INFINITY, l = 0.f;  // m in raw score units; l: this half's partial sum
      for (int kb = 0; kb < tl.nt; ++kb, ++n) {
        const int sb = n % 3;
        if (!mbar_wait(bar(bSFull0 + sb), (n / 3) & 1)) { ok = false; break; }
        tc::fence_after_sync();
        float s[64];
        tc::tmem_ld32(trow + uint32_t(sb * kBN + h * 64), *reinterpret_cast<float(*)[32]>(s));
        tc::tmem_ld32(trow + uint32_t(sb * kBN + h * 64 + 32), *reinterpret_cast<float(*)[32]>(s + 32));
        tc::tmem_wait_ld();
        const int key0 = kb * kBN + h * 64;
        if (kb * kBN + kBN - 1 > tl.pos0) {  // a diagonal tile: causal mask
#pragma unroll
          for (int c = 0; c < 64; ++c) s[c] = (key0 + c <= mypos) ? s[c] : -INFINITY;
        }
        // row max of this half: 3-input max tree (64 -> 22 -> 8 -> 3 -> 1)
        float m22[22];
#pragma unroll
        for (int c = 0; c < 21; ++c) m22[c] = fmax3(s[3 * c], s[3 * c + 1], s[3 * c + 2]);
        m22[21] = s[63];
        float m8[8];
#pragma unroll
        for (int c = 0; c < 7; ++c) m8[c] = fmax3(m22[3 * c], m22[3 * c + 1], m22[3 * c + 2]);
        m8[7] = m22[21];
        const float mt = fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
        tc::fence_before_sync();  // S reads done before the other half overwrites S with P
        float mo;
        if (!exchange(mt, mo)) { ok = false; break; }
        tc::fence_after_sync();
        const float m_new = fmaxf(m_used, fmaxf(mt, mo));
        const bool grow = (m_new - m_used) * sc > 8.f;  // also true on the first tile
        const float m_use = grow ? m_new : m_used;
        const float alpha = exp2f((m_used - m_use) * sc);
        const float bias = -m_use * sc;
        // p = 2^(s * scale_log2 - m * scale_log2): one packed FMA per pair, hardware ex2
        float2 rs[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
        float pk[32];
        const float2 sc2 = make_float2(sc, sc), bias2 = make_float2(bias, bias);
#pragma unroll
        for (int c = 0; c < 64; c += 2) {
          const float2 x = ffma2v(make_float2(s[c], s[c + 1]), sc2, bias2);
          const float2 pp = make_float2(ex2_ftz(x.x), ex2_ftz(x.y));
          rs[(c >> 1) & 3] = fadd2(rs[(c >> 1) & 3], pp);
          __nv_bfloat162 hh = __floats2bfloat162_rn(pp.x, pp.y);
          pk[c / 2] = __uint_as_float(*reinterpret_cast<uint32_t*>(&hh));
        }
        const float2 r01 = fadd2(rs[0], rs[1]), r23 = fadd2(rs[2], rs[3]);
        l = l * alpha + ((r01.x + r01.y) + (r23.x + r23.y));
        m_used = m_use;
        // O rescale needs the previous P.V finished (rare with the lazy threshold)
        if (kb > 0 && __any_sync(0xffffffffu, grow)) {
          if (!mbar_wait(bar(bPVDone), (n - 1) & 1)) { ok = false; break; }
          tc::fence_after_sync();
          const float a = grow ? alpha : 1.f;
#pragma unroll
          for (int c = 0; c < DH / 32; ++c) {
            float o[32];
            tc::tmem_ld32(trow + kOCol + uint32_t(h * DH + c * 32), o);
            tc::tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] *= a;
            tc::tmem_st32(trow + kOCol + uint32_t(h * DH + c * 32), o);
          }
        }
        // P (bf16 pairs) into the first 64 columns of this S buffer: half h -> 32 columns
        tc::tmem_st32(trow + uint32_t(sb * kBN + h * 32), pk);
        tc::tmem_wait_st();
        // last tile: V rows past the keys this tile needs may hold stale or invalid data;
        // P is 0 there, but 0 * NaN is NaN in the MMA: zero them
        if (kb == tl.nt - 1 && tl.leff - kb * kBN < kBN) {
          const int st = n % kVStages;
          if (!mbar_wait(bar(bVFull0 + st), (n / kVStages) & 1)) { ok = false; break; }
          if (r >= tl.leff - kb * kBN && h < NH) {  // thread h clears V dim-half h of row r
#pragma unroll
            for (int ch = 0; ch < 8; ++ch)
              *reinterpret_cast<uint4*>(sm + LY::V + uint32_t(st * NH + h) * kHalf + uint32_t(r) * 128 + ch * 16) =
                  make_uint4(0, 0, 0, 0);
          }
          tc::fence_proxy_async_smem();
        }
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(bPFull));
      }
      if (!ok) break;
      // ---- epilogue: O / l -> out
      float lo;
      if (!exchange(l, lo)) { ok = false; break; }
      if (!mbar_wait(bar(bPVDone), (n - 1) & 1)) { ok = false; break; }
      tc::fence_after_sync();
      const float lt = l + lo;
      const float inv = lt > 0.f ? 1.f / lt : 0.f;
      __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out) +
                           (int64_t(tl.qs + tl.q0 + i) * p.num_heads + tl.hk * G + g) * D + h * DH;
#pragma unroll
      for (int c = 0; c < DH / 32; ++c) {
        float o[32];
        tc::tmem_ld32(trow + kOCol + uint32_t(h * DH + c * 32), o);
        tc::tmem_wait_ld();
        if (active) {
#pragma unroll
          for (int e = 0; e < 32; e += 8) {
            float f[8];
#pragma unroll
            for (int x = 0; x < 8; ++x) f[x] = o[e + x] * inv;
            *reinterpret_cast<uint4*>(out + c * 32 + e) = Elem<__nv_bfloat16>::pack(f);
          }
        }
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(bOEmpty));
    }
    if (!ok) fail();
  }

  // ---- teardown: everyone done with TMEM, then the allocating warp frees it
  tc::fence_before_sync();
  __syncthreads();
  if (warp == kSoftmaxWarps + 1) {
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

// 3-D bf16 map over [d2][d1][d0] (d0 contiguous), box {64, b1, b2}, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* ptr, uint64_t d0, uint64_t d1, uint64_t d2, uint32_t b1, uint32_t b2) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {d0 * 2, d0 * d1 * 2};
  const cuuint32_t box[3] = {64, b1, b2};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, int G>
cudaError_t run(const AttnArgs& a, int num_ctas, cudaStream_t stream) {
  CUtensorMap qm, km, vm;
  const int B = a.block_size;
  if (!make_map(&qm, a.q, D, uint64_t(a.num_heads), uint64_t(a.num_tokens), G, kBM / G) ||
      !make_map(&km, a.k_cache, D, uint64_t(a.num_kv_heads), uint64_t(a.num_blocks) * B, 1, B) ||
      !make_map(&vm, a.v_cache, D, uint64_t(a.num_kv_heads), uint64_t(a.num_blocks) * B, 1, B))
    return cudaErrorInvalidValue;
  PrefillParams p;
  p.out = a.out;
  p.block_table = a.block_table;
  p.seq_lens = a.seq_lens;
  p.qsl = a.query_start_loc;
  p.err = a.err;
  p.num_blocks = a.num_blocks;
  p.max_blocks_per_seq = a.max_blocks_per_seq;
  p.num_seqs = a.num_seqs;
  p.num_heads = a.num_heads;
  p.num_kv_heads = a.num_kv_heads;
  p.block_size = a.block_size;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  auto kern = prefill_tc_kernel<D, G>;
  const size_t smem = Layout<D>::SMEM;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(num_ctas), dim3(kThreads), smem, stream, p, qm, km, vm);
}

template <int D>
cudaError_t run_g(const AttnArgs& a, int G, int num_ctas, cudaStream_t stream) {
  switch (G) {
    case 1: return run<D, 1>(a, num_ctas, stream);
    case 2: return run<D, 2>(a, num_ctas, stream);
    case 4: return run<D, 4>(a, num_ctas, stream);
    case 8: return run<D, 8>(a, num_ctas, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

bool prefill_tc_supported(const AttnArgs& a) {
  const int B = a.block_size;
  return a.dtype == PA_BF16 && (a.head_dim == 64 || a.head_dim == 128) && B >= 8 && B <= kBN && kBN % B == 0 &&
         a.num_seqs <= kMaxSeqs && encode_fn() != nullptr;
}

cudaError_t launch_prefill_tc(const AttnArgs& a, int num_ctas, cudaStream_t stream) {
  const int G = a.num_heads / a.num_kv_heads;
  if (a.head_dim == 64) return run_g<64>(a, G, num_ctas, stream);
  return run_g<128>(a, G, num_ctas, stream);
}

}  // namespace pa
