// Host block manager of include/pa.h (pa_bm_*): the accounting that produces the slot
// mappings, block tables and copy-on-write pairs the device kernels consume.
//
// Sources: "vLLM" docs page -- PagedAttention algorithm flow (a request's blocks are
// taken on demand: a new physical block only when the current one is full; all released
// when the request ends), memory-utilisation arithmetic (n tokens hold ceil(n / B)
// blocks), Copy-on-Write (reference counts: +1 per sharer, -1 when a holder ends or
// moves away, released at 0; a write into a block with count > 1 first copies it to a
// fresh block). Code-reading page 5.1.1 / 5.2.1 (the worked examples). vLLM 0.10.0 flow
// page 3.3 (pool of free blocks; slot = block * B + offset).
//
// Swapping (optional, pa_bm_enable_swap): code-reading page 6.2.1 (a preempted sequence
// group's KV blocks are swapped out to the CPU and back in when resources return); a CPU
// pool with its own FIFO free queue and reference counts; each distinct block of a group
// moves once, and a block still held outside the group stays on the GPU.
//
// Prefix caching (optional, pa_bm_enable_prefix_caching): "vLLM" docs page, Copy-on-Write ›
// shared-prefix detection (hash the prompt prefix; reuse cached prefix KV, counts + 1) and
// Prefix Caching › mechanism (look up on arrival, reuse on a hit, cache on a miss); vLLM
// 0.10.0 flow page 3.3 (the pool's blocks on a doubly linked list, LRU eviction).
//
// Free blocks sit on a doubly linked list whose initial order is given by the caller: new
// blocks come from the head, released blocks join the tail, and (with prefix caching) a
// lookup that reuses a released block unlinks it from the middle. The list is the LRU
// order. An append that cannot complete changes nothing.
//
// With prefix caching, a full block is keyed by its whole token prefix (every token of
// the sequence up to the block's last slot), encoded as a 128-bit hash chain: the key of
// block i is the key of block i - 1 folded with block i's token ids (fold_block). It is registered
// when its last slot is written unless the key is already registered (the first block
// stays); it keeps its registration while released and loses it when the free list hands
// it out again (eviction). Two different prefixes share a key only through a 128-bit hash
// collision.
#include <cstdint>
#include <cstring>
#include <deque>
#include <new>
#include <unordered_map>
#include <vector>

#include "pa.h"

namespace {

struct Key {
  uint64_t a, b;
  bool operator==(const Key& o) const { return a == o.a && b == o.b; }
};

struct KeyHash {
  size_t operator()(const Key& k) const { return size_t(k.a ^ (k.b * 0x9E3779B97F4A7C15ull)); }
};

// Finaliser of the SplitMix64 generator (Steele, Lea and Flood, OOPSLA 2014): a
// bijective 64-bit mixer.
uint64_t mix64(uint64_t z) {
  z ^= z >> 30;
  z *= 0xBF58476D1CE4E5B9ull;
  z ^= z >> 27;
  z *= 0x94D049BB133111EBull;
  z ^= z >> 31;
  return z;
}

// Key of a full block: its parent's key (the prefix before it) folded with its B token
// ids. Each lane absorbs the ids two at a time as one 64-bit word with one multiply
// (lane a: xor then multiply, as in FNV-1a over 64-bit words; lane b: add then multiply
// by another odd constant), then goes through the bijective mixer, so the next block
// starts from a well-mixed state.
Key fold_block(Key parent, const int32_t* tokens, int64_t n) {
  uint64_t a = parent.a, b = parent.b;
  int64_t i = 0;
  for (; i + 1 < n; i += 2) {
    const uint64_t w = uint64_t(uint32_t(tokens[i])) | (uint64_t(uint32_t(tokens[i + 1])) << 32);
    a = (a ^ w) * 0x00000100000001B3ull;
    b = (b + w + 1) * 0xD1B54A32D192ED03ull;
  }
  if (i < n) {
    const uint64_t w = uint64_t(uint32_t(tokens[i])) | (uint64_t(0xFFFFFFFFu) << 32);
    a = (a ^ w) * 0x00000100000001B3ull;
    b = (b + w + 1) * 0xD1B54A32D192ED03ull;
  }
  return Key{mix64(a ^ uint64_t(n)), mix64(b + 0x632BE59BD9B4E019ull)};
}

constexpr Key kRootKey{0x243F6A8885A308D3ull, 0x13198A2E03707344ull};  // the empty prefix

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace

struct pa_bm {
  struct Seq {
    std::vector<int32_t> table;
    int64_t len = 0;
    Key chain = kRootKey;          // key of the prefix through the last full block
    std::vector<int32_t> partial;  // token ids of the partially filled last block
    bool swapped = false;          // its table holds CPU block ids
  };
  int64_t num_blocks = 0;
  int block_size = 0;
  // free list (doubly linked over block ids; -1 ends it)
  std::vector<int32_t> nxt, prv;
  std::vector<char> in_free;
  int32_t head = -1, tail = -1;
  int64_t nfree = 0;
  std::vector<int32_t> ref;
  std::unordered_map<int64_t, Seq> seqs;
  std::deque<int64_t> copies;  // src, dst, src, dst, ...
  // prefix caching
  bool caching = false;
  std::unordered_map<Key, int32_t, KeyHash> cache;
  std::vector<Key> block_key;
  std::vector<char> registered;
  int64_t hit_blocks = 0, evictions = 0;
  // CPU block pool for swapping (FIFO free queue, reference counts)
  bool swap = false;
  int64_t num_cpu_blocks = 0;
  std::deque<int32_t> cpu_free;
  std::vector<int32_t> cpu_ref;

  void push_free(int32_t b) {
    nxt[b] = -1;
    prv[b] = tail;
    if (tail >= 0) nxt[tail] = b; else head = b;
    tail = b;
    in_free[b] = 1;
    ++nfree;
  }
  void unlink_free(int32_t b) {
    if (prv[b] >= 0) nxt[prv[b]] = nxt[b]; else head = nxt[b];
    if (nxt[b] >= 0) prv[nxt[b]] = prv[b]; else tail = prv[b];
    in_free[b] = 0;
    --nfree;
  }
  int32_t take_block() {
    const int32_t b = head;
    unlink_free(b);
    if (caching && registered[b]) {  // evicted: its content is about to be overwritten
      cache.erase(block_key[b]);
      registered[b] = 0;
      ++evictions;
    }
    ref[b] = 1;
    return b;
  }
  // Token `tok` was just written at position len - 1 of `sq`; register a block it filled.
  void note_token(Seq& sq, int32_t tok) {
    sq.partial.push_back(tok);
    if (sq.len % block_size != 0) return;
    const Key k = fold_block(sq.chain, sq.partial.data(), int64_t(sq.partial.size()));
    sq.partial.clear();
    sq.chain = k;
    const int32_t b = sq.table.back();
    if (cache.emplace(k, b).second) {
      block_key[b] = k;
      registered[b] = 1;
    }
  }
};

namespace {

// Shared by pa_bm_append and pa_bm_append_tokens: tokens == nullptr without caching.
int append_impl(pa_bm* bm, int64_t seq, int64_t n, const int32_t* tokens, int64_t* slots_out) {
  auto it = bm->seqs.find(seq);
  if (it == bm->seqs.end()) return PA_ERR_NOT_FOUND;
  pa_bm::Seq& sq = it->second;
  if (sq.swapped) return PA_ERR_INVALID_ARG;
  const int64_t B = bm->block_size;
  if (n == 0) return PA_OK;
  if (ceil_div(sq.len + n, B) > bm->num_blocks) return PA_ERR_TOO_LARGE;
  // Blocks this append takes: the ones that open new logical blocks, plus one copy if
  // the first token lands in a partially filled block that others still hold.
  const bool cow = (sq.len % B != 0) && bm->ref[size_t(sq.table.back())] > 1;
  const int64_t need = ceil_div(sq.len + n, B) - ceil_div(sq.len, B) + (cow ? 1 : 0);
  if (need > bm->nfree) return PA_ERR_NO_BLOCKS;
  for (int64_t i = 0; i < n; ++i) {
    const int64_t pos = sq.len;
    if (pos % B == 0) {
      sq.table.push_back(bm->take_block());
    } else if (bm->ref[size_t(sq.table.back())] > 1) {
      const int32_t src = sq.table.back();
      const int32_t dst = bm->take_block();
      bm->copies.push_back(src);
      bm->copies.push_back(dst);
      bm->ref[size_t(src)] -= 1;
      sq.table.back() = dst;
    }
    slots_out[i] = int64_t(sq.table[size_t(pos / B)]) * B + pos % B;
    sq.len = pos + 1;
    if (tokens) bm->note_token(sq, tokens[i]);
  }
  return PA_OK;
}

}  // namespace

extern "C" {

pa_bm* pa_bm_create(int64_t num_blocks, int block_size, const int32_t* free_order) {
  if (num_blocks < 1 || num_blocks > 0x7fffffff || block_size < 1 || !free_order) return nullptr;
  pa_bm* bm = new (std::nothrow) pa_bm();
  if (!bm) return nullptr;
  bm->num_blocks = num_blocks;
  bm->block_size = block_size;
  const size_t nb = size_t(num_blocks);
  bm->nxt.assign(nb, -1);
  bm->prv.assign(nb, -1);
  bm->in_free.assign(nb, 0);
  for (int64_t i = 0; i < num_blocks; ++i) {
    const int32_t b = free_order[i];
    if (b < 0 || b >= num_blocks || bm->in_free[size_t(b)]) {
      delete bm;
      return nullptr;
    }
    bm->push_free(b);
  }
  bm->ref.assign(nb, 0);
  return bm;
}

int pa_bm_enable_prefix_caching(pa_bm* bm) {
  if (!bm || !bm->seqs.empty() || bm->nfree != bm->num_blocks) return PA_ERR_INVALID_ARG;
  bm->caching = true;
  bm->block_key.assign(size_t(bm->num_blocks), Key{0, 0});
  bm->registered.assign(size_t(bm->num_blocks), 0);
  return PA_OK;
}

void pa_bm_destroy(pa_bm* bm) { delete bm; }

int pa_bm_add_seq(pa_bm* bm, int64_t seq) {
  if (!bm) return PA_ERR_INVALID_ARG;
  if (bm->seqs.count(seq)) return PA_ERR_NOT_FOUND;
  bm->seqs.emplace(seq, pa_bm::Seq());
  return PA_OK;
}

int pa_bm_append(pa_bm* bm, int64_t seq, int64_t n, int64_t* slots_out) {
  if (!bm || n < 0 || (n > 0 && !slots_out)) return PA_ERR_INVALID_ARG;
  if (bm->caching) return PA_ERR_INVALID_ARG;  // needs the token ids: pa_bm_append_tokens
  return append_impl(bm, seq, n, nullptr, slots_out);
}

int pa_bm_append_tokens(pa_bm* bm, int64_t seq, const int32_t* token_ids, int64_t n, int64_t* slots_out) {
  if (!bm || n < 0 || (n > 0 && (!slots_out || !token_ids))) return PA_ERR_INVALID_ARG;
  return append_impl(bm, seq, n, bm->caching ? token_ids : nullptr, slots_out);
}

int pa_bm_append_tokens_batch(pa_bm* bm, const int64_t* seqs, const int64_t* counts, int64_t n,
                              const int32_t* token_ids, int64_t* slots_out, int64_t* done_out) {
  if (done_out) *done_out = 0;
  if (!bm || n < 0 || (n > 0 && (!seqs || !counts))) return PA_ERR_INVALID_ARG;
  int64_t off = 0;
  for (int64_t i = 0; i < n; ++i) {
    const int st = pa_bm_append_tokens(bm, seqs[i], counts[i] > 0 ? token_ids + off : nullptr, counts[i],
                                       counts[i] > 0 ? slots_out + off : nullptr);
    if (st != PA_OK) return st;
    off += counts[i];
    if (done_out) *done_out = i + 1;
  }
  return PA_OK;
}

int pa_bm_add_seq_cached(pa_bm* bm, int64_t seq, const int32_t* prompt, int64_t n, int64_t max_hit,
                         int64_t* hit_out) {
  if (!bm || !bm->caching || n < 0 || (n > 0 && !prompt) || !hit_out) return PA_ERR_INVALID_ARG;
  if (bm->seqs.count(seq)) return PA_ERR_NOT_FOUND;
  pa_bm::Seq sq;
  const int64_t B = bm->block_size;
  const int64_t lim = max_hit < n ? max_hit : n;
  Key k = kRootKey;
  sq.table.reserve(size_t(n / B + 1));
  while (sq.len + B <= lim) {
    const Key kk = fold_block(k, prompt + sq.len, B);
    auto it = bm->cache.find(kk);
    if (it == bm->cache.end()) break;
    const int32_t b = it->second;
    if (bm->ref[size_t(b)] == 0) bm->unlink_free(b);
    bm->ref[size_t(b)] += 1;
    sq.table.push_back(b);
    sq.len += B;
    k = kk;
  }
  sq.chain = k;
  bm->hit_blocks += int64_t(sq.table.size());
  *hit_out = sq.len;
  bm->seqs.emplace(seq, std::move(sq));
  return PA_OK;
}

int pa_bm_prefix_stats(const pa_bm* bm, int64_t* cached_blocks, int64_t* hit_blocks, int64_t* evictions) {
  if (!bm || !cached_blocks || !hit_blocks || !evictions) return PA_ERR_INVALID_ARG;
  *cached_blocks = int64_t(bm->cache.size());
  *hit_blocks = bm->hit_blocks;
  *evictions = bm->evictions;
  return PA_OK;
}

int pa_bm_append_batch(pa_bm* bm, const int64_t* seqs, const int64_t* counts, int64_t n, int64_t* slots_out,
                       int64_t* done_out) {
  if (done_out) *done_out = 0;
  if (!bm || n < 0 || (n > 0 && (!seqs || !counts))) return PA_ERR_INVALID_ARG;
  int64_t off = 0;
  for (int64_t i = 0; i < n; ++i) {
    const int st = pa_bm_append(bm, seqs[i], counts[i], counts[i] > 0 ? slots_out + off : nullptr);
    if (st != PA_OK) return st;
    off += counts[i];
    if (done_out) *done_out = i + 1;
  }
  return PA_OK;
}

int pa_bm_fork(pa_bm* bm, int64_t parent, int64_t child) {
  if (!bm) return PA_ERR_INVALID_ARG;
  auto it = bm->seqs.find(parent);
  if (it == bm->seqs.end() || bm->seqs.count(child)) return PA_ERR_NOT_FOUND;
  if (it->second.swapped) return PA_ERR_INVALID_ARG;
  pa_bm::Seq c = it->second;
  for (int32_t b : c.table) bm->ref[size_t(b)] += 1;
  bm->seqs.emplace(child, std::move(c));
  return PA_OK;
}

int pa_bm_free_seq(pa_bm* bm, int64_t seq) {
  if (!bm) return PA_ERR_INVALID_ARG;
  auto it = bm->seqs.find(seq);
  if (it == bm->seqs.end()) return PA_ERR_NOT_FOUND;
  if (it->second.swapped) {
    for (int32_t c : it->second.table)
      if (--bm->cpu_ref[size_t(c)] == 0) bm->cpu_free.push_back(c);
  } else {
    for (int32_t b : it->second.table) {
      if (--bm->ref[size_t(b)] == 0) bm->push_free(b);
    }
  }
  bm->seqs.erase(it);
  return PA_OK;
}

int64_t pa_bm_seq_len(const pa_bm* bm, int64_t seq) {
  if (!bm) return -1;
  auto it = bm->seqs.find(seq);
  return it == bm->seqs.end() ? -1 : it->second.len;
}

int64_t pa_bm_num_seq_blocks(const pa_bm* bm, int64_t seq) {
  if (!bm) return -1;
  auto it = bm->seqs.find(seq);
  return it == bm->seqs.end() ? -1 : int64_t(it->second.table.size());
}

int pa_bm_ref_count(const pa_bm* bm, int64_t block) {
  if (!bm || block < 0 || block >= bm->num_blocks) return -1;
  return bm->ref[size_t(block)];
}

int64_t pa_bm_num_free(const pa_bm* bm) { return bm ? bm->nfree : -1; }

int pa_bm_free_queue(const pa_bm* bm, int32_t* out, int64_t capacity) {
  if (!bm || (!out && bm->nfree > 0)) return PA_ERR_INVALID_ARG;
  if (capacity < bm->nfree) return PA_ERR_INVALID_ARG;
  int64_t i = 0;
  for (int32_t b = bm->head; b >= 0; b = bm->nxt[size_t(b)]) out[i++] = b;
  return PA_OK;
}

int pa_bm_block_table(const pa_bm* bm, int64_t seq, int32_t* out, int64_t capacity) {
  if (!bm) return PA_ERR_INVALID_ARG;
  auto it = bm->seqs.find(seq);
  if (it == bm->seqs.end()) return PA_ERR_NOT_FOUND;
  const auto& t = it->second.table;
  if (capacity < int64_t(t.size()) || (!out && !t.empty())) return PA_ERR_INVALID_ARG;
  if (!t.empty()) std::memcpy(out, t.data(), t.size() * sizeof(int32_t));
  return PA_OK;
}

int pa_bm_batch_tables(const pa_bm* bm, const int64_t* seqs, int64_t n, int32_t* table_out,
                       int64_t width, int32_t* seq_lens_out) {
  if (!bm || n < 0 || width < 1 || (n > 0 && (!seqs || !table_out || !seq_lens_out)))
    return PA_ERR_INVALID_ARG;
  for (int64_t i = 0; i < n; ++i) {
    auto it = bm->seqs.find(seqs[i]);
    if (it == bm->seqs.end()) return PA_ERR_NOT_FOUND;
    const auto& t = it->second.table;
    if (it->second.swapped) return PA_ERR_INVALID_ARG;  // its blocks are not on the GPU
    if (int64_t(t.size()) > width || it->second.len > 0x7fffffff) return PA_ERR_INVALID_ARG;
    int32_t* row = table_out + i * width;
    if (!t.empty()) std::memcpy(row, t.data(), t.size() * sizeof(int32_t));
    std::memset(row + t.size(), 0, size_t(width - int64_t(t.size())) * sizeof(int32_t));
    seq_lens_out[i] = int32_t(it->second.len);
  }
  return PA_OK;
}

int64_t pa_bm_num_pending_copies(const pa_bm* bm) { return bm ? int64_t(bm->copies.size() / 2) : -1; }

int64_t pa_bm_take_copies(pa_bm* bm, int64_t* pairs_out, int64_t capacity) {
  if (!bm || capacity < 0 || (capacity > 0 && !pairs_out)) return -1;
  int64_t k = 0;
  while (k < capacity && !bm->copies.empty()) {
    pairs_out[2 * k] = bm->copies.front();
    bm->copies.pop_front();
    pairs_out[2 * k + 1] = bm->copies.front();
    bm->copies.pop_front();
    ++k;
  }
  return k;
}

// ---------------------------------------------------------------- swapping
int pa_bm_enable_swap(pa_bm* bm, int64_t num_cpu_blocks, const int32_t* cpu_free_order) {
  if (!bm || bm->swap || num_cpu_blocks < 1 || num_cpu_blocks > 0x7fffffff || !cpu_free_order)
    return PA_ERR_INVALID_ARG;
  std::vector<char> seen(size_t(num_cpu_blocks), 0);
  for (int64_t i = 0; i < num_cpu_blocks; ++i) {
    const int32_t c = cpu_free_order[i];
    if (c < 0 || c >= num_cpu_blocks || seen[size_t(c)]) return PA_ERR_INVALID_ARG;
    seen[size_t(c)] = 1;
  }
  bm->swap = true;
  bm->num_cpu_blocks = num_cpu_blocks;
  bm->cpu_free.assign(cpu_free_order, cpu_free_order + num_cpu_blocks);
  bm->cpu_ref.assign(size_t(num_cpu_blocks), 0);
  return PA_OK;
}

namespace {

// Distinct blocks of the group's tables, first met walking the sequences in order and each
// table from its first block, with how many of the sequences hold each.
void group_blocks(pa_bm* bm, const int64_t* seqs, int64_t n, std::vector<int32_t>& order,
                  std::unordered_map<int32_t, int32_t>& holders) {
  for (int64_t i = 0; i < n; ++i)
    for (int32_t b : bm->seqs.find(seqs[i])->second.table)
      if (holders[b]++ == 0) order.push_back(b);
}

// Checks shared by both directions: swap on, distinct known sequences, all on the side the
// move starts from.
int check_group(pa_bm* bm, const int64_t* seqs, int64_t n, bool want_swapped) {
  if (!bm || !bm->swap || n < 0 || (n > 0 && !seqs)) return PA_ERR_INVALID_ARG;
  std::unordered_map<int64_t, char> seen;
  for (int64_t i = 0; i < n; ++i) {
    auto it = bm->seqs.find(seqs[i]);
    if (it == bm->seqs.end()) return PA_ERR_NOT_FOUND;
    if (it->second.swapped != want_swapped || seen[seqs[i]]++) return PA_ERR_INVALID_ARG;
  }
  return PA_OK;
}

}  // namespace

int pa_bm_swap_out(pa_bm* bm, const int64_t* seqs, int64_t n, int64_t* pairs_out, int64_t capacity,
                   int64_t* num_pairs_out) {
  int st = check_group(bm, seqs, n, false);
  if (st != PA_OK) return st;
  if (!num_pairs_out) return PA_ERR_INVALID_ARG;
  std::vector<int32_t> order;
  std::unordered_map<int32_t, int32_t> holders;
  group_blocks(bm, seqs, n, order, holders);
  if (int64_t(order.size()) > capacity || (!order.empty() && !pairs_out)) return PA_ERR_INVALID_ARG;
  if (int64_t(order.size()) > int64_t(bm->cpu_free.size())) return PA_ERR_NO_BLOCKS;
  std::unordered_map<int32_t, int32_t> where;
  int64_t k = 0;
  for (int32_t g : order) {
    const int32_t c = bm->cpu_free.front();
    bm->cpu_free.pop_front();
    const int32_t h = holders[g];
    bm->cpu_ref[size_t(c)] = h;
    bm->ref[size_t(g)] -= h;
    if (bm->ref[size_t(g)] == 0) bm->push_free(g);
    where[g] = c;
    pairs_out[2 * k] = g;
    pairs_out[2 * k + 1] = c;
    ++k;
  }
  for (int64_t i = 0; i < n; ++i) {
    pa_bm::Seq& sq = bm->seqs.find(seqs[i])->second;
    for (int32_t& b : sq.table) b = where[b];
    sq.swapped = true;
  }
  *num_pairs_out = k;
  return PA_OK;
}

int pa_bm_swap_in(pa_bm* bm, const int64_t* seqs, int64_t n, int64_t* pairs_out, int64_t capacity,
                  int64_t* num_pairs_out) {
  int st = check_group(bm, seqs, n, true);
  if (st != PA_OK) return st;
  if (!num_pairs_out) return PA_ERR_INVALID_ARG;
  std::vector<int32_t> order;
  std::unordered_map<int32_t, int32_t> holders;
  group_blocks(bm, seqs, n, order, holders);
  if (int64_t(order.size()) > capacity || (!order.empty() && !pairs_out)) return PA_ERR_INVALID_ARG;
  if (int64_t(order.size()) > bm->nfree) return PA_ERR_NO_BLOCKS;
  std::unordered_map<int32_t, int32_t> where;
  int64_t k = 0;
  for (int32_t c : order) {
    const int32_t g = bm->take_block();
    const int32_t h = holders[c];
    bm->ref[size_t(g)] = h;
    bm->cpu_ref[size_t(c)] -= h;
    if (bm->cpu_ref[size_t(c)] == 0) bm->cpu_free.push_back(c);
    where[c] = g;
    pairs_out[2 * k] = c;
    pairs_out[2 * k + 1] = g;
    ++k;
  }
  for (int64_t i = 0; i < n; ++i) {
    pa_bm::Seq& sq = bm->seqs.find(seqs[i])->second;
    for (int32_t& b : sq.table) b = where[b];
    sq.swapped = false;
  }
  *num_pairs_out = k;
  return PA_OK;
}

int pa_bm_is_swapped(const pa_bm* bm, int64_t seq) {
  if (!bm) return -1;
  auto it = bm->seqs.find(seq);
  return it == bm->seqs.end() ? -1 : (it->second.swapped ? 1 : 0);
}

int64_t pa_bm_num_free_cpu(const pa_bm* bm) { return bm && bm->swap ? int64_t(bm->cpu_free.size()) : -1; }

int pa_bm_cpu_ref_count(const pa_bm* bm, int64_t block) {
  if (!bm || !bm->swap || block < 0 || block >= bm->num_cpu_blocks) return -1;
  return bm->cpu_ref[size_t(block)];
}

int pa_bm_batch_groups(const pa_bm* bm, const int64_t* seqs, int64_t n, int max_members, int32_t* seq_group_out,
                       int32_t* group_range_out, int32_t* shared_len_out, int64_t capacity,
                       int64_t* num_groups_out) {
  if (!bm || n < 0 || max_members < 2 || !num_groups_out || (n > 0 && (!seqs || !seq_group_out)))
    return PA_ERR_INVALID_ARG;
  if (n > 0x7fffffff) return PA_ERR_INVALID_ARG;
  std::vector<const pa_bm::Seq*> sq(static_cast<size_t>(n));
  for (int64_t i = 0; i < n; ++i) {
    auto it = bm->seqs.find(seqs[i]);
    if (it == bm->seqs.end()) return PA_ERR_NOT_FOUND;
    sq[size_t(i)] = &it->second;
  }
  int64_t ng = 0;
  int64_t i = 0;
  while (i < n) {
    const auto& first = *sq[size_t(i)];
    int64_t j = i + 1;
    int64_t common = int64_t(first.table.size());  // leading entries shared with the first member
    int64_t min_len = first.len;
    while (j < n && j - i < max_members && !first.swapped && !sq[size_t(j)]->swapped) {
      const auto& t = sq[size_t(j)]->table;
      int64_t k = 0;
      while (k < common && k < int64_t(t.size()) && t[size_t(k)] == first.table[size_t(k)]) ++k;
      if (k == 0) break;
      common = k;
      min_len = sq[size_t(j)]->len < min_len ? sq[size_t(j)]->len : min_len;
      ++j;
    }
    if (j - i >= 2) {
      if (ng >= capacity || !group_range_out || !shared_len_out) return PA_ERR_INVALID_ARG;
      group_range_out[2 * ng] = int32_t(i);
      group_range_out[2 * ng + 1] = int32_t(j);
      const int64_t shared = common * bm->block_size;
      shared_len_out[ng] = int32_t(shared < min_len ? shared : min_len);
      for (int64_t m = i; m < j; ++m) seq_group_out[m] = int32_t(ng);
      ++ng;
    } else {
      seq_group_out[i] = -1;
    }
    i = j;
  }
  *num_groups_out = ng;
  return PA_OK;
}

}  // extern "C"
