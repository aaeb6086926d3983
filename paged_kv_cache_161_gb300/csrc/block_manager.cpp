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
// Free blocks leave a FIFO queue whose initial order is given by the caller; released
// blocks join its tail. An append that cannot complete changes nothing.
#include <cstdint>
#include <cstring>
#include <deque>
#include <new>
#include <unordered_map>
#include <vector>

#include "pa.h"

struct pa_bm {
  struct Seq {
    std::vector<int32_t> table;
    int64_t len = 0;
  };
  int64_t num_blocks = 0;
  int block_size = 0;
  std::deque<int32_t> free_q;
  std::vector<int32_t> ref;
  std::unordered_map<int64_t, Seq> seqs;
  std::deque<int64_t> copies;  // src, dst, src, dst, ...

  int32_t take_block() {
    const int32_t b = free_q.front();
    free_q.pop_front();
    ref[b] = 1;
    return b;
  }
};

namespace {

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace

extern "C" {

pa_bm* pa_bm_create(int64_t num_blocks, int block_size, const int32_t* free_order) {
  if (num_blocks < 1 || num_blocks > 0x7fffffff || block_size < 1 || !free_order) return nullptr;
  pa_bm* bm = new (std::nothrow) pa_bm();
  if (!bm) return nullptr;
  bm->num_blocks = num_blocks;
  bm->block_size = block_size;
  std::vector<char> seen(size_t(num_blocks), 0);
  for (int64_t i = 0; i < num_blocks; ++i) {
    const int32_t b = free_order[i];
    if (b < 0 || b >= num_blocks || seen[size_t(b)]) {
      delete bm;
      return nullptr;
    }
    seen[size_t(b)] = 1;
    bm->free_q.push_back(b);
  }
  bm->ref.assign(size_t(num_blocks), 0);
  return bm;
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
  auto it = bm->seqs.find(seq);
  if (it == bm->seqs.end()) return PA_ERR_NOT_FOUND;
  pa_bm::Seq& sq = it->second;
  const int64_t B = bm->block_size;
  if (n == 0) return PA_OK;
  if (ceil_div(sq.len + n, B) > bm->num_blocks) return PA_ERR_TOO_LARGE;
  // Blocks this append takes: the ones that open new logical blocks, plus one copy if
  // the first token lands in a partially filled block that others still hold.
  const bool cow = (sq.len % B != 0) && bm->ref[size_t(sq.table.back())] > 1;
  const int64_t need = ceil_div(sq.len + n, B) - ceil_div(sq.len, B) + (cow ? 1 : 0);
  if (need > int64_t(bm->free_q.size())) return PA_ERR_NO_BLOCKS;
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
  }
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
  pa_bm::Seq c = it->second;
  for (int32_t b : c.table) bm->ref[size_t(b)] += 1;
  bm->seqs.emplace(child, std::move(c));
  return PA_OK;
}

int pa_bm_free_seq(pa_bm* bm, int64_t seq) {
  if (!bm) return PA_ERR_INVALID_ARG;
  auto it = bm->seqs.find(seq);
  if (it == bm->seqs.end()) return PA_ERR_NOT_FOUND;
  for (int32_t b : it->second.table) {
    if (--bm->ref[size_t(b)] == 0) bm->free_q.push_back(b);
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

int64_t pa_bm_num_free(const pa_bm* bm) { return bm ? int64_t(bm->free_q.size()) : -1; }

int pa_bm_free_queue(const pa_bm* bm, int32_t* out, int64_t capacity) {
  if (!bm || (!out && !bm->free_q.empty())) return PA_ERR_INVALID_ARG;
  if (capacity < int64_t(bm->free_q.size())) return PA_ERR_INVALID_ARG;
  int64_t i = 0;
  for (int32_t b : bm->free_q) out[i++] = b;
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

}  // extern "C"
