// Host block manager of the paged KV cache ("PagedAttention: the KV cache
// was the bottleneck all along", section "Virtual memory for attention"):
// blocks are taken on demand as sequences grow, shared between forked
// sequences by reference count, and replaced by a private copy when a
// sequence writes into a block that another live sequence still holds.
//
// Plain C++ on the host: no CUDA call. Every entry point validates first and
// mutates only once the whole request is known to succeed.
#include <algorithm>
#include <cstdint>
#include <limits>
#include <new>
#include <vector>

#include "pkv_block_manager.h"

struct pkv_block_manager {
  struct Seq {
    std::vector<int32_t> table;  // physical block of each logical block
    int64_t len = 0;             // tokens
    bool live = false;
  };
  int32_t num_blocks = 0;
  int32_t block_size = 0;
  std::vector<int32_t> free_stack;  // next block to hand out at the back
  std::vector<int32_t> ref;         // table entries of live sequences pointing at each block
  std::vector<Seq> seqs;
  std::vector<int32_t> free_ids;    // ids of ended sequences, reused last-in first-out
  int64_t cow_copies = 0;

  // Scratch of the batched pre-checks (sized on first use, all zero between
  // calls): per-block reference changes and copies, the blocks touched, and
  // per-sequence marks for duplicate detection.
  std::vector<int32_t> blk_delta, blk_drop;
  std::vector<uint8_t> blk_seen, seq_mark;
  std::vector<int32_t> touched, marked;

  void ensure_scratch() {
    if (blk_delta.size() != (size_t)num_blocks) {
      blk_delta.assign((size_t)num_blocks, 0);
      blk_drop.assign((size_t)num_blocks, 0);
      blk_seen.assign((size_t)num_blocks, 0);
    }
    if (seq_mark.size() < seqs.size()) seq_mark.resize(seqs.size(), 0);
  }
  void touch(int32_t b) {
    if (!blk_seen[(size_t)b]) {
      blk_seen[(size_t)b] = 1;
      touched.push_back(b);
    }
  }
  // false when `s` was marked already (a repeated id)
  bool mark(int32_t s) {
    if (seq_mark[(size_t)s]) return false;
    seq_mark[(size_t)s] = 1;
    marked.push_back(s);
    return true;
  }
  void reset_scratch() {
    for (int32_t b : touched) {
      blk_delta[(size_t)b] = 0;
      blk_drop[(size_t)b] = 0;
      blk_seen[(size_t)b] = 0;
    }
    touched.clear();
    for (int32_t q : marked) seq_mark[(size_t)q] = 0;
    marked.clear();
  }

  bool is_live(int32_t s) const { return s >= 0 && (size_t)s < seqs.size() && seqs[(size_t)s].live; }

  int32_t take_block() {
    const int32_t b = free_stack.back();
    free_stack.pop_back();
    ref[(size_t)b] = 1;
    return b;
  }

  void drop_ref(int32_t b) {
    if (--ref[(size_t)b] == 0) free_stack.push_back(b);
  }

  // A fresh or recycled sequence id with an empty, live record.
  int32_t new_id() {
    int32_t id;
    if (!free_ids.empty()) {
      id = free_ids.back();
      free_ids.pop_back();
    } else {
      id = (int32_t)seqs.size();
      seqs.emplace_back();
    }
    Seq& s = seqs[(size_t)id];
    s.table.clear();
    s.len = 0;
    s.live = true;
    return id;
  }
};

namespace {

// splitmix64: a small counter-based generator, enough to scatter block ids.
uint64_t splitmix64(uint64_t& state) {
  uint64_t z = (state += 0x9e3779b97f4a7c15ull);
  z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ull;
  z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;
  return z ^ (z >> 31);
}

// Uniform integer in [0, n) by rejection (no modulo bias).
uint64_t below(uint64_t& state, uint64_t n) {
  const uint64_t limit = std::numeric_limits<uint64_t>::max() - std::numeric_limits<uint64_t>::max() % n;
  uint64_t r;
  do r = splitmix64(state);
  while (r >= limit);
  return r % n;
}

}  // namespace

extern "C" {

pkv_status pkv_bm_create(int32_t num_blocks, int32_t block_size, uint64_t seed, pkv_block_manager** out) {
  if (out == nullptr || num_blocks < 1 || block_size < 1) return PKV_ERR_INVALID_ARG;
  *out = nullptr;
  pkv_block_manager* bm = new (std::nothrow) pkv_block_manager();
  if (bm == nullptr) return PKV_ERR_OUT_OF_BLOCKS;
  try {
    bm->num_blocks = num_blocks;
    bm->block_size = block_size;
    bm->ref.assign((size_t)num_blocks, 0);
    // hand-out order: order[0] first. Fisher-Yates over the ids when seeded.
    std::vector<int32_t> order((size_t)num_blocks);
    for (int32_t i = 0; i < num_blocks; ++i) order[(size_t)i] = i;
    if (seed != 0) {
      uint64_t st = seed;
      for (int32_t i = num_blocks - 1; i > 0; --i) {
        const int32_t j = (int32_t)below(st, (uint64_t)i + 1);
        const int32_t t = order[(size_t)i];
        order[(size_t)i] = order[(size_t)j];
        order[(size_t)j] = t;
      }
    }
    bm->free_stack.assign(order.rbegin(), order.rend());
  } catch (...) {
    delete bm;
    return PKV_ERR_OUT_OF_BLOCKS;
  }
  *out = bm;
  return PKV_OK;
}

void pkv_bm_destroy(pkv_block_manager* bm) { delete bm; }

pkv_status pkv_bm_add_seq(pkv_block_manager* bm, int32_t* seq) {
  if (bm == nullptr || seq == nullptr) return PKV_ERR_INVALID_ARG;
  try {
    *seq = bm->new_id();
  } catch (...) {
    return PKV_ERR_OUT_OF_BLOCKS;
  }
  return PKV_OK;
}

pkv_status pkv_bm_fork(pkv_block_manager* bm, int32_t parent, int32_t* child) {
  if (bm == nullptr || child == nullptr || !bm->is_live(parent)) return PKV_ERR_INVALID_ARG;
  try {
    // reserve first: new_id() may grow `seqs` and move the parent's record
    std::vector<int32_t> table = bm->seqs[(size_t)parent].table;
    const int64_t len = bm->seqs[(size_t)parent].len;
    const int32_t c = bm->new_id();
    pkv_block_manager::Seq& s = bm->seqs[(size_t)c];
    s.table.swap(table);
    s.len = len;
    for (int32_t b : s.table) ++bm->ref[(size_t)b];
    *child = c;
  } catch (...) {
    return PKV_ERR_OUT_OF_BLOCKS;
  }
  return PKV_OK;
}

pkv_status pkv_bm_free_seq(pkv_block_manager* bm, int32_t seq) {
  if (bm == nullptr || !bm->is_live(seq)) return PKV_ERR_INVALID_ARG;
  pkv_block_manager::Seq& s = bm->seqs[(size_t)seq];
  try {
    bm->free_ids.reserve(bm->free_ids.size() + 1);
  } catch (...) {
    return PKV_ERR_OUT_OF_BLOCKS;
  }
  for (int32_t b : s.table) bm->drop_ref(b);
  s.table.clear();
  s.table.shrink_to_fit();
  s.len = 0;
  s.live = false;
  bm->free_ids.push_back(seq);
  return PKV_OK;
}

pkv_status pkv_bm_append(pkv_block_manager* bm, int32_t seq, int32_t n, int64_t* slots, int64_t* cow_pair,
                         int32_t* num_cow) {
  if (bm == nullptr || n < 0 || !bm->is_live(seq)) return PKV_ERR_INVALID_ARG;
  if (num_cow != nullptr) *num_cow = 0;
  if (n == 0) return PKV_OK;
  pkv_block_manager::Seq& s = bm->seqs[(size_t)seq];
  const int64_t bs = bm->block_size;
  const int64_t off0 = s.len % bs;
  // a write into a partly filled last block that others still hold copies it
  const bool cow = off0 != 0 && bm->ref[(size_t)s.table.back()] > 1;
  const int64_t new_blocks = (s.len + n + bs - 1) / bs - (s.len + bs - 1) / bs;
  const int64_t need = new_blocks + (cow ? 1 : 0);
  if (need > (int64_t)bm->free_stack.size()) return PKV_ERR_OUT_OF_BLOCKS;
  try {
    s.table.reserve(s.table.size() + (size_t)new_blocks);
  } catch (...) {
    return PKV_ERR_OUT_OF_BLOCKS;
  }
  if (cow) {
    const int32_t src = s.table.back();
    const int32_t dst = bm->take_block();
    --bm->ref[(size_t)src];  // still held by another sequence: never reaches 0 here
    s.table.back() = dst;
    ++bm->cow_copies;
    if (cow_pair != nullptr) {
      cow_pair[0] = src;
      cow_pair[1] = dst;
    }
    if (num_cow != nullptr) *num_cow = 1;
  }
  for (int32_t i = 0; i < n; ++i) {
    const int64_t off = s.len % bs;
    if (off == 0) s.table.push_back(bm->take_block());
    if (slots != nullptr) slots[i] = (int64_t)s.table.back() * bs + off;
    ++s.len;
  }
  return PKV_OK;
}

pkv_status pkv_bm_append_batch(pkv_block_manager* bm, const int32_t* seqs, const int32_t* counts, int32_t n,
                               int64_t* slots, int64_t* cow_pairs, int32_t* num_cow) {
  if (bm == nullptr || n < 0 || (n > 0 && (seqs == nullptr || counts == nullptr))) return PKV_ERR_INVALID_ARG;
  if (num_cow != nullptr) *num_cow = 0;
  if (n == 0) return PKV_OK;
  const int64_t bs = bm->block_size;
  int64_t need = 0;
  pkv_status bad = PKV_OK;
  try {
    bm->ensure_scratch();
    // blocks the batch takes, with the reference drops of earlier copies in it
    for (int32_t i = 0; i < n && bad == PKV_OK; ++i) {
      if (!bm->is_live(seqs[i]) || counts[i] < 0 || !bm->mark(seqs[i])) {
        bad = PKV_ERR_INVALID_ARG;
        break;
      }
      if (counts[i] == 0) continue;
      const pkv_block_manager::Seq& s = bm->seqs[(size_t)seqs[i]];
      if (s.len % bs != 0) {
        const int32_t last = s.table.back();
        if (bm->ref[(size_t)last] - bm->blk_drop[(size_t)last] > 1) {
          ++need;
          bm->touch(last);
          ++bm->blk_drop[(size_t)last];
        }
      }
      need += (s.len + counts[i] + bs - 1) / bs - (s.len + bs - 1) / bs;
    }
  } catch (...) {
    bad = PKV_ERR_OUT_OF_BLOCKS;
  }
  bm->reset_scratch();
  if (bad != PKV_OK) return bad;
  if (need > (int64_t)bm->free_stack.size()) return PKV_ERR_OUT_OF_BLOCKS;
  int64_t at = 0;
  int32_t ncow = 0;
  for (int32_t i = 0; i < n; ++i) {
    int32_t c = 0;
    const pkv_status st = pkv_bm_append(bm, seqs[i], counts[i], slots != nullptr ? slots + at : nullptr,
                                        cow_pairs != nullptr ? cow_pairs + 2 * (size_t)ncow : nullptr, &c);
    if (st != PKV_OK) return st;  // not reached: the batch was checked to fit
    ncow += c;
    at += counts[i];
  }
  if (num_cow != nullptr) *num_cow = ncow;
  return PKV_OK;
}

pkv_status pkv_bm_beam_step_many(pkv_block_manager* bm, const int32_t* beams, const int32_t* parents,
                                 int32_t requests, int32_t width, int32_t n_new, int32_t* new_beams, int64_t* slots,
                                 int64_t* cow_pairs, int32_t* num_cow, int32_t* shared_blocks) {
  if (bm == nullptr || beams == nullptr || parents == nullptr || new_beams == nullptr || requests < 0 ||
      width < 1 || n_new < 0)
    return PKV_ERR_INVALID_ARG;
  if (num_cow != nullptr) *num_cow = 0;
  if (requests == 0) return PKV_OK;
  const int64_t bs = bm->block_size;
  const size_t total = (size_t)requests * (size_t)width;
  std::vector<int32_t> children;
  std::vector<char> taken;  // a parent's first child already placed
  pkv_status bad = PKV_OK;
  int64_t need = 0, released = 0;
  try {  // every allocation of the call happens here, before anything changes
    children.assign(total, 0);
    taken.assign(total, 0);
    bm->ensure_scratch();
    for (size_t k = 0; k < total; ++k)
      if (!bm->is_live(beams[k]) || !bm->mark(beams[k])) {
        bad = PKV_ERR_INVALID_ARG;
        break;
      }
    for (size_t k = 0; k < total && bad == PKV_OK; ++k) {
      if (parents[k] < 0 || parents[k] >= width) {
        bad = PKV_ERR_INVALID_ARG;
        break;
      }
      ++children[k / (size_t)width * (size_t)width + (size_t)parents[k]];
    }
    if (bad == PKV_OK) {
      // reference counts after every request's forks and ends
      for (size_t k = 0; k < total; ++k) {
        const int32_t d = children[k] == 0 ? -1 : children[k] - 1;
        if (d == 0) continue;
        for (int32_t b : bm->seqs[(size_t)beams[k]].table) {
          bm->touch(b);
          bm->blk_delta[(size_t)b] += d;
        }
      }
      for (int32_t b : bm->touched)
        if (bm->ref[(size_t)b] > 0 && bm->ref[(size_t)b] + bm->blk_delta[(size_t)b] == 0) ++released;
      // blocks the appends take, in order (copies made earlier in the step counted)
      if (n_new > 0)
        for (size_t k = 0; k < total; ++k) {
          const size_t r0 = k / (size_t)width * (size_t)width;
          const pkv_block_manager::Seq& s = bm->seqs[(size_t)beams[r0 + (size_t)parents[k]]];
          if (s.len % bs != 0) {
            const int32_t last = s.table.back();
            bm->touch(last);
            if (bm->ref[(size_t)last] + bm->blk_delta[(size_t)last] - bm->blk_drop[(size_t)last] > 1) {
              ++need;
              ++bm->blk_drop[(size_t)last];
            }
          }
          need += (s.len + n_new + bs - 1) / bs - (s.len + bs - 1) / bs;
        }
    }
    if (bad == PKV_OK) {
      bm->seqs.reserve(bm->seqs.size() + total);
      bm->free_ids.reserve(bm->free_ids.size() + total);
    }
  } catch (...) {
    bad = PKV_ERR_OUT_OF_BLOCKS;
  }
  bm->reset_scratch();
  if (bad != PKV_OK) return bad;
  if (need > (int64_t)bm->free_stack.size() + released) return PKV_ERR_OUT_OF_BLOCKS;
  // every request's ends, then its forks (a parent's first child keeps its id)
  for (size_t k = 0; k < total; ++k)
    if (children[k] == 0) pkv_bm_free_seq(bm, beams[k]);
  for (size_t k = 0; k < total; ++k) {
    const size_t j = k / (size_t)width * (size_t)width + (size_t)parents[k];
    if (!taken[j]) {
      taken[j] = 1;
      new_beams[k] = beams[j];
    } else if (pkv_bm_fork(bm, beams[j], &new_beams[k]) != PKV_OK) {
      return PKV_ERR_OUT_OF_BLOCKS;  // host memory ran out while copying a table
    }
  }
  // then every new beam's tokens, in order
  int64_t at = 0;
  int32_t ncow = 0;
  if (n_new > 0)
    for (size_t k = 0; k < total; ++k) {
      int32_t c = 0;
      const pkv_status st = pkv_bm_append(bm, new_beams[k], n_new, slots != nullptr ? slots + at : nullptr,
                                          cow_pairs != nullptr ? cow_pairs + 2 * (size_t)ncow : nullptr, &c);
      if (st != PKV_OK) return st;  // not reached: the step was checked to fit
      ncow += c;
      at += n_new;
    }
  if (num_cow != nullptr) *num_cow = ncow;
  if (shared_blocks != nullptr)
    for (int32_t r = 0; r < requests; ++r)
      pkv_bm_common_prefix(bm, new_beams + (size_t)r * width, width, shared_blocks + r);
  return PKV_OK;
}

pkv_status pkv_bm_beam_step(pkv_block_manager* bm, const int32_t* beams, const int32_t* parents, int32_t width,
                            int32_t n_new, int32_t* new_beams, int64_t* slots, int64_t* cow_pairs,
                            int32_t* num_cow) {
  return pkv_bm_beam_step_many(bm, beams, parents, 1, width, n_new, new_beams, slots, cow_pairs, num_cow, nullptr);
}

pkv_status pkv_bm_seq_info(const pkv_block_manager* bm, int32_t seq, int64_t* length, int32_t* num_blocks) {
  if (bm == nullptr || !bm->is_live(seq)) return PKV_ERR_INVALID_ARG;
  const pkv_block_manager::Seq& s = bm->seqs[(size_t)seq];
  if (length != nullptr) *length = s.len;
  if (num_blocks != nullptr) *num_blocks = (int32_t)s.table.size();
  return PKV_OK;
}

pkv_status pkv_bm_export(const pkv_block_manager* bm, const int32_t* seqs, int32_t n, int32_t max_blocks,
                         int32_t* block_tables, int32_t* context_lens) {
  if (bm == nullptr || n < 0 || max_blocks < 0) return PKV_ERR_INVALID_ARG;
  if (n > 0 && (seqs == nullptr || block_tables == nullptr || context_lens == nullptr)) return PKV_ERR_INVALID_ARG;
  for (int32_t i = 0; i < n; ++i) {
    if (!bm->is_live(seqs[i])) return PKV_ERR_INVALID_ARG;
    const pkv_block_manager::Seq& s = bm->seqs[(size_t)seqs[i]];
    if (s.table.size() > (size_t)max_blocks || s.len > std::numeric_limits<int32_t>::max())
      return PKV_ERR_INVALID_ARG;
  }
  for (int32_t i = 0; i < n; ++i) {
    const pkv_block_manager::Seq& s = bm->seqs[(size_t)seqs[i]];
    int32_t* row = block_tables + (size_t)i * (size_t)max_blocks;
    size_t j = 0;
    for (; j < s.table.size(); ++j) row[j] = s.table[j];
    for (; j < (size_t)max_blocks; ++j) row[j] = -1;
    context_lens[i] = (int32_t)s.len;
  }
  return PKV_OK;
}

pkv_status pkv_bm_common_prefix(const pkv_block_manager* bm, const int32_t* seqs, int32_t n, int32_t* blocks) {
  if (bm == nullptr || blocks == nullptr || n < 1 || seqs == nullptr) return PKV_ERR_INVALID_ARG;
  for (int32_t i = 0; i < n; ++i)
    if (!bm->is_live(seqs[i])) return PKV_ERR_INVALID_ARG;
  const std::vector<int32_t>& t0 = bm->seqs[(size_t)seqs[0]].table;
  size_t k = t0.size();
  for (int32_t i = 1; i < n && k > 0; ++i) {
    const std::vector<int32_t>& t = bm->seqs[(size_t)seqs[i]].table;
    size_t j = 0;
    const size_t lim = k < t.size() ? k : t.size();
    while (j < lim && t[j] == t0[j]) ++j;
    k = j;
  }
  *blocks = (int32_t)k;
  return PKV_OK;
}

pkv_status pkv_bm_get_stats(const pkv_block_manager* bm, pkv_bm_stats* stats) {
  if (bm == nullptr || stats == nullptr) return PKV_ERR_INVALID_ARG;
  pkv_bm_stats st{};
  st.num_blocks = bm->num_blocks;
  st.free_blocks = (int64_t)bm->free_stack.size();
  st.used_blocks = st.num_blocks - st.free_blocks;
  st.cow_copies = bm->cow_copies;
  for (int32_t r : bm->ref)
    if (r > 1) ++st.shared_blocks;
  // furthest token kept in each used block by any live sequence
  std::vector<int32_t> reach;
  try {
    reach.assign((size_t)bm->num_blocks, 0);
  } catch (...) {
    return PKV_ERR_OUT_OF_BLOCKS;
  }
  const int64_t bs = bm->block_size;
  for (const pkv_block_manager::Seq& s : bm->seqs) {
    if (!s.live) continue;
    ++st.live_seqs;
    st.logical_tokens += s.len;
    st.logical_blocks += (int64_t)s.table.size();
    for (size_t j = 0; j < s.table.size(); ++j) {
      const int64_t rest = s.len - (int64_t)j * bs;
      const int32_t used = (int32_t)(rest < bs ? rest : bs);
      int32_t& r = reach[(size_t)s.table[j]];
      if (used > r) r = used;
    }
  }
  for (int32_t r : reach) st.filled_slots += r;
  *stats = st;
  return PKV_OK;
}

}  // extern "C"
