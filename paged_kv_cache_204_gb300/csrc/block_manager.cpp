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
#include <unordered_map>
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
  try {
    std::vector<int32_t> ids(seqs, seqs + n);
    std::sort(ids.begin(), ids.end());
    if (std::adjacent_find(ids.begin(), ids.end()) != ids.end()) return PKV_ERR_INVALID_ARG;
    // blocks the batch takes, with the reference drops of earlier copies in it
    std::unordered_map<int32_t, int32_t> dropped;
    for (int32_t i = 0; i < n; ++i) {
      if (!bm->is_live(seqs[i]) || counts[i] < 0) return PKV_ERR_INVALID_ARG;
      if (counts[i] == 0) continue;
      const pkv_block_manager::Seq& s = bm->seqs[(size_t)seqs[i]];
      if (s.len % bs != 0) {
        const int32_t last = s.table.back();
        auto it = dropped.find(last);
        const int32_t d = it == dropped.end() ? 0 : it->second;
        if (bm->ref[(size_t)last] - d > 1) {
          ++need;
          ++dropped[last];
        }
      }
      need += (s.len + counts[i] + bs - 1) / bs - (s.len + bs - 1) / bs;
    }
  } catch (...) {
    return PKV_ERR_OUT_OF_BLOCKS;
  }
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

pkv_status pkv_bm_beam_step(pkv_block_manager* bm, const int32_t* beams, const int32_t* parents, int32_t width,
                            int32_t n_new, int32_t* new_beams, int64_t* slots, int64_t* cow_pairs,
                            int32_t* num_cow) {
  if (bm == nullptr || beams == nullptr || parents == nullptr || new_beams == nullptr || width < 1 || n_new < 0)
    return PKV_ERR_INVALID_ARG;
  if (num_cow != nullptr) *num_cow = 0;
  const int64_t bs = bm->block_size;
  std::vector<int32_t> children((size_t)width, 0);
  try {
    std::vector<int32_t> ids(beams, beams + width);
    std::sort(ids.begin(), ids.end());
    if (std::adjacent_find(ids.begin(), ids.end()) != ids.end()) return PKV_ERR_INVALID_ARG;
    for (int32_t j = 0; j < width; ++j)
      if (!bm->is_live(beams[j])) return PKV_ERR_INVALID_ARG;
    for (int32_t i = 0; i < width; ++i) {
      if (parents[i] < 0 || parents[i] >= width) return PKV_ERR_INVALID_ARG;
      ++children[(size_t)parents[i]];
    }
    // reference counts after the step's forks and ends, for the blocks involved
    std::unordered_map<int32_t, int32_t> delta;
    for (int32_t j = 0; j < width; ++j) {
      const int32_t d = children[(size_t)j] == 0 ? -1 : children[(size_t)j] - 1;
      if (d == 0) continue;
      for (int32_t b : bm->seqs[(size_t)beams[j]].table) delta[b] += d;
    }
    int64_t released = 0;
    for (const auto& kv : delta)
      if (bm->ref[(size_t)kv.first] + kv.second == 0) ++released;
    // blocks the appends take (copies made earlier in the step counted)
    int64_t need = 0;
    std::unordered_map<int32_t, int32_t> dropped;
    if (n_new > 0) {
      for (int32_t i = 0; i < width; ++i) {
        const pkv_block_manager::Seq& s = bm->seqs[(size_t)beams[parents[i]]];
        if (s.len % bs != 0) {
          const int32_t last = s.table.back();
          auto it = delta.find(last);
          const int32_t holders = bm->ref[(size_t)last] + (it == delta.end() ? 0 : it->second) - dropped[last];
          if (holders > 1) {
            ++need;
            ++dropped[last];
          }
        }
        need += (s.len + n_new + bs - 1) / bs - (s.len + bs - 1) / bs;
      }
    }
    if (need > (int64_t)bm->free_stack.size() + released) return PKV_ERR_OUT_OF_BLOCKS;
    bm->seqs.reserve(bm->seqs.size() + (size_t)width);
    bm->free_ids.reserve(bm->free_ids.size() + (size_t)width);
  } catch (...) {
    return PKV_ERR_OUT_OF_BLOCKS;
  }
  // end the beams nobody continues, then hand out the survivors
  for (int32_t j = 0; j < width; ++j)
    if (children[(size_t)j] == 0) pkv_bm_free_seq(bm, beams[j]);
  std::vector<char> taken((size_t)width, 0);
  for (int32_t i = 0; i < width; ++i) {
    const int32_t j = parents[i];
    if (!taken[(size_t)j]) {
      taken[(size_t)j] = 1;
      new_beams[i] = beams[j];
    } else if (pkv_bm_fork(bm, beams[j], &new_beams[i]) != PKV_OK) {
      return PKV_ERR_OUT_OF_BLOCKS;  // host memory ran out while copying a table
    }
  }
  std::vector<int32_t> counts((size_t)width, n_new);
  return pkv_bm_append_batch(bm, new_beams, counts.data(), width, slots, cow_pairs, num_cow);
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
