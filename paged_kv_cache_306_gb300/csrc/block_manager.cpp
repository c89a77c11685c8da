// block_manager.cpp -- host-side block manager of a paged KV pool (pa_block_manager.h).
//
// The bookkeeping the pages describe ("vLLM's PagedAttention: why the KV cache is
// paged", §4.1, §4.2): a free list of physical blocks, per-block reference
// counts, per-sequence logical -> physical block lists, sharing by fork and
// copy-on-write of a shared, partly filled last block before a token is appended
// to it.  Every call checks all of its preconditions before it changes
// anything, so a failed call leaves the manager as it was.
#include <stdint.h>

#include <cstdio>
#include <mutex>
#include <unordered_map>
#include <unordered_set>
#include <vector>

#include "pa.h"
#include "pa_block_manager.h"

namespace pa {
pa_status record_failure(pa_status st, const char* message);
}

namespace {

struct Sequence {
  int64_t len = 0;
  std::vector<int32_t> blocks;  // logical block i -> physical block
};

pa_status failf(pa_status st, const char* fmt, long long a, long long b = 0) {
  char msg[256];
  std::snprintf(msg, sizeof msg, fmt, a, b);
  return pa::record_failure(st, msg);
}

}  // namespace

struct pa_block_manager {
  int64_t num_blocks = 0;
  int block_size = 0;
  std::vector<int32_t> free_list;  // a stack: the lowest free id on top
  std::vector<int32_t> refcount;
  std::unordered_map<int64_t, Sequence> seqs;
  mutable std::mutex mu;

  int32_t take() {
    const int32_t b = free_list.back();
    free_list.pop_back();
    refcount[b] = 1;
    return b;
  }
  void drop(int32_t b) {
    if (--refcount[b] == 0) free_list.push_back(b);
  }
  int64_t blocks_for(int64_t tokens) const { return (tokens + block_size - 1) / block_size; }
};

extern "C" {

pa_status pa_bm_create(int64_t num_blocks, int block_size, pa_block_manager** out) {
  if (!out) return pa::record_failure(PA_ERR_INVALID_ARG, "null output pointer");
  *out = nullptr;
  if (num_blocks < 1 || num_blocks > 0x7fffffffLL)
    return failf(PA_ERR_INVALID_ARG, "num_blocks %lld outside [1, 2^31 - 1]", num_blocks);
  if (block_size < 1) return failf(PA_ERR_INVALID_ARG, "block_size %lld < 1", block_size);
  auto* bm = new pa_block_manager;
  bm->num_blocks = num_blocks;
  bm->block_size = block_size;
  bm->refcount.assign(static_cast<size_t>(num_blocks), 0);
  bm->free_list.reserve(static_cast<size_t>(num_blocks));
  for (int64_t b = num_blocks - 1; b >= 0; --b) bm->free_list.push_back(static_cast<int32_t>(b));
  *out = bm;
  return PA_OK;
}

void pa_bm_destroy(pa_block_manager* bm) { delete bm; }

int64_t pa_bm_num_free_blocks(const pa_block_manager* bm) {
  if (!bm) return 0;
  std::lock_guard<std::mutex> lock(bm->mu);
  return static_cast<int64_t>(bm->free_list.size());
}

pa_status pa_bm_add_sequence(pa_block_manager* bm, int64_t seq_id, int64_t num_tokens, int64_t* slots) {
  if (!bm) return pa::record_failure(PA_ERR_INVALID_ARG, "null manager");
  std::lock_guard<std::mutex> lock(bm->mu);
  if (num_tokens < 0) return failf(PA_ERR_INVALID_ARG, "num_tokens %lld < 0", num_tokens);
  if (bm->seqs.count(seq_id)) return failf(PA_ERR_INVALID_ARG, "sequence %lld exists", seq_id);
  const int64_t need = bm->blocks_for(num_tokens);
  if (need > static_cast<int64_t>(bm->free_list.size()))
    return failf(PA_ERR_OUT_OF_BLOCKS, "%lld blocks needed, %lld free", need, (long long)bm->free_list.size());
  Sequence sq;
  sq.len = num_tokens;
  sq.blocks.reserve(static_cast<size_t>(need));
  for (int64_t i = 0; i < need; ++i) sq.blocks.push_back(bm->take());
  if (slots)
    for (int64_t t = 0; t < num_tokens; ++t)
      slots[t] = static_cast<int64_t>(sq.blocks[t / bm->block_size]) * bm->block_size + t % bm->block_size;
  bm->seqs.emplace(seq_id, std::move(sq));
  return PA_OK;
}

pa_status pa_bm_fork(pa_block_manager* bm, int64_t parent_id, int64_t child_id) {
  if (!bm) return pa::record_failure(PA_ERR_INVALID_ARG, "null manager");
  std::lock_guard<std::mutex> lock(bm->mu);
  auto it = bm->seqs.find(parent_id);
  if (it == bm->seqs.end()) return failf(PA_ERR_INVALID_ARG, "no sequence %lld", parent_id);
  if (bm->seqs.count(child_id)) return failf(PA_ERR_INVALID_ARG, "sequence %lld exists", child_id);
  Sequence child = it->second;
  for (int32_t b : child.blocks) ++bm->refcount[b];
  bm->seqs.emplace(child_id, std::move(child));
  return PA_OK;
}

pa_status pa_bm_free_sequence(pa_block_manager* bm, int64_t seq_id) {
  if (!bm) return pa::record_failure(PA_ERR_INVALID_ARG, "null manager");
  std::lock_guard<std::mutex> lock(bm->mu);
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return failf(PA_ERR_INVALID_ARG, "no sequence %lld", seq_id);
  // return blocks last first, so that a freed sequence's first block is on top
  for (auto b = it->second.blocks.rbegin(); b != it->second.blocks.rend(); ++b) bm->drop(*b);
  bm->seqs.erase(it);
  return PA_OK;
}

pa_status pa_bm_append_tokens(pa_block_manager* bm, const int64_t* seq_ids, int num_seqs, int64_t* slot_mapping,
                              int64_t* copies, int64_t max_copies, int64_t* num_copies) {
  if (!bm) return pa::record_failure(PA_ERR_INVALID_ARG, "null manager");
  std::lock_guard<std::mutex> lock(bm->mu);
  if (num_seqs < 0) return failf(PA_ERR_INVALID_ARG, "num_seqs %lld < 0", num_seqs);
  if (num_seqs > 0 && (!seq_ids || !slot_mapping || !num_copies))
    return pa::record_failure(PA_ERR_INVALID_ARG, "null pointer");
  if (num_copies) *num_copies = 0;
  // Check everything first: known, distinct ids, enough free blocks and copy
  // room.  The decisions are simulated in batch order on the reference counts,
  // so that of several sequences of the batch that share a partly filled last
  // block, all but the last to append copy it and the last writes in place.
  std::unordered_set<int64_t> seen;
  std::unordered_map<int32_t, int32_t> dropped;  // simulated lost references per block
  int64_t need_blocks = 0, need_copies = 0;
  for (int i = 0; i < num_seqs; ++i) {
    auto it = bm->seqs.find(seq_ids[i]);
    if (it == bm->seqs.end()) return failf(PA_ERR_INVALID_ARG, "no sequence %lld", seq_ids[i]);
    if (!seen.insert(seq_ids[i]).second) return failf(PA_ERR_INVALID_ARG, "sequence %lld listed twice", seq_ids[i]);
    const Sequence& sq = it->second;
    if (sq.len % bm->block_size == 0) {
      ++need_blocks;  // the last block is full (or there is none): a fresh one
    } else {
      const int32_t last = sq.blocks.back();
      if (bm->refcount[last] - dropped[last] > 1) {  // shared, partly filled: copy-on-write
        ++need_blocks;
        ++need_copies;
        ++dropped[last];
      }
    }
  }
  if (need_blocks > static_cast<int64_t>(bm->free_list.size()))
    return failf(PA_ERR_OUT_OF_BLOCKS, "%lld blocks needed, %lld free", need_blocks, (long long)bm->free_list.size());
  if (need_copies > max_copies || (need_copies > 0 && !copies))
    return failf(PA_ERR_WORKSPACE, "%lld copy pairs, room for %lld", need_copies, max_copies);
  // Apply the same decisions to the real counts.  A copied block keeps at least
  // one reference (the sequence that writes in place, or one outside the batch),
  // so it is not freed and cannot be handed out as the copy's destination.
  int64_t nc = 0;
  for (int i = 0; i < num_seqs; ++i) {
    Sequence& sq = bm->seqs[seq_ids[i]];
    if (sq.len % bm->block_size == 0) {
      sq.blocks.push_back(bm->take());
    } else if (bm->refcount[sq.blocks.back()] > 1) {
      const int32_t src = sq.blocks.back();
      const int32_t dst = bm->take();
      copies[2 * nc] = src;
      copies[2 * nc + 1] = dst;
      ++nc;
      bm->drop(src);
      sq.blocks.back() = dst;
    }
    slot_mapping[i] = static_cast<int64_t>(sq.blocks.back()) * bm->block_size + sq.len % bm->block_size;
    ++sq.len;
  }
  *num_copies = nc;
  return PA_OK;
}

pa_status pa_bm_seq_len(const pa_block_manager* bm, int64_t seq_id, int64_t* len) {
  if (!bm || !len) return pa::record_failure(PA_ERR_INVALID_ARG, "null pointer");
  std::lock_guard<std::mutex> lock(bm->mu);
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return failf(PA_ERR_INVALID_ARG, "no sequence %lld", seq_id);
  *len = it->second.len;
  return PA_OK;
}

pa_status pa_bm_block_tables(const pa_block_manager* bm, const int64_t* seq_ids, int num_seqs, int32_t* block_tables,
                             int max_blocks_per_seq, int32_t* seq_lens) {
  if (!bm) return pa::record_failure(PA_ERR_INVALID_ARG, "null manager");
  std::lock_guard<std::mutex> lock(bm->mu);
  if (num_seqs < 0 || max_blocks_per_seq < 1)
    return failf(PA_ERR_INVALID_ARG, "num_seqs %lld, max_blocks_per_seq %lld", num_seqs, max_blocks_per_seq);
  if (num_seqs > 0 && (!seq_ids || !block_tables || !seq_lens)) return pa::record_failure(PA_ERR_INVALID_ARG, "null pointer");
  for (int i = 0; i < num_seqs; ++i) {
    auto it = bm->seqs.find(seq_ids[i]);
    if (it == bm->seqs.end()) return failf(PA_ERR_INVALID_ARG, "no sequence %lld", seq_ids[i]);
    if (static_cast<int64_t>(it->second.blocks.size()) > max_blocks_per_seq)
      return failf(PA_ERR_INVALID_ARG, "sequence %lld has more than %lld blocks", seq_ids[i], max_blocks_per_seq);
    if (it->second.len > 0x7fffffffLL) return failf(PA_ERR_INVALID_ARG, "sequence %lld longer than int32", seq_ids[i]);
  }
  for (int i = 0; i < num_seqs; ++i) {
    const Sequence& sq = bm->seqs.at(seq_ids[i]);
    int32_t* row = block_tables + static_cast<int64_t>(i) * max_blocks_per_seq;
    for (int j = 0; j < max_blocks_per_seq; ++j) row[j] = j < static_cast<int>(sq.blocks.size()) ? sq.blocks[j] : -1;
    seq_lens[i] = static_cast<int32_t>(sq.len);
  }
  return PA_OK;
}

pa_status pa_bm_prefix_groups(const pa_block_manager* bm, const int64_t* seq_ids, int num_seqs, int32_t* prefix_group,
                              int32_t* prefix_blocks) {
  if (!bm) return pa::record_failure(PA_ERR_INVALID_ARG, "null manager");
  std::lock_guard<std::mutex> lock(bm->mu);
  if (num_seqs < 0) return failf(PA_ERR_INVALID_ARG, "num_seqs %lld", static_cast<long long>(num_seqs));
  if (num_seqs > 0 && (!seq_ids || !prefix_group || !prefix_blocks))
    return pa::record_failure(PA_ERR_INVALID_ARG, "null pointer");
  std::vector<const std::vector<int32_t>*> rows(static_cast<size_t>(num_seqs));
  for (int i = 0; i < num_seqs; ++i) {
    auto it = bm->seqs.find(seq_ids[i]);
    if (it == bm->seqs.end()) return failf(PA_ERR_INVALID_ARG, "no sequence %lld", seq_ids[i]);
    rows[static_cast<size_t>(i)] = &it->second.blocks;
  }
  // a group: consecutive sequences whose first block is one physical block (sharing is
  // always a prefix, so two sequences that share anything share block 0); each is
  // compared with the longest sequence of its group
  for (int i = 0; i < num_seqs;) {
    int j = i + 1;
    while (j < num_seqs && !rows[i]->empty() && !rows[j]->empty() && (*rows[j])[0] == (*rows[i])[0]) ++j;
    int ref = i;
    for (int t = i; t < j; ++t)
      if (rows[t]->size() > rows[ref]->size()) ref = t;
    for (int t = i; t < j; ++t) {
      const std::vector<int32_t>& a = *rows[t];
      const std::vector<int32_t>& r = *rows[ref];
      size_t n = 0;
      while (n < a.size() && n < r.size() && a[n] == r[n]) ++n;
      prefix_group[t] = i;
      prefix_blocks[t] = j - i > 1 ? static_cast<int32_t>(n) : 0;
    }
    i = j;
  }
  return PA_OK;
}

pa_status pa_bm_refcount(const pa_block_manager* bm, int64_t block, int* refcount) {
  if (!bm || !refcount) return pa::record_failure(PA_ERR_INVALID_ARG, "null pointer");
  std::lock_guard<std::mutex> lock(bm->mu);
  if (block < 0 || block >= bm->num_blocks) return failf(PA_ERR_INVALID_ARG, "block %lld outside the pool", block);
  *refcount = bm->refcount[static_cast<size_t>(block)];
  return PA_OK;
}

}  // extern "C"
