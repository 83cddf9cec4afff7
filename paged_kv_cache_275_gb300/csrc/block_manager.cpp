// Host block manager of the paged KV cache (declared in include/pagedkv.h).
//
// "跟着 Claude Code，我用 Python 实现了一个轻量级的 vLLM", section
// "核心机制一：分页 KV Cache": the cache is a pool of fixed 16-token blocks, a
// sequence takes a new block only when it needs more room, and all of its
// blocks are returned when it ends.  "从零实现一个 mini vLLM--开篇", section 5
// (phase 4): every request owns a block table.  "v0版本介绍", section
// "为什么需要推理框架": a block is taken only when the current one is full, and
// requests may share the KV blocks of a common prompt.
//
// Sharing is by reference count.  fork() makes a child that points at all of
// its parent's blocks.  A sequence about to append into a partly filled
// block that others still reference first moves onto a fresh block
// (copy-on-write): the manager reports the (src, dst) pair and the caller
// copies the block on the GPU (pkv_copy_blocks) before appending.
//
// Host memory only; one mutex per manager serialises its calls.  Every call
// validates first and changes nothing when it fails.
#include <cstdint>
#include <cstdio>
#include <deque>
#include <mutex>
#include <unordered_map>
#include <unordered_set>
#include <vector>

#include "pagedkv.h"
#include "pkv_internal.h"

namespace {

constexpr int64_t kBlock = PKV_BLOCK_SIZE;

struct Sequence {
  std::vector<int64_t> blocks;
  int64_t length = 0;
};

pkv_status bm_fail(pkv_status status, const char* fmt, long long a = 0, long long b = 0) {
  char msg[256];
  snprintf(msg, sizeof msg, fmt, a, b);
  pkv::set_error_message(msg);
  return status;
}

pkv_status bm_ok() {
  pkv::set_error_message("");
  return PKV_OK;
}

}  // namespace

struct pkv_block_manager {
  std::mutex mu;
  int64_t num_blocks = 0;
  std::deque<int64_t> free_list;     // front = next block handed out
  std::vector<int32_t> refs;         // references per block (0 = on the free list)
  std::unordered_map<int64_t, Sequence> seqs;

  int64_t take() {
    const int64_t b = free_list.front();
    free_list.pop_front();
    refs[b] = 1;
    return b;
  }
  void release(int64_t b) {
    if (--refs[b] == 0) free_list.push_back(b);
  }
};

extern "C" {

pkv_status pkv_bm_create(int64_t num_blocks, const int64_t* initial_free_order, pkv_block_manager** out) {
  if (!out) return bm_fail(PKV_ERR_INVALID_ARGUMENT, "out is null");
  if (num_blocks <= 0 || num_blocks > (int64_t{1} << 31))
    return bm_fail(PKV_ERR_INVALID_ARGUMENT, "num_blocks out of range (got %lld)", num_blocks);
  auto* bm = new pkv_block_manager();
  bm->num_blocks = num_blocks;
  bm->refs.assign(static_cast<size_t>(num_blocks), 0);
  if (initial_free_order) {
    std::vector<char> seen(static_cast<size_t>(num_blocks), 0);
    for (int64_t i = 0; i < num_blocks; ++i) {
      const int64_t b = initial_free_order[i];
      if (b < 0 || b >= num_blocks || seen[b]) {
        delete bm;
        return bm_fail(PKV_ERR_INVALID_ARGUMENT, "initial_free_order is not a permutation (entry %lld = %lld)", i, b);
      }
      seen[b] = 1;
      bm->free_list.push_back(b);
    }
  } else {
    for (int64_t b = 0; b < num_blocks; ++b) bm->free_list.push_back(b);
  }
  *out = bm;
  return bm_ok();
}

pkv_status pkv_bm_destroy(pkv_block_manager* bm) {
  if (!bm) return bm_fail(PKV_ERR_INVALID_ARGUMENT, "manager is null");
  delete bm;
  return bm_ok();
}

pkv_status pkv_bm_num_free(pkv_block_manager* bm, int64_t* num_free) {
  if (!bm || !num_free) return bm_fail(PKV_ERR_INVALID_ARGUMENT, "null argument");
  std::lock_guard<std::mutex> lock(bm->mu);
  *num_free = static_cast<int64_t>(bm->free_list.size());
  return bm_ok();
}

pkv_status pkv_bm_add_sequence(pkv_block_manager* bm, int64_t seq_id, int64_t num_tokens, int64_t* slots) {
  if (!bm) return bm_fail(PKV_ERR_INVALID_ARGUMENT, "manager is null");
  if (seq_id < 0) return bm_fail(PKV_ERR_INVALID_ARGUMENT, "seq_id must be >= 0 (got %lld)", seq_id);
  if (num_tokens < 0) return bm_fail(PKV_ERR_INVALID_ARGUMENT, "num_tokens must be >= 0 (got %lld)", num_tokens);
  std::lock_guard<std::mutex> lock(bm->mu);
  if (bm->seqs.count(seq_id)) return bm_fail(PKV_ERR_INVALID_ARGUMENT, "sequence %lld already exists", seq_id);
  const int64_t need = (num_tokens + kBlock - 1) / kBlock;
  if (need > static_cast<int64_t>(bm->free_list.size()))
    return bm_fail(PKV_ERR_NO_FREE_BLOCKS, "need %lld blocks, %lld free", need,
                   static_cast<long long>(bm->free_list.size()));
  Sequence s;
  s.length = num_tokens;
  s.blocks.reserve(static_cast<size_t>(need));
  for (int64_t i = 0; i < need; ++i) s.blocks.push_back(bm->take());
  if (slots)
    for (int64_t p = 0; p < num_tokens; ++p) slots[p] = s.blocks[p / kBlock] * kBlock + p % kBlock;
  bm->seqs.emplace(seq_id, std::move(s));
  return bm_ok();
}

pkv_status pkv_bm_append_slots(pkv_block_manager* bm, const int64_t* seq_ids, int32_t num_seqs, int64_t* slots,
                               int64_t* copies, int32_t* num_copies) {
  if (!bm || !num_copies) return bm_fail(PKV_ERR_INVALID_ARGUMENT, "null argument");
  if (num_seqs < 0) return bm_fail(PKV_ERR_INVALID_ARGUMENT, "num_seqs must be >= 0 (got %lld)", num_seqs);
  if (num_seqs > 0 && (!seq_ids || !slots || !copies)) return bm_fail(PKV_ERR_INVALID_ARGUMENT, "null argument");
  std::lock_guard<std::mutex> lock(bm->mu);
  // Validate, and count the blocks this call takes: a full last block needs a
  // new one; a partly filled last block that others still reference needs a
  // copy.  References drop as earlier sequences of the same call move off a
  // shared block, so the count replays those drops.
  std::unordered_set<int64_t> ids;
  std::unordered_map<int64_t, int32_t> dropped;
  int64_t need = 0;
  for (int32_t i = 0; i < num_seqs; ++i) {
    auto it = bm->seqs.find(seq_ids[i]);
    if (it == bm->seqs.end()) return bm_fail(PKV_ERR_INVALID_ARGUMENT, "unknown sequence %lld", seq_ids[i]);
    if (!ids.insert(seq_ids[i]).second) return bm_fail(PKV_ERR_INVALID_ARGUMENT, "sequence %lld listed twice", seq_ids[i]);
    const Sequence& s = it->second;
    if (s.length % kBlock == 0) {
      ++need;
    } else {
      const int64_t last = s.blocks.back();
      if (bm->refs[last] - dropped[last] > 1) {
        ++need;
        ++dropped[last];
      }
    }
  }
  if (need > static_cast<int64_t>(bm->free_list.size()))
    return bm_fail(PKV_ERR_NO_FREE_BLOCKS, "need %lld blocks, %lld free", need,
                   static_cast<long long>(bm->free_list.size()));
  int32_t n_copies = 0;
  for (int32_t i = 0; i < num_seqs; ++i) {
    Sequence& s = bm->seqs[seq_ids[i]];
    const int64_t pos = s.length;
    if (pos % kBlock == 0) {
      s.blocks.push_back(bm->take());
    } else {
      const int64_t last = s.blocks.back();
      if (bm->refs[last] > 1) {  // copy-on-write: move onto a private copy
        const int64_t fresh = bm->take();
        copies[2 * n_copies] = last;
        copies[2 * n_copies + 1] = fresh;
        ++n_copies;
        bm->release(last);
        s.blocks.back() = fresh;
      }
    }
    slots[i] = s.blocks.back() * kBlock + pos % kBlock;
    s.length = pos + 1;
  }
  *num_copies = n_copies;
  return bm_ok();
}

pkv_status pkv_bm_fork(pkv_block_manager* bm, int64_t parent_id, int64_t child_id) {
  if (!bm) return bm_fail(PKV_ERR_INVALID_ARGUMENT, "manager is null");
  if (child_id < 0) return bm_fail(PKV_ERR_INVALID_ARGUMENT, "child id must be >= 0 (got %lld)", child_id);
  std::lock_guard<std::mutex> lock(bm->mu);
  auto it = bm->seqs.find(parent_id);
  if (it == bm->seqs.end()) return bm_fail(PKV_ERR_INVALID_ARGUMENT, "unknown sequence %lld", parent_id);
  if (bm->seqs.count(child_id)) return bm_fail(PKV_ERR_INVALID_ARGUMENT, "sequence %lld already exists", child_id);
  Sequence child = it->second;
  for (int64_t b : child.blocks) ++bm->refs[b];
  bm->seqs.emplace(child_id, std::move(child));
  return bm_ok();
}

pkv_status pkv_bm_free_sequence(pkv_block_manager* bm, int64_t seq_id) {
  if (!bm) return bm_fail(PKV_ERR_INVALID_ARGUMENT, "manager is null");
  std::lock_guard<std::mutex> lock(bm->mu);
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return bm_fail(PKV_ERR_INVALID_ARGUMENT, "unknown sequence %lld", seq_id);
  for (int64_t b : it->second.blocks) bm->release(b);
  bm->seqs.erase(it);
  return bm_ok();
}

pkv_status pkv_bm_block_tables(pkv_block_manager* bm, const int64_t* seq_ids, int32_t num_seqs, int32_t width,
                               int32_t* tables, int32_t* lengths) {
  if (!bm) return bm_fail(PKV_ERR_INVALID_ARGUMENT, "manager is null");
  if (num_seqs < 0 || width <= 0) return bm_fail(PKV_ERR_INVALID_ARGUMENT, "bad num_seqs %lld or width %lld", num_seqs, width);
  if (num_seqs > 0 && (!seq_ids || !tables || !lengths)) return bm_fail(PKV_ERR_INVALID_ARGUMENT, "null argument");
  std::lock_guard<std::mutex> lock(bm->mu);
  for (int32_t i = 0; i < num_seqs; ++i) {
    auto it = bm->seqs.find(seq_ids[i]);
    if (it == bm->seqs.end()) return bm_fail(PKV_ERR_INVALID_ARGUMENT, "unknown sequence %lld", seq_ids[i]);
    if (static_cast<int64_t>(it->second.blocks.size()) > width)
      return bm_fail(PKV_ERR_INVALID_ARGUMENT, "sequence %lld needs %lld table entries", seq_ids[i],
                     static_cast<long long>(it->second.blocks.size()));
    if (it->second.length > INT32_MAX) return bm_fail(PKV_ERR_UNSUPPORTED, "sequence %lld too long", seq_ids[i]);
  }
  for (int32_t i = 0; i < num_seqs; ++i) {
    const Sequence& s = bm->seqs[seq_ids[i]];
    int32_t* row = tables + static_cast<int64_t>(i) * width;
    for (int32_t j = 0; j < width; ++j)
      row[j] = j < static_cast<int32_t>(s.blocks.size()) ? static_cast<int32_t>(s.blocks[j]) : -1;
    lengths[i] = static_cast<int32_t>(s.length);
  }
  return bm_ok();
}

pkv_status pkv_bm_ref_count(pkv_block_manager* bm, int64_t block, int32_t* count) {
  if (!bm || !count) return bm_fail(PKV_ERR_INVALID_ARGUMENT, "null argument");
  std::lock_guard<std::mutex> lock(bm->mu);
  if (block < 0 || block >= bm->num_blocks) return bm_fail(PKV_ERR_INVALID_ARGUMENT, "block %lld out of range", block);
  *count = bm->refs[block];
  return bm_ok();
}

}  // extern "C"
