// block_manager.cpp -- host-side KV block manager (C++): the bookkeeping that decides
// which physical block every token lives in.
//
// Pages: "anthology-of-the-sota note-023", Method (allocate blocks on demand as a
// sequence grows, free them when it finishes, share physical blocks between
// sequences with identical prefixes, copy on write when one diverges) and Concepts
// (internal fragmentation = the unused tail of the last block); "Paged Attention"
// glossary, paragraphs 1-3 (waste only in the last block; a shared block is copied
// only when a sequence writes to it); "PagedAttention & Continuous Batching", the
// shared-system-prompt paragraph (blocks of a finished request are reclaimed and
// handed to a new request on the very next step).
//
// Policy (the pages fix none): free blocks form a LIFO stack, initially handing out
// 0, 1, 2, ...; a freed block is reused first.  An append that lands in a block
// whose reference count is above one copies that block first (copy-on-write); an
// append at a block boundary takes a fresh block.  Every call either succeeds as a
// whole or leaves the manager unchanged.
#include <algorithm>
#include <cstdio>
#include <string>
#include <unordered_map>
#include <vector>

#include "launch.h"
#include "pagedkv.h"

struct pkv_block_manager {
  int32_t num_blocks = 0;
  int32_t block_size = 0;
  std::vector<int32_t> free_stack;  // top = back
  std::vector<int32_t> refcount;    // per physical block
  std::vector<int32_t> filled;      // valid rows written into each block
  struct Seq {
    std::vector<int32_t> blocks;
    int64_t len = 0;
  };
  std::unordered_map<int64_t, Seq> seqs;
  std::unordered_map<int64_t, int64_t> swapped;  // swapped-out sequence -> length
  int64_t copies = 0;  // copy-on-write copies made so far
};

namespace {

pkv_status err(pkv_status st, const std::string& msg) { return pkv::record_error(st, msg.c_str()); }

int64_t blocks_for(int64_t tokens, int32_t bs) { return (tokens + bs - 1) / bs; }

int32_t take_block(pkv_block_manager* m) {
  const int32_t b = m->free_stack.back();
  m->free_stack.pop_back();
  m->refcount[b] = 1;
  m->filled[b] = 0;
  return b;
}

void release_block(pkv_block_manager* m, int32_t b) {
  if (--m->refcount[b] == 0) {
    m->filled[b] = 0;
    m->free_stack.push_back(b);
  }
}

}  // namespace

extern "C" {

pkv_status pkv_bm_create(int32_t num_blocks, int32_t block_size, pkv_block_manager** out) {
  if (!out) return err(PKV_ERR_INVALID_ARG, "out is NULL");
  if (num_blocks <= 0 || block_size <= 0) return err(PKV_ERR_INVALID_ARG, "num_blocks and block_size must be positive");
  auto* m = new pkv_block_manager;
  m->num_blocks = num_blocks;
  m->block_size = block_size;
  m->free_stack.resize(num_blocks);
  for (int32_t i = 0; i < num_blocks; ++i) m->free_stack[i] = num_blocks - 1 - i;  // pops 0, 1, 2, ...
  m->refcount.assign(num_blocks, 0);
  m->filled.assign(num_blocks, 0);
  *out = m;
  return PKV_OK;
}

void pkv_bm_destroy(pkv_block_manager* m) { delete m; }

pkv_status pkv_bm_add_sequence(pkv_block_manager* m, int64_t seq_id, int64_t num_tokens) {
  if (!m) return err(PKV_ERR_INVALID_ARG, "manager is NULL");
  if (num_tokens < 0) return err(PKV_ERR_INVALID_ARG, "num_tokens < 0");
  if (m->seqs.count(seq_id) || m->swapped.count(seq_id))
    return err(PKV_ERR_INVALID_ARG, "sequence id already present");
  const int64_t need = blocks_for(num_tokens, m->block_size);
  if (need > static_cast<int64_t>(m->free_stack.size()))
    return err(PKV_ERR_OUT_OF_BLOCKS, "not enough free blocks for the prompt");
  auto& s = m->seqs[seq_id];
  for (int64_t i = 0; i < need; ++i) {
    const int32_t b = take_block(m);
    const int64_t rows = std::min<int64_t>(m->block_size, num_tokens - i * m->block_size);
    m->filled[b] = static_cast<int32_t>(rows);
    s.blocks.push_back(b);
  }
  s.len = num_tokens;
  return PKV_OK;
}

pkv_status pkv_bm_fork(pkv_block_manager* m, int64_t parent, int64_t child) {
  if (!m) return err(PKV_ERR_INVALID_ARG, "manager is NULL");
  auto it = m->seqs.find(parent);
  if (it == m->seqs.end()) return err(PKV_ERR_INVALID_ARG, "unknown parent sequence");
  if (m->seqs.count(child) || m->swapped.count(child)) return err(PKV_ERR_INVALID_ARG, "child id already present");
  const auto copy = it->second;  // the child shares every physical block by reference
  for (int32_t b : copy.blocks) ++m->refcount[b];
  m->seqs[child] = copy;
  return PKV_OK;
}

pkv_status pkv_bm_append(pkv_block_manager* m, const int64_t* seq_ids, int32_t n, int64_t* slots,
                         int64_t* cow_pairs, int32_t* num_cow) {
  if (!m || (n > 0 && (!seq_ids || !slots || !cow_pairs || !num_cow)))
    return err(PKV_ERR_INVALID_ARG, "NULL argument");
  if (n < 0) return err(PKV_ERR_INVALID_ARG, "n < 0");
  // first pass: validate and count the fresh blocks needed, so failure changes nothing
  int64_t need = 0;
  {
    std::unordered_map<int64_t, int> seen;
    std::unordered_map<int32_t, int32_t> refs;  // simulated reference counts
    for (int32_t i = 0; i < n; ++i) {
      auto it = m->seqs.find(seq_ids[i]);
      if (it == m->seqs.end()) return err(PKV_ERR_INVALID_ARG, "unknown sequence id");
      if (seen[seq_ids[i]]++) return err(PKV_ERR_INVALID_ARG, "a sequence appears twice in one append");
      const auto& s = it->second;
      if (s.len % m->block_size == 0) {
        ++need;
      } else {
        const int32_t b = s.blocks.back();
        auto r = refs.find(b);
        int32_t& rc = r == refs.end() ? (refs[b] = m->refcount[b]) : r->second;
        if (rc > 1) {
          ++need;
          --rc;
        }
      }
    }
  }
  if (need > static_cast<int64_t>(m->free_stack.size()))
    return err(PKV_ERR_OUT_OF_BLOCKS, "not enough free blocks for this append");
  int32_t ncow = 0;
  for (int32_t i = 0; i < n; ++i) {
    auto& s = m->seqs[seq_ids[i]];
    const int32_t row = static_cast<int32_t>(s.len % m->block_size);
    if (row == 0) {
      s.blocks.push_back(take_block(m));
    } else if (m->refcount[s.blocks.back()] > 1) {
      // copy-on-write: this sequence gets its own copy of the shared last block
      const int32_t old = s.blocks.back();
      const int32_t fresh = take_block(m);
      m->filled[fresh] = m->filled[old];
      cow_pairs[2 * ncow] = old;
      cow_pairs[2 * ncow + 1] = fresh;
      ++ncow;
      --m->refcount[old];
      s.blocks.back() = fresh;
      ++m->copies;
    }
    const int32_t b = s.blocks.back();
    slots[i] = static_cast<int64_t>(b) * m->block_size + row;
    m->filled[b] = std::max(m->filled[b], row + 1);
    ++s.len;
  }
  *num_cow = ncow;
  return PKV_OK;
}

pkv_status pkv_bm_free_sequence(pkv_block_manager* m, int64_t seq_id) {
  if (!m) return err(PKV_ERR_INVALID_ARG, "manager is NULL");
  auto it = m->seqs.find(seq_id);
  if (it == m->seqs.end()) return err(PKV_ERR_INVALID_ARG, "unknown sequence id");
  // release in reverse so the first block of the sequence ends on top of the stack
  for (auto b = it->second.blocks.rbegin(); b != it->second.blocks.rend(); ++b) release_block(m, *b);
  m->seqs.erase(it);
  return PKV_OK;
}

pkv_status pkv_bm_swap_out(pkv_block_manager* m, int64_t seq_id, int32_t* blocks_out, int32_t capacity,
                           int32_t* num_out) {
  if (!m || !num_out) return err(PKV_ERR_INVALID_ARG, "NULL argument");
  auto it = m->seqs.find(seq_id);
  if (it == m->seqs.end()) return err(PKV_ERR_INVALID_ARG, "unknown (or already swapped) sequence id");
  const auto& blocks = it->second.blocks;
  if (static_cast<int64_t>(blocks.size()) > capacity || (!blocks.empty() && !blocks_out))
    return err(PKV_ERR_INVALID_ARG, "blocks_out too small");
  for (size_t i = 0; i < blocks.size(); ++i) blocks_out[i] = blocks[i];
  *num_out = static_cast<int32_t>(blocks.size());
  const int64_t len = it->second.len;
  for (auto b = blocks.rbegin(); b != blocks.rend(); ++b) release_block(m, *b);
  m->seqs.erase(it);
  m->swapped[seq_id] = len;
  return PKV_OK;
}

pkv_status pkv_bm_swap_in(pkv_block_manager* m, int64_t seq_id, int32_t* blocks_out, int32_t capacity,
                          int32_t* num_out) {
  if (!m || !num_out) return err(PKV_ERR_INVALID_ARG, "NULL argument");
  auto it = m->swapped.find(seq_id);
  if (it == m->swapped.end()) return err(PKV_ERR_INVALID_ARG, "sequence is not swapped out");
  const int64_t len = it->second;
  const int64_t need = blocks_for(len, m->block_size);
  if (need > capacity || (need > 0 && !blocks_out)) return err(PKV_ERR_INVALID_ARG, "blocks_out too small");
  if (need > static_cast<int64_t>(m->free_stack.size()))
    return err(PKV_ERR_OUT_OF_BLOCKS, "not enough free blocks to swap the sequence in");
  auto& s = m->seqs[seq_id];
  for (int64_t i = 0; i < need; ++i) {
    const int32_t b = take_block(m);
    m->filled[b] = static_cast<int32_t>(std::min<int64_t>(m->block_size, len - i * m->block_size));
    s.blocks.push_back(b);
    blocks_out[i] = b;
  }
  s.len = len;
  *num_out = static_cast<int32_t>(need);
  m->swapped.erase(it);
  return PKV_OK;
}

pkv_status pkv_bm_block_tables(const pkv_block_manager* m, const int64_t* seq_ids, int32_t n,
                               int32_t max_blocks, int32_t* tables, int32_t* lens) {
  if (!m || (n > 0 && (!seq_ids || !tables || !lens))) return err(PKV_ERR_INVALID_ARG, "NULL argument");
  for (int32_t i = 0; i < n; ++i) {
    auto it = m->seqs.find(seq_ids[i]);
    if (it == m->seqs.end()) return err(PKV_ERR_INVALID_ARG, "unknown sequence id");
    if (static_cast<int64_t>(it->second.blocks.size()) > max_blocks)
      return err(PKV_ERR_INVALID_ARG, "max_blocks too small for a sequence");
    if (it->second.len > INT32_MAX) return err(PKV_ERR_UNSUPPORTED, "sequence longer than int32");
  }
  for (int32_t i = 0; i < n; ++i) {
    const auto& s = m->seqs.at(seq_ids[i]);
    int32_t* row = tables + static_cast<size_t>(i) * max_blocks;
    for (int32_t j = 0; j < max_blocks; ++j)
      row[j] = j < static_cast<int32_t>(s.blocks.size()) ? s.blocks[j] : -1;
    lens[i] = static_cast<int32_t>(s.len);
  }
  return PKV_OK;
}

pkv_status pkv_bm_stats(const pkv_block_manager* m, pkv_block_stats* out) {
  if (!m || !out) return err(PKV_ERR_INVALID_ARG, "NULL argument");
  pkv_block_stats st{};
  st.num_blocks = m->num_blocks;
  st.free_blocks = static_cast<int32_t>(m->free_stack.size());
  st.used_blocks = m->num_blocks - st.free_blocks;
  st.num_sequences = static_cast<int32_t>(m->seqs.size());
  for (int32_t b = 0; b < m->num_blocks; ++b) {
    if (m->refcount[b] > 0) st.stored_tokens += m->filled[b];
    if (m->refcount[b] > 1) ++st.shared_blocks;
  }
  for (const auto& kv : m->seqs) {
    st.logical_tokens += kv.second.len;
    st.max_len = std::max(st.max_len, kv.second.len);
  }
  st.allocated_slots = static_cast<int64_t>(st.used_blocks) * m->block_size;
  st.copies = m->copies;
  st.swapped = static_cast<int64_t>(m->swapped.size());
  *out = st;
  return PKV_OK;
}

}  // extern "C"
