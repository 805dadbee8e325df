// block_manager.cpp -- host-side block pool of a paged KV cache: free list,
// reference counts, fork (prefix sharing), the decode step's slot mapping
// and copy-on-write pairs.  The rules are stated in
// include/pkv_block_manager.h ("Running Out of Cache": fixed blocks, a new
// block only when the last is full, copy only on write).
#include <cstdint>
#include <new>
#include <vector>

#include "pkv_block_manager.h"

namespace pkv {
void set_last_error_message(const char* msg);
}

struct pkv_block_manager {
  struct Seq {
    std::vector<int32_t> blocks;
    int64_t len = 0;
    bool alive = false;
  };
  int32_t num_blocks = 0;
  int32_t block_size = 0;
  std::vector<int32_t> free_stack;  // top = next block handed out
  std::vector<int32_t> refs;        // per block
  std::vector<Seq> seqs;
  // scratch of one append call
  std::vector<int32_t> mark;

  int32_t take() {
    const int32_t b = free_stack.back();
    free_stack.pop_back();
    refs[b] = 1;
    return b;
  }
  void drop(int32_t b) {
    if (--refs[b] == 0) free_stack.push_back(b);
  }
  bool valid(int32_t s) const {
    return s >= 0 && s < static_cast<int32_t>(seqs.size()) && seqs[s].alive;
  }
};

namespace {

pkv_status bm_fail(pkv_status s, const char* msg) {
  pkv::set_last_error_message(msg);
  return s;
}

}  // namespace

extern "C" {

pkv_block_manager* pkv_bm_create(int32_t num_blocks, int32_t block_size,
                                 const int32_t* free_order) {
  if (num_blocks < 0 || block_size <= 0) {
    bm_fail(PKV_ERR_INVALID_ARG, "num_blocks < 0 or block_size < 1");
    return nullptr;
  }
  pkv_block_manager* bm = new (std::nothrow) pkv_block_manager();
  if (bm == nullptr) {
    bm_fail(PKV_ERR_INVALID_ARG, "out of host memory");
    return nullptr;
  }
  bm->num_blocks = num_blocks;
  bm->block_size = block_size;
  bm->refs.assign(num_blocks, 0);
  bm->mark.assign(num_blocks, 0);
  bm->free_stack.resize(num_blocks);
  std::vector<char> seen(num_blocks, 0);
  for (int32_t i = 0; i < num_blocks; ++i) {
    const int32_t b = free_order != nullptr ? free_order[i] : i;
    if (b < 0 || b >= num_blocks || seen[b]) {
      delete bm;
      bm_fail(PKV_ERR_INVALID_ARG, "free_order is not a permutation of the block ids");
      return nullptr;
    }
    seen[b] = 1;
    bm->free_stack[num_blocks - 1 - i] = b;  // free_order[0] on top
  }
  return bm;
}

void pkv_bm_destroy(pkv_block_manager* bm) { delete bm; }

int32_t pkv_bm_add_sequence(pkv_block_manager* bm, int64_t num_tokens) {
  if (bm == nullptr || num_tokens < 0) {
    bm_fail(PKV_ERR_INVALID_ARG, "null manager or negative length");
    return -1;
  }
  const int64_t need = (num_tokens + bm->block_size - 1) / bm->block_size;
  if (need > static_cast<int64_t>(bm->free_stack.size())) {
    bm_fail(PKV_ERR_OUT_OF_BLOCKS, "not enough free blocks for the sequence");
    return -1;
  }
  pkv_block_manager::Seq s;
  s.alive = true;
  s.len = num_tokens;
  s.blocks.reserve(static_cast<size_t>(need));
  for (int64_t i = 0; i < need; ++i) s.blocks.push_back(bm->take());
  bm->seqs.push_back(std::move(s));
  return static_cast<int32_t>(bm->seqs.size() - 1);
}

int32_t pkv_bm_fork(pkv_block_manager* bm, int32_t parent) {
  if (bm == nullptr || !bm->valid(parent)) {
    bm_fail(PKV_ERR_INVALID_ARG, "bad parent sequence");
    return -1;
  }
  pkv_block_manager::Seq s = bm->seqs[parent];
  for (int32_t b : s.blocks) ++bm->refs[b];
  bm->seqs.push_back(std::move(s));
  return static_cast<int32_t>(bm->seqs.size() - 1);
}

pkv_status pkv_bm_append(pkv_block_manager* bm, const int32_t* seq_ids, int32_t n,
                         int64_t* slot_mapping_out, int64_t* cow_pairs_out,
                         int32_t* num_cow_out) {
  if (bm == nullptr || n < 0 || (n > 0 && (!seq_ids || !slot_mapping_out || !cow_pairs_out)) ||
      !num_cow_out)
    return bm_fail(PKV_ERR_INVALID_ARG, "null argument or negative count");
  *num_cow_out = 0;
  for (int32_t i = 0; i < n; ++i)
    if (!bm->valid(seq_ids[i])) return bm_fail(PKV_ERR_INVALID_ARG, "bad or retired sequence id");
  {
    std::vector<char> seen(bm->seqs.size(), 0);
    for (int32_t i = 0; i < n; ++i) {
      if (seen[seq_ids[i]]) return bm_fail(PKV_ERR_INVALID_ARG, "a sequence appears twice");
      seen[seq_ids[i]] = 1;
    }
  }
  // Count the blocks the step needs before changing anything.  A sequence
  // needs one when its last block is full, or to copy its last block away
  // while another sequence still holds it; of the holders of a shared block,
  // every one but the last in order copies (mark counts the copies so far).
  const int32_t bs = bm->block_size;
  std::vector<int32_t> remaining;  // blocks whose mark this call set
  int64_t need = 0;
  for (int32_t i = 0; i < n; ++i) {
    const auto& q = bm->seqs[seq_ids[i]];
    if (q.len % bs == 0) {
      ++need;
      continue;
    }
    const int32_t last = q.blocks.back();
    // references to `last` dropped earlier in this step
    const int32_t held = bm->refs[last] - bm->mark[last];
    if (held > 1) {
      ++need;
      if (bm->mark[last]++ == 0) remaining.push_back(last);
    }
  }
  for (int32_t b : remaining) bm->mark[b] = 0;
  if (need > static_cast<int64_t>(bm->free_stack.size()))
    return bm_fail(PKV_ERR_OUT_OF_BLOCKS, "not enough free blocks for this step");
  // Apply.
  int32_t ncow = 0;
  for (int32_t i = 0; i < n; ++i) {
    auto& q = bm->seqs[seq_ids[i]];
    const int64_t off = q.len % bs;
    int32_t blk;
    if (off == 0) {
      blk = bm->take();
      q.blocks.push_back(blk);
    } else {
      blk = q.blocks.back();
      if (bm->refs[blk] > 1) {
        const int32_t fresh = bm->take();
        cow_pairs_out[2 * ncow] = blk;
        cow_pairs_out[2 * ncow + 1] = fresh;
        ++ncow;
        --bm->refs[blk];
        q.blocks.back() = fresh;
        blk = fresh;
      }
    }
    slot_mapping_out[i] = static_cast<int64_t>(blk) * bs + off;
    ++q.len;
  }
  *num_cow_out = ncow;
  return PKV_OK;
}

pkv_status pkv_bm_free_sequence(pkv_block_manager* bm, int32_t seq) {
  if (bm == nullptr || !bm->valid(seq)) return bm_fail(PKV_ERR_INVALID_ARG, "bad sequence id");
  auto& q = bm->seqs[seq];
  // release in reverse, so the sequence's first block is handed out first
  for (auto it = q.blocks.rbegin(); it != q.blocks.rend(); ++it) bm->drop(*it);
  q.blocks.clear();
  q.blocks.shrink_to_fit();
  q.len = 0;
  q.alive = false;
  return PKV_OK;
}

int32_t pkv_bm_block_table(const pkv_block_manager* bm, int32_t seq, int32_t* out,
                           int32_t max_blocks) {
  if (bm == nullptr || !bm->valid(seq)) return -1;
  const auto& q = bm->seqs[seq];
  const int32_t nb = static_cast<int32_t>(q.blocks.size());
  if (nb > max_blocks || (nb > 0 && out == nullptr)) return -1;
  for (int32_t i = 0; i < nb; ++i) out[i] = q.blocks[i];
  return nb;
}

pkv_status pkv_bm_export(const pkv_block_manager* bm, const int32_t* seq_ids, int32_t n,
                         int32_t* tables_out, int32_t max_blocks, int32_t filler,
                         int32_t* context_lens_out) {
  if (bm == nullptr || n < 0 || max_blocks < 0 ||
      (n > 0 && (!seq_ids || !tables_out || !context_lens_out)))
    return bm_fail(PKV_ERR_INVALID_ARG, "null argument or negative count");
  for (int32_t i = 0; i < n; ++i) {
    if (!bm->valid(seq_ids[i])) return bm_fail(PKV_ERR_INVALID_ARG, "bad sequence id");
    const auto& q = bm->seqs[seq_ids[i]];
    if (static_cast<int32_t>(q.blocks.size()) > max_blocks)
      return bm_fail(PKV_ERR_INVALID_ARG, "max_blocks smaller than a block table");
    if (q.len > INT32_MAX) return bm_fail(PKV_ERR_UNSUPPORTED, "context longer than int32");
  }
  for (int32_t i = 0; i < n; ++i) {
    const auto& q = bm->seqs[seq_ids[i]];
    int32_t* row = tables_out + static_cast<int64_t>(i) * max_blocks;
    const int32_t nb = static_cast<int32_t>(q.blocks.size());
    for (int32_t j = 0; j < max_blocks; ++j) row[j] = j < nb ? q.blocks[j] : filler;
    context_lens_out[i] = static_cast<int32_t>(q.len);
  }
  return PKV_OK;
}

int64_t pkv_bm_length(const pkv_block_manager* bm, int32_t seq) {
  return bm != nullptr && bm->valid(seq) ? bm->seqs[seq].len : -1;
}

int32_t pkv_bm_num_free_blocks(const pkv_block_manager* bm) {
  return bm != nullptr ? static_cast<int32_t>(bm->free_stack.size()) : -1;
}

int32_t pkv_bm_ref_count(const pkv_block_manager* bm, int32_t block) {
  if (bm == nullptr || block < 0 || block >= bm->num_blocks) return -1;
  return bm->refs[block];
}

}  // extern "C"
