// block_manager.cpp -- host-side block pool of a paged KV cache: free list,
// reference counts, fork (prefix sharing), the decode step's slot mapping
// and copy-on-write pairs, and pre-emption (eviction for recompute or to a
// host swap space, and resume).  The rules are stated in
// include/pkv_block_manager.h ("Running Out of Cache": fixed blocks, a new
// block only when the last is full, copy only on write, pre-empt a request
// when even paging runs out).
#include <cstdint>
#include <new>
#include <vector>

#include "pkv_block_manager.h"

namespace pkv {
void set_last_error_message(const char* msg);
}

struct pkv_block_manager {
  struct Seq {
    // device blocks (running), host slots (swapped) or nothing (recompute)
    std::vector<int32_t> blocks;
    int64_t len = 0;
    int32_t state = PKV_BM_RETIRED;
  };
  int32_t num_blocks = 0;
  int32_t block_size = 0;
  std::vector<int32_t> free_stack;  // top = next block handed out
  std::vector<int32_t> refs;        // per block
  std::vector<Seq> seqs;
  // swap space
  int32_t num_host = 0;
  std::vector<int32_t> host_free;   // top = next slot handed out
  std::vector<int32_t> host_refs;   // per slot
  pkv_bm_counters counters{};
  // scratch, all zero (mark) or -1 (hmap, dmap) between calls
  mutable std::vector<int32_t> mark;  // per block: references dropped so far in a count
  std::vector<int32_t> hmap;          // per block: host slot given in this call
  std::vector<int32_t> dmap;          // per slot: device block given in this call

  int32_t take() {
    const int32_t b = free_stack.back();
    free_stack.pop_back();
    refs[b] = 1;
    return b;
  }
  void drop(int32_t b) {
    if (--refs[b] == 0) free_stack.push_back(b);
  }
  int32_t take_host() {
    const int32_t h = host_free.back();
    host_free.pop_back();
    host_refs[h] = 1;
    return h;
  }
  void drop_host(int32_t h) {
    if (--host_refs[h] == 0) host_free.push_back(h);
  }
  bool live(int32_t s) const {
    return s >= 0 && s < static_cast<int32_t>(seqs.size()) && seqs[s].state != PKV_BM_RETIRED;
  }
  bool valid(int32_t s) const { return live(s) && seqs[s].state == PKV_BM_RUNNING; }
  void release_device(Seq& q) {
    // in reverse, so the sequence's first block is handed out first
    for (auto it = q.blocks.rbegin(); it != q.blocks.rend(); ++it) drop(*it);
    q.blocks.clear();
  }

  // Free blocks an append of ids[0..n) needs when dropped[b] references to
  // block b are about to go (null: none).  A sequence needs one when its last
  // block is full, or to copy its last block away while another sequence
  // still holds it; of the holders of a shared block, every one but the last
  // in order copies (mark counts the copies so far).
  int64_t count_step(const int32_t* ids, int32_t n, const std::vector<int32_t>* dropped) const {
    std::vector<int32_t> touched;
    int64_t need = 0;
    for (int32_t i = 0; i < n; ++i) {
      const Seq& q = seqs[ids[i]];
      if (q.len % block_size == 0) {
        ++need;
        continue;
      }
      const int32_t last = q.blocks.back();
      const int32_t held = refs[last] - mark[last] - (dropped ? (*dropped)[last] : 0);
      if (held > 1) {
        ++need;
        if (mark[last]++ == 0) touched.push_back(last);
      }
    }
    for (int32_t b : touched) mark[b] = 0;
    return need;
  }
};

namespace {

pkv_status bm_fail(pkv_status s, const char* msg) {
  pkv::set_last_error_message(msg);
  return s;
}

// Ids in [0, n) all pass `ok` and appear once.
template <class Ok>
bool distinct_and(const pkv_block_manager* bm, const int32_t* ids, int32_t n, Ok ok) {
  for (int32_t i = 0; i < n; ++i)
    if (!ok(ids[i])) return false;
  std::vector<char> seen(bm->seqs.size(), 0);
  for (int32_t i = 0; i < n; ++i) {
    if (seen[ids[i]]) return false;
    seen[ids[i]] = 1;
  }
  return true;
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
  bm->hmap.assign(num_blocks, -1);
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
  s.state = PKV_BM_RUNNING;
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
  // Count the blocks the step needs before changing anything.
  const int32_t bs = bm->block_size;
  const int64_t need = bm->count_step(seq_ids, n, nullptr);
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
  bm->counters.cow_copies += ncow;
  return PKV_OK;
}

pkv_status pkv_bm_free_sequence(pkv_block_manager* bm, int32_t seq) {
  if (bm == nullptr || !bm->live(seq)) return bm_fail(PKV_ERR_INVALID_ARG, "bad sequence id");
  auto& q = bm->seqs[seq];
  if (q.state == PKV_BM_RUNNING) {
    bm->release_device(q);
  } else if (q.state == PKV_BM_SWAPPED) {
    for (auto it = q.blocks.rbegin(); it != q.blocks.rend(); ++it) bm->drop_host(*it);
    q.blocks.clear();
  }
  q.blocks.shrink_to_fit();
  q.len = 0;
  q.state = PKV_BM_RETIRED;
  return PKV_OK;
}

int32_t pkv_bm_block_table(const pkv_block_manager* bm, int32_t seq, int32_t* out,
                           int32_t max_blocks) {
  if (bm == nullptr || !bm->live(seq)) return -1;
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
  return bm != nullptr && bm->live(seq) ? bm->seqs[seq].len : -1;
}

int32_t pkv_bm_num_free_blocks(const pkv_block_manager* bm) {
  return bm != nullptr ? static_cast<int32_t>(bm->free_stack.size()) : -1;
}

int32_t pkv_bm_ref_count(const pkv_block_manager* bm, int32_t block) {
  if (bm == nullptr || block < 0 || block >= bm->num_blocks) return -1;
  return bm->refs[block];
}

pkv_status pkv_bm_set_swap_space(pkv_block_manager* bm, int32_t num_host_blocks) {
  if (bm == nullptr || num_host_blocks < 0)
    return bm_fail(PKV_ERR_INVALID_ARG, "null manager or negative swap space");
  if (static_cast<int32_t>(bm->host_free.size()) != bm->num_host)
    return bm_fail(PKV_ERR_INVALID_ARG, "the swap space holds swapped sequences");
  bm->num_host = num_host_blocks;
  bm->host_refs.assign(num_host_blocks, 0);
  bm->dmap.assign(num_host_blocks, -1);
  bm->host_free.resize(num_host_blocks);
  for (int32_t i = 0; i < num_host_blocks; ++i) bm->host_free[num_host_blocks - 1 - i] = i;
  return PKV_OK;
}

int64_t pkv_bm_step_blocks(const pkv_block_manager* bm, const int32_t* seq_ids, int32_t n) {
  if (bm == nullptr || n < 0 || (n > 0 && !seq_ids) ||
      !distinct_and(bm, seq_ids, n, [bm](int32_t s) { return bm->valid(s); })) {
    bm_fail(PKV_ERR_INVALID_ARG, "null argument, bad, repeated or evicted sequence id");
    return -1;
  }
  return bm->count_step(seq_ids, n, nullptr);
}

pkv_status pkv_bm_plan_preemption(const pkv_block_manager* bm, const int32_t* seq_ids, int32_t n,
                                  int32_t* num_victims_out) {
  if (bm == nullptr || n < 0 || (n > 0 && !seq_ids) || !num_victims_out)
    return bm_fail(PKV_ERR_INVALID_ARG, "null argument or negative count");
  if (!distinct_and(bm, seq_ids, n, [bm](int32_t s) { return bm->valid(s); }))
    return bm_fail(PKV_ERR_INVALID_ARG, "bad, repeated or evicted sequence id");
  // Evict from the back one sequence at a time: a block returns to the free
  // list once every reference to it belongs to an evicted sequence.
  std::vector<int32_t> dropped(bm->num_blocks, 0);
  int64_t free_blocks = static_cast<int64_t>(bm->free_stack.size());
  int32_t k = 0;
  for (; k < n; ++k) {
    if (bm->count_step(seq_ids, n - k, &dropped) <= free_blocks) break;
    for (int32_t b : bm->seqs[seq_ids[n - 1 - k]].blocks)
      if (++dropped[b] == bm->refs[b]) ++free_blocks;
  }
  *num_victims_out = k;
  return PKV_OK;
}

pkv_status pkv_bm_preempt(pkv_block_manager* bm, const int32_t* seq_ids, int32_t n, int32_t mode,
                          int64_t* swap_pairs_out, int32_t* num_swap_out) {
  if (bm == nullptr || n < 0 || (n > 0 && !seq_ids) || !num_swap_out ||
      (mode != PKV_PREEMPT_RECOMPUTE && mode != PKV_PREEMPT_SWAP) ||
      (mode == PKV_PREEMPT_SWAP && n > 0 && !swap_pairs_out))
    return bm_fail(PKV_ERR_INVALID_ARG, "null argument, negative count or bad mode");
  *num_swap_out = 0;
  if (!distinct_and(bm, seq_ids, n, [bm](int32_t s) { return bm->valid(s); }))
    return bm_fail(PKV_ERR_INVALID_ARG, "bad, repeated or evicted sequence id");
  if (mode == PKV_PREEMPT_RECOMPUTE) {
    for (int32_t i = 0; i < n; ++i) {
      auto& q = bm->seqs[seq_ids[i]];
      bm->release_device(q);
      q.state = PKV_BM_RECOMPUTE;
    }
    bm->counters.preempted_recompute += n;
    return PKV_OK;
  }
  // Swap: one host slot per distinct device block, counted first.
  std::vector<int32_t> distinct;
  for (int32_t i = 0; i < n; ++i)
    for (int32_t b : bm->seqs[seq_ids[i]].blocks)
      if (bm->hmap[b] == -1) {
        bm->hmap[b] = -2;
        distinct.push_back(b);
      }
  for (int32_t b : distinct) bm->hmap[b] = -1;
  if (distinct.size() > bm->host_free.size())
    return bm_fail(PKV_ERR_OUT_OF_BLOCKS, "not enough free host blocks in the swap space");
  int32_t np = 0;
  for (int32_t i = 0; i < n; ++i) {
    auto& q = bm->seqs[seq_ids[i]];
    std::vector<int32_t> slots(q.blocks.size());
    for (size_t j = 0; j < q.blocks.size(); ++j) {
      const int32_t b = q.blocks[j];
      if (bm->hmap[b] < 0) {
        bm->hmap[b] = bm->take_host();
        swap_pairs_out[2 * np] = b;
        swap_pairs_out[2 * np + 1] = bm->hmap[b];
        ++np;
      } else {
        ++bm->host_refs[bm->hmap[b]];
      }
      slots[j] = bm->hmap[b];
    }
    bm->release_device(q);
    q.blocks = std::move(slots);
    q.state = PKV_BM_SWAPPED;
  }
  for (int32_t b : distinct) bm->hmap[b] = -1;
  *num_swap_out = np;
  bm->counters.preempted_swap += n;
  bm->counters.blocks_swapped_out += np;
  return PKV_OK;
}

pkv_status pkv_bm_resume(pkv_block_manager* bm, const int32_t* seq_ids, int32_t n,
                         int64_t* swap_pairs_out, int32_t* num_swap_out) {
  if (bm == nullptr || n < 0 || (n > 0 && !seq_ids) || !num_swap_out)
    return bm_fail(PKV_ERR_INVALID_ARG, "null argument or negative count");
  *num_swap_out = 0;
  auto evicted = [bm](int32_t s) {
    return bm->live(s) && bm->seqs[s].state != PKV_BM_RUNNING;
  };
  if (!distinct_and(bm, seq_ids, n, evicted))
    return bm_fail(PKV_ERR_INVALID_ARG, "bad, repeated or running sequence id");
  // Blocks needed: a table's worth per recomputed sequence, one per distinct
  // host slot of the swapped ones.
  const int32_t bs = bm->block_size;
  int64_t need = 0;
  std::vector<int32_t> distinct;
  for (int32_t i = 0; i < n; ++i) {
    const auto& q = bm->seqs[seq_ids[i]];
    if (q.state == PKV_BM_RECOMPUTE) {
      need += (q.len + bs - 1) / bs;
    } else {
      if (!swap_pairs_out && !q.blocks.empty()) {
        for (int32_t h : distinct) bm->dmap[h] = -1;
        return bm_fail(PKV_ERR_INVALID_ARG, "swap_pairs_out is null");
      }
      for (int32_t h : q.blocks)
        if (bm->dmap[h] == -1) {
          bm->dmap[h] = -2;
          distinct.push_back(h);
        }
    }
  }
  for (int32_t h : distinct) bm->dmap[h] = -1;
  need += static_cast<int64_t>(distinct.size());
  if (need > static_cast<int64_t>(bm->free_stack.size()))
    return bm_fail(PKV_ERR_OUT_OF_BLOCKS, "not enough free blocks to resume");
  int32_t np = 0;
  for (int32_t i = 0; i < n; ++i) {
    auto& q = bm->seqs[seq_ids[i]];
    if (q.state == PKV_BM_RECOMPUTE) {
      const int64_t nb = (q.len + bs - 1) / bs;
      q.blocks.reserve(static_cast<size_t>(nb));
      for (int64_t j = 0; j < nb; ++j) q.blocks.push_back(bm->take());
      bm->counters.tokens_recomputed += q.len;
    } else {
      for (auto& e : q.blocks) {
        const int32_t h = e;
        if (bm->dmap[h] < 0) {
          bm->dmap[h] = bm->take();
          swap_pairs_out[2 * np] = h;
          swap_pairs_out[2 * np + 1] = bm->dmap[h];
          ++np;
        } else {
          ++bm->refs[bm->dmap[h]];
        }
        e = bm->dmap[h];
        bm->drop_host(h);
      }
    }
    q.state = PKV_BM_RUNNING;
  }
  for (int32_t h : distinct) bm->dmap[h] = -1;
  *num_swap_out = np;
  bm->counters.resumed += n;
  bm->counters.blocks_swapped_in += np;
  return PKV_OK;
}

int32_t pkv_bm_state(const pkv_block_manager* bm, int32_t seq) {
  return bm != nullptr && bm->live(seq) ? bm->seqs[seq].state : PKV_BM_RETIRED;
}

int32_t pkv_bm_num_free_host_blocks(const pkv_block_manager* bm) {
  return bm != nullptr ? static_cast<int32_t>(bm->host_free.size()) : -1;
}

int32_t pkv_bm_host_ref_count(const pkv_block_manager* bm, int32_t slot) {
  if (bm == nullptr || slot < 0 || slot >= bm->num_host) return -1;
  return bm->host_refs[slot];
}

pkv_status pkv_bm_get_counters(const pkv_block_manager* bm, pkv_bm_counters* out) {
  if (bm == nullptr || out == nullptr) return bm_fail(PKV_ERR_INVALID_ARG, "null argument");
  *out = bm->counters;
  return PKV_OK;
}

}  // extern "C"
