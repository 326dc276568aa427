// Host block allocator (see the allocator section of include/pkv.h).
//
// The block manager of mini-runtime "ch.12 Paged KV Cache" §2.2-2.4 and of
// "vLLM PagedAttention source notes" §2.1: a FIFO deque of free block ids
// (allocate from the front, release to the back at ref_count zero),
// per-block reference counts for sharing, per-sequence block tables with a
// first-block offset, and copy-on-write when an append would write into a
// shared block (ch.12 §3.1).  Every operation checks all its conditions
// before changing anything, so a failing call leaves the state unchanged.
#include <climits>
#include <cstdint>
#include <deque>
#include <new>
#include <unordered_map>
#include <vector>

#include "pkv.h"

struct pkv_allocator {
  struct Seq {
    std::vector<int32_t> blocks;
    int32_t offset = 0;
    int64_t num_tokens = 0;
  };
  int64_t num_blocks = 0;
  int32_t block_size = 0;
  std::vector<int32_t> ref;
  std::deque<int32_t> free_q;
  std::unordered_map<int64_t, Seq> seqs;

  // blocks spanned by num_tokens tokens starting at row `offset`
  int64_t span(int32_t offset, int64_t num_tokens) const {
    return num_tokens > 0 ? (offset + num_tokens + block_size - 1) / block_size : 0;
  }
  int32_t take() {
    const int32_t b = free_q.front();
    free_q.pop_front();
    ref[b] = 1;
    return b;
  }
  void release(int32_t b) {
    if (--ref[b] == 0) free_q.push_back(b);
  }
  bool valid_block(int64_t b) const { return b >= 0 && b < num_blocks; }
};

extern "C" {

pkv_status pkv_alloc_create(int64_t num_blocks, int32_t block_size, const int32_t* free_order,
                            pkv_allocator** out) {
  if (!out || num_blocks <= 0 || num_blocks > INT32_MAX || block_size <= 0 ||
      (block_size & (block_size - 1)) != 0 || block_size > 1024)
    return PKV_ERR_INVALID_ARG;
  pkv_allocator* a = new (std::nothrow) pkv_allocator;
  if (!a) return PKV_ERR_INVALID_ARG;
  a->num_blocks = num_blocks;
  a->block_size = block_size;
  a->ref.assign((size_t)num_blocks, 0);
  if (free_order) {
    std::vector<char> seen((size_t)num_blocks, 0);
    for (int64_t i = 0; i < num_blocks; ++i) {
      const int32_t b = free_order[i];
      if (b < 0 || b >= num_blocks || seen[(size_t)b]) {
        delete a;
        return PKV_ERR_INVALID_ARG;  // not a permutation of the ids
      }
      seen[(size_t)b] = 1;
      a->free_q.push_back(b);
    }
  } else {
    for (int64_t i = 0; i < num_blocks; ++i) a->free_q.push_back((int32_t)i);
  }
  *out = a;
  return PKV_OK;
}

pkv_status pkv_alloc_destroy(pkv_allocator* a) {
  if (!a) return PKV_ERR_INVALID_ARG;
  delete a;
  return PKV_OK;
}

int64_t pkv_alloc_num_free(const pkv_allocator* a) {
  return a ? (int64_t)a->free_q.size() : -1;
}

int32_t pkv_alloc_ref_count(const pkv_allocator* a, int64_t block) {
  if (!a || !a->valid_block(block)) return -1;
  return a->ref[(size_t)block];
}

pkv_status pkv_alloc_blocks(pkv_allocator* a, int64_t n, int32_t* out_ids) {
  if (!a || n < 0 || (n > 0 && !out_ids)) return PKV_ERR_INVALID_ARG;
  if ((size_t)n > a->free_q.size()) return PKV_ERR_NO_BLOCKS;
  for (int64_t i = 0; i < n; ++i) out_ids[i] = a->take();
  return PKV_OK;
}

pkv_status pkv_alloc_inc_ref(pkv_allocator* a, int32_t block) {
  if (!a || !a->valid_block(block) || a->ref[block] <= 0) return PKV_ERR_INVALID_ARG;
  ++a->ref[block];
  return PKV_OK;
}

pkv_status pkv_alloc_dec_ref(pkv_allocator* a, int32_t block) {
  if (!a || !a->valid_block(block) || a->ref[block] <= 0) return PKV_ERR_INVALID_ARG;
  a->release(block);
  return PKV_OK;
}

pkv_status pkv_seq_new(pkv_allocator* a, int64_t seq_id, int32_t offset) {
  if (!a || offset < 0 || offset >= a->block_size) return PKV_ERR_INVALID_ARG;
  if (a->seqs.count(seq_id)) return PKV_ERR_INVALID_ARG;
  pkv_allocator::Seq s;
  s.offset = offset;
  a->seqs.emplace(seq_id, std::move(s));
  return PKV_OK;
}

pkv_status pkv_seq_share(pkv_allocator* a, int64_t seq_id, const int32_t* blocks, int32_t n,
                         int64_t num_tokens) {
  if (!a || n < 0 || num_tokens < 0 || (n > 0 && !blocks)) return PKV_ERR_INVALID_ARG;
  auto it = a->seqs.find(seq_id);
  if (it == a->seqs.end() || !it->second.blocks.empty() || it->second.num_tokens != 0)
    return PKV_ERR_INVALID_ARG;
  auto& s = it->second;
  if (a->span(s.offset, num_tokens) != n) return PKV_ERR_CAPACITY;
  for (int32_t i = 0; i < n; ++i)
    if (!a->valid_block(blocks[i]) || a->ref[blocks[i]] <= 0) return PKV_ERR_INVALID_ARG;
  for (int32_t i = 0; i < n; ++i) {
    ++a->ref[blocks[i]];
    s.blocks.push_back(blocks[i]);
  }
  s.num_tokens = num_tokens;
  return PKV_OK;
}

pkv_status pkv_seq_append(pkv_allocator* a, int64_t seq_id, int64_t num_tokens,
                          int64_t* slots_out, int32_t* cow_src, int32_t* cow_dst,
                          int32_t* n_cow) {
  if (!a || num_tokens < 0) return PKV_ERR_INVALID_ARG;
  auto it = a->seqs.find(seq_id);
  if (it == a->seqs.end()) return PKV_ERR_INVALID_ARG;
  auto& s = it->second;
  const int64_t bs = a->block_size;
  const int64_t start = s.offset + s.num_tokens;  // table position of the first new token
  const int64_t end = start + num_tokens;
  const int64_t have = (int64_t)s.blocks.size();
  const int64_t after = num_tokens > 0 ? (end + bs - 1) / bs : have;
  const int64_t fresh = after > have ? after - have : 0;
  const int64_t first_blk = start / bs;
  const bool cow = num_tokens > 0 && first_blk < have && a->ref[s.blocks[first_blk]] > 1;
  if (fresh + (cow ? 1 : 0) > (int64_t)a->free_q.size()) return PKV_ERR_NO_BLOCKS;
  if (n_cow) *n_cow = 0;
  if (cow) {
    const int32_t old = s.blocks[first_blk];
    const int32_t nb = a->take();
    a->release(old);
    s.blocks[first_blk] = nb;
    if (cow_src) *cow_src = old;
    if (cow_dst) *cow_dst = nb;
    if (n_cow) *n_cow = 1;
  }
  for (int64_t i = 0; i < fresh; ++i) s.blocks.push_back(a->take());
  if (slots_out) {
    for (int64_t p = start; p < end; ++p)
      slots_out[p - start] = (int64_t)s.blocks[p / bs] * bs + p % bs;
  }
  s.num_tokens += num_tokens;
  return PKV_OK;
}

pkv_status pkv_seq_append_batch(pkv_allocator* a, const int64_t* seq_ids, int32_t n,
                                const int64_t* num_tokens, int64_t* slots_out, int32_t* cow_src,
                                int32_t* cow_dst, int32_t* n_cow) {
  if (!a || n < 0 || (n > 0 && !seq_ids)) return PKV_ERR_INVALID_ARG;
  // dry run: blocks the whole batch needs, with the reference counts the
  // earlier appends of the batch leave behind (copy-on-write drops the count
  // of the shared block it leaves)
  std::unordered_map<int64_t, char> seen;
  std::unordered_map<int32_t, int32_t> ref_delta;
  const int64_t bs = a->block_size;
  int64_t need = 0;
  for (int32_t i = 0; i < n; ++i) {
    auto it = a->seqs.find(seq_ids[i]);
    if (it == a->seqs.end() || !seen.emplace(seq_ids[i], 1).second) return PKV_ERR_INVALID_ARG;
    const int64_t k = num_tokens ? num_tokens[i] : 1;
    if (k < 0) return PKV_ERR_INVALID_ARG;
    if (k == 0) continue;
    const auto& s = it->second;
    const int64_t start = s.offset + s.num_tokens, end = start + k;
    const int64_t have = (int64_t)s.blocks.size();
    const int64_t after = (end + bs - 1) / bs;
    need += after > have ? after - have : 0;
    const int64_t first_blk = start / bs;
    if (first_blk < have) {
      const int32_t b = s.blocks[first_blk];
      auto d = ref_delta.find(b);
      const int32_t r = a->ref[b] + (d == ref_delta.end() ? 0 : d->second);
      if (r > 1) {
        need += 1;
        ref_delta[b] = (d == ref_delta.end() ? 0 : d->second) - 1;
      }
    }
  }
  if (need > (int64_t)a->free_q.size()) return PKV_ERR_NO_BLOCKS;
  int64_t w = 0;
  int32_t c = 0;
  for (int32_t i = 0; i < n; ++i) {
    const int64_t k = num_tokens ? num_tokens[i] : 1;
    int32_t one = 0, src = 0, dst = 0;
    pkv_seq_append(a, seq_ids[i], k, slots_out ? slots_out + w : nullptr, &src, &dst, &one);
    w += k;
    if (one) {
      if (cow_src) cow_src[c] = src;
      if (cow_dst) cow_dst[c] = dst;
      ++c;
    }
  }
  if (n_cow) *n_cow = c;
  return PKV_OK;
}

pkv_status pkv_seq_fork(pkv_allocator* a, int64_t src, int64_t dst) {
  if (!a || src == dst) return PKV_ERR_INVALID_ARG;
  auto it = a->seqs.find(src);
  if (it == a->seqs.end() || a->seqs.count(dst)) return PKV_ERR_INVALID_ARG;
  pkv_allocator::Seq copy = it->second;
  for (int32_t b : copy.blocks) ++a->ref[b];
  a->seqs.emplace(dst, std::move(copy));
  return PKV_OK;
}

pkv_status pkv_seq_free(pkv_allocator* a, int64_t seq_id) {
  if (!a) return PKV_ERR_INVALID_ARG;
  auto it = a->seqs.find(seq_id);
  if (it == a->seqs.end()) return PKV_ERR_INVALID_ARG;
  for (int32_t b : it->second.blocks) a->release(b);
  a->seqs.erase(it);
  return PKV_OK;
}

pkv_status pkv_seq_info(const pkv_allocator* a, int64_t seq_id, int64_t* num_tokens,
                        int32_t* offset, int32_t* num_blocks) {
  if (!a) return PKV_ERR_INVALID_ARG;
  auto it = a->seqs.find(seq_id);
  if (it == a->seqs.end()) return PKV_ERR_INVALID_ARG;
  if (num_tokens) *num_tokens = it->second.num_tokens;
  if (offset) *offset = it->second.offset;
  if (num_blocks) *num_blocks = (int32_t)it->second.blocks.size();
  return PKV_OK;
}

pkv_status pkv_seq_tables(const pkv_allocator* a, const int64_t* seq_ids, int32_t batch,
                          int32_t max_blocks, int32_t* tables, int32_t* seq_lens,
                          int32_t* offsets) {
  if (!a || batch < 0 || max_blocks <= 0 || (batch > 0 && (!seq_ids || !tables)))
    return PKV_ERR_INVALID_ARG;
  for (int32_t b = 0; b < batch; ++b) {  // check everything before writing
    auto it = a->seqs.find(seq_ids[b]);
    if (it == a->seqs.end()) return PKV_ERR_INVALID_ARG;
    if ((int64_t)it->second.blocks.size() > max_blocks) return PKV_ERR_CAPACITY;
    if (it->second.num_tokens > INT32_MAX) return PKV_ERR_CAPACITY;
  }
  for (int32_t b = 0; b < batch; ++b) {
    const auto& s = a->seqs.find(seq_ids[b])->second;
    int32_t* row = tables + (int64_t)b * max_blocks;
    const int32_t n = (int32_t)s.blocks.size();
    for (int32_t k = 0; k < max_blocks; ++k) row[k] = k < n ? s.blocks[k] : -1;
    if (seq_lens) seq_lens[b] = (int32_t)s.num_tokens;
    if (offsets) offsets[b] = s.offset;
  }
  return PKV_OK;
}

pkv_status pkv_alloc_stats(const pkv_allocator* a, int64_t* allocated_blocks, int64_t* used_slots,
                           double* fragmentation) {
  if (!a) return PKV_ERR_INVALID_ARG;
  const int64_t bs = a->block_size;
  int64_t allocated = 0;
  for (int32_t r : a->ref) allocated += r > 0 ? 1 : 0;
  // rows in use: union over the sequences holding each block
  std::unordered_map<int32_t, std::vector<char>> rows;
  for (const auto& kv : a->seqs) {
    const auto& s = kv.second;
    for (int64_t i = 0; i < s.num_tokens; ++i) {
      const int64_t p = s.offset + i;
      auto& r = rows[s.blocks[(size_t)(p / bs)]];
      if (r.empty()) r.assign((size_t)bs, 0);
      r[(size_t)(p % bs)] = 1;
    }
  }
  int64_t used = 0;
  for (const auto& kv : rows)
    for (char c : kv.second) used += c;
  if (allocated_blocks) *allocated_blocks = allocated;
  if (used_slots) *used_slots = used;
  if (fragmentation)
    *fragmentation = allocated ? (double)(allocated * bs - used) / (double)(allocated * bs) : 0.0;
  return PKV_OK;
}

}  // extern "C"
