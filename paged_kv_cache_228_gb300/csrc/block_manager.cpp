// Host block manager: LIFO free list + per-block refcounts.
//
// "Paged Attention and KV Cache Fragmentation", section "How PagedAttention
// maps an OS concept onto GPU memory": blocks are all the same size, so any
// freed block fits any request; a sequence gets a block only when it grows
// past its last one; blocks return the moment a request finishes; sequences
// sharing a prefix point at the same physical blocks and diverge only where
// their content differs (copy-on-write of the shared partial tail).
//
// Every entry point validates first and mutates second, so a failing call
// leaves the allocator exactly as it was.
#include <cstdint>
#include <new>
#include <unordered_map>
#include <vector>

#include "pa.h"

struct pa_allocator {
  std::vector<int32_t> refcount;   // per block; 0 = free
  std::vector<int32_t> free_stack; // back() is the next block handed out
};

namespace {

inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

inline bool live(const pa_allocator* a, int32_t id) {
  return id >= 0 && id < static_cast<int32_t>(a->refcount.size()) &&
         a->refcount[id] > 0;
}

}  // namespace

extern "C" pa_status pa_allocator_create(int32_t num_blocks,
                                         pa_allocator** out) {
  if (out == nullptr || num_blocks < 0) return PA_ERR_INVALID_ARG;
  pa_allocator* a = new (std::nothrow) pa_allocator;
  if (a == nullptr) return PA_ERR_INVALID_ARG;
  try {
    a->refcount.assign(static_cast<size_t>(num_blocks), 0);
    a->free_stack.resize(static_cast<size_t>(num_blocks));
  } catch (...) {
    delete a;
    return PA_ERR_INVALID_ARG;
  }
  // Highest id at the bottom: a fresh allocator hands out 0, 1, 2, ...
  for (int32_t i = 0; i < num_blocks; ++i)
    a->free_stack[static_cast<size_t>(i)] = num_blocks - 1 - i;
  *out = a;
  return PA_OK;
}

extern "C" void pa_allocator_destroy(pa_allocator* a) { delete a; }

extern "C" int32_t pa_block_num_free(const pa_allocator* a) {
  return a ? static_cast<int32_t>(a->free_stack.size()) : -1;
}

extern "C" pa_status pa_block_refcount(const pa_allocator* a, int32_t id,
                                       int32_t* rc) {
  if (a == nullptr || rc == nullptr) return PA_ERR_INVALID_ARG;
  if (id < 0 || id >= static_cast<int32_t>(a->refcount.size()))
    return PA_ERR_BAD_BLOCK_ID;
  *rc = a->refcount[id];
  return PA_OK;
}

extern "C" pa_status pa_block_alloc(pa_allocator* a, int32_t n,
                                    int32_t* ids_out) {
  if (a == nullptr || n < 0 || (n > 0 && ids_out == nullptr))
    return PA_ERR_INVALID_ARG;
  if (static_cast<size_t>(n) > a->free_stack.size())
    return PA_ERR_OUT_OF_BLOCKS;
  for (int32_t i = 0; i < n; ++i) {
    const int32_t id = a->free_stack.back();
    a->free_stack.pop_back();
    a->refcount[id] = 1;
    ids_out[i] = id;
  }
  return PA_OK;
}

extern "C" pa_status pa_block_free(pa_allocator* a, const int32_t* ids,
                                   int32_t n) {
  if (a == nullptr || n < 0 || (n > 0 && ids == nullptr))
    return PA_ERR_INVALID_ARG;
  std::unordered_map<int32_t, int32_t> need;
  for (int32_t i = 0; i < n; ++i) {
    const int32_t id = ids[i];
    if (id < 0 || id >= static_cast<int32_t>(a->refcount.size()))
      return PA_ERR_BAD_BLOCK_ID;
    ++need[id];
  }
  for (const auto& kv : need)
    if (a->refcount[kv.first] < kv.second) return PA_ERR_BAD_BLOCK_ID;
  for (int32_t i = 0; i < n; ++i) {
    const int32_t id = ids[i];
    if (--a->refcount[id] == 0) a->free_stack.push_back(id);
  }
  return PA_OK;
}

extern "C" pa_status pa_block_fork(pa_allocator* a, const int32_t* ids,
                                   int32_t n) {
  if (a == nullptr || n < 0 || (n > 0 && ids == nullptr))
    return PA_ERR_INVALID_ARG;
  for (int32_t i = 0; i < n; ++i)
    if (!live(a, ids[i])) return PA_ERR_BAD_BLOCK_ID;
  for (int32_t i = 0; i < n; ++i) ++a->refcount[ids[i]];
  return PA_OK;
}

extern "C" pa_status pa_seq_append_slots(pa_allocator* a, int32_t* table,
                                         int32_t max_blocks, int32_t len,
                                         int32_t n, int32_t block_size,
                                         int64_t* slots_out,
                                         int32_t* cow_pair_out,
                                         int32_t* num_cow) {
  if (a == nullptr || num_cow == nullptr || len < 0 || n < 0 ||
      block_size <= 0 || max_blocks < 0)
    return PA_ERR_INVALID_ARG;
  if ((max_blocks > 0 && table == nullptr) || (n > 0 && slots_out == nullptr))
    return PA_ERR_INVALID_ARG;
  const int64_t held = cdiv(len, block_size);
  const int64_t want = cdiv(static_cast<int64_t>(len) + n, block_size);
  if (want > max_blocks) return PA_ERR_INVALID_ARG;
  for (int64_t j = 0; j < held; ++j)
    if (!live(a, table[j])) return PA_ERR_BAD_BLOCK_ID;
  const bool cow = n > 0 && (len % block_size) != 0 &&
                   a->refcount[table[held - 1]] > 1;
  if (cow && cow_pair_out == nullptr) return PA_ERR_INVALID_ARG;
  const int64_t extra = (want - held) + (cow ? 1 : 0);
  if (extra > static_cast<int64_t>(a->free_stack.size()))
    return PA_ERR_OUT_OF_BLOCKS;

  *num_cow = 0;
  if (cow) {
    const int32_t old_id = table[held - 1];
    const int32_t new_id = a->free_stack.back();
    a->free_stack.pop_back();
    a->refcount[new_id] = 1;
    --a->refcount[old_id];
    table[held - 1] = new_id;
    cow_pair_out[0] = old_id;
    cow_pair_out[1] = new_id;
    cow_pair_out[2] = len % block_size;
    *num_cow = 1;
  }
  for (int64_t j = held; j < want; ++j) {
    const int32_t id = a->free_stack.back();
    a->free_stack.pop_back();
    a->refcount[id] = 1;
    table[j] = id;
  }
  for (int32_t i = 0; i < n; ++i) {
    const int64_t p = static_cast<int64_t>(len) + i;
    slots_out[i] = static_cast<int64_t>(table[p / block_size]) * block_size +
                   p % block_size;
  }
  return PA_OK;
}

extern "C" pa_status pa_batch_append_slots(pa_allocator* a, int32_t* tables,
                                           int32_t max_blocks, const int32_t* lens,
                                           const int32_t* n_new, int32_t num_seqs,
                                           int32_t block_size, int64_t* slots_out,
                                           int32_t* cow_pairs_out, int32_t* n_cow_out,
                                           int32_t* num_done) {
  if (num_done == nullptr) return PA_ERR_INVALID_ARG;
  *num_done = 0;
  if (a == nullptr || num_seqs < 0 || max_blocks < 0) return PA_ERR_INVALID_ARG;
  if (num_seqs > 0 && (lens == nullptr || n_new == nullptr || cow_pairs_out == nullptr ||
                       n_cow_out == nullptr || (max_blocks > 0 && tables == nullptr)))
    return PA_ERR_INVALID_ARG;
  int64_t at = 0;  // next slot index in slots_out
  for (int32_t i = 0; i < num_seqs; ++i) {
    const pa_status st = pa_seq_append_slots(
        a, tables + static_cast<int64_t>(i) * max_blocks, max_blocks, lens[i], n_new[i],
        block_size, slots_out == nullptr ? nullptr : slots_out + at, cow_pairs_out + 3 * i,
        n_cow_out + i);
    if (st != PA_OK) return st;
    at += n_new[i];
    *num_done = i + 1;
  }
  return PA_OK;
}

extern "C" pa_status pa_allocator_usage(const pa_allocator* a, const int32_t* tables,
                                        int32_t max_blocks, const int32_t* lens,
                                        int32_t num_seqs, int32_t block_size, int64_t* out) {
  if (a == nullptr || out == nullptr || num_seqs < 0 || max_blocks < 0 || block_size <= 0)
    return PA_ERR_INVALID_ARG;
  if (num_seqs > 0 && (lens == nullptr || (max_blocks > 0 && tables == nullptr)))
    return PA_ERR_INVALID_ARG;
  // per block: the furthest offset any sequence fills (slots 0..fill-1 of a
  // block hold tokens of its holders; a sequence fills its blocks from 0)
  std::vector<int32_t> fill(a->refcount.size(), 0);
  int64_t logical = 0;
  for (int32_t i = 0; i < num_seqs; ++i) {
    const int64_t n = lens[i];
    if (n < 0 || cdiv(n, block_size) > max_blocks) return PA_ERR_INVALID_ARG;
    logical += n;
    const int32_t* t = tables + static_cast<int64_t>(i) * max_blocks;
    for (int64_t j = 0; j < cdiv(n, block_size); ++j) {
      if (!live(a, t[j])) return PA_ERR_BAD_BLOCK_ID;
      const int64_t f = n - j * block_size < block_size ? n - j * block_size : block_size;
      if (f > fill[t[j]]) fill[t[j]] = static_cast<int32_t>(f);
    }
  }
  int64_t live_blocks = 0, stored = 0;
  for (size_t b = 0; b < fill.size(); ++b) {
    live_blocks += a->refcount[b] > 0;
    stored += fill[b];
  }
  out[0] = live_blocks;
  out[1] = live_blocks * block_size;
  out[2] = stored;
  out[3] = logical;
  return PA_OK;
}
