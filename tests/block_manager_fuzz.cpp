// Randomised driver of the host block manager, built with AddressSanitizer
// and UndefinedBehaviorSanitizer by tests/test_block_manager_sanitized.py.
//
// It calls every allocator entry point of include/pa.h -- valid and invalid
// arguments alike -- and checks the invariants of "Paged Attention and KV
// Cache Fragmentation", section "How PagedAttention maps an OS concept onto
// GPU memory": blocks are all the same size, a block is free exactly when
// nothing references it, and a failing call changes nothing.
//   free blocks + distinct referenced blocks == pool size
//   refcount(id) == number of sequences (and extra references) holding id
// Any sanitizer report aborts with a non-zero status; an invariant failure
// returns 1.
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <map>
#include <random>
#include <vector>

#include "pa.h"

namespace {

constexpr int32_t kPool = 96;
constexpr int32_t kBs = 8;
constexpr int32_t kMaxBlocks = 24;

struct Seq {
  std::vector<int32_t> table;  // kMaxBlocks entries, -1 past the held ones
  int32_t len = 0;
};

int held(const Seq& s) { return (s.len + kBs - 1) / kBs; }

bool check(pa_allocator* a, const std::vector<Seq>& seqs, const std::vector<int32_t>& extra) {
  std::map<int32_t, int32_t> refs;
  for (const Seq& s : seqs)
    for (int j = 0; j < held(s); ++j) ++refs[s.table[j]];
  for (int32_t id : extra) ++refs[id];
  for (int32_t id = 0; id < kPool; ++id) {
    int32_t rc = -1;
    if (pa_block_refcount(a, id, &rc) != PA_OK) return false;
    const auto it = refs.find(id);
    if (rc != (it == refs.end() ? 0 : it->second)) {
      std::fprintf(stderr, "block %d: refcount %d, holders %d\n", id, rc,
                   it == refs.end() ? 0 : it->second);
      return false;
    }
  }
  if (pa_block_num_free(a) + static_cast<int32_t>(refs.size()) != kPool) {
    std::fprintf(stderr, "free %d + live %zu != %d\n", pa_block_num_free(a), refs.size(), kPool);
    return false;
  }
  return true;
}

}  // namespace

int main(int argc, char** argv) {
  const uint32_t seed = argc > 1 ? static_cast<uint32_t>(std::atoi(argv[1])) : 1u;
  const int steps = argc > 2 ? std::atoi(argv[2]) : 20000;
  std::mt19937 rng(seed);
  auto pick = [&](int n) { return static_cast<int>(rng() % static_cast<uint32_t>(n)); };

  pa_allocator* a = nullptr;
  if (pa_allocator_create(-1, &a) != PA_ERR_INVALID_ARG) return 1;
  if (pa_allocator_create(kPool, &a) != PA_OK || a == nullptr) return 1;
  std::vector<Seq> seqs;
  std::vector<int32_t> extra;  // references taken by pa_block_alloc / fork
  std::vector<int64_t> slots(4 * kMaxBlocks * kBs);
  int32_t cow[3 * 64];

  for (int step = 0; step < steps; ++step) {
    const int op = pick(9);
    if (op <= 2) {  // append n tokens to a (possibly new) sequence
      if (seqs.empty() || pick(4) == 0) {
        seqs.emplace_back();
        seqs.back().table.assign(kMaxBlocks, -1);
      }
      Seq& s = seqs[pick(static_cast<int>(seqs.size()))];
      const int32_t n = pick(3 * kBs);
      int32_t ncow = -1;
      const pa_status st = pa_seq_append_slots(a, s.table.data(), kMaxBlocks, s.len, n, kBs,
                                               slots.data(), cow, &ncow);
      if (st == PA_OK) {
        for (int32_t i = 0; i < n; ++i) {
          const int64_t p = s.len + i;
          if (slots[i] != static_cast<int64_t>(s.table[p / kBs]) * kBs + p % kBs) return 1;
        }
        s.len += n;
      } else if (st != PA_ERR_OUT_OF_BLOCKS && st != PA_ERR_INVALID_ARG) {
        return 1;
      }
    } else if (op == 3 && !seqs.empty()) {  // fork a sequence
      const Seq src = seqs[pick(static_cast<int>(seqs.size()))];
      if (pa_block_fork(a, src.table.data(), held(src)) != PA_OK) return 1;
      seqs.push_back(src);
    } else if (op == 4 && !seqs.empty()) {  // finish a sequence
      const int i = pick(static_cast<int>(seqs.size()));
      if (pa_block_free(a, seqs[i].table.data(), held(seqs[i])) != PA_OK) return 1;
      seqs.erase(seqs.begin() + i);
    } else if (op == 5) {  // raw alloc / free of extra references
      const int32_t n = pick(6);
      std::vector<int32_t> ids(static_cast<size_t>(n) + 1);
      const pa_status st = pa_block_alloc(a, n, ids.data());
      if (st == PA_OK)
        extra.insert(extra.end(), ids.begin(), ids.begin() + n);
      else if (st != PA_ERR_OUT_OF_BLOCKS)
        return 1;
      if (!extra.empty() && pick(2) == 0) {
        const int32_t id = extra.back();
        extra.pop_back();
        if (pa_block_free(a, &id, 1) != PA_OK) return 1;
      }
    } else if (op == 6) {  // invalid calls: nothing may change
      const int32_t bad[3] = {-1, kPool, kPool + 7};
      const int32_t id = bad[pick(3)];
      int32_t rc = 0;
      if (pa_block_free(a, &id, 1) != PA_ERR_BAD_BLOCK_ID) return 1;
      if (pa_block_fork(a, &id, 1) != PA_ERR_BAD_BLOCK_ID) return 1;
      if (pa_block_refcount(a, id, &rc) != PA_ERR_BAD_BLOCK_ID) return 1;
      if (pa_block_alloc(a, -1, nullptr) != PA_ERR_INVALID_ARG) return 1;
      if (pa_block_alloc(a, kPool + 1, slots.data() != nullptr ? cow : nullptr) !=
          PA_ERR_OUT_OF_BLOCKS)
        return 1;
      int32_t ncow = 0;
      int32_t table[kMaxBlocks];
      if (pa_seq_append_slots(a, table, kMaxBlocks, 0, kMaxBlocks * kBs + 1, kBs,
                              slots.data(), cow, &ncow) != PA_ERR_INVALID_ARG)
        return 1;
    } else if (op == 7 && !seqs.empty()) {  // a batch of one-token appends
      const int32_t b = static_cast<int32_t>(seqs.size());
      std::vector<int32_t> tables(static_cast<size_t>(b) * kMaxBlocks), lens(b), ones(b, 1);
      std::vector<int32_t> ncow(b);
      std::vector<int32_t> pairs(3 * static_cast<size_t>(b));
      std::vector<int64_t> out(b);
      for (int32_t i = 0; i < b; ++i) {
        for (int j = 0; j < kMaxBlocks; ++j) tables[i * kMaxBlocks + j] = seqs[i].table[j];
        lens[i] = seqs[i].len;
      }
      int32_t done = -1;
      const pa_status st =
          pa_batch_append_slots(a, tables.data(), kMaxBlocks, lens.data(), ones.data(), b, kBs,
                                out.data(), pairs.data(), ncow.data(), &done);
      if (st != PA_OK && st != PA_ERR_OUT_OF_BLOCKS && st != PA_ERR_INVALID_ARG) return 1;
      for (int32_t i = 0; i < done; ++i) {  // the sequences the call completed
        for (int j = 0; j < kMaxBlocks; ++j) seqs[i].table[j] = tables[i * kMaxBlocks + j];
        seqs[i].len += 1;
      }
    } else if (op == 8 && !seqs.empty()) {  // usage report
      const int32_t b = static_cast<int32_t>(seqs.size());
      std::vector<int32_t> tables(static_cast<size_t>(b) * kMaxBlocks), lens(b);
      for (int32_t i = 0; i < b; ++i) {
        for (int j = 0; j < kMaxBlocks; ++j) tables[i * kMaxBlocks + j] = seqs[i].table[j];
        lens[i] = seqs[i].len;
      }
      int64_t u[4];
      if (pa_allocator_usage(a, tables.data(), kMaxBlocks, lens.data(), b, kBs, u) != PA_OK)
        return 1;
      if (u[1] != u[0] * kBs || u[2] > u[1] || u[2] > u[3]) return 1;
    }
    if (!check(a, seqs, extra)) {
      std::fprintf(stderr, "invariant broken at step %d (op %d)\n", step, op);
      return 1;
    }
  }
  for (const Seq& s : seqs)
    if (pa_block_free(a, s.table.data(), held(s)) != PA_OK) return 1;
  if (!extra.empty() && pa_block_free(a, extra.data(), static_cast<int32_t>(extra.size())) != PA_OK)
    return 1;
  if (pa_block_num_free(a) != kPool) return 1;
  pa_allocator_destroy(a);
  std::printf("ok %d steps\n", steps);
  return 0;
}
