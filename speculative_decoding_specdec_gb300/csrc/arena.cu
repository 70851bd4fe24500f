// Host-side allocator of SequencePool arena columns (host code only; no kernels).
//
// "Batch Speculative Decoding Done Right", section 2.3: the pool's sequences come and go.  Each
// admitted sequence takes a run of consecutive columns of the pool's K/V arena, sized for its
// length limit, and gives it back when it finishes.  Runs are handed out first fit (the lowest
// column where enough consecutive columns are free); a freed run merges with free neighbours.
//
// The free runs live in an ordered map (start -> length), the allocations in another; first fit
// walks the free runs in column order.  One mutex per arena makes the calls thread safe.
#include <cstdint>
#include <iterator>
#include <map>
#include <mutex>
#include <new>

#include "specdec.h"

struct specdec_arena {
  int64_t cols = 0;
  std::map<int64_t, int64_t> free_runs;  // start -> length, disjoint and never adjacent
  std::map<int64_t, int64_t> used;       // start -> length of each allocation
  std::mutex mu;
};

extern "C" int specdec_arena_create(int64_t cols, specdec_arena** out) {
  if (!out || cols < 1) return SPECDEC_ERR_INVALID_ARG;
  specdec_arena* a = new (std::nothrow) specdec_arena;
  if (!a) return SPECDEC_ERR_CAPACITY;
  a->cols = cols;
  a->free_runs.emplace(0, cols);
  *out = a;
  return SPECDEC_OK;
}

extern "C" void specdec_arena_destroy(specdec_arena* a) { delete a; }

extern "C" int specdec_arena_alloc(specdec_arena* a, int64_t ncols, int64_t* col) {
  if (!a || !col || ncols < 1) return SPECDEC_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(a->mu);
  for (auto it = a->free_runs.begin(); it != a->free_runs.end(); ++it) {
    if (it->second < ncols) continue;
    const int64_t start = it->first, len = it->second;
    a->free_runs.erase(it);
    if (len > ncols) a->free_runs.emplace(start + ncols, len - ncols);
    a->used.emplace(start, ncols);
    *col = start;
    return SPECDEC_OK;
  }
  return SPECDEC_ERR_CAPACITY;
}

extern "C" int specdec_arena_free(specdec_arena* a, int64_t col) {
  if (!a) return SPECDEC_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(a->mu);
  auto u = a->used.find(col);
  if (u == a->used.end()) return SPECDEC_ERR_INVALID_ARG;
  int64_t start = u->first, len = u->second;
  a->used.erase(u);
  auto next = a->free_runs.lower_bound(start);
  if (next != a->free_runs.begin()) {  // merge with the free run just below
    auto prev = std::prev(next);
    if (prev->first + prev->second == start) {
      start = prev->first;
      len += prev->second;
      a->free_runs.erase(prev);
    }
  }
  if (next != a->free_runs.end() && start + len == next->first) {  // and the one just above
    len += next->second;
    a->free_runs.erase(next);
  }
  a->free_runs.emplace(start, len);
  return SPECDEC_OK;
}

extern "C" int specdec_arena_stats(specdec_arena* a, int64_t* free_cols, int64_t* largest_free,
                                   int64_t* allocations) {
  if (!a) return SPECDEC_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(a->mu);
  int64_t total = 0, big = 0;
  for (const auto& r : a->free_runs) {
    total += r.second;
    if (r.second > big) big = r.second;
  }
  if (free_cols) *free_cols = total;
  if (largest_free) *largest_free = big;
  if (allocations) *allocations = static_cast<int64_t>(a->used.size());
  return SPECDEC_OK;
}
