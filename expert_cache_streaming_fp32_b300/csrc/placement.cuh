// Expert-placement policies replayed on a routing trace (host only): the
// shared LRU of the cache, a hot set frozen at prefill time, and a static
// split by layer.  Part of the single translation unit ft.cu.
#pragma once

#include <algorithm>
#include <set>
#include <utility>
#include <vector>

#include "common.cuh"

namespace ft {

// Unique valid experts of one layer step, ascending.
static void unique_experts(const int32_t* ids, int width, int E, std::vector<int>& out) {
  out.clear();
  for (int i = 0; i < width; ++i)
    if (ids[i] >= 0 && ids[i] < E) out.push_back(ids[i]);
  std::sort(out.begin(), out.end());
  out.erase(std::unique(out.begin(), out.end()), out.end());
}

// The shared LRU with every miss filled: the cache step's rules (one stamp per
// layer step, victims empty slots first by slot, then the oldest (stamp, slot)).
// capacity >= E, so a layer step never needs more slots than there are.
static void replay_lru(int L, int E, int C, const int32_t* trace, int n_steps, int width, uint64_t& acc,
                       uint64_t& miss) {
  std::vector<int> key(C, -1), where((size_t)L * E, -1);
  std::vector<uint32_t> stamp(C, 0);
  std::set<std::pair<uint32_t, int>> occupied;
  std::set<int> empty;
  for (int s = 0; s < C; ++s) empty.insert(s);
  uint32_t clock = 0;
  std::vector<int> U, misses;
  for (int t = 0; t < n_steps; ++t) {
    for (int l = 0; l < L; ++l) {
      unique_experts(trace + ((size_t)t * L + l) * width, width, E, U);
      acc += U.size();
      if (U.empty()) continue;
      ++clock;
      misses.clear();
      for (int e : U) {
        const int k = l * E + e, s = where[k];
        if (s >= 0) {
          occupied.erase({stamp[s], s});
          stamp[s] = clock;
          occupied.insert({clock, s});
        } else {
          misses.push_back(e);
        }
      }
      for (int e : misses) {
        int s;
        if (!empty.empty()) {
          s = *empty.begin();
          empty.erase(empty.begin());
        } else {
          auto it = occupied.begin();  // oldest; never this step's (capacity >= E)
          s = it->second;
          occupied.erase(it);
          where[key[s]] = -1;
        }
        const int k = l * E + e;
        key[s] = k;
        stamp[s] = clock;
        where[k] = s;
        occupied.insert({clock, s});
        ++miss;
      }
    }
  }
}

static void replay_fixed(int L, int E, const std::vector<char>& resident, const int32_t* trace, int n_steps,
                         int width, uint64_t& acc, uint64_t& miss) {
  std::vector<int> U;
  for (int t = 0; t < n_steps; ++t)
    for (int l = 0; l < L; ++l) {
      unique_experts(trace + ((size_t)t * L + l) * width, width, E, U);
      acc += U.size();
      for (int e : U) miss += !resident[(size_t)l * E + e];
    }
}

}  // namespace ft
