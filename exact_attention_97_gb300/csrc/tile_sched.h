// tile_sched.h -- static work schedule of the persistent attention kernels.
//
// A kernel's work is BH heads x nt tiles per head (query tiles for the
// forward and the dQ pass, key blocks for the dK/dV pass). Under the causal
// mask tiles differ in cost; the schedule sees them only through their rank:
// rank 0 is the most expensive tile of a head, rank nt-1 the cheapest, and
// the cost never grows with the rank. The kernel maps a rank back to its tile.
//
// G persistent CTAs each walk their own list of (rank, head) items;
// sched_item gives item k of CTA c. Two modes, both fixed before the launch
// (no atomics, no device-side state):
//
//   kSnake  items in head-major order, ranks ascending within a head; position
//           v goes to CTA v % G in even rounds (v / G) and to G-1 - v % G in
//           odd rounds. Consecutive positions share heads, so the CTAs running
//           together read the K/V (or Q/dO) of a few heads through L2.
//   kPairs  (causal only) the first P = (BH - hs) * ceil(nt/2) units pair
//           rank p with rank nt-1-p of one head -- every pair costs about the
//           same -- and are dealt round-robin; the last hs heads are then cut
//           into single tiles, heaviest first, dealt in snake order starting
//           at the CTAs that got one pair fewer.
//
// The host evaluates the makespan of both (exact tile costs) and launches the
// cheaper one. This header compiles as plain C++ too, so the CPU tests can
// check that every item is scheduled exactly once.
#pragma once

#include <mutex>
#include <vector>

#if defined(__CUDACC__)
#define FA_HD __host__ __device__ __forceinline__
#else
#define FA_HD inline
#endif

namespace fa {

enum SchedMode : int { kSnake = 0, kPairs = 1 };

struct TileSched {
  int mode;  // SchedMode
  int G;     // CTAs
  int nt;    // tiles per head
  int BH;    // heads (batch x heads)
  int per;   // kPairs: pair units per head, ceil(nt / 2)
  int hs;    // kPairs: heads cut into single tiles at the end
  int P;     // kPairs: pair units, (BH - hs) * per
};

// Item k of CTA c, in closed form (no state carried between calls):
// returns kItem and sets (rank, bh), kSkip for an empty slot (the second half
// of the middle unit of an odd head under kPairs: every role skips it alike),
// or kDone past the CTA's last item. Positions stay below 2^31: the host
// limits B*H*N.
enum SchedStep : int { kDone = 0, kItem = 1, kSkip = 2 };

// position of CTA c in snake round q (odd rounds run the CTAs backwards)
FA_HD int sched_snake_pos(const TileSched &s, int c, int q) { return q * s.G + ((q & 1) ? s.G - 1 - c : c); }

FA_HD int sched_item(const TileSched &s, int c, int k, int &rank, int &bh) {
  if (s.mode == kSnake) {
    const int v = sched_snake_pos(s, c, k);
    if (v >= s.BH * s.nt) return kDone;
    bh = v / s.nt;
    rank = v - bh * s.nt;
    return kItem;
  }
  // pairs: CTA c holds units c, c + G, ... below P, two slots each
  const int units = c < s.P ? (s.P - 1 - c) / s.G + 1 : 0;
  if (k < 2 * units) {
    const int u = c + (k >> 1) * s.G;
    bh = u / s.per;
    const int p = u - bh * s.per;
    if ((k & 1) == 0) {
      rank = p;
      return kItem;
    }
    if (2 * p + 1 == s.nt) return kSkip;
    rank = s.nt - 1 - p;
    return kItem;
  }
  // singles of the last hs heads, heaviest first, snake order offset by P % G
  const int o = s.P % s.G;
  const int q = (k - 2 * units) + (sched_snake_pos(s, c, 0) < o ? 1 : 0);
  const int v = sched_snake_pos(s, c, q) - o;
  if (v >= s.hs * s.nt) return kDone;
  rank = v / s.hs;
  bh = (s.BH - s.hs) + (v - rank * s.hs);
  return kItem;
}

// Above this many items the host does not compare the modes.
constexpr long long kSchedEvalItems = 1ll << 16;

// True when sched_make needs the per-rank costs.
inline bool sched_needs_cost(int BH, int nt, bool causal) {
  return causal && static_cast<long long>(BH) * nt <= kSchedEvalItems;
}

// Host side: pick the mode and grid for BH heads of nt tiles whose costs by
// rank are cost[0..nt-1] (non-increasing), on num_sms SMs.
inline TileSched sched_make(int BH, int nt, const long long *cost, bool causal, int num_sms) {
  TileSched best{};
  long long best_span = -1;
  const long long items = static_cast<long long>(BH) * nt;
  // equal costs: the snake is optimal; very many items: pairs, whose balance
  // only improves with the count (and evaluating would cost host time)
  const bool many = items > kSchedEvalItems;
  const int first = (causal && many) ? kPairs : kSnake;
  const int last = (causal && !many) ? kPairs : first;
  for (int mode = first; mode <= last; ++mode) {
    TileSched s{};
    s.mode = mode;
    s.nt = nt;
    s.BH = BH;
    s.per = (nt + 1) / 2;
    if (mode == kPairs) {
      const int want = (2 * num_sms + nt - 1) / nt;  // about two singles per CTA
      s.hs = want < BH ? want : BH;
      s.P = (BH - s.hs) * s.per;
    }
    long long units = mode == kPairs ? static_cast<long long>(s.P) + static_cast<long long>(s.hs) * nt : items;
    s.G = static_cast<int>(units < num_sms ? units : num_sms);
    if (s.G < 1) s.G = 1;
    if (first == last) return s;
    // exact makespan: the largest total cost over CTAs
    long long span = 0;
    for (int c = 0; c < s.G; ++c) {
      long long load = 0;
      int rank, bh, st;
      for (int k = 0; (st = sched_item(s, c, k, rank, bh)) != kDone; ++k)
        if (st == kItem) load += cost[rank];
      if (load > span) span = load;
    }
    if (best_span < 0 || span < best_span) {
      best = s;
      best_span = span;
    }
  }
  return best;
}

// Memoised sched_make for one kind of kernel: the mode comparison walks every
// item once, so its result is kept per shape (a few dozen shapes at most).
// cost_of(rank) gives the cost of a rank when the comparison needs it.
template <typename CostFn>
TileSched sched_cached(int kind, int BH, int N, int Nk, bool causal, int nt, int num_sms, CostFn cost_of) {
  struct Entry {
    int kind, BH, N, Nk, causal, num_sms;
    TileSched s;
  };
  static std::mutex mu;
  static std::vector<Entry> cache;
  {
    std::lock_guard<std::mutex> lock(mu);
    for (const Entry &e : cache)
      if (e.kind == kind && e.BH == BH && e.N == N && e.Nk == Nk && e.causal == (causal ? 1 : 0) &&
          e.num_sms == num_sms)
        return e.s;
  }
  std::vector<long long> cost;
  if (sched_needs_cost(BH, nt, causal)) {
    cost.resize(nt);
    for (int r = 0; r < nt; ++r) cost[r] = cost_of(r);
  }
  const TileSched s = sched_make(BH, nt, cost.empty() ? nullptr : cost.data(), causal, num_sms);
  std::lock_guard<std::mutex> lock(mu);
  if (cache.size() >= 64) cache.erase(cache.begin());
  cache.push_back(Entry{kind, BH, N, Nk, causal ? 1 : 0, num_sms, s});
  return s;
}

}  // namespace fa
