// Host-side check of the persistent kernels' static work schedule: every
// (tile, head) item is handed to exactly one CTA, whatever the mode, shape or
// grid, and the chosen mode balances the causal costs. Prints one line per
// case: "ok <N> <Nk> <BH> <causal> <sms> <mode> <G> <balance>" or "FAIL ...".
#include <algorithm>
#include <cstdio>
#include <vector>

#include "tile_sched.h"

using fa::TileSched;

// cost by rank of a query tile (forward, dQ pass): key tiles it visits + 1
static std::vector<long long> fwd_costs(int N, int Nk, bool causal) {
  const int nt = (N + 127) / 128, nall = (Nk + 127) / 128, off = Nk - N;
  std::vector<long long> c(nt);
  for (int r = 0; r < nt; ++r) {
    const int q = nt - 1 - r;
    c[r] = (causal ? std::min(nall, (q * 128 + 127 + off) / 128 + 1) : nall) + 1;
  }
  return c;
}

static bool run(int N, int Nk, int BH, bool causal, int sms, double min_balance) {
  const std::vector<long long> cost = fwd_costs(N, Nk, causal);
  const int nt = static_cast<int>(cost.size());
  bool ok = true;
  double balance = 0;
  TileSched chosen = fa::sched_make(BH, nt, cost.data(), causal, sms);
  // the chosen schedule and every mode on its own must cover each item once
  for (int mode = -1; mode <= (causal ? 1 : 0); ++mode) {
    TileSched s = chosen;
    if (mode >= 0) {
      s.mode = mode;
      s.per = (nt + 1) / 2;
      s.hs = 0;
      s.P = 0;
      if (mode == fa::kPairs) {
        const int want = (2 * sms + nt - 1) / nt;
        s.hs = std::min(want, BH);
        s.P = (BH - s.hs) * s.per;
      }
    }
    std::vector<int> seen(static_cast<size_t>(BH) * nt, 0);
    long long span = 0, total = 0;
    for (int c = 0; c < s.G; ++c) {
      int rank, bh, st;
      long long load = 0;
      for (int k = 0; (st = fa::sched_item(s, c, k, rank, bh)) != fa::kDone; ++k) {
        if (st == fa::kSkip) continue;
        if (st != fa::kItem || rank < 0 || rank >= nt || bh < 0 || bh >= BH || k > 4 * BH * nt + 8) {
          ok = false;
          break;
        }
        ++seen[static_cast<size_t>(bh) * nt + rank];
        load += cost[rank];
      }
      span = std::max(span, load);
      total += load;
    }
    for (int v : seen) ok = ok && v == 1;
    if (mode < 0) balance = static_cast<double>(total) / s.G / static_cast<double>(span);
  }
  ok = ok && chosen.G >= 1 && chosen.G <= sms && balance >= min_balance;
  std::printf("%s %d %d %d %d %d %d %d %.3f\n", ok ? "ok" : "FAIL", N, Nk, BH, causal ? 1 : 0, sms, chosen.mode,
              chosen.G, balance);
  return ok;
}

// The mode sched_make picks for a causal shape with the forward's costs.
static bool expect_mode(int N, int Nk, int BH, int sms, int mode) {
  const std::vector<long long> cost = fwd_costs(N, Nk, true);
  const TileSched s = fa::sched_make(BH, static_cast<int>(cost.size()), cost.data(), true, sms);
  const bool ok = s.mode == mode;
  std::printf("%s mode %d %d %d %d\n", ok ? "ok" : "FAIL", N, Nk, BH, s.mode);
  return ok;
}

int main() {
  bool ok = true;
  // balance floors where the schedule has enough work per CTA to balance
  ok &= run(4096, 4096, 256, false, 152, 0.99);
  ok &= run(4096, 4096, 256, true, 152, 0.99);
  ok &= run(65536, 65536, 32, true, 152, 0.99);
  ok &= run(16384, 16384, 32, true, 152, 0.98);
  ok &= run(8192, 8192, 16, true, 152, 0.97);
  ok &= run(4096, 16384, 32, true, 152, 0.9);
  ok &= run(128, 8192, 2048, true, 152, 0.9);
  // the shapes of the GPU schedule test: the mode each one exercises
  ok &= expect_mode(2048, 2048, 48, 152, fa::kPairs);
  ok &= expect_mode(1000, 4000, 40, 152, fa::kSnake);
  ok &= expect_mode(1400, 1400, 60, 152, fa::kPairs);
  // coverage only: small, ragged and odd shapes, other SM counts
  const int Ns[] = {1, 100, 128, 129, 255, 256, 300, 1000, 1152, 2049};
  const int BHs[] = {1, 2, 3, 7, 19, 64};
  const int smss[] = {1, 2, 5, 148, 152};
  for (int N : Ns)
    for (int BH : BHs)
      for (int sms : smss)
        for (int causal = 0; causal < 2; ++causal)
          for (int extra : {0, 77, 1024}) ok &= run(N, N + extra, BH, causal != 0, sms, 0.0);
  std::printf(ok ? "ALL OK\n" : "SOME FAILED\n");
  return ok ? 0 : 1;
}
