// ne_sched.cu -- work schedule of the persistent attention backward (host code).
//
// The backward main kernel runs one CTA per SM over a list of work units of
// unequal length, indexed longest first: unit r is key tile j = r / (nseq H)
// of one (sequence, head), and takes one step per query tile i >= j
// (n_tiles - j steps).  Every unit also costs a roughly fixed amount at its
// boundaries (its K', V loads, its dV/dK epilogue): measured on GB300 with
// globaltimer stamps of every CTA, 1.2-1.8 steps, so short units cost far
// more than their steps.  The kernel's time is that of its busiest CTA.
//
// For a fixed-length batch the host packs the list instead of letting the
// kernel deal it in a snake order.  The packer tries a few candidates -- the
// snake order itself, a round-robin longest-processing-time deal (every CTA
// takes one unit per round, the round's longest units going to the
// least-loaded CTAs), and MULTIFIT (first fit decreasing inside a capacity
// found by bisection; Coffman, Garey and Johnson, "An application of
// bin-packing to multiprocessor scheduling", SIAM J. Comput. 7, 1978) on
// steps plus a per-unit overhead -- and keeps the one whose busiest CTA is
// lowest relative to the mean, taken at the worst of three overheads across
// the measured range.  Only the assignment changes: every unit is computed
// the same way by whichever CTA gets it (dK, dV bitwise the same).
//
// Measured on GB300 (training pair, L2 flushed): the GPT-2-small step gains
// 2-3 us (the round-robin deal: busiest CTA 1.066 of the mean against 1.096);
// at 4096 and 16384 positions the snake order is kept or the packing changes
// nothing measurable.  Packing the forward's items the same way (pairs of
// query tiles, ~2 steps of overhead each) saved 2 us at 4096 positions but
// cost 1 us on GPT-2-small: CTAs doing identical work differ by up to 30%
// there (cold start after the flush), more than the packing moves, so the
// forward keeps the snake order.
#include <algorithm>
#include <cstddef>
#include <numeric>
#include <vector>

namespace ne {

namespace {

using Bins = std::vector<std::vector<int>>;

// Busiest CTA over the mean, with per-unit overhead c.
double balance(const Bins& bins, const std::vector<int>& w, double c) {
  double total = 0.0, worst = 0.0;
  for (int x : w) total += x + c;
  for (const auto& b : bins) {
    double load = 0.0;
    for (int i : b) load += w[i] + c;
    worst = std::max(worst, load);
  }
  const double mean = total / static_cast<double>(bins.size());
  return mean > 0.0 ? worst / mean : 1.0;
}

double worst_balance(const Bins& bins, const std::vector<int>& w, const double (&cs)[3]) {
  double v = 0.0;
  for (double c : cs) v = std::max(v, balance(bins, w, c));
  return v;
}

Bins snake(int n, int G) {
  Bins bins(G);
  for (int k = 0; static_cast<long long>(k) * G < n; ++k)
    for (int c = 0; c < G; ++c) {
      const long long r = static_cast<long long>(k) * G + ((k & 1) ? (G - 1 - c) : c);
      if (r < n) bins[c].push_back(static_cast<int>(r));
    }
  return bins;
}

// Units by decreasing steps (ties: increasing index, i.e. the list order).
std::vector<int> by_length(const std::vector<int>& w) {
  std::vector<int> order(w.size());
  std::iota(order.begin(), order.end(), 0);
  std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return w[a] > w[b]; });
  return order;
}

Bins round_robin_lpt(const std::vector<int>& w, int G) {
  const std::vector<int> order = by_length(w);
  Bins bins(G);
  std::vector<long long> load(G, 0);
  std::vector<int> cta(G);
  for (size_t s = 0; s < order.size(); s += G) {
    std::iota(cta.begin(), cta.end(), 0);
    std::stable_sort(cta.begin(), cta.end(), [&](int a, int b) { return load[a] < load[b]; });
    for (size_t j = 0; j < static_cast<size_t>(G) && s + j < order.size(); ++j) {
      const int i = order[s + j];
      bins[cta[j]].push_back(i);
      load[cta[j]] += w[i];
    }
  }
  return bins;
}

// First fit decreasing of units with cost w + c into bins of capacity cap;
// false if it needs more than G bins.
bool first_fit(const std::vector<int>& order, const std::vector<int>& w, double c, double cap,
               int G, Bins& bins) {
  bins.assign(G, {});
  std::vector<double> load(G, 0.0);
  int used = 0;
  for (int i : order) {
    const double x = w[i] + c;
    int b = 0;
    while (b < used && load[b] + x > cap + 1e-9) ++b;
    if (b == used) {
      if (used == G) return false;
      ++used;
    }
    load[b] += x;
    bins[b].push_back(i);
  }
  return true;
}

Bins multifit(const std::vector<int>& w, int G, double c) {
  const std::vector<int> order = by_length(w);
  double total = 0.0, big = 0.0;
  for (int x : w) {
    total += x + c;
    big = std::max(big, x + c);
  }
  // First fit always succeeds at mean + largest: a unit that fits nowhere
  // would mean every bin holds more than the mean.
  double lo = std::max(big, total / G), hi = total / G + big;
  Bins best, trial;
  first_fit(order, w, c, hi, G, best);
  for (int it = 0; it < 24 && hi - lo > 1e-3; ++it) {
    const double mid = 0.5 * (lo + hi);
    if (first_fit(order, w, c, mid, G, trial)) {
      hi = mid;
      best.swap(trial);
    } else {
      lo = mid;
    }
  }
  return best;
}

}  // namespace

// Steps of every backward unit, in the kernel's longest-first index order.
std::vector<int> unit_steps(int nseq, int H, int T) {
  const int n_tiles = (T + 127) / 128;
  const long long per = static_cast<long long>(nseq) * H;
  std::vector<int> w(static_cast<size_t>(n_tiles * per));
  for (size_t r = 0; r < w.size(); ++r) w[r] = n_tiles - static_cast<int>(r / per);
  return w;
}

// The schedule table for G CTAs (offsets [G + 1], then the units of each CTA
// in increasing index order, i.e. longest first), or an empty vector when the
// snake order is as good.  c_lo, c_hi: the range of per-unit overheads, in
// steps.
std::vector<int> pack_schedule(const std::vector<int>& w, int G, double c_lo, double c_hi) {
  const int n = static_cast<int>(w.size());
  if (G <= 1 || n <= G) return {};  // one unit per CTA at most: nothing to balance
  const double cs[3] = {c_lo, 0.5 * (c_lo + c_hi), c_hi};
  const Bins base = snake(n, G);
  const double base_v = worst_balance(base, w, cs);
  Bins best;
  double best_v = base_v;
  auto consider = [&](Bins&& b) {
    const double v = worst_balance(b, w, cs);
    if (v < best_v - 1e-9) {
      best_v = v;
      best = std::move(b);
    }
  };
  consider(round_robin_lpt(w, G));
  // First fit costs O(units x CTAs) per trial capacity; large lists balance
  // well enough by the deals above.
  if (static_cast<long long>(n) * G <= 4000000LL)
    for (double c : {0.5 * (c_lo + c_hi), c_hi, 2.0 * c_hi + 0.5}) consider(multifit(w, G, c));
  if (best.empty()) return {};
  std::vector<int> tab(static_cast<size_t>(G) + 1 + n);
  int at = 0;
  for (int c = 0; c < G; ++c) {
    std::sort(best[c].begin(), best[c].end());
    tab[c] = at;
    for (int i : best[c]) tab[G + 1 + at++] = i;
  }
  tab[G] = at;
  return tab;
}

}  // namespace ne
