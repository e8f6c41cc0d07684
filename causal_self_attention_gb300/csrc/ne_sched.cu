// ne_sched.cu -- work dealing of the persistent attention kernels: the
// backward's schedule packed on the host for a fixed-length batch, and the
// compaction of a packed batch's work lists on the device.
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

#include "ne_sm100.cuh"

namespace ne {

// ---------------------------------------------------------------------------
// Packed (variable-length) batches: the work lists of both persistent kernels
// enumerate every (block, sequence, head), and a sequence shorter than the
// longest has no items for the higher blocks.  Dealt with those holes, the
// snake order left the busiest forward CTA at 1.6 times the mean work on a
// batch of lengths 64..2048; without the holes but in block order, the
// backward's units (whose length also depends on their sequence's length)
// were worse still.  The lengths are on the device, so one CTA builds the
// list there before the kernel runs: the items that are not empty, sorted by
// their number of steps, longest first (a counting sort: steps are small
// integers), which the kernel then deals in the snake order.  out[0] = the
// number of items, out[1 ..] their indices; items of equal length in no fixed
// order (every item is computed the same way by whichever CTA gets it).
// Items of a sequence whose bounds are invalid are kept, last, so that the
// kernel reports them as before.
//   kind 0: forward items, r -> block n_blocks - 1 - r / (nseq H) (pairs of
//           128-row query tiles), steps = key tiles of its last query tile;
//   kind 1: backward units, r -> key tile r / (nseq H), steps = query tiles
//           from it to the end of its sequence.
// Bucket b of the sort holds the items of b steps; bucket 0 the kept items of
// invalid sequences; -1 marks an empty item.
// ---------------------------------------------------------------------------
__device__ __forceinline__ int item_bucket(const Problem& pb, int kind, int n_blocks, int r) {
  const int per = pb.nseq * pb.H;
  const int blk = r / per;
  const int seq = (r - blk * per) / pb.H;
  int start, len;
  if (!seq_bounds(pb, seq, start, len, nullptr)) return 0;
  if (kind == 0) {
    const int b = n_blocks - 1 - blk;  // the item's block of two query tiles
    if (2 * b * kBM >= len) return -1;
    return (2 * b + 1) * kBM < len ? 2 * b + 2 : 2 * b + 1;
  }
  if (blk * kBM >= len) return -1;
  return (len + kBM - 1) / kBM - blk;
}

// Add 1 to ctr[key] for every active lane, one atomic per distinct key in the
// warp; returns this lane's slot among the lanes that added (old value + rank).
__device__ __forceinline__ int warp_counted_add(int* ctr, int key, bool active) {
  const unsigned act = __ballot_sync(0xffffffffu, active);
  if (!active) return 0;
  const int lane = threadIdx.x & 31;
  const unsigned peers = __match_any_sync(act, key);
  const int leader = __ffs(peers) - 1;
  int base = 0;
  if (lane == leader) base = atomicAdd(ctr + key, __popc(peers));
  base = __shfl_sync(peers, base, leader);
  return base + __popc(peers & ((1u << lane) - 1u));
}

__global__ void __launch_bounds__(1024)
    ne_compact_items_kernel(const Problem pb, int kind, int n_blocks, int n_buckets,
                            int* __restrict__ out) {
  pdl_wait();  // cu_seqlens may come from the kernel before
  extern __shared__ int bucket[];  // counts, then the next free slot of each bucket
  const int n = n_blocks * pb.nseq * pb.H;
  for (int b = threadIdx.x; b < n_buckets; b += blockDim.x) bucket[b] = 0;
  __syncthreads();
  for (int r0 = 0; r0 < n; r0 += blockDim.x) {
    const int r = r0 + threadIdx.x;
    const int b = r < n ? item_bucket(pb, kind, n_blocks, r) : -1;
    warp_counted_add(bucket, b < 0 ? 0 : b, b >= 0);
  }
  __syncthreads();
  if (threadIdx.x == 0) {  // first slots: the most steps first, bucket 0 last
    int at = 0;
    for (int b = n_buckets - 1; b >= 1; --b) {
      const int c = bucket[b];
      bucket[b] = at;
      at += c;
    }
    const int c0 = bucket[0];
    bucket[0] = at;
    out[0] = at + c0;
  }
  __syncthreads();
  for (int r0 = 0; r0 < n; r0 += blockDim.x) {
    const int r = r0 + threadIdx.x;
    const int b = r < n ? item_bucket(pb, kind, n_blocks, r) : -1;
    const int slot = warp_counted_add(bucket, b < 0 ? 0 : b, b >= 0);
    if (b >= 0) out[1 + slot] = r;
  }
  pdl_launch_dependents();
}

// n_buckets: the largest number of steps an item can have, plus one.
cudaError_t launch_compact_items(const Problem& pb, int kind, int n_blocks, int n_buckets,
                                 int* out, cudaStream_t stream) {
  return launch_pdl(ne_compact_items_kernel, dim3(1), dim3(1024),
                    static_cast<size_t>(n_buckets) * sizeof(int), stream, pb, kind, n_blocks,
                    n_buckets, out);
}

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
