// block_sched.cu - dynamic block-size scheduling (host logic, no device code).
//
// The DFlash notes' ablation ("DFlash - Block Diffusion for Flash Speculative
// Decoding", 6.5, block size) finds that a drafter trained at block 16 also
// serves block 8, which enables choosing the block size per cycle. The
// scheduler keeps, per draft position j, exponentially decayed counts of
// cycles that reached j (every earlier draft accepted) and that accepted it,
// read from each cycle's acceptance length tau (tau - 1 leading drafts
// accepted, notes 2.2). Each position's rate is shrunk toward the pooled
// rate of all positions, so positions a smaller block never reaches inherit
// it: with w = prior_a + prior_r,
//     pooled = (sum accepted + prior_a) / (sum reached + w),
//     a_j = (accepted_j + w * pooled) / (reached_j + w),
// and a block of B drafts is expected to yield
//     E[tau | B] = 1 + sum_{j=1}^{B-1} prod_{i<=j} a_i
// tokens, and among the sizes whose cycle cost T(B) is known the scheduler
// picks the largest E[tau | B] / T(B) (the smaller size on ties).
#include <algorithm>
#include <cmath>
#include <new>
#include <vector>

#include "dflash.h"
#include "internal.h"

struct dflash_block_sched {
  std::vector<int> sizes;        // ascending, distinct
  double decay, prior_a, prior_r;
  std::vector<double> reached;   // [max size - 1], index j - 1 for draft position j
  std::vector<double> accepted;
  std::vector<double> cost;      // [max size + 1] cycle cost per size, < 0 unknown
};

namespace {

double expected_tau(const dflash_block_sched* s, int B) {
  const double w = s->prior_a + s->prior_r;
  double sa = 0.0, sr = 0.0;
  for (size_t j = 0; j < s->reached.size(); ++j) {
    sa += s->accepted[j];
    sr += s->reached[j];
  }
  const double pooled = (sa + s->prior_a) / (sr + w);
  double e = 1.0, prod = 1.0;
  for (int j = 1; j < B; ++j) {
    prod *= (s->accepted[j - 1] + w * pooled) / (s->reached[j - 1] + w);
    e += prod;
  }
  return e;
}

}  // namespace

extern "C" {

dflash_status dflash_block_sched_create(const int32_t* sizes, int n_sizes, float decay, float prior_accept,
                                        float prior_reject, dflash_block_sched** out) {
  if (!out) return DFLASH_EINVAL;
  *out = nullptr;
  if (!sizes || n_sizes < 1 || n_sizes > dfl::kMaxBlock) return DFLASH_EINVAL;
  if (!(decay > 0.f && decay <= 1.f) || !(prior_accept > 0.f) || !(prior_reject > 0.f)) return DFLASH_EINVAL;
  std::vector<int> v(sizes, sizes + n_sizes);
  std::sort(v.begin(), v.end());
  for (size_t i = 0; i < v.size(); ++i)
    if (v[i] < 1 || v[i] > dfl::kMaxBlock || (i && v[i] == v[i - 1])) return DFLASH_EINVAL;
  dflash_block_sched* s = new (std::nothrow) dflash_block_sched();
  if (!s) return DFLASH_ENOMEM;
  s->sizes = v;
  s->decay = decay;
  s->prior_a = prior_accept;
  s->prior_r = prior_reject;
  s->reached.assign(std::max(1, v.back() - 1), 0.0);
  s->accepted.assign(std::max(1, v.back() - 1), 0.0);
  s->cost.assign(v.back() + 1, -1.0);
  *out = s;
  return DFLASH_OK;
}

dflash_status dflash_block_sched_destroy(dflash_block_sched* s) {
  if (!s) return DFLASH_EINVAL;
  delete s;
  return DFLASH_OK;
}

dflash_status dflash_block_sched_observe(dflash_block_sched* s, int B, const int32_t* taus, int n) {
  if (!s || B < 1 || B > s->sizes.back() || n < 0 || (n > 0 && !taus)) return DFLASH_EINVAL;
  for (int k = 0; k < n; ++k)
    if (taus[k] < 1 || taus[k] > B) return DFLASH_EINVAL;
  for (int k = 0; k < n; ++k) {
    for (size_t j = 0; j < s->reached.size(); ++j) {
      s->reached[j] *= s->decay;
      s->accepted[j] *= s->decay;
    }
    const int a = taus[k] - 1;   // leading drafts accepted
    for (int j = 1; j < B && j <= a + 1; ++j) {
      s->reached[j - 1] += 1.0;
      if (j <= a) s->accepted[j - 1] += 1.0;
    }
  }
  return DFLASH_OK;
}

dflash_status dflash_block_sched_set_cost(dflash_block_sched* s, int B, float cycle_ms) {
  if (!s || !(cycle_ms > 0.f) || std::find(s->sizes.begin(), s->sizes.end(), B) == s->sizes.end())
    return DFLASH_EINVAL;
  s->cost[B] = cycle_ms;
  return DFLASH_OK;
}

dflash_status dflash_block_sched_expected_tau(const dflash_block_sched* s, int B, double* out) {
  if (!s || !out || B < 1 || B > s->sizes.back()) return DFLASH_EINVAL;
  *out = expected_tau(s, B);
  return DFLASH_OK;
}

dflash_status dflash_block_sched_choose(const dflash_block_sched* s, int* B_out) {
  if (!s || !B_out) return DFLASH_EINVAL;
  int best = s->sizes.front();
  double best_rate = -1.0;
  for (int b : s->sizes) {
    if (s->cost[b] <= 0.0) continue;
    const double rate = expected_tau(s, b) / s->cost[b];
    if (rate > best_rate) {
      best = b;
      best_rate = rate;
    }
  }
  *B_out = best;
  return DFLASH_OK;
}

}  // extern "C"
