"""CPU oracle of dynamic block-size scheduling.

TEST INFRASTRUCTURE. Only the tests may import this module. The library's
scheduler (csrc/block_sched.cu) shares no code with it.

What it computes. The DFlash notes' ablation ("DFlash - Block Diffusion for
Flash Speculative Decoding", 6.5 "Key Ablation Findings", block size) finds
that a drafter trained at block 16 generalises to block 8 at inference and
that this enables dynamic block-size scheduling; no policy is printed. The
reading taken, the plainest one the rest supports:
  - the acceptance length of a cycle with block B is tau = 1 + the number of
    leading drafts accepted (notes 2.2), so tau - 1 = a means positions
    1..a were accepted, position a + 1 (if a + 1 <= B - 1) was rejected and
    later positions were not reached;
  - per draft position j the scheduler keeps exponentially decayed counts of
    "reached" and "accepted" (every observation first multiplies the old
    counts by `decay`), and estimates the acceptance probability of position
    j given that every earlier draft was accepted by shrinking its own rate
    toward the pooled rate of all positions,
        pooled = (sum_j accepted_j + prior_a) / (sum_j reached_j + prior_a + prior_r),
        a_j = (accepted_j + w * pooled) / (reached_j + w),  w = prior_a + prior_r,
    so positions a smaller block never reaches inherit the pooled rate
    instead of the bare prior (a scheduler running block 8 at high
    acceptance can then see that block 16 pays);
  - the expected acceptance length of block B is
    E[tau | B] = 1 + sum_{j=1}^{B-1} prod_{i=1}^{j} a_i;
  - given the cycle cost T(B) of each allowed size (measured by the caller),
    it picks the size with the largest E[tau | B] / T(B), the smaller size on
    ties.
Pins (tests/test_block_sched_pins.py): with a constant acceptance a the
expectation is the geometric sum (1 - a^B) / (1 - a); the counts after a
hand-worked stream of observations; a worked choice.
"""
from __future__ import annotations

from typing import Dict, Sequence

import numpy as np


class BlockScheduler:
    def __init__(self, sizes: Sequence[int], decay: float = 0.99, prior_a: float = 1.0, prior_r: float = 1.0):
        self.sizes = sorted(int(b) for b in sizes)
        self.decay = float(decay)
        self.prior_a, self.prior_r = float(prior_a), float(prior_r)
        n = max(self.sizes)
        self.reached = np.zeros(n)    # index j - 1 for draft position j
        self.accepted = np.zeros(n)
        self.cost: Dict[int, float] = {}

    def observe(self, B: int, taus: Sequence[int]) -> None:
        for tau in taus:
            self.reached *= self.decay
            self.accepted *= self.decay
            a = int(tau) - 1
            for j in range(1, B):
                if j <= a:
                    self.reached[j - 1] += 1
                    self.accepted[j - 1] += 1
                elif j == a + 1:
                    self.reached[j - 1] += 1
                else:
                    break

    def acceptance(self) -> np.ndarray:
        w = self.prior_a + self.prior_r
        pooled = (self.accepted.sum() + self.prior_a) / (self.reached.sum() + w)
        return (self.accepted + w * pooled) / (self.reached + w)

    def expected_tau(self, B: int) -> float:
        a = self.acceptance()
        return 1.0 + float(np.sum(np.cumprod(a[: B - 1])))

    def set_cost(self, B: int, ms: float) -> None:
        self.cost[int(B)] = float(ms)

    def choose(self) -> int:
        best, best_rate = self.sizes[0], -1.0
        for b in self.sizes:
            if b not in self.cost:
                continue
            rate = self.expected_tau(b) / self.cost[b]
            if rate > best_rate:
                best, best_rate = b, rate
        return best
