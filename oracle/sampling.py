"""CPU oracle of temperature sampling and lossless rejection-sampling verify.

TEST INFRASTRUCTURE. Only the tests, the smoke check and the bench's CPU
baseline leg may import this module. The CUDA library shares no code with it.

What it computes. The pages evaluate DFlash and DFlash 2 at temperature 1
with lossless rejection sampling ("DFlash - Block Diffusion for Flash
Speculative Decoding" notes, 6.2 "Sampling (Temperature = 1)" and the
"Lossless Guarantee"; "DFlash 2" notes, 7.2, run at temp 1.0, top-p 0.95,
top-k 20). They name the scheme but print no algorithm. Readings, the plainest
ones the rest supports:
  - a distribution over the vocabulary is the temperature softmax of the
    logits restricted to the top_k largest logits (largest first, lower id
    first among equal logits), then to the shortest prefix of that order whose
    probability mass reaches top_p, renormalised (temperature, then top-k,
    then top-p, as serving stacks apply them);
  - the drafter samples each masked position j from its own filtered
    distribution q_j, independently (one forward pass gives every q_j);
  - verify is standard speculative sampling: walking j = 0, 1, ..., draft x_j
    is accepted when u_j < min(1, p_j(x_j) / q_j(x_j)), p_j the target's
    filtered distribution after block position j; at the first rejection the
    token is drawn from max(0, p_j - q_j) renormalised; if every draft is
    accepted, the bonus token is drawn from p_{B-1};
  - a draw from a distribution (ids in filter order, probs) with a uniform
    u in [0, 1) takes the first entry whose cumulative probability exceeds u
    (for the residual, the cumulative residual exceeds u times its total);
  - tau = accepted + 1 and the bonus, as in greedy verify.
Random numbers are inputs (uniforms in [0, 1)), so the GPU path consumes the
same draws.

Pins (tests/test_sampling_pins.py): the verify's output distribution equals
p_j exactly (integrated over the draft and both uniforms on a tiny
vocabulary); top_k = 1 gives the argmax; no filter gives the plain softmax;
a worked top-p case; temperature scaling; the greedy limit reduces to the
greedy verify.
"""
from __future__ import annotations

from typing import List, Sequence, Tuple

import numpy as np

MAX_TOP_K = 32


def filtered_probs(logits: np.ndarray, temperature: float, top_k: int, top_p: float):
    """(ids, probs) of the filtered temperature softmax, in decreasing order."""
    logits = np.asarray(logits, dtype=np.float64)
    k = min(int(top_k), logits.shape[0])
    order = np.lexsort((np.arange(logits.shape[0]), -logits))[:k]
    z = (logits[order] - logits[order[0]]) / float(temperature)
    w = np.exp(z)
    w = w / w.sum()
    c = np.cumsum(w)
    n = int(np.searchsorted(c, top_p, side="left")) + 1   # first prefix whose mass reaches top_p
    n = min(n, k)
    p = w[:n] / w[:n].sum()
    return order[:n].astype(np.int64), p


def draw(ids: np.ndarray, probs: np.ndarray, u: float) -> int:
    """Inverse-CDF draw: the first entry whose cumulative probability exceeds u."""
    c = np.cumsum(probs)
    i = int(np.searchsorted(c, u * c[-1], side="right"))
    return int(ids[min(i, len(ids) - 1)])


def prob_of(ids: np.ndarray, probs: np.ndarray, x: int) -> float:
    hit = np.flatnonzero(np.asarray(ids) == int(x))
    return float(probs[hit[0]]) if hit.size else 0.0


def verify_sample(drafts: Sequence[int], q: List[Tuple[np.ndarray, np.ndarray]],
                  p: List[Tuple[np.ndarray, np.ndarray]], u_accept: Sequence[float],
                  u_resample: Sequence[float]):
    """Speculative-sampling verify of one block.

    drafts x_1..x_{B-1}; q[j] = (ids, probs) the drafter's filtered
    distribution the draft x_{j+1} was drawn from; p[j] the target's after
    block position j, j = 0..B-1; u_accept [B-1], u_resample [B].
    Returns (tau, token, accepted_ratio_list).
    """
    B = len(p)
    for j in range(B - 1):
        x = int(drafts[j])
        px = prob_of(*p[j], x)
        qx = prob_of(*q[j], x)
        if qx > 0 and u_accept[j] < min(1.0, px / qx):
            continue
        ids = p[j][0]
        r = np.array([max(0.0, pv - prob_of(*q[j], int(y))) for y, pv in zip(ids, p[j][1])])
        return j + 1, draw(ids, r, u_resample[j])
    return B, draw(*p[B - 1], u_resample[B - 1])


def draft_sample(logits_rows: np.ndarray, temperature: float, top_k: int, top_p: float, u: Sequence[float]):
    """Per masked position: (drawn id, filtered (ids, probs)) from the drafter's logits rows."""
    out = []
    for row, uu in zip(logits_rows, u):
        ids, pr = filtered_probs(row, temperature, top_k, top_p)
        out.append((draw(ids, pr, uu), (ids, pr)))
    return out
