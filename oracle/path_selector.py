"""CPU oracle of the DFlash 2 path selector.

TEST INFRASTRUCTURE. Only the tests, the smoke check and the bench's CPU
baseline leg may import this module. The CUDA library shares no code with it.

What it computes (DFlash 2 notes, "Problem 1: Selection Headroom" and
"Solution - Lightweight Path Selector"): the drafter keeps its top-16
candidate tokens at every masked position; each adjacent pair (predecessor a,
candidate b) gets the score

    S_t(a, b) = U_t(b) + < A(a) * H(h_t), B(b) >

(U_t the drafter's own logit of b at position t, A and B 256-dimensional
embeddings of the two tokens, H a context gate from the drafter's hidden
state at t, * elementwise), all pairs scored in parallel; a greedy walk over
the precomputed scores then picks one token per position.

Readings taken where the notes give the score but not the maps:
  - A(a) = W_A E[a] and B(b) = W_B E[b], linear maps of the drafter's token
    embedding E, and H(h_t) = W_H h~_t, a linear map of the final-normalised
    hidden state h~_t that the LM head reads; W_A, W_B, W_H are 256 x hidden
    (three such maps are the stated 2.0M parameters at hidden 2560);
  - the candidates C_t of masked position t are the 16 largest logits U_t
    (largest first, lower token id first among equal logits);
  - the predecessor of the first masked position is the anchor (the last
    verified token); every later position's predecessor is the walk's pick at
    the position before;
  - the walk picks argmax_b S_t(x_{t-1}, b); among equal scores the
    higher-ranked candidate (larger logit, then lower id).

Pins (tests/test_path_selector_pins.py): with W_H = 0 the walk returns the
plain greedy drafts; adding a constant to one position's logits leaves the
walk unchanged; one-hot embeddings give scores and a walk that can be worked
out by hand; top_k agrees with a brute-force sort.
"""
from __future__ import annotations

from typing import Dict, Sequence

import numpy as np

import oracle.dflash_oracle as od

K_SEL = 16     # candidates per masked position
D_SEL = 256    # width of the pair embeddings


def top_k(row: np.ndarray, k: int = K_SEL):
    """Indices of the k largest entries of a 1D array, largest first, the lower
    index first among equal values; returns (indices, values)."""
    row = np.asarray(row)
    order = np.lexsort((np.arange(row.shape[0]), -row))[:k]
    return order.astype(np.int64), row[order]


def pair_scores(u: np.ndarray, cand: np.ndarray, prev: Sequence[int], E: np.ndarray, w_a: np.ndarray,
                w_b: np.ndarray, h_gate: np.ndarray) -> np.ndarray:
    """S[i, j] = u[j] + <A(prev[i]) * h_gate, B(cand[j])> with A = W_A E, B = W_B E.

    u [k] logits of the candidates, cand [k] their ids, prev predecessor ids,
    h_gate [D] = H(h_t) = W_H h~_t.
    """
    a = E[np.asarray(prev, dtype=np.int64)] @ w_a.T       # [n_prev, D]
    b = E[np.asarray(cand, dtype=np.int64)] @ w_b.T       # [k, D]
    return u[None, :] + (a * h_gate[None, :]) @ b.T


def greedy_walk(anchor: int, cands: np.ndarray, u: np.ndarray, E: np.ndarray, w_a: np.ndarray, w_b: np.ndarray,
                h_gates: np.ndarray):
    """Walk the masked positions in order.

    cands [T, k], u [T, k] candidate ids and logits per position, h_gates
    [T, D]. Returns (ids [T], gap [T] = best minus second-best score, pick
    [T] = rank of the picked candidate).
    """
    prev = int(anchor)
    ids, gaps, picks = [], [], []
    for t in range(cands.shape[0]):
        s = pair_scores(u[t], cands[t], [prev], E, w_a, w_b, h_gates[t])[0]
        j = int(np.argmax(s))    # first maximum: the higher-ranked candidate on ties
        srt = np.sort(s)[::-1]
        ids.append(int(cands[t, j]))
        gaps.append(float(srt[0] - srt[1]) if s.shape[0] > 1 else np.inf)
        picks.append(j)
        prev = int(cands[t, j])
    return np.array(ids, dtype=np.int64), np.array(gaps), np.array(picks, dtype=np.int64)


def select_block(weights, shape, sel: Dict[str, np.ndarray], anchor: int, k_ctx, v_ctx, B: int):
    """One drafter pass (as dflash_oracle.draft_block) followed by the path
    selector. sel holds w_a, w_b, w_h, each [D_SEL, H]."""
    base = od.draft_block(weights, shape, anchor, k_ctx, v_ctx, B)
    hf = od.rms_norm(base["hidden"], weights["g_final"], shape.rms_eps)[1:]   # h~_t of the masked positions
    logits = hf @ weights["lm_head"].T
    T = B - 1
    cands = np.zeros((T, K_SEL), dtype=np.int64)
    u = np.zeros((T, K_SEL))
    gap16 = np.zeros(T)
    for t in range(T):
        cands[t], u[t] = top_k(logits[t])
        srt = np.sort(logits[t])[::-1]
        gap16[t] = srt[K_SEL - 1] - srt[K_SEL] if logits.shape[1] > K_SEL else np.inf
    h_gates = hf @ sel["w_h"].T
    ids, gaps, picks = greedy_walk(anchor, cands, u, weights["embed"], sel["w_a"], sel["w_b"], h_gates)
    return {"draft": ids, "gap": gaps, "pick": picks, "cand": cands, "u": u, "gap16": gap16,
            "h_gate": h_gates, "logits": logits, "plain_draft": base["draft"], "hidden": base["hidden"]}


def drafter_select(orc, seq_ids, anchors, B: int, sel: Dict[str, np.ndarray]):
    """select_block for every sequence against an OracleDrafter's cache."""
    dt = orc.w["embed"].dtype
    s_w = {k: np.asarray(v, dtype=dt) for k, v in sel.items()}
    out = []
    for s, a in zip(seq_ids, anchors):
        st = orc._state(int(s))
        kc = [k[: st["len"]] for k in st["k"]]
        vc = [v[: st["len"]] for v in st["v"]]
        out.append(select_block(orc.w, orc.shape, s_w, int(a), kc, vc, B))
    return out
