"""Pins of the path-selector oracle (DFlash 2 notes, "Solution - Lightweight
Path Selector"): special cases that reduce it to the plain greedy drafter,
an invariance of the score, a walk worked out by hand with one-hot
embeddings, and top_k against a brute-force sort."""
import numpy as np
import pytest

import oracle
from oracle import path_selector as ps
from synth import TINY, make_weights_np, make_features_np, make_anchor_ids_np


def _sel(sh, seed, scale=0.05):
    rng = np.random.Generator(np.random.PCG64(seed))
    return {k: rng.standard_normal((ps.D_SEL, sh.hidden)) * scale for k in ("w_a", "w_b", "w_h")}


def test_top_k_matches_brute_force_with_ties():
    rng = np.random.Generator(np.random.PCG64(3))
    for _ in range(50):
        row = np.round(rng.standard_normal(40) * 2)   # many exact ties
        idx, val = ps.top_k(row, 16)
        brute = sorted(range(40), key=lambda i: (-row[i], i))[:16]
        assert list(idx) == brute
        np.testing.assert_array_equal(val, row[brute])


def _tiny_orc(seed=5):
    sh = TINY
    wn = make_weights_np(sh, seed=seed, gamma="jitter", std=0.05)
    orc = oracle.OracleDrafter(sh, wn)
    width = sh.n_feat_layers * sh.hidden
    orc.fuse_ctx([0, 1], [40, 7], make_features_np(47, width, seed=seed + 1), pending=False)
    return sh, wn, orc


def test_zero_gate_reduces_to_greedy_drafts():
    """H = 0 removes the pair term: S_t(a, b) = U_t(b), so the walk takes every
    position's top candidate, the plain drafter's argmax."""
    sh, wn, orc = _tiny_orc()
    sel = _sel(sh, 7)
    sel["w_h"] = np.zeros_like(sel["w_h"])
    anchors = make_anchor_ids_np(2, sh.vocab, seed=9)
    for r in ps.drafter_select(orc, [0, 1], anchors, 8, sel):
        np.testing.assert_array_equal(r["draft"], r["plain_draft"])
        np.testing.assert_array_equal(r["pick"], np.zeros(7, dtype=np.int64))


def test_constant_logit_shift_leaves_walk_unchanged():
    """Adding c to every candidate logit of one position adds c to every score
    of that position, so no choice changes."""
    rng = np.random.Generator(np.random.PCG64(11))
    V, T, H = 300, 6, 32
    E = rng.standard_normal((V, H))
    w = {k: rng.standard_normal((ps.D_SEL, H)) for k in ("w_a", "w_b")}
    gates = rng.standard_normal((T, ps.D_SEL))
    cands = np.stack([rng.choice(V, 16, replace=False) for _ in range(T)])
    u = rng.standard_normal((T, 16))
    ids, _, _ = ps.greedy_walk(5, cands, u, E, w["w_a"], w["w_b"], gates)
    u2 = u.copy()
    u2[3] += 17.0
    ids2, _, _ = ps.greedy_walk(5, cands, u2, E, w["w_a"], w["w_b"], gates)
    np.testing.assert_array_equal(ids, ids2)


def test_one_hot_walk_worked_by_hand():
    """Embeddings e_i = one-hot(i) in 256 dims, W_A = W_B = I (first 256
    columns), gate = g * ones: <A(a) * H, B(b)> = g if a == b else 0.
    Candidates [[7, 3], [9, 3], [9, 3]] (padded with tokens far below),
    logits [[1, 0.9], [1, 0.95], [1, 0.99]]:
      anchor 3, g = 0.05: t0 7 (1 > 0.95), t1 after 7: 9 (1 > 0.95), t2 after
        9: 9 (1.05 > 0.99)                                  -> 7, 9, 9;
      anchor 3, g = 0.2: t0 3 (1.1 > 1), t1 after 3: 3 (1.15 > 1), t2 after
        3: 3 (1.19 > 1)                                     -> 3, 3, 3;
      anchor 7, g = 0.2: t0 7 (1.2 > 0.9), t1 after 7: 9 (1 > 0.95) - the
        choice at t1 differs from the walk above only through t0's pick -
        t2 after 9: 9 (1.2 > 0.99)                          -> 7, 9, 9."""
    V = ps.D_SEL
    E = np.eye(V)
    I = np.eye(ps.D_SEL, V)
    pad = [200 + j for j in range(14)]
    cands = np.array([[7, 3] + pad, [9, 3] + pad, [9, 3] + pad])
    u = np.array([[1.0, 0.9] + [-100.0] * 14, [1.0, 0.95] + [-100.0] * 14, [1.0, 0.99] + [-100.0] * 14])

    def walk(anchor, g):
        gates = np.full((3, ps.D_SEL), g)
        return list(ps.greedy_walk(anchor, cands, u, E, I, I, gates)[0])

    assert walk(3, 0.05) == [7, 9, 9]
    assert walk(3, 0.2) == [3, 3, 3]
    assert walk(7, 0.2) == [7, 9, 9]
    # and the score itself: S_0(3, 3) = 0.9 + g
    s = ps.pair_scores(u[0], cands[0], [3, 7], E, I, I, np.full(ps.D_SEL, 0.2))
    assert s[0, 1] == pytest.approx(1.1)
    assert s[0, 0] == pytest.approx(1.0)
    assert s[1, 0] == pytest.approx(1.2)


def test_asymmetric_maps_and_position_gates_worked_by_hand():
    """W_A = I, W_B a permutation P (B(b) = e_{P(b)}), so the pair term is g_t
    when a == P(b): the maps enter in their roles, not symmetrically. P is the
    3-cycle 3 -> 5 -> 4 -> 3 (P(4) = 3, P(3) = 5, P(5) = 4) and swaps 8 <-> 9,
    so a == P(b) and P(a) == b differ. Candidates [[7, 4], [8, 4], [8, 4]], logits
    [[1, 0.9], [1, 0.95], [1, 0.99]], gates g = (0.2, 0.05, 0.05):
      t0 after anchor 3: B(4) = e_3 matches A(3): 0.9 + 0.2 = 1.1 > 1 -> 4;
      t1 after 4: P(8) = 9 != 4, P(4) = 3 != 4: 1 > 0.95           -> 8;
      t2 after 8: P(8) = 9 != 8, P(4) = 3 != 8: 1 > 0.99           -> 8.
    With the gates of t0 and t1 exchanged (0.05, 0.2, 0.05): t0 after 3:
    0.95 < 1 -> 7; t1 after 7: no match -> 8; t2 after 8 -> 8. A third case
    makes the gate of t1 decide."""
    V = ps.D_SEL
    E = np.eye(V)
    I = np.eye(ps.D_SEL, V)
    perm = np.arange(V)
    perm[[3, 4, 5, 8, 9]] = [5, 3, 4, 9, 8]
    wb = np.eye(ps.D_SEL, V)[perm].T.copy()   # B(b) = W_B e_b = e_{perm[b]}
    assert np.array_equal(wb @ E[4], E[3][: ps.D_SEL]) and np.array_equal(wb @ E[8], E[9][: ps.D_SEL])
    pad = [200 + j for j in range(14)]
    cands = np.array([[7, 4] + pad, [8, 4] + pad, [8, 4] + pad])
    u = np.array([[1.0, 0.9] + [-100.0] * 14, [1.0, 0.95] + [-100.0] * 14, [1.0, 0.99] + [-100.0] * 14])

    def walk(gs):
        gates = np.stack([np.full(ps.D_SEL, g) for g in gs])
        return list(ps.greedy_walk(3, cands, u, E, I, wb, gates)[0])

    assert walk((0.2, 0.05, 0.05)) == [4, 8, 8]
    assert walk((0.05, 0.2, 0.05)) == [7, 8, 8]
    # the gate of position t, not t-1: candidates [[7, 4], [8, 5], [8, 4]],
    # logits [[1, 0.9], [1, 0.97], [1, 0.99]], gates (0.2, 0.01, 0.3):
    # t0 after 3 -> 4 (1.1); t1 after 4: P(5) = 4 matches, 0.97 + 0.01 < 1
    # -> 8 (with t0's gate it would be 1.17 -> 5); t2 after 8: no match -> 8
    cands3 = np.array([[7, 4] + pad, [8, 5] + pad, [8, 4] + pad])
    u3 = np.array([[1.0, 0.9] + [-100.0] * 14, [1.0, 0.97] + [-100.0] * 14, [1.0, 0.99] + [-100.0] * 14])
    gates3 = np.stack([np.full(ps.D_SEL, g) for g in (0.2, 0.01, 0.3)])
    assert list(ps.greedy_walk(3, cands3, u3, E, I, wb, gates3)[0]) == [4, 8, 8]
