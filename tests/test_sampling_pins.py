"""Pins of the sampling oracle (oracle/sampling.py) against facts that do not
come from the oracle itself: the losslessness of speculative sampling
(the verify's output law equals the target's distribution, integrated
exactly over the draft and both uniforms), closed forms of the filters, a
worked top-p case, and the greedy limit."""
import numpy as np
import pytest
from scipy.special import softmax

import oracle
from oracle import sampling as osm


def _rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def _output_law(q, p0, p1, grid=1000):
    """Law of the first emitted token of a B = 2 block: draft x ~ q, accept
    with u_a, else resample with u_r; if accepted the first token is x. Each
    uniform is integrated on a midpoint grid (exact up to 1/(2 grid) per
    probability boundary); the resample branch does not depend on u_a once
    the draft is rejected."""
    V = 1 + max(int(np.max(q[0])), int(np.max(p0[0])), int(np.max(p1[0])))
    law = np.zeros(V)
    us = (np.arange(grid) + 0.5) / grid
    for x, qx in zip(*q):
        acc = [osm.verify_sample([x], [q], [p0, p1], [ua], [0.5, 0.5])[0] == 2 for ua in us]
        f = float(np.mean(acc))
        law[int(x)] += qx * f
        if f < 1.0:
            ua_rej = us[acc.index(False)]
            for ur in us:
                tau, tok = osm.verify_sample([x], [q], [p0, p1], [ua_rej], [ur, 0.5])
                assert tau == 1
                law[tok] += qx * (1.0 - f) / grid
    return law


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_speculative_sampling_is_lossless(seed):
    """The first token's law equals p_0 whatever the drafter's q: the
    accept test and the residual exactly make up p_0 (the scheme's lossless
    property). Tiny vocabulary, supports that partly overlap."""
    rng = _rng(seed)
    V = 6
    lq = rng.standard_normal(V) * 1.5
    lp = rng.standard_normal(V) * 1.5
    q = osm.filtered_probs(lq, 1.0, 4, 1.0)      # drafter: top-4
    p0 = osm.filtered_probs(lp, 1.0, 5, 1.0)     # target: top-5
    p1 = osm.filtered_probs(lp[::-1].copy(), 1.0, 5, 1.0)
    law = _output_law(q, p0, p1)
    want = np.zeros(V)
    want[p0[0]] = p0[1]
    np.testing.assert_allclose(law, want, atol=3e-3)


def test_acceptance_rate_is_the_overlap():
    """Expected acceptance of one draft = sum_x min(p(x), q(x))."""
    rng = _rng(7)
    V = 8
    q = osm.filtered_probs(rng.standard_normal(V), 1.0, 8, 1.0)
    p0 = osm.filtered_probs(rng.standard_normal(V), 1.0, 8, 1.0)
    p1 = p0
    grid = 2000
    us = (np.arange(grid) + 0.5) / grid
    acc = 0.0
    for x, qx in zip(*q):
        acc += qx * np.mean([osm.verify_sample([x], [q], [p0, p1], [u], [0.5, 0.5])[0] == 2 for u in us])
    overlap = sum(min(osm.prob_of(*p0, v), osm.prob_of(*q, v)) for v in range(V))
    assert abs(acc - overlap) < 2e-3


def test_filters_closed_forms():
    rng = _rng(11)
    x = rng.standard_normal(50)
    ids, pr = osm.filtered_probs(x, 1.0, 1, 0.9)
    assert list(ids) == [int(np.argmax(x))] and pr[0] == 1.0
    ids, pr = osm.filtered_probs(x, 1.0, 50, 1.0)        # no filter: the plain softmax, sorted
    s = softmax(x)
    np.testing.assert_allclose(pr, s[ids], rtol=1e-12)
    assert list(ids) == list(np.argsort(-x, kind="stable"))
    # temperature T on logits c*x equals temperature T/c on x
    a = osm.filtered_probs(3.0 * x, 1.5, 20, 0.95)
    b = osm.filtered_probs(x, 0.5, 20, 0.95)
    assert list(a[0]) == list(b[0])
    np.testing.assert_allclose(a[1], b[1], rtol=1e-12)
    # top-k keeps the k largest, renormalised
    ids, pr = osm.filtered_probs(x, 1.0, 5, 1.0)
    top = np.argsort(-x, kind="stable")[:5]
    np.testing.assert_allclose(pr, softmax(x[top]), rtol=1e-12)


def test_top_p_worked_case():
    # probabilities 0.5, 0.3, 0.2 (logits ln p): top-p 0.75 keeps two (0.5 < 0.75 <= 0.8)
    lg = np.log(np.array([0.2, 0.5, 0.3]))
    ids, pr = osm.filtered_probs(lg, 1.0, 3, 0.75)
    assert list(ids) == [1, 2]
    np.testing.assert_allclose(pr, [0.625, 0.375], rtol=1e-12)
    # exactly reaching the mass keeps the token that reaches it (four equal
    # logits: probabilities 0.25 exactly, cumulative 0.5 after two)
    ids, pr = osm.filtered_probs(np.zeros(4), 1.0, 4, 0.5)
    assert list(ids) == [0, 1]
    np.testing.assert_array_equal(pr, [0.5, 0.5])
    ids, pr = osm.filtered_probs(lg, 1.0, 3, 0.5)
    assert list(ids) == [1]
    # ties: lower id first
    ids, _ = osm.filtered_probs(np.zeros(5), 1.0, 3, 1.0)
    assert list(ids) == [0, 1, 2]


def test_draw_inverse_cdf():
    ids = np.array([7, 3, 9])
    pr = np.array([0.5, 0.3, 0.2])
    assert osm.draw(ids, pr, 0.0) == 7
    assert osm.draw(ids, pr, 0.49) == 7
    assert osm.draw(ids, pr, 0.5) == 3     # cumulative 0.5 does not exceed 0.5
    assert osm.draw(ids, pr, 0.79) == 3
    assert osm.draw(ids, pr, 0.81) == 9
    assert osm.draw(ids, pr, 0.999999) == 9
    # unnormalised weights scale u by their total
    assert osm.draw(ids, 2 * pr, 0.6) == 3


def test_greedy_limit_is_greedy_verify():
    """top_k = 1 on both sides: p_j and q_j are point masses, so a draft is
    accepted exactly when it equals the target's argmax and the emitted token
    is the target's argmax: the greedy verify."""
    rng = _rng(13)
    V, B = 30, 6
    for _ in range(40):
        tl = rng.standard_normal((B, V))
        t = tl.argmax(axis=1)
        drafts = np.where(rng.random(B - 1) < 0.6, t[:-1], rng.integers(0, V, B - 1))
        p = [osm.filtered_probs(r, 1.0, 1, 1.0) for r in tl]
        q = [(np.array([d]), np.array([1.0])) for d in drafts]
        got = osm.verify_sample(drafts, q, p, rng.random(B - 1), rng.random(B))
        assert got == oracle.verify_block(drafts, t)
