"""Dynamic block-size scheduling: the oracle (oracle/block_sched.py) pinned to
closed forms and hand-worked counts, and the library's host scheduler
(dflash_block_sched_*, no GPU involved) against the oracle."""
import numpy as np
import pytest

from oracle.block_sched import BlockScheduler as OracleSched


def test_constant_acceptance_gives_the_geometric_sum():
    """With every a_j equal to a, E[tau | B] = sum_{j<B} a^j = (1 - a^B) / (1 - a)
    (no data: every position takes the pooled prior rate 3/4)."""
    s = OracleSched([4, 8, 16, 32], decay=1.0, prior_a=3.0, prior_r=1.0)   # no data: a = 3/4 everywhere
    for B in (1, 4, 8, 16, 32):
        a = 0.75
        assert abs(s.expected_tau(B) - (1 - a ** B) / (1 - a)) < 1e-12


def test_counts_after_worked_observations():
    s = OracleSched([8], decay=1.0, prior_a=1.0, prior_r=1.0)
    s.observe(8, [3, 1, 8])
    # tau 3: positions 1, 2 accepted, 3 rejected; tau 1: position 1 rejected; tau 8: 1..7 accepted
    np.testing.assert_array_equal(s.reached[:7], [3, 2, 2, 1, 1, 1, 1])
    np.testing.assert_array_equal(s.accepted[:7], [2, 2, 1, 1, 1, 1, 1])
    # pooled rate (9 + 1) / (11 + 2) = 10/13, w = 2: a_1 = (2 + 20/13) / 5,
    # a_3 = (1 + 20/13) / 4, and the never-reached position 8 gets 10/13
    a = s.acceptance()
    assert abs(a[0] - 46 / 65) < 1e-12 and abs(a[2] - 33 / 52) < 1e-12
    s16 = OracleSched([16], decay=1.0, prior_a=1.0, prior_r=1.0)
    s16.observe(8, [3, 1, 8])
    assert abs(s16.acceptance()[8] - 10 / 13) < 1e-12
    # decay multiplies the old counts before each observation
    t = OracleSched([4], decay=0.5, prior_a=1.0, prior_r=1.0)
    t.observe(4, [4, 1])
    np.testing.assert_allclose(t.reached[:3], [0.5 + 1, 0.5, 0.5])
    np.testing.assert_allclose(t.accepted[:3], [0.5, 0.5, 0.5])


def test_worked_choice():
    """High acceptance favours the long block, low acceptance the short one,
    at costs 1.0 (B = 8) and 1.3 (B = 16)."""
    hi = OracleSched([8, 16], decay=1.0)
    hi.observe(16, [16] * 50)
    lo = OracleSched([8, 16], decay=1.0)
    lo.observe(16, [2] * 50)
    for s in (hi, lo):
        s.set_cost(8, 1.0)
        s.set_cost(16, 1.3)
    assert hi.expected_tau(16) / 1.3 > hi.expected_tau(8) / 1.0 and hi.choose() == 16
    assert lo.choose() == 8
    # no cost known: the smallest size
    assert OracleSched([8, 16]).choose() == 8


@pytest.fixture(scope="module")
def dfl():
    import __graft_entry__
    __graft_entry__.build()
    import block_diffusion_drafter_pass_gb300 as m
    return m


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_library_scheduler_matches_oracle(dfl, seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    sizes = [4, 8, 16, 32]
    lib = dfl.BlockScheduler(sizes, decay=0.97, prior_accept=1.0, prior_reject=1.0)
    orc = OracleSched(sizes, decay=0.97, prior_a=1.0, prior_r=1.0)
    costs = {4: 0.55, 8: 0.6, 16: 0.7, 32: 0.95}
    for b, c in costs.items():
        lib.set_cost(b, c)
        orc.set_cost(b, c)
    for cycle in range(200):
        B = int(rng.choice(sizes))
        p = 0.6 + 0.35 * np.sin(cycle / 25.0)   # a drifting acceptance rate
        taus = [1 + int(np.sum(np.cumprod(rng.random(B - 1) < p))) for _ in range(int(rng.integers(1, 5)))]
        lib.observe(B, taus)
        orc.observe(B, taus)
        for b in sizes:
            assert abs(lib.expected_tau(b) - orc.expected_tau(b)) < 1e-6 * orc.expected_tau(b)
        rates = sorted(orc.expected_tau(b) / costs[b] for b in sizes)
        if rates[-1] - rates[-2] > 1e-6 * rates[-1]:
            assert lib.choose() == orc.choose()
    lib.close()


def test_library_scheduler_rejects_bad_arguments(dfl):
    with pytest.raises(dfl.DFlashError):
        dfl.BlockScheduler([8, 8])
    with pytest.raises(dfl.DFlashError):
        dfl.BlockScheduler([0, 8])
    with pytest.raises(dfl.DFlashError):
        dfl.BlockScheduler([8], decay=0.0)
    s = dfl.BlockScheduler([8, 16])
    with pytest.raises(dfl.DFlashError):
        s.observe(8, [9])      # tau above B
    with pytest.raises(dfl.DFlashError):
        s.set_cost(12, 1.0)    # not one of the sizes
    s.close()


def test_scheduler_converges_to_the_best_block():
    """I.i.d. acceptance p = 0.85 per draft and cycle costs 0.5 + 0.01 B ms:
    E[tau | B] / T(B) = (1 - p^B) / (1 - p) / T(B) peaks at B = 16 among
    4, 8, 16, 32. Starting from whatever the empty scheduler picks, choosing
    and observing 400 cycles must settle on 16 (positions beyond the running
    block inherit the pooled rate, so growing the block can pay off)."""
    p, sizes = 0.85, [4, 8, 16, 32]
    cost = {b: 0.5 + 0.01 * b for b in sizes}
    rate = {b: (1 - p ** b) / (1 - p) / cost[b] for b in sizes}
    assert max(rate, key=rate.get) == 16
    rng = np.random.Generator(np.random.PCG64(9))
    s = OracleSched(sizes, decay=0.99)
    for b in sizes:
        s.set_cost(b, cost[b])
    picks = []
    for _ in range(400):
        b = s.choose()
        picks.append(b)
        tau = 1 + int(np.sum(np.cumprod(rng.random(b - 1) < p)))
        s.observe(b, [tau])
    assert all(b == 16 for b in picks[-100:])


def test_library_scheduler_converges_too(dfl):
    """The library's host scheduler in the same loop: low acceptance (0.3)
    settles on the shortest block, high acceptance (0.85) on 16."""
    sizes = [4, 8, 16, 32]
    cost = {b: 0.5 + 0.01 * b for b in sizes}
    for p, want in ((0.3, 4), (0.85, 16)):
        rate = {b: (1 - p ** b) / (1 - p) / cost[b] for b in sizes}
        assert max(rate, key=rate.get) == want
        rng = np.random.Generator(np.random.PCG64(int(p * 100)))
        s = dfl.BlockScheduler(sizes, decay=0.99)
        for b in sizes:
            s.set_cost(b, cost[b])
        picks = []
        for _ in range(400):
            b = s.choose()
            picks.append(b)
            s.observe(b, [1 + int(np.sum(np.cumprod(rng.random(b - 1) < p)))])
        s.close()
        assert all(b == want for b in picks[-100:]), (p, picks[-20:])
