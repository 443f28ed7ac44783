"""The top-K selection scheme of the library's top-K pass (csrc/topk.cuh),
restated in numpy and checked against a brute-force top-K on adversarial rows.

This checks the design, not the CUDA code: that the per-slice lower bound
(the smallest over 8 warps of each warp's (K/8)-th largest lane maximum) never
excludes a true top-K key, that the bounded tie rounds always end with the
exact top-K, and that the merge bound over slice lists (the larger of the
slices' largest K-th key and the smallest c-th key, c = ceil(K / slices))
keeps every true top-K key. Keys order (value, column): larger value first,
lower column first among equal values; NaN never counts.
"""
import numpy as np
import pytest

THREADS, WARP, CAP = 256, 32, 4096


def _keys(vals, cols):
    """Sortable keys: (value, -column) as a structured order via a tuple list."""
    return [(float(v), -int(c)) for v, c in zip(vals, cols) if v == v]


def _brute_topk(row, K):
    order = sorted(_keys(row, np.arange(len(row))), reverse=True)
    return [-c for _, c in order[:K]]


def _slice_topk(row, c0, c1, K, per=32):
    """One CTA: thread t holds per values laid out as the kernel's loads
    (4-wide fp32 loads: column c0 + 4 (t + 256 u) + e)."""
    R = K // 8
    lane_max = np.full(THREADS, -np.inf)
    cols_of = np.zeros((THREADS, per), dtype=np.int64)
    for t in range(THREADS):
        for q in range(per):
            c = c0 + 4 * (t + THREADS * (q // 4)) + q % 4
            cols_of[t, q] = c
            if c < c1 and row[c] == row[c]:
                lane_max[t] = max(lane_max[t], row[c])
    # the warp's R-th largest lane maximum (ties broken by lane), smallest over warps
    rth = []
    for w in range(THREADS // WARP):
        lm = lane_max[w * WARP:(w + 1) * WARP]
        rth.append(np.sort(lm)[::-1][R - 1])
    bound = min(rth)
    thr = (bound, -np.inf)                  # keys at or above: values at or above the bound
    valid = [(c, row[c]) for t in range(THREADS) for c in cols_of[t] if c < c1 and row[c] == row[c]]
    rounds = 0
    while True:
        cand = [(v, -c) for c, v in valid if (v, -c) >= thr]
        if len(cand) <= CAP:
            break
        buf = cand[:CAP]                    # whichever keys won the slots
        kth = sorted(buf, reverse=True)[K - 1]
        assert kth > thr
        thr = kth
        rounds += 1
        assert rounds < 64
    top = sorted(cand, reverse=True)[:K]
    return top, rounds


def _merge(lists, K):
    S = len(lists)
    c = (K + S - 1) // S
    pad = lambda L, i: L[i] if i < len(L) else (-np.inf, -np.inf)
    t1 = max(pad(L, K - 1) for L in lists)
    t2 = min(pad(L, c - 1) for L in lists)
    t = max(t1, t2)
    kept = [k for L in lists for k in L if k >= t]
    return [-col for _, col in sorted(kept, reverse=True)[:K]]


def _select(row, K, slice_cols=8192):
    lists, rounds = [], 0
    for c0 in range(0, len(row), slice_cols):
        top, r = _slice_topk(row, c0, min(len(row), c0 + slice_cols), K)
        lists.append(top)
        rounds += r
    return _merge(lists, K), rounds


def _rows():
    rng = np.random.Generator(np.random.PCG64(0))
    V = 20000
    out = {
        "normal": rng.standard_normal(V).astype(np.float32),
        "ascending": np.linspace(-3, 3, V).astype(np.float32),
        "descending": np.linspace(3, -3, V).astype(np.float32),
        "equal": np.zeros(V, dtype=np.float32),
        "three_levels": rng.integers(0, 3, V).astype(np.float32),
        "spikes_in_one_lane": np.full(V, -1.0, dtype=np.float32),
        "periodic": np.tile(np.arange(64, dtype=np.float32), V // 64 + 1)[:V],
    }
    sp = out["spikes_in_one_lane"]
    sp[[4 * 7 + 1024 * u for u in range(8)]] = 5.0      # every value of one thread is large
    nan = rng.standard_normal(V).astype(np.float32)
    nan[rng.integers(0, V, 500)] = np.nan
    out["with_nan"] = nan
    return out


@pytest.mark.parametrize("name", sorted(_rows()))
@pytest.mark.parametrize("K", [16, 32])
def test_scheme_returns_the_exact_top_k(name, K):
    row = _rows()[name]
    got, rounds = _select(row, K)
    assert got == _brute_topk(row, K), name
    if name == "equal":
        assert rounds > 0            # the tie rounds ran


@pytest.mark.parametrize("K", [16, 32])
def test_scheme_over_many_slices(K):
    """Vocabulary 300000: 37 slice lists merged under the merge bound."""
    rng = np.random.Generator(np.random.PCG64(K))
    row = (rng.standard_normal(300000) * 3).astype(np.float32)
    row[rng.integers(0, 300000, 40)] = 9.0       # ties at the very top, spread over slices
    got, _ = _select(row, K)
    assert got == _brute_topk(row, K)
