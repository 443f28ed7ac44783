"""Pins of the two-tap convolution oracle (oracle/two_tap_conv.py): identity
kernels reproduce the plain drafter pass bit for bit, zero output kernels
leave the embedding rows, a pure shift kernel moves rows down by one, the
output at t depends on inputs t and t-1 only, and the correction's effect
scales linearly with U (a dropped or misplaced correction fails)."""
import numpy as np

import oracle
import oracle.dflash_oracle as od
from oracle import two_tap_conv as tc
from synth import TINY, make_weights_np, make_features_np


def _rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def _random_conv(rng, H, r, scale=0.1):
    return {"base": 1.0 + scale * rng.standard_normal((2, H)), "U": scale * rng.standard_normal((2, H, r)),
            "V": scale * rng.standard_normal((2, r, H)) / np.sqrt(H)}


def _setup(seed=3, C=40):
    w = make_weights_np(TINY, seed=seed)
    orc = oracle.OracleDrafter(TINY, w)
    f = make_features_np(C, TINY.n_feat_layers * TINY.hidden, seed=seed + 1)
    orc.fuse_ctx([0], [C], f, pending=False)
    st = orc._state(0)
    kc = [k[: st["len"]] for k in st["k"]]
    vc = [v[: st["len"]] for v in st["v"]]
    return orc.w, kc, vc


def test_identity_kernels_reproduce_the_plain_pass():
    w, kc, vc = _setup()
    H, r = TINY.hidden, 8
    convs = [{t: tc.identity_conv(H, r) for t in tc.TAPS} for _ in range(TINY.n_layers)]
    got = tc.draft_block_conv(w, TINY, convs, 17, kc, vc, 8)
    ref = od.draft_block(w, TINY, 17, kc, vc, 8)
    np.testing.assert_array_equal(got["hidden"], ref["hidden"])
    np.testing.assert_array_equal(got["draft"], ref["draft"])


def test_zero_output_kernels_leave_the_embedding():
    """With the output convolutions zero, every residual add adds zero: the
    final residual stream is the block's embedding rows."""
    w, kc, vc = _setup(seed=5)
    H, r = TINY.hidden, 8
    rng = _rng(6)
    zero = {"base": np.zeros((2, H)), "U": np.zeros((2, H, r)), "V": np.zeros((2, r, H))}
    convs = [{"ai": _random_conv(rng, H, r), "ao": zero, "fi": _random_conv(rng, H, r), "fo": zero}
             for _ in range(TINY.n_layers)]
    got = tc.draft_block_conv(w, TINY, convs, 9, kc, vc, 6)
    ids = np.array([9] + [TINY.mask_id] * 5)
    np.testing.assert_array_equal(got["hidden"], w["embed"][ids])


def test_shift_kernel_moves_rows_down():
    rng = _rng(7)
    x = rng.standard_normal((6, 16))
    shift = {"base": np.stack([np.zeros(16), np.ones(16)]), "U": np.zeros((2, 16, 3)), "V": np.zeros((2, 3, 16))}
    y = tc.conv2(x, shift)
    np.testing.assert_array_equal(y[0], np.zeros(16))     # the anchor has no predecessor
    np.testing.assert_array_equal(y[1:], x[:-1])


def test_output_depends_on_the_position_and_its_predecessor_only():
    rng = _rng(8)
    H, r, B = 32, 4, 7
    c = _random_conv(rng, H, r, scale=0.5)
    x = rng.standard_normal((B, H))
    y = tc.conv2(x, c)
    for s in range(B):
        x2 = x.copy()
        x2[s] += rng.standard_normal(H)
        y2 = tc.conv2(x2, c)
        changed = sorted(set(np.flatnonzero(np.any(y2 != y, axis=1)).tolist()))
        assert changed == [t for t in (s, s + 1) if t < B], (s, changed)


def test_correction_scales_with_U_and_is_absent_without_it():
    rng = _rng(9)
    H, r = 24, 5
    c = _random_conv(rng, H, r, scale=0.3)
    x = rng.standard_normal((5, H))
    plain = dict(c, U=np.zeros_like(c["U"]))
    y0 = tc.conv2(x, plain)
    # without a correction the convolution is linear in x
    np.testing.assert_allclose(tc.conv2(2.5 * x, plain), 2.5 * y0, rtol=1e-12)
    d1 = tc.conv2(x, c) - y0
    d3 = tc.conv2(x, dict(c, U=3.0 * c["U"])) - y0
    assert np.abs(d1).max() > 1e-3
    np.testing.assert_allclose(d3, 3.0 * d1, rtol=1e-10, atol=1e-12)


def test_tap0_only_kernel_is_pointwise():
    """With tap 1 off (zero base and correction), y_t = (base_0 + U_0 V_0 x_t) * x_t:
    each output depends on its own position only, so the coefficients come
    from the position's own input."""
    rng = _rng(10)
    H, r, B = 20, 4, 6
    c = _random_conv(rng, H, r, scale=0.5)
    c["base"][1] = 0.0
    c["U"][1] = 0.0
    x = rng.standard_normal((B, H))
    y = tc.conv2(x, c)
    for s in range(B):
        x2 = x.copy()
        x2[s] += rng.standard_normal(H)
        changed = np.flatnonzero(np.any(tc.conv2(x2, c) != y, axis=1)).tolist()
        assert changed == [s], (s, changed)
