"""Pins of the 8-bit block KV format oracle (oracle/kv_quant.py)."""
import numpy as np

import oracle
import oracle.dflash_oracle as od
from oracle import kv_quant as kq
from synth import TINY, make_weights_np, make_features_np


def _rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def test_exact_multiples_decode_exactly():
    """Blocks whose largest magnitude is 127 * 2^-e (a scale of 2^-e, exact in
    fp16) and whose values are integer multiples of the scale round-trip."""
    rng = _rng(1)
    for e in (0, 3, 7, 11):
        s = 2.0 ** -e
        codes = rng.integers(-127, 128, size=(5, 4, 64))
        codes[..., 0] = 127          # every block of 32 reaches the full range
        codes[..., 32] = -127
        x = codes * s
        np.testing.assert_array_equal(kq.roundtrip(x), x)


def test_decode_error_bound():
    """|x - decode(x)| <= d/2 + 127 |d - fp16(d)| per block, d = max|x|/127:
    half a quantisation step plus the scale's storage rounding."""
    rng = _rng(2)
    x = rng.standard_normal((50, 8, 128)) * rng.uniform(0.01, 100, size=(50, 8, 1))
    q, sc = kq.quantize(x)
    y = kq.dequantize(q, sc)
    blocks = x.reshape(50, 8, 4, 32)
    d = np.abs(blocks).max(axis=-1) / 127
    bound = d / 2 + 127 * np.abs(d - sc.astype(np.float64)) + 1e-12
    err = np.abs(blocks - y.reshape(50, 8, 4, 32)).max(axis=-1)
    assert np.all(err <= bound)
    assert np.all(np.abs(q.astype(int)) <= 127)
    # decoded values sit on the grid of the stored (fp16) scale
    grid = y.reshape(50, 8, 4, 32) / np.where(sc == 0, 1, sc.astype(np.float64))[..., None]
    np.testing.assert_array_equal(grid, np.round(grid))


def test_zero_blocks_and_symmetry():
    x = np.zeros((3, 64))
    x[1, 32:] = np.linspace(-1, 1, 32)
    q, sc = kq.quantize(x)
    assert np.all(q[0] == 0) and sc[0, 0] == 0 and np.all(kq.dequantize(q, sc)[0] == 0)
    assert np.all(q[1, :32] == 0)
    rng = _rng(3)
    z = rng.standard_normal((10, 96))
    np.testing.assert_array_equal(kq.quantize(-z)[0], -kq.quantize(z)[0])
    # halves round away from zero: 0.5 and 1.5 steps
    h = np.zeros((1, 32))
    h[0, 0], h[0, 1], h[0, 2] = 127.0, 0.5, -1.5
    np.testing.assert_array_equal(kq.quantize(h)[0][0, :3], [127, 1, -2])


def _ctx(seed, C):
    w = make_weights_np(TINY, seed=seed)
    orc = oracle.OracleDrafter(TINY, w)
    f = make_features_np(C, TINY.n_feat_layers * TINY.hidden, seed=seed + 1)
    orc.fuse_ctx([0], [C], f, pending=False)
    st = orc._state(0)
    return orc.w, [k[: st["len"]] for k in st["k"]], [v[: st["len"]] for v in st["v"]]


def test_pass_over_representable_context_is_the_plain_pass():
    w, kc, vc = _ctx(4, 48)
    # snap the context to the format: decoding again changes nothing
    kc2 = [kq.roundtrip(k) for k in kc]
    vc2 = [kq.roundtrip(v) for v in vc]
    np.testing.assert_array_equal(kq.roundtrip(kc2[0]), kc2[0])
    got = kq.draft_block_quantized_ctx(w, TINY, 11, kc2, vc2, 8)
    ref = od.draft_block(w, TINY, 11, kc2, vc2, 8)
    np.testing.assert_array_equal(got["hidden"], ref["hidden"])


def test_pass_with_quantized_context_stays_close():
    """Relative decode error is about 1/254 per value; over the tiny drafter
    the final residual stream moves by well under 2% of its row norm."""
    w, kc, vc = _ctx(5, 64)
    got = kq.draft_block_quantized_ctx(w, TINY, 12, kc, vc, 8)["hidden"]
    ref = od.draft_block(w, TINY, 12, kc, vc, 8)["hidden"]
    rel = np.linalg.norm(got - ref, axis=1) / np.linalg.norm(ref, axis=1)
    assert np.all(rel < 2e-2), rel.max()
    assert np.any(got != ref)
