"""Temperature sampling and the speculative-sampling verify on the GPU against
oracle/sampling.py, through the C ABI.

- dflash_sample_filter on bf16 target logits: the oracle filters the very same
  values, so the lists must agree id for id (ties included: bf16 logits tie
  often) and the probabilities within fp32 rounding; the kept count may
  differ only where the cumulative mass sits within 1e-5 of top_p, a draw only
  where the uniform sits within 1e-5 of a cumulative boundary.
- dflash_draft_sample: the drafter's logits differ from the oracle's within the
  logit tolerance, so its lists are checked for validity (distinct ids,
  decreasing probabilities summing to 1, ids a top-k of the oracle's logits
  within the tolerance) and for the oracle's probabilities within what that
  tolerance allows; each draw must be the list entry the uniform selects.
- dflash_verify_sample on lists built on the host: tau and the emitted token
  equal the oracle's except within 1e-5 of an acceptance or draw boundary,
  and the committed lengths advance by min(tau, pending). With top_k = 1 on
  both sides it is the greedy verify.
"""
import numpy as np
import pytest

import oracle
from oracle import sampling as osm
from synth import TINY, make_weights_np, make_features_np, make_anchor_ids_np, make_target_logits_bf16_np, bits_to_f32
from tests.gpu_util import np_weights_to_device, bf16_dev, i32_dev, ATOL, RTOL

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
DEV = "cuda:0"
EPS = 1e-5


@pytest.fixture(scope="module")
def dfl():
    import __graft_entry__
    __graft_entry__.build()
    import block_diffusion_drafter_pass_gb300 as m
    return m


def _drafter(dfl, max_batch=64, max_block=16, seed=3):
    wn = make_weights_np(TINY, seed=seed)
    d = dfl.Drafter(TINY, np_weights_to_device(wn, DEV), max_seqs=max_batch, max_batch=max_batch,
                    max_block=max_block, max_ctx=512, max_fuse_tokens=8192)
    return d, wn


def _f32_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(DEV)


def _check_filter_rows(ids, probs, drawn, vals, us, temperature, top_k, top_p, what):
    ambiguous = 0
    for r in range(vals.shape[0]):
        oi, op = osm.filtered_probs(vals[r], temperature, top_k, top_p)
        n_g = int((ids[r] >= 0).sum())
        assert np.all(ids[r][n_g:] == -1) and np.all(probs[r][n_g:] == 0), f"{what} row {r}: padding"
        # the unfiltered top-k masses decide the kept count
        full_i, full_p = osm.filtered_probs(vals[r], temperature, top_k, 1.0)
        cum = np.cumsum(full_p)
        near = np.any(np.abs(cum[:-1] - top_p) < EPS)
        if n_g != len(oi):
            assert near, f"{what} row {r}: kept {n_g} vs {len(oi)}"
            ambiguous += 1
            continue
        np.testing.assert_array_equal(ids[r][:n_g], oi, err_msg=f"{what} row {r}: ids")
        np.testing.assert_allclose(probs[r][:n_g], op, rtol=1e-5, atol=1e-7, err_msg=f"{what} row {r}: probs")
        if drawn is not None:
            c = np.cumsum(op)
            if np.all(np.abs(c[:-1] - us[r]) > EPS):
                assert drawn[r] == osm.draw(oi, op, us[r]), f"{what} row {r}: draw"
            else:
                ambiguous += 1
    return ambiguous


@pytest.mark.parametrize("temperature,top_k,top_p", [(1.0, 20, 0.95), (0.7, 32, 0.8), (1.3, 5, 1.0), (1.0, 1, 0.95)])
def test_filter_target_logits_matches_oracle(dfl, temperature, top_k, top_p):
    """1024 rows of bf16 N(0, 3) logits over vocabulary 151936 (19 column
    slices, the last ragged)."""
    d, _ = _drafter(dfl)
    with d:
        rows, V = 1024, 151936
        bits = make_target_logits_bf16_np(rows, V, seed=int(temperature * 10) + top_k)
        vals = bits_to_f32(bits).astype(np.float64)
        us = np.random.Generator(np.random.PCG64(top_k)).random(rows)
        logits = torch.from_numpy(bits.view(np.int16)).to(DEV).view(torch.bfloat16)
        ids, probs, drawn = d.sample_filter(logits, temperature, top_k, top_p, uniforms=_f32_dev(us))
        d.sync()
        amb = _check_filter_rows(ids.cpu().numpy(), probs.cpu().numpy(), drawn.cpu().numpy(), vals, us,
                                 temperature, top_k, top_p, "target")
        assert amb <= rows // 100


def test_filter_ties_small_and_ragged_rows(dfl):
    """All-equal rows (ties overflow the threshold buffer: the exact-key
    rounds), rows of three distinct values, ascending rows, a 40-column row,
    a row with a few large values, and rows whose width is not a multiple of
    the slice."""
    d, _ = _drafter(dfl)
    with d:
        for V, fill in ((20000, "zeros"), (40, "normal"), (16392, "spiky"), (32776, "normal"), (24576, "ascending"),
                        (16384, "few_levels")):
            rng = np.random.Generator(np.random.PCG64(V))
            if fill == "zeros":
                vals = np.zeros((6, V), dtype=np.float32)
            elif fill == "ascending":   # the largest values in the last columns of the last slice
                vals = np.tile(np.linspace(-4, 4, V, dtype=np.float32), (6, 1))
            elif fill == "few_levels":  # three distinct values: long runs of ties at the bound
                vals = rng.integers(0, 3, size=(6, V)).astype(np.float32)
            elif fill == "spiky":
                vals = np.full((6, V), -5.0, dtype=np.float32)
                for r in range(6):
                    vals[r, rng.integers(0, V, 40)] = rng.standard_normal(40).astype(np.float32) * 2
            else:
                vals = rng.standard_normal((6, V)).astype(np.float32) * 2
            from synth import bf16_bits
            bits = bf16_bits(vals)
            v64 = bits_to_f32(bits).astype(np.float64)
            us = rng.random(6)
            logits = torch.from_numpy(bits.view(np.int16)).to(DEV).view(torch.bfloat16)
            for top_k, top_p in ((32, 1.0), (20, 0.95), (7, 0.5)):
                ids, probs, drawn = d.sample_filter(logits, 1.0, top_k, top_p, uniforms=_f32_dev(us))
                d.sync()
                _check_filter_rows(ids.cpu().numpy(), probs.cpu().numpy(), drawn.cpu().numpy(), v64, us, 1.0,
                                   top_k, top_p, f"V={V} {fill}")
            if fill == "zeros":   # seven equal logits, top-p 0.5: the lowest four ids (4/7 reaches 0.5)
                got = ids.cpu().numpy()
                np.testing.assert_array_equal(got[:, :4], np.tile(np.arange(4), (6, 1)))
                assert np.all(got[:, 4:] == -1)


def test_draft_sample_lists_and_draws(dfl):
    d, wn = _drafter(dfl, max_batch=8, max_block=16, seed=5)
    orc = oracle.OracleDrafter(TINY, wn)
    with d:
        width = TINY.n_feat_layers * TINY.hidden
        lens = [0, 17, 64, 130, 200, 255]
        seqs = list(range(len(lens)))
        f = make_features_np(sum(lens), width, seed=51)
        d.fuse_ctx(seqs, lens, bf16_dev(f, DEV), pending=False)
        orc.fuse_ctx(seqs, lens, f, pending=False)
        anchors = make_anchor_ids_np(len(seqs), TINY.vocab, seed=52)
        B, temperature, top_k, top_p = 16, 1.0, 20, 0.95
        us = np.random.Generator(np.random.PCG64(53)).random((len(seqs), B - 1))
        drafts, q_ids, q_probs = d.draft_sample(seqs, i32_dev(anchors, DEV), B, temperature, top_k, top_p,
                                                _f32_dev(us))
        d.sync()
        drafts, q_ids, q_probs = drafts.cpu().numpy(), q_ids.cpu().numpy(), q_probs.cpu().numpy()
        import oracle.dflash_oracle as od
        for i, s in enumerate(seqs):
            st = orc._state(s)
            base = od.draft_block(orc.w, orc.shape, int(anchors[i]),
                                  [k[: st["len"]] for k in st["k"]], [v[: st["len"]] for v in st["v"]], B)
            hf = od.rms_norm(base["hidden"], orc.w["g_final"], orc.shape.rms_eps)[1:]
            logits = hf @ orc.w["lm_head"].T
            for j in range(B - 1):
                tag = f"seq {s} pos {j + 1}"
                ids, pr = q_ids[i, j], q_probs[i, j]
                n = int((ids >= 0).sum())
                assert 1 <= n <= top_k and len(set(ids[:n].tolist())) == n, tag
                assert np.all(np.diff(pr[:n]) <= 1e-7) and abs(pr[:n].sum() - 1) < 1e-5, tag
                L = logits[j]
                tol = ATOL + RTOL * np.abs(L)
                out = np.ones(L.shape[0], dtype=bool)
                out[ids[:n]] = False
                # the kept ids are among the oracle's top_k within the tolerance
                kth = np.sort(L)[::-1][top_k - 1]
                assert np.all(L[ids[:n]] + tol[ids[:n]] >= kth - tol.max()), tag
                # probabilities: the oracle's softmax of the library's kept ids, within what the logit
                # tolerance moves them (a shift of e in a logit scales its weight by exp(+-e))
                w = np.exp((L[ids[:n]] - L[ids[0]]) / temperature)
                p_ref = w / w.sum()
                e = 2 * np.max(tol[ids[:n]]) / temperature
                assert np.all(np.abs(pr[:n] - p_ref) <= p_ref * (np.exp(2 * e) - 1) + 1e-6), tag
                # the draw is the list entry the uniform selects (the library's own list)
                c = np.cumsum(pr[:n])
                if np.all(np.abs(c[:-1] - us[i, j]) > EPS):
                    assert drafts[i, j] == osm.draw(ids[:n], pr[:n], us[i, j]), tag


def _random_list(rng, V, k):
    ids = rng.choice(V, size=k, replace=False)
    p = rng.random(k) ** 2 + 1e-3
    p = np.sort(p)[::-1]
    p = (p / p.sum()).astype(np.float32)
    out_i = np.full(32, -1, dtype=np.int32)
    out_p = np.zeros(32, dtype=np.float32)
    out_i[:k] = ids
    out_p[:k] = p
    return out_i, out_p


@pytest.mark.parametrize("B", [2, 8, 16, 32])
def test_verify_sample_matches_oracle(dfl, B):
    n, V = 48, 60    # a small vocabulary so that p and q overlap often
    rng = np.random.Generator(np.random.PCG64(B))
    d, _ = _drafter(dfl, max_batch=n, max_block=32)
    with d:
        seqs = list(range(n))
        width = TINY.n_feat_layers * TINY.hidden
        pend = [int(x) for x in rng.integers(0, B + 1, size=n)]
        f = make_features_np(sum(pend), width, seed=B + 7)
        d.fuse_ctx(seqs, pend, bf16_dev(f, DEV), pending=True)
        q = [[_random_list(rng, V, int(rng.integers(1, 33))) for _ in range(B - 1)] for _ in seqs]
        p = [[_random_list(rng, V, int(rng.integers(1, 33))) for _ in range(B)] for _ in seqs]
        # drafts drawn from q, sometimes made equal to p's top entry so acceptance paths run long
        drafts = np.zeros((n, B - 1), dtype=np.int32)
        for i in seqs:
            for j in range(B - 1):
                qi, qp = q[i][j]
                k = int((qi >= 0).sum())
                drafts[i, j] = qi[rng.choice(k, p=qp[:k] / qp[:k].sum())]
                if rng.random() < 0.5:   # make p agree on the draft with a high probability
                    pi, pp = p[i][j]
                    if drafts[i, j] not in pi:
                        pi[0] = drafts[i, j]
        ua = rng.random((n, B - 1)).astype(np.float32)
        ur = rng.random((n, B)).astype(np.float32)
        q_ids = np.array([[x[0] for x in row] for row in q], dtype=np.int32).reshape(n, B - 1, 32)
        q_pr = np.array([[x[1] for x in row] for row in q], dtype=np.float32).reshape(n, B - 1, 32)
        p_ids = np.array([[x[0] for x in row] for row in p], dtype=np.int32).reshape(n, B, 32)
        p_pr = np.array([[x[1] for x in row] for row in p], dtype=np.float32).reshape(n, B, 32)
        tau, tok = d.verify_sample(seqs, B, i32_dev(drafts, DEV), i32_dev(q_ids, DEV), _f32_dev(q_pr),
                                   i32_dev(p_ids, DEV), _f32_dev(p_pr), _f32_dev(ua), _f32_dev(ur))
        d.sync()
        tau, tok = tau.cpu().numpy(), tok.cpu().numpy()
        checked = 0
        for i in seqs:
            lists = lambda ids, pr: (ids[ids >= 0].astype(np.int64), pr[ids >= 0].astype(np.float64))
            qi = [lists(q_ids[i, j], q_pr[i, j]) for j in range(B - 1)]
            pi = [lists(p_ids[i, j], p_pr[i, j]) for j in range(B)]
            rt, rtok = osm.verify_sample(drafts[i], qi, pi, ua[i].astype(np.float64), ur[i].astype(np.float64))
            # ambiguity: a ratio or a cumulative boundary within EPS of its uniform
            amb = False
            for j in range(min(rt, B - 1)):
                px, qx = osm.prob_of(*pi[j], drafts[i, j]), osm.prob_of(*qi[j], drafts[i, j])
                if qx > 0 and abs(ua[i, j] - min(1.0, px / qx)) < EPS:
                    amb = True
            jj = rt - 1
            if rt <= B - 1:
                r = np.array([max(0.0, pv - osm.prob_of(*qi[jj], int(y))) for y, pv in zip(*pi[jj])])
                c = np.cumsum(r)
                amb |= bool(np.any(np.abs(c[:-1] - ur[i, jj] * c[-1]) < EPS * max(c[-1], 1e-30)))
            else:
                c = np.cumsum(pi[B - 1][1])
                amb |= bool(np.any(np.abs(c[:-1] - ur[i, B - 1] * c[-1]) < EPS))
            if amb:
                continue
            assert (tau[i], tok[i]) == (rt, rtok), f"seq {i}"
            assert d.seq_len(i) == (min(rt, pend[i]), 0), f"seq {i}: commit"
            checked += 1
        assert checked >= n - 3


def test_verify_sample_greedy_limit(dfl):
    """top_k = 1 on both sides: point masses, so the result is the greedy verify."""
    n, B, V = 32, 16, 1000
    rng = np.random.Generator(np.random.PCG64(77))
    d, _ = _drafter(dfl, max_batch=n, max_block=B)
    with d:
        seqs = list(range(n))
        t = rng.integers(0, V, size=(n, B)).astype(np.int32)
        drafts = np.where(rng.random((n, B - 1)) < 0.8, t[:, :-1], rng.integers(0, V, (n, B - 1))).astype(np.int32)
        one = lambda ids: (np.concatenate([ids[..., None], np.full(ids.shape + (31,), -1)], -1).astype(np.int32),
                           np.concatenate([np.ones(ids.shape + (1,)), np.zeros(ids.shape + (31,))], -1)
                           .astype(np.float32))
        qi, qp = one(drafts)
        pi, pp = one(t)
        tau, tok = d.verify_sample(seqs, B, i32_dev(drafts, DEV), i32_dev(qi, DEV), _f32_dev(qp), i32_dev(pi, DEV),
                                   _f32_dev(pp), _f32_dev(rng.random((n, B - 1))), _f32_dev(rng.random((n, B))))
        d.sync()
        for i in seqs:
            assert (int(tau[i]), int(tok[i])) == oracle.verify_block(drafts[i], t[i])


def test_sampling_block_of_one(dfl):
    """B = 1: no drafts; the verify draws the bonus from p_0 and commits one
    pending token; the sampling draft runs the layers and returns no ids."""
    n = 4
    rng = np.random.Generator(np.random.PCG64(5))
    d, _ = _drafter(dfl, max_batch=n, max_block=8)
    with d:
        seqs = list(range(n))
        width = TINY.n_feat_layers * TINY.hidden
        d.fuse_ctx(seqs, [1] * n, bf16_dev(make_features_np(n, width, seed=6), DEV), pending=True)
        p = [_random_list(rng, 50, int(rng.integers(1, 33))) for _ in seqs]
        p_ids = np.array([x[0] for x in p], dtype=np.int32).reshape(n, 1, 32)
        p_pr = np.array([x[1] for x in p], dtype=np.float32).reshape(n, 1, 32)
        ur = rng.random((n, 1)).astype(np.float32)
        tau, tok = d.verify_sample(seqs, 1, None, None, None, i32_dev(p_ids, DEV), _f32_dev(p_pr), None, _f32_dev(ur))
        d.sync()
        for i in seqs:
            ids = p_ids[i, 0][p_ids[i, 0] >= 0]
            pr = p_pr[i, 0][p_ids[i, 0] >= 0].astype(np.float64)
            c = np.cumsum(pr)
            if np.all(np.abs(c[:-1] - ur[i, 0] * c[-1]) > EPS):
                assert (int(tau[i]), int(tok[i])) == (1, osm.draw(ids, pr, ur[i, 0]))
            assert d.seq_len(i) == (1, 0)
        out, q_ids, q_probs = d.draft_sample(seqs, i32_dev(np.arange(n), DEV), 1, 1.0, 20, 0.95, None)
        d.sync()
        assert out.numel() == 0


def test_sampling_argument_errors(dfl):
    d, _ = _drafter(dfl, max_batch=2, max_block=8)
    with d:
        x = torch.zeros(4, 64, dtype=torch.bfloat16, device=DEV)
        for bad in ((0.0, 20, 0.9), (1.0, 0, 0.9), (1.0, 33, 0.9), (1.0, 20, 0.0), (1.0, 20, 1.5)):
            with pytest.raises(dfl.DFlashError) as e:
                d.sample_filter(x, *bad)
            assert e.value.status == dfl.DFLASH_EINVAL
        with pytest.raises(dfl.DFlashError):
            d.sample_filter(torch.zeros(4, 60, dtype=torch.bfloat16, device=DEV), 1.0, 20, 0.9)   # cols % 8
