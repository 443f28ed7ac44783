"""The path selector's CUDA path against the CPU oracle through the C ABI.

What must agree with oracle.path_selector ("DFlash 2" notes, "Solution -
Lightweight Path Selector"): each row's 16 candidates form a top-16 of the
oracle's logits within the logit tolerance (the oracle's exact set where its
16th and 17th logits are more than GAP apart), carry the oracle's logits, and
every pair score S_t(a, b) = U + pair term over those lists matches the
oracle's within the logit tolerance of U plus the same tolerance on the pair
term; the walk's
pick at each position, given its own previous pick, is the oracle's argmax
wherever the oracle's best and second-best scores are more than GAP apart.
Cases: the tiny drafter with ragged contexts at B = 2, 8, 16 and 32 (one to
32 column slices per row, up to 31 positions in the walk), 32 sequences of
the tiny drafter (512 block rows: CTA-pair LM head with the H rows stacked),
and the Qwen3-8B shape (vocabulary 151936, 11 column slices) at 2 layers.
With W_H = 0 the walk must return the plain greedy draft.
"""
import dataclasses

import numpy as np
import pytest

import oracle
from oracle import path_selector as ops
from synth import (TINY, QWEN3_8B, make_weights_np, make_selector_weights_np, make_features_np,
                   make_anchor_ids_np, make_weights_torch, torch_weights_to_np)
from tests.gpu_util import np_weights_to_device, bf16_dev, i32_dev, assert_close, GAP, ATOL, RTOL

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def dfl():
    import __graft_entry__
    __graft_entry__.build()
    import block_diffusion_drafter_pass_gb300 as m
    return m


def _sel_dev(sel):
    return {k: bf16_dev(v, DEV) for k, v in sel.items()}


def _compare_selection(d, orc, sel_np, seqs, anchors, B, got_ids, what, ref=None):
    """Check one selector draft; returns (walk decisions checked, oracle results).

    Candidate lists: distinct ids in non-increasing logit order, logits within
    the logit tolerance of the oracle's, and a valid top-16 of the oracle's
    logits (no excluded id beats an included one by more than twice the
    tolerance); where the oracle's 16th and 17th logits are more than GAP
    apart, the oracle's own set. Pair scores: the oracle's S_t(a, b) over the
    library's candidate lists. Walk: at every position, given the library's
    own previous pick, the pick must be the oracle's argmax wherever the
    oracle's best and second-best scores are more than GAP apart.
    """
    if ref is None:
        ref = ops.drafter_select(orc, seqs, anchors, B, sel_np)
    cand, u, sc = d.last_selection(len(seqs), B)
    T = B - 1
    E = orc.w["embed"]
    s_w = {k: np.asarray(v, dtype=E.dtype) for k, v in sel_np.items()}
    checked = 0
    for i, r in enumerate(ref):
        for t in range(T):
            row = i * T + t
            c = cand[row]
            L = r["logits"][t]
            tag = f"{what} seq {i} t {t}"
            assert len(set(c.tolist())) == ops.K_SEL and c.min() >= 0 and c.max() < L.shape[0], f"{tag}: ids"
            assert np.all(np.diff(u[row]) <= 0), f"{tag}: candidates not in logit order"
            assert_close(u[row], L[c], f"{tag}: candidate logits")
            out = np.ones(L.shape[0], dtype=bool)
            out[c] = False
            tol = ATOL + RTOL * np.abs(L)
            worst_in = np.min(L[c] + tol[c])
            if out.any():
                assert np.max(L[out] - tol[out]) <= worst_in, f"{tag}: not a top-16 of the oracle's logits"
            if r["gap16"][t] > GAP:
                assert sorted(c.tolist()) == sorted(r["cand"][t].tolist()), f"{tag}: candidate set"
            prev = [int(anchors[i])] if t == 0 else cand[row - 1].tolist()
            s_ref = ops.pair_scores(L[c], c, prev, E, s_w["w_a"], s_w["w_b"], r["h_gate"][t])
            # S = U + pair term: each part carries its own tolerance (the
            # logits' for U, the same form for the pair term)
            pair_ref = s_ref - L[c][None, :]
            bound = 2 * ATOL + RTOL * (np.abs(L[c])[None, :] + np.abs(pair_ref))
            err = np.abs(sc[row][: len(prev)] - s_ref)
            assert np.all(err <= bound), f"{tag}: pair scores, worst excess {float((err - bound).max()):.4g}"
            p = 0 if t == 0 else int(np.flatnonzero(cand[row - 1] == got_ids[i, t - 1])[0])
            srt = np.sort(s_ref[p])[::-1]
            if srt[0] - srt[1] > GAP:
                assert got_ids[i, t] == c[int(np.argmax(s_ref[p]))], f"{tag}: walk id"
                checked += 1
    return checked, ref


def _tiny(dfl, max_batch, max_block, seed=3, shape=TINY, edit=None):
    wn = make_weights_np(shape, seed=seed)
    if edit:
        edit(wn)
    d = dfl.Drafter(shape, np_weights_to_device(wn, DEV), max_seqs=max_batch, max_batch=max_batch,
                    max_block=max_block, max_ctx=512, max_fuse_tokens=10000)
    return d, wn, oracle.OracleDrafter(shape, wn)


def _run_case(dfl, d, orc, shape, sel_seed, lens, B, what, feat_seed=61):
    sel = make_selector_weights_np(shape, seed=sel_seed)
    d.set_path_selector(**_sel_dev(sel))
    width = shape.n_feat_layers * shape.hidden
    seqs = list(range(len(lens)))
    f = make_features_np(sum(lens), width, seed=feat_seed)
    d.fuse_ctx(seqs, lens, bf16_dev(f, DEV), pending=False)
    orc.fuse_ctx(seqs, lens, f, pending=False)
    anchors = make_anchor_ids_np(len(lens), shape.vocab, seed=feat_seed + 1)
    ids = d.draft(seqs, i32_dev(anchors, DEV), B)
    d.sync()
    return _compare_selection(d, orc, sel, seqs, anchors, B, ids.cpu().numpy(), what)


def test_tiny_selector_ragged_block_sizes(dfl):
    d, wn, orc = _tiny(dfl, max_batch=6, max_block=32)
    with d:
        sel = make_selector_weights_np(TINY, seed=21)
        d.set_path_selector(**_sel_dev(sel))
        width = TINY.n_feat_layers * TINY.hidden
        lens = [0, 1, 63, 64, 130, 257]
        f = make_features_np(sum(lens), width, seed=22)
        seqs = list(range(6))
        d.fuse_ctx(seqs, lens, bf16_dev(f, DEV), pending=False)
        orc.fuse_ctx(seqs, lens, f, pending=False)
        anchors = make_anchor_ids_np(6, TINY.vocab, seed=23)
        total, differs = 0, 0
        for B, idx in ((16, seqs), (8, seqs), (2, seqs), (32, [5]), (16, [2])):
            a = anchors[idx]
            ids = d.draft(idx, i32_dev(a, DEV), B)
            d.sync()
            walked, ref = _compare_selection(d, orc, sel, idx, a, B, ids.cpu().numpy(), f"tiny B={B}")
            total += walked
            differs += sum(int((r["draft"] != r["plain_draft"]).any()) for r in ref)
        assert total >= 40, total
        assert differs > 0, "the walk never left the greedy path: the case does not exercise the pair term"


def test_tiny_selector_batch32_pair_tiles(dfl):
    d, wn, orc = _tiny(dfl, max_batch=32, max_block=16, seed=5)
    with d:
        sel = make_selector_weights_np(TINY, seed=31)
        d.set_path_selector(**_sel_dev(sel))
        width = TINY.n_feat_layers * TINY.hidden
        rng = np.random.default_rng(32)
        lens = [int(x) for x in rng.integers(0, 300, size=32)]
        f = make_features_np(sum(lens), width, seed=33)
        seqs = list(range(32))
        d.fuse_ctx(seqs, lens, bf16_dev(f, DEV), pending=False)
        orc.fuse_ctx(seqs, lens, f, pending=False)
        anchors = make_anchor_ids_np(32, TINY.vocab, seed=34)
        ids = d.draft(seqs, i32_dev(anchors, DEV), 16)
        d.sync()
        walked, _ = _compare_selection(d, orc, sel, seqs, anchors, 16, ids.cpu().numpy(), "tiny batch 32")
        assert walked >= 100, walked


def test_selector_with_zero_gate_is_greedy(dfl):
    """W_H = 0 leaves S_t(a, b) = U_t(b): the walk is the plain argmax draft."""
    d, wn, orc = _tiny(dfl, max_batch=4, max_block=16, seed=7)
    with d:
        width = TINY.n_feat_layers * TINY.hidden
        lens = [40, 0, 200, 77]
        f = make_features_np(sum(lens), width, seed=41)
        seqs = [0, 1, 2, 3]
        d.fuse_ctx(seqs, lens, bf16_dev(f, DEV), pending=False)
        anchors = i32_dev(make_anchor_ids_np(4, TINY.vocab, seed=42), DEV)
        plain = d.draft(seqs, anchors, 16).cpu().numpy()
        _, top = d.last_draft(4, 16)
        sel = make_selector_weights_np(TINY, seed=43)
        sel["w_h"] = np.zeros_like(sel["w_h"])
        d.set_path_selector(**_sel_dev(sel))
        walk = d.draft(seqs, anchors, 16).cpu().numpy()
        cand, u, _ = d.last_selection(4, 16)
        d.sync()
        gap = u[:, 0] - u[:, 1]
        sure = (gap > 1e-3).reshape(4, 15)
        np.testing.assert_array_equal(walk[sure], plain[sure])
        np.testing.assert_array_equal(cand[:, 0].reshape(4, 15)[sure], plain[sure])
        assert_close(u[:, 0], top, "top logits with and without the selector")
        # removing the selector restores the plain draft
        d.set_path_selector()
        again = d.draft(seqs, anchors, 16).cpu().numpy()
        d.sync()
        np.testing.assert_array_equal(again, plain)


def test_qwen3_8b_shape_selector_two_layers(dfl):
    shape = QWEN3_8B.with_layers(2)
    wt = make_weights_torch(shape, seed=51, device=DEV, gamma="jitter")
    wn = torch_weights_to_np(wt)
    orc = oracle.OracleDrafter(shape, wn, dtype=np.float32)
    width = shape.n_feat_layers * shape.hidden
    with dfl.Drafter(shape, wt, max_seqs=2, max_batch=2, max_block=16, max_ctx=1024,
                     max_fuse_tokens=1024) as d:
        sel = make_selector_weights_np(shape, seed=52)
        d.set_path_selector(**_sel_dev(sel))
        f = make_features_np(900, width, seed=53)
        d.fuse_ctx([0, 1], [200, 700], bf16_dev(f, DEV), pending=False)
        orc.fuse_ctx([0, 1], [200, 700], f, pending=False)
        anchors = make_anchor_ids_np(2, shape.vocab, seed=54)
        ids = d.draft([0, 1], i32_dev(anchors, DEV), 16)
        d.sync()
        walked, _ = _compare_selection(d, orc, sel, [0, 1], anchors, 16, ids.cpu().numpy(), "8B 2-layer")
        assert walked >= 4, walked


def test_selector_argument_errors(dfl):
    d, wn, _ = _tiny(dfl, max_batch=2, max_block=8)
    with d:
        sel = _sel_dev(make_selector_weights_np(TINY, seed=1))
        with pytest.raises(dfl.DFlashError) as e:
            d.set_path_selector(sel["w_a"], sel["w_b"], None)
        assert e.value.status == dfl.DFLASH_EINVAL
        lib = dfl.load_library()
        st = lib.dflash_set_path_selector(d.ctx, sel["w_a"].data_ptr(), sel["w_b"].data_ptr(),
                                          sel["w_h"].data_ptr(), 128, None)
        assert st == dfl.DFLASH_EINVAL
        # no selection to read before a selector draft
        with pytest.raises(dfl.DFlashError):
            d.last_selection(1, 8)


def test_selector_all_equal_logits(dfl):
    """A zero LM head makes every logit 0: the candidates are the 16 lowest
    ids in order (the tie rule). Vocabulary 10000: the first 8192-column
    slice holds more tied keys than the threshold filter's buffer and takes
    the exact-key path, the second (1808 columns) does not."""
    def zero_head(wn):
        wn["lm_head"] = np.zeros_like(wn["lm_head"])
    shape = dataclasses.replace(TINY, vocab=10000, mask_id=9999)
    d, wn, orc = _tiny(dfl, max_batch=2, max_block=16, seed=9, shape=shape, edit=zero_head)
    with d:
        checked, _ = _run_case(dfl, d, orc, shape, 71, [30, 100], 16, "zero LM head")
        cand, u, _ = d.last_selection(2, 16)
        np.testing.assert_array_equal(cand, np.tile(np.arange(16), (30, 1)))
        assert np.all(u == 0)


def test_selector_vocab_16_and_wide_vocab(dfl):
    """Vocabulary 16 (every token a candidate) and vocabulary 300000 (37
    column slices of 8192: the merge ranks more than 512 keys)."""
    small = dataclasses.replace(TINY, vocab=16, mask_id=15)
    d, wn, orc = _tiny(dfl, max_batch=2, max_block=8, seed=11, shape=small)
    with d:
        _run_case(dfl, d, orc, small, 81, [5, 70], 8, "vocab 16")
        cand, _, _ = d.last_selection(2, 8)
        assert all(sorted(r.tolist()) == list(range(16)) for r in cand)
    wide = dataclasses.replace(TINY, vocab=300000, mask_id=299999)
    d, wn, orc = _tiny(dfl, max_batch=2, max_block=8, seed=12, shape=wide)
    with d:
        checked, _ = _run_case(dfl, d, orc, wide, 82, [64, 9], 8, "vocab 300000")
        assert checked >= 2, checked


def test_qwen3_8b_full_depth_selector_and_sampling_head(dfl):
    """The benchmarked configuration (5 layers, context 4096, B = 16, batch 1):
    the selector's lists, pair scores and walk, then the sampling head's lists
    (validity within the logit tolerance) and its draws from its own lists.
    Five layers of bf16 activation storage move the hidden state past the
    two-layer guard (as in the full-depth draft test), so the reference
    logits and gates come from the oracle's pass with the library's bf16
    storage points emulated."""
    from tests.emulate import bf16_context, bf16_storage_hidden
    from oracle import sampling as osm
    import oracle.dflash_oracle as od
    shape = QWEN3_8B
    wt = make_weights_torch(shape, seed=0, device=DEV, gamma="jitter")
    wn = torch_weights_to_np(wt)
    orc = oracle.OracleDrafter(shape, wn, dtype=np.float32)
    width = shape.n_feat_layers * shape.hidden
    with dfl.Drafter(shape, wt, max_seqs=1, max_batch=1, max_block=16, max_ctx=4096 + 64,
                     max_fuse_tokens=4096) as d:
        f = make_features_np(4096, width, seed=1)
        d.fuse_ctx([0], [4096], bf16_dev(f, DEV), pending=False)
        orc.fuse_ctx([0], [4096], f, pending=False)
        anchors = make_anchor_ids_np(1, shape.vocab, seed=2)
        sel = make_selector_weights_np(shape, seed=3)
        d.set_path_selector(**_sel_dev(sel))
        ids = d.draft([0], i32_dev(anchors, DEV), 16)
        d.sync()
        kb, vb = bf16_context(wn, shape, f, dtype=np.float32)
        emu = bf16_storage_hidden(wn, shape, int(anchors[0]), kb, vb, 16, dtype=np.float32)
        hf = od.rms_norm(emu, wn["g_final"], shape.rms_eps)[1:]
        logits = hf @ np.asarray(wn["lm_head"], dtype=np.float32).T
        w_h = np.asarray(sel["w_h"], dtype=np.float32)
        gap16 = np.array([np.sort(r)[::-1][15] - np.sort(r)[::-1][16] for r in logits])
        cand = np.array([ops.top_k(r)[0] for r in logits])
        ref = [{"logits": logits, "h_gate": hf @ w_h.T, "gap16": gap16, "cand": cand}]
        checked, _ = _compare_selection(d, orc, sel, [0], anchors, 16, ids.cpu().numpy(), "8B full depth", ref=ref)
        assert checked >= 3, checked
        d.set_path_selector()
        us = np.random.Generator(np.random.PCG64(4)).random((1, 15))
        drafts, q_ids, q_probs = d.draft_sample([0], i32_dev(anchors, DEV), 16, 1.0, 20, 0.95,
                                                torch.from_numpy(us.astype(np.float32)).to(DEV))
        d.sync()
        drafts, q_ids, q_probs = drafts.cpu().numpy()[0], q_ids.cpu().numpy()[0], q_probs.cpu().numpy()[0]
        for j in range(15):
            n = int((q_ids[j] >= 0).sum())
            c = q_ids[j][:n]
            L = logits[j]
            assert 1 <= n <= 20 and len(set(c.tolist())) == n
            tol = ATOL + RTOL * np.abs(L)
            kth = np.sort(L)[::-1][19]
            assert np.all(L[c] + tol[c] >= kth - tol.max()), f"pos {j + 1}: not among the top 20"
            cum = np.cumsum(q_probs[j][:n])
            if np.all(np.abs(cum[:-1] - us[0, j]) > 1e-5):
                assert drafts[j] == osm.draw(c, q_probs[j][:n], us[0, j])
