"""The target-shaped verify pass on the GPU against the target-pass oracle
(oracle/target_pass.py), through the C ABI: prefill in committed blocks, a
pending verify block, greedy ids at every block position (bit-exact where the
oracle's top-1/top-2 gap exceeds 0.1, a near-top logit elsewhere), the
features of the feature layers, the K/V the pass caches, the commit of tau;
causal masking in both query-row layouts of the attention kernel; and the
whole DFlash cycle (drafter + target) run in lockstep with the oracles."""
from dataclasses import replace

import numpy as np
import pytest

import oracle
from oracle import target_pass as tp
from synth import TINY, QWEN3_8B, make_weights_np, make_weights_torch, torch_weights_to_np, make_anchor_ids_np
from tests.gpu_util import (np_weights_to_device, bf16_dev, i32_dev, assert_close, assert_hidden_close,
                            check_near_top, GAP, ROW_REL_HIGH_GAIN)

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def dfl():
    import __graft_entry__
    __graft_entry__.build()
    import block_diffusion_drafter_pass_gb300 as m
    return m


def _compare_pass(got_ids, hid, top, feats, ref, what, row_rel=None):
    """One sequence's target pass against the oracle's result."""
    got_ids = np.asarray(got_ids, dtype=np.int64)
    assert_hidden_close(hid, ref["hidden"], f"{what}: final residual stream")
    assert_close(top, ref["top1"], f"{what}: winning logits", row_rel=row_rel)
    sure = ref["gap"] > GAP
    np.testing.assert_array_equal(got_ids[sure], ref["ids"][sure], err_msg=f"{what}: target ids (gap > {GAP})")
    check_near_top(got_ids, top, {"logits": ref["logits"], "top1": ref["top1"]}, what, row_rel)
    if feats is not None:
        assert_hidden_close(feats, ref["feats"], f"{what}: features")
    return int(sure.sum())


def _tiny_target(n_layers=4, **kw):
    sh = replace(TINY, n_layers=n_layers, n_feat_layers=2, **kw)
    return sh


def _run_prefill(t, orc, seq, ids, chunk):
    """Committed passes over `ids` in blocks of at most `chunk` tokens; per
    block the GPU's ids, features, (residual stream, winning logits) read
    right after the pass, and the oracle's result."""
    out = []
    for p0 in range(0, len(ids), chunk):
        blk = np.array([ids[p0:p0 + chunk]], dtype=np.int32)
        g_ids, g_feats = t.forward([seq], i32_dev(blk, DEV), blk.shape[1], pending=False)
        last = t.last_pass(1, blk.shape[1])
        r = orc.forward([seq], blk, pending=False)[0]
        out.append((g_ids, g_feats, last, r))
    return out


@pytest.mark.parametrize("std,n_layers", [(0.05, 4), (0.03, 8)])
def test_tiny_target_prefill_verify_and_commit(dfl, std, n_layers):
    """Tiny width (features of the last two layers): a 70-token prompt in
    committed blocks of 32, 32 and 6 tokens, then pending verify blocks of
    B = 8 with the commit of tau, over two cycles and two sequences; 4 layers
    and a deeper 8-layer target."""
    sh = _tiny_target(n_layers)
    fl = [n_layers - 2, n_layers - 1]
    wn = make_weights_np(sh, seed=301, gamma="jitter", std=std)
    orc = tp.OracleTarget(sh, wn, fl)
    row_rel = None
    rng = np.random.Generator(np.random.PCG64(302))
    with dfl.Target(sh, np_weights_to_device(wn, DEV), fl, max_seqs=2, max_batch=2, max_block=32, max_ctx=512) as t:
        checked = 0
        for s, plen in ((0, 70), (1, 21)):
            prompt = rng.integers(0, sh.vocab, size=plen).astype(np.int32)
            for k, (g_ids, g_feats, (hid, top), r) in enumerate(_run_prefill(t, orc, s, prompt, 32)):
                checked += _compare_pass(g_ids.cpu().numpy()[0], hid, top, g_feats.float().cpu().numpy(), r,
                                         f"prefill seq {s} block {k}", row_rel)
            assert t.seq_len(s) == orc.seq_len(s)
        B = 8
        for cyc in range(2):
            blocks = rng.integers(0, sh.vocab, size=(2, B)).astype(np.int32)
            g_ids, g_feats = t.forward([0, 1], i32_dev(blocks, DEV), B, pending=True)
            refs = orc.forward([0, 1], blocks, pending=True)
            hid, top = t.last_pass(2, B)
            got = g_ids.cpu().numpy()
            feats = g_feats.float().cpu().numpy()
            for i in range(2):
                checked += _compare_pass(got[i], hid[i * B:(i + 1) * B], top[i * B:(i + 1) * B],
                                         feats[i * B:(i + 1) * B], refs[i], f"cycle {cyc} seq {i}", row_rel)
            # drafts agree with the oracle's target ids for a seeded count, then
            # differ; both verifies take the oracle's ids
            ref_ids = np.stack([refs[i]["ids"] for i in range(2)]).astype(np.int32)
            drafts = ref_ids[:, : B - 1].copy()
            for i, m in enumerate(rng.integers(0, B, size=2)):
                if m < B - 1:
                    drafts[i, m] = (drafts[i, m] + 1) % sh.vocab
            tau, bonus = t.verify([0, 1], B, i32_dev(drafts, DEV), i32_dev(ref_ids, DEV))
            rt, rb = orc.verify([0, 1], B, drafts, ref_ids)
            t.sync()
            np.testing.assert_array_equal(tau.cpu().numpy(), rt)
            np.testing.assert_array_equal(bonus.cpu().numpy(), rb)
            for s in (0, 1):
                assert t.seq_len(s) == orc.seq_len(s)
                n = orc.seq_len(s)[0]
                for l in (0, n_layers - 1):
                    k, v = t.read_kv(l, s, 0, n)
                    assert_close(k, orc.seqs[s]["k"][l][:n], f"cached K layer {l} seq {s}", row_rel=row_rel)
                    assert_close(v, orc.seqs[s]["v"][l][:n], f"cached V layer {l} seq {s}", row_rel=row_rel)
        assert checked > 20


@pytest.mark.parametrize("n_heads,n_kv,blocks", [(8, 2, (32, 16, 1)), (6, 2, (32, 5))])
def test_causal_mask_in_both_row_layouts(dfl, n_heads, n_kv, blocks):
    """G*B = 128 and 96 (one thread per query row), G*B <= 64 (rows spread 16
    per TMEM lane quarter): each block position attends to its own prefix of
    the block only."""
    sh = replace(TINY, n_heads=n_heads, n_kv_heads=n_kv, n_layers=2, n_feat_layers=1)
    fl = [0]
    wn = make_weights_np(sh, seed=311, gamma="jitter", std=0.05)
    orc = tp.OracleTarget(sh, wn, fl)
    rng = np.random.Generator(np.random.PCG64(312))
    with dfl.Target(sh, np_weights_to_device(wn, DEV), fl, max_seqs=1, max_batch=1, max_block=32, max_ctx=1024) as t:
        _run_prefill(t, orc, 0, rng.integers(0, sh.vocab, size=100).astype(np.int32), 32)
        for B in blocks:
            blk = rng.integers(0, sh.vocab, size=(1, B)).astype(np.int32)
            g_ids, g_feats = t.forward([0], i32_dev(blk, DEV), B, pending=False)
            r = orc.forward([0], blk, pending=False)[0]
            hid, top = t.last_pass(1, B)
            _compare_pass(g_ids.cpu().numpy()[0], hid, top, g_feats.float().cpu().numpy(), r,
                          f"G={n_heads // n_kv} B={B}")


def test_qwen3_8b_width_target_two_layers(dfl):
    """8B width, 2 target layers (features of both): a 300-token prompt in
    committed blocks of 32, then a pending B = 16 verify block."""
    shape = replace(QWEN3_8B.with_layers(2), n_feat_layers=2)
    fl = [0, 1]
    wt = make_weights_torch(shape, seed=321, device=DEV, gamma="jitter")
    wn = torch_weights_to_np(wt)
    orc = tp.OracleTarget(shape, wn, fl, dtype=np.float32)
    rng = np.random.Generator(np.random.PCG64(322))
    with dfl.Target(shape, wt, fl, max_seqs=1, max_batch=1, max_block=32, max_ctx=1024) as t:
        _run_prefill(t, orc, 0, rng.integers(0, shape.vocab, size=300).astype(np.int32), 32)
        blk = rng.integers(0, shape.vocab, size=(1, 16)).astype(np.int32)
        g_ids, g_feats = t.forward([0], i32_dev(blk, DEV), 16, pending=True)
        r = orc.forward([0], blk, pending=True)[0]
        hid, top = t.last_pass(1, 16)
        checked = _compare_pass(g_ids.cpu().numpy()[0], hid, top, g_feats.float().cpu().numpy(), r, "8B target")
        assert checked >= 3
        for l in (0, 1):
            for p0 in (0, 63, 64, 299, 300, 315):
                k, v = t.read_kv(l, 0, p0, 1)
                assert_close(k, orc.seqs[0]["k"][l][p0:p0 + 1], f"8B target K layer {l} pos {p0}")
                assert_close(v, orc.seqs[0]["v"][l][p0:p0 + 1], f"8B target V layer {l} pos {p0}")


def test_dflash_cycle_with_a_target_in_lockstep(dfl):
    """The whole cycle on the GPU, driven by the oracles' choices: prefill
    through the target, features into the drafter's context, then drafter
    pass -> target verify pass over [anchor, drafts] -> dflash_verify on both
    contexts -> the block's features into the drafter (pending), anchor =
    bonus. Every GPU pass is compared with the oracle's on the same inputs
    (ids bit-exact where the gap exceeds 0.1, features within the hidden-state
    tolerance); tau, bonus and every length exactly. The drafters consume the
    oracle target's features rounded to bf16, so no oracle input comes from
    the GPU."""
    from synth import bf16_round
    tsh = replace(TINY, n_layers=4, n_feat_layers=3)
    fl = [1, 2, 3]
    dsh = replace(TINY, n_layers=1, n_feat_layers=3)
    tw = make_weights_np(tsh, seed=331, gamma="jitter", std=0.05)
    dw = make_weights_np(dsh, seed=332, gamma="jitter", std=0.05)
    to = tp.OracleTarget(tsh, tw, fl)
    do = oracle.OracleDrafter(dsh, dw)
    rng = np.random.Generator(np.random.PCG64(333))
    B = 8
    with dfl.Target(tsh, np_weights_to_device(tw, DEV), fl, max_seqs=1, max_batch=1, max_block=32,
                    max_ctx=512) as t, \
            dfl.Drafter(dsh, np_weights_to_device(dw, DEV), max_seqs=1, max_batch=1, max_block=B, max_ctx=512,
                        max_fuse_tokens=256) as d:
        prompt = rng.integers(0, tsh.vocab, size=40).astype(np.int32)
        checked = 0
        for k, (g_ids, g_feats, (hid, top), r) in enumerate(_run_prefill(t, to, 0, prompt, 32)):
            n = r["ids"].shape[0]
            checked += _compare_pass(g_ids.cpu().numpy()[0], hid, top, g_feats.float().cpu().numpy(), r,
                                     f"prefill block {k}")
            f = bf16_round(np.asarray(r["feats"], dtype=np.float32))
            d.fuse_ctx([0], [n], bf16_dev(f, DEV), pending=False)
            do.fuse_ctx([0], [n], f, pending=False)
        anchor = int(r["ids"][-1])
        taus = []
        for cyc in range(6):
            ref_d = do.draft([0], [anchor], B)[0]
            drafts = d.draft([0], i32_dev([anchor], DEV), B)
            got_d = drafts.cpu().numpy()[0]
            sure = ref_d["gap"] > GAP
            np.testing.assert_array_equal(got_d[sure], ref_d["draft"][sure], err_msg=f"cycle {cyc} drafts")
            od = ref_d["draft"].astype(np.int32)
            block = np.array([[anchor] + [int(x) for x in od]], dtype=np.int32)
            g_ids, g_feats = t.forward([0], i32_dev(block, DEV), B, pending=True)
            r = to.forward([0], block, pending=True)[0]
            hid, top = t.last_pass(1, B)
            checked += _compare_pass(g_ids.cpu().numpy()[0], hid, top, g_feats.float().cpu().numpy(), r,
                                     f"cycle {cyc} target")
            f = bf16_round(np.asarray(r["feats"], dtype=np.float32))
            d.fuse_ctx([0], [B], bf16_dev(f, DEV), pending=True)
            do.fuse_ctx([0], [B], f, pending=True)
            # the drafts agree with the oracle target's ids for a seeded count,
            # so tau varies from cycle to cycle
            tgt = r["ids"].astype(np.int32)
            m = int(rng.integers(0, B))
            drafts_v = tgt[: B - 1].copy()
            if m < B - 1:
                drafts_v[m] = (drafts_v[m] + 1) % tsh.vocab
            tau_t, bonus_t = t.verify([0], B, i32_dev(drafts_v[None, :], DEV), i32_dev(tgt[None, :], DEV))
            tau_d, bonus_d = d.verify([0], B, i32_dev(drafts_v[None, :], DEV), i32_dev(tgt[None, :], DEV))
            rt, rb = to.verify([0], B, drafts_v[None, :], tgt[None, :])
            do.verify([0], B, drafts_v[None, :], tgt[None, :])
            t.sync()
            assert int(tau_t.item()) == int(rt[0]) == int(tau_d.item())
            assert int(bonus_t.item()) == int(rb[0]) == int(bonus_d.item())
            assert t.seq_len(0) == to.seq_len(0) and d.seq_len(0) == do.seq_len(0)
            n = to.seq_len(0)[0]
            k_, v_ = t.read_kv(3, 0, 0, n)
            assert_close(k_, to.seqs[0]["k"][3][:n], f"cycle {cyc} target K")
            taus.append(int(rt[0]))
            anchor = int(rb[0])
        assert checked > 10 and max(taus) > 1
