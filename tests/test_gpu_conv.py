"""Two-tap dynamic convolutions (DFlash 2) on the GPU against the conv oracle.

The drafter pass with the four convolutions per layer (attention in/out,
feed-forward in/out) is compared with oracle.two_tap_conv.draft_block_conv
over the oracle drafter's own context K/V (the injected context does not pass
through a convolution): draft ids, winning logits and the final residual
stream. Cases: two layers (so an output site hands its V products to the
next layer's input site), rank 16 and 8, several sequences with ragged
contexts, B = 8, 5 and 1 (row counts that are and are not multiples of the
kernel's 16-row tiles, a block of the anchor alone), removing the
convolutions again, identity convolutions against the plain oracle pass, and
the 8B width at rank 80.
"""
from dataclasses import replace

import numpy as np
import pytest

import oracle
from oracle import two_tap_conv as ttc
from synth import (TINY, QWEN3_8B, make_weights_np, make_features_np, make_anchor_ids_np, make_conv_weights_np,
                   make_weights_torch, torch_weights_to_np)
from tests.gpu_util import np_weights_to_device, bf16_dev, i32_dev, compare_draft

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def dfl():
    import __graft_entry__
    __graft_entry__.build()
    import block_diffusion_drafter_pass_gb300 as m
    return m


def _conv_dev(convs):
    return [{site: {k: bf16_dev(np.ascontiguousarray(v), DEV) for k, v in c.items()} for site, c in layer.items()}
            for layer in convs]


def _conv_np(convs, dtype):
    return [{site: {k: np.asarray(v, dtype=dtype) for k, v in c.items()} for site, c in layer.items()}
            for layer in convs]


def _ref_conv(orc, convs, seqs, anchors, B):
    out = []
    for s, a in zip(seqs, anchors):
        st = orc.seqs[int(s)]
        kc = [k[: st["len"]] for k in st["k"]]
        vc = [v[: st["len"]] for v in st["v"]]
        out.append(ttc.draft_block_conv(orc.w, orc.shape, convs, int(a), kc, vc, B))
    return out


def _draft_compare(d, refs, seqs, anchors, B, what):
    ids = d.draft(seqs, i32_dev(anchors, DEV), B)
    d.sync()
    hid, top = d.last_draft(len(seqs), B)
    got = ids.cpu().numpy()
    checked = 0
    for i in range(len(seqs)):
        checked += compare_draft(got[i] if B > 1 else [], hid[i * B:(i + 1) * B], top[i * (B - 1):(i + 1) * (B - 1)],
                                 refs[i], B, f"{what} seq {seqs[i]}")
    return checked


@pytest.mark.parametrize("rank", [16, 8])
def test_conv_two_layers_ragged(dfl, rank):
    sh = replace(TINY, n_layers=2)
    wn = make_weights_np(sh, seed=61, gamma="jitter", std=0.02)
    cw = make_conv_weights_np(sh, rank=rank, seed=62)
    orc = oracle.OracleDrafter(sh, wn)
    convs = _conv_np(cw, np.float64)
    width = sh.n_feat_layers * sh.hidden
    seqs = [0, 1, 2]
    with dfl.Drafter(sh, np_weights_to_device(wn, DEV), max_seqs=3, max_batch=3, max_block=8, max_ctx=512,
                     max_fuse_tokens=512) as d:
        ctx = [70, 0, 200]
        f = make_features_np(sum(ctx), width, seed=63)
        d.fuse_ctx(seqs, ctx, bf16_dev(f, DEV), pending=False)
        orc.fuse_ctx(seqs, ctx, f, pending=False)
        d.set_conv(_conv_dev(cw), rank)
        anchors = make_anchor_ids_np(3, sh.vocab, seed=64)
        checked = 0
        for B in (8, 5, 1):
            refs = _ref_conv(orc, convs, seqs, anchors, B)
            checked += _draft_compare(d, refs, seqs, anchors, B, f"conv r={rank} B={B}")
        # removed again: the plain pass
        d.set_conv(None)
        refs = orc.draft(seqs, anchors, 8)
        checked += _draft_compare(d, refs, seqs, anchors, 8, "conv removed")
        assert checked > 0


def test_conv_changes_the_pass(dfl):
    """The convolutions are not a no-op at these weights: the oracle's conv pass
    and plain pass differ well beyond the tolerance, and the GPU follows the
    conv pass."""
    sh = replace(TINY, n_layers=2)
    wn = make_weights_np(sh, seed=71, gamma="jitter", std=0.02)
    cw = make_conv_weights_np(sh, rank=16, seed=72, corr=0.5, tap1_std=0.5)
    orc = oracle.OracleDrafter(sh, wn)
    width = sh.n_feat_layers * sh.hidden
    with dfl.Drafter(sh, np_weights_to_device(wn, DEV), max_seqs=1, max_batch=1, max_block=8, max_ctx=512,
                     max_fuse_tokens=512) as d:
        f = make_features_np(100, width, seed=73)
        d.fuse_ctx([0], [100], bf16_dev(f, DEV), pending=False)
        orc.fuse_ctx([0], [100], f, pending=False)
        d.set_conv(_conv_dev(cw), 16)
        anchors = make_anchor_ids_np(1, sh.vocab, seed=74)
        refs = _ref_conv(orc, _conv_np(cw, np.float64), [0], anchors, 8)
        plain = orc.draft([0], anchors, 8)
        diff = np.abs(refs[0]["hidden"] - plain[0]["hidden"]).max() / np.abs(plain[0]["hidden"]).max()
        assert diff > 0.05, f"conv and plain passes differ by only {diff:.3g} of the hidden range"
        _draft_compare(d, refs, [0], anchors, 8, "conv vs plain")


def test_identity_conv_is_the_plain_pass(dfl):
    sh = replace(TINY, n_layers=2)
    wn = make_weights_np(sh, seed=81, gamma="jitter", std=0.02)
    orc = oracle.OracleDrafter(sh, wn)
    width = sh.n_feat_layers * sh.hidden
    ident = []
    for _ in range(sh.n_layers):
        c = ttc.identity_conv(sh.hidden, 8, dtype=np.float32)
        ident.append({site: c for site in ttc.TAPS})
    with dfl.Drafter(sh, np_weights_to_device(wn, DEV), max_seqs=2, max_batch=2, max_block=16, max_ctx=512,
                     max_fuse_tokens=512) as d:
        f = make_features_np(150, width, seed=83)
        d.fuse_ctx([0, 1], [50, 100], bf16_dev(f, DEV), pending=False)
        orc.fuse_ctx([0, 1], [50, 100], f, pending=False)
        d.set_conv(_conv_dev(ident), 8)
        anchors = make_anchor_ids_np(2, sh.vocab, seed=84)
        refs = orc.draft([0, 1], anchors, 16)
        # the residual stream and every row's near-top check (few rows of this
        # low-gain pass have a top-1/top-2 gap wide enough for an id match)
        _draft_compare(d, refs, [0, 1], anchors, 16, "identity conv")


def test_conv_8b_width_rank80(dfl):
    """8B width, 2 layers, rank 80 (the reading's rank), context 600, B = 16."""
    shape = QWEN3_8B.with_layers(2)
    wt = make_weights_torch(shape, seed=91, device=DEV, gamma="jitter")
    wn = torch_weights_to_np(wt)
    cw = make_conv_weights_np(shape, rank=80, seed=92)
    orc = oracle.OracleDrafter(shape, wn, dtype=np.float32)
    width = shape.n_feat_layers * shape.hidden
    with dfl.Drafter(shape, wt, max_seqs=1, max_batch=1, max_block=16, max_ctx=1024, max_fuse_tokens=1024) as d:
        f = make_features_np(600, width, seed=93)
        d.fuse_ctx([0], [600], bf16_dev(f, DEV), pending=False)
        orc.fuse_ctx([0], [600], f, pending=False)
        d.set_conv(_conv_dev(cw), 80)
        anchors = make_anchor_ids_np(1, shape.vocab, seed=94)
        refs = _ref_conv(orc, _conv_np(cw, np.float32), [0], anchors, 16)
        assert _draft_compare(d, refs, [0], anchors, 16, "8B conv r=80") > 0


def test_set_conv_rejects_bad_arguments(dfl):
    sh = replace(TINY, n_layers=1)
    wn = make_weights_np(sh, seed=95, gamma="jitter", std=0.02)
    cw = make_conv_weights_np(sh, rank=16, seed=96)
    with dfl.Drafter(sh, np_weights_to_device(wn, DEV), max_seqs=1, max_batch=1, max_block=8, max_ctx=256,
                     max_fuse_tokens=256) as d:
        for rank in (0, 12, 136):
            with pytest.raises(dfl.DFlashError):
                d.set_conv(_conv_dev(cw), rank)
