"""8-bit context pages (kv_format 1, the q8_0 block format) on the GPU against
the oracle (oracle/kv_quant.py over the drafter oracle's K/V), through the C
ABI: the stored codes and fp16 scales of every appended token, the decoded
K/V, and drafts over the quantised context (the attention kernel's converter
warps decode the pages into the bf16 tiles its tensor cores read)."""
from dataclasses import replace

import numpy as np
import pytest

import oracle
from oracle import kv_quant as kq
from synth import TINY, QWEN3_8B, make_weights_np, make_features_np, make_anchor_ids_np, make_weights_torch, \
    torch_weights_to_np
from tests.gpu_util import np_weights_to_device, bf16_dev, i32_dev, assert_close, compare_draft, GAP, \
    ROW_REL_HIGH_GAIN

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def dfl():
    import __graft_entry__
    __graft_entry__.build()
    import block_diffusion_drafter_pass_gb300 as m
    return m


def _check_codes(d, orc, s, layers, what):
    """Stored blocks against the format and against the oracle's K/V. The
    library quantises its own K/V, which sit within the K/V tolerance of the
    oracle's (bf16-stored normalised features), so codes are not compared
    bit for bit. Checked: codes in [-127, 127] and every block with a nonzero
    scale reaches +-127 (its largest value maps to 127 exactly); 127 x scale
    (the block maximum, through its fp16 rounding) within the K/V tolerance of
    the oracle's block maximum; codes within one step of the oracle's where
    the scales agree to 1%; decoded values within the K/V tolerance of the
    oracle's decoded values. Returns the number of blocks checked."""
    from tests.gpu_util import ATOL, RTOL
    n = sum(orc.seq_len(s))
    if n == 0:
        return 0
    blocks = 0
    for l in layers:
        kc, ksc, vc, vsc = d.read_kv_q8(l, s, 0, n)
        for name, got_c, got_s, ref in (("K", kc, ksc, orc.seqs[s]["k"][l][:n]), ("V", vc, vsc, orc.seqs[s]["v"][l][:n])):
            gc = got_c.astype(np.int32).reshape(got_c.shape[:-1] + (-1, 32))
            assert np.abs(gc).max() <= 127, f"{what} {name} layer {l}: code outside [-127, 127]"
            nz = got_s > 0
            np.testing.assert_array_equal(np.abs(gc).max(-1)[nz], 127, err_msg=f"{what} {name} layer {l}: block max")
            amax = np.abs(ref).reshape(ref.shape[:-1] + (-1, 32)).max(-1)
            excess = np.abs(127.0 * got_s - amax) - (ATOL + RTOL * amax)
            assert excess.max() <= 0, f"{what} {name} layer {l}: block maximum off by {excess.max() + ATOL:.3g}"
            rq, rs = kq.quantize(ref)
            close = np.abs(got_s - rs.astype(np.float32)) <= 1e-2 * np.maximum(rs.astype(np.float32), 1e-30)
            dq = np.abs(gc - rq.astype(np.int32).reshape(gc.shape))
            assert dq[close].max() <= 1, f"{what} {name} layer {l}: codes off by {dq[close].max()}"
            blocks += int(nz.sum())
        k, v = d.read_kv(l, s, 0, n)
        assert_close(k, kq.roundtrip(orc.seqs[s]["k"][l][:n]), f"{what} decoded K layer {l}")
        assert_close(v, kq.roundtrip(orc.seqs[s]["v"][l][:n]), f"{what} decoded V layer {l}")
    return blocks


def _compare_q8(got_ids, hid, top, ref_q, ref_x, B, what, row_rel=None):
    """A draft over 8-bit context pages against the oracle's pass over its
    own quantised context (ref_q). The library quantises its own K/V, within
    the K/V tolerance of the oracle's, so near a rounding boundary the two
    land a step apart; the effect of such steps is bounded by the effect of
    quantising at all, which the oracle measures on the same inputs (ref_q
    against the exact pass ref_x). So each bound is the stated one plus that
    effect: row L2 2e-2 + |ref_q - ref_x| / |ref_x| for the residual stream;
    logit tolerance + max |logits_q - logits_x| of the row for the winning
    logits and the near-top check; ids bit-exact where the oracle's gap
    exceeds 0.1 + twice that logit effect."""
    from tests.gpu_util import HID_REL_L2, RTOL, ATOL, logit_tol
    got = np.asarray(hid, dtype=np.float64)
    hq, hx = np.asarray(ref_q["hidden"]), np.asarray(ref_x["hidden"])
    q8_h = np.linalg.norm(hq - hx, axis=-1) / np.maximum(np.linalg.norm(hx, axis=-1), 1e-30)
    rel = np.linalg.norm(got - hq, axis=-1) / np.maximum(np.linalg.norm(hq, axis=-1), 1e-30)
    assert (rel <= HID_REL_L2 + q8_h).all(), (
        f"{what}: row relative L2 {rel.max():.4g} above {HID_REL_L2} + the quantisation effect {q8_h.max():.4g}")
    if B == 1:
        return 0
    lq, lx = np.asarray(ref_q["logits"]), np.asarray(ref_x["logits"])
    q8_l = np.abs(lq - lx).max(axis=-1)
    tol = logit_tol(ref_q["top1"], row_rel) + q8_l
    assert (np.abs(np.asarray(top, dtype=np.float64) - ref_q["top1"]) <= tol).all(), f"{what}: winning logits"
    ids = np.asarray(got_ids, dtype=np.int64)
    sure = ref_q["gap"] > GAP + 2 * q8_l
    np.testing.assert_array_equal(ids[sure], ref_q["draft"][sure], err_msg=f"{what}: draft ids")
    at_id = lq[np.arange(len(ids)), ids]
    assert (at_id >= ref_q["top1"] - 2 * tol).all(), f"{what}: a draft id far below the top logit"
    return int(sure.sum())


def _draft_q8(d, orc, seqs, anchors, B, what, row_rel=None):
    import oracle.dflash_oracle as od
    ids = d.draft(seqs, i32_dev(anchors, DEV), B)
    d.sync()
    hid, top = d.last_draft(len(seqs), B)
    got = ids.cpu().numpy()
    checked = 0
    for i, s in enumerate(seqs):
        kc = [orc.context(s, l)[0] for l in range(orc.shape.n_layers)]
        vc = [orc.context(s, l)[1] for l in range(orc.shape.n_layers)]
        ref_q = kq.draft_block_quantized_ctx(orc.w, orc.shape, int(anchors[i]), kc, vc, B)
        ref_x = od.draft_block(orc.w, orc.shape, int(anchors[i]), kc, vc, B)
        checked += _compare_q8(got[i] if B > 1 else [], hid[i * B:(i + 1) * B], top[i * (B - 1):(i + 1) * (B - 1)],
                               ref_q, ref_x, B, f"{what} seq {s}", row_rel=row_rel)
    return checked


def test_tiny_q8_pages_codes_and_drafts(dfl):
    """Tiny drafter (d = 64): contexts appended in ragged chunks (odd and even
    first slots, page crossings), the stored blocks of every token, drafts at
    B = 4, 8, 16 over the quantised context, then a pending append, verify
    and commit, and a draft over the committed context."""
    sh = TINY
    wn = make_weights_np(sh, seed=401, gamma="jitter", std=0.05)
    orc = oracle.OracleDrafter(sh, wn)
    width = sh.n_feat_layers * sh.hidden
    with dfl.Drafter(sh, np_weights_to_device(wn, DEV), max_seqs=3, max_batch=3, max_block=16, max_ctx=1024,
                     max_fuse_tokens=512, kv_format=1) as d:
        seed = 402
        for s, chunks in {0: [64, 37], 1: [5, 130, 1], 2: [200]}.items():
            for n in chunks:
                f = make_features_np(n, width, seed=seed)
                seed += 1
                d.fuse_ctx([s], [n], bf16_dev(f, DEV), pending=False)
                orc.fuse_ctx([s], [n], f, pending=False)
        d.sync()
        blocks = sum(_check_codes(d, orc, s, range(sh.n_layers), f"seq {s}") for s in (0, 1, 2))
        assert blocks > 1000
        anchors = make_anchor_ids_np(3, sh.vocab, seed=410)
        total = 0
        for B in (4, 8, 16):
            total += _draft_q8(d, orc, [0, 1, 2], anchors, B, f"q8 B={B}")
        assert total > 0
        # a pending block, verify (commit tau of it), then draft
        B = 8
        f = make_features_np(3 * B, width, seed=420)
        d.fuse_ctx([0, 1, 2], [B] * 3, bf16_dev(f, DEV), pending=True)
        orc.fuse_ctx([0, 1, 2], [B] * 3, f, pending=True)
        rng = np.random.Generator(np.random.PCG64(421))
        drafts = rng.integers(0, sh.vocab, size=(3, B - 1)).astype(np.int32)
        targets = rng.integers(0, sh.vocab, size=(3, B)).astype(np.int32)
        targets[0, :3] = drafts[0, :3]   # seq 0 accepts three drafts
        tau, bonus = d.verify([0, 1, 2], B, i32_dev(drafts, DEV), i32_dev(targets, DEV))
        rt, rb = orc.verify([0, 1, 2], B, drafts, targets)
        d.sync()
        np.testing.assert_array_equal(tau.cpu().numpy(), rt)
        for s in (0, 1, 2):
            assert d.seq_len(s) == orc.seq_len(s)
            _check_codes(d, orc, s, range(sh.n_layers), f"after verify seq {s}")
        _draft_q8(d, orc, [0, 1, 2], rb.astype(np.int32), 16, "q8 after commit")


def test_q8_mqa_long_context_many_chunks(dfl):
    """One key/value head of d = 128 over 6000 tokens: the attention work is
    split into many chunks, every context unit decoded by the converter warps
    from its raw 8-bit region (d = 128 layout), the combine takes its general
    path."""
    sh = replace(TINY, n_heads=2, n_kv_heads=1, head_dim=128)
    wn = make_weights_np(sh, seed=431, gamma="jitter", std=0.05)
    orc = oracle.OracleDrafter(sh, wn)
    width = sh.n_feat_layers * sh.hidden
    with dfl.Drafter(sh, np_weights_to_device(wn, DEV), max_seqs=2, max_batch=2, max_block=16, max_ctx=6400,
                     max_fuse_tokens=2048, kv_format=1) as d:
        for part, n in enumerate((2000, 2000, 1700, 300)):
            f = make_features_np(n, width, seed=432 + part)
            d.fuse_ctx([0], [n], bf16_dev(f, DEV), pending=False)
            orc.fuse_ctx([0], [n], f, pending=False)
        f = make_features_np(77, width, seed=439)
        d.fuse_ctx([1], [77], bf16_dev(f, DEV), pending=False)
        orc.fuse_ctx([1], [77], f, pending=False)
        d.sync()
        _check_codes(d, orc, 1, [0], "short seq")
        kc, ksc, vc, vsc = d.read_kv_q8(0, 0, 5000, 64)
        assert np.abs(kc.astype(np.int32).reshape(64, 1, 4, 32)).max(-1).min() == 127
        anchors = make_anchor_ids_np(2, sh.vocab, seed=440)
        assert _draft_q8(d, orc, [0, 1], anchors, 16, "q8 MQA C=6000", ROW_REL_HIGH_GAIN) > 0


def test_qwen3_8b_width_q8_two_layers(dfl):
    """8B width, 2 layers, 8 kv heads of d = 128: a 1000-token context in
    8-bit pages (blocks sampled at page and chunk boundaries), drafts at
    B = 16 and 8."""
    shape = QWEN3_8B.with_layers(2)
    wt = make_weights_torch(shape, seed=451, device=DEV, gamma="jitter")
    wn = torch_weights_to_np(wt)
    orc = oracle.OracleDrafter(shape, wn, dtype=np.float32)
    width = shape.n_feat_layers * shape.hidden
    with dfl.Drafter(shape, wt, max_seqs=2, max_batch=2, max_block=16, max_ctx=2048, max_fuse_tokens=1024,
                     kv_format=1) as d:
        f = make_features_np(1300, width, seed=452)
        d.fuse_ctx([0, 1], [300, 700], bf16_dev(f[:1000], DEV), pending=False)
        orc.fuse_ctx([0, 1], [300, 700], f[:1000], pending=False)
        d.fuse_ctx([1], [300], bf16_dev(f[1000:], DEV), pending=False)
        orc.fuse_ctx([1], [300], f[1000:], pending=False)
        d.sync()
        for s, p0 in ((0, 0), (0, 250), (1, 640), (1, 960)):
            for l in (0, 1):
                kc, ksc, vc, vsc = d.read_kv_q8(l, s, p0, 40)
                for got, ref in ((kc, orc.seqs[s]["k"][l][p0:p0 + 40]), (vc, orc.seqs[s]["v"][l][p0:p0 + 40])):
                    g = got.astype(np.int32).reshape(40, 8, 4, 32)
                    assert (np.abs(g).max(-1) == 127).all()
        anchors = make_anchor_ids_np(2, shape.vocab, seed=453)
        total = 0
        for B in (16, 8):
            total += _draft_q8(d, orc, [0, 1], anchors, B, f"8B q8 B={B}")
        assert total > 0


def test_q8_long_positions_262144(dfl):
    """The longest configuration in 8-bit pages: 262144 injected tokens, one
    key/value head of d = 128 at tiny width (the fp64 oracle holds the whole
    cache). Every stored block of the context is checked against the format
    and the oracle's blocks (RoPE angles up to 2.6e5 rad before quantising),
    then drafts at B = 8, 16 and 32 over the whole quantised context: 4096
    context units per pass through the raw loader's slots and the converter
    warps, thousands of chunks in the combine."""
    sh = replace(TINY, n_heads=2, n_kv_heads=1, head_dim=128)
    wn = make_weights_np(sh, seed=461, gamma="jitter", std=0.05)
    orc = oracle.OracleDrafter(sh, wn)
    width = sh.n_feat_layers * sh.hidden
    C, chunk = 262144, 32768
    with dfl.Drafter(sh, np_weights_to_device(wn, DEV), max_seqs=1, max_batch=1, max_block=32, max_ctx=C + 64,
                     max_fuse_tokens=chunk, kv_format=1) as d:
        for i in range(C // chunk):
            f = make_features_np(chunk, width, seed=462 + i)
            d.fuse_ctx([0], [chunk], bf16_dev(f, DEV), pending=False)
            orc.fuse_ctx([0], [chunk], f, pending=False)
            del f
        d.sync()
        assert d.seq_len(0) == (C, 0)
        assert _check_codes(d, orc, 0, [0], "C=262144") == 2 * C * 4
        anchors = make_anchor_ids_np(1, sh.vocab, seed=470)
        # every row: residual stream, winning logit and the near-top check;
        # at this length the oracle's own quantisation effect on the logits
        # puts the id-exact threshold (0.1 + twice that effect) above every
        # row's top-1/top-2 gap, so no row is required to match bit for bit
        for B in (8, 16, 32):
            _draft_q8(d, orc, [0], anchors, B, f"q8 C=262144 B={B}", ROW_REL_HIGH_GAIN)
