"""CUDA path against the CPU oracle through the C ABI.

Tiny drafter (oracle in fp64): cached K/V after fusion, draft ids / residual
stream / winning logits, verify + commit + rollback over several cycles,
ragged and empty contexts, B = 1..8, several sequences per call.
Qwen3-8B-shaped drafter (oracle in fp32): reduced depth at ragged contexts,
and the full 5-layer pass at context 4096, B = 16 (the benchmarked shape).
"""
import numpy as np
import pytest

import oracle
from synth import (TINY, QWEN3_8B, make_weights_np, make_features_np, make_anchor_ids_np,
                   make_weights_torch, torch_weights_to_np)
from tests.gpu_util import (np_weights_to_device, bf16_dev, i32_dev, assert_close, compare_draft, GAP,
                            ROW_REL_HIGH_GAIN)
from tests.emulate import bf16_context, bf16_storage_hidden

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def dfl():
    import __graft_entry__
    __graft_entry__.build()
    import block_diffusion_drafter_pass_gb300 as m
    return m


def _check_kv(d, orc, seqs, layers, what, row_rel=None):
    for s in seqs:
        n = orc.seq_len(s)[0] + orc.seq_len(s)[1]
        if n == 0:
            continue
        st = orc.seqs[s]
        for l in layers:
            k, v = d.read_kv(l, s, 0, n)
            assert_close(k, st["k"][l][:n], f"{what}: K layer {l} seq {s}", row_rel=row_rel)
            assert_close(v, st["v"][l][:n], f"{what}: V layer {l} seq {s}", row_rel=row_rel)


def _draft_and_compare(d, orc, seqs, anchors, B, what, row_rel=None):
    ids = d.draft(seqs, i32_dev(anchors, DEV), B)
    d.sync()
    ref = orc.draft(seqs, anchors, B)
    hid, top = d.last_draft(len(seqs), B)
    got = ids.cpu().numpy()
    checked = 0
    for i in range(len(seqs)):
        checked += compare_draft(got[i] if B > 1 else [], hid[i * B:(i + 1) * B],
                                 top[i * (B - 1):(i + 1) * (B - 1)], ref[i], B, f"{what} seq {seqs[i]}",
                                 row_rel=row_rel)
    return got, ref, checked


@pytest.mark.parametrize("std", [0.02, 0.1])
def test_tiny_fuse_draft_parity(dfl, std):
    row_rel = None if std == 0.02 else ROW_REL_HIGH_GAIN
    sh = TINY
    wn = make_weights_np(sh, seed=21, gamma="jitter", std=std)
    orc = oracle.OracleDrafter(sh, wn)
    width = sh.n_feat_layers * sh.hidden
    with dfl.Drafter(sh, np_weights_to_device(wn, DEV), max_seqs=6, max_batch=4, max_block=8, max_ctx=512,
                     max_fuse_tokens=512) as d:
        # seq 0: one full page; seq 1: ragged; seq 2: empty; seq 3: three chunks crossing pages
        plan = {0: [64], 1: [100], 2: [], 3: [30, 70, 100]}
        rng_seed = 100
        for s, chunks in plan.items():
            for n in chunks:
                f = make_features_np(n, width, seed=rng_seed)
                rng_seed += 1
                d.fuse_ctx([s], [n], bf16_dev(f, DEV), pending=False)
                orc.fuse_ctx([s], [n], f, pending=False)
        d.sync()
        _check_kv(d, orc, [0, 1, 3], range(sh.n_layers), "tiny fuse", row_rel)
        seqs = [0, 1, 2, 3]
        anchors = make_anchor_ids_np(4, sh.vocab, seed=7)
        total = 0
        for B in (4, 1, 2, 8):
            _, _, c = _draft_and_compare(d, orc, seqs, anchors, B, f"tiny std={std} B={B}", row_rel)
            total += c
        # a multi-sequence fuse call with rows grouped per sequence
        f = make_features_np(3 + 5, width, seed=999)
        d.fuse_ctx([2, 1], [3, 5], bf16_dev(f, DEV), pending=False)
        orc.fuse_ctx([2, 1], [3, 5], f, pending=False)
        _check_kv(d, orc, [1, 2], range(sh.n_layers), "tiny multi-seq fuse", row_rel)
        _, _, c = _draft_and_compare(d, orc, [2, 1], anchors[:2], 4, "tiny after multi-seq fuse", row_rel)
        total += c
        assert total > 0


def test_tiny_speculative_cycles_commit_and_rollback(dfl):
    """Draft -> fuse the block's features as pending -> verify against target
    ids that agree for a seeded number of positions -> commit tau, roll back
    the rest; repeated, with the caches compared after every cycle."""
    sh = TINY
    wn = make_weights_np(sh, seed=31, gamma="jitter", std=0.1)
    orc = oracle.OracleDrafter(sh, wn)
    width = sh.n_feat_layers * sh.hidden
    B = 6
    seqs = [0, 1, 2]
    rng = np.random.Generator(np.random.PCG64(32))
    with dfl.Drafter(sh, np_weights_to_device(wn, DEV), max_seqs=3, max_batch=3, max_block=B, max_ctx=1024,
                     max_fuse_tokens=512) as d:
        ctx = [70, 5, 128]
        f = make_features_np(sum(ctx), width, seed=33)
        d.fuse_ctx(seqs, ctx, bf16_dev(f, DEV), pending=False)
        orc.fuse_ctx(seqs, ctx, f, pending=False)
        anchors = make_anchor_ids_np(3, sh.vocab, seed=34)
        taus = []
        for cyc in range(6):
            got, ref, _ = _draft_and_compare(d, orc, seqs, anchors, B, f"cycle {cyc}", ROW_REL_HIGH_GAIN)
            drafts = np.stack([r["draft"] for r in ref]).astype(np.int32)
            # targets agree with the oracle's drafts for m positions, then differ
            t = rng.integers(0, sh.vocab, size=(3, B)).astype(np.int32)
            for i in range(3):
                m = int(rng.integers(0, B))
                t[i, :m] = drafts[i, :m]
                if m < B - 1:
                    t[i, m] = (drafts[i, m] + 1) % sh.vocab
            fb = make_features_np(3 * B, width, seed=200 + cyc)
            d.fuse_ctx(seqs, [B] * 3, bf16_dev(fb, DEV), pending=True)
            orc.fuse_ctx(seqs, [B] * 3, fb, pending=True)
            tau, bonus = d.verify(seqs, B, i32_dev(drafts, DEV), i32_dev(t, DEV))
            rt, rb = orc.verify(seqs, B, drafts, t)
            d.sync()
            np.testing.assert_array_equal(tau.cpu().numpy(), rt)
            np.testing.assert_array_equal(bonus.cpu().numpy(), rb)
            taus += list(rt)
            for s in seqs:
                assert d.seq_len(s) == orc.seq_len(s)
            _check_kv(d, orc, seqs, [0], f"cycle {cyc}", ROW_REL_HIGH_GAIN)
            anchors = rb.astype(np.int32)
        assert max(taus) > 1 and min(taus) < B


def _big_setup(n_layers, seed):
    shape = QWEN3_8B.with_layers(n_layers)
    wt = make_weights_torch(shape, seed=seed, device=DEV, gamma="jitter")
    wn = torch_weights_to_np(wt)
    return shape, wt, wn


def test_qwen3_8b_shape_two_layers_ragged(dfl):
    """8B width, 2 layers: two sequences with ragged contexts (300 and 1000
    tokens, appended in uneven chunks), B = 16 and B = 8."""
    shape, wt, wn = _big_setup(2, seed=41)
    orc = oracle.OracleDrafter(shape, wn, dtype=np.float32)
    width = shape.n_feat_layers * shape.hidden
    with dfl.Drafter(shape, wt, max_seqs=2, max_batch=2, max_block=16, max_ctx=2048,
                     max_fuse_tokens=1024) as d:
        f = make_features_np(1300, width, seed=42)
        d.fuse_ctx([0, 1], [300, 700], bf16_dev(f[:1000], DEV), pending=False)
        orc.fuse_ctx([0, 1], [300, 700], f[:1000], pending=False)
        d.fuse_ctx([1], [300], bf16_dev(f[1000:], DEV), pending=False)
        orc.fuse_ctx([1], [300], f[1000:], pending=False)
        d.sync()
        for s in (0, 1):
            n = orc.seq_len(s)[0]
            for l in range(2):
                k, v = d.read_kv(l, s, 0, n)
                kr, vr = orc.context(s, l)
                assert_close(k, kr, f"8B K layer {l} seq {s}")
                assert_close(v, vr, f"8B V layer {l} seq {s}")
        anchors = make_anchor_ids_np(2, shape.vocab, seed=43)
        for B in (16, 8):
            _, _, checked = _draft_and_compare(d, orc, [0, 1], anchors, B, f"8B 2-layer B={B}")
            assert checked > 0


def test_qwen3_8b_full_depth_context_4096(dfl):
    """The benchmarked workload: 5 layers, batch 1, context 4096, B = 16."""
    shape, wt, wn = _big_setup(5, seed=0)
    orc = oracle.OracleDrafter(shape, wn, dtype=np.float32)
    width = shape.n_feat_layers * shape.hidden
    with dfl.Drafter(shape, wt, max_seqs=1, max_batch=1, max_block=16, max_ctx=4096 + 64,
                     max_fuse_tokens=4096) as d:
        f = make_features_np(4096, width, seed=1)
        d.fuse_ctx([0], [4096], bf16_dev(f, DEV), pending=False)
        orc.fuse_ctx([0], [4096], f, pending=False)
        d.sync()
        # sampled cache rows: first, page boundaries, last
        for l in (0, 4):
            for p0 in (0, 63, 64, 2047, 4095):
                k, v = d.read_kv(l, 0, p0, 1)
                st = orc.seqs[0]
                assert_close(k, st["k"][l][p0:p0 + 1], f"8B K layer {l} pos {p0}")
                assert_close(v, st["v"][l][p0:p0 + 1], f"8B V layer {l} pos {p0}")
        anchors = make_anchor_ids_np(1, shape.vocab, seed=2)
        ids = d.draft([0], i32_dev(anchors, DEV), 16)
        d.sync()
        ref = orc.draft([0], anchors, 16)[0]
        hid, top = d.last_draft(1, 16)
    # five layers of bf16 storage move single elements past the 2-layer guard;
    # hold the kernels to what an exact bf16-storage pass of the same inputs does
    kb, vb = bf16_context(wn, shape, f, dtype=np.float32)
    emu = bf16_storage_hidden(wn, shape, int(anchors[0]), kb, vb, 16, dtype=np.float32)
    checked = compare_draft(ids.cpu().numpy()[0], hid, top, ref, 16, "8B full depth C=4096", emu_hidden=emu)
    assert checked >= 5, f"only {checked} rows with gap > {GAP}"


@pytest.mark.parametrize("n_heads,n_kv,blocks", [(8, 2, (32, 16, 5)), (6, 2, (32, 8, 1))])
def test_gqa_group_layouts(dfl, n_heads, n_kv, blocks):
    """Query-row layouts of the attention kernel: G*B = 128 and 96 (one thread
    per row, row r in TMEM lane r), G*B <= 64 (rows spread 16 per TMEM lane
    quarter, two threads per row), for G = 4 and G = 3, B = 1 .. 32."""
    from dataclasses import replace
    sh = replace(TINY, n_heads=n_heads, n_kv_heads=n_kv)
    wn = make_weights_np(sh, seed=51, gamma="jitter", std=0.05)
    orc = oracle.OracleDrafter(sh, wn)
    width = sh.n_feat_layers * sh.hidden
    with dfl.Drafter(sh, np_weights_to_device(wn, DEV), max_seqs=3, max_batch=3, max_block=32, max_ctx=1024,
                     max_fuse_tokens=512) as d:
        ctx = [200, 64, 7]
        f = make_features_np(sum(ctx), width, seed=52)
        d.fuse_ctx([0, 1, 2], ctx, bf16_dev(f, DEV), pending=False)
        orc.fuse_ctx([0, 1, 2], ctx, f, pending=False)
        anchors = make_anchor_ids_np(3, sh.vocab, seed=53)
        total = 0
        for B in blocks:
            _, _, c = _draft_and_compare(d, orc, [0, 1, 2], anchors, B, f"G={n_heads // n_kv} B={B}",
                                         ROW_REL_HIGH_GAIN)
            total += c
        assert total > 0


def test_tiny_batch16_cluster_split(dfl):
    """16 sequences x B = 16 (256 block tokens) and a 256-row fuse: every
    projection (fuse, QKV with RoPE, O and down with the residual, gate/up
    with SwiGLU and an odd weight-tile count, LM head with argmax) runs as
    clusters of two CTA pairs (cta_group::2 MMAs), each pair over half of the
    k-blocks, exchanging half sums through distributed shared memory."""
    sh = TINY
    wn = make_weights_np(sh, seed=81, gamma="jitter", std=0.05)
    orc = oracle.OracleDrafter(sh, wn)
    width = sh.n_feat_layers * sh.hidden
    n = 16
    with dfl.Drafter(sh, np_weights_to_device(wn, DEV), max_seqs=n, max_batch=n, max_block=16, max_ctx=1024,
                     max_fuse_tokens=512) as d:
        rng = np.random.default_rng(82)
        lens = rng.integers(1, 300, size=n)
        for s in range(n):
            f = make_features_np(int(lens[s]), width, seed=83 + s)
            d.fuse_ctx([s], [int(lens[s])], bf16_dev(f, DEV), pending=False)
            orc.fuse_ctx([s], [int(lens[s])], f, pending=False)
        # one fuse call of 16 rows per sequence: M = 256
        f = make_features_np(16 * n, width, seed=99)
        d.fuse_ctx(list(range(n)), [16] * n, bf16_dev(f, DEV), pending=False)
        orc.fuse_ctx(list(range(n)), [16] * n, f, pending=False)
        d.sync()
        _check_kv(d, orc, range(n), range(sh.n_layers), "tiny 256-row fuse", ROW_REL_HIGH_GAIN)
        anchors = make_anchor_ids_np(n, sh.vocab, seed=100)
        total = 0
        for B in (16, 8):
            _, _, c = _draft_and_compare(d, orc, list(range(n)), anchors, B, f"tiny batch {n} B={B}",
                                         ROW_REL_HIGH_GAIN)
            total += c
        assert total > 0


def test_qwen3_8b_batch16_two_layers(dfl):
    """8B width, 2 layers, 16 sequences x B = 16 = 256 block tokens: QKV, O,
    down and the 256-row fuse run as clusters of two CTA pairs splitting the
    k-blocks at full width; gate/up and the LM head run as CTA pairs over
    whole pair tiles."""
    shape, wt, wn = _big_setup(2, seed=91)
    orc = oracle.OracleDrafter(shape, wn, dtype=np.float32)
    width = shape.n_feat_layers * shape.hidden
    n = 16
    with dfl.Drafter(shape, wt, max_seqs=n, max_batch=n, max_block=16, max_ctx=512,
                     max_fuse_tokens=4096) as d:
        rng = np.random.default_rng(92)
        lens = [int(x) for x in rng.integers(16, 240, size=n)]
        f = make_features_np(sum(lens), width, seed=93)
        d.fuse_ctx(list(range(n)), lens, bf16_dev(f, DEV), pending=False)
        orc.fuse_ctx(list(range(n)), lens, f, pending=False)
        f = make_features_np(16 * n, width, seed=94)
        d.fuse_ctx(list(range(n)), [16] * n, bf16_dev(f, DEV), pending=False)
        orc.fuse_ctx(list(range(n)), [16] * n, f, pending=False)
        d.sync()
        for s in (0, 7, 15):
            m = orc.seq_len(s)[0]
            for l in range(2):
                k, v = d.read_kv(l, s, 0, m)
                kr, vr = orc.context(s, l)
                assert_close(k, kr, f"8B batch {n} K layer {l} seq {s}")
                assert_close(v, vr, f"8B batch {n} V layer {l} seq {s}")
        anchors = make_anchor_ids_np(n, shape.vocab, seed=95)
        _, _, checked = _draft_and_compare(d, orc, list(range(n)), anchors, 16, f"8B 2-layer batch {n}")
        assert checked > 0


def test_qwen3_8b_batch32_two_layers(dfl):
    """8B width, 2 layers, 32 sequences x B = 16 = 512 block tokens: QKV
    (RoPE), gate/up (SwiGLU) and the LM head (argmax over 1187 weight tiles,
    an odd count) run as CTA pairs issuing cta_group::2 MMAs over whole pair
    tiles; O, down and the fuse run as clusters of two pairs splitting the
    k-blocks."""
    shape, wt, wn = _big_setup(2, seed=101)
    orc = oracle.OracleDrafter(shape, wn, dtype=np.float32)
    width = shape.n_feat_layers * shape.hidden
    n = 32
    with dfl.Drafter(shape, wt, max_seqs=n, max_batch=n, max_block=16, max_ctx=256,
                     max_fuse_tokens=4096) as d:
        rng = np.random.default_rng(102)
        lens = [int(x) for x in rng.integers(16, 96, size=n)]
        f = make_features_np(sum(lens), width, seed=103)
        d.fuse_ctx(list(range(n)), lens, bf16_dev(f, DEV), pending=False)
        orc.fuse_ctx(list(range(n)), lens, f, pending=False)
        f = make_features_np(16 * n, width, seed=104)
        d.fuse_ctx(list(range(n)), [16] * n, bf16_dev(f, DEV), pending=False)
        orc.fuse_ctx(list(range(n)), [16] * n, f, pending=False)
        d.sync()
        for s in (0, 31):
            m = orc.seq_len(s)[0]
            for l in range(2):
                k, v = d.read_kv(l, s, 0, m)
                kr, vr = orc.context(s, l)
                assert_close(k, kr, f"8B batch {n} K layer {l} seq {s}")
                assert_close(v, vr, f"8B batch {n} V layer {l} seq {s}")
        anchors = make_anchor_ids_np(n, shape.vocab, seed=105)
        _, _, checked = _draft_and_compare(d, orc, list(range(n)), anchors, 16, f"8B 2-layer batch {n}")
        assert checked > 0


def test_mqa_long_context_many_chunks(dfl):
    """One key/value head (d = 128, two query heads) over a 6000-token
    context: the attention work is split into 2-unit chunks (94 pages plus the
    block per row on 152 SMs), so one (sequence, head) row has 48 chunk
    partials and the combine kernel takes its general path (more than 32
    chunks, weights recomputed per chunk). A second, short sequence shares the
    call."""
    from dataclasses import replace
    sh = replace(TINY, n_heads=2, n_kv_heads=1, head_dim=128)
    wn = make_weights_np(sh, seed=71, gamma="jitter", std=0.05)
    orc = oracle.OracleDrafter(sh, wn)
    width = sh.n_feat_layers * sh.hidden
    with dfl.Drafter(sh, np_weights_to_device(wn, DEV), max_seqs=2, max_batch=2, max_block=16, max_ctx=6400,
                     max_fuse_tokens=2048) as d:
        for part, n in enumerate((2000, 2000, 1700, 300)):
            f = make_features_np(n, width, seed=72 + part)
            d.fuse_ctx([0], [n], bf16_dev(f, DEV), pending=False)
            orc.fuse_ctx([0], [n], f, pending=False)
        f = make_features_np(300, width, seed=79)
        d.fuse_ctx([1], [300], bf16_dev(f, DEV), pending=False)
        orc.fuse_ctx([1], [300], f, pending=False)
        assert orc.seq_len(0)[0] == 6000
        anchors = make_anchor_ids_np(2, sh.vocab, seed=80)
        _, _, c = _draft_and_compare(d, orc, [0, 1], anchors, 16, "MQA C=6000", ROW_REL_HIGH_GAIN)
        assert c > 0


def test_draft_is_bit_reproducible(dfl):
    """Repeated drafts over the same cache give bit-identical ids, logits and
    residual streams: split GEMM tiles are summed in a fixed order, whichever
    CTA finishes them (8B width, 2 layers, batch 1, so the projections run
    stream-K with tiles split over several CTAs)."""
    shape, wt, _ = _big_setup(2, seed=61)
    width = shape.n_feat_layers * shape.hidden
    with dfl.Drafter(shape, wt, max_seqs=1, max_batch=1, max_block=16, max_ctx=1024 + 64,
                     max_fuse_tokens=1024) as d:
        d.fuse_ctx([0], [1000], bf16_dev(make_features_np(1000, width, seed=62), DEV), pending=False)
        anchors = i32_dev(make_anchor_ids_np(1, shape.vocab, seed=63), DEV)
        first = None
        for _ in range(8):
            ids = d.draft([0], anchors, 16)
            d.sync()
            hid, top = d.last_draft(1, 16)
            cur = (ids.cpu().numpy().copy(), np.asarray(hid).copy(), np.asarray(top).copy())
            if first is None:
                first = cur
                continue
            for a, b in zip(cur, first):
                np.testing.assert_array_equal(a, b)


# ----------------------------------------------------------------------------
# The long-context, 32K and serving-batch configurations
# ----------------------------------------------------------------------------

def test_long_positions_262144(dfl):
    """A context of 262144 injected tokens (the longest configuration): one
    key/value head of d = 128 at tiny width, so the fp64 oracle holds the whole
    cache. K/V are compared at positions around 2^17 and up to 2^18 - 1, where
    RoPE angles reach 2.6e5 rad (the library's fp64-built table), and the
    draft over the whole context at B = 8, 16 and 32."""
    from dataclasses import replace
    sh = replace(TINY, n_heads=2, n_kv_heads=1, head_dim=128)
    wn = make_weights_np(sh, seed=111, gamma="jitter", std=0.05)
    orc = oracle.OracleDrafter(sh, wn)
    width = sh.n_feat_layers * sh.hidden
    C, chunk = 262144, 32768
    with dfl.Drafter(sh, np_weights_to_device(wn, DEV), max_seqs=1, max_batch=1, max_block=32,
                     max_ctx=C + 64, max_fuse_tokens=chunk) as d:
        for i in range(C // chunk):
            f = make_features_np(chunk, width, seed=112 + i)
            d.fuse_ctx([0], [chunk], bf16_dev(f, DEV), pending=False)
            orc.fuse_ctx([0], [chunk], f, pending=False)
            del f
        d.sync()
        assert d.seq_len(0) == (C, 0)
        st = orc.seqs[0]
        for p in (0, 63, 131071, 131072, 131073, 200001, 262080, 262143):
            k, v = d.read_kv(0, 0, p, 1)
            assert_close(k, st["k"][0][p:p + 1], f"K pos {p}", row_rel=ROW_REL_HIGH_GAIN)
            assert_close(v, st["v"][0][p:p + 1], f"V pos {p}", row_rel=ROW_REL_HIGH_GAIN)
        anchors = make_anchor_ids_np(1, sh.vocab, seed=120)
        total = 0
        for B in (8, 16, 32):
            _, _, c = _draft_and_compare(d, orc, [0], anchors, B, f"C=262144 B={B}", ROW_REL_HIGH_GAIN)
            total += c
        assert total > 0


def test_qwen3_8b_context_32768_two_layers(dfl):
    """Batch 1 at context 32768 (the context of the bandwidth target) at the
    8B width: 5 fused target layers, 2 drafter layers, the context appended in
    4096-token chunks; K/V at page and chunk boundaries, then the B = 16 draft."""
    shape, wt, wn = _big_setup(2, seed=131)
    orc = oracle.OracleDrafter(shape, wn, dtype=np.float32)
    width = shape.n_feat_layers * shape.hidden
    C, chunk = 32768, 4096
    with dfl.Drafter(shape, wt, max_seqs=1, max_batch=1, max_block=16, max_ctx=C + 64,
                     max_fuse_tokens=chunk) as d:
        for i in range(C // chunk):
            f = make_features_np(chunk, width, seed=132 + i)
            d.fuse_ctx([0], [chunk], bf16_dev(f, DEV), pending=False)
            orc.fuse_ctx([0], [chunk], f, pending=False)
            del f
        d.sync()
        st = orc.seqs[0]
        for l in (0, 1):
            for p in (0, 4095, 4096, 16383, 16384, 32767):
                k, v = d.read_kv(l, 0, p, 1)
                assert_close(k, st["k"][l][p:p + 1], f"8B C=32768 K layer {l} pos {p}")
                assert_close(v, st["v"][l][p:p + 1], f"8B C=32768 V layer {l} pos {p}")
        anchors = make_anchor_ids_np(1, shape.vocab, seed=140)
        _, _, checked = _draft_and_compare(d, orc, [0], anchors, 16, "8B 2-layer C=32768")
        assert checked > 0


def test_qwen3_8b_batch32_serving_lengths(dfl):
    """The serving batch: 32 sequences with contexts uniform in [1024, 8192]
    (the benchmark's seeded lengths), B = 16, at the 8B width with 2 drafter
    layers (one fused target layer keeps the host oracle's fusion short; the
    drafter side is the benchmarked one). The attention work is dealt largest
    first over several chunks per CTA at these lengths."""
    from dataclasses import replace
    from synth import make_serving_lengths
    shape = replace(QWEN3_8B.with_layers(2), n_feat_layers=1)
    wt = make_weights_torch(shape, seed=151, device=DEV, gamma="jitter")
    wn = torch_weights_to_np(wt)
    orc = oracle.OracleDrafter(shape, wn, dtype=np.float32)
    width = shape.n_feat_layers * shape.hidden
    n = 32
    lens = [int(x) for x in make_serving_lengths(n, 1024, 8192, seed=0)]
    with dfl.Drafter(shape, wt, max_seqs=n, max_batch=n, max_block=16, max_ctx=8192 + 64,
                     max_fuse_tokens=8192) as d:
        for s in range(n):
            f = make_features_np(lens[s], width, seed=152 + s)
            d.fuse_ctx([s], [lens[s]], bf16_dev(f, DEV), pending=False)
            orc.fuse_ctx([s], [lens[s]], f, pending=False)
            del f
        d.sync()
        for s in (0, 13, 31):
            st = orc.seqs[s]
            m = lens[s]
            for l in (0, 1):
                for p in (0, 63, 64, m // 2, m - 1):
                    k, v = d.read_kv(l, s, p, 1)
                    assert_close(k, st["k"][l][p:p + 1], f"batch 32 K seq {s} layer {l} pos {p}")
                    assert_close(v, st["v"][l][p:p + 1], f"batch 32 V seq {s} layer {l} pos {p}")
        anchors = make_anchor_ids_np(n, shape.vocab, seed=190)
        _, _, checked = _draft_and_compare(d, orc, list(range(n)), anchors, 16, "8B 2-layer batch 32 U[1024, 8192]")
        assert checked > 0


def test_kv_append_512_rows_stream_k_pairs(dfl):
    """A 512-row append into 5 layers of 8 key/value heads of d = 128 (the 8B
    drafter's K/V width on a narrow hidden size): the fused K/V projection
    has 80 pair tiles for 76 SM pairs, so the pairs split them stream-K and
    the split tiles are finished by whichever CTA takes the last ticket. The
    cached K/V of every layer, at page-aligned and odd slot offsets, and a
    batch-32 draft over them are compared with the oracle."""
    from dataclasses import replace
    sh = replace(TINY, n_heads=8, n_kv_heads=8, head_dim=128, n_layers=5)
    wn = make_weights_np(sh, seed=201, gamma="jitter", std=0.05)
    orc = oracle.OracleDrafter(sh, wn, dtype=np.float32)
    width = sh.n_feat_layers * sh.hidden
    n = 32
    with dfl.Drafter(sh, np_weights_to_device(wn, DEV), max_seqs=n, max_batch=n, max_block=16, max_ctx=512,
                     max_fuse_tokens=8192) as d:
        rng = np.random.default_rng(202)
        lens = [int(x) for x in rng.integers(0, 150, size=n)]   # odd and even first slots of the append
        f = make_features_np(sum(lens), width, seed=203)
        d.fuse_ctx(list(range(n)), lens, bf16_dev(f, DEV), pending=False)
        orc.fuse_ctx(list(range(n)), lens, f, pending=False)
        f = make_features_np(16 * n, width, seed=204)
        d.fuse_ctx(list(range(n)), [16] * n, bf16_dev(f, DEV), pending=False)
        orc.fuse_ctx(list(range(n)), [16] * n, f, pending=False)
        d.sync()
        _check_kv(d, orc, range(n), range(sh.n_layers), "512-row append", ROW_REL_HIGH_GAIN)
        anchors = make_anchor_ids_np(n, sh.vocab, seed=205)
        _, _, c = _draft_and_compare(d, orc, list(range(n)), anchors, 16, "batch 32 after a stream-K append",
                                     ROW_REL_HIGH_GAIN)
        assert c > 0
