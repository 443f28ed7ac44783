"""Kernel-level GPU checks through the C ABI: the tcgen05 GEMM against a plain
fp32 matmul, the bf16 row argmax and greedy verify/commit against the oracle
(integer outputs bit-exact)."""
import numpy as np
import pytest

import oracle
from synth import (TINY, make_weights_np, make_features_np, make_target_logits_bf16_np, make_verify_case_np,
                   bits_to_f32)
from tests.gpu_util import np_weights_to_device, bf16_dev, i32_dev, assert_close

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dfl():
    import __graft_entry__
    __graft_entry__.build()
    import block_diffusion_drafter_pass_gb300 as m
    return m


DEV = "cuda:0"


@pytest.mark.parametrize("N,M,K,splits", [
    (256, 16, 256, 1),        # one tile
    (384, 5, 1024, 0),        # ragged tokens, automatic split-K
    (100, 33, 200, 0),        # ragged everything, K not a multiple of 64
    (4096, 16, 4096, 0),      # batch-1 weight streaming shape (O): stream-K over all SMs
    (6144, 16, 4096, 0),      # batch-1 QKV shape
    (4096, 5, 4096, 0),       # the same with a ragged token tile
    (4256, 16, 4096, 0),      # a ragged last weight tile (34 tiles)
    (2048, 16, 1000, 0),      # 16 k-blocks, the last one ragged
    (2048, 16, 1088, 0),      # 17 k-blocks: pieces of uneven length
    (4096, 16, 12288, 0),     # batch-1 down shape
    (1024, 300, 512, 1),      # two 256-token tiles with a ragged tail
    (640, 64, 2048, 3),       # explicit split-K
    (256, 128, 128, 2),
    (2048, 512, 1024, 0),     # clusters of two CTA pairs splitting each pair tile's k-blocks
    (1024, 300, 512, 0),      # the same with a ragged token tail
    (512, 272, 960, 0),       # the same with an odd k-block count (15 = 7 + 8)
    (128, 512, 512, 0),       # one weight tile: 256-token tiles split over K by 2-CTA clusters
    (384, 200, 64, 0),        # one k-block: CTA pairs, odd weight-tile count
    (6144, 512, 1024, 0),     # CTA pairs (cta_group::2), one pair tile per pair
    (24576, 512, 512, 0),     # CTA pairs, pair tiles dealt round-robin (3 rounds)
    (4992, 512, 256, 0),      # CTA pairs, odd weight-tile count (last pair half empty)
    (5120, 300, 320, 0),      # CTA pairs, ragged token tail in the second CTA's half
    (10240, 512, 512, 0),     # 80 pair tiles on 76 pairs: stream-K over the pairs (split tiles finished by tickets)
    (10112, 300, 1024, 0),    # stream-K pairs, odd weight-tile count and a ragged token tail
])
def test_gemm_matches_fp32_matmul(dfl, N, M, K, splits):
    g = torch.Generator(device="cpu").manual_seed(N * 7 + M * 3 + K)
    W = torch.randn(N, K, generator=g).to(torch.bfloat16)
    X = torch.randn(M, K, generator=g).to(torch.bfloat16)
    ref = X.float() @ W.float().T
    Y = dfl.dflash_debug_gemm(W.to(DEV), X.to(DEV), splits=splits)
    torch.cuda.synchronize()
    err = (Y.cpu() - ref).abs()
    assert float(err.max()) <= 1e-3 * np.sqrt(K), float(err.max())


def test_rows_argmax_full_size_bit_exact(dfl):
    rows, V = 64 * 16, 151936
    bits = make_target_logits_bf16_np(rows, V, seed=5)
    ref = oracle.rows_argmax(bits_to_f32(bits))
    logits = torch.from_numpy(bits.view(np.int16)).to(DEV).view(torch.bfloat16)
    got = dfl.dflash_rows_argmax_bf16(logits).cpu().numpy()
    np.testing.assert_array_equal(got, ref)


@pytest.mark.parametrize("cols", [1, 7, 13, 4096, 4099])
def test_rows_argmax_ties_and_ragged(dfl, cols):
    rng = np.random.Generator(np.random.PCG64(cols))
    vals = np.round(rng.standard_normal((37, cols)) * 2).astype(np.float32)   # many exact ties
    from synth import bf16_bits
    bits = bf16_bits(vals)
    ref = oracle.rows_argmax(bits_to_f32(bits))
    logits = torch.from_numpy(bits.view(np.int16)).to(DEV).view(torch.bfloat16)
    got = dfl.dflash_rows_argmax_bf16(logits).cpu().numpy()
    np.testing.assert_array_equal(got, ref)


@pytest.mark.parametrize("rows", [100, 131, 300, 1029])
@pytest.mark.parametrize("cols", [4096, 4099, 20008])
def test_rows_argmax_split_and_ring(dfl, rows, cols):
    """Row counts that split a row over clusters of 4 and 2 CTAs or give each
    row one CTA, on the bulk-copy ring (cols % 8 == 0, several 8192-column
    stages and a short last one) and the direct path (cols % 8 != 0)."""
    rng = np.random.Generator(np.random.PCG64(rows * 10 + cols))
    vals = np.round(rng.standard_normal((rows, cols)) * 3).astype(np.float32)
    from synth import bf16_bits
    bits = bf16_bits(vals)
    ref = oracle.rows_argmax(bits_to_f32(bits))
    logits = torch.from_numpy(bits.view(np.int16)).to(DEV).view(torch.bfloat16)
    got = dfl.dflash_rows_argmax_bf16(logits).cpu().numpy()
    np.testing.assert_array_equal(got, ref)


def test_rows_argmax_signed_zero_is_one_value(dfl):
    """-0 and +0 compare equal: a row whose maximum is zero takes the first
    zero, whichever sign it has (a float comparison, as the oracle's)."""
    cols = 20008   # three ring stages
    from synth import bf16_bits
    vals = -np.ones((4, cols), dtype=np.float32)
    vals[0, 100], vals[0, 9000] = 0.0, -0.0
    vals[1, 100], vals[1, 9000] = -0.0, 0.0
    vals[2, 9000], vals[2, 9001] = -0.0, 0.0
    vals[3, 5], vals[3, 20007] = 0.0, 1.0
    bits = bf16_bits(vals)
    ref = oracle.rows_argmax(bits_to_f32(bits))
    np.testing.assert_array_equal(ref, [100, 100, 9000, 20007])
    logits = torch.from_numpy(bits.view(np.int16)).to(DEV).view(torch.bfloat16)
    got = dfl.dflash_rows_argmax_bf16(logits).cpu().numpy()
    np.testing.assert_array_equal(got, ref)


def _tiny_drafter(dfl, max_batch=64, max_block=16, max_ctx=256, max_pages=None):
    wn = make_weights_np(TINY, seed=3)
    d = dfl.Drafter(TINY, np_weights_to_device(wn, DEV), max_seqs=max_batch, max_batch=max_batch,
                    max_block=max_block, max_ctx=max_ctx, max_pages=max_pages, max_fuse_tokens=4096)
    return d, wn


def test_verify_and_commit_bit_exact_batch64(dfl):
    """Batch 64, B = 16, vocab 151936: targets are the argmax of bf16 N(0, 3)
    logits; drafts agree up to a geometric mismatch. tau, bonus and the
    commit of pending slots are compared exactly with the oracle."""
    b, B, V = 64, 16, 151936
    bits = make_target_logits_bf16_np(b * B, V, seed=11)
    logits = torch.from_numpy(bits.view(np.int16)).to(DEV).view(torch.bfloat16)
    t_gpu = dfl.dflash_rows_argmax_bf16(logits).view(b, B)
    t_ref = oracle.rows_argmax(bits_to_f32(bits)).reshape(b, B)
    np.testing.assert_array_equal(t_gpu.cpu().numpy(), t_ref)
    drafts, ms = make_verify_case_np(t_ref, V, seed=12)

    d, wn = _tiny_drafter(dfl)
    orc = oracle.OracleDrafter(TINY, wn)
    seqs = list(range(b))
    width = TINY.n_feat_layers * TINY.hidden
    ctx_len = [int(x) for x in np.random.Generator(np.random.PCG64(13)).integers(0, 100, size=b)]
    feats = make_features_np(sum(ctx_len) + b * B, width, seed=14)
    d.fuse_ctx(seqs, ctx_len, bf16_dev(feats[:sum(ctx_len)], DEV), pending=False)
    orc.fuse_ctx(seqs, ctx_len, feats[:sum(ctx_len)], pending=False)
    d.fuse_ctx(seqs, [B] * b, bf16_dev(feats[sum(ctx_len):], DEV), pending=True)
    orc.fuse_ctx(seqs, [B] * b, feats[sum(ctx_len):], pending=True)
    # every cached byte (committed context and the pending block) before verify
    before = {s: d.read_kv(0, s, 0, ctx_len[s] + B) for s in seqs}
    tau, bonus = d.verify(seqs, B, i32_dev(drafts, DEV), t_gpu)
    rt, rb = orc.verify(seqs, B, drafts, t_ref)
    d.sync()
    np.testing.assert_array_equal(tau.cpu().numpy(), rt)
    np.testing.assert_array_equal(bonus.cpu().numpy(), rb)
    assert (rt == np.minimum(ms, B - 1) + 1).all()
    for s in seqs:
        assert d.seq_len(s) == orc.seq_len(s)
    # the committed slots keep exactly the bytes appended before verify (bf16
    # bit patterns compared, so -0 and +0 differ), and they are the oracle's
    # K/V within the tolerance
    for s in seqs:
        n = orc.seq_len(s)[0]
        assert n == ctx_len[s] + int(rt[seqs.index(s)])
        k, v = d.read_kv(0, s, 0, n)
        np.testing.assert_array_equal(k.view(np.uint32), before[s][0][:n].view(np.uint32))
        np.testing.assert_array_equal(v.view(np.uint32), before[s][1][:n].view(np.uint32))
        kr, vr = orc.context(s, 0)
        assert_close(k, kr, f"committed K seq {s}")
        assert_close(v, vr, f"committed V seq {s}")
    # the next cycle appends at the committed length: the rolled-back slots are
    # overwritten by the new block and the committed prefix is untouched
    feats2 = make_features_np(b * B, width, seed=15)
    d.fuse_ctx(seqs, [B] * b, bf16_dev(feats2, DEV), pending=True)
    orc.fuse_ctx(seqs, [B] * b, feats2, pending=True)
    for s in (0, 17, 63):
        n = orc.seq_len(s)[0]
        k, v = d.read_kv(0, s, 0, n + B)
        np.testing.assert_array_equal(k[:n].view(np.uint32), before[s][0][:n].view(np.uint32))
        np.testing.assert_array_equal(v[:n].view(np.uint32), before[s][1][:n].view(np.uint32))
        st = orc.seqs[s]
        assert_close(k[n:], st["k"][0][n:n + B], f"re-appended K seq {s}")
        assert_close(v[n:], st["v"][0][n:n + B], f"re-appended V seq {s}")
    d.close()


def test_verify_edge_cases(dfl):
    d, wn = _tiny_drafter(dfl, max_batch=4, max_block=32)
    cases = [
        (1, np.zeros((1, 0), np.int32), np.array([[9]], np.int32)),             # B = 1: tau 1, bonus t_0
        (32, np.arange(31, dtype=np.int32)[None], np.arange(32, dtype=np.int32)[None]),  # all accepted
        (5, np.array([[1, 2, 3, 4]], np.int32), np.array([[0, 2, 3, 4, 5]], np.int32)),  # first rejected
    ]
    for B, dr, tg in cases:
        tau, bonus = d.verify([0], B, i32_dev(dr, DEV) if dr.size else None, i32_dev(tg, DEV))
        rt, rb = oracle.verify_block(dr[0], tg[0])
        d.sync()
        assert (int(tau.item()), int(bonus.item())) == (rt, rb)
    d.close()


def test_invalid_arguments_are_rejected(dfl):
    d, _ = _tiny_drafter(dfl, max_batch=2, max_block=8, max_ctx=128, max_pages=2)
    width = TINY.n_feat_layers * TINY.hidden
    f = bf16_dev(make_features_np(200, width, seed=1), DEV)
    anchors = i32_dev([1, 2], DEV)
    with pytest.raises(dfl.DFlashError) as e:
        d.draft([0, 0], anchors, 4)            # duplicate sequence
    assert e.value.status == dfl.DFLASH_EINVAL
    with pytest.raises(dfl.DFlashError):
        d.draft([0], anchors, 9)               # B > max_block
    with pytest.raises(dfl.DFlashError):
        d.fuse_ctx([0], [129], f, pending=False)   # beyond max_ctx
    with pytest.raises(dfl.DFlashError) as e:
        d.fuse_ctx([0, 1], [100, 100], f, pending=False)   # 4 pages needed, pool holds 2
    assert e.value.status == dfl.DFLASH_ENOMEM
    d.fuse_ctx([0], [10], f, pending=True)
    with pytest.raises(dfl.DFlashError):
        d.fuse_ctx([0], [1], f, pending=False)     # committed append over pending tokens
    d.sync()
    assert d.seq_len(0) == (0, 10) and d.seq_len(1) == (0, 0)
    d.seq_reset(0)
    assert d.seq_len(0) == (0, 0)
    d.close()
