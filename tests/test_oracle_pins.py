"""Pins of the CPU oracle to things other than itself.

Each test checks an oracle function against a closed form, an invariant, a
library routine, brute force on tiny inputs, or a number the pages print
(tests/golden/worked_numbers.json). None of them calls the CUDA library.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from synth import TINY, DrafterShape, make_weights_np, make_features_np

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_numbers.json")

# A micro drafter for explicit-loop brute force (GQA group 2, ffn not a power of 2).
MICRO = DrafterShape(hidden=16, n_heads=4, n_kv_heads=2, head_dim=4, ffn=24, vocab=37,
                     n_layers=2, n_feat_layers=3, rope_base=100.0, rms_eps=1e-6, mask_id=36)


def _rng(seed=0):
    return np.random.Generator(np.random.PCG64(seed))


def _f64_weights(shape, seed=0, gamma="jitter", std=0.3):
    w = make_weights_np(shape, seed=seed, gamma=gamma, std=std)
    cv = lambda a: np.asarray(a, dtype=np.float64)
    out = {k: cv(v) for k, v in w.items() if k != "layers"}
    out["layers"] = [{k: cv(v) for k, v in lw.items()} for lw in w["layers"]]
    return out


# ----------------------------------------------------------------------------
# RMSNorm, SiLU
# ----------------------------------------------------------------------------

def test_rmsnorm_unit_rms_closed_form():
    x = _rng(1).standard_normal((7, 64)) * 5.0
    y = oracle.rms_norm(x, np.ones(64), 0.0)
    np.testing.assert_allclose(np.sqrt(np.mean(y * y, axis=-1)), 1.0, rtol=1e-12)


def test_rmsnorm_matches_torch():
    r = _rng(2)
    x = r.standard_normal((5, 48))
    g = 1.0 + 0.1 * r.standard_normal(48)
    ref = F.rms_norm(torch.from_numpy(x), (48,), torch.from_numpy(g), eps=1e-6).numpy()
    np.testing.assert_allclose(oracle.rms_norm(x, g, 1e-6), ref, rtol=1e-12, atol=1e-14)


def test_silu_matches_torch():
    x = np.linspace(-20, 20, 1001)
    np.testing.assert_allclose(oracle.silu(x), F.silu(torch.from_numpy(x)).numpy(), rtol=1e-12, atol=1e-15)


# ----------------------------------------------------------------------------
# RoPE
# ----------------------------------------------------------------------------

def _rope_complex(x, positions, base):
    """Closed form: pair (x_i, x_{i+d/2}) as x_i + i*x_{i+d/2}, multiply by e^{i*pos*theta_i}."""
    n, h, d = x.shape
    half = d // 2
    z = x[..., :half] + 1j * x[..., half:]
    theta = base ** (-(2.0 * np.arange(half)) / d)
    rot = np.exp(1j * np.asarray(positions, dtype=np.float64)[:, None, None] * theta[None, None, :])
    w = z * rot
    return np.concatenate([w.real, w.imag], axis=-1)


def test_rope_matches_complex_rotation():
    x = _rng(3).standard_normal((9, 3, 64))
    pos = np.array([0, 1, 2, 7, 63, 1000, 4095, 32768, 262143])
    np.testing.assert_allclose(oracle.apply_rope(x, pos, 1e6), _rope_complex(x, pos, 1e6),
                               rtol=1e-12, atol=1e-12)


def test_rope_theta_values():
    # theta_i = base^(-2i/d): theta_0 = 1 and theta_1 = base^(-2/d)
    a = oracle.rope_angles(np.array([1]), 64, 1e4)[0]
    assert a[0] == 1.0
    assert abs(a[1] - 10000 ** (-2 / 64)) < 1e-15
    assert abs(a[31] - 10000 ** (-62 / 64)) < 1e-18


def test_rope_identity_at_zero_and_norm_preserving():
    x = _rng(4).standard_normal((4, 2, 128))
    np.testing.assert_array_equal(oracle.apply_rope(x, np.zeros(4, dtype=int), 1e6), x)
    y = oracle.apply_rope(x, np.array([5, 77, 1 << 17, 262100]), 1e6)
    np.testing.assert_allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-12)


def test_rope_relative_position_invariance():
    r = _rng(5)
    q = r.standard_normal((1, 1, 128))
    k = r.standard_normal((1, 1, 128))
    for s in (0, 13, 4096, 200000):
        qs = oracle.apply_rope(q, np.array([s + 40]), 1e6)
        ks = oracle.apply_rope(k, np.array([s + 3]), 1e6)
        q0 = oracle.apply_rope(q, np.array([40]), 1e6)
        k0 = oracle.apply_rope(k, np.array([3]), 1e6)
        assert abs(float(np.sum(qs * ks)) - float(np.sum(q0 * k0))) < 1e-9


# ----------------------------------------------------------------------------
# Attention
# ----------------------------------------------------------------------------

def _attention_loops(q, k, v):
    """Explicit-loop softmax attention (GQA by integer division of the head)."""
    B, nq, d = q.shape
    T, nkv, _ = k.shape
    g = nq // nkv
    out = np.zeros_like(q)
    for b in range(B):
        for h in range(nq):
            kh = h // g
            scores = [sum(q[b, h, i] * k[t, kh, i] for i in range(d)) / math.sqrt(d) for t in range(T)]
            m = max(scores)
            w = [math.exp(s - m) for s in scores]
            z = sum(w)
            for i in range(d):
                out[b, h, i] = sum(w[t] * v[t, kh, i] for t in range(T)) / z
    return out


def test_attention_matches_explicit_loops():
    r = _rng(6)
    q = r.standard_normal((3, 4, 8))
    k = r.standard_normal((11, 2, 8))
    v = r.standard_normal((11, 2, 8))
    np.testing.assert_allclose(oracle.block_attention(q, k, v), _attention_loops(q, k, v), rtol=1e-12, atol=1e-12)


def test_attention_rows_are_distributions():
    r = _rng(7)
    q = r.standard_normal((16, 8, 32)) * 3
    k = r.standard_normal((100, 2, 32)) * 3
    v = r.standard_normal((100, 2, 32))
    _, p = oracle.block_attention(q, k, v, return_probs=True)
    assert np.all(p >= 0)
    np.testing.assert_allclose(p.sum(-1), 1.0, rtol=0, atol=1e-12)


def test_attention_matches_torch_sdpa_and_gqa_equals_repeated_mha():
    r = _rng(8)
    q = r.standard_normal((16, 8, 32))
    k = r.standard_normal((40, 2, 32))
    v = r.standard_normal((40, 2, 32))
    out = oracle.block_attention(q, k, v)
    kr = np.repeat(k, 4, axis=1)
    vr = np.repeat(v, 4, axis=1)
    np.testing.assert_allclose(oracle.block_attention(q, kr, vr), out, rtol=1e-12, atol=1e-12)
    tq = torch.from_numpy(q).permute(1, 0, 2)
    tk = torch.from_numpy(kr).permute(1, 0, 2)
    tv = torch.from_numpy(vr).permute(1, 0, 2)
    ref = F.scaled_dot_product_attention(tq, tk, tv, is_causal=False).permute(1, 0, 2).numpy()
    np.testing.assert_allclose(out, ref, rtol=1e-10, atol=1e-12)


def test_attention_single_key_returns_value():
    r = _rng(9)
    q = r.standard_normal((1, 4, 8)) * 10
    k = r.standard_normal((1, 2, 8))
    v = r.standard_normal((1, 2, 8))
    out = oracle.block_attention(q, k, v)
    np.testing.assert_allclose(out[0], np.repeat(v[0], 2, axis=0), rtol=1e-14)


# ----------------------------------------------------------------------------
# Decoder layer / draft pass
# ----------------------------------------------------------------------------

def _matvec(w, x):
    return [sum(w[i][j] * x[j] for j in range(len(x))) for i in range(len(w))]


def _rms_loop(x, g, eps):
    s = math.sqrt(sum(t * t for t in x) / len(x) + eps)
    return [x[i] / s * g[i] for i in range(len(x))]


def _single_step_loops(x, lw, sh):
    """One decoder step for a lone token with no context: its only key is
    itself, so every head's attention weight is exactly 1 and RoPE drops out."""
    x = list(x)
    h = _rms_loop(x, lw["g_attn"], sh.rms_eps)
    v = _matvec(lw["w_v"], h)
    g = sh.n_heads // sh.n_kv_heads
    d = sh.head_dim
    attn = []
    for head in range(sh.n_heads):
        kvh = head // g
        attn += v[kvh * d:(kvh + 1) * d]
    o = _matvec(lw["w_o"], attn)
    x = [x[i] + o[i] for i in range(len(x))]
    h2 = _rms_loop(x, lw["g_ffn"], sh.rms_eps)
    gate = _matvec(lw["w_gate"], h2)
    up = _matvec(lw["w_up"], h2)
    act = [gate[i] / (1 + math.exp(-gate[i])) * up[i] for i in range(len(gate))]
    dn = _matvec(lw["w_down"], act)
    return [x[i] + dn[i] for i in range(len(x))]


def test_decoder_B1_C0_is_a_single_step():
    sh = MICRO
    w = _f64_weights(sh, seed=11)
    x = w["embed"][[5]]
    empty = np.zeros((0, sh.n_kv_heads, sh.head_dim))
    got = oracle.decoder_layer(x, w["layers"][0], empty, empty, 0, sh)[0]
    ref = _single_step_loops(x[0], w["layers"][0], sh)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def _rope_loops(vec, pos, base):
    d = len(vec)
    half = d // 2
    out = [0.0] * d
    for i in range(half):
        a = pos * base ** (-2.0 * i / d)
        c, s = math.cos(a), math.sin(a)
        out[i] = vec[i] * c - vec[i + half] * s
        out[i + half] = vec[i + half] * c + vec[i] * s
    return out


def _draft_loops(w, sh, anchor, feats_ctx, B):
    """Brute-force draft pass with scalar loops (fuse, inject, decode, argmax)."""
    H, d, nq, nkv = sh.hidden, sh.head_dim, sh.n_heads, sh.n_kv_heads
    g = nq // nkv
    C = len(feats_ctx)
    # context K/V per layer
    ht = [_rms_loop(_matvec(w["w_c"], f), w["g_c"], sh.rms_eps) for f in feats_ctx]
    ck, cv = [], []
    for lw in w["layers"]:
        ks, vs = [], []
        for p in range(C):
            kf = _matvec(lw["w_k"], ht[p])
            vf = _matvec(lw["w_v"], ht[p])
            ks.append([_rope_loops(kf[j * d:(j + 1) * d], p, sh.rope_base) for j in range(nkv)])
            vs.append([vf[j * d:(j + 1) * d] for j in range(nkv)])
        ck.append(ks)
        cv.append(vs)
    ids = [anchor] + [sh.mask_id] * (B - 1)
    x = [list(w["embed"][i]) for i in ids]
    for li, lw in enumerate(w["layers"]):
        hs = [_rms_loop(r, lw["g_attn"], sh.rms_eps) for r in x]
        q = [_matvec(lw["w_q"], h) for h in hs]
        k = [_matvec(lw["w_k"], h) for h in hs]
        v = [_matvec(lw["w_v"], h) for h in hs]
        qh = [[_rope_loops(q[b][j * d:(j + 1) * d], C + b, sh.rope_base) for j in range(nq)] for b in range(B)]
        kh = [[_rope_loops(k[b][j * d:(j + 1) * d], C + b, sh.rope_base) for j in range(nkv)] for b in range(B)]
        vh = [[v[b][j * d:(j + 1) * d] for j in range(nkv)] for b in range(B)]
        keys = ck[li] + kh
        vals = cv[li] + vh
        new_x = []
        for b in range(B):
            attn = []
            for hq in range(nq):
                kv = hq // g
                sc = [sum(qh[b][hq][i] * keys[t][kv][i] for i in range(d)) / math.sqrt(d) for t in range(len(keys))]
                m = max(sc)
                e = [math.exp(s - m) for s in sc]
                z = sum(e)
                attn += [sum(e[t] * vals[t][kv][i] for t in range(len(keys))) / z for i in range(d)]
            o = _matvec(lw["w_o"], attn)
            new_x.append([x[b][i] + o[i] for i in range(H)])
        x = new_x
        for b in range(B):
            h2 = _rms_loop(x[b], lw["g_ffn"], sh.rms_eps)
            gt = _matvec(lw["w_gate"], h2)
            up = _matvec(lw["w_up"], h2)
            act = [gt[i] / (1 + math.exp(-gt[i])) * up[i] for i in range(len(gt))]
            dn = _matvec(lw["w_down"], act)
            x[b] = [x[b][i] + dn[i] for i in range(H)]
    drafts, all_logits = [], []
    for b in range(1, B):
        hf = _rms_loop(x[b], w["g_final"], sh.rms_eps)
        logits = _matvec(w["lm_head"], hf)
        best = 0
        for i in range(1, len(logits)):
            if logits[i] > logits[best]:
                best = i
        drafts.append(best)
        all_logits.append(logits)
    return drafts, x, all_logits


def test_draft_pass_matches_scalar_brute_force():
    sh = MICRO
    w = _f64_weights(sh, seed=12)
    feats = make_features_np(6, sh.n_feat_layers * sh.hidden, seed=13).astype(np.float64)
    od = oracle.OracleDrafter(sh, w)
    od.fuse_ctx([0], [6], feats, pending=False)
    res = od.draft([0], [7], 4)[0]
    ref_ids, ref_x, ref_logits = _draft_loops(w, sh, 7, feats, 4)
    np.testing.assert_allclose(res["hidden"], np.array(ref_x), rtol=1e-11, atol=1e-11)
    np.testing.assert_array_equal(res["draft"], ref_ids)
    np.testing.assert_allclose(res["logits"], np.array(ref_logits), rtol=1e-11, atol=1e-11)
    # top logit and top-1/top-2 gap of each row, by a scan of the brute-force logits
    for r, row in enumerate(ref_logits):
        first, second = _two_largest_scan(row)
        assert abs(res["top1"][r] - first) <= 1e-11
        assert abs(res["gap"][r] - (first - second)) <= 1e-11


def test_draft_is_invariant_to_a_global_position_shift():
    sh = MICRO
    w = _f64_weights(sh, seed=14)
    feats = make_features_np(5, sh.n_feat_layers * sh.hidden, seed=15).astype(np.float64)
    ht = oracle.fuse_features(feats, w["w_c"], w["g_c"], sh.rms_eps)
    outs = []
    for shift in (0, 1000):
        pos = shift + np.arange(5)
        x = w["embed"][[3, sh.mask_id, sh.mask_id]].copy()
        for lw in w["layers"]:
            k, v = oracle.context_kv(ht, lw, pos, sh.n_kv_heads, sh.head_dim, sh.rope_base)
            x = oracle.decoder_layer(x, lw, k, v, shift + 5, sh)
        outs.append(x)
    np.testing.assert_allclose(outs[0], outs[1], rtol=1e-9, atol=1e-9)


def test_fusion_chunked_append_equals_single_append():
    sh = TINY
    w = make_weights_np(sh, seed=16, gamma="jitter")
    feats = make_features_np(40, sh.n_feat_layers * sh.hidden, seed=17)
    a = oracle.OracleDrafter(sh, w)
    b = oracle.OracleDrafter(sh, w)
    a.fuse_ctx([0], [40], feats, pending=False)
    b.fuse_ctx([0], [13], feats[:13], pending=False)
    b.fuse_ctx([0], [27], feats[13:], pending=False)
    for l in range(sh.n_layers):
        np.testing.assert_allclose(a.context(0, l)[0], b.context(0, l)[0], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(a.context(0, l)[1], b.context(0, l)[1], rtol=1e-12, atol=1e-13)


def test_fusion_weight_size_matches_the_printed_42MB():
    g = json.load(open(GOLDEN))["fusion_weight_bytes"][0]
    shape = DrafterShape(hidden=g["hidden"], n_heads=1, n_kv_heads=1, head_dim=8, ffn=8, vocab=8,
                         n_layers=0, n_feat_layers=g["n_feat_layers"], rope_base=1e4,
                         rms_eps=1e-6, mask_id=7)
    # fuse_features takes W_c as [H, L_f*H]; its byte count must match the page.
    D = shape.hidden
    w_c = np.zeros((D, shape.n_feat_layers * D), dtype=np.float32)
    out = oracle.fuse_features(np.ones((1, shape.n_feat_layers * D), dtype=np.float32), w_c,
                               np.ones(D, dtype=np.float32), 1e-6)
    assert out.shape == (1, D)
    assert round(w_c.size * g["bytes_per_elem"] / 1e6) == g["printed_mb"]


# ----------------------------------------------------------------------------
# Argmax and verify
# ----------------------------------------------------------------------------

def test_rows_argmax_lowest_index_on_ties():
    r = _rng(18)
    x = np.round(r.standard_normal((50, 30)) * 2) / 2  # many exact ties
    got = oracle.rows_argmax(x)
    for i in range(50):
        best = 0
        for j in range(30):
            if x[i, j] > x[i, best]:
                best = j
        assert got[i] == best


def _two_largest_scan(row):
    """The largest and second-largest entries of a row by one scan that keeps
    both, a repeat of the maximum counting as the second largest."""
    first, second = -math.inf, -math.inf
    for v in row:
        if v > first:
            first, second = v, first
        elif v > second:
            second = v
    return first, second


def test_top2_gap_matches_a_scan_and_a_sort():
    """top2_gap decides which draft rows must match bit for bit, so it is
    pinned on its own: random rows, rows whose maximum repeats (gap 0), rows
    whose second value repeats, all-equal rows, a two-column row and rows with
    infinities, against a two-value scan and against Python's sorted()."""
    r = _rng(19)
    rows = [r.standard_normal(40) for _ in range(20)]
    rows += [np.round(r.standard_normal(40) * 2) / 2 for _ in range(20)]   # many exact ties
    tie_top = r.standard_normal(40)
    tie_top[[3, 31]] = tie_top.max() + 1.0                               # maximum occurs twice
    tie_second = r.standard_normal(40)
    tie_second[[5, 6, 7]] = tie_second.max() + 1.0
    tie_second[20] = tie_second.max() + 0.25                             # second value occurs three times
    rows += [tie_top, tie_second, np.full(40, 1.5), np.array([2.0, -1.0])]
    inf_row = r.standard_normal(40)
    inf_row[9] = -math.inf
    rows.append(inf_row)
    x = np.stack([np.resize(row, 40) for row in rows])
    got = oracle.top2_gap(x)
    assert got.shape == (x.shape[0],)
    for i, row in enumerate(x):
        first, second = _two_largest_scan(row)
        srt = sorted(row.tolist(), reverse=True)
        assert got[i] == first - second == srt[0] - srt[1]
    assert got[40] == 0.0 and got[42] == 0.0                              # repeated maximum, all equal
    assert got[41] == 0.25                                               # the repeated second value counts once
    assert (got >= 0).all()


def _tau_bruteforce(d, t):
    B = len(t)
    best = 1
    for k in range(1, B + 1):       # tau = k means the first k-1 drafts agree
        if all(d[j] == t[j] for j in range(k - 1)):
            best = k
    return best, t[best - 1]


def test_verify_bruteforce_tiny_vocab():
    V = 3
    for B in (1, 2, 3, 4):
        for t in itertools.product(range(V), repeat=B):
            for d in itertools.product(range(V), repeat=B - 1):
                tau, bonus = oracle.verify_block(d, t)
                assert (tau, bonus) == _tau_bruteforce(d, t)
                assert 1 <= tau <= B


def test_verify_commit_bookkeeping():
    sh = TINY
    w = make_weights_np(sh, seed=19)
    od = oracle.OracleDrafter(sh, w)
    feats = make_features_np(20, sh.n_feat_layers * sh.hidden, seed=20)
    od.fuse_ctx([3], [10], feats[:10], pending=False)
    od.fuse_ctx([3], [4], feats[10:14], pending=True)
    assert od.seq_len(3) == (10, 4)
    t = np.array([[5, 6, 7, 8]])
    d = np.array([[5, 9, 9]])            # first draft agrees, second does not
    tau, bonus = od.verify([3], 4, d, t)
    assert (tau[0], bonus[0]) == (2, 6)
    assert od.seq_len(3) == (12, 0)
    assert od.context(3, 0)[0].shape[0] == 12
    # tau larger than the pending count commits only what was appended
    od.fuse_ctx([3], [1], feats[14:15], pending=True)
    tau, _ = od.verify([3], 4, np.array([[5, 6, 7]]), t)
    assert tau[0] == 4 and od.seq_len(3) == (13, 0)
    with pytest.raises(ValueError):
        od.fuse_ctx([3], [2], feats[:2], pending=True)
        od.fuse_ctx([3], [1], feats[:1], pending=False)


def test_speculative_loop_is_lossless_against_a_fake_target():
    """Draft, verify against a deterministic target, commit: the emitted
    stream equals the target's own greedy stream (DFlash notes, §4.5)."""
    sh = TINY
    w = make_weights_np(sh, seed=21)
    od = oracle.OracleDrafter(sh, w)
    memo = {}
    rng = _rng(22)
    width = sh.n_feat_layers * sh.hidden

    def target_next(prefix, proposal):
        key = tuple(prefix)
        if key not in memo:
            # agree with the drafter's proposal 70% of the time, else a fixed other id
            memo[key] = int(proposal) if rng.random() < 0.7 else int((proposal + 1 + rng.integers(0, sh.vocab - 1)) % sh.vocab)
        return memo[key]

    def features(prefix_len):
        return make_features_np(1, width, seed=10_000 + prefix_len)[0]

    prompt = [11, 12, 13, 14, 15]
    od.fuse_ctx([0], [len(prompt)], np.stack([features(i + 1) for i in range(len(prompt))]), pending=False)
    out = list(prompt)
    anchor = target_next(out, 0)
    out.append(anchor)
    B = 4
    taus = []
    while len(out) < 40:
        dr = od.draft([0], [anchor], B)[0]["draft"]
        block = [anchor] + [int(x) for x in dr]
        prefix = out[:-1]
        t = []
        for j in range(B):
            prop = block[j + 1] if j + 1 < B else 0
            t.append(target_next(prefix + block[: j + 1], prop))
        feats = np.stack([features(len(prefix) + j + 1) for j in range(B)])
        od.fuse_ctx([0], [B], feats, pending=True)
        tau, bonus = od.verify([0], B, np.array([dr]), np.array([t]))
        tau, bonus = int(tau[0]), int(bonus[0])
        taus.append(tau)
        out += block[1:tau] + [bonus]
        anchor = bonus
        assert od.seq_len(0)[0] == len(out) - 1
    # replay plain greedy decoding with the same target
    greedy = list(prompt)
    while len(greedy) < len(out):
        greedy.append(memo[tuple(greedy)])
    assert greedy == out
    assert max(taus) > 1  # acceptance paths were exercised


# ----------------------------------------------------------------------------
# Latency model and acceptance accounting (numbers printed on the pages)
# ----------------------------------------------------------------------------

def test_worked_numbers_from_the_pages():
    g = json.load(open(GOLDEN))
    for e in g["speedup"]:
        eta = oracle.speedup(1.0 / e["plain_tok_s"], 1.0 / e["dflash_tok_s"])
        assert round(eta, e["decimals"]) == e["printed_speedup"], e["source"]
    for e in g["acceptance_logs"]:
        acc, mean_len = oracle.acceptance_stats(e["accepted"], e["generated"], e["drafts_per_cycle"])
        assert round(acc, e["acceptance_decimals"]) == e["printed_acceptance"], e["source"]
        assert round(mean_len, e["mean_len_decimals"]) == e["printed_mean_len"], e["source"]
    for e in g["acceptance_percent"]:
        acc, _ = oracle.acceptance_stats(e["accepted"], e["generated"], 1)
        assert round(100 * acc, 2) == e["printed_percent"], e["source"]
    for e in g["acceptance_average_percent"]:
        assert round(float(np.mean(e["turn_percents"])), 2) == e["printed_average"], e["source"]
    for e in g["throughput"]:
        assert round(oracle.tokens_per_second(e["tokens"], e["ms"]), 2) == e["printed_tok_s"], e["source"]


def test_latency_model_closed_form():
    # tau = 1 and no draft cost reproduces the target's own latency
    assert oracle.per_token_latency(0.0, 20.0, 1.0) == 20.0
    L = oracle.per_token_latency(2.0, 20.0, 6.49)
    assert abs(oracle.speedup(20.0, L) - 20.0 * 6.49 / 22.0) < 1e-12
