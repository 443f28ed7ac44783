"""Pins of the target-pass oracle (oracle/target_pass.py) against what the
pages print and what the mathematics fixes: the feature layers of the setup
table, causal attention written as explicit loops, a scalar-loop brute force
of a whole target pass, the KV-cache equivalence of one block pass and B
one-token passes, prefix independence, and losslessness of the speculative
cycle against the target's own greedy decoding."""
import math
from dataclasses import replace

import numpy as np

import oracle
from oracle import dflash_oracle as od
from oracle import target_pass as tp
from synth import DrafterShape, make_weights_np

# micro target: 3 layers, hidden 16, 4 query / 2 kv heads of 8, FFN 24, vocab 37
MICRO = DrafterShape(hidden=16, n_heads=4, n_kv_heads=2, head_dim=8, ffn=24, vocab=37, n_layers=3, n_feat_layers=2,
                     rope_base=1.0e4, rms_eps=1e-6, mask_id=36)


def _rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def _f64_weights(shape, seed, std=0.4):
    w = make_weights_np(shape, seed=seed, gamma="jitter", std=std)
    cv = lambda a: np.asarray(a, dtype=np.float64)
    out = {k: cv(v) for k, v in w.items() if k != "layers"}
    out["layers"] = [{k: cv(v) for k, v in lw.items()} for lw in w["layers"]]
    return out


def test_feature_layers_match_the_setup_table():
    """5 layers uniformly sampled between layer 2 and the third-to-last: for a
    36-layer Qwen3-8B target the 1-based layers 2, 10, 18, 26, 34."""
    assert [l + 1 for l in tp.feature_layers(36, 5)] == [2, 10, 18, 26, 34]
    for L in (8, 12, 28, 36, 40):
        fl = [l + 1 for l in tp.feature_layers(L, 5)]
        assert fl[0] == 2 and fl[-1] == L - 2            # layer 2 and the third-to-last
        assert all(b > a for a, b in zip(fl, fl[1:]))
        step = (L - 4) / 4
        assert all(abs(fl[k] - (2 + k * step)) <= 0.5 for k in range(5))


def _causal_loops(q, k, v, n_ctx):
    B, nq, d = q.shape
    g = nq // k.shape[1]
    out = np.zeros_like(q)
    for j in range(B):
        for h in range(nq):
            keys = range(n_ctx + j + 1)
            sc = [sum(q[j, h, i] * k[t, h // g, i] for i in range(d)) / math.sqrt(d) for t in keys]
            m = max(sc)
            e = [math.exp(x - m) for x in sc]
            z = sum(e)
            for i in range(d):
                out[j, h, i] = sum(e[t] * v[t, h // g, i] for t in keys) / z
    return out


def test_causal_attention_matches_explicit_loops():
    r = _rng(1)
    q = r.standard_normal((5, 4, 8))
    k = r.standard_normal((7 + 5, 2, 8))
    v = r.standard_normal((7 + 5, 2, 8))
    np.testing.assert_allclose(tp.causal_block_attention(q, k, v, 7), _causal_loops(q, k, v, 7), rtol=1e-12, atol=1e-12)
    # one block token sees every key: the non-causal attention
    np.testing.assert_allclose(tp.causal_block_attention(q[:1], k[:8], v[:8], 7), od.block_attention(q[:1], k[:8], v[:8]),
                               rtol=1e-13, atol=1e-13)
    # the first block token of an empty context sees only itself
    np.testing.assert_allclose(tp.causal_block_attention(q, k[:5], v[:5], 0)[0],
                               np.repeat(v[0], 2, axis=0), rtol=1e-13, atol=1e-13)


def _matvec(w, x):
    return [sum(w[i][j] * x[j] for j in range(len(x))) for i in range(len(w))]


def _rms(x, g, eps):
    s = math.sqrt(sum(t * t for t in x) / len(x) + eps)
    return [x[i] / s * g[i] for i in range(len(x))]


def _rope(vec, pos, base):
    d = len(vec)
    out = list(vec)
    for i in range(d // 2):
        a = pos * base ** (-2.0 * i / d)
        c, s = math.cos(a), math.sin(a)
        out[i] = vec[i] * c - vec[i + d // 2] * s
        out[i + d // 2] = vec[i + d // 2] * c + vec[i] * s
    return out


def _target_loops(w, sh, ids, feat_layers):
    """Scalar-loop causal pass over the whole sequence `ids` from an empty
    cache (positions 0..n-1): logits, features and every layer's K/V."""
    H, d, nq, nkv = sh.hidden, sh.head_dim, sh.n_heads, sh.n_kv_heads
    g = nq // nkv
    n = len(ids)
    x = [list(w["embed"][i]) for i in ids]
    feats = [[] for _ in range(n)]
    ks, vs = [], []
    for li, lw in enumerate(w["layers"]):
        hs = [_rms(row, lw["g_attn"], sh.rms_eps) for row in x]
        qf = [_matvec(lw["w_q"], h) for h in hs]
        kf = [_matvec(lw["w_k"], h) for h in hs]
        vf = [_matvec(lw["w_v"], h) for h in hs]
        q = [[_rope(qf[t][j * d:(j + 1) * d], t, sh.rope_base) for j in range(nq)] for t in range(n)]
        k = [[_rope(kf[t][j * d:(j + 1) * d], t, sh.rope_base) for j in range(nkv)] for t in range(n)]
        v = [[vf[t][j * d:(j + 1) * d] for j in range(nkv)] for t in range(n)]
        ks.append(k)
        vs.append(v)
        new_x = []
        for t in range(n):
            att = []
            for hq in range(nq):
                kv = hq // g
                sc = [sum(q[t][hq][i] * k[u][kv][i] for i in range(d)) / math.sqrt(d) for u in range(t + 1)]
                m = max(sc)
                e = [math.exp(s - m) for s in sc]
                z = sum(e)
                att += [sum(e[u] * v[u][kv][i] for u in range(t + 1)) / z for i in range(d)]
            o = _matvec(lw["w_o"], att)
            new_x.append([x[t][i] + o[i] for i in range(H)])
        x = new_x
        for t in range(n):
            h2 = _rms(x[t], lw["g_ffn"], sh.rms_eps)
            gt = _matvec(lw["w_gate"], h2)
            up = _matvec(lw["w_up"], h2)
            act = [gt[i] / (1 + math.exp(-gt[i])) * up[i] for i in range(len(gt))]
            dn = _matvec(lw["w_down"], act)
            x[t] = [x[t][i] + dn[i] for i in range(H)]
        if li in feat_layers:
            for t in range(n):
                feats[t].append(list(x[t]))
    logits = [_matvec(w["lm_head"], _rms(row, w["g_final"], sh.rms_eps)) for row in x]
    order = sorted(feat_layers)
    feats = [sum((f[order.index(l)] for l in feat_layers), []) for f in feats]
    return np.array(logits), np.array(feats), ks, vs


def test_target_pass_matches_scalar_brute_force():
    """Prefill of 4 tokens, then a block of 3 at positions 4..6: the oracle's
    logits, greedy ids, features and cached K/V equal a scalar-loop causal
    pass over all 7 tokens."""
    sh = MICRO
    w = _f64_weights(sh, seed=2)
    fl = [0, 2]
    ids = [3, 17, 8, 30, 5, 11, 22]
    t = tp.OracleTarget(sh, w, fl)
    t.forward([0], np.array([ids[:4]]), pending=False)
    r = t.forward([0], np.array([ids[4:]]), pending=True)[0]
    logits, feats, ks, vs = _target_loops(w, sh, ids, fl)
    np.testing.assert_allclose(r["logits"], logits[4:], rtol=1e-11, atol=1e-11)
    np.testing.assert_array_equal(r["ids"], np.argmax(logits[4:], axis=-1))
    np.testing.assert_allclose(r["feats"], feats[4:], rtol=1e-11, atol=1e-11)
    for l in range(sh.n_layers):
        np.testing.assert_allclose(t.seqs[0]["k"][l], np.array(ks[l]), rtol=1e-11, atol=1e-11)
        np.testing.assert_allclose(t.seqs[0]["v"][l], np.array(vs[l]), rtol=1e-11, atol=1e-11)
    assert t.seq_len(0) == (4, 3)


def test_block_pass_equals_one_token_passes():
    """The KV-cache equivalence that makes verification one pass: a block of
    B tokens gives the same logits, features and cached K/V as B passes of
    one token each, every token appended before the next runs."""
    sh = MICRO
    w = _f64_weights(sh, seed=3)
    fl = [1, 2]
    prompt, block = [4, 9, 1, 33, 12], [7, 7, 20, 2, 35, 0]
    a = tp.OracleTarget(sh, w, fl)
    a.forward([0], np.array([prompt]), pending=False)
    ra = a.forward([0], np.array([block]), pending=False)[0]
    b = tp.OracleTarget(sh, w, fl)
    b.forward([0], np.array([prompt]), pending=False)
    rb = [b.forward([0], np.array([[x]]), pending=False)[0] for x in block]
    np.testing.assert_allclose(ra["logits"], np.concatenate([r["logits"] for r in rb]), rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(ra["feats"], np.concatenate([r["feats"] for r in rb]), rtol=1e-11, atol=1e-11)
    for l in range(sh.n_layers):
        np.testing.assert_allclose(a.seqs[0]["k"][l], b.seqs[0]["k"][l], rtol=1e-11, atol=1e-11)
        np.testing.assert_allclose(a.seqs[0]["v"][l], b.seqs[0]["v"][l], rtol=1e-11, atol=1e-11)


def test_prefix_independence():
    """A block token changes nothing at earlier block positions."""
    sh = MICRO
    w = _f64_weights(sh, seed=4)
    fl = [0, 1]
    ctx = [5, 6, 7]
    for j in range(4):
        blk = np.array([10, 11, 12, 13])
        alt = blk.copy()
        alt[j] = 30
        outs = []
        for b in (blk, alt):
            t = tp.OracleTarget(sh, w, fl)
            t.forward([0], np.array([ctx]), pending=False)
            outs.append(t.forward([0], b[None, :], pending=True)[0])
        np.testing.assert_allclose(outs[0]["logits"][:j], outs[1]["logits"][:j], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(outs[0]["feats"][:j], outs[1]["feats"][:j], rtol=1e-12, atol=1e-12)
        if j < 3:
            assert np.abs(outs[0]["logits"][j:] - outs[1]["logits"][j:]).max() > 1e-6


def test_verify_commits_tau_of_the_pending_block():
    sh = MICRO
    w = _f64_weights(sh, seed=5)
    t = tp.OracleTarget(sh, w, [0, 1])
    t.forward([0], np.array([[1, 2, 3]]), pending=False)
    r = t.forward([0], np.array([[4, 5, 6, 7]]), pending=True)[0]
    drafts = np.array([[int(r["ids"][0]), (int(r["ids"][1]) + 1) % sh.vocab, 9]])
    tau, bonus = t.verify([0], 4, drafts, r["ids"][None, :])
    assert int(tau[0]) == 2 and int(bonus[0]) == int(r["ids"][1])
    assert t.seq_len(0) == (5, 0)
    assert t.seqs[0]["k"][0].shape[0] == 5


class _ScriptedDrafter:
    """A drafter that knows the greedy stream and proposes its next B-1
    tokens with one seeded position corrupted per cycle (or none), so the
    acceptance lengths of the cycle vary; it keeps the drafter's cache
    bookkeeping (committed length) to know where the anchor stands."""

    def __init__(self, stream, prompt_len, seed, vocab):
        self.stream, self.n0, self.vocab = stream, prompt_len, vocab
        self.rng = _rng(seed)
        self.len = self.pend = 0

    def fuse_ctx(self, seq_ids, n_new, feats, pending):
        if pending:
            self.pend += int(n_new[0])
        else:
            self.len += int(n_new[0])

    def verify(self, seq_ids, B, drafts, targets):
        tau, bonus = od.verify_block(drafts[0], targets[0])
        self.len += min(tau, self.pend)
        self.pend = 0
        return np.array([tau]), np.array([bonus])

    def draft(self, seq_ids, anchors, B):
        k = self.len - self.n0                     # index of the anchor in the generated stream
        assert self.stream[k] == anchors[0]
        d = np.array([self.stream[min(k + 1 + j, len(self.stream) - 1)] for j in range(B - 1)], dtype=np.int64)
        bad = int(self.rng.integers(0, B + 2))
        if bad < B - 1:
            d[bad] = (d[bad] + 1) % self.vocab
        return [{"draft": d}]


def test_speculative_cycle_is_lossless():
    """Prefill, then draft / one-pass verify / commit cycles emit exactly the
    target's own one-token-at-a-time greedy stream: with a random drafter
    (almost every cycle tau = 1) and with a scripted one (tau from 1 to B)."""
    sh = MICRO
    w = _f64_weights(sh, seed=6, std=0.5)
    fl = [0, 2]
    prompt = [3, 14, 15, 9, 26]
    ref = tp.greedy_decode(tp.OracleTarget(sh, w, fl), prompt, 40)
    dw = _f64_weights(replace(sh, n_layers=1), seed=7)
    for B in (2, 4, 6):
        got = tp.speculative_decode(tp.OracleTarget(sh, w, fl), od.OracleDrafter(replace(sh, n_layers=1), dw), prompt,
                                    B, 40)
        assert got == ref, B
        taus = []
        drafter = _ScriptedDrafter(ref + [0] * 64, len(prompt), seed=B, vocab=sh.vocab)
        orig = drafter.verify

        def rec(*a, **k):
            out = orig(*a, **k)
            taus.append(int(out[0][0]))
            return out
        drafter.verify = rec
        got = tp.speculative_decode(tp.OracleTarget(sh, w, fl), drafter, prompt, B, 40)
        assert got == ref, B
        assert max(taus) == B and min(taus) < B
