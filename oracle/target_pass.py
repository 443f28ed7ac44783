"""CPU oracle of a target-shaped verify pass (the other half of a DFlash cycle).

TEST INFRASTRUCTURE. Only the tests, the smoke check and the bench's CPU
baseline leg may import this module. The CUDA library shares no code, table or
helper with it and never calls it.

What it computes, and where the pages define it:

* Block verification (DFlash notes, §4.5 "The Decoding Loop", the decoding
  cycle figure): the target LLM computes logits for all positions of the
  drafted block in one batched forward pass; the acceptance check compares
  each draft with the target's greedy choice there.
* T_verify (DFlash notes, §2.2 "The Speedup Formula"): the time of that one
  forward pass; with L_target, the time of one plain decoding step, it gives
  eta = L_target / L.
* Feature extraction (DFlash notes, §4.2 "Feature Fusion", and §6.1 "Setup"):
  during the target's forward pass (prefill or verification) the hidden
  states of 5 layers, uniformly sampled between layer 2 and the third-to-last
  layer, are taken for the drafter.

Readings taken where the pages are silent:
  - the target is a Qwen-style pre-norm decoder, the drafter's layer (RMSNorm,
    rotate-half RoPE, GQA attention, SwiGLU; no QK-norm) with causal
    attention: block position j sees the cached context and block positions
    0..j;
  - layers are numbered from 1, and feature k of L_f is the output residual
    stream of layer 2 + k (L - 4) / (L_f - 1), rounded to the nearest layer
    (the third-to-last layer is L - 2; for L = 36 this is layers 2, 10, 18,
    26, 34, integers, which is what fixes the 1-based reading); the features
    are concatenated
    layer-major, shallow to deep, as the fusion projection expects;
  - the block is [last verified token, d_1 .. d_{B-1}] at positions
    C .. C+B-1; its K/V are appended to the target's own cache, pending until
    the verify, which commits min(tau, pending) of them like the drafter's
    cache (prefill appends them committed);
  - t_j is the argmax of the target's logits at block position j (lowest index
    on ties).

Pins (tests/test_target_pass_pins.py): the feature layers the setup table
prints, causal attention against explicit loops, a scalar-loop brute force of
the whole pass on a micro target, the KV-cache equivalence (one block pass
equals B one-token passes), prefix independence, and losslessness of the
speculative loop against the target's own greedy decoding.
"""
from __future__ import annotations

import math
from typing import Dict, List, Sequence

import numpy as np

from oracle import dflash_oracle as od


def feature_layers(n_layers: int, n_feat: int) -> List[int]:
    """0-based indices of the target layers whose outputs are the features:
    uniformly spaced from layer 2 to the third-to-last layer (1-based), each
    rounded to the nearest layer."""
    first, last = 2, n_layers - 2
    if n_feat == 1:
        return [first - 1]
    out = []
    for k in range(n_feat):
        pos = first + k * (last - first) / (n_feat - 1)
        out.append(int(math.floor(pos + 0.5)) - 1)
    return out


def causal_block_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, n_ctx: int) -> np.ndarray:
    """Attention of block queries q [B, n_q, d] over keys/values [n_ctx + B,
    n_kv, d] (context first, then the block): block position j sees the
    context and block positions 0..j. Scale 1/sqrt(d); query head h reads kv
    head h // (n_q / n_kv)."""
    B, n_q, d = q.shape
    n_kv = k.shape[1]
    group = n_q // n_kv
    T = k.shape[0]
    allowed = np.arange(T)[None, :] <= (n_ctx + np.arange(B))[:, None]     # [B, T]
    out = np.empty_like(q)
    scale = 1.0 / math.sqrt(d)
    for h in range(n_q):
        s = (q[:, h, :] @ k[:, h // group, :].T) * scale
        s = np.where(allowed, s, -np.inf)
        s = s - np.max(s, axis=-1, keepdims=True)
        p = np.exp(s)
        p = p / np.sum(p, axis=-1, keepdims=True)
        out[:, h, :] = p @ v[:, h // group, :]
    return out


def target_layer(x: np.ndarray, layer: Dict[str, np.ndarray], k_ctx: np.ndarray, v_ctx: np.ndarray, pos0: int,
                 shape):
    """One pre-norm target layer over the block x [B, H] at positions
    pos0 .. pos0+B-1 with causal attention over the cached context and the
    block. Returns the new residual stream and the block's K (rotated) and V,
    which the cache appends."""
    B = x.shape[0]
    nq, nkv, d = shape.n_heads, shape.n_kv_heads, shape.head_dim
    pos = pos0 + np.arange(B)
    h = od.rms_norm(x, layer["g_attn"], shape.rms_eps)
    q = od.apply_rope((h @ layer["w_q"].T).reshape(B, nq, d), pos, shape.rope_base)
    k = od.apply_rope((h @ layer["w_k"].T).reshape(B, nkv, d), pos, shape.rope_base)
    v = (h @ layer["w_v"].T).reshape(B, nkv, d)
    a = causal_block_attention(q, np.concatenate([k_ctx, k], axis=0), np.concatenate([v_ctx, v], axis=0),
                               k_ctx.shape[0]).reshape(B, nq * d)
    x = x + a @ layer["w_o"].T
    h2 = od.rms_norm(x, layer["g_ffn"], shape.rms_eps)
    x = x + (od.silu(h2 @ layer["w_gate"].T) * (h2 @ layer["w_up"].T)) @ layer["w_down"].T
    return x, k, v


def target_block_pass(weights, shape, ids: Sequence[int], k_ctx: Sequence[np.ndarray], v_ctx: Sequence[np.ndarray],
                      feat_layers: Sequence[int]) -> Dict[str, object]:
    """The target's forward pass over one block of token ids at positions
    C .. C+B-1 (C = cached length). Returns the greedy ids t_j [B], the
    logits [B, V], the top logit and top-1/top-2 gap per position, the final
    residual stream [B, H], the features [B, L_f * H] (outputs of the feature
    layers, layer-major) and the block's K/V per layer ([B, n_kv, d] each)."""
    C = k_ctx[0].shape[0] if len(k_ctx) else 0
    x = weights["embed"][np.asarray(ids, dtype=np.int64)].copy()
    feats, ks, vs = [], [], []
    for l, layer in enumerate(weights["layers"]):
        x, k, v = target_layer(x, layer, k_ctx[l], v_ctx[l], C, shape)
        ks.append(k)
        vs.append(v)
        if l in feat_layers:
            feats.append(x.copy())
    feats = [feats[sorted(feat_layers).index(l)] for l in feat_layers]
    hf = od.rms_norm(x, weights["g_final"], shape.rms_eps)
    logits = hf @ weights["lm_head"].T
    return {"ids": od.rows_argmax(logits), "logits": logits, "top1": np.max(logits, axis=-1),
            "gap": od.top2_gap(logits), "hidden": x, "feats": np.concatenate(feats, axis=-1), "k": ks, "v": vs}


class OracleTarget:
    """The target with its own per-sequence KV cache (committed tokens, then
    the pending block of the current cycle)."""

    def __init__(self, shape, weights, feat_layers: Sequence[int], dtype=np.float64):
        self.shape = shape
        cv = lambda a: np.asarray(a, dtype=dtype)
        self.w = {k: cv(v) for k, v in weights.items() if k != "layers"}
        self.w["layers"] = [{k: cv(v) for k, v in lw.items()} for lw in weights["layers"]]
        self.feat_layers = list(feat_layers)
        self.dtype = dtype
        self.seqs: Dict[int, dict] = {}

    def _state(self, s: int) -> dict:
        if s not in self.seqs:
            sh = self.shape
            empty = np.zeros((0, sh.n_kv_heads, sh.head_dim), dtype=self.dtype)
            self.seqs[s] = {"k": [empty.copy() for _ in range(sh.n_layers)],
                            "v": [empty.copy() for _ in range(sh.n_layers)], "len": 0, "pend": 0}
        return self.seqs[s]

    def seq_len(self, s: int):
        st = self._state(s)
        return st["len"], st["pend"]

    def forward(self, seq_ids, block_ids: np.ndarray, pending: bool) -> List[Dict[str, object]]:
        """One pass per sequence over block_ids[i] (B ids) at positions after
        its committed tokens; the block's K/V are appended pending (verify
        commits tau of them) or committed (prefill). A sequence with pending
        tokens must be verified first."""
        out = []
        for i, s in enumerate(seq_ids):
            st = self._state(int(s))
            if st["pend"]:
                raise ValueError("a target pass over a sequence with pending tokens")
            n = st["len"]
            kc = [k[:n] for k in st["k"]]
            vc = [v[:n] for v in st["v"]]
            r = target_block_pass(self.w, self.shape, block_ids[i], kc, vc, self.feat_layers)
            B = len(block_ids[i])
            for l in range(self.shape.n_layers):
                st["k"][l] = np.concatenate([kc[l], r["k"][l]], axis=0)
                st["v"][l] = np.concatenate([vc[l], r["v"][l]], axis=0)
            if pending:
                st["pend"] = B
            else:
                st["len"] += B
            out.append(r)
        return out

    def verify(self, seq_ids, B: int, drafts: np.ndarray, targets: np.ndarray):
        """Greedy verify per sequence (as the drafter's), committing
        min(tau, pending) of the pending block and dropping the rest."""
        taus, bonuses = [], []
        for i, s in enumerate(seq_ids):
            st = self._state(int(s))
            tau, bonus = od.verify_block(drafts[i], targets[i])
            st["len"] += min(tau, st["pend"])
            st["pend"] = 0
            for l in range(self.shape.n_layers):
                st["k"][l] = st["k"][l][: st["len"]]
                st["v"][l] = st["v"][l][: st["len"]]
            taus.append(tau)
            bonuses.append(bonus)
        return np.array(taus, dtype=np.int64), np.array(bonuses, dtype=np.int64)


def speculative_decode(target: OracleTarget, drafter: od.OracleDrafter, prompt: Sequence[int], B: int,
                       n_tokens: int) -> List[int]:
    """The DFlash cycle end to end for one sequence (slot 0 of both models).
    Prefill: the target runs over the prompt (committed); its features of the
    prompt tokens fill the drafter's context, and its choice after the last
    prompt token is the first generated token, the first anchor (the last
    verified token, not yet cached). Then each cycle drafts from the anchor,
    verifies [anchor, drafts] in one target pass (pending), commits tau on
    both caches and emits the accepted drafts and the bonus token, which is
    the next anchor. Returns the first n_tokens generated tokens."""
    prompt = [int(t) for t in prompt]
    r = target.forward([0], np.array([prompt]), pending=False)[0]
    drafter.fuse_ctx([0], [len(prompt)], r["feats"], pending=False)
    anchor = int(r["ids"][-1])
    out = [anchor]
    while len(out) < n_tokens:
        drafts = np.asarray(drafter.draft([0], [anchor], B)[0]["draft"], dtype=np.int64)
        block = np.array([[anchor] + [int(x) for x in drafts]])
        tr = target.forward([0], block, pending=True)[0]
        drafter.fuse_ctx([0], [B], tr["feats"], pending=True)
        tau, bonus = target.verify([0], B, drafts[None, :], tr["ids"][None, :])
        drafter.verify([0], B, drafts[None, :], tr["ids"][None, :])
        out.extend(int(x) for x in drafts[: int(tau[0]) - 1])
        out.append(int(bonus[0]))
        anchor = int(bonus[0])
    return out[:n_tokens]


def greedy_decode(target: OracleTarget, prompt: Sequence[int], n_tokens: int) -> List[int]:
    """The target alone, one token per pass (slot 1): the output the
    speculative cycle must reproduce exactly."""
    r = target.forward([1], np.array([[int(t) for t in prompt]]), pending=False)[0]
    out = [int(r["ids"][-1])]
    while len(out) < n_tokens:
        r = target.forward([1], np.array([[out[-1]]]), pending=False)[0]
        out.append(int(r["ids"][-1]))
    return out
