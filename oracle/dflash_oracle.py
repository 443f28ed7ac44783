"""CPU oracle of the DFlash drafter pass and greedy verify.

TEST INFRASTRUCTURE. Only the tests, the smoke check and the bench's CPU
baseline leg may import this module. The CUDA library shares no code, table or
helper with it and never calls it.

What it computes, and where the pages define it:

* Feature fusion (DFlash notes, §4.2, fusion equation): the hidden states of
  L_f target layers are concatenated (shallow to deep), projected by one
  shared W_c of shape [H, L_f*H] and RMS-normalised:
  H_t = RMSNorm(W_c [H^(l1); ...; H^(lLf)]).
* KV injection (DFlash notes, §4.3, the two K_i / V_i equations): every
  drafter layer i projects the fused context with its own W_i^K, W_i^V and
  prepends the result, along the sequence axis, to the K/V of the draft
  block. The context skips Q, O, the residual update and the FFN.
* Parallel block drafting (DFlash notes, §4.4; Trying DFlash on Gemma,
  appendix): the block is the last verified (anchor) token followed by B-1
  MASK tokens, embedded with the shared embedding, run once through a
  Qwen-style pre-norm decoder (RMSNorm, RoPE, GQA attention, SwiGLU FFN) whose
  attention is non-causal; every masked position is decoded independently
  with the shared LM head (greedy: argmax).
* Greedy acceptance (DFlash notes, §4.5 "acceptance check"; §2.2 for tau):
  drafts are compared in order with the target's greedy choices; acceptance
  stops at the first mismatch and the target supplies one bonus token;
  tau counts the accepted drafts plus the bonus.
* Latency model (DFlash notes, §2.2): L = (T_draft + T_verify) / tau,
  speedup eta = L_target / L; acceptance accounting as printed in the
  llama-server logs (Trying DFlash on Gemma, Tables 4-5 and the n-max-15 log).

Readings taken where the pages are silent:
  - mask position j of the block predicts the token at absolute position C+j
    (the anchor's own output is unused), so a block of B yields B-1 drafts;
  - RoPE is the rotate-half form with theta_i = base^(-2i/d), at absolute
    positions: context 0..C-1, block C..C+B-1, K rotated before caching;
  - RMSNorm is x / sqrt(mean(x^2) + eps) * gain, no biases, no QK-norm;
  - the attention scale is 1/sqrt(d) and kv head h // (n_q/n_kv) serves
    query head h;
  - argmax ties go to the lowest index;
  - t_j is the target's greedy token after block position j; accept while
    d_{j+1} == t_j; tau = a + 1, bonus = t_a;
  - with pending features, verify commits the first min(tau, pending) slots
    (anchor plus accepted drafts) and discards the rest.

Pins: every function here is checked, in tests/test_oracle_pins.py, against
closed forms, invariants, library routines or values the pages print.
Parity unpinned: the trained behaviour (acceptance rates of a real drafter)
needs trained weights; the full-depth draft ids are pinned only through the
per-part pins above.
"""
from __future__ import annotations

import math
from typing import Dict, List, Optional, Sequence

import numpy as np


# ----------------------------------------------------------------------------
# Building blocks
# ----------------------------------------------------------------------------

def rms_norm(x: np.ndarray, gain: np.ndarray, eps: float) -> np.ndarray:
    """x / sqrt(mean(x^2) + eps) * gain over the last axis."""
    mean_sq = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(mean_sq + eps) * gain


def rope_angles(positions: np.ndarray, head_dim: int, base: float) -> np.ndarray:
    """Angles pos * theta_i, theta_i = base^(-2i/d), i < d/2, always in fp64."""
    i = np.arange(head_dim // 2, dtype=np.float64)
    theta = np.power(np.float64(base), -2.0 * i / head_dim)
    return np.asarray(positions, dtype=np.float64)[:, None] * theta[None, :]


def apply_rope(x: np.ndarray, positions: np.ndarray, base: float) -> np.ndarray:
    """Rotate-half RoPE. x [n, heads, d]; position per row n.

    Dimension i is paired with i + d/2 and the pair is rotated by the angle
    pos * theta_i.
    """
    n, _, d = x.shape
    ang = rope_angles(positions, d, base)
    cos = np.cos(ang)[:, None, :].astype(x.dtype)
    sin = np.sin(ang)[:, None, :].astype(x.dtype)
    lo = x[..., : d // 2]
    hi = x[..., d // 2:]
    return np.concatenate([lo * cos - hi * sin, hi * cos + lo * sin], axis=-1)


def silu(x: np.ndarray) -> np.ndarray:
    return x / (1.0 + np.exp(-x))


def rows_argmax(logits: np.ndarray) -> np.ndarray:
    """Index of the largest value per row; among equal values the lowest index."""
    return np.argmax(logits, axis=-1).astype(np.int64)


def top2_gap(logits: np.ndarray) -> np.ndarray:
    """Largest minus second-largest value per row, counting repeats: a row
    whose maximum occurs twice has gap 0."""
    part = np.partition(logits, -2, axis=-1)
    return part[..., -1] - part[..., -2]


# ----------------------------------------------------------------------------
# Fusion and KV injection
# ----------------------------------------------------------------------------

def fuse_features(feats: np.ndarray, w_c: np.ndarray, g_c: np.ndarray, eps: float) -> np.ndarray:
    """H_t = RMSNorm(W_c [H^(l1); ...; H^(lLf)]); feats [n, L_f*H] layer-major."""
    return rms_norm(feats @ w_c.T, g_c, eps)


def context_kv(h_t: np.ndarray, layer: Dict[str, np.ndarray], positions: np.ndarray,
               n_kv: int, head_dim: int, base: float):
    """The context half of the KV-injection equations for one drafter layer:
    K = RoPE(W^K H_t) at the tokens' absolute positions, V = W^V H_t."""
    n = h_t.shape[0]
    k = (h_t @ layer["w_k"].T).reshape(n, n_kv, head_dim)
    v = (h_t @ layer["w_v"].T).reshape(n, n_kv, head_dim)
    return apply_rope(k, positions, base), v


# ----------------------------------------------------------------------------
# Drafter forward
# ----------------------------------------------------------------------------

def block_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray,
                    return_probs: bool = False):
    """Non-causal attention of every block query over all keys.

    q [B, n_q, d]; k, v [T, n_kv, d] (T = context + block). Query head h reads
    kv head h // (n_q / n_kv). Scale 1/sqrt(d). No mask.
    """
    B, n_q, d = q.shape
    n_kv = k.shape[1]
    group = n_q // n_kv
    out = np.empty_like(q)
    probs = [] if return_probs else None
    scale = 1.0 / math.sqrt(d)
    for h in range(n_q):
        kh = k[:, h // group, :]
        vh = v[:, h // group, :]
        s = (q[:, h, :] @ kh.T) * scale          # [B, T]
        s = s - np.max(s, axis=-1, keepdims=True)
        p = np.exp(s)
        p = p / np.sum(p, axis=-1, keepdims=True)
        out[:, h, :] = p @ vh
        if return_probs:
            probs.append(p)
    if return_probs:
        return out, np.stack(probs, axis=1)      # [B, n_q, T]
    return out


def decoder_layer(x: np.ndarray, layer: Dict[str, np.ndarray], k_ctx: np.ndarray,
                  v_ctx: np.ndarray, pos0: int, shape) -> np.ndarray:
    """One Qwen-style pre-norm drafter layer over the block x [B, H].

    Block positions are pos0 .. pos0+B-1. The block's K/V are appended after
    the injected context K/V (already rotated), and every block query attends
    to all of them.
    """
    B = x.shape[0]
    nq, nkv, d = shape.n_heads, shape.n_kv_heads, shape.head_dim
    pos = pos0 + np.arange(B)
    h = rms_norm(x, layer["g_attn"], shape.rms_eps)
    q = apply_rope((h @ layer["w_q"].T).reshape(B, nq, d), pos, shape.rope_base)
    k = apply_rope((h @ layer["w_k"].T).reshape(B, nkv, d), pos, shape.rope_base)
    v = (h @ layer["w_v"].T).reshape(B, nkv, d)
    keys = np.concatenate([k_ctx, k], axis=0)
    vals = np.concatenate([v_ctx, v], axis=0)
    a = block_attention(q, keys, vals).reshape(B, nq * d)
    x = x + a @ layer["w_o"].T
    h2 = rms_norm(x, layer["g_ffn"], shape.rms_eps)
    x = x + (silu(h2 @ layer["w_gate"].T) * (h2 @ layer["w_up"].T)) @ layer["w_down"].T
    return x


def draft_block(weights, shape, anchor: int, k_ctx: Sequence[np.ndarray],
                v_ctx: Sequence[np.ndarray], B: int) -> Dict[str, np.ndarray]:
    """One drafter pass over [anchor, MASK x (B-1)] against a committed context.

    k_ctx[l], v_ctx[l] [C, n_kv, d] are layer l's injected context K/V.
    Returns draft ids [B-1] (greedy per masked position), the final residual
    stream [B, H], the logits of every masked position [B-1, V], the top logit
    and the top-1/top-2 gap per masked position.
    """
    C = k_ctx[0].shape[0] if len(k_ctx) else 0
    ids = np.array([anchor] + [shape.mask_id] * (B - 1), dtype=np.int64)
    x = weights["embed"][ids].copy()
    for layer, kc, vc in zip(weights["layers"], k_ctx, v_ctx):
        x = decoder_layer(x, layer, kc, vc, C, shape)
    hf = rms_norm(x, weights["g_final"], shape.rms_eps)
    if B > 1:
        logits = hf[1:] @ weights["lm_head"].T
        draft = rows_argmax(logits)
        top1 = np.max(logits, axis=-1)
        gap = top2_gap(logits)
    else:
        logits = np.zeros((0, weights["lm_head"].shape[0]))
        draft = np.zeros(0, dtype=np.int64)
        top1 = np.zeros(0)
        gap = np.zeros(0)
    return {"draft": draft, "hidden": x, "logits": logits, "top1": top1, "gap": gap}


# ----------------------------------------------------------------------------
# Verify
# ----------------------------------------------------------------------------

def verify_block(drafts: Sequence[int], targets: Sequence[int]):
    """Greedy acceptance of one block.

    drafts d_1..d_{B-1}; targets t_0..t_{B-1}, t_j being the target's greedy
    token after block position j. a = number of leading j with d_{j+1} == t_j;
    tau = a + 1 (accepted drafts plus the bonus); bonus = t_a.
    """
    B = len(targets)
    a = 0
    while a < B - 1 and int(drafts[a]) == int(targets[a]):
        a += 1
    return a + 1, int(targets[a])


# ----------------------------------------------------------------------------
# Stateful drafter with a per-sequence injected-context cache
# ----------------------------------------------------------------------------

class OracleDrafter:
    """The drafter with its own context cache, separate from the target's.

    Per sequence it keeps, for every layer, the context K/V of the committed
    tokens followed by any pending (appended, not yet verified) tokens.
    """

    def __init__(self, shape, weights, dtype=np.float64):
        self.shape = shape
        cv = lambda a: np.asarray(a, dtype=dtype)
        self.w = {k: cv(v) for k, v in weights.items() if k != "layers"}
        self.w["layers"] = [{k: cv(v) for k, v in lw.items()} for lw in weights["layers"]]
        self.dtype = dtype
        self.seqs: Dict[int, dict] = {}

    def _state(self, s: int) -> dict:
        if s not in self.seqs:
            sh = self.shape
            empty = np.zeros((0, sh.n_kv_heads, sh.head_dim), dtype=self.dtype)
            self.seqs[s] = {"k": [empty.copy() for _ in range(sh.n_layers)],
                            "v": [empty.copy() for _ in range(sh.n_layers)],
                            "len": 0, "pend": 0}
        return self.seqs[s]

    def seq_reset(self, s: int) -> None:
        self.seqs.pop(s, None)

    def seq_len(self, s: int):
        st = self._state(s)
        return st["len"], st["pend"]

    def fuse_ctx(self, seq_ids, n_new, feats: np.ndarray, pending: bool) -> None:
        """Append fused target features for n_new[i] tokens of seq_ids[i]
        (rows of feats in that order) at positions len + pend + (0..n-1)."""
        sh = self.shape
        r = 0
        for s, n in zip(seq_ids, n_new):
            st = self._state(int(s))
            if not pending and st["pend"]:
                raise ValueError("committed append with pending slots outstanding")
            n = int(n)
            base = st["len"] + st["pend"]
            pos = base + np.arange(n)
            h_t = fuse_features(np.asarray(feats[r:r + n], dtype=self.dtype),
                                self.w["w_c"], self.w["g_c"], sh.rms_eps)
            for l, layer in enumerate(self.w["layers"]):
                k, v = context_kv(h_t, layer, pos, sh.n_kv_heads, sh.head_dim, sh.rope_base)
                st["k"][l] = np.concatenate([st["k"][l][:base], k], axis=0)
                st["v"][l] = np.concatenate([st["v"][l][:base], v], axis=0)
            if pending:
                st["pend"] += n
            else:
                st["len"] += n
            r += n

    def context(self, s: int, layer: int):
        st = self._state(s)
        return st["k"][layer][: st["len"]], st["v"][layer][: st["len"]]

    def draft(self, seq_ids, anchors, B: int) -> List[Dict[str, np.ndarray]]:
        out = []
        for s, a in zip(seq_ids, anchors):
            st = self._state(int(s))
            kc = [k[: st["len"]] for k in st["k"]]
            vc = [v[: st["len"]] for v in st["v"]]
            out.append(draft_block(self.w, self.shape, int(a), kc, vc, B))
        return out

    def verify(self, seq_ids, B: int, drafts: np.ndarray, targets: np.ndarray):
        """Greedy verify per sequence, then commit min(tau, pending) pending
        slots and discard the rest. Returns (tau [n], bonus [n])."""
        taus, bonuses = [], []
        for i, s in enumerate(seq_ids):
            st = self._state(int(s))
            tau, bonus = verify_block(drafts[i], targets[i])
            commit = min(tau, st["pend"])
            st["len"] += commit
            st["pend"] = 0
            for l in range(self.shape.n_layers):
                st["k"][l] = st["k"][l][: st["len"]]
                st["v"][l] = st["v"][l][: st["len"]]
            taus.append(tau)
            bonuses.append(bonus)
        return np.array(taus, dtype=np.int64), np.array(bonuses, dtype=np.int64)


# ----------------------------------------------------------------------------
# Latency model and acceptance accounting
# ----------------------------------------------------------------------------

def per_token_latency(t_draft: float, t_verify: float, tau: float) -> float:
    """L = (T_draft + T_verify) / tau (DFlash notes, §2.2)."""
    return (t_draft + t_verify) / tau


def speedup(l_target: float, l_spec: float) -> float:
    """eta = L_target / L (DFlash notes, §2.2)."""
    return l_target / l_spec


def acceptance_stats(accepted: int, generated: int, drafts_per_cycle: float):
    """Acceptance = accepted drafts / generated drafts; mean accepted length
    per cycle, counting the bonus token, = 1 + accepted / cycles where
    cycles = generated / drafts_per_cycle."""
    acceptance = accepted / generated
    cycles = generated / drafts_per_cycle
    return acceptance, 1.0 + accepted / cycles


def tokens_per_second(tokens: int, milliseconds: float) -> float:
    return tokens / (milliseconds / 1000.0)
