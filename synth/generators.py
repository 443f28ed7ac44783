"""Seeded synthetic workloads for the DFlash drafter pass.

The pages measure on math/code/chat suites that are not available here; these
draws stand in for them with the shapes and distributions the drafter pass
sees (weights N(0, 0.02), target features N(0, 1) per token, ids uniform,
per-sequence context lengths uniform, verify agreement to a geometric
mismatch position).

Everything stored in bf16 on the device is drawn in float32 and rounded to
bf16 here (round to nearest even), so the oracle can consume exactly the
values the CUDA path consumes, upcast.

Nothing in this module is part of the drafter's computation.
"""
from __future__ import annotations

from dataclasses import dataclass, replace
from typing import Dict, List

import numpy as np


@dataclass(frozen=True)
class DrafterShape:
    """Sizes of a DFlash drafter (notation of the DFlash notes, §4)."""

    hidden: int          # H: drafter (and target) hidden size
    n_heads: int         # query heads
    n_kv_heads: int      # key/value heads (GQA group = n_heads / n_kv_heads)
    head_dim: int        # d
    ffn: int             # SwiGLU intermediate size F
    vocab: int           # V (shared embedding and LM head)
    n_layers: int        # drafter layers L
    n_feat_layers: int   # target layers whose hidden states are fused (L_f)
    rope_base: float
    rms_eps: float
    mask_id: int         # id of the MASK token that fills the block after the anchor

    def with_layers(self, n_layers: int) -> "DrafterShape":
        return replace(self, n_layers=n_layers)


# 1-layer tiny drafter checked in fp64 (hidden 256, 4/4 heads of 64, FFN 688,
# vocab 4096, RoPE base 1e4, 3 target feature layers).
TINY = DrafterShape(hidden=256, n_heads=4, n_kv_heads=4, head_dim=64, ffn=688,
                    vocab=4096, n_layers=1, n_feat_layers=3, rope_base=1.0e4,
                    rms_eps=1e-6, mask_id=4095)

# Qwen3-8B-shaped drafter: 5 layers, hidden 4096, 32 q / 8 kv heads of 128,
# SwiGLU 12288, vocab 151936, RoPE base 1e6, 5 fused target layers.
QWEN3_8B = DrafterShape(hidden=4096, n_heads=32, n_kv_heads=8, head_dim=128,
                        ffn=12288, vocab=151936, n_layers=5, n_feat_layers=5,
                        rope_base=1.0e6, rms_eps=1e-6, mask_id=151935)


# ----------------------------------------------------------------------------
# bf16 storage helpers (storage format only)
# ----------------------------------------------------------------------------

def bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round to nearest even."""
    a = np.ascontiguousarray(x, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    u = (u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    return u.astype(np.uint16)


def bits_to_f32(b: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float32 values."""
    u = np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32)


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 value (returned as float32)."""
    return bits_to_f32(bf16_bits(x))


# ----------------------------------------------------------------------------
# Weights
# ----------------------------------------------------------------------------

def _normal(rng: np.random.Generator, shape, std: float) -> np.ndarray:
    return bf16_round(rng.standard_normal(shape, dtype=np.float32) * np.float32(std))


def _gamma(rng: np.random.Generator, n: int, mode: str) -> np.ndarray:
    if mode == "ones":
        return np.ones(n, dtype=np.float32)
    if mode == "jitter":  # exercises the gain path in parity tests
        return bf16_round(1.0 + 0.1 * rng.standard_normal(n, dtype=np.float32))
    raise ValueError(mode)


def make_weights_np(shape: DrafterShape, seed: int = 0, gamma: str = "ones",
                    std: float = 0.02) -> Dict[str, object]:
    """All drafter weights as float32 arrays holding bf16 values.

    Layout is nn.Linear style, [out_features, in_features]:
      w_c     [H, L_f*H]   fusion projection (DFlash notes §4.2)
      g_c     [H]          fusion RMSNorm gain
      embed   [V, H]       shared token embedding
      lm_head [V, H]       shared LM head (untied from embed)
      g_final [H]          final RMSNorm gain
      layers[i]: w_q [n_q*d, H], w_k/w_v [n_kv*d, H], w_o [H, n_q*d],
                 w_gate/w_up [F, H], w_down [H, F], g_attn/g_ffn [H]
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    H, d = shape.hidden, shape.head_dim
    out: Dict[str, object] = {}
    out["w_c"] = _normal(rng, (H, shape.n_feat_layers * H), std)
    out["g_c"] = _gamma(rng, H, gamma)
    out["embed"] = _normal(rng, (shape.vocab, H), std)
    out["lm_head"] = _normal(rng, (shape.vocab, H), std)
    out["g_final"] = _gamma(rng, H, gamma)
    layers: List[Dict[str, np.ndarray]] = []
    for _ in range(shape.n_layers):
        lw = {
            "w_q": _normal(rng, (shape.n_heads * d, H), std),
            "w_k": _normal(rng, (shape.n_kv_heads * d, H), std),
            "w_v": _normal(rng, (shape.n_kv_heads * d, H), std),
            "w_o": _normal(rng, (H, shape.n_heads * d), std),
            "w_gate": _normal(rng, (shape.ffn, H), std),
            "w_up": _normal(rng, (shape.ffn, H), std),
            "w_down": _normal(rng, (H, shape.ffn), std),
            "g_attn": _gamma(rng, H, gamma),
            "g_ffn": _gamma(rng, H, gamma),
        }
        layers.append(lw)
    out["layers"] = layers
    return out


def make_weights_torch(shape: DrafterShape, seed: int = 0, device="cuda",
                       gamma: str = "ones", std: float = 0.02):
    """Same structure as make_weights_np, drawn on the device with a seeded
    torch.Generator and stored as bf16 tensors (for the 8B-sized drafter,
    whose 4.6 GB of weights are too slow to draw on the host)."""
    import torch

    g = torch.Generator(device=device)
    g.manual_seed(seed)
    H, d = shape.hidden, shape.head_dim

    def normal(*sz):
        t = torch.empty(sz, dtype=torch.float32, device=device)
        t.normal_(0.0, std, generator=g)
        return t.to(torch.bfloat16)

    def gain(n):
        if gamma == "ones":
            return torch.ones(n, dtype=torch.bfloat16, device=device)
        t = torch.empty(n, dtype=torch.float32, device=device)
        t.normal_(1.0, 0.1, generator=g)
        return t.to(torch.bfloat16)

    out = {"w_c": normal(H, shape.n_feat_layers * H), "g_c": gain(H),
           "embed": normal(shape.vocab, H), "lm_head": normal(shape.vocab, H),
           "g_final": gain(H), "layers": []}
    for _ in range(shape.n_layers):
        out["layers"].append({
            "w_q": normal(shape.n_heads * d, H), "w_k": normal(shape.n_kv_heads * d, H),
            "w_v": normal(shape.n_kv_heads * d, H), "w_o": normal(H, shape.n_heads * d),
            "w_gate": normal(shape.ffn, H), "w_up": normal(shape.ffn, H),
            "w_down": normal(H, shape.ffn), "g_attn": gain(H), "g_ffn": gain(H)})
    return out


def torch_weights_to_np(w) -> Dict[str, object]:
    """Host float32 copies of make_weights_torch's tensors (input plumbing)."""
    def cvt(t):
        return t.float().cpu().numpy()
    out = {k: cvt(v) for k, v in w.items() if k != "layers"}
    out["layers"] = [{k: cvt(v) for k, v in lw.items()} for lw in w["layers"]]
    return out


# ----------------------------------------------------------------------------
# Activations, ids, lengths
# ----------------------------------------------------------------------------

def make_selector_weights_np(shape: DrafterShape, seed: int = 0, dim: int = 256,
                             std: float = None, embed_std: float = 0.02,
                             lm_std: float = 0.02) -> Dict[str, np.ndarray]:
    """Path-selector maps W_A, W_B, W_H [dim, H] as float32 arrays of bf16 values.

    The default std makes the pair term's spread comparable to the logits'
    spread, so the selector's walk both follows and leaves the plain greedy
    path: with E ~ N(0, embed_std^2), normalised hidden rows of unit RMS and
    W ~ N(0, std^2), the pair term has std sqrt(dim) std^3 embed_std^2 H^1.5
    and a logit std lm_std sqrt(H); std solves their equality.
    """
    H = shape.hidden
    if std is None:
        std = float((lm_std / (np.sqrt(dim) * embed_std ** 2 * H)) ** (1.0 / 3.0))
    rng = np.random.Generator(np.random.PCG64(seed))
    return {k: _normal(rng, (dim, H), std) for k in ("w_a", "w_b", "w_h")}


def make_conv_weights_np(shape: DrafterShape, rank: int = 80, seed: int = 0, corr: float = 0.2,
                         base_jitter: float = 0.1, tap1_std: float = 0.3):
    """Two-tap convolution weights for every layer: a list over layers of
    dicts {"ai", "ao", "fi", "fo"} -> {"base" [2, H], "U" [2, H, r],
    "V" [2, r, H]}, float32 arrays of bf16 values.

    base tap 0 ~ 1 + N(0, base_jitter^2), tap 1 ~ N(0, tap1_std^2); U and V
    entries N(0, s^2) with s^2 = corr / sqrt(r H), so that for inputs of unit
    RMS the rank-r correction U V x has RMS about corr.
    """
    H = shape.hidden
    s = float(np.sqrt(corr / np.sqrt(rank * H)))
    rng = np.random.Generator(np.random.PCG64(seed))
    layers = []
    for _ in range(shape.n_layers):
        sites = {}
        for name in ("ai", "ao", "fi", "fo"):
            base = np.stack([1.0 + rng.standard_normal(H) * base_jitter, rng.standard_normal(H) * tap1_std])
            sites[name] = {"base": bf16_round(base.astype(np.float32)),
                           "U": _normal(rng, (2, H, rank), s), "V": _normal(rng, (2, rank, H), s)}
        layers.append(sites)
    return layers


def make_features_np(n_tokens: int, width: int, seed: int) -> np.ndarray:
    """Concatenated target features [n, L_f*H], N(0, 1) per element, bf16 values."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return bf16_round(rng.standard_normal((n_tokens, width), dtype=np.float32))


def make_anchor_ids_np(n: int, vocab: int, seed: int) -> np.ndarray:
    """Anchor ids uniform on [0, V-2] (V-1 is reserved for the mask token)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return rng.integers(0, vocab - 1, size=n, dtype=np.int64).astype(np.int32)


def make_serving_lengths(batch: int, lo: int, hi: int, seed: int) -> np.ndarray:
    """Per-sequence committed context lengths, integer uniform on [lo, hi]."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return rng.integers(lo, hi + 1, size=batch, dtype=np.int64).astype(np.int32)


def make_target_logits_bf16_np(rows: int, vocab: int, seed: int, std: float = 3.0) -> np.ndarray:
    """Target logits N(0, std^2) stored as bf16 bit patterns [rows, vocab]."""
    rng = np.random.Generator(np.random.PCG64(seed))
    x = rng.standard_normal((rows, vocab), dtype=np.float32) * np.float32(std)
    return bf16_bits(x)


def make_verify_case_np(targets: np.ndarray, vocab: int, seed: int,
                        p_mismatch: float = 0.3):
    """Draft ids that agree with the target ids up to a seeded mismatch.

    targets [b, B] are the target's greedy ids t_0..t_{B-1}. For each row a
    mismatch position m ~ Geometric(p_mismatch) on {0, 1, ...} is drawn:
    d_{j+1} = t_j for j < m; d_{m+1} differs from t_m; later drafts are
    uniform. m >= B-1 means every draft agrees. Returns (drafts [b, B-1], m [b]).
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    t = np.asarray(targets, dtype=np.int64)
    b, B = t.shape
    drafts = np.empty((b, B - 1), dtype=np.int64)
    ms = rng.geometric(p_mismatch, size=b) - 1
    for r in range(b):
        m = int(ms[r])
        for j in range(B - 1):
            if j < m:
                drafts[r, j] = t[r, j]
            elif j == m:
                drafts[r, j] = (t[r, j] + 1 + rng.integers(0, vocab - 1)) % vocab
            else:
                drafts[r, j] = rng.integers(0, vocab)
    return drafts.astype(np.int32), ms.astype(np.int32)
