"""CPU oracle of the DFlash 2 two-tap dynamic convolution.

TEST INFRASTRUCTURE. Only the tests, the smoke check and the bench's CPU
baseline leg may import this module. The CUDA library (conv.cu and the draft
pass) shares no code, table or helper with it and never calls it.

What it computes ("DFlash 2" notes, "Solution - Two-Tap Dynamic
Convolution"): a short depthwise convolution reaching one block position back,
    Conv(x)_t = k_{t,0} * x_t + k_{t,1} * x_{t-1}     (* elementwise),
inserted before and after every attention and feed-forward sublayer, whose
coefficients combine a learned base kernel with a content-dependent
correction. Readings taken where the notes stop:
  - the correction of tap i at position t is a rank-r linear map of that
    position's own input: k_{t,i} = base_i + U_i (V_i x_t), base_i [H],
    V_i [r, H], U_i [H, r] (20 convolutions of two such taps with r = 80 at
    hidden 2560 come to the stated 16.5M parameters);
  - the block's first position (the anchor) has no predecessor: x_{-1} = 0;
    the first masked position reads the anchor, the last verified token, and
    every later position its predecessor;
  - "before" a sublayer is its normalised input, "after" its output before
    the residual add:
        x <- x + Conv_ao(Attn(Conv_ai(RMSNorm(x))))
        x <- x + Conv_fo(FFN(Conv_fi(RMSNorm(x))))
    (ai/ao/fi/fo: attention in/out, feed-forward in/out);
  - the injected context K/V do not pass through a convolution: it mixes
    block positions only.
Pins (tests/test_two_tap_conv_pins.py): identity kernels reproduce the plain
drafter pass exactly; zero output kernels leave the embedding rows; a pure
shift kernel moves rows down by one with a zero first row; the output at t
depends on inputs t and t - 1 only; the kernel is linear in x without a
correction, and the correction's effect scales with U.
"""
from __future__ import annotations

from typing import Dict, Sequence

import numpy as np

import oracle.dflash_oracle as od

TAPS = ("ai", "ao", "fi", "fo")


def conv2(x: np.ndarray, c: Dict[str, np.ndarray]) -> np.ndarray:
    """Two-tap dynamic convolution over block positions. x [B, H];
    c: base [2, H], U [2, H, r], V [2, r, H]."""
    prev = np.zeros_like(x)
    prev[1:] = x[:-1]
    out = np.zeros_like(x)
    for i, xi in ((0, x), (1, prev)):
        k = c["base"][i][None, :] + (x @ c["V"][i].T) @ c["U"][i].T   # coefficients from the position's own input
        out = out + k * xi
    return out


def decoder_layer_conv(x: np.ndarray, layer: Dict[str, np.ndarray], convs: Dict[str, Dict[str, np.ndarray]],
                       k_ctx: np.ndarray, v_ctx: np.ndarray, pos0: int, shape) -> np.ndarray:
    """One pre-norm drafter layer (as dflash_oracle.decoder_layer) with the
    four convolutions around its sublayers."""
    B = x.shape[0]
    nq, nkv, d = shape.n_heads, shape.n_kv_heads, shape.head_dim
    pos = pos0 + np.arange(B)
    h = conv2(od.rms_norm(x, layer["g_attn"], shape.rms_eps), convs["ai"])
    q = od.apply_rope((h @ layer["w_q"].T).reshape(B, nq, d), pos, shape.rope_base)
    k = od.apply_rope((h @ layer["w_k"].T).reshape(B, nkv, d), pos, shape.rope_base)
    v = (h @ layer["w_v"].T).reshape(B, nkv, d)
    keys = np.concatenate([k_ctx, k], axis=0)
    vals = np.concatenate([v_ctx, v], axis=0)
    a = od.block_attention(q, keys, vals).reshape(B, nq * d)
    x = x + conv2(a @ layer["w_o"].T, convs["ao"])
    h2 = conv2(od.rms_norm(x, layer["g_ffn"], shape.rms_eps), convs["fi"])
    f = (od.silu(h2 @ layer["w_gate"].T) * (h2 @ layer["w_up"].T)) @ layer["w_down"].T
    return x + conv2(f, convs["fo"])


def draft_block_conv(weights, shape, conv_weights: Sequence[Dict[str, Dict[str, np.ndarray]]], anchor: int,
                     k_ctx: Sequence[np.ndarray], v_ctx: Sequence[np.ndarray], B: int) -> Dict[str, np.ndarray]:
    """dflash_oracle.draft_block with the two-tap convolutions of every layer
    (conv_weights[l][tap] for tap in TAPS)."""
    C = k_ctx[0].shape[0] if len(k_ctx) else 0
    ids = np.array([anchor] + [shape.mask_id] * (B - 1), dtype=np.int64)
    x = weights["embed"][ids].copy()
    for layer, convs, kc, vc in zip(weights["layers"], conv_weights, k_ctx, v_ctx):
        x = decoder_layer_conv(x, layer, convs, kc, vc, C, shape)
    hf = od.rms_norm(x, weights["g_final"], shape.rms_eps)
    if B > 1:
        logits = hf[1:] @ weights["lm_head"].T
        return {"draft": od.rows_argmax(logits), "hidden": x, "top1": np.max(logits, axis=-1),
                "gap": od.top2_gap(logits), "logits": logits}
    return {"draft": np.zeros(0, dtype=np.int64), "hidden": x, "top1": np.zeros(0), "gap": np.zeros(0),
            "logits": np.zeros((0, weights["lm_head"].shape[0]))}


def identity_conv(H: int, r: int, dtype=np.float64) -> Dict[str, np.ndarray]:
    base = np.zeros((2, H), dtype=dtype)
    base[0] = 1.0
    return {"base": base, "U": np.zeros((2, H, r), dtype=dtype), "V": np.zeros((2, r, H), dtype=dtype)}
