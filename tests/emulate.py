"""bf16-storage emulation of the drafter pass (test infrastructure).

The library keeps the block's activations in bf16 between kernels (layer
inputs after RMSNorm, q/k/v after RoPE, attention output, SwiGLU output, the
cached K/V and H_t) and accumulates in fp32. This module repeats the oracle's
arithmetic with exactly those values rounded to bf16, so a test can measure how
far bf16 storage alone moves a pass from the exact oracle, and hold the CUDA
path to that. It uses the oracle's functions and no CUDA code.
"""
import numpy as np

import oracle.dflash_oracle as od
from synth import bf16_round


def r16(x, dtype=np.float64):
    """Round to the nearest bf16 value, returned in `dtype`."""
    return bf16_round(np.asarray(x, dtype=np.float32)).astype(dtype)


def bf16_context(w, sh, feats, dtype=np.float64):
    """Per-layer context K/V as the library caches them: H_t rounded to bf16,
    then K = RoPE(W_K H_t) and V = W_V H_t rounded to bf16."""
    ht = r16(od.fuse_features(np.asarray(feats, dtype), w["w_c"], w["g_c"], sh.rms_eps), dtype)
    pos = np.arange(ht.shape[0])
    kc, vc = [], []
    for lw in w["layers"]:
        k, v = od.context_kv(ht, lw, pos, sh.n_kv_heads, sh.head_dim, sh.rope_base)
        kc.append(r16(k, dtype))
        vc.append(r16(v, dtype))
    return kc, vc


def bf16_storage_hidden(w, sh, anchor, kc, vc, B, dtype=np.float64):
    """Final residual stream of one block with bf16 storage at the library's
    rounding points (the residual stream itself stays in full precision)."""
    C = kc[0].shape[0]
    x = np.asarray(w["embed"][[anchor] + [sh.mask_id] * (B - 1)], dtype).copy()
    pos = C + np.arange(B)
    for lw, k_ctx, v_ctx in zip(w["layers"], kc, vc):
        h = r16(od.rms_norm(x, lw["g_attn"], sh.rms_eps), dtype)
        q = r16(od.apply_rope((h @ lw["w_q"].T).reshape(B, sh.n_heads, sh.head_dim), pos, sh.rope_base), dtype)
        k = r16(od.apply_rope((h @ lw["w_k"].T).reshape(B, sh.n_kv_heads, sh.head_dim), pos, sh.rope_base), dtype)
        v = r16((h @ lw["w_v"].T).reshape(B, sh.n_kv_heads, sh.head_dim), dtype)
        a = r16(od.block_attention(q, np.concatenate([k_ctx, k]), np.concatenate([v_ctx, v])).reshape(B, -1), dtype)
        x = x + a @ lw["w_o"].T
        h2 = r16(od.rms_norm(x, lw["g_ffn"], sh.rms_eps), dtype)
        x = x + r16(od.silu(h2 @ lw["w_gate"].T) * (h2 @ lw["w_up"].T), dtype) @ lw["w_down"].T
    return x
