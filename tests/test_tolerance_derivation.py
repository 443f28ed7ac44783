"""Where the parity tolerance comes from.

The library stores the block's activations in bf16 between kernels (layer
inputs after RMSNorm, q/k/v, attention output, SwiGLU output, cached K/V,
H_t) and accumulates in fp32. This test emulates exactly those rounding
points in numpy on a drafter with the Qwen3-8B per-layer gain (weights of
std 0.04 at hidden 1024, i.e. std * sqrt(H) = 1.28, as 0.02 * sqrt(4096))
and checks how far an exact bf16-storage pass lands from the oracle: the
per-row relative L2 error stays near 1%, inside 2e-2, while single elements can
exceed an elementwise 5e-2 + 2e-2|x| bound. The GPU tests use the per-row
reading (tests/gpu_util.py). No CUDA code is involved.
"""
import numpy as np

import oracle.dflash_oracle as od
from synth import DrafterShape, make_weights_np, make_features_np
from tests.emulate import bf16_context, bf16_storage_hidden

SHAPE = DrafterShape(hidden=1024, n_heads=8, n_kv_heads=2, head_dim=128, ffn=3072, vocab=512, n_layers=2,
                     n_feat_layers=5, rope_base=1e6, rms_eps=1e-6, mask_id=511)


def test_bf16_storage_error_fits_the_row_relative_reading():
    sh = SHAPE
    wn = make_weights_np(sh, seed=5, gamma="jitter", std=0.04)
    w = {k: np.asarray(v, np.float64) for k, v in wn.items() if k != "layers"}
    w["layers"] = [{k: np.asarray(v, np.float64) for k, v in lw.items()} for lw in wn["layers"]]
    C, B = 200, 16
    f = make_features_np(C, sh.n_feat_layers * sh.hidden, seed=6).astype(np.float64)
    ht = od.fuse_features(f, w["w_c"], w["g_c"], sh.rms_eps)
    kc, vc = [], []
    for lw in w["layers"]:
        k, v = od.context_kv(ht, lw, np.arange(C), sh.n_kv_heads, sh.head_dim, sh.rope_base)
        kc.append(k)
        vc.append(v)
    kb, vb = bf16_context(w, sh, f)
    ref = od.draft_block(w, sh, 3, kc, vc, B)["hidden"]
    emu = bf16_storage_hidden(w, sh, 3, kb, vb, B)
    rel = np.linalg.norm(emu - ref, axis=1) / np.linalg.norm(ref, axis=1)
    assert rel.max() < 0.6 * 2e-2                     # the per-row reading holds with margin
    err = np.abs(emu - ref)
    assert (err <= 5e-2 + 2e-2 * np.abs(ref).max(axis=1, keepdims=True)).all()   # elementwise guard
    # the elementwise reading fails for some elements even for an exact bf16-storage pass
    assert (err > 5e-2 + 2e-2 * np.abs(ref)).any()
