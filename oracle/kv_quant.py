"""CPU oracle of 8-bit block quantisation of the drafter's context K/V cache.

TEST INFRASTRUCTURE. Only the tests may import this module. The CUDA library
does not store quantised pages yet; when it does, it shares no code with this
module.

What it computes. The pages run the target with its KV cache in the q8_0
format (the llama.cpp command lines of the Gemma write-up pass -ctk q8_0
-ctv q8_0); per-page 8-bit KV is the compression the long-context drafter
pass needs (its context K/V are the dominant traffic at 262K tokens).
Readings, restating that published block format:
  - a K or V row of one head (head_dim values) is cut into blocks of 32
    consecutive values; a block's scale is d = max|x| / 127, stored as fp16;
    its codes are q = round(x / d) as int8, halves rounded away from zero
    (q = 0 for an all-zero block); the decoded value is q * fp16(d);
  - every row written to the paged cache (committed or pending context) is
    stored this way; the block's own K/V, computed inside the pass, are not
    cached and stay unquantised;
  - attention reads the decoded values.
Pins (tests/test_kv_quant_pins.py): rows that are exact multiples of a scale
representable in fp16 decode exactly; the decode error is within half a step
plus the scale's fp16 rounding; zero blocks decode to zero; the code is odd
in x; the drafter pass over exactly representable context K/V equals the plain
pass, and with arbitrary context it moves the hidden state by no more than
the decode error allows.
"""
from __future__ import annotations

from typing import Dict, Sequence

import numpy as np

import oracle.dflash_oracle as od

BLOCK = 32
QMAX = 127


def _round_half_away(x: np.ndarray) -> np.ndarray:
    return np.sign(x) * np.floor(np.abs(x) + 0.5)


def quantize(x: np.ndarray):
    """x [..., n] with n a multiple of 32 -> (codes int8 [..., n], scales fp16 [..., n/32])."""
    x = np.asarray(x, dtype=np.float64)
    blocks = x.reshape(x.shape[:-1] + (x.shape[-1] // BLOCK, BLOCK))
    amax = np.max(np.abs(blocks), axis=-1)
    d = amax / QMAX
    inv = np.where(d > 0, 1.0 / np.where(d > 0, d, 1.0), 0.0)
    q = _round_half_away(blocks * inv[..., None]).astype(np.int8)
    return q.reshape(x.shape), d.astype(np.float16)


def dequantize(q: np.ndarray, scales: np.ndarray) -> np.ndarray:
    blocks = q.astype(np.float64).reshape(q.shape[:-1] + (q.shape[-1] // BLOCK, BLOCK))
    return (blocks * scales.astype(np.float64)[..., None]).reshape(q.shape)


def roundtrip(x: np.ndarray) -> np.ndarray:
    return dequantize(*quantize(x))


def draft_block_quantized_ctx(weights, shape, anchor: int, k_ctx: Sequence[np.ndarray],
                              v_ctx: Sequence[np.ndarray], B: int) -> Dict[str, np.ndarray]:
    """dflash_oracle.draft_block with every context K/V row stored in the
    8-bit block format (per head row of head_dim values) and decoded for attention."""
    kq = [roundtrip(k) for k in k_ctx]
    vq = [roundtrip(v) for v in v_ctx]
    return od.draft_block(weights, shape, anchor, kq, vq, B)
