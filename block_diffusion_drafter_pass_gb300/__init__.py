"""Python binding of libdflash (the DFlash drafter pass on GB300).

Argument marshalling only: every step of the drafter pass runs in the CUDA
kernels behind include/dflash.h. The functions named dflash_* mirror the C
entry points one to one; `Drafter` bundles a context with the torch tensors
it borrows. PyTorch supplies device memory and streams.

There is no fallback: if libdflash.so is missing or cannot load, every call
raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

from . import _build

LIB_PATH = _build.LIB

DFLASH_OK, DFLASH_EINVAL, DFLASH_ENOMEM, DFLASH_ECUDA, DFLASH_ETIMEOUT, DFLASH_EDEVICE = range(6)
_STATUS_NAMES = {0: "OK", 1: "EINVAL", 2: "ENOMEM", 3: "ECUDA", 4: "ETIMEOUT", 5: "EDEVICE"}

# Entry points declared in include/dflash.h.
EXPORTED = (
    "dflash_create", "dflash_destroy", "dflash_last_error", "dflash_seq_reset", "dflash_seq_len",
    "dflash_fuse_ctx", "dflash_draft", "dflash_verify", "dflash_rows_argmax_bf16", "dflash_sync",
    "dflash_debug_read_kv", "dflash_debug_last_draft", "dflash_debug_gemm", "dflash_debug_profile",
    "dflash_debug_profile_read", "dflash_gemm_noalloc", "dflash_set_path_selector", "dflash_debug_last_selection",
    "dflash_draft_sample", "dflash_sample_filter", "dflash_verify_sample",
    "dflash_block_sched_create", "dflash_block_sched_destroy", "dflash_block_sched_observe",
    "dflash_block_sched_set_cost", "dflash_block_sched_expected_tau", "dflash_block_sched_choose",
    "dflash_debug_wait_timeout", "dflash_target_feature_layers", "dflash_target_create", "dflash_target_forward",
    "dflash_debug_read_kv_q8", "dflash_set_conv",
)
SAMPLE_WIDTH = 32   # DFLASH_SAMPLE_WIDTH

# Kernel classes of the per-kernel accounting (DFLASH_K_* in include/dflash.h).
KERNEL_CLASSES = ("qkv", "attn", "attn_combine", "o", "gateup", "down", "lmhead", "fuse_wc", "fuse_kv", "norm",
                  "verify", "other", "select", "sample", "conv")


class DFlashError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"dflash {_STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class dflash_config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("hidden", "n_heads", "n_kv_heads", "head_dim", "ffn", "vocab",
                                            "n_layers", "n_feat_layers")] + [
        ("rope_base", ctypes.c_float), ("rms_eps", ctypes.c_float)] + [
        (n, ctypes.c_int) for n in ("mask_id", "max_seqs", "max_batch", "max_block", "max_ctx", "max_pages",
                                    "max_fuse_tokens", "kv_format")]


class dflash_layer_weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("w_q", "w_k", "w_v", "w_o", "w_gate", "w_up", "w_down",
                                               "g_attn", "g_ffn")]


class dflash_conv_site(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("base", "u", "v")]


CONV_SITES = ("ai", "ao", "fi", "fo")   # per layer: attention in/out, feed-forward in/out


class dflash_kernel_stat(ctypes.Structure):
    _fields_ = [("launches", ctypes.c_longlong), ("ms", ctypes.c_double), ("bytes", ctypes.c_double),
                ("flops", ctypes.c_double)]


class dflash_weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("w_c", "g_c", "embed", "lm_head", "g_final")] + [
        ("layers", ctypes.POINTER(dflash_layer_weights))]


_lib = None


def load_library() -> ctypes.CDLL:
    """Load libdflash.so (built by __graft_entry__.build()). Raises if absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise DFlashError(DFLASH_ECUDA, f"{LIB_PATH} is missing; build it with __graft_entry__.build()")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, VP = ctypes.POINTER, ctypes.c_int, ctypes.c_void_p
    i32p = P(ctypes.c_int32)
    sigs = {
        "dflash_create": ([P(dflash_config), P(dflash_weights), P(VP)], I),
        "dflash_destroy": ([VP], I),
        "dflash_last_error": ([VP], ctypes.c_char_p),
        "dflash_seq_reset": ([VP, I], I),
        "dflash_seq_len": ([VP, I, P(I), P(I)], I),
        "dflash_fuse_ctx": ([VP, i32p, I, i32p, VP, I, VP], I),
        "dflash_draft": ([VP, i32p, I, VP, I, VP, VP], I),
        "dflash_verify": ([VP, i32p, I, I, VP, VP, VP, VP, VP], I),
        "dflash_rows_argmax_bf16": ([VP, I, I, VP, VP], I),
        "dflash_sync": ([VP], I),
        "dflash_debug_read_kv": ([VP, I, I, I, I, VP, VP], I),
        "dflash_debug_read_kv_q8": ([VP, I, I, I, I, VP, VP, VP, VP], I),
        "dflash_debug_last_draft": ([VP, VP, VP], I),
        "dflash_debug_gemm": ([VP, VP, VP, I, I, I, I, VP], I),
        "dflash_debug_profile": ([VP, I], I),
        "dflash_debug_profile_read": ([VP, P(dflash_kernel_stat), I], I),
        "dflash_gemm_noalloc": ([VP, VP, VP, I, I, I, I, VP], I),
        "dflash_set_path_selector": ([VP, VP, VP, VP, I, VP], I),
        "dflash_set_conv": ([VP, VP, I, VP], I),
        "dflash_debug_last_selection": ([VP, VP, VP, VP], I),
        "dflash_draft_sample": ([VP, i32p, I, VP, I, ctypes.c_float, I, ctypes.c_float, VP, VP, VP, VP, VP], I),
        "dflash_sample_filter": ([VP, VP, I, I, ctypes.c_float, I, ctypes.c_float, VP, VP, VP, VP, VP], I),
        "dflash_verify_sample": ([VP, i32p, I, I, VP, VP, VP, VP, VP, VP, VP, VP, VP, VP], I),
        "dflash_block_sched_create": ([i32p, I, ctypes.c_float, ctypes.c_float, ctypes.c_float, P(VP)], I),
        "dflash_block_sched_destroy": ([VP], I),
        "dflash_block_sched_observe": ([VP, I, i32p, I], I),
        "dflash_block_sched_set_cost": ([VP, I, ctypes.c_float], I),
        "dflash_block_sched_expected_tau": ([VP, I, P(ctypes.c_double)], I),
        "dflash_block_sched_choose": ([VP, P(I)], I),
        "dflash_debug_wait_timeout": ([VP, I, VP], I),
        "dflash_target_feature_layers": ([I, I, i32p], I),
        "dflash_target_create": ([P(dflash_config), P(dflash_weights), i32p, P(VP)], I),
        "dflash_target_forward": ([VP, i32p, I, VP, I, I, VP, VP, VP], I),
    }
    for name, (args, res) in sigs.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def _check(status: int, ctx=None) -> None:
    if status != DFLASH_OK:
        msg = load_library().dflash_last_error(ctx)
        raise DFlashError(status, msg.decode() if msg else "")


def _i32(seq: Sequence[int]):
    arr = (ctypes.c_int32 * max(1, len(seq)))(*[int(v) for v in seq])
    return arr


def _stream(stream) -> Optional[int]:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t) -> int:
    return 0 if t is None else t.data_ptr()


# --- one-to-one wrappers of the C entry points -------------------------------

def dflash_rows_argmax_bf16(logits, out=None, stream=None):
    """Row argmax of bf16 logits [rows, cols] (lowest index on ties) -> int32 [rows]."""
    import torch
    assert logits.dtype == torch.bfloat16 and logits.is_cuda and logits.is_contiguous()
    rows, cols = logits.shape
    if out is None:
        out = torch.empty(rows, dtype=torch.int32, device=logits.device)
    _check(load_library().dflash_rows_argmax_bf16(_ptr(logits), rows, cols, _ptr(out), _stream(stream)))
    return out


def dflash_debug_gemm(W, X, splits: int = 0, stream=None):
    """Y = X W^T in fp32 with the library's tcgen05 GEMM (W [N,K], X [M,K] bf16)."""
    import torch
    N, K = W.shape
    M = X.shape[0]
    Y = torch.empty(M, N, dtype=torch.float32, device=W.device)
    _check(load_library().dflash_debug_gemm(_ptr(W), _ptr(X), _ptr(Y), N, M, K, splits, _stream(stream)))
    return Y


def dflash_gemm_noalloc(W, X, Y=None, splits: int = 0, stream=None):
    """Y = X W^T (fp32) with no device allocation inside the library; the
    split-K scratch is a fixed array the library keeps on each GPU. Pass Y
    (fp32 [M, N], preallocated) when the caller itself cannot allocate."""
    import torch
    N, K = W.shape
    M = X.shape[0]
    if Y is None:
        Y = torch.empty(M, N, dtype=torch.float32, device=W.device)
    _check(load_library().dflash_gemm_noalloc(_ptr(W), _ptr(X), _ptr(Y), N, M, K, splits, _stream(stream)))
    return Y


class BlockScheduler:
    """Dynamic block-size scheduling (host logic in the library, no GPU needed):
    observe acceptance lengths, set per-size cycle costs, choose the next B."""

    def __init__(self, sizes, decay: float = 0.99, prior_accept: float = 1.0, prior_reject: float = 1.0):
        lib = load_library()
        h = ctypes.c_void_p()
        _check(lib.dflash_block_sched_create(_i32(sizes), len(sizes), float(decay), float(prior_accept),
                                             float(prior_reject), ctypes.byref(h)))
        self.h = h

    def observe(self, B: int, taus) -> None:
        taus = [int(t) for t in taus]
        _check(load_library().dflash_block_sched_observe(self.h, int(B), _i32(taus), len(taus)))

    def set_cost(self, B: int, cycle_ms: float) -> None:
        _check(load_library().dflash_block_sched_set_cost(self.h, int(B), float(cycle_ms)))

    def expected_tau(self, B: int) -> float:
        v = ctypes.c_double()
        _check(load_library().dflash_block_sched_expected_tau(self.h, int(B), ctypes.byref(v)))
        return v.value

    def choose(self) -> int:
        b = ctypes.c_int()
        _check(load_library().dflash_block_sched_choose(self.h, ctypes.byref(b)))
        return b.value

    def close(self) -> None:
        if getattr(self, "h", None):
            load_library().dflash_block_sched_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class Drafter:
    """A dflash context plus the bf16 device weights it borrows.

    `weights` follows synth.make_weights_torch: w_c, g_c, embed, lm_head,
    g_final and layers[i] = {w_q, w_k, w_v, w_o, w_gate, w_up, w_down,
    g_attn, g_ffn}, all contiguous torch.bfloat16 CUDA tensors.
    """

    def __init__(self, shape, weights, *, max_seqs: int = 4, max_batch: int = 4, max_block: int = 16,
                 max_ctx: int = 4096, max_pages: Optional[int] = None, max_fuse_tokens: int = 1024,
                 kv_format: int = 0, _feat_layers=None):
        import torch
        lib = load_library()
        self.shape = shape
        self._weights = weights  # keep the borrowed tensors alive
        top = ("embed", "lm_head", "g_final") if _feat_layers is not None else ("w_c", "g_c", "embed", "lm_head",
                                                                                "g_final")
        for t in [weights[k] for k in top] + [v for lw in weights["layers"] for v in lw.values()]:
            if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
                raise DFlashError(DFLASH_EINVAL, "weights must be contiguous bf16 CUDA tensors")
        if max_pages is None:
            max_pages = max_seqs * ((max_ctx + 63) // 64)
        self.cfg = dflash_config(shape.hidden, shape.n_heads, shape.n_kv_heads, shape.head_dim, shape.ffn,
                                 shape.vocab, shape.n_layers, shape.n_feat_layers, shape.rope_base,
                                 shape.rms_eps, shape.mask_id, max_seqs, max_batch, max_block, max_ctx,
                                 max_pages, max_fuse_tokens, kv_format)
        layers = (dflash_layer_weights * shape.n_layers)()
        for i, lw in enumerate(weights["layers"]):
            layers[i] = dflash_layer_weights(*[_ptr(lw[k]) for k in ("w_q", "w_k", "w_v", "w_o", "w_gate",
                                                                      "w_up", "w_down", "g_attn", "g_ffn")])
        self._layers = layers
        w = dflash_weights(_ptr(weights.get("w_c")), _ptr(weights.get("g_c")), _ptr(weights["embed"]),
                           _ptr(weights["lm_head"]), _ptr(weights["g_final"]), layers)
        ctx = ctypes.c_void_p()
        if _feat_layers is None:
            _check(lib.dflash_create(ctypes.byref(self.cfg), ctypes.byref(w), ctypes.byref(ctx)), None)
        else:
            _check(lib.dflash_target_create(ctypes.byref(self.cfg), ctypes.byref(w), _i32(_feat_layers),
                                            ctypes.byref(ctx)), None)
        self.ctx = ctx
        self.device = weights["embed"].device

    # lifecycle ---------------------------------------------------------------
    def close(self) -> None:
        if getattr(self, "ctx", None):
            load_library().dflash_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    # the hot path ----------------------------------------------------------------
    def fuse_ctx(self, seq_ids, n_new, feats, pending: bool, stream=None) -> None:
        import torch
        assert feats is None or (feats.dtype == torch.bfloat16 and feats.is_cuda and feats.is_contiguous())
        _check(load_library().dflash_fuse_ctx(self.ctx, _i32(seq_ids), len(seq_ids), _i32(n_new), _ptr(feats),
                                              1 if pending else 0, _stream(stream)), self.ctx)

    def draft(self, seq_ids, anchor_ids, B: int, out=None, stream=None):
        import torch
        n = len(seq_ids)
        if out is None:
            out = torch.empty(n, max(B - 1, 0), dtype=torch.int32, device=self.device)
        assert anchor_ids.dtype == torch.int32 and anchor_ids.is_cuda
        _check(load_library().dflash_draft(self.ctx, _i32(seq_ids), n, _ptr(anchor_ids), B,
                                           _ptr(out) if out.numel() else 0, _stream(stream)), self.ctx)
        return out

    def verify(self, seq_ids, B: int, draft_ids, target_ids, tau=None, bonus=None, stream=None):
        import torch
        n = len(seq_ids)
        if tau is None:
            tau = torch.empty(n, dtype=torch.int32, device=self.device)
        if bonus is None:
            bonus = torch.empty(n, dtype=torch.int32, device=self.device)
        dptr = _ptr(draft_ids) if draft_ids is not None and draft_ids.numel() else 0
        _check(load_library().dflash_verify(self.ctx, _i32(seq_ids), n, B, dptr, _ptr(target_ids), _ptr(tau),
                                            _ptr(bonus), _stream(stream)), self.ctx)
        return tau, bonus

    def set_path_selector(self, w_a=None, w_b=None, w_h=None, stream=None) -> None:
        """Install the DFlash 2 path selector (W_A, W_B, W_H: contiguous bf16
        CUDA tensors [256, H]); no arguments removes it. While installed,
        draft() returns the selector's walk over the top-16 candidates."""
        import torch
        ws = (w_a, w_b, w_h)
        if all(w is None for w in ws):
            _check(load_library().dflash_set_path_selector(self.ctx, 0, 0, 0, 256, _stream(stream)), self.ctx)
            self._sel = None
            return
        for w in ws:
            if w is None or w.dtype != torch.bfloat16 or not w.is_cuda or not w.is_contiguous() or w.dim() != 2:
                raise DFlashError(DFLASH_EINVAL, "selector weights must be contiguous bf16 CUDA matrices")
        _check(load_library().dflash_set_path_selector(self.ctx, _ptr(w_a), _ptr(w_b), _ptr(w_h), w_a.shape[0],
                                                       _stream(stream)), self.ctx)
        self._sel = ws   # W_H is read by every draft

    def set_conv(self, sites=None, rank: int = 0, stream=None) -> None:
        """Install the DFlash 2 two-tap convolutions: `sites` is a list over
        layers of dicts {"ai", "ao", "fi", "fo"} of dicts {"base" [2, H],
        "U" [2, H, r], "V" [2, r, H]} (contiguous bf16 CUDA tensors); None
        removes them."""
        import torch
        if sites is None:
            _check(load_library().dflash_set_conv(self.ctx, None, 0, _stream(stream)), self.ctx)
            self._conv = None
            return
        arr = (dflash_conv_site * (4 * len(sites)))()
        keep = []
        for l, layer in enumerate(sites):
            for k, name in enumerate(CONV_SITES):
                c = layer[name]
                for key in ("base", "U", "V"):
                    t = c[key]
                    if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
                        raise DFlashError(DFLASH_EINVAL, "conv arrays must be contiguous bf16 CUDA tensors")
                    keep.append(t)
                arr[4 * l + k] = dflash_conv_site(_ptr(c["base"]), _ptr(c["U"]), _ptr(c["V"]))
        _check(load_library().dflash_set_conv(self.ctx, ctypes.cast(arr, ctypes.c_void_p), rank, _stream(stream)),
               self.ctx)
        self._conv = keep   # borrowed by every draft

    # temperature sampling ------------------------------------------------------
    def draft_sample(self, seq_ids, anchor_ids, B: int, temperature: float, top_k: int, top_p: float, uniforms,
                     out=None, q_ids=None, q_probs=None, stream=None):
        """Drafter pass with a sampling head: (draft ids [n, B-1], q ids
        [n, B-1, 32], q probs [n, B-1, 32]); uniforms fp32 [n, B-1] on the device."""
        import torch
        n = len(seq_ids)
        T = max(B - 1, 0)
        if out is None:
            out = torch.empty(n, T, dtype=torch.int32, device=self.device)
        if q_ids is None:
            q_ids = torch.empty(n, T, SAMPLE_WIDTH, dtype=torch.int32, device=self.device)
        if q_probs is None:
            q_probs = torch.empty(n, T, SAMPLE_WIDTH, dtype=torch.float32, device=self.device)
        assert anchor_ids.dtype == torch.int32 and anchor_ids.is_cuda
        assert uniforms is None or (uniforms.dtype == torch.float32 and uniforms.is_contiguous())
        _check(load_library().dflash_draft_sample(self.ctx, _i32(seq_ids), n, _ptr(anchor_ids), B, float(temperature),
                                                  int(top_k), float(top_p), _ptr(uniforms),
                                                  _ptr(out) if out.numel() else 0, _ptr(q_ids) if q_ids.numel() else 0,
                                                  _ptr(q_probs) if q_probs.numel() else 0, _stream(stream)), self.ctx)
        return out, q_ids, q_probs

    def sample_filter(self, logits, temperature: float, top_k: int, top_p: float, uniforms=None, ids=None,
                      probs=None, drawn=None, stream=None):
        """Filtered distributions of bf16 logit rows [rows, V]: (ids [rows, 32],
        probs [rows, 32], draws [rows] or None when no uniforms are given)."""
        import torch
        assert logits.dtype == torch.bfloat16 and logits.is_cuda and logits.is_contiguous()
        rows, cols = logits.shape
        if ids is None:
            ids = torch.empty(rows, SAMPLE_WIDTH, dtype=torch.int32, device=logits.device)
        if probs is None:
            probs = torch.empty(rows, SAMPLE_WIDTH, dtype=torch.float32, device=logits.device)
        if uniforms is not None and drawn is None:
            drawn = torch.empty(rows, dtype=torch.int32, device=logits.device)
        _check(load_library().dflash_sample_filter(self.ctx, _ptr(logits), rows, cols, float(temperature), int(top_k),
                                                   float(top_p), _ptr(uniforms), _ptr(ids), _ptr(probs),
                                                   _ptr(drawn), _stream(stream)), self.ctx)
        return ids, probs, drawn

    def verify_sample(self, seq_ids, B: int, draft_ids, q_ids, q_probs, p_ids, p_probs, u_accept, u_resample,
                      tau=None, bonus=None, stream=None):
        """Lossless speculative-sampling verify + commit -> (tau, token)."""
        import torch
        n = len(seq_ids)
        if tau is None:
            tau = torch.empty(n, dtype=torch.int32, device=self.device)
        if bonus is None:
            bonus = torch.empty(n, dtype=torch.int32, device=self.device)
        nz = lambda t: _ptr(t) if t is not None and t.numel() else 0
        _check(load_library().dflash_verify_sample(self.ctx, _i32(seq_ids), n, B, nz(draft_ids), nz(q_ids),
                                                   nz(q_probs), _ptr(p_ids), _ptr(p_probs), nz(u_accept),
                                                   _ptr(u_resample), _ptr(tau), _ptr(bonus), _stream(stream)),
               self.ctx)
        return tau, bonus

    # state and inspection ------------------------------------------------------
    def seq_reset(self, seq: int) -> None:
        _check(load_library().dflash_seq_reset(self.ctx, seq), self.ctx)

    def seq_len(self, seq: int):
        c, p = ctypes.c_int(), ctypes.c_int()
        _check(load_library().dflash_seq_len(self.ctx, seq, ctypes.byref(c), ctypes.byref(p)), self.ctx)
        return c.value, p.value

    def sync(self) -> None:
        _check(load_library().dflash_sync(self.ctx), self.ctx)

    def debug_wait_timeout(self, limit_us: int, stream=None) -> None:
        """Launch one bounded wait that runs out after limit_us (failure-path check)."""
        _check(load_library().dflash_debug_wait_timeout(self.ctx, int(limit_us), _stream(stream)), self.ctx)

    def read_kv(self, layer: int, seq: int, pos0: int, n: int):
        """Cached K, V of `n` positions as float32 arrays [n, n_kv, d]."""
        import numpy as np
        sh = self.shape
        k = np.empty((n, sh.n_kv_heads, sh.head_dim), dtype=np.uint16)
        v = np.empty_like(k)
        _check(load_library().dflash_debug_read_kv(self.ctx, layer, seq, pos0, n, k.ctypes.data, v.ctypes.data),
               self.ctx)
        f = lambda a: (a.astype(np.uint32) << 16).view(np.float32)
        return f(k), f(v)

    def read_kv_q8(self, layer: int, seq: int, pos0: int, n: int):
        """The stored 8-bit blocks (kv_format 1): K codes, K scales, V codes,
        V scales; codes int8 [n, n_kv, d], scales float32 [n, n_kv, d/32]
        (the stored fp16 values)."""
        import numpy as np
        sh = self.shape
        kc = np.empty((n, sh.n_kv_heads, sh.head_dim), dtype=np.int8)
        vc = np.empty_like(kc)
        ks = np.empty((n, sh.n_kv_heads, sh.head_dim // 32), dtype=np.uint16)
        vs = np.empty_like(ks)
        _check(load_library().dflash_debug_read_kv_q8(self.ctx, layer, seq, pos0, n, kc.ctypes.data, ks.ctypes.data,
                                                      vc.ctypes.data, vs.ctypes.data), self.ctx)
        return kc, ks.view(np.float16).astype(np.float32), vc, vs.view(np.float16).astype(np.float32)

    def profile(self, enable: bool) -> None:
        """Event-time every kernel launch (on its launch stream) while enabled."""
        _check(load_library().dflash_debug_profile(self.ctx, 1 if enable else 0), self.ctx)

    def profile_read(self):
        """Per kernel class: launches, summed ms, algorithmic bytes and flops
        since the last read (synchronises, then resets the totals)."""
        n = len(KERNEL_CLASSES)
        arr = (dflash_kernel_stat * n)()
        _check(load_library().dflash_debug_profile_read(self.ctx, arr, n), self.ctx)
        return {name: {"launches": int(a.launches), "ms": float(a.ms), "bytes": float(a.bytes),
                       "flops": float(a.flops)} for name, a in zip(KERNEL_CLASSES, arr)}

    def last_draft(self, n_seq: int, B: int):
        """(final residual stream [n_seq*B, H] fp32, winning logits [n_seq*(B-1)] fp32) of the last draft."""
        import numpy as np
        hid = np.empty((n_seq * B, self.shape.hidden), dtype=np.float32)
        top = np.empty(max(1, n_seq * (B - 1)), dtype=np.float32)
        _check(load_library().dflash_debug_last_draft(self.ctx, hid.ctypes.data, top.ctypes.data), self.ctx)
        return hid, top[: n_seq * (B - 1)]

    def last_selection(self, n_seq: int, B: int):
        """(candidate ids [rows, 16], their logits [rows, 16], pair scores
        [rows, 16, 16]) of the last draft that ran the path selector, rows =
        n_seq * (B - 1) in sequence-major order."""
        import numpy as np
        rows = n_seq * (B - 1)
        cand = np.empty((max(1, rows), 16), dtype=np.int32)
        u = np.empty((max(1, rows), 16), dtype=np.float32)
        sc = np.empty((max(1, rows), 16, 16), dtype=np.float32)
        _check(load_library().dflash_debug_last_selection(self.ctx, cand.ctypes.data, u.ctypes.data,
                                                          sc.ctypes.data), self.ctx)
        return cand[:rows], u[:rows], sc[:rows]


def target_feature_layers(n_layers: int, n_feat: int = 5):
    """The library's default feature layers (0-based) of an n_layers target."""
    out = (ctypes.c_int32 * n_feat)()
    _check(load_library().dflash_target_feature_layers(n_layers, n_feat, out), None)
    return [int(x) for x in out]


class Target(Drafter):
    """A target context (dflash_target_create): the causal verify pass that
    caches its own K/V and hands its feature layers' outputs to the drafter.
    `shape.n_feat_layers` is the number of feature layers; `weights` as for
    Drafter without w_c and g_c. dflash_verify, seq_len, read_kv and the
    other inspection hooks work as on a Drafter."""

    def __init__(self, shape, weights, feat_layers=None, *, max_seqs: int = 4, max_batch: int = 4,
                 max_block: int = 16, max_ctx: int = 4096, max_pages: Optional[int] = None):
        if feat_layers is None:
            feat_layers = target_feature_layers(shape.n_layers, shape.n_feat_layers)
        self.feat_layers = list(feat_layers)
        super().__init__(shape, weights, max_seqs=max_seqs, max_batch=max_batch, max_block=max_block,
                         max_ctx=max_ctx, max_pages=max_pages, max_fuse_tokens=1, _feat_layers=self.feat_layers)

    def forward(self, seq_ids, block_ids, B: int, pending: bool, out=None, feats=None, want_feats: bool = True,
                stream=None):
        """One causal pass over block_ids [n, B] (int32 CUDA). Returns
        (target ids [n, B], features [n * B, n_feat * H] bf16 or None)."""
        import torch
        n = len(seq_ids)
        assert block_ids.dtype == torch.int32 and block_ids.is_cuda and block_ids.is_contiguous()
        if out is None:
            out = torch.empty(n, B, dtype=torch.int32, device=self.device)
        if feats is None and want_feats and self.feat_layers:
            feats = torch.empty(n * B, len(self.feat_layers) * self.shape.hidden, dtype=torch.bfloat16,
                                device=self.device)
        _check(load_library().dflash_target_forward(self.ctx, _i32(seq_ids), n, _ptr(block_ids), B,
                                                    1 if pending else 0, _ptr(out), _ptr(feats), _stream(stream)),
               self.ctx)
        return out, feats

    def last_pass(self, n_seq: int, B: int):
        """(final residual stream [n_seq*B, H] fp32, winning logit of every
        block position [n_seq*B] fp32) of the last forward."""
        import numpy as np
        hid = np.empty((n_seq * B, self.shape.hidden), dtype=np.float32)
        top = np.empty(n_seq * B, dtype=np.float32)
        _check(load_library().dflash_debug_last_draft(self.ctx, hid.ctypes.data, top.ctypes.data), self.ctx)
        return hid, top
