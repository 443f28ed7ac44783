"""Plant plausible mistakes in the oracle and check that some pin catches each.

Each mutation replaces one oracle function (on the CPU, for the duration of one
test) with a subtly wrong version: a dropped term, a wrong sign or index, a
transposed operand. The pins in test_oracle_pins.py must then fail.
"""
import math

import numpy as np
import pytest

import oracle
import oracle.dflash_oracle as od
from tests import test_oracle_pins as pins


def _patch(monkeypatch, name, fn):
    monkeypatch.setattr(od, name, fn)
    monkeypatch.setattr(oracle, name, fn)


def _expect_failure(test_fn):
    with pytest.raises(AssertionError):
        test_fn()


def test_rope_sign_error_is_caught(monkeypatch):
    def bad(x, positions, base):
        n, _, d = x.shape
        ang = od.rope_angles(positions, d, base)
        c, s = np.cos(ang)[:, None, :], np.sin(ang)[:, None, :]
        lo, hi = x[..., : d // 2], x[..., d // 2:]
        return np.concatenate([lo * c + hi * s, hi * c - lo * s], axis=-1)
    _patch(monkeypatch, "apply_rope", bad)
    _expect_failure(pins.test_rope_matches_complex_rotation)
    _expect_failure(pins.test_draft_pass_matches_scalar_brute_force)


def test_rope_interleaved_pairing_is_caught(monkeypatch):
    def bad(x, positions, base):
        n, _, d = x.shape
        ang = od.rope_angles(positions, d, base)
        c, s = np.cos(ang)[:, None, :], np.sin(ang)[:, None, :]
        ev, odd = x[..., 0::2], x[..., 1::2]
        out = np.empty_like(x)
        out[..., 0::2] = ev * c - odd * s
        out[..., 1::2] = odd * c + ev * s
        return out
    _patch(monkeypatch, "apply_rope", bad)
    _expect_failure(pins.test_rope_matches_complex_rotation)


def test_gqa_head_mapping_error_is_caught(monkeypatch):
    orig = od.block_attention

    def bad(q, k, v, return_probs=False):
        n_kv = k.shape[1]
        g = q.shape[1] // n_kv
        perm = [h % n_kv for h in range(q.shape[1])]  # modulo instead of integer division
        kk = k[:, perm, :]
        vv = v[:, perm, :]
        return orig(q, kk, vv, return_probs) if g > 1 else orig(q, k, v, return_probs)
    _patch(monkeypatch, "block_attention", bad)
    _expect_failure(pins.test_attention_matches_explicit_loops)


def test_missing_attention_scale_is_caught(monkeypatch):
    orig = od.block_attention

    def bad(q, k, v, return_probs=False):
        return orig(q * math.sqrt(q.shape[-1]), k, v, return_probs)
    _patch(monkeypatch, "block_attention", bad)
    _expect_failure(pins.test_attention_matches_explicit_loops)


def test_dropped_ffn_residual_is_caught(monkeypatch):
    def bad(x, layer, k_ctx, v_ctx, pos0, shape):
        B = x.shape[0]
        nq, nkv, d = shape.n_heads, shape.n_kv_heads, shape.head_dim
        pos = pos0 + np.arange(B)
        h = od.rms_norm(x, layer["g_attn"], shape.rms_eps)
        q = od.apply_rope((h @ layer["w_q"].T).reshape(B, nq, d), pos, shape.rope_base)
        k = od.apply_rope((h @ layer["w_k"].T).reshape(B, nkv, d), pos, shape.rope_base)
        v = (h @ layer["w_v"].T).reshape(B, nkv, d)
        a = od.block_attention(q, np.concatenate([k_ctx, k]), np.concatenate([v_ctx, v])).reshape(B, nq * d)
        x = x + a @ layer["w_o"].T
        h2 = od.rms_norm(x, layer["g_ffn"], shape.rms_eps)
        return (od.silu(h2 @ layer["w_gate"].T) * (h2 @ layer["w_up"].T)) @ layer["w_down"].T
    _patch(monkeypatch, "decoder_layer", bad)
    _expect_failure(pins.test_decoder_B1_C0_is_a_single_step)


def test_transposed_output_projection_is_caught(monkeypatch):
    orig = od.decoder_layer

    def bad(x, layer, k_ctx, v_ctx, pos0, shape):
        lw = dict(layer)
        lw["w_o"] = layer["w_o"].T.copy()
        return orig(x, lw, k_ctx, v_ctx, pos0, shape)
    _patch(monkeypatch, "decoder_layer", bad)
    _expect_failure(pins.test_decoder_B1_C0_is_a_single_step)


def test_swapped_gate_and_up_is_caught(monkeypatch):
    orig = od.decoder_layer

    def bad(x, layer, k_ctx, v_ctx, pos0, shape):
        lw = dict(layer)
        lw["w_gate"], lw["w_up"] = layer["w_up"], layer["w_gate"]
        return orig(x, lw, k_ctx, v_ctx, pos0, shape)
    _patch(monkeypatch, "decoder_layer", bad)
    _expect_failure(pins.test_decoder_B1_C0_is_a_single_step)


def test_fusion_without_norm_is_caught(monkeypatch):
    def bad(feats, w_c, g_c, eps):
        return (feats @ w_c.T) * g_c
    _patch(monkeypatch, "fuse_features", bad)
    _expect_failure(pins.test_draft_pass_matches_scalar_brute_force)


def test_causal_mask_is_caught(monkeypatch):
    """A causal block (mask positions blind to later positions) is not the
    non-causal attention the pages describe."""
    def bad(q, k, v, return_probs=False):
        B, n_q, d = q.shape
        T = k.shape[0]
        g = n_q // k.shape[1]
        out = np.empty_like(q)
        for h in range(n_q):
            s = q[:, h, :] @ k[:, h // g, :].T / math.sqrt(d)
            for b in range(B):
                s[b, T - B + b + 1:] = -np.inf
            s = s - s.max(-1, keepdims=True)
            p = np.exp(s)
            p /= p.sum(-1, keepdims=True)
            out[:, h, :] = p @ v[:, h // g, :]
        return out
    _patch(monkeypatch, "block_attention", bad)
    _expect_failure(pins.test_draft_pass_matches_scalar_brute_force)


@pytest.mark.parametrize("kind", ["third_value", "distinct_values", "wrong_axis"])
def test_top2_gap_mistakes_are_caught(monkeypatch, kind):
    """top2_gap picks the rows whose draft ids must match bit for bit; a
    mistake would silently grow or shrink that set."""
    def bad(logits):
        if kind == "third_value":        # top-1 minus the third-largest value
            part = np.partition(logits, -3, axis=-1)
            return part[..., -1] - part[..., -3]
        if kind == "distinct_values":    # a repeated maximum skipped: ties look certain
            out = []
            for row in np.reshape(logits, (-1, logits.shape[-1])):
                u = np.unique(row)
                out.append(u[-1] - u[-2] if len(u) > 1 else 0.0)
            return np.reshape(np.array(out), logits.shape[:-1])
        part = np.partition(logits, -2, axis=0)   # partitioned over rows, not columns
        return part[-1] - part[-2]
    _patch(monkeypatch, "top2_gap", bad)
    _expect_failure(pins.test_top2_gap_matches_a_scan_and_a_sort)


def test_verify_off_by_one_is_caught(monkeypatch):
    def bad(drafts, targets):
        B = len(targets)
        a = 0
        while a < B - 1 and int(drafts[a]) == int(targets[a + 1]):
            a += 1
        return a + 1, int(targets[a])
    _patch(monkeypatch, "verify_block", bad)
    _expect_failure(pins.test_verify_bruteforce_tiny_vocab)


def test_verify_without_bonus_is_caught(monkeypatch):
    def bad(drafts, targets):
        B = len(targets)
        a = 0
        while a < B - 1 and int(drafts[a]) == int(targets[a]):
            a += 1
        return max(a, 1), int(targets[a])
    _patch(monkeypatch, "verify_block", bad)
    _expect_failure(pins.test_verify_bruteforce_tiny_vocab)


def test_mean_len_without_bonus_is_caught(monkeypatch):
    def bad(accepted, generated, drafts_per_cycle):
        cycles = generated / drafts_per_cycle
        return accepted / generated, accepted / cycles
    _patch(monkeypatch, "acceptance_stats", bad)
    _expect_failure(pins.test_worked_numbers_from_the_pages)


# ----------------------------------------------------------------------------
# Sampling oracle (oracle/sampling.py)
# ----------------------------------------------------------------------------

def test_sampling_residual_sign_error_is_caught(monkeypatch):
    """Resampling from max(0, q - p) instead of max(0, p - q)."""
    from oracle import sampling as osm
    from tests import test_sampling_pins as spins

    def bad(drafts, q, p, u_accept, u_resample):
        B = len(p)
        for j in range(B - 1):
            x = int(drafts[j])
            px, qx = osm.prob_of(*p[j], x), osm.prob_of(*q[j], x)
            if qx > 0 and u_accept[j] < min(1.0, px / qx):
                continue
            ids = q[j][0]
            r = np.array([max(0.0, qv - osm.prob_of(*p[j], int(y))) for y, qv in zip(ids, q[j][1])])
            return j + 1, osm.draw(ids, r, u_resample[j])
        return B, osm.draw(*p[B - 1], u_resample[B - 1])
    monkeypatch.setattr(osm, "verify_sample", bad)
    _expect_failure(lambda: spins.test_speculative_sampling_is_lossless(1))


def test_sampling_inverted_ratio_is_caught(monkeypatch):
    """Accepting with min(1, q/p) instead of min(1, p/q)."""
    from oracle import sampling as osm
    from tests import test_sampling_pins as spins

    def bad(drafts, q, p, u_accept, u_resample):
        B = len(p)
        for j in range(B - 1):
            x = int(drafts[j])
            px, qx = osm.prob_of(*p[j], x), osm.prob_of(*q[j], x)
            if px > 0 and u_accept[j] < min(1.0, qx / px):
                continue
            ids = p[j][0]
            r = np.array([max(0.0, pv - osm.prob_of(*q[j], int(y))) for y, pv in zip(ids, p[j][1])])
            if r.sum() == 0:
                r = np.asarray(p[j][1], dtype=float)
            return j + 1, osm.draw(ids, r, u_resample[j])
        return B, osm.draw(*p[B - 1], u_resample[B - 1])
    monkeypatch.setattr(osm, "verify_sample", bad)
    _expect_failure(lambda: spins.test_speculative_sampling_is_lossless(2))


def test_sampling_top_p_off_by_one_is_caught(monkeypatch):
    """Keeping the tokens strictly below top_p (dropping the one that reaches it)."""
    from oracle import sampling as osm
    from tests import test_sampling_pins as spins
    orig = osm.filtered_probs

    def bad(logits, temperature, top_k, top_p):
        ids, p = orig(logits, temperature, top_k, 1.0)
        c = np.cumsum(p)
        n = max(1, int(np.searchsorted(c, top_p, side="left")))
        return ids[:n], p[:n] / p[:n].sum()
    monkeypatch.setattr(osm, "filtered_probs", bad)
    _expect_failure(spins.test_top_p_worked_case)


# ----------------------------------------------------------------------------
# Path selector oracle (oracle/path_selector.py)
# ----------------------------------------------------------------------------

def _walk_variant(kind):
    from oracle import path_selector as ps

    def bad(anchor, cands, u, E, w_a, w_b, h_gates):
        prev = int(anchor)
        ids, gaps, picks = [], [], []
        for t in range(cands.shape[0]):
            if kind == "swap_maps":
                s = ps.pair_scores(u[t], cands[t], [prev], E, w_b, w_a, h_gates[t])[0]
            elif kind == "gate_shift":
                s = ps.pair_scores(u[t], cands[t], [prev], E, w_a, w_b, h_gates[max(t - 1, 0)])[0]
            else:
                s = ps.pair_scores(u[t], cands[t], [prev], E, w_a, w_b, h_gates[t])[0]
            j = int(np.argmax(s))
            ids.append(int(cands[t, j]))
            gaps.append(0.0)
            picks.append(j)
            if kind != "anchor_only":
                prev = int(cands[t, j])
        return np.array(ids), np.array(gaps), np.array(picks)
    return bad


@pytest.mark.parametrize("kind", ["anchor_only", "swap_maps", "gate_shift"])
def test_path_selector_walk_mistakes_are_caught(monkeypatch, kind):
    """The walk keeping the anchor as predecessor, A and B exchanged, or the
    gate taken from the previous position: a worked pin fails."""
    from oracle import path_selector as ps
    from tests import test_path_selector_pins as sp
    monkeypatch.setattr(ps, "greedy_walk", _walk_variant(kind))

    def both():
        sp.test_one_hot_walk_worked_by_hand()
        sp.test_asymmetric_maps_and_position_gates_worked_by_hand()
    _expect_failure(both)


def test_block_sched_counting_the_rejected_position_is_caught(monkeypatch):
    """Counting the rejected position as accepted (tau drafts accepted
    instead of tau - 1)."""
    from oracle import block_sched as obs
    from tests import test_block_sched_pins as bp

    def bad_observe(self, B, taus):
        for tau in taus:
            self.reached *= self.decay
            self.accepted *= self.decay
            a = min(int(tau), B - 1)
            for j in range(1, B):
                if j <= a:
                    self.reached[j - 1] += 1
                    self.accepted[j - 1] += 1
                elif j == a + 1:
                    self.reached[j - 1] += 1
                else:
                    break
    monkeypatch.setattr(obs.BlockScheduler, "observe", bad_observe)
    _expect_failure(bp.test_counts_after_worked_observations)


# ----------------------------------------------------------------------------
# Two-tap convolution oracle (oracle/two_tap_conv.py)
# ----------------------------------------------------------------------------

def _conv_variant(kind):
    def bad(x, c):
        nb = np.zeros_like(x)
        if kind == "successor":
            nb[:-1] = x[1:]
        else:
            nb[1:] = x[:-1]
        src = nb if kind == "coeff_from_prev" else x
        out = np.zeros_like(x)
        for i, xi in ((0, x), (1, nb)):
            k = c["base"][i][None, :]
            if kind != "no_correction":
                k = k + (src @ c["V"][i].T) @ c["U"][i].T
            out = out + k * xi
        return out
    return bad


@pytest.mark.parametrize("kind", ["successor", "coeff_from_prev", "no_correction"])
def test_two_tap_conv_mistakes_are_caught(monkeypatch, kind):
    from oracle import two_tap_conv as tc
    from tests import test_two_tap_conv_pins as cp
    monkeypatch.setattr(tc, "conv2", _conv_variant(kind))

    def pins():
        cp.test_shift_kernel_moves_rows_down()
        cp.test_tap0_only_kernel_is_pointwise()
        cp.test_correction_scales_with_U_and_is_absent_without_it()
    _expect_failure(pins)


def test_two_tap_conv_output_after_the_residual_is_caught(monkeypatch):
    """The output convolution applied to the residual stream after the add."""
    import oracle.dflash_oracle as od
    from oracle import two_tap_conv as tc
    from tests import test_two_tap_conv_pins as cp

    def bad_layer(x, layer, convs, k_ctx, v_ctx, pos0, shape):
        B = x.shape[0]
        nq, nkv, d = shape.n_heads, shape.n_kv_heads, shape.head_dim
        pos = pos0 + np.arange(B)
        h = tc.conv2(od.rms_norm(x, layer["g_attn"], shape.rms_eps), convs["ai"])
        q = od.apply_rope((h @ layer["w_q"].T).reshape(B, nq, d), pos, shape.rope_base)
        k = od.apply_rope((h @ layer["w_k"].T).reshape(B, nkv, d), pos, shape.rope_base)
        v = (h @ layer["w_v"].T).reshape(B, nkv, d)
        a = od.block_attention(q, np.concatenate([k_ctx, k]), np.concatenate([v_ctx, v])).reshape(B, nq * d)
        x = tc.conv2(x + a @ layer["w_o"].T, convs["ao"])
        h2 = tc.conv2(od.rms_norm(x, layer["g_ffn"], shape.rms_eps), convs["fi"])
        f = (od.silu(h2 @ layer["w_gate"].T) * (h2 @ layer["w_up"].T)) @ layer["w_down"].T
        return tc.conv2(x + f, convs["fo"])
    monkeypatch.setattr(tc, "decoder_layer_conv", bad_layer)
    _expect_failure(cp.test_zero_output_kernels_leave_the_embedding)


# ----------------------------------------------------------------------------
# 8-bit block KV format oracle (oracle/kv_quant.py)
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("kind", ["half_even", "exact_scale", "block16"])
def test_kv_quant_mistakes_are_caught(monkeypatch, kind):
    from oracle import kv_quant as kq
    from tests import test_kv_quant_pins as qp
    orig_q, orig_d = kq.quantize, kq.dequantize
    if kind == "half_even":
        monkeypatch.setattr(kq, "_round_half_away", np.round)
    elif kind == "exact_scale":
        def q2(x):
            q, sc = orig_q(x)
            blocks = np.asarray(x, dtype=np.float64).reshape(x.shape[:-1] + (x.shape[-1] // 32, 32))
            return q, np.abs(blocks).max(axis=-1) / 127      # the scale kept unrounded
        monkeypatch.setattr(kq, "quantize", q2)
    else:
        monkeypatch.setattr(kq, "BLOCK", 16)

    def pins():
        qp.test_exact_multiples_decode_exactly()
        qp.test_decode_error_bound()
        qp.test_zero_blocks_and_symmetry()
    _expect_failure(pins)


# ----------------------------------------------------------------------------
# target pass
# ----------------------------------------------------------------------------
from oracle import target_pass as otp
from tests import test_target_pass_pins as tpins


@pytest.mark.parametrize("kind", ["off_by_one", "non_causal"])
def test_target_causal_mask_mistakes_are_caught(monkeypatch, kind):
    orig = otp.causal_block_attention

    def bad(q, k, v, n_ctx):
        if kind == "non_causal":
            return od.block_attention(q, k, v)
        # each block position misses its own key (keeps at least one key)
        B = q.shape[0]
        out = np.empty_like(q)
        for j in range(B):
            lim = max(1, n_ctx + j)
            out[j:j + 1] = orig(q[j:j + 1], k[:lim], v[:lim], lim - 1)
        return out
    monkeypatch.setattr(otp, "causal_block_attention", bad)
    _expect_failure(tpins.test_causal_attention_matches_explicit_loops)
    _expect_failure(tpins.test_target_pass_matches_scalar_brute_force)


def test_target_feature_layers_zero_based_reading_is_caught(monkeypatch):
    orig = otp.feature_layers
    monkeypatch.setattr(otp, "feature_layers", lambda n, f: [l + 1 for l in orig(n, f)])
    _expect_failure(tpins.test_feature_layers_match_the_setup_table)


def test_target_caching_unrotated_keys_is_caught(monkeypatch):
    orig = otp.target_layer

    def bad(x, layer, k_ctx, v_ctx, pos0, shape):
        x2, k, v = orig(x, layer, k_ctx, v_ctx, pos0, shape)
        B = x.shape[0]
        h = od.rms_norm(x, layer["g_attn"], shape.rms_eps)
        k_raw = (h @ layer["w_k"].T).reshape(B, shape.n_kv_heads, shape.head_dim)
        return x2, k_raw, v
    monkeypatch.setattr(otp, "target_layer", bad)
    _expect_failure(tpins.test_block_pass_equals_one_token_passes)
    _expect_failure(tpins.test_target_pass_matches_scalar_brute_force)
