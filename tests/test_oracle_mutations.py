"""The pins have teeth: plant a plausible mistake in the oracle (on the CPU, by
monkeypatching one function) and check that at least one pin then fails."""
import numpy as np
import pytest

from oracle import msa_oracle as O
from tests import test_oracle_pins as P


def _rope_adjacent_pairs(x, pos, rope_dim=64, base=1.0e7):
    x = np.asarray(x, dtype=np.float64)
    ang = np.asarray(pos, dtype=np.float64)[:, None] * O.rope_inv_freq(rope_dim, base)[None, :]
    shape = (x.shape[0],) + (1,) * (x.ndim - 2) + (rope_dim // 2,)
    c, s = np.cos(ang).reshape(shape), np.sin(ang).reshape(shape)
    y = x.copy()
    y[..., 0:rope_dim:2] = x[..., 0:rope_dim:2] * c - x[..., 1:rope_dim:2] * s
    y[..., 1:rope_dim:2] = x[..., 1:rope_dim:2] * c + x[..., 0:rope_dim:2] * s
    return y


def _norm_without_one(x, w, eps=1e-6):
    x = np.asarray(x, dtype=np.float64)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps) * w


def _norm_eps_outside(x, w, eps=1e-6):
    x = np.asarray(x, dtype=np.float64)
    return x / (np.sqrt(np.mean(x * x, axis=-1, keepdims=True)) + 1e-2) * (1 + w)


def _select_higher_id_on_tie(scores, own, topk=O.TOPK, n_init=0):
    s = scores.copy()
    n = s.shape[1]
    s = s + 1e-12 * np.arange(n)[None, :]      # breaks ties towards the higher id
    return _ORIG["select_from_scores"](s, own, topk, n_init)


def _select_init_rescored(scores, own, topk=O.TOPK, n_init=0):
    # keeps the init blocks but still lets them compete for the scored slots
    n = scores.shape[0]
    sel = np.full((n, topk), -1, dtype=np.int64)
    for r in range(n):
        o = int(own[r])
        ni = min(n_init, o)
        cand = np.arange(o)
        order = cand[np.lexsort((cand, -scores[r, :o]))] if o > 0 else cand
        ids = np.unique(np.concatenate([np.arange(ni), order[:topk - 1 - ni], [o]]))
        sel[r, :len(ids)] = ids
    return sel, np.full(n, np.inf)


def _select_streaming_insert_skips_ties(scores, own, topk=O.TOPK, n_init=0):
    # blocks taken in ascending order into a list kept by score, each new one
    # placed where it first beats an entry and the displaced entries carried on
    # with a strict comparison, so a displaced entry passes entries of equal
    # score (ties then stay in block order only while nothing larger arrives)
    n = scores.shape[0]
    sel = np.full((n, topk), -1, dtype=np.int64)
    for r in range(n):
        o = int(own[r])
        ni = min(n_init, o)
        slots = topk - 1 - ni
        best = [(-np.inf, -1)] * max(slots, 0)
        for b in range(ni, o):
            cv, ci = scores[r, b], b
            for i in range(len(best)):
                if cv > best[i][0]:
                    best[i], (cv, ci) = (cv, ci), best[i]
        keep = [b for _, b in best if b >= 0]
        ids = np.sort(np.concatenate([np.arange(ni), np.array(keep, dtype=np.int64), [o]]))
        sel[r, :len(ids)] = ids
    return sel, _ORIG["select_from_scores"](scores, own, topk, n_init)[1]


def _gap_variant(scores, own, topk, n_init, shift, denom):
    """select_from_scores with its near-tie gap taken between scored candidates
    `slots - 1 + shift` and `slots + shift`, relative to `denom` of the two."""
    sel, _ = _ORIG["select_from_scores"](scores, own, topk, n_init)
    gap = np.full(scores.shape[0], np.inf)
    for r in range(scores.shape[0]):
        o = int(own[r])
        ni = min(n_init, o)
        slots = topk - 1 - ni
        cand = np.arange(ni, o)
        order = cand[np.lexsort((cand, -scores[r, ni:o]))] if o > ni else cand
        i = slots - 1 + shift
        if slots > 0 and 0 <= i and i + 1 < len(order):
            a, b = scores[r, order[i]], scores[r, order[i + 1]]
            den = denom(abs(a), abs(b))
            gap[r] = abs(a - b) / den if den > 0 else 0.0
    return sel, gap


def _gap_one_past_the_cut(scores, own, topk=O.TOPK, n_init=0):
    # off by one toward the dropped side: first dropped vs second dropped
    return _gap_variant(scores, own, topk, n_init, 1, max)


def _gap_min_denominator(scores, own, topk=O.TOPK, n_init=0):
    # divides by the smaller magnitude of the two
    return _gap_variant(scores, own, topk, n_init, 0, min)


def _select_own_not_forced(scores, own, topk=O.TOPK, n_init=0):
    n = scores.shape[0]
    sel = np.full((n, topk), -1, dtype=np.int64)
    for r in range(n):
        cand = np.arange(int(own[r]) + 1)
        order = cand[np.argsort(-scores[r, :len(cand)], kind="stable")]
        ids = np.sort(order[:topk])
        sel[r, :len(ids)] = ids
    return sel, np.full(n, np.inf)


def _keys_one_past_causal(sel_row, p, block=O.BLOCK):
    # off by one: lets the key right after the query through (j <= p + 1)
    parts = [np.arange(b * block, min((b + 1) * block, p + 2)) for b in sel_row if b >= 0]
    return np.concatenate(parts)


def _keys_ignore_selection(sel_row, p, block=O.BLOCK):
    return np.arange(p + 1)


def _grads_without_delta(qt, do_t, kJ, vJ, scale):
    logits = scale * (qt @ kJ.T)
    e = np.exp(logits - logits.max(axis=1, keepdims=True))
    P_ = e / e.sum(axis=1, keepdims=True)
    return P_, P_ * (do_t @ vJ.T)


def _grads_transposed_dp(qt, do_t, kJ, vJ, scale):
    logits = scale * (qt @ kJ.T)
    e = np.exp(logits - logits.max(axis=1, keepdims=True))
    P_ = e / e.sum(axis=1, keepdims=True)
    o = P_ @ vJ
    dP = do_t @ kJ.T                        # wrong operand: K instead of V
    return P_, P_ * (dP - np.sum(do_t * o, axis=1, keepdims=True))


def _scores_no_causal(qi, ki, rows=None, block=O.BLOCK):
    L = qi.shape[0]
    nb = (L + block - 1) // block
    rows = np.arange(L) if rows is None else np.asarray(rows)
    s = qi[rows] @ ki.T
    out = np.stack([s[:, b * block:(b + 1) * block].max(axis=1) for b in range(nb)], axis=1)
    out[np.arange(nb)[None, :] > (rows // block)[:, None]] = -np.inf
    return out


def _bwd_rotate_forward(x, w, dy, cu_seqlens, eps=1e-6, rope_dim=64, base=1.0e7):
    # rotates the gradient by +angle instead of -angle
    dz = O.partial_rope(np.asarray(dy, np.float64), O.positions(cu_seqlens).astype(np.float64),
                        rope_dim, base)
    x = np.asarray(x, np.float64)
    r = 1.0 / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
    xh = x * r
    g = dz * (1.0 + np.asarray(w, np.float64))
    return r * (g - xh * np.mean(g * xh, axis=-1, keepdims=True)), np.sum(dz * xh, axis=(0, 1))


def _bwd_drop_norm_term(x, w, dy, cu_seqlens, eps=1e-6, rope_dim=64, base=1.0e7):
    # forgets that the rms depends on x
    dz = O.partial_rope(np.asarray(dy, np.float64), -O.positions(cu_seqlens).astype(np.float64),
                        rope_dim, base)
    x = np.asarray(x, np.float64)
    r = 1.0 / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
    return r * dz * (1.0 + np.asarray(w, np.float64)), np.sum(dz * x * r, axis=(0, 1))


def _bwd_dw_scaled(x, w, dy, cu_seqlens, eps=1e-6, rope_dim=64, base=1.0e7):
    # weight gradient taken through the (1 + w) factor a second time
    dx, dw = _ORIG["qk_norm_rope_bwd"](x, w, dy, cu_seqlens, eps, rope_dim, base)
    return dx, dw * (1.0 + np.asarray(w, np.float64))


def _append_at_length(q, k, v, q_idx, k_idx, w_q, w_k, w_qi, w_ki, k_cache, v_cache,
                      kidx_cache, block_table, cache_lens, eps=1e-6, rope_dim=64, base=1.0e7):
    # the new token placed at position L instead of L - 1
    return _ORIG["decode_append"](q, k, v, q_idx, k_idx, w_q, w_k, w_qi, w_ki, k_cache, v_cache,
                                  kidx_cache, block_table, np.asarray(cache_lens) + 1, eps,
                                  rope_dim, base)


_ORIG = {"select_from_scores": O.select_from_scores, "qk_norm_rope_bwd": O.qk_norm_rope_bwd,
         "decode_append": O.decode_append}

MUTATIONS = [
    ("partial_rope", _rope_adjacent_pairs, [P.test_rope_matches_complex_rotation]),
    ("gemma_rmsnorm", _norm_without_one, [P.test_gemma_rmsnorm_matches_torch_rms_norm]),
    ("gemma_rmsnorm", _norm_eps_outside, [P.test_gemma_rmsnorm_zero_weight_gives_unit_rms]),
    ("select_from_scores", _select_higher_id_on_tie, [P.test_selection_tie_prefers_lower_block]),
    ("select_from_scores", _select_streaming_insert_skips_ties,
     [P.test_selection_with_exact_ties_then_larger_scores]),
    ("select_from_scores", _select_own_not_forced, [P.test_selection_invariants]),
    ("select_from_scores", _select_init_rescored, [P.test_init_rule_by_enumeration]),
    ("select_from_scores", _gap_one_past_the_cut, [P.test_near_tie_gap_exact_values]),
    ("select_from_scores", _gap_min_denominator, [P.test_near_tie_gap_exact_values]),
    ("_keys_of", _keys_one_past_causal,
     [P.test_sparse_forward_and_backward_match_masked_library_attention]),
    ("_keys_of", _keys_ignore_selection,
     [P.test_sparse_forward_and_backward_match_masked_library_attention]),
    ("_row_grads", _grads_without_delta, [P.test_backward_finite_differences]),
    ("_row_grads", _grads_transposed_dp, [P.test_backward_finite_differences]),
    ("block_scores_seq", _scores_no_causal, [P.test_block_scores_brute_force]),
    ("qk_norm_rope_bwd", _bwd_rotate_forward, [P.test_prologue_backward_finite_differences]),
    ("qk_norm_rope_bwd", _bwd_drop_norm_term, [P.test_prologue_backward_scale_invariance]),
    ("qk_norm_rope_bwd", _bwd_dw_scaled, [P.test_prologue_backward_matches_autograd]),
    ("decode_append", _append_at_length, [P.test_decode_append_matches_prefill_prologue]),
]


@pytest.mark.parametrize("name,fn,pins", MUTATIONS,
                         ids=[f"{m[0]}-{m[1].__name__}" for m in MUTATIONS])
def test_planted_mistake_is_caught(monkeypatch, name, fn, pins):
    monkeypatch.setattr(O, name, fn)
    caught = False
    for pin in pins:
        try:
            pin()
        except (AssertionError, ValueError, IndexError):
            caught = True
    assert caught, f"no pin caught the planted mistake in {name}"
