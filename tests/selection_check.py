"""Checks a block selection made by the CUDA path against the CPU oracle's.

Test infrastructure: used by the GPU tests, the smoke check and the parity
report of the benchmark's CPU-baseline leg.

The rule ("MiniMax-M3.1-Flash", 1. Model Introduction: each query keeps its
own block and the best of its earlier blocks, 16 in all; "[1/4] Add
MiniMax-M3 support - #4581", Kernel tuning, and "MiniMax-M3.1-Flash",
5.4 Notable quirks: two implementations' selections differ only at
near-ties):

* every selected row must be a valid selection: its own block, the
  min(16, own + 1) - 1 other ids distinct, ascending and earlier than the own
  block, the first min(n_init, own) blocks present when the init rule is on,
  and -1 in every unused slot;
* a row may differ from the oracle's only where the oracle marks it a
  near-tie (its last kept and first dropped scored blocks within 1e-3
  relative), and then only in blocks whose oracle score lies within 1e-3
  relative of the oracle's cut (the lowest score it kept).  Several results
  are correct on such rows, so the check is on what all of them share.
"""
from __future__ import annotations

from typing import Callable, Optional

import numpy as np

from oracle import msa_oracle as O


def invalid_rows(sel: np.ndarray, own: np.ndarray, n_init: int = 0) -> np.ndarray:
    """Boolean [n, H]: rows of sel [n, H, topk] that are not a valid selection
    for a query whose own block is own [n]."""
    sel = np.asarray(sel, dtype=np.int64)
    n, H, K = sel.shape
    own = np.asarray(own, dtype=np.int64)[:, None]                    # [n, 1]
    live = sel >= 0
    cnt = live.sum(-1)                                                 # [n, H]
    need = np.minimum(K, own + 1)                                      # [n, 1]
    bad = cnt != need
    j = np.arange(K)[None, None, :]
    bad |= np.any(live != (j < cnt[..., None]), axis=-1)               # -1 only after the ids
    step_ok = (np.diff(sel, axis=-1) > 0) | (j[..., :-1] >= cnt[..., None] - 1)
    bad |= ~np.all(step_ok, axis=-1)                                   # strictly ascending
    last = np.take_along_axis(sel, np.maximum(cnt - 1, 0)[..., None], axis=-1)[..., 0]
    bad |= last != own                                                 # ends with the own block
    bad |= sel[..., 0] < 0
    if n_init > 0:
        ni = np.minimum(n_init, own)                                   # [n, 1]
        init_ok = (j >= ni[..., None]) | (sel == j)
        bad |= ~np.all(init_ok, axis=-1)
    return bad


def tie_band_problem(grow, orow, scores, own: int, n_init: int = 0) -> Optional[str]:
    """Why the GPU row `grow` is not a near-tie variant of the oracle row `orow`
    given the oracle's block scores of that row, or None."""
    ni = min(n_init, own)
    g = {int(b) for b in grow if ni <= b < own}
    o = {int(b) for b in orow if ni <= b < own}
    if not o:
        return "the oracle keeps no scored block, yet the rows differ"
    cut = min(float(scores[b]) for b in o)
    for b in sorted(g ^ o):
        s = float(scores[b])
        if abs(s - cut) >= O.NEAR_TIE_REL * max(abs(s), abs(cut)):
            side = "dropped" if b in o else "added"
            return (f"block {b} {side} with oracle score {s!r}, outside the 1e-3 band "
                    f"around the cut {cut!r}")
    return None


def check_selection(gsel, osel, gap, own, scores_of: Callable[[int, int], np.ndarray],
                    what: str = "", n_init: int = 0) -> dict:
    """Compare gsel with osel (both [n, H, topk]); gap [n, H] is the oracle's
    near-tie gap, own [n] the own-block id of each compared row, and
    scores_of(r, h) returns the oracle's block scores of compared row r, index
    head h (called for differing rows only).  Raises AssertionError on any
    violation; returns the counts for the report."""
    gsel = np.asarray(gsel, dtype=np.int64)
    osel = np.asarray(osel, dtype=np.int64)
    gap = np.asarray(gap, dtype=np.float64)
    own = np.asarray(own, dtype=np.int64)
    bad = invalid_rows(gsel, own, n_init)
    assert not bad.any(), (f"{what}: {int(bad.sum())} invalid GPU selections, first at "
                           f"{np.argwhere(bad)[0].tolist()}: {gsel[tuple(np.argwhere(bad)[0])]}")
    diff = np.any(gsel != osel, axis=-1)
    near = gap < O.NEAR_TIE_REL
    outside = diff & ~near
    assert not outside.any(), (f"{what}: {int(outside.sum())} rows differ outside near-ties "
                               f"(first {np.argwhere(outside)[:3].tolist()})")
    for r, h in np.argwhere(diff):
        why = tie_band_problem(gsel[r, h], osel[r, h], scores_of(int(r), int(h)), int(own[r]),
                               n_init)
        assert why is None, f"{what}: row {int(r)} head {int(h)}: {why}"
    return {"rows": int(diff.size), "differing": int(diff.sum()), "near_tie": int(near.sum())}


def prefill_scores_of(qi: np.ndarray, ki: np.ndarray, cu: np.ndarray, tokens) -> Callable:
    """scores_of for prefill rows: compared row r is packed token tokens[r];
    qi, ki are the oracle's post-prologue index tensors [T, Hi, D]."""
    toks = np.asarray(tokens, dtype=np.int64)
    cu = np.asarray(cu, dtype=np.int64)

    def scores_of(r: int, h: int) -> np.ndarray:
        t = int(toks[r])
        s = int(np.searchsorted(cu, t, side="right") - 1)
        a, b = int(cu[s]), int(cu[s + 1])
        return O.block_scores_seq(np.asarray(qi[a:b, h], np.float64),
                                  np.asarray(ki[a:b, h], np.float64), np.array([t - a]))[0]

    return scores_of


def decode_scores_of(q_idx, kidx_cache, block_table, cache_lens) -> Callable:
    """scores_of for decode rows: compared row r is batch row r of q_idx
    [n, Hi, D] with its pages block_table[r] of kidx_cache [P, Hi, 128, D] and
    cache length cache_lens[r]; the new token sits at position L - 1."""
    q_idx = np.asarray(q_idx, dtype=np.float64)
    table = np.asarray(block_table, dtype=np.int64)
    lens = np.asarray(cache_lens, dtype=np.int64)

    def scores_of(r: int, h: int) -> np.ndarray:
        L = int(lens[r])
        npg = (L + O.BLOCK - 1) // O.BLOCK
        keys = np.asarray(kidx_cache[table[r, :npg], h], dtype=np.float64).reshape(-1, q_idx.shape[-1])
        qrows = np.zeros((L, q_idx.shape[-1]))
        qrows[L - 1] = q_idx[r, h]
        return O.block_scores_seq(qrows, keys[:L], np.array([L - 1]))[0]

    return scores_of
