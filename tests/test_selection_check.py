"""The selection checker used by the GPU tests catches what it must: invalid
rows of every kind, rows that differ away from a near-tie, and near-tie rows
that swap a block outside the tie band; and it accepts a swap inside it.
CPU only: the "GPU" selections here are edited copies of the oracle's."""
import numpy as np
import pytest

from oracle import msa_oracle as O
from tests import selection_check as SC


def _row(ids, k=16):
    r = np.full(k, -1, dtype=np.int64)
    r[:len(ids)] = ids
    return r


@pytest.mark.parametrize("ids,own,why", [
    (list(range(15)) + [20], 20, None),
    ([0, 1, 2], 2, None),
    (list(range(15)) + [19], 20, "own block missing"),
    (list(range(14)) + [20], 20, "one id short"),
    (list(range(14)) + [13, 20], 20, "duplicate"),
    ([1, 0] + list(range(2, 15)) + [20], 20, "not ascending"),
    (list(range(15)) + [21], 20, "future block"),
    ([0, 1], 2, "own block of a short row missing"),
    ([0, -1, 1, 2], 2, "hole before the ids"),
])
def test_invalid_rows(ids, own, why):
    sel = _row(ids)[None, None, :]
    bad = SC.invalid_rows(sel, np.array([own]))
    assert bool(bad[0, 0]) == (why is not None), why


def test_invalid_rows_init_rule():
    sel = np.stack([_row(list(range(15)) + [20]), _row([1] + list(range(2, 16)) + [20])])
    bad = SC.invalid_rows(sel[:, None, :], np.array([20, 20]), n_init=1)
    assert list(bad[:, 0]) == [False, True]          # the second drops init block 0


def _scored_row(scores_earlier, topk=4):
    own = len(scores_earlier)
    sc = np.concatenate([scores_earlier, [0.0]])
    sel, gap = O.select_from_scores(sc[None, :], np.array([own]), topk=topk)
    return sc, own, sel[:, None, :], gap[:, None]


def test_check_selection_accepts_a_swap_inside_the_band():
    sc, own, osel, gap = _scored_row(np.array([9.0, 7.0, 5.0, 4.9999, 1.0]))
    gsel = osel.copy()
    gsel[0, 0] = [0, 1, 3, 5]                         # 5.0 and 4.9999 swapped
    rep = SC.check_selection(gsel, osel, gap, np.array([own]), lambda r, h: sc, "swap")
    assert rep == {"rows": 1, "differing": 1, "near_tie": 1}


def test_check_selection_rejects_a_difference_away_from_a_near_tie():
    sc, own, osel, gap = _scored_row(np.array([9.0, 7.0, 5.0, 4.0, 1.0]))
    gsel = osel.copy()
    gsel[0, 0] = [0, 1, 3, 5]
    with pytest.raises(AssertionError, match="outside near-ties"):
        SC.check_selection(gsel, osel, gap, np.array([own]), lambda r, h: sc, "far")


def test_check_selection_rejects_a_swap_outside_the_band_on_a_near_tie_row():
    # a near-tie row (5.0 vs 4.9999) whose GPU row keeps block 4 (score 1.0) instead
    sc, own, osel, gap = _scored_row(np.array([9.0, 7.0, 5.0, 4.9999, 1.0]))
    gsel = osel.copy()
    gsel[0, 0] = [0, 1, 4, 5]
    with pytest.raises(AssertionError, match="outside the 1e-3 band"):
        SC.check_selection(gsel, osel, gap, np.array([own]), lambda r, h: sc, "band")


def test_check_selection_rejects_an_invalid_near_tie_row():
    sc, own, osel, gap = _scored_row(np.array([9.0, 7.0, 5.0, 4.9999, 1.0]))
    gsel = osel.copy()
    gsel[0, 0] = [0, 1, 3, -1]                        # own block dropped
    with pytest.raises(AssertionError, match="invalid GPU selections"):
        SC.check_selection(gsel, osel, gap, np.array([own]), lambda r, h: sc, "invalid")


def test_scores_of_helpers_match_the_oracle_scores():
    r = np.random.default_rng(3)
    cu = np.array([0, 300, 700])
    qi = r.standard_normal((700, 2, 16))
    ki = r.standard_normal((700, 2, 16))
    toks = [5, 299, 300, 699]
    f = SC.prefill_scores_of(qi, ki, cu, toks)
    for n, t in enumerate(toks):
        s = 0 if t < 300 else 1
        a, b = cu[s], cu[s + 1]
        want = O.block_scores_seq(qi[a:b, 1], ki[a:b, 1], np.array([t - a]))[0]
        np.testing.assert_array_equal(f(n, 1), want)
    # decode: the same keys laid out in pages, the query at the last position
    L = 300
    pages = np.array([2, 0, 1])
    cache = np.zeros((3, 2, 128, 16))
    keys = np.zeros((384, 2, 16))
    keys[:L] = ki[:L]
    for c, p in enumerate(pages):
        cache[p] = keys[c * 128:(c + 1) * 128].transpose(1, 0, 2)
    g = SC.decode_scores_of(qi[L - 1][None], cache, pages[None], np.array([L]))
    want = O.block_scores_seq(qi[:L, 1], ki[:L, 1], np.array([L - 1]))[0]
    np.testing.assert_array_equal(g(0, 1), want)
