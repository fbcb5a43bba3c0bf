"""Pins for the CPU oracle: library routines, closed forms, invariants, brute force
on tiny inputs and the facts the pages state.  None of these calls the CUDA path."""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import msa_oracle as O

HERE = os.path.dirname(os.path.abspath(__file__))
FACTS = json.load(open(os.path.join(HERE, "golden", "msa_page_facts.json")))


def rng(seed=0):
    return np.random.default_rng(seed)


# ------------------------------------------------------------------ bf16 rounding

def test_bf16_round_matches_torch_on_float32_values():
    r = rng(1)
    x = np.concatenate([
        r.standard_normal(20000) * 10.0 ** r.integers(-40, 38, 20000),
        r.standard_normal(2000) * 1e-39,                 # bf16 subnormals
        np.array([0.0, -0.0, 1.0, -2.5, 3.0e38, -3.3e38]),
    ]).astype(np.float32)
    # exact halfway points between neighbouring bf16 values
    base = torch.randn(4000, dtype=torch.float32).to(torch.bfloat16).float().numpy()
    half = (base.view(np.uint32) | np.uint32(0x8000)).view(np.float32)
    x = np.concatenate([x, half])
    want = torch.from_numpy(x).to(torch.bfloat16).double().numpy()
    got = O.bf16_round(x.astype(np.float64))
    np.testing.assert_array_equal(got, want)


def test_bf16_round_from_float64_is_single_rounding():
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7: ties go to the even value 1.
    assert O.bf16_round(1.0 + 2.0 ** -8) == 1.0
    # slightly above halfway (not representable in float32) must round up.
    assert O.bf16_round(1.0 + 2.0 ** -8 + 2.0 ** -40) == 1.0 + 2.0 ** -7
    # 1 + 3*2^-8 is halfway between 1+2^-7 and 1+2^-6: even is 1+2^-6.
    assert O.bf16_round(1.0 + 3 * 2.0 ** -8) == 1.0 + 2.0 ** -6
    assert O.bf16_round(2.0 ** -133) == 2.0 ** -133
    assert O.bf16_round(0.49 * 2.0 ** -133) == 0.0
    assert np.isinf(O.bf16_round(3.4e38))


# ------------------------------------------------------------------ prologue

def test_gemma_rmsnorm_matches_torch_rms_norm():
    r = rng(2)
    x = r.standard_normal((7, 3, 128)) * 3.0
    w = r.standard_normal(128) * 0.1
    want = F.rms_norm(torch.from_numpy(x), (128,), weight=torch.from_numpy(1.0 + w),
                      eps=1e-6).numpy()
    np.testing.assert_allclose(O.gemma_rmsnorm(x, w, 1e-6), want, rtol=1e-12, atol=1e-12)


def test_gemma_rmsnorm_zero_weight_gives_unit_rms():
    x = rng(3).standard_normal((50, 128)) * 7.0
    y = O.gemma_rmsnorm(x, np.zeros(128), eps=0.0)
    np.testing.assert_allclose(np.sqrt(np.mean(y * y, axis=-1)), 1.0, rtol=1e-12)


def test_rope_matches_complex_rotation():
    # channel i and i+32 form the complex number x_i + i*x_{i+32}; RoPE multiplies
    # it by exp(i * p * base^(-2i/64)); channels 64..127 pass through.
    r = rng(4)
    T, H = 9, 2
    x = r.standard_normal((T, H, 128))
    pos = r.integers(0, 40000, T)
    base = FACTS["rope_base"]["value"]
    y = O.partial_rope(x, pos, 64, base)
    theta = base ** (-np.arange(32) * 2.0 / 64.0)
    z = (x[..., :32] + 1j * x[..., 32:64]) * np.exp(1j * pos[:, None, None] * theta)
    np.testing.assert_allclose(y[..., :32], z.real, rtol=1e-9, atol=1e-9)
    np.testing.assert_allclose(y[..., 32:64], z.imag, rtol=1e-9, atol=1e-9)
    np.testing.assert_array_equal(y[..., 64:], x[..., 64:])


def test_rope_closed_form_values():
    x = np.zeros((2, 1, 128))
    x[:, 0, 0] = 1.0     # pair (0, 32) has frequency 1
    x[:, 0, 31] = 1.0    # pair (31, 63) has frequency base^(-62/64)
    y = O.partial_rope(x, np.array([0, 1]), 64, 1e7)
    np.testing.assert_allclose(y[0, 0], x[0, 0], atol=0)          # p = 0 is the identity
    assert y[1, 0, 0] == pytest.approx(math.cos(1.0), abs=1e-15)
    assert y[1, 0, 32] == pytest.approx(math.sin(1.0), abs=1e-15)
    f = 1e7 ** (-62.0 / 64.0)
    assert y[1, 0, 31] == pytest.approx(math.cos(f), abs=1e-15)
    assert y[1, 0, 63] == pytest.approx(math.sin(f), abs=1e-15)


def test_rope_relative_position_and_norm():
    r = rng(5)
    q = r.standard_normal((1, 1, 128))
    k = r.standard_normal((1, 1, 128))
    def dot(p1, p2):
        a = O.partial_rope(q, np.array([p1]), 64, 1e7)
        b = O.partial_rope(k, np.array([p2]), 64, 1e7)
        return float(np.sum(a * b))
    assert dot(100, 37) == pytest.approx(dot(1100, 1037), rel=1e-9)
    assert dot(5, 5) == pytest.approx(float(np.sum(q * k)), rel=1e-9)
    y = O.partial_rope(q, np.array([12345]), 64, 1e7)
    assert np.linalg.norm(y[..., :64]) == pytest.approx(np.linalg.norm(q[..., :64]), rel=1e-12)


def test_positions_restart_per_sequence():
    np.testing.assert_array_equal(O.positions([0, 3, 5, 5, 9]),
                                  [0, 1, 2, 0, 1, 0, 1, 2, 3])


def test_prologue_is_norm_then_rope_then_bf16():
    r = rng(6)
    cu = [0, 130, 300]
    x = r.standard_normal((300, 2, 128))
    w = r.standard_normal(128) * 0.1
    y = O.qk_norm_rope(x, w, cu)
    xt = torch.from_numpy(x)
    n = F.rms_norm(xt, (128,), weight=torch.from_numpy(1.0 + w), eps=1e-6).numpy()
    pos = np.concatenate([np.arange(130), np.arange(170)])
    ref = O.partial_rope(n, pos, 64, 1e7)
    np.testing.assert_array_equal(y, O.bf16_round(ref))
    assert np.all(O.bf16_round(y) == y)


def _prologue_case(seed, T=9, H=2, D=128, cu=(0, 4, 9)):
    r = rng(seed)
    x = r.standard_normal((T, H, D)) * 1.5
    w = r.standard_normal(D) * 0.3
    dy = r.standard_normal((T, H, D))
    return x, w, dy, np.array(cu)


def test_prologue_backward_finite_differences():
    """Central differences of L = sum(dy * y(x, w)) against the closed form, for
    rotated and pass-through channels, at several positions."""
    x, w, dy, cu = _prologue_case(21)
    loss = lambda x_, w_: float(np.sum(dy * O.qk_norm_rope(x_, w_, cu, round_bf16=False)))
    dx, dw = O.qk_norm_rope_bwd(x, w, dy, cu)
    h = 1e-6
    for idx in [(0, 0, 3), (2, 1, 40), (3, 0, 70), (5, 1, 10), (8, 0, 127), (7, 1, 33)]:
        xp = x.copy(); xp[idx] += h
        xm = x.copy(); xm[idx] -= h
        fd = (loss(xp, w) - loss(xm, w)) / (2 * h)
        assert fd == pytest.approx(dx[idx], rel=1e-6, abs=1e-8), idx
    for c in [0, 31, 32, 63, 64, 100]:
        wp = w.copy(); wp[c] += h
        wm = w.copy(); wm[c] -= h
        fd = (loss(x, wp) - loss(x, wm)) / (2 * h)
        assert fd == pytest.approx(dw[c], rel=1e-6, abs=1e-8), c


def test_prologue_backward_matches_autograd():
    """fp64 torch autograd through an independent statement of the forward."""
    x, w, dy, cu = _prologue_case(22, T=13, H=3, cu=(0, 5, 6, 13))
    pos = torch.tensor(O.positions(cu), dtype=torch.float64)
    xt = torch.tensor(x, requires_grad=True)
    wt = torch.tensor(w, requires_grad=True)
    z = xt * torch.rsqrt((xt * xt).mean(-1, keepdim=True) + 1e-6) * (1 + wt)
    inv = 1e7 ** (-torch.arange(0, 64, 2, dtype=torch.float64) / 64)
    ang = pos[:, None, None] * inv[None, None, :]
    z1, z2, rest = z[..., :32], z[..., 32:64], z[..., 64:]
    y = torch.cat([z1 * torch.cos(ang) - z2 * torch.sin(ang),
                   z2 * torch.cos(ang) + z1 * torch.sin(ang), rest], dim=-1)
    (y * torch.tensor(dy)).sum().backward()
    dx, dw = O.qk_norm_rope_bwd(x, w, dy, cu)
    np.testing.assert_allclose(dx, xt.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dw, wt.grad.numpy(), rtol=1e-10, atol=1e-12)


def test_prologue_backward_reduces_to_plain_rmsnorm():
    """w = 0 and every token at position 0 (one-token sequences): the textbook
    RMSNorm gradient dx = (dy - y mean(dy y)) / rms, and dw = sum dy * y."""
    T = 5
    x, _, dy, _ = _prologue_case(23, T=T)
    cu = np.arange(T + 1)
    w = np.zeros(x.shape[-1])
    rms = np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + 1e-6)
    y = x / rms
    want = (dy - y * np.mean(dy * y, axis=-1, keepdims=True)) / rms
    dx, dw = O.qk_norm_rope_bwd(x, w, dy, cu)
    np.testing.assert_allclose(dx, want, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(dw, np.sum(dy * y, axis=(0, 1)), rtol=1e-12, atol=1e-12)


def test_prologue_backward_scale_invariance():
    """With eps -> 0 the norm output does not depend on the scale of x, so the
    gradient is orthogonal to x and scales as 1/c."""
    x, w, dy, cu = _prologue_case(24)
    dx, _ = O.qk_norm_rope_bwd(x, w, dy, cu, eps=0.0)
    assert np.max(np.abs(np.sum(dx * x, axis=-1))) < 1e-10
    dx3, _ = O.qk_norm_rope_bwd(3.0 * x, w, dy, cu, eps=0.0)
    np.testing.assert_allclose(dx3, dx / 3.0, rtol=1e-10, atol=1e-14)


# ------------------------------------------------------------------ indexer

def test_decode_append_matches_prefill_prologue():
    """The appended token's stored k / index-k and its q / index-q equal the
    prefill prologue of the same token at the same position of its sequence;
    v is stored verbatim; nothing else in the caches changes."""
    r = rng(31)
    lens = np.array([1, 130, 257, 128])
    B, H, D = len(lens), 2, 128
    pages = [(L + 127) // 128 for L in lens]
    P = sum(pages) + 3
    perm = r.permutation(P)
    table = np.full((B, max(pages)), -1)
    at = 0
    for b in range(B):
        table[b, :pages[b]] = perm[at:at + pages[b]]
        at += pages[b]
    kc, vc, ic = (O.bf16_round(r.standard_normal((P, H, 128, D))) for _ in range(3))
    q, k, v, qi, ki = (r.standard_normal((B, H, D)) for _ in range(5))
    v = O.bf16_round(v)
    w_q, w_k, w_qi, w_ki = (r.standard_normal(D) * 0.2 for _ in range(4))
    q_out, qi_out, kc2, vc2, ic2 = O.decode_append(q, k, v, qi, ki, w_q, w_k, w_qi, w_ki,
                                                   kc, vc, ic, table, lens)
    touched = np.zeros((P, 128), dtype=bool)
    for b in range(B):
        # the same token placed at position L-1 of a packed sequence of length L
        L = int(lens[b])
        cu = np.array([0, L])
        pack = lambda x: np.concatenate([r.standard_normal((L - 1, H, D)), x[b][None]], axis=0)
        for got, x, w in ((q_out[b], q, w_q), (qi_out[b], qi, w_qi)):
            np.testing.assert_array_equal(got, O.qk_norm_rope(pack(x), w, cu)[-1])
        page, slot = int(table[b, (L - 1) // 128]), (L - 1) % 128
        np.testing.assert_array_equal(kc2[page, :, slot], O.qk_norm_rope(pack(k), w_k, cu)[-1])
        np.testing.assert_array_equal(ic2[page, :, slot], O.qk_norm_rope(pack(ki), w_ki, cu)[-1])
        np.testing.assert_array_equal(vc2[page, :, slot], v[b])
        touched[page, slot] = True
    keep = np.broadcast_to(~touched[:, None, :, None], kc.shape)
    for old, new in ((kc, kc2), (vc, vc2), (ic, ic2)):
        np.testing.assert_array_equal(old[keep], new[keep])


def _brute_scores(qi, ki, block):
    L = qi.shape[0]
    nb = (L + block - 1) // block
    out = np.full((L, nb), -np.inf)
    for t in range(L):
        for b in range(nb):
            for j in range(b * block, min((b + 1) * block, t + 1)):
                out[t, b] = max(out[t, b], float(np.dot(qi[t], ki[j])))
    return out


def test_block_scores_brute_force():
    r = rng(7)
    qi = r.standard_normal((23, 8))
    ki = r.standard_normal((23, 8))
    np.testing.assert_array_equal(O.block_scores_seq(qi, ki, block=4), _brute_scores(qi, ki, 4))


def test_selection_is_best_subset_by_enumeration():
    # the top-(k-1) earlier blocks are the subset of that size with the largest
    # total score; check against enumeration of all subsets on tiny inputs.
    r = rng(8)
    block, topk = 4, 3
    for trial in range(20):
        L = int(r.integers(1, 40))
        qi = r.standard_normal((L, 6))
        ki = r.standard_normal((L, 6))
        sc = _brute_scores(qi, ki, block)
        own = np.arange(L) // block
        sel, _ = O.select_from_scores(sc, own, topk)
        for t in range(L):
            o = own[t]
            m = min(topk - 1, o)
            best = max(itertools.combinations(range(o), m), key=lambda c: sum(sc[t, list(c)]))
            want = sorted(list(best) + [o]) + [-1] * (topk - 1 - m)
            assert list(sel[t]) == want


def test_init_rule_by_enumeration():
    """With the init rule ("#4581", Kernel tuning names it; read here as: the first
    n_init blocks of the sequence are always kept) the scored slots hold the best
    subset of the blocks between the init blocks and the own block."""
    r = rng(31)
    block, topk = 4, 4
    for n_init in (1, 2, 3):
        for trial in range(12):
            L = int(r.integers(1, 48))
            qi = r.standard_normal((L, 6))
            ki = r.standard_normal((L, 6))
            sc = _brute_scores(qi, ki, block)
            own = np.arange(L) // block
            sel, _ = O.select_from_scores(sc, own, topk, n_init=n_init)
            for t in range(L):
                o = int(own[t])
                ni = min(n_init, o)
                m = min(topk - 1 - ni, o - ni)
                best = max(itertools.combinations(range(ni, o), m),
                           key=lambda c: sum(sc[t, list(c)]))
                want = sorted(list(range(ni)) + list(best) + [o])
                want += [-1] * (topk - len(want))
                assert list(sel[t]) == want, (n_init, t)


def test_init_rule_is_infinite_score_for_the_first_blocks():
    """Keeping the first n_init blocks equals the plain rule on scores where those
    blocks score +inf (they then win every comparison), on a real index pack."""
    qi, ki, cu = _small_pack(33, [700, 1, 2600], hi=2)
    for n_init in (1, 2):
        sel, _ = O.index_select(qi, ki, cu, n_init=n_init)
        pos = O.positions(cu)
        for s in range(len(cu) - 1):
            a, b = cu[s], cu[s + 1]
            for h in range(2):
                sc = O.block_scores_seq(qi[a:b, h], ki[a:b, h])
                sc[:, :n_init] = np.inf
                want, _ = O.select_from_scores(sc, pos[a:b] // 128)
                np.testing.assert_array_equal(sel[a:b, h], want)
    sel0, _ = O.index_select(qi, ki, cu, n_init=0)
    np.testing.assert_array_equal(sel0, O.index_select(qi, ki, cu)[0])


def test_selection_tie_prefers_lower_block():
    sc = np.array([[5.0, 7.0, 5.0, 5.0, 1.0, 0.0]])
    sel, gap = O.select_from_scores(sc, np.array([5]), topk=3)
    assert list(sel[0]) == [0, 1, 5]
    assert gap[0] == 0.0


def test_selection_with_exact_ties_then_larger_scores():
    """Key blocks 0 .. 9 copies of one block B, later ones copies of 2B: every
    earlier block scores exactly m or 2m (m > 0 for these queries), so the
    rule alone gives each row's selection: the lowest 2B blocks first, then
    the lowest B blocks in the places left, then the own block."""
    g = rng(9)
    L = 20 * 128
    blk = g.standard_normal((128, 1, 128))
    ki = np.concatenate([blk * (2.0 if b >= 10 else 1.0) for b in range(20)], axis=0)
    qi = g.standard_normal((L, 1, 128))
    assert np.all((qi[:, 0] @ blk[:, 0].T).max(axis=1) > 0)
    sel, gap = O.index_select(qi, ki, np.array([0, L]))
    for t in range(L):
        o = t // 128
        hi = list(range(10, o))[:15]
        lo = list(range(min(o, 10)))[:15 - len(hi)]
        want = sorted(hi + lo + [o])
        assert list(sel[t, 0, :len(want)]) == want and np.all(sel[t, 0, len(want):] == -1), t
        # with more than 15 earlier blocks the cut falls between two equal
        # scores (gap 0) except at o = 25, where it falls between the last of
        # the fifteen 2m blocks and block 0 (gap (2m - m) / 2m = 1/2)
        if o > 15:
            assert gap[t, 0] == (0.5 if o == 25 else 0.0), t


def test_near_tie_gap_exact_values():
    """The near-tie gap compares the last kept scored block with the first
    dropped one, relative to the larger magnitude of the two (the parity rule:
    rows whose cut straddles scores within 1e-3 relative are near-ties;
    "[1/4] Add MiniMax-M3 support - #4581", Kernel tuning, and
    "MiniMax-M3.1-Flash", 5.4 Notable quirks: selections differ only at
    near-ties).  Hand-chosen distinct scores, values worked out by hand:

      top-4 (own + 3 scored), earlier scores 9, 7, 5, 4.99, 1 (own block 5):
        kept 9, 7, 5; first dropped 4.99; gap = 0.01 / 5
      same with negative scores -1, -2, -3, -3.001, -10:
        kept -1, -2, -3; first dropped -3.001; gap = 0.001 / 3.001
      the scored order need not follow block ids: 4.99 at block 0, 9 at block 4
      top-16 on 20 earlier blocks with scores 20 - b (b = 0..19), block 14 at
      5.5 and block 15 at 5.4945: kept blocks 0..13 and 14; first dropped 15;
      gap = 0.0055 / 5.5 = 1e-3 exactly at the boundary (not a near-tie)."""
    own = np.array([5])
    sel, gap = O.select_from_scores(np.array([[9.0, 7.0, 5.0, 4.99, 1.0, 0.0]]), own, topk=4)
    assert list(sel[0]) == [0, 1, 2, 5]
    assert gap[0] == pytest.approx(0.01 / 5.0, rel=1e-9)

    sel, gap = O.select_from_scores(np.array([[-1.0, -2.0, -3.0, -3.001, -10.0, 0.0]]), own,
                                    topk=4)
    assert list(sel[0]) == [0, 1, 2, 5]
    assert gap[0] == pytest.approx(0.001 / 3.001, rel=1e-9)

    sel, gap = O.select_from_scores(np.array([[4.99, 7.0, 1.0, 5.0, 9.0, 0.0]]), own, topk=4)
    assert list(sel[0]) == [1, 3, 4, 5]
    assert gap[0] == pytest.approx(0.01 / 5.0, rel=1e-9)

    sc = np.concatenate([20.0 - np.arange(20), [0.0]])
    sc[14], sc[15] = 5.5, 5.4945
    sel, gap = O.select_from_scores(sc[None, :], np.array([20]), topk=16)
    assert list(sel[0]) == list(range(15)) + [20]
    assert gap[0] == pytest.approx(0.0055 / 5.5, rel=1e-9)
    assert not (gap[0] < O.NEAR_TIE_REL * (1 - 1e-9))


def test_near_tie_gap_through_index_select():
    """The gap that index_select reports for a row is the one its block scores
    give: one sequence of 6 blocks of 4 keys (block 4, top-4), index keys built
    so that every block's maximum logit is a chosen value (one key per block
    along the query direction, the others orthogonal and smaller)."""
    D, blk = 8, 4
    q = np.zeros(D)
    q[0] = 1.0
    want = [9.0, 5.0, 7.0, 4.999, 1.0]                 # earlier blocks 0..4
    keys = np.zeros((24, D))
    for b, s in enumerate(want + [0.5]):
        keys[b * blk, 0] = s                           # logit s
        keys[b * blk + 1:(b + 1) * blk, 1] = 3.0       # logit 0, never the max here
    qi = np.zeros((24, 1, D))
    qi[:, 0] = q
    ki = keys[:, None, :]
    sel, gap = O.index_select(qi, ki, np.array([0, 24]), topk=4, block=blk)
    assert list(sel[23, 0]) == [0, 1, 2, 5]
    assert gap[23, 0] == pytest.approx((5.0 - 4.999) / 5.0, rel=1e-9)
    assert gap[23, 0] < O.NEAR_TIE_REL


def _small_pack(seed, seqlens, hi=2, d=32):
    r = rng(seed)
    T = sum(seqlens)
    cu = np.concatenate([[0], np.cumsum(seqlens)])
    return r.standard_normal((T, hi, d)), r.standard_normal((T, hi, d)), cu


def test_selection_invariants():
    qi, ki, cu = _small_pack(9, [2500, 100, 3000, 1])
    sel, gap = O.index_select(qi, ki, cu)
    pos = O.positions(cu)
    for t in range(len(pos)):
        own = pos[t] // 128
        for h in range(qi.shape[1]):
            ids = sel[t, h][sel[t, h] >= 0]
            assert own in ids
            assert ids.max() == own
            assert len(ids) == min(16, own + 1) == len(set(ids))
            assert np.all(np.diff(ids) > 0)
            assert np.all(sel[t, h][len(ids):] == -1)
    # the result does not depend on the logit scale
    sel2, _ = O.index_select(qi * 0.37, ki, cu)
    np.testing.assert_array_equal(sel, sel2)


def test_selection_keeps_every_block_up_to_2048_tokens():
    n = FACTS["dense_equivalent_tokens"]["value"]
    assert n == FACTS["topk_blocks"]["value"] * FACTS["block"]["value"]
    qi, ki, cu = _small_pack(10, [n + 1], hi=1)
    sel, gap = O.index_select(qi, ki, cu)
    for t in range(n):
        assert list(sel[t, 0]) == list(range(t // 128 + 1)) + [-1] * (15 - t // 128)
        assert gap[t, 0] == np.inf
    # token 2048 (17 causal blocks) is the first that drops one
    assert len(set(sel[n, 0])) == 16 and np.isfinite(gap[n, 0])


# ------------------------------------------------------------------ attention

def _sdpa_masked(q, k, v, mask, scale):
    """Library attention (fp64, torch CPU) with a boolean allow-mask per head."""
    qt = torch.from_numpy(q).requires_grad_(True)
    kt = torch.from_numpy(k).requires_grad_(True)
    vt = torch.from_numpy(v).requires_grad_(True)
    out = F.scaled_dot_product_attention(qt, kt, vt, attn_mask=torch.from_numpy(mask), scale=scale)
    return qt, kt, vt, out


def _allow_mask(sel_g, cu, block):
    """allow[t, j]: j is in t's sequence, in one of t's selected blocks, and j <= t."""
    T = sel_g.shape[0]
    pos = O.positions(cu)
    seq = np.searchsorted(cu, np.arange(T), side="right") - 1
    allow = np.zeros((T, T), dtype=bool)
    for t in range(T):
        for j in range(T):
            if seq[j] == seq[t] and pos[j] <= pos[t] and (pos[j] // block) in set(sel_g[t]):
                allow[t, j] = True
    return allow


def _gqa_reference(q, k, v, do, sel, cu, scale, block):
    """Dense library attention per KV group with the selection as a mask; returns
    o, lse, dq, dk, dv from torch autograd in fp64."""
    T, Hq, D = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    o = np.zeros_like(q); lse = np.zeros((T, Hq))
    dq = np.zeros_like(q); dk = np.zeros_like(k); dv = np.zeros_like(v)
    for g in range(Hkv):
        mask = _allow_mask(sel[:, g], cu, block)
        qg = np.ascontiguousarray(q[:, g * G:(g + 1) * G].transpose(1, 0, 2))
        kg = np.repeat(k[None, :, g], G, axis=0)
        vg = np.repeat(v[None, :, g], G, axis=0)
        qt, kt, vt, out = _sdpa_masked(qg, kg, vg, mask[None], scale)
        out.backward(torch.from_numpy(np.ascontiguousarray(do[:, g * G:(g + 1) * G].transpose(1, 0, 2))))
        o[:, g * G:(g + 1) * G] = out.detach().numpy().transpose(1, 0, 2)
        logits = torch.from_numpy(qg) @ torch.from_numpy(kg).transpose(1, 2) * scale
        logits = logits.masked_fill(~torch.from_numpy(mask)[None], float("-inf"))
        lse[:, g * G:(g + 1) * G] = torch.logsumexp(logits, dim=-1).numpy().T
        dq[:, g * G:(g + 1) * G] = qt.grad.numpy().transpose(1, 0, 2)
        dk[:, g] = kt.grad.numpy().sum(0)
        dv[:, g] = vt.grad.numpy().sum(0)
    return o, lse, dq, dk, dv


def test_dense_equivalence_up_to_2048_tokens():
    """Every causal block is selected for sequences of <= 2048 tokens, so the
    block-sparse forward equals plain causal attention (Megatron-Bridge MiniMax-M3
    page, Known Limitations)."""
    r = rng(11)
    seqlens = [300, 700, 2048]
    cu = np.concatenate([[0], np.cumsum(seqlens)])
    T, Hq, Hkv, D = sum(seqlens), 4, 2, 16
    q, k, v = (r.standard_normal((T, h, D)) for h in (Hq, Hkv, Hkv))
    qi, ki = r.standard_normal((T, Hkv, D)), r.standard_normal((T, Hkv, D))
    sel, _ = O.index_select(qi, ki, cu)
    scale = 1 / math.sqrt(D)
    o, lse = O.sparse_attn_fwd(q, k, v, sel, cu, scale)
    G = Hq // Hkv
    for s in range(len(seqlens)):
        a, b = cu[s], cu[s + 1]
        qq = torch.from_numpy(q[a:b].transpose(1, 0, 2).copy())
        kk = torch.from_numpy(np.repeat(k[a:b], G, axis=1).transpose(1, 0, 2).copy())
        vv = torch.from_numpy(np.repeat(v[a:b], G, axis=1).transpose(1, 0, 2).copy())
        want = F.scaled_dot_product_attention(qq, kk, vv, is_causal=True, scale=scale)
        np.testing.assert_allclose(o[a:b], want.numpy().transpose(1, 0, 2), rtol=1e-10, atol=1e-12)


def test_sparse_forward_and_backward_match_masked_library_attention():
    block, topk = 4, 3
    r = rng(12)
    seqlens = [13, 30, 1, 21]
    cu = np.concatenate([[0], np.cumsum(seqlens)])
    T, Hq, Hkv, D = sum(seqlens), 6, 2, 8
    q, k, v, do = (r.standard_normal((T, h, D)) for h in (Hq, Hkv, Hkv, Hq))
    qi, ki = r.standard_normal((T, Hkv, D)), r.standard_normal((T, Hkv, D))
    sel, _ = O.index_select(qi, ki, cu, topk=topk, block=block)
    assert np.any(sel[:, :, -1] >= 0) and np.any(O.positions(cu) // block >= topk)
    scale = 0.3
    o, lse = O.sparse_attn_fwd(q, k, v, sel, cu, scale, block=block)
    ro, rlse, rdq, rdk, rdv = _gqa_reference(q, k, v, do, sel, cu, scale, block)
    np.testing.assert_allclose(o, ro, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(lse, rlse, rtol=1e-10, atol=1e-12)
    dq, dk, dv = O.sparse_attn_bwd(q, k, v, do, sel, cu, scale, block=block)
    np.testing.assert_allclose(dq, rdq, rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(dk, rdk, rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(dv, rdv, rtol=1e-9, atol=1e-11)
    # sampled mode agrees with full mode
    out = O.sparse_attn_bwd(q, k, v, do, sel, cu, scale, dq_tokens=[0, 20, 63],
                            dkv_blocks=[(1, 0, 2), (3, 1, 0)], block=block)
    np.testing.assert_allclose(out["dq"], dq[[0, 20, 63]], rtol=1e-12, atol=1e-13)
    (dkb, dvb), (dkb2, dvb2) = out["dkv"]
    np.testing.assert_allclose(dkb, dk[cu[1] + 8:cu[1] + 12, 0], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dvb2, dv[cu[3]:cu[3] + 4, 1], rtol=1e-12, atol=1e-13)


def test_narrow_block_regime_matches_masked_library_attention():
    """The narrow-block variant ("#4581", Kernel tuning: 12 q / 1 kv head, head dim
    256, 4-token blocks) runs the same oracle with block=4: forward, lse and all
    three gradients equal masked library attention (fp64 autograd) on a ragged
    pack with seeded random block subsets, own block kept."""
    import workloads as W
    seqlens = (9, 23, 1)
    cu = np.concatenate([[0], np.cumsum(seqlens)])
    T, Hq, Hkv, D = sum(seqlens), 12, 1, 256
    r = rng(21)
    q, k, v, do = (r.standard_normal((T, h, D)) for h in (Hq, Hkv, Hkv, Hq))
    g = torch.Generator().manual_seed(3)
    sel = W.qsa_selection(seqlens, Hkv, 3, g, "cpu").numpy()
    assert np.all(sel[:, 0, 0] >= 0) and np.any(sel[:, 0, -1] >= 0)
    assert np.any(O.positions(cu) // 4 >= 3)        # some rows keep a strict subset
    scale = 1 / math.sqrt(D)
    o, lse = O.sparse_attn_fwd(q, k, v, sel, cu, scale, block=4)
    ro, rlse, rdq, rdk, rdv = _gqa_reference(q, k, v, do, sel, cu, scale, 4)
    np.testing.assert_allclose(o, ro, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(lse, rlse, rtol=1e-10, atol=1e-12)
    dq, dk, dv = O.sparse_attn_bwd(q, k, v, do, sel, cu, scale, block=4)
    np.testing.assert_allclose(dq, rdq, rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(dk, rdk, rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(dv, rdv, rtol=1e-9, atol=1e-11)


def test_narrow_block_full_selection_is_causal_attention():
    """With every causal 4-token block selected the narrow-block forward is plain
    causal GQA attention (two KV heads of 12 query heads each, head dim 256)."""
    import workloads as W
    seqlens = (37, 5)
    cu = np.concatenate([[0], np.cumsum(seqlens)])
    T, Hq, Hkv, D = sum(seqlens), 24, 2, 256
    r = rng(22)
    q, k, v = (r.standard_normal((T, h, D)) for h in (Hq, Hkv, Hkv))
    g = torch.Generator().manual_seed(4)
    sel = W.qsa_selection(seqlens, Hkv, 16, g, "cpu").numpy()    # 16 >= 10 blocks
    scale = 1 / math.sqrt(D)
    o, _ = O.sparse_attn_fwd(q, k, v, sel, cu, scale, block=4)
    G = Hq // Hkv
    for s in range(len(seqlens)):
        a, b = cu[s], cu[s + 1]
        qq = torch.from_numpy(q[a:b].transpose(1, 0, 2).copy())
        kk = torch.from_numpy(np.repeat(k[a:b], G, axis=1).transpose(1, 0, 2).copy())
        vv = torch.from_numpy(np.repeat(v[a:b], G, axis=1).transpose(1, 0, 2).copy())
        want = F.scaled_dot_product_attention(qq, kk, vv, is_causal=True, scale=scale)
        np.testing.assert_allclose(o[a:b], want.numpy().transpose(1, 0, 2), rtol=1e-10,
                                   atol=1e-12)


def test_backward_finite_differences():
    block, topk = 4, 2
    r = rng(13)
    cu = np.array([0, 11, 19])
    T, Hq, Hkv, D = 19, 2, 1, 4
    q, k, v, do = (r.standard_normal((T, h, D)) for h in (Hq, Hkv, Hkv, Hq))
    sel, _ = O.index_select(r.standard_normal((T, 1, D)), r.standard_normal((T, 1, D)), cu,
                            topk=topk, block=block)
    scale = 0.7
    loss = lambda q_, k_, v_: float(np.sum(O.sparse_attn_fwd(q_, k_, v_, sel, cu, scale, block=block)[0] * do))
    dq, dk, dv = O.sparse_attn_bwd(q, k, v, do, sel, cu, scale, block=block)
    h = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        for idx in [(0, 0, 0), (10, 0, 3), (15, 0, 1), (18, 0, 2)]:
            if idx[1] >= x.shape[1]:
                continue
            xp = x.copy(); xp[idx] += h
            xm = x.copy(); xm[idx] -= h
            args_p = {"q": (xp, k, v), "k": (q, xp, v), "v": (q, k, xp)}[name]
            args_m = {"q": (xm, k, v), "k": (q, xm, v), "v": (q, k, xm)}[name]
            fd = (loss(*args_p) - loss(*args_m)) / (2 * h)
            assert fd == pytest.approx(g[idx], rel=1e-6, abs=1e-8), (name, idx)


def test_lse_and_normalisation():
    r = rng(14)
    cu = np.array([0, 2600])
    q, k, v = r.standard_normal((2600, 2, 16)), r.standard_normal((2600, 1, 16)), np.ones((2600, 1, 16))
    sel, _ = O.index_select(r.standard_normal((2600, 1, 16)), r.standard_normal((2600, 1, 16)), cu)
    toks = [0, 5, 2047, 2048, 2599]
    o, lse = O.sparse_attn_fwd(q, k, v, sel, cu, 0.25, tokens=toks)
    np.testing.assert_allclose(o, 1.0, rtol=1e-12)    # softmax weights sum to one
    for n, t in enumerate(toks):
        own0 = (t // 128) * 128            # the own block is always attended
        assert lse[n, 0] >= 0.25 * float(np.max(k[own0:t + 1, 0] @ q[t, 0])) - 1e-12
        if t < 2048:                       # dense region: every key attended
            lg = 0.25 * (k[:t + 1, 0] @ q[t, 0])
            assert lse[n, 0] == pytest.approx(float(np.log(np.sum(np.exp(lg)))), rel=1e-12)


# ------------------------------------------------------------------ decode

def test_decode_equals_prefill_at_last_token():
    r = rng(15)
    lens = [2100, 130, 2560, 1]
    Hq, Hkv, D = 4, 2, 16
    pages_per = [(L + 127) // 128 for L in lens]
    P = sum(pages_per)
    perm = r.permutation(P)
    maxp = max(pages_per)
    table = np.full((len(lens), maxp), -1)
    kc = np.zeros((P, Hkv, 128, D)); vc = np.zeros((P, Hkv, 128, D)); ic = np.zeros((P, Hkv, 128, D))
    qd = r.standard_normal((len(lens), Hq, D)); qid = r.standard_normal((len(lens), Hkv, D))
    pos = 0
    for b, L in enumerate(lens):
        kk, vv, ii = (r.standard_normal((L, Hkv, D)) for _ in range(3))
        pg = perm[pos:pos + pages_per[b]]; pos += pages_per[b]
        table[b, :len(pg)] = pg
        for c, p in enumerate(pg):
            n = min(128, L - 128 * c)
            kc[p, :, :n] = kk[128 * c:128 * c + n].transpose(1, 0, 2)
            vc[p, :, :n] = vv[128 * c:128 * c + n].transpose(1, 0, 2)
            ic[p, :, :n] = ii[128 * c:128 * c + n].transpose(1, 0, 2)
        # prefill view of the same sequence: the new token is the last one
        qf = np.zeros((L, Hq, D)); qf[-1] = qd[b]
        qif = np.zeros((L, Hkv, D)); qif[-1] = qid[b]
        cu = np.array([0, L])
        sel_p, gap_p = O.index_select(qif, ii, cu, tokens=[L - 1])
        o_p, _ = O.sparse_attn_fwd(qf, kk, vv, _expand(sel_p, L), cu, 0.2, tokens=[L - 1])
        o_d, sel_d, gap_d = O.decode_step(qd, qid, kc, vc, ic, table, lens, 0.2, batch=[b])
        np.testing.assert_array_equal(sel_d[0], sel_p[0])
        np.testing.assert_allclose(o_d[0], o_p[0], rtol=1e-11, atol=1e-12)


def _expand(sel_last, L):
    s = np.full((L,) + sel_last.shape[1:], -1, dtype=np.int64)
    s[-1] = sel_last[0]
    return s


# ------------------------------------------------------------------ page facts

def test_page_facts_fixture():
    assert FACTS["hq"]["value"] // FACTS["hkv"]["value"] == 16
    assert FACTS["index_heads"]["value"] == FACTS["hkv"]["value"]
    assert FACTS["rope_dims"]["value"] * 2 == FACTS["d_head"]["value"]
    assert O.BLOCK == FACTS["block"]["value"] and O.TOPK == FACTS["topk_blocks"]["value"]
