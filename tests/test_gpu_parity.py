"""GPU parity: each C-ABI call against the fp64 CPU oracle on the same seeded
inputs.  Small packs (several tiles, ragged tails, an empty sequence) compare
every output element; the full workload sizes compare sampled outputs that the
oracle computes one by one.

Tolerances (from the statement of the method's acceptance): selected block sets are
bit-exact except on rows the oracle marks as near-ties (relative gap between
the 15th and 16th earlier block below 1e-3), which are counted; given the same
selection, o is within max-abs 2e-2 and rel-L2 1e-2 (bf16 I/O, fp32
accumulation) and gradients within rel-L2 1e-2.  lse is fp32 of an fp32
softmax: max-abs 1e-3.  The prologue output is bf16 of an fp32 computation:
within one bf16 step of the oracle's bf16 value, with < 1% of elements off.
"""
import math

import numpy as np
import pytest
import torch

import workloads as W
from oracle import msa_oracle as O
from tests import selection_check as SC

pytestmark = pytest.mark.gpu

SCALE = 1.0 / math.sqrt(128)
DEV = "cuda:0"


@pytest.fixture(scope="module")
def m():
    import __graft_entry__ as ge
    ge.build()
    import msa_block_sparse_gb300 as mod
    return mod


def f64(t):
    return t.detach().float().cpu().double().numpy()


def rel_l2(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def assert_close(got, want, max_abs, rel, what):
    err = float(np.max(np.abs(got - want))) if got.size else 0.0
    r = rel_l2(got, want)
    assert err <= max_abs and r <= rel, f"{what}: max-abs {err:.3e}, rel-L2 {r:.3e}"


def bf16_step(v):
    """Spacing of bf16 values around |v| (the oracle's value)."""
    a = np.maximum(np.abs(v), 2.0 ** -126)
    return np.ldexp(1.0, np.floor(np.log2(a)).astype(np.int64) - 7)


def compare_selection(gsel, osel, gap, what, own, scores_of, n_init=0):
    """Every GPU row a valid selection; rows that differ from the oracle's are
    near-ties and differ only inside the tie band (tests/selection_check.py).
    Returns (differing rows, near-tie rows)."""
    rep = SC.check_selection(gsel, osel, gap, own, scores_of, what, n_init)
    print(f"{what}: {rep['differing']} differing rows, {rep['near_tie']} near-tie rows "
          f"of {rep['rows']}")
    return rep["differing"], rep["near_tie"]


def own_blocks(cpu, tokens=None):
    pos = O.positions(cpu["cu_seqlens"].numpy())
    return (pos if tokens is None else pos[np.asarray(tokens)]) // 128


RAGGED = W.PrefillShape("ragged-64q4kv", (300, 0, 1, 2000, 129, 2433), 64, 4, 4, runs_bwd=True)
SMALL = {
    "tiny": W.config(0),
    "ragged": RAGGED,
}


def sample_tokens(shape, n_random=96, seed=0):
    cu = shape.cu_seqlens().tolist()
    toks = set()
    for s in range(shape.S):
        a, b = cu[s], cu[s + 1]
        if b <= a:
            continue
        for p in (0, 1, 127, 128, 2047, 2048, 2049, b - a - 1):
            if 0 <= p < b - a:
                toks.add(a + p)
    r = np.random.default_rng(seed)
    toks.update(int(x) for x in r.integers(0, shape.T, n_random))
    return sorted(toks)


# ------------------------------------------------------------------ inputs and oracle caches

_cache = {}


def inputs(name, shape, seed=0):
    key = (name, seed)
    if key not in _cache:
        big = shape.T > 8192
        x = W.make_prefill(shape, seed=seed, device=DEV if big else "cpu",
                           with_grad_out=True)
        gpu = {k: v.to(DEV) for k, v in x.items()}
        cpu = {k: v.cpu() for k, v in x.items()}
        _cache[key] = (cpu, gpu)
    return _cache[key]


def oracle_selection(name, shape, cpu):
    key = ("sel", name)
    if key not in _cache:
        _cache[key] = O.index_select(f64(cpu["q_idx"]), f64(cpu["k_idx"]),
                                     cpu["cu_seqlens"].numpy())
    return _cache[key]


def oracle_gap(name, shape, cpu):
    return oracle_selection(name, shape, cpu)[1]


# ------------------------------------------------------------------ prologue

@pytest.mark.parametrize("name", ["tiny", "ragged"])
def test_prologue_matches_oracle(m, name):
    shape = SMALL[name]
    cpu, gpu = inputs(name, shape)
    cu = gpu["cu_seqlens"]
    q, k, qi, ki = m.msa_qk_norm_rope4(gpu["q"], gpu["k"], gpu["q_idx"], gpu["k_idx"],
                                       gpu["w_q"], gpu["w_k"], gpu["w_qi"], gpu["w_ki"], cu)
    q1 = m.msa_qk_norm_rope(gpu["q"], gpu["w_q"], cu)
    k2 = gpu["k"].clone()
    m.msa_qk_norm_rope(k2, gpu["w_k"], cu, out=k2)          # in place
    m.msa_check_status()
    assert torch.equal(q1, q) and torch.equal(k2, k)
    cun = cpu["cu_seqlens"].numpy()
    for got, n, wn in ((q, "q", "w_q"), (k, "k", "w_k"), (qi, "q_idx", "w_qi"), (ki, "k_idx", "w_ki")):
        assert_prologue_close(f64(got), O.qk_norm_rope(f64(cpu[n]), f64(cpu[wn]), cun), n)


def assert_prologue_close(g, want, n):
    """Each bf16 output within one bf16 step of the oracle's bf16 value: fp32
    evaluation leaves an absolute error of a few 2^-24 of the row's magnitude
    before the rounding (cancellation in the rotation makes it large relative
    to small outputs), and the rounding may then land one step off; fewer
    than 1% of the elements may be off."""
    off = np.abs(g - want)
    row_scale = np.max(np.abs(want), axis=-1, keepdims=True)
    tol = bf16_step(want) * 1.0001 + 1e-5 * row_scale
    worst = float(np.max(off - tol))
    assert worst <= 0, f"{n}: {int(np.sum(off > tol))} elements beyond tolerance, " \
                       f"worst excess {worst:.3e}, max off {float(off.max()):.3e}"
    assert np.mean(off > 0) < 0.01, f"{n}: {np.mean(off > 0):.4f} of elements off by a step"


def oracle_prologue_rows(cpu, name, wname, tokens):
    """The oracle's prologue (gemma norm, partial RoPE at each token's position,
    bf16 storage) of the given packed rows only: the prologue acts row by row."""
    pos = O.positions(cpu["cu_seqlens"].numpy())[tokens]
    x = f64(cpu[name][tokens])
    return O.bf16_round(O.partial_rope(O.gemma_rmsnorm(x, f64(cpu[wname])), pos))


def test_prologue_full_size_sampled(m):
    """The four prologue outputs of the full layer shape (64 q / 4 kv / 4 index
    heads, 16k pack of 8 sequences) on sampled rows of every sequence."""
    shape = W.config(2)
    cpu, gpu = inputs("cfg2", shape)
    q, k, qi, ki = m.msa_qk_norm_rope4(gpu["q"], gpu["k"], gpu["q_idx"], gpu["k_idx"],
                                       gpu["w_q"], gpu["w_k"], gpu["w_qi"], gpu["w_ki"],
                                       gpu["cu_seqlens"])
    m.msa_check_status()
    toks = sample_tokens(shape, n_random=512, seed=31)
    for got, n, wn in ((q, "q", "w_q"), (k, "k", "w_k"), (qi, "q_idx", "w_qi"), (ki, "k_idx", "w_ki")):
        assert_prologue_close(f64(got[toks]), oracle_prologue_rows(cpu, n, wn, toks), f"cfg2 {n}")


@pytest.mark.parametrize("heads", [(3, 5, 1), (7, 2, 3)])
def test_prologue_odd_head_counts(m, heads):
    """Head counts that do not fill the kernels' row slots evenly (the four
    tensors' rows of a token interleave across slots and CTAs), on a ragged
    pack with an empty and a one-token sequence: the forward of the 4-tensor
    call and the backward of each tensor against the oracle."""
    hq, hkv, hi = heads
    shape = W.PrefillShape("odd-heads", (300, 0, 1, 777, 129), hq, hkv, hi)
    gen = torch.Generator().manual_seed(101 + hq)
    T = shape.T
    x = {n: torch.randn((T, h, 128), generator=gen).to(torch.bfloat16)
         for n, h in (("q", hq), ("k", hkv), ("q_idx", hi), ("k_idx", hi))}
    w = {n: (0.1 * torch.randn(128, generator=gen)).to(torch.bfloat16)
         for n in ("w_q", "w_k", "w_qi", "w_ki")}
    cu_cpu = shape.cu_seqlens()
    cun = cu_cpu.numpy()
    g = {n: v.to(DEV) for n, v in list(x.items()) + list(w.items())}
    cu = cu_cpu.to(DEV)
    outs = m.msa_qk_norm_rope4(g["q"], g["k"], g["q_idx"], g["k_idx"], g["w_q"], g["w_k"],
                               g["w_qi"], g["w_ki"], cu)
    m.msa_check_status()
    for got, n, wn in zip(outs, ("q", "k", "q_idx", "k_idx"), ("w_q", "w_k", "w_qi", "w_ki")):
        assert_prologue_close(f64(got), O.qk_norm_rope(f64(x[n]), f64(w[wn]), cun), f"{heads} {n}")
    for n, wn in (("q", "w_q"), ("k", "w_k")):
        dy_cpu = torch.randn(x[n].shape, generator=gen).to(torch.bfloat16)
        dx, dw = m.msa_qk_norm_rope_bwd(g[n], dy_cpu.to(DEV), g[wn], cu)
        m.msa_check_status()
        want_dx, want_dw = O.qk_norm_rope_bwd(f64(x[n]), f64(w[wn]), f64(dy_cpu), cun)
        off = np.abs(f64(dx) - want_dx)
        tol = bf16_step(want_dx) * 1.0001 + 1e-5 * np.max(np.abs(want_dx), axis=-1, keepdims=True)
        assert float(np.max(off - tol)) <= 0, f"{heads} {n} dx"
        assert rel_l2(f64(dw), want_dw) <= 1e-4, f"{heads} {n} dw"


def test_prologue_head_limit(m):
    """256 heads per tensor (the most the prologue kernels take: a CTA's rows of
    one tensor reach 16 x 256) against the oracle, forward and backward, on a
    ragged pack; 257 heads are refused with an error before anything runs."""
    cu_cpu = torch.tensor([0, 3, 20, 21], dtype=torch.int32)
    cun = cu_cpu.numpy()
    T = int(cun[-1])
    gen = torch.Generator().manual_seed(256)
    x = torch.randn((T, 256, 128), generator=gen).to(torch.bfloat16)
    w = (0.1 * torch.randn(128, generator=gen)).to(torch.bfloat16)
    dy = torch.randn((T, 256, 128), generator=gen).to(torch.bfloat16)
    cu = cu_cpu.to(DEV)
    y = m.msa_qk_norm_rope(x.to(DEV), w.to(DEV), cu)
    dx, dw = m.msa_qk_norm_rope_bwd(x.to(DEV), dy.to(DEV), w.to(DEV), cu)
    m.msa_check_status()
    assert_prologue_close(f64(y), O.qk_norm_rope(f64(x), f64(w), cun), "256 heads")
    want_dx, want_dw = O.qk_norm_rope_bwd(f64(x), f64(w), f64(dy), cun)
    off = np.abs(f64(dx) - want_dx)
    tol = bf16_step(want_dx) * 1.0001 + 1e-5 * np.max(np.abs(want_dx), axis=-1, keepdims=True)
    assert float(np.max(off - tol)) <= 0, "256 heads dx"
    assert rel_l2(f64(dw), want_dw) <= 1e-4, "256 heads dw"
    big = torch.zeros((T, 257, 128), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(m.MSAError):
        m.msa_qk_norm_rope(big, w.to(DEV), cu)
    with pytest.raises(m.MSAError):
        m.msa_qk_norm_rope_bwd(big, big, w.to(DEV), cu)
    m.msa_check_status()


@pytest.mark.parametrize("name", ["tiny", "ragged"])
def test_prologue_backward_matches_oracle(m, name):
    """dx (bf16) and dw (fp32) of the q and k prologues against the fp64 closed
    form: every element of dx within one bf16 step (plus a small fp32 term),
    dw to 1e-4 relative; dx written over dy gives the same bits; dw is the same
    on a second run."""
    shape = SMALL[name]
    cpu, gpu = inputs(name, shape)
    cu = gpu["cu_seqlens"]
    cun = cpu["cu_seqlens"].numpy()
    gen = torch.Generator().manual_seed(7)
    for n, wn in (("q", "w_q"), ("k", "w_k")):
        dy_cpu = torch.randn(cpu[n].shape, generator=gen).to(torch.bfloat16)
        dy = dy_cpu.to(DEV)
        dx, dw = m.msa_qk_norm_rope_bwd(gpu[n], dy, gpu[wn], cu)
        dy2 = dy.clone()
        dx2, dw2 = m.msa_qk_norm_rope_bwd(gpu[n], dy2, gpu[wn], cu, dx=dy2)
        m.msa_check_status()
        assert torch.equal(dx2, dx) and torch.equal(dw2, dw), n
        want_dx, want_dw = O.qk_norm_rope_bwd(f64(cpu[n]), f64(cpu[wn]), f64(dy_cpu), cun)
        g = f64(dx)
        off = np.abs(g - want_dx)
        row_scale = np.max(np.abs(want_dx), axis=-1, keepdims=True)
        tol = bf16_step(want_dx) * 1.0001 + 1e-5 * row_scale
        worst = float(np.max(off - tol))
        assert worst <= 0, f"{n} dx: {int(np.sum(off > tol))} elements beyond tolerance, " \
                           f"worst excess {worst:.3e}"
        assert rel_l2(f64(dw), want_dw) <= 1e-4, f"{n} dw rel-L2 {rel_l2(f64(dw), want_dw):.3e}"


# ------------------------------------------------------------------ index select

@pytest.mark.parametrize("name", ["tiny", "ragged"])
def test_index_select_small(m, name):
    shape = SMALL[name]
    cpu, gpu = inputs(name, shape)
    sel = m.msa_index_select(gpu["q_idx"], gpu["k_idx"], gpu["cu_seqlens"], max(shape.max_seqlen, 1))
    m.msa_check_status()
    osel, gap = oracle_selection(name, shape, cpu)
    cun = cpu["cu_seqlens"].numpy()
    compare_selection(sel.cpu().numpy(), osel, gap, name, own_blocks(cpu),
                      SC.prefill_scores_of(f64(cpu["q_idx"]), f64(cpu["k_idx"]), cun,
                                           np.arange(shape.T)))


@pytest.mark.parametrize("idx", [1, 2, 4])
def test_index_select_full_size(m, idx):
    shape = W.config(idx)
    cpu, gpu = inputs(f"cfg{idx}", shape)
    sel = m.msa_index_select(gpu["q_idx"], gpu["k_idx"], gpu["cu_seqlens"], shape.max_seqlen)
    m.msa_check_status()
    toks = sample_tokens(shape, n_random=1024, seed=idx)
    osel, gap = O.index_select(f64(cpu["q_idx"]), f64(cpu["k_idx"]), cpu["cu_seqlens"].numpy(),
                               tokens=toks)
    compare_selection(sel.cpu().numpy()[toks], osel, gap, f"cfg{idx}", own_blocks(cpu, toks),
                      SC.prefill_scores_of(f64(cpu["q_idx"]), f64(cpu["k_idx"]),
                                           cpu["cu_seqlens"].numpy(), toks))


@pytest.mark.parametrize("n_init", [1, 3])
def test_index_select_init_rule(m, n_init):
    """The init rule (msa_index_select_ex): the first n_init blocks are always
    kept, on the ragged pack and sampled rows of the 16k pack."""
    for name, shape in (("ragged", RAGGED), ("cfg1", W.config(1))):
        cpu, gpu = inputs(name, shape)
        sel = m.msa_index_select(gpu["q_idx"], gpu["k_idx"], gpu["cu_seqlens"],
                                 max(shape.max_seqlen, 1), n_init=n_init)
        m.msa_check_status()
        toks = None if shape.T <= 8192 else sample_tokens(shape, n_random=512, seed=7)
        osel, gap = O.index_select(f64(cpu["q_idx"]), f64(cpu["k_idx"]),
                                   cpu["cu_seqlens"].numpy(), tokens=toks, n_init=n_init)
        g = sel.cpu().numpy() if toks is None else sel.cpu().numpy()[toks]
        rows = np.arange(shape.T) if toks is None else toks
        compare_selection(g, osel, gap, f"{name} n_init={n_init}", own_blocks(cpu, rows),
                          SC.prefill_scores_of(f64(cpu["q_idx"]), f64(cpu["k_idx"]),
                                               cpu["cu_seqlens"].numpy(), rows), n_init=n_init)
        pos = O.positions(cpu["cu_seqlens"].numpy())
        own = (pos if toks is None else pos[toks]) // 128
        for i in range(n_init):
            keep = own > i
            assert np.all(np.any(g[keep] == i, axis=-1)), f"{name}: block {i} not kept"


def test_index_select_exact_ties(m):
    """Key blocks 0 .. 9 of each sequence copies of one block B, every later
    one a copy of 2B (exact in bf16), so a token's earlier blocks score
    exactly m or 2m (m > 0): by the selection rule (equal scores: lower block
    first) a token with own block o keeps the lowest min(15, o - 10) of the 2B
    blocks 10 .. o - 1, then the lowest B blocks 0 .. in the places left, and
    o.  The larger scores arrive after the tied ones, so a list kept in
    score order must move tied entries down without reordering them.  The
    150-block sequence makes the pack's chunks longer than 16 blocks, so both
    the sorted-at-the-end path (units of at most 16 blocks) and the
    insert-as-they-come path run, and chunk lists with tied entries are
    merged across CTAs."""
    lens = (150 * 128, 300, 0, 2100)
    cu_cpu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32)
    T = int(cu_cpu[-1])
    gen = torch.Generator().manual_seed(77)
    qi = torch.randn((T, 1, 128), generator=gen).to(torch.bfloat16)
    blk = torch.randn((128, 1, 128), generator=gen).to(torch.bfloat16)
    ki = torch.empty((T, 1, 128), dtype=torch.bfloat16)
    k = 10
    for s0, L in zip(cu_cpu[:-1].tolist(), lens):
        for b in range((L + 127) // 128):
            n = min(128, L - 128 * b)
            ki[s0 + 128 * b:s0 + 128 * b + n] = blk[:n] * (2 if b >= k else 1)
    # every token's block maximum over B must be positive for 2B to score higher
    q64, b64 = f64(qi)[:, 0, :], f64(blk)[:, 0, :]
    assert np.all((q64 @ b64.T).max(axis=1) > 0)
    sel = m.msa_index_select(qi.to(DEV), ki.to(DEV), cu_cpu.to(DEV), max(lens))
    m.msa_check_status()
    got = sel.cpu().numpy()[:, 0, :]
    own = O.positions(cu_cpu.numpy()) // 128
    want = np.full((T, 16), -1, dtype=np.int64)
    for t in range(T):
        o = int(own[t])
        hi = np.arange(k, o)[:15]                       # 2B blocks, lowest first
        lo = np.arange(min(o, k))[:15 - hi.size]        # then B blocks, lowest first
        row = np.sort(np.concatenate([hi, lo, [o]]))
        want[t, :row.size] = row
    bad = np.nonzero(np.any(got != want, axis=1))[0]
    assert bad.size == 0, f"{bad.size} rows differ, first {bad[:4].tolist()}: " \
                          f"{got[bad[0]].tolist()} != {want[bad[0]].tolist()}"


def test_index_select_max_seqlen(m):
    """One sequence of the longest supported length (1024 blocks of 128 tokens)
    beside a short one: the plans' largest histograms, chunks longer than 16
    blocks (the insert-as-they-come path) and up to 1023 earlier blocks per
    query tile; sampled rows against the oracle.  One token more is refused
    before anything runs."""
    L = 1024 * 128
    cu_cpu = torch.tensor([0, L, L + 300], dtype=torch.int32)
    T = L + 300
    gen = torch.Generator().manual_seed(1024)
    qi = torch.randn((T, 1, 128), generator=gen).to(torch.bfloat16)
    ki = torch.randn((T, 1, 128), generator=gen).to(torch.bfloat16)
    sel = m.msa_index_select(qi.to(DEV), ki.to(DEV), cu_cpu.to(DEV), L)
    m.msa_check_status()
    rng = np.random.default_rng(1024)
    toks = sorted({0, 127, 128, 2047, 16383, 16384, 65535, 65536, L - 129, L - 128, L - 1, L,
                   T - 1} | set(int(x) for x in rng.integers(0, T, 24)))
    cun = cu_cpu.numpy()
    osel, gap = O.index_select(f64(qi), f64(ki), cun, tokens=toks)
    compare_selection(sel.cpu().numpy()[toks], osel, gap, "max seqlen",
                      own_blocks({"cu_seqlens": cu_cpu}, toks),
                      SC.prefill_scores_of(f64(qi), f64(ki), cun, toks))
    cu2 = torch.tensor([0, L + 1, T], dtype=torch.int32, device=DEV)
    with pytest.raises(m.MSAError):
        m.msa_index_select(qi.to(DEV), ki.to(DEV), cu2, L + 1)
    m.msa_check_status()


# ------------------------------------------------------------------ forward

@pytest.mark.parametrize("name", ["tiny", "ragged"])
def test_sparse_fwd_small(m, name):
    shape = SMALL[name]
    cpu, gpu = inputs(name, shape)
    osel, _ = oracle_selection(name, shape, cpu)
    sel = torch.from_numpy(osel.astype(np.int32)).to(DEV)
    o, lse = m.msa_sparse_attn_fwd(gpu["q"], gpu["k"], gpu["v"], sel, gpu["cu_seqlens"],
                                   max(shape.max_seqlen, 1))
    m.msa_check_status()
    oo, olse = O.sparse_attn_fwd(f64(cpu["q"]), f64(cpu["k"]), f64(cpu["v"]), osel,
                                 cpu["cu_seqlens"].numpy(), SCALE)
    assert_close(f64(o), oo, 2e-2, 1e-2, f"{name} o")
    assert_close(lse.cpu().numpy().astype(np.float64), olse, 1e-3, 1e-4, f"{name} lse")
    o2, lse2 = m.msa_sparse_attn_fwd(gpu["q"], gpu["k"], gpu["v"], sel, gpu["cu_seqlens"],
                                     max(shape.max_seqlen, 1))
    assert torch.equal(o, o2) and torch.equal(lse, lse2), "forward is not deterministic"


@pytest.mark.parametrize("idx", [1, 2, 4])
def test_sparse_fwd_full_size(m, idx):
    shape = W.config(idx)
    cpu, gpu = inputs(f"cfg{idx}", shape)
    osel, _ = oracle_selection(f"cfg{idx}", shape, cpu)
    sel = torch.from_numpy(osel.astype(np.int32)).to(DEV)
    o, lse = m.msa_sparse_attn_fwd(gpu["q"], gpu["k"], gpu["v"], sel, gpu["cu_seqlens"],
                                   shape.max_seqlen)
    m.msa_check_status()
    toks = sample_tokens(shape, n_random=160, seed=10 + idx)
    oo, olse = O.sparse_attn_fwd(f64(cpu["q"]), f64(cpu["k"]), f64(cpu["v"]), osel,
                                 cpu["cu_seqlens"].numpy(), SCALE, tokens=toks)
    assert_close(f64(o[toks]), oo, 2e-2, 1e-2, f"cfg{idx} o")
    assert_close(lse[toks].cpu().numpy().astype(np.float64), olse, 1e-3, 1e-4, f"cfg{idx} lse")


LONG = W.PrefillShape("long-17000-16q1kv", (17000, 700), 16, 1, 1)


def test_sparse_fwd_long_sequence(m):
    """A sequence longer than 16,384 tokens: the query blocks past that point
    form their 8-token tiles from consecutive tokens (their selection masks do
    not fit the grouping's registers), the earlier ones by selection
    similarity; rows on both sides compare with the oracle."""
    shape = LONG
    cpu, gpu = inputs("long", shape)
    osel, _ = oracle_selection("long", shape, cpu)
    sel = torch.from_numpy(osel.astype(np.int32)).to(DEV)
    o, lse = m.msa_sparse_attn_fwd(gpu["q"], gpu["k"], gpu["v"], sel, gpu["cu_seqlens"],
                                   shape.max_seqlen)
    m.msa_check_status()
    toks = sorted(set(sample_tokens(shape, n_random=64, seed=21))
                  | {16383, 16384, 16385, 16391, 16392, 16511, 16512, 16999})
    oo, olse = O.sparse_attn_fwd(f64(cpu["q"]), f64(cpu["k"]), f64(cpu["v"]), osel,
                                 cpu["cu_seqlens"].numpy(), SCALE, tokens=toks)
    assert_close(f64(o[toks]), oo, 2e-2, 1e-2, "long o")
    assert_close(lse[toks].cpu().numpy().astype(np.float64), olse, 1e-3, 1e-4, "long lse")
    # the index select on the same pack: the long sequence's query tiles have
    # up to 132 earlier blocks, cut into several chunks whose top-15 lists the
    # last chunk merges
    gsel = m.msa_index_select(gpu["q_idx"], gpu["k_idx"], gpu["cu_seqlens"], shape.max_seqlen)
    m.msa_check_status()
    compare_selection(gsel.cpu().numpy()[toks], osel[toks], oracle_gap("long", shape, cpu)[toks],
                      "long select", own_blocks(cpu, toks),
                      SC.prefill_scores_of(f64(cpu["q_idx"]), f64(cpu["k_idx"]),
                                           cpu["cu_seqlens"].numpy(), toks))


# ------------------------------------------------------------------ backward

BWD_SMALL = {
    "2seq-16q1kv": W.PrefillShape("2seq-16q1kv", (2100, 1400), 16, 1, 1, runs_bwd=True),
    "3seq-32q2kv": W.PrefillShape("3seq-32q2kv", (700, 1, 2433), 32, 2, 2, runs_bwd=True),
}


@pytest.mark.parametrize("name", list(BWD_SMALL))
def test_sparse_bwd_small(m, name):
    shape = BWD_SMALL[name]
    cpu, gpu = inputs(name, shape)
    osel, _ = oracle_selection(name, shape, cpu)
    sel = torch.from_numpy(osel.astype(np.int32)).to(DEV)
    cu = gpu["cu_seqlens"]
    o, lse = m.msa_sparse_attn_fwd(gpu["q"], gpu["k"], gpu["v"], sel, cu, shape.max_seqlen)
    dq, dk, dv = m.msa_sparse_attn_bwd(gpu["q"], gpu["k"], gpu["v"], o, gpu["do"], lse, sel, cu,
                                       shape.max_seqlen)
    m.msa_check_status()
    rq, rk, rv = O.sparse_attn_bwd(f64(cpu["q"]), f64(cpu["k"]), f64(cpu["v"]), f64(cpu["do"]),
                                   osel, cpu["cu_seqlens"].numpy(), SCALE)
    for got, want, n in ((dq, rq, "dq"), (dk, rk, "dk"), (dv, rv, "dv")):
        r = rel_l2(f64(got), want)
        assert r <= 1e-2, f"{name} {n}: rel-L2 {r:.3e}"


def test_sparse_bwd_prepared_on_a_second_stream(m):
    """msa_sparse_attn_bwd_prepare on another stream (ordered by an event) and
    msa_sparse_attn_bwd_prepared give the oracle's gradients; the workspace is
    dirty before the prepare (a previous backward ran in it)."""
    name = "2seq-16q1kv"
    shape = BWD_SMALL[name]
    cpu, gpu = inputs(name, shape)
    osel, _ = oracle_selection(name, shape, cpu)
    sel = torch.from_numpy(osel.astype(np.int32)).to(DEV)
    cu = gpu["cu_seqlens"]
    L = shape.max_seqlen
    o, lse = m.msa_sparse_attn_fwd(gpu["q"], gpu["k"], gpu["v"], sel, cu, L)
    ws = torch.empty(m.workspace_bytes("sparse_attn_bwd", shape.T, shape.S, shape.hq, shape.hkv, L),
                     dtype=torch.uint8, device=DEV)
    ref = m.msa_sparse_attn_bwd(gpu["q"], gpu["k"], gpu["v"], o, gpu["do"], lse, sel, cu, L,
                                workspace=ws)
    side = torch.cuda.Stream(DEV)
    ready, cleared = torch.cuda.Event(), torch.cuda.Event()
    ready.record(torch.cuda.current_stream())
    side.wait_event(ready)
    m.msa_sparse_attn_bwd_prepare(gpu["q"], gpu["k"], cu, L, ws, stream=side)
    cleared.record(side)
    torch.cuda.current_stream().wait_event(cleared)
    got = m.msa_sparse_attn_bwd(gpu["q"], gpu["k"], gpu["v"], o, gpu["do"], lse, sel, cu, L,
                                workspace=ws, prepared=True)
    m.msa_check_status()
    rq, rk, rv = O.sparse_attn_bwd(f64(cpu["q"]), f64(cpu["k"]), f64(cpu["v"]), f64(cpu["do"]),
                                   osel, cpu["cu_seqlens"].numpy(), SCALE)
    for g_, r_, want, n in zip(got, ref, (rq, rk, rv), ("dq", "dk", "dv")):
        assert rel_l2(f64(g_), want) <= 1e-2, n
        # the same kernels on the same inputs: only the order of the fp32
        # atomic additions may differ between the two runs
        assert rel_l2(f64(g_), f64(r_)) <= 1e-3, n
    with pytest.raises(ValueError):
        m.msa_sparse_attn_bwd(gpu["q"], gpu["k"], gpu["v"], o, gpu["do"], lse, sel, cu, L,
                              prepared=True)


def bwd_sample_blocks(shape, seed):
    """(sequence, KV head, block) triples whose dk/dv a full-size backward test
    compares: for every sequence and KV head block 0 or 1 (selected by almost
    every query of the sequence, so its work spans all 256-position windows),
    one random block past them and the sequence's last block (partly causal,
    claimed late from the largest-first tail)."""
    r = np.random.default_rng(seed)
    out = []
    for s in range(shape.S):
        nb = (shape.seqlens[s] + 127) // 128
        for g in range(shape.hkv):
            picks = {int(r.integers(0, min(2, nb))), nb - 1}
            if nb > 3:
                picks.add(int(r.integers(2, nb - 1)))
            out += [(s, g, b) for b in sorted(picks)]
    return out


def check_bwd_sampled(cpu, dq, dk, dv, sel, shape, toks, blocks, what, q=None, k=None):
    """dq on the sampled tokens and dk/dv of the sampled blocks against the
    oracle's sampled backward (blocks computed in a spawned process pool)."""
    from tests import oracle_pool
    cun = cpu["cu_seqlens"].numpy()
    qq = f64(cpu["q"]) if q is None else q
    kk = f64(cpu["k"]) if k is None else k
    vv, dd = f64(cpu["v"]), f64(cpu["do"])
    ref = O.sparse_attn_bwd(qq, kk, vv, dd, sel, cun, SCALE, dq_tokens=toks)
    r = rel_l2(f64(dq[toks]), ref["dq"])
    assert r <= 1e-2, f"{what} dq rel-L2 {r:.3e}"
    dkv = oracle_pool.dkv_blocks(qq, kk, vv, dd, sel, cun, SCALE, blocks)
    worst = 0.0
    for (s, g, b), (rk, rv) in zip(blocks, dkv):
        k0 = int(cun[s]) + 128 * b
        n = rk.shape[0]
        rk_ = rel_l2(f64(dk[k0:k0 + n, g]), rk)
        rv_ = rel_l2(f64(dv[k0:k0 + n, g]), rv)
        worst = max(worst, rk_, rv_)
        assert rk_ <= 1e-2 and rv_ <= 1e-2, f"{what} block {(s, g, b)}: dk {rk_:.3e} dv {rv_:.3e}"
    print(f"{what}: dq on {len(toks)} tokens rel-L2 {r:.2e}; dk/dv on {len(blocks)} blocks, "
          f"worst rel-L2 {worst:.2e}")


@pytest.mark.parametrize("name", ["tiny", "ragged"])
def test_sparse_fwd_train_clears_bwd_workspace(m, name):
    """msa_sparse_attn_fwd_train zeroes the backward workspace's accumulators
    while it runs: with the workspace first filled with NaN bytes, its o and
    lse equal the plain forward's bit for bit and the prepared backward that
    follows matches the oracle and the unprepared backward."""
    shape = SMALL[name]
    cpu, gpu = inputs(name, shape)
    osel, _ = oracle_selection(name, shape, cpu)
    sel = torch.from_numpy(osel.astype(np.int32)).to(DEV)
    cu = gpu["cu_seqlens"]
    L = shape.max_seqlen
    o_ref, lse_ref = m.msa_sparse_attn_fwd(gpu["q"], gpu["k"], gpu["v"], sel, cu, L)
    ref = m.msa_sparse_attn_bwd(gpu["q"], gpu["k"], gpu["v"], o_ref, gpu["do"], lse_ref, sel, cu,
                                L)
    ws = torch.full((m.workspace_bytes("sparse_attn_bwd", shape.T, shape.S, shape.hq, shape.hkv,
                                       L),), 0xFF, dtype=torch.uint8, device=DEV)
    o, lse = m.msa_sparse_attn_fwd(gpu["q"], gpu["k"], gpu["v"], sel, cu, L, bwd_workspace=ws)
    got = m.msa_sparse_attn_bwd(gpu["q"], gpu["k"], gpu["v"], o, gpu["do"], lse, sel, cu, L,
                                workspace=ws, prepared=True)
    m.msa_check_status()
    assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)
    rq, rk, rv = O.sparse_attn_bwd(f64(cpu["q"]), f64(cpu["k"]), f64(cpu["v"]), f64(cpu["do"]),
                                   osel, cpu["cu_seqlens"].numpy(), SCALE)
    for g_, r_, want, n in zip(got, ref, (rq, rk, rv), ("dq", "dk", "dv")):
        assert torch.isfinite(g_.float()).all(), n
        assert rel_l2(f64(g_), want) <= 1e-2, n
        assert rel_l2(f64(g_), f64(r_)) <= 1e-3, n


@pytest.mark.parametrize("idx", [1, 4])
def test_sparse_bwd_full_size(m, idx):
    """Full-size backward with the oracle's selection: dq on >= 256 sampled
    tokens, dk / dv on 2-3 blocks of every (sequence, KV head)."""
    shape = W.config(idx)
    cpu, gpu = inputs(f"cfg{idx}", shape)
    osel, _ = oracle_selection(f"cfg{idx}", shape, cpu)
    sel = torch.from_numpy(osel.astype(np.int32)).to(DEV)
    cu = gpu["cu_seqlens"]
    o, lse = m.msa_sparse_attn_fwd(gpu["q"], gpu["k"], gpu["v"], sel, cu, shape.max_seqlen)
    dq, dk, dv = m.msa_sparse_attn_bwd(gpu["q"], gpu["k"], gpu["v"], o, gpu["do"], lse, sel, cu,
                                       shape.max_seqlen)
    m.msa_check_status()
    toks = sample_tokens(shape, n_random=256, seed=20 + idx)
    blocks = bwd_sample_blocks(shape, seed=40 + idx)
    assert len(toks) >= 256 and len(blocks) >= (12 if idx == 1 else 32)
    check_bwd_sampled(cpu, dq, dk, dv, osel, shape, toks, blocks, f"cfg{idx}")


def test_pipeline_full_size_sampled(m):
    """The whole training step of the 16k pack (16 q / 1 kv / 1 index head) on
    the GPU -- prologue, index select, forward, backward -- against the oracle
    pipeline on sampled rows: prologue outputs, the selection (near-tie rule),
    o and lse, dq, and dk / dv of sampled blocks.  The oracle's attention and
    backward take the GPU's selection (validated on the sampled rows) and its
    own prologue outputs."""
    shape = W.config(1)
    cpu, gpu = inputs("cfg1", shape)
    cu = gpu["cu_seqlens"]
    L = shape.max_seqlen
    q, k, qi, ki = m.msa_qk_norm_rope4(gpu["q"], gpu["k"], gpu["q_idx"], gpu["k_idx"],
                                       gpu["w_q"], gpu["w_k"], gpu["w_qi"], gpu["w_ki"], cu)
    sel = m.msa_index_select(qi, ki, cu, L)
    o, lse = m.msa_sparse_attn_fwd(q, k, gpu["v"], sel, cu, L)
    dq, dk, dv = m.msa_sparse_attn_bwd(q, k, gpu["v"], o, gpu["do"], lse, sel, cu, L)
    m.msa_check_status()
    cun = cpu["cu_seqlens"].numpy()
    pq = O.qk_norm_rope(f64(cpu["q"]), f64(cpu["w_q"]), cun)
    pk = O.qk_norm_rope(f64(cpu["k"]), f64(cpu["w_k"]), cun)
    pqi = O.qk_norm_rope(f64(cpu["q_idx"]), f64(cpu["w_qi"]), cun)
    pki = O.qk_norm_rope(f64(cpu["k_idx"]), f64(cpu["w_ki"]), cun)
    toks = sample_tokens(shape, n_random=512, seed=51)
    for got, want, n in ((q, pq, "q"), (k, pk, "k"), (qi, pqi, "q_idx"), (ki, pki, "k_idx")):
        assert_prologue_close(f64(got[toks]), want[toks], f"pipeline {n}")
    gsel = sel.cpu().numpy().astype(np.int64)
    osel, gap = O.index_select(pqi, pki, cun, tokens=toks)
    compare_selection(gsel[toks], osel, gap, "pipeline cfg1", own_blocks(cpu, toks),
                      SC.prefill_scores_of(pqi, pki, cun, toks))
    oo, olse = O.sparse_attn_fwd(pq, pk, f64(cpu["v"]), gsel, cun, SCALE, tokens=toks)
    assert_close(f64(o[toks]), oo, 2e-2, 1e-2, "pipeline o")
    assert_close(lse[toks].cpu().numpy().astype(np.float64), olse, 1e-3, 1e-4, "pipeline lse")
    blocks = [(s, 0, b) for (s, _, b) in bwd_sample_blocks(shape, seed=52)]
    check_bwd_sampled(cpu, dq, dk, dv, gsel, shape, toks, blocks, "pipeline cfg1", q=pq, k=pk)


# ------------------------------------------------------------------ decode

def _decode_check(m, shape, seed, rows=None, n_init=0):
    big = shape.B > 16
    x = W.make_decode(shape, seed=seed, device=DEV if big else "cpu")
    g = {k: v.to(DEV) for k, v in x.items()}
    o, sel = m.msa_decode_step(g["q"], g["q_idx"], g["k_cache"], g["v_cache"], g["kidx_cache"],
                               g["block_table"], g["cache_lens"], n_init=n_init)
    m.msa_check_status()
    rows = list(range(shape.B)) if rows is None else rows
    # copy to the host only the pages the sampled rows use, with a remapped table
    table = x["block_table"].cpu().numpy()
    lens = x["cache_lens"].cpu().numpy()
    used = sorted({int(p) for b in rows for p in table[b, :(lens[b] + 127) // 128]})
    remap = {p: i for i, p in enumerate(used)}
    sub_table = np.full((len(rows), table.shape[1]), -1, dtype=np.int64)
    for n, b in enumerate(rows):
        for c in range((lens[b] + 127) // 128):
            sub_table[n, c] = remap[int(table[b, c])]
    idx = torch.tensor(used, dtype=torch.long, device=x["k_cache"].device)
    kc, vc, ic = (x[n].index_select(0, idx).float().cpu().numpy()
                  for n in ("k_cache", "v_cache", "kidx_cache"))
    ro, rsel, rgap = O.decode_step(f64(x["q"][rows]), f64(x["q_idx"][rows]), kc, vc, ic,
                                   sub_table, lens[rows], SCALE, n_init=n_init)
    gsel = sel.cpu().numpy()[rows]
    compare_selection(gsel, rsel, rgap, shape.name, (lens[rows] - 1) // 128,
                      SC.decode_scores_of(f64(x["q_idx"][rows]), ic, sub_table, lens[rows]),
                      n_init=n_init)
    same = np.all(np.all(gsel == rsel, axis=-1), axis=-1)
    assert same.mean() > 0.5
    assert_close(f64(o)[rows][same], ro[same], 2e-2, 1e-2, f"{shape.name} o")


def test_decode_small_edges(m):
    shape = W.DecodeShape("decode-edges", (1, 127, 128, 129, 2048, 2049, 5000, 300), 32, 2, 2)
    _decode_check(m, shape, seed=5)


def test_decode_init_rule(m):
    shape = W.DecodeShape("decode-init", (1, 127, 128, 129, 2048, 2049, 5000, 300), 32, 2, 2)
    _decode_check(m, shape, seed=6, n_init=2)


def test_decode_exact_ties(m):
    """Twenty earlier blocks of sequence 0 share one dominant index-key page, so
    their scores are exactly equal and straddle the 15-block cut: the rule
    (equal scores: lower block id first) must keep the 15 lowest of them."""
    shape = W.DecodeShape("decode-ties", (5120, 3000, 129, 4096), 32, 2, 2)
    x = W.make_decode(shape, seed=11, device="cpu")
    table = x["block_table"].numpy()
    tied = [2, 3, 5, 7, 8, 11, 13, 14, 17, 19, 21, 22, 24, 26, 27, 29, 31, 33, 35, 37]
    kidx = x["kidx_cache"].clone()
    for h in range(shape.hi):
        row = (x["q_idx"][0, h].float() * 4.0).to(torch.bfloat16)
        for blk in tied:
            kidx[int(table[0, blk]), h] = row
    x["kidx_cache"] = kidx
    g = {k: v.to(DEV) for k, v in x.items()}
    o, sel = m.msa_decode_step(g["q"], g["q_idx"], g["k_cache"], g["v_cache"], g["kidx_cache"],
                               g["block_table"], g["cache_lens"])
    m.msa_check_status()
    lens = x["cache_lens"].numpy()
    ro, rsel, rgap = O.decode_step(f64(x["q"]), f64(x["q_idx"]), f64(x["k_cache"]),
                                   f64(x["v_cache"]), f64(x["kidx_cache"]), table, lens, SCALE)
    gsel = sel.cpu().numpy()
    own0 = (lens[0] + 127) // 128 - 1
    want = sorted(tied[:15]) + [own0]
    for h in range(shape.hi):
        assert list(rsel[0, h]) == want, (h, rsel[0, h])      # the oracle applies the rule
        assert list(gsel[0, h]) == want, (h, gsel[0, h])      # and so must the kernels
    np.testing.assert_array_equal(gsel, rsel)
    assert_close(f64(o), ro, 2e-2, 1e-2, "decode-ties o")


def test_decode_full_size(m):
    _decode_check(m, W.config(3), seed=0, rows=[0, 1, 17, 33, 63])


def test_decode_append_then_step(m):
    """New tokens appended (prologue + page write) at ragged positions, including
    the first slot of a fresh page and a one-token cache, then a decode step on
    the result: append outputs within one bf16 step of the oracle, every other
    cache byte unchanged, the decode step as in test_decode_small_edges."""
    shape = W.DecodeShape("decode-append", (1, 128, 129, 300, 2049, 4096), 32, 2, 2)
    x = W.make_decode(shape, seed=9, device="cpu")
    gen = torch.Generator().manual_seed(3)
    B, hq, hkv = shape.B, shape.hq, shape.hkv
    raw = {n: torch.randn((B, h, 128), generator=gen).to(torch.bfloat16)
           for n, h in (("q", hq), ("q_idx", hkv), ("k", hkv), ("v", hkv), ("k_idx", hkv))}
    ws = {n: (torch.randn(128, generator=gen) * 0.2).to(torch.bfloat16)
          for n in ("w_q", "w_qi", "w_k", "w_ki")}
    g = {k: v.to(DEV) for k, v in x.items()}
    gr = {k: v.to(DEV) for k, v in raw.items()}
    gw = {k: v.to(DEV) for k, v in ws.items()}
    q_out, qi_out = m.msa_decode_append(gr["q"], gr["q_idx"], gr["k"], gr["v"], gr["k_idx"],
                                        gw["w_q"], gw["w_qi"], gw["w_k"], gw["w_ki"],
                                        g["k_cache"], g["v_cache"], g["kidx_cache"],
                                        g["block_table"], g["cache_lens"])
    m.msa_check_status()
    table = x["block_table"].numpy()
    lens = x["cache_lens"].numpy()
    oq, oqi, okc, ovc, oic = O.decode_append(
        f64(raw["q"]), f64(raw["k"]), f64(raw["v"]), f64(raw["q_idx"]), f64(raw["k_idx"]),
        f64(ws["w_q"]), f64(ws["w_k"]), f64(ws["w_qi"]), f64(ws["w_ki"]),
        f64(x["k_cache"]), f64(x["v_cache"]), f64(x["kidx_cache"]), table, lens)

    def within_step(got, want, what):
        off = np.abs(got - want)
        tol = bf16_step(want) * 1.0001 + 1e-5 * np.max(np.abs(want), axis=-1, keepdims=True)
        assert np.all(off <= tol), f"{what}: {int(np.sum(off > tol))} elements beyond one bf16 step"

    within_step(f64(q_out), oq, "q_out")
    within_step(f64(qi_out), oqi, "q_idx_out")
    touched = np.zeros(x["k_cache"].shape, dtype=bool)
    for b in range(B):
        p = int(lens[b]) - 1
        touched[int(table[b, p // 128]), :, p % 128] = True
    for n, want in (("k_cache", okc), ("kidx_cache", oic), ("v_cache", ovc)):
        got = f64(g[n])
        within_step(got[touched].reshape(-1, 128), want[touched].reshape(-1, 128), n)
        assert np.array_equal(got[~touched], f64(x[n])[~touched]), f"{n}: untouched bytes changed"
    # the decode step on the appended caches
    o, sel = m.msa_decode_step(q_out, qi_out, g["k_cache"], g["v_cache"], g["kidx_cache"],
                               g["block_table"], g["cache_lens"])
    m.msa_check_status()
    ro, rsel, rgap = O.decode_step(f64(q_out), f64(qi_out), f64(g["k_cache"]), f64(g["v_cache"]),
                                   f64(g["kidx_cache"]), table, lens, SCALE)
    gsel = sel.cpu().numpy()
    compare_selection(gsel, rsel, rgap, shape.name, (lens - 1) // 128,
                      SC.decode_scores_of(f64(qi_out), f64(g["kidx_cache"]), table, lens))
    same = np.all(np.all(gsel == rsel, axis=-1), axis=-1)
    assert_close(f64(o)[same], ro[same], 2e-2, 1e-2, "decode after append")


# ------------------------------------------------------------------ pipeline

def test_prefill_pipeline_tiny(m):
    """prologue -> select -> forward on the GPU against the oracle pipeline."""
    shape = W.config(0)
    cpu, gpu = inputs("tiny", shape)
    cu = gpu["cu_seqlens"]
    q, k, qi, ki = m.msa_qk_norm_rope4(gpu["q"], gpu["k"], gpu["q_idx"], gpu["k_idx"],
                                       gpu["w_q"], gpu["w_k"], gpu["w_qi"], gpu["w_ki"], cu)
    sel = m.msa_index_select(qi, ki, cu, shape.max_seqlen)
    o, lse = m.msa_sparse_attn_fwd(q, k, gpu["v"], sel, cu, shape.max_seqlen)
    m.msa_check_status()
    cun = cpu["cu_seqlens"].numpy()
    pq = O.qk_norm_rope(f64(cpu["q"]), f64(cpu["w_q"]), cun)
    pk = O.qk_norm_rope(f64(cpu["k"]), f64(cpu["w_k"]), cun)
    pqi = O.qk_norm_rope(f64(cpu["q_idx"]), f64(cpu["w_qi"]), cun)
    pki = O.qk_norm_rope(f64(cpu["k_idx"]), f64(cpu["w_ki"]), cun)
    osel, gap = O.index_select(pqi, pki, cun)
    gsel = sel.cpu().numpy()
    ndiff, nnear = compare_selection(gsel, osel, gap, "pipeline", own_blocks(cpu),
                                     SC.prefill_scores_of(pqi, pki, cun, np.arange(shape.T)))
    rows = np.nonzero(np.all(gsel == osel, axis=(1, 2)))[0]
    oo, olse = O.sparse_attn_fwd(pq, pk, f64(cpu["v"]), osel, cun, SCALE, tokens=rows)
    assert_close(f64(o)[rows], oo, 2e-2, 1e-2, "pipeline o")
    print(f"pipeline: {ndiff} rows select differently (all near-ties), {nnear} near-tie rows")
