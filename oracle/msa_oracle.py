"""Plain fp64 CPU oracle for MiniMax-M3 MSA block-sparse attention.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or run
this module: only the test-suite, the smoke check and the CPU-baseline leg of
the benchmark use it.  It shares no code with the CUDA library; it only reads
the seeded tensors that the `workloads` module draws.

Sources (web pages, cited by title and section):
  [M31]  "MiniMax-M3.1-Flash" (miles docs), "1. Model Introduction": a 4-head
         indexer (dim 128, own gemma q/k norm and RoPE) scores every causal
         128-token block by its maximum logit; each query attends to the 16 best
         blocks, its own block always included; index head h selects the blocks
         of KV head h.  GQA with 64 query / 4 KV heads of dim 128, per-head gemma
         q/k norm, RoPE on the first 64 dims with base 1e7.
  [M31q] same page, "5.4 Notable quirks": the indexer is frozen; the block
         selection receives no gradient.
  [M31p] same page, "5.1 Parallelism": the sparse attention runs on THD-packed
         sequences.
  [PR]   "[1/4] Add MiniMax-M3 support - #4581" (radixark/miles), "Kernel tuning":
         per-block max logits, then top-k; selections that differ do so only at
         near-ties; gradients agree to bf16 noise.
  [MB]   "MiniMax-M3" (Megatron-Bridge docs), "Architecture Notes": Gemma-style
         RMSNorm x*(1+w), per-head QK RMSNorm, partial RoPE (64 of 128 channels).
  [MBk]  same page, "Known Limitations": selection keeps 16 x 128 = 2048 key
         tokens, so full causal attention is identical up to that length.

Readings where the pages are silent (each is listed with its reason in the
design notes): RoPE pairs channel i with i+32 inside the rotated 64 channels
(rotate-half), inverse frequency base^(-2i/64); positions restart at 0 at each
sequence start of the pack; RMSNorm eps 1e-6, norm before RoPE, one [128]
weight per tensor shared by its heads; selected block ids are relative to the
sequence start, sorted ascending, padded with -1; equal scores prefer the lower
block id; query head i uses KV head i // (Hq/Hkv).

Every floating-point step runs in float64.  Values that the library stores as
bf16 (prologue outputs) are rounded to the bf16 grid with `bf16_round`, the
dtype of that boundary, so that both sides score the same stored keys.
"""
from __future__ import annotations

import math
from typing import Iterable, Optional

import numpy as np

BLOCK = 128
TOPK = 16
NEAR_TIE_REL = 1e-3


# --------------------------------------------------------------------------- bf16

def bf16_round(x) -> np.ndarray:
    """Round float64 values to the nearest bfloat16 value, ties to even.

    bf16 keeps 8 significant bits and float32's exponent range: for |x| in
    [2^(e-1), 2^e) the spacing is 2^(e-8); below the smallest normal 2^-126 the
    spacing stays 2^-133.  Dividing by a power of two is exact, so np.rint
    (round-half-even) on x/spacing is the rounding itself."""
    x = np.asarray(x, dtype=np.float64)
    _, e = np.frexp(x)
    e = np.maximum(e, -125)
    ulp = np.ldexp(1.0, e - 8)
    r = np.rint(x / ulp) * ulp
    big = np.abs(r) >= 2.0 ** 128
    if np.any(big):
        r = np.where(big, np.copysign(np.inf, x), r)
    return np.where(np.isfinite(x), r, x)


# --------------------------------------------------------------------------- prologue

def positions(cu_seqlens) -> np.ndarray:
    """Position of every packed token inside its own sequence [M31p]."""
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    T = int(cu[-1])
    pos = np.empty(T, dtype=np.int64)
    for s in range(len(cu) - 1):
        pos[cu[s]:cu[s + 1]] = np.arange(cu[s + 1] - cu[s])
    return pos


def gemma_rmsnorm(x: np.ndarray, w: np.ndarray, eps: float = 1e-6) -> np.ndarray:
    """Gemma-style RMSNorm over the last axis: x / sqrt(mean(x^2) + eps) * (1 + w) [MB]."""
    x = np.asarray(x, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    rms = np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
    return x / rms * (1.0 + w)


def rope_inv_freq(rope_dim: int = 64, base: float = 1.0e7) -> np.ndarray:
    i = np.arange(rope_dim // 2, dtype=np.float64)
    return base ** (-(2.0 * i) / rope_dim)


def partial_rope(x: np.ndarray, pos: np.ndarray, rope_dim: int = 64,
                 base: float = 1.0e7) -> np.ndarray:
    """Rotate the first `rope_dim` channels of x[t, ..., :] by position pos[t];
    channel i pairs with channel i + rope_dim/2; the rest pass through [M31, MB]."""
    x = np.asarray(x, dtype=np.float64)
    half = rope_dim // 2
    ang = np.asarray(pos, dtype=np.float64)[:, None] * rope_inv_freq(rope_dim, base)[None, :]
    shape = (x.shape[0],) + (1,) * (x.ndim - 2) + (half,)
    c = np.cos(ang).reshape(shape)
    s = np.sin(ang).reshape(shape)
    y = x.copy()
    x1 = x[..., :half]
    x2 = x[..., half:rope_dim]
    y[..., :half] = x1 * c - x2 * s
    y[..., half:rope_dim] = x2 * c + x1 * s
    return y


def qk_norm_rope(x, w, cu_seqlens, eps: float = 1e-6, rope_dim: int = 64,
                 base: float = 1.0e7, round_bf16: bool = True) -> np.ndarray:
    """Prologue for one tensor [T, H, 128]: per-head gemma norm, then partial RoPE
    at each token's in-sequence position; the result is stored as bf16."""
    y = partial_rope(gemma_rmsnorm(x, w, eps), positions(cu_seqlens), rope_dim, base)
    return bf16_round(y) if round_bf16 else y


def qk_norm_rope_bwd(x, w, dy, cu_seqlens, eps: float = 1e-6, rope_dim: int = 64,
                     base: float = 1.0e7):
    """Gradients of the prologue of one tensor [T, H, 128] (gemma norm, then
    partial RoPE [M31, MB]) for an upstream gradient dy = dL/dy.

    RoPE is a rotation, so dL/dz = R^T dy: the same pairs rotated by the
    negative angle.  With r = 1 / sqrt(mean(x^2) + eps), xh = x r and
    z = xh (1 + w):
        dL/dw = sum over tokens and heads of dz * xh                 [128]
        dL/dx = r (g - xh * mean(g * xh)),   g = dz (1 + w)          [T, H, 128]
    (the norm's own derivative: d xh_i / d x_k = r (delta_ik - xh_i xh_k / D)).
    Returns (dx, dw) in fp64."""
    x = np.asarray(x, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    dy = np.asarray(dy, dtype=np.float64)
    dz = partial_rope(dy, -positions(cu_seqlens).astype(np.float64), rope_dim, base)
    r = 1.0 / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
    xh = x * r
    dw = np.sum(dz * xh, axis=tuple(range(x.ndim - 1)))
    g = dz * (1.0 + w)
    dx = r * (g - xh * np.mean(g * xh, axis=-1, keepdims=True))
    return dx, dw


def decode_append(q, k, v, q_idx, k_idx, w_q, w_k, w_qi, w_ki, k_cache, v_cache,
                  kidx_cache, block_table, cache_lens, eps: float = 1e-6,
                  rope_dim: int = 64, base: float = 1.0e7):
    """Prologue of one new token per sequence, appended to a paged cache.

    Sequence b's new token sits at position p = cache_lens[b] - 1 (the length
    counts it).  Its q and index-q ([B, H, 128], pre-norm) get the prologue at
    p; its k and index-k get the same and, with v unchanged, are stored in slot
    p % 128 of page block_table[b, p // 128] ([page, head, slot, 128] caches).
    Returns (q_out, q_idx_out, k_cache, v_cache, kidx_cache) as new arrays, the
    prologue outputs rounded to bf16 like every stored value [M31, MB]."""
    lens = np.asarray(cache_lens, dtype=np.int64)
    pos = lens - 1

    def pro(x, w):
        return bf16_round(partial_rope(gemma_rmsnorm(x, w, eps), pos, rope_dim, base))

    q_out, qi_out = pro(q, w_q), pro(q_idx, w_qi)
    kn, kin = pro(k, w_k), pro(k_idx, w_ki)
    kc = np.array(k_cache, dtype=np.float64, copy=True)
    vc = np.array(v_cache, dtype=np.float64, copy=True)
    ic = np.array(kidx_cache, dtype=np.float64, copy=True)
    for b in range(len(lens)):
        page = int(block_table[b, pos[b] // BLOCK])
        slot = int(pos[b] % BLOCK)
        kc[page, :, slot] = kn[b]
        vc[page, :, slot] = np.asarray(v[b], dtype=np.float64)
        ic[page, :, slot] = kin[b]
    return q_out, qi_out, kc, vc, ic


# --------------------------------------------------------------------------- indexer

def block_scores_seq(qi: np.ndarray, ki: np.ndarray, rows: Optional[np.ndarray] = None,
                     block: int = BLOCK) -> np.ndarray:
    """Per-block max logit for one sequence and one index head [M31, PR].

    qi, ki: [L, D].  Returns [n, nb] with score[t, b] = max over keys j of block b
    with j <= t of qi[t] . ki[j]; blocks after the query's own block are -inf."""
    L = qi.shape[0]
    nb = (L + block - 1) // block
    rows = np.arange(L) if rows is None else np.asarray(rows)
    out = np.full((len(rows), nb), -np.inf)
    for c0 in range(0, len(rows), 1024):
        r = rows[c0:c0 + 1024]
        s = qi[r] @ ki.T
        s[np.arange(L)[None, :] > r[:, None]] = -np.inf
        for b in range(nb):
            out[c0:c0 + len(r), b] = s[:, b * block:(b + 1) * block].max(axis=1)
    return out


def select_from_scores(scores: np.ndarray, own: np.ndarray, topk: int = TOPK, n_init: int = 0):
    """Top-k blocks with the own block forced [M31]: own block plus the best
    min(topk-1, own) earlier blocks by score (equal scores: lower id first);
    output sorted ascending, padded with -1.

    With n_init > 0 the "init" rule named in [PR] (Kernel tuning) is applied as
    read here: the first n_init blocks of the sequence (those before the own
    block) are kept as well, and the best of the remaining earlier blocks fill
    the other topk - 1 - min(n_init, own) slots.

    Also returns, per row, the relative gap between the last kept and the first
    dropped scored block (inf when no scored block is dropped or none is kept),
    which the near-tie rule compares with 1e-3."""
    n = scores.shape[0]
    sel = np.full((n, topk), -1, dtype=np.int64)
    gap = np.full(n, np.inf)
    for r in range(n):
        o = int(own[r])
        ni = min(n_init, o)
        slots = topk - 1 - ni
        cand = np.arange(ni, o)
        order = cand[np.lexsort((cand, -scores[r, ni:o]))] if o > ni else cand
        keep = order[:max(slots, 0)]
        ids = np.sort(np.concatenate([np.arange(ni), keep, [o]]))
        sel[r, :len(ids)] = ids
        if slots > 0 and len(cand) > slots:
            a = scores[r, order[slots - 1]]
            b = scores[r, order[slots]]
            den = max(abs(a), abs(b))
            gap[r] = abs(a - b) / den if den > 0 else 0.0
    return sel, gap


def index_select(q_idx, k_idx, cu_seqlens, topk: int = TOPK,
                 tokens: Optional[Iterable[int]] = None, block: int = BLOCK, n_init: int = 0):
    """Block selection of every (token, index head) [M31, PR].

    q_idx, k_idx: [T, Hi, D] post-prologue values.  Returns sel [n, Hi, topk]
    (ids relative to the sequence start) and gap [n, Hi] for the requested
    tokens (all when None), in the order given.  n_init: see select_from_scores."""
    q_idx = np.asarray(q_idx, dtype=np.float64)
    k_idx = np.asarray(k_idx, dtype=np.float64)
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    T, Hi, _ = q_idx.shape
    toks = np.arange(T) if tokens is None else np.asarray(list(tokens), dtype=np.int64)
    seq_of = np.searchsorted(cu, toks, side="right") - 1
    sel = np.full((len(toks), Hi, topk), -1, dtype=np.int64)
    gap = np.full((len(toks), Hi), np.inf)
    for s in np.unique(seq_of):
        idx = np.nonzero(seq_of == s)[0]
        b0, b1 = cu[s], cu[s + 1]
        rows = toks[idx] - b0
        for h in range(Hi):
            sc = block_scores_seq(q_idx[b0:b1, h], k_idx[b0:b1, h], rows, block)
            ss, gg = select_from_scores(sc, rows // block, topk, n_init)
            sel[idx, h] = ss
            gap[idx, h] = gg
    return sel, gap


# --------------------------------------------------------------------------- attention

def _keys_of(sel_row: np.ndarray, p: int, block: int = BLOCK) -> np.ndarray:
    """In-sequence key positions a query at position p attends to: the union of
    its selected blocks, causally limited to keys <= p."""
    parts = [np.arange(b * block, min((b + 1) * block, p + 1)) for b in sel_row if b >= 0]
    return np.concatenate(parts) if parts else np.zeros(0, dtype=np.int64)


def sparse_attn_fwd(q, k, v, sel, cu_seqlens, scale: float,
                    tokens: Optional[Iterable[int]] = None, block: int = BLOCK):
    """Block-sparse GQA attention forward [M31, PR].

    q [T, Hq, D], k/v [T, Hkv, D], sel [T, Hkv, topk].  For query head i of token
    t (KV head g = i // (Hq/Hkv)): o = softmax(scale * q k_j) v_j over the keys j
    of the selected blocks with j <= t; lse = log(sum_j exp(scale * q k_j)).
    Returns o [n, Hq, D] and lse [n, Hq] for the requested tokens."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    T, Hq, D = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    toks = np.arange(T) if tokens is None else np.asarray(list(tokens), dtype=np.int64)
    o = np.zeros((len(toks), Hq, D))
    lse = np.zeros((len(toks), Hq))
    for n, t in enumerate(toks):
        s = int(np.searchsorted(cu, t, side="right") - 1)
        p = int(t - cu[s])
        for g in range(Hkv):
            J = cu[s] + _keys_of(sel[t, g], p, block)
            logits = scale * (q[t, g * G:(g + 1) * G] @ k[J, g].T)
            m = logits.max(axis=1, keepdims=True)
            e = np.exp(logits - m)
            l = e.sum(axis=1, keepdims=True)
            o[n, g * G:(g + 1) * G] = (e / l) @ v[J, g]
            lse[n, g * G:(g + 1) * G] = (m + np.log(l))[:, 0]
    return o, lse


def _row_grads(qt, do_t, kJ, vJ, scale):
    """Softmax-attention gradients of one token's G query rows over keys kJ/vJ."""
    logits = scale * (qt @ kJ.T)
    m = logits.max(axis=1, keepdims=True)
    e = np.exp(logits - m)
    P = e / e.sum(axis=1, keepdims=True)
    o = P @ vJ
    dP = do_t @ vJ.T
    delta = np.sum(do_t * o, axis=1, keepdims=True)
    dS = P * (dP - delta)
    return P, dS


def sparse_attn_bwd(q, k, v, do, sel, cu_seqlens, scale: float,
                    dq_tokens: Optional[Iterable[int]] = None,
                    dkv_blocks: Optional[Iterable[tuple]] = None, block: int = BLOCK,
                    only_tokens: Optional[Iterable[int]] = None):
    """Gradients of sum(o * do) w.r.t. q, k, v for the block-sparse attention;
    the selection is a constant (frozen indexer) [M31q, PR].

    With P = softmax(scale q k^T) over the selected causal keys and
    dP = do v^T:  dS = P * (dP - rowsum(dP * P)),  dq = scale dS k,
    dk = scale dS^T q,  dv = P^T do, the sums running over every query row that
    attends to the key.

    Full mode (both selectors None) returns dq [T,Hq,D], dk, dv [T,Hkv,D];
    with `only_tokens` it sums the contributions of those query tokens only.
    Sampled mode returns dq for `dq_tokens` and, for every (s, g, b) in
    `dkv_blocks`, dk/dv of the keys of block b of sequence s, KV head g."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    do = np.asarray(do, dtype=np.float64)
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    T, Hq, D = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    seq_of = np.searchsorted(cu, np.arange(T), side="right") - 1
    full = dq_tokens is None and dkv_blocks is None

    if full:
        dq = np.zeros_like(q)
        dk = np.zeros_like(k)
        dv = np.zeros_like(v)
        for t in (range(T) if only_tokens is None else only_tokens):
            s = int(seq_of[t])
            p = int(t - cu[s])
            for g in range(Hkv):
                J = cu[s] + _keys_of(sel[t, g], p, block)
                hs = slice(g * G, (g + 1) * G)
                P, dS = _row_grads(q[t, hs], do[t, hs], k[J, g], v[J, g], scale)
                dq[t, hs] = scale * dS @ k[J, g]
                dk[J, g] += scale * dS.T @ q[t, hs]
                dv[J, g] += P.T @ do[t, hs]
        return dq, dk, dv

    out = {}
    if dq_tokens is not None:
        toks = np.asarray(list(dq_tokens), dtype=np.int64)
        dq = np.zeros((len(toks), Hq, D))
        for n, t in enumerate(toks):
            s = int(seq_of[t])
            p = int(t - cu[s])
            for g in range(Hkv):
                J = cu[s] + _keys_of(sel[t, g], p, block)
                hs = slice(g * G, (g + 1) * G)
                _, dS = _row_grads(q[t, hs], do[t, hs], k[J, g], v[J, g], scale)
                dq[n, hs] = scale * dS @ k[J, g]
        out["dq"] = dq
    if dkv_blocks is not None:
        res = []
        for (s, g, b) in dkv_blocks:
            k0 = int(cu[s] + b * block)
            k1 = int(min(cu[s] + (b + 1) * block, cu[s + 1]))
            dkb = np.zeros((k1 - k0, D))
            dvb = np.zeros((k1 - k0, D))
            for t in range(k0, int(cu[s + 1])):
                if b not in sel[t, g]:
                    continue
                p = int(t - cu[s])
                J = cu[s] + _keys_of(sel[t, g], p, block)
                hs = slice(g * G, (g + 1) * G)
                P, dS = _row_grads(q[t, hs], do[t, hs], k[J, g], v[J, g], scale)
                inb = (J >= k0) & (J < k1)
                jj = J[inb] - k0
                dkb[jj] += scale * dS[:, inb].T @ q[t, hs]
                dvb[jj] += P[:, inb].T @ do[t, hs]
            res.append((dkb, dvb))
        out["dkv"] = res
    return out


# --------------------------------------------------------------------------- decode

def decode_step(q, q_idx, k_cache, v_cache, kidx_cache, block_table, cache_lens,
                scale: float, topk: int = TOPK, batch: Optional[Iterable[int]] = None,
                block: int = BLOCK, n_init: int = 0):
    """One decode step against a paged cache (page = one 128-token block,
    layout [page, head, token, dim]).

    For sequence b with cache length L (the new token sits at position L-1 and is
    already cached) and index head h: every block 0..(L-1)//128 is scored by its
    max logit q_idx[b,h] . kidx over its cached keys, the own block is forced and
    the best others fill it up to `topk` [M31]; the 16 query heads of KV head h
    then attend over the selected keys.  Returns o [n, Hq, D], sel [n, Hi, topk]
    and gap [n, Hi] for the requested batch rows (all when None).  n_init: see
    select_from_scores."""
    q = np.asarray(q, dtype=np.float64)
    q_idx = np.asarray(q_idx, dtype=np.float64)
    bt = np.asarray(block_table, dtype=np.int64)
    lens = np.asarray(cache_lens, dtype=np.int64)
    B, Hq, D = q.shape
    Hkv = k_cache.shape[1]
    Hi = q_idx.shape[1]
    G = Hq // Hkv
    rows = np.arange(B) if batch is None else np.asarray(list(batch), dtype=np.int64)
    o = np.zeros((len(rows), Hq, D))
    sel = np.full((len(rows), Hi, topk), -1, dtype=np.int64)
    gap = np.full((len(rows), Hi), np.inf)
    for n, b in enumerate(rows):
        L = int(lens[b])
        npg = (L + block - 1) // block
        pages = bt[b, :npg]
        kk = np.asarray(k_cache[pages], dtype=np.float64)       # [npg, Hkv, 128, D]
        vv = np.asarray(v_cache[pages], dtype=np.float64)
        ki = np.asarray(kidx_cache[pages], dtype=np.float64)    # [npg, Hi, 128, D]
        kk = kk.transpose(1, 0, 2, 3).reshape(Hkv, npg * block, D)[:, :L]
        vv = vv.transpose(1, 0, 2, 3).reshape(Hkv, npg * block, D)[:, :L]
        ki = ki.transpose(1, 0, 2, 3).reshape(Hi, npg * block, D)[:, :L]
        own = (L - 1) // block
        for h in range(Hi):
            logits = ki[h] @ q_idx[b, h]
            sc = np.array([logits[c * block:min((c + 1) * block, L)].max() for c in range(npg)])
            ss, gg = select_from_scores(sc[None, :], np.array([own]), topk, n_init)
            sel[n, h] = ss[0]
            gap[n, h] = gg[0]
        for g in range(Hkv):
            J = _keys_of(sel[n, g], L - 1, block)
            hs = slice(g * G, (g + 1) * G)
            lg = scale * (q[b, hs] @ kk[g, J].T)
            e = np.exp(lg - lg.max(axis=1, keepdims=True))
            o[n, hs] = (e / e.sum(axis=1, keepdims=True)) @ vv[g, J]
    return o, sel, gap
