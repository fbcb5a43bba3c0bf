"""Algorithmic work of each call, for roofline reporting.

Counts only the useful work of the method (the dense work that block sparsity
avoids is not counted, nor are padded or masked tensor-core lanes):
  forward  : 4 * D FLOPs per (query head, attended key)   (q.k and p.v)
  backward : 2.5 x the forward                           (S recompute, dP, dV, dQ, dK)
  select   : 2 * D FLOPs per (index head, causal key)     (dense causal indexer q.k)
  prologue : bytes = read + write of q, k, index-q, index-k (bf16)
  decode   : bytes = every cached index key of every head + the selected keys'
             K and V + q, index-q and o
A query at position p attends to 128 * (min(16, p // 128 + 1) - 1) + p % 128 + 1
keys: the full earlier selected blocks and its own block up to itself.
Narrow-block calls (4-token blocks, head dim 256) count the keys of the actual
selection: every listed block contributes its keys at positions <= p.
"""
from __future__ import annotations

import numpy as np

D = 128
BLOCK = 128
TOPK = 16


def _positions(seqlens):
    return np.concatenate([np.arange(int(L)) for L in seqlens if L > 0]) if len(seqlens) else \
        np.zeros(0, dtype=np.int64)


def attended_keys(seqlens) -> np.ndarray:
    pos = _positions(seqlens)
    nsel = np.minimum(TOPK, pos // BLOCK + 1)
    return BLOCK * (nsel - 1) + pos % BLOCK + 1


def prefill_work(seqlens, hq: int, hkv: int, hi: int) -> dict:
    pos = _positions(seqlens)
    keys = attended_keys(seqlens)
    T = int(len(pos))
    fwd = float(keys.sum()) * hq * 4 * D
    return {
        "tokens": T,
        "fwd_flops": fwd,
        "bwd_flops": 2.5 * fwd,
        "select_flops": float((pos + 1).sum()) * hi * 2 * D,
        "prologue_bytes": float(T) * D * 2 * 2 * (hq + hkv + 2 * hi),
    }


def decode_bytes(cache_lens, hq: int, hkv: int) -> float:
    total = 0.0
    for L in cache_lens:
        L = int(L)
        p = L - 1
        nsel = min(TOPK, p // BLOCK + 1)
        keys = BLOCK * (nsel - 1) + p % BLOCK + 1
        total += L * hkv * D * 2              # index keys, every head
        total += 2 * hkv * keys * D * 2       # selected K and V
        total += (hq + hkv + hq) * D * 2      # q, index-q, o
    return total


def qsa_work(seqlens, sel: np.ndarray, hq: int, block: int = 4, d: int = 256) -> dict:
    """Useful work of the narrow-block forward / backward for a selection
    sel [T, Hkv, topk] (block ids relative to the sequence start, -1 unused)."""
    pos = _positions(seqlens)
    T, hkv, _ = sel.shape
    b = sel.astype(np.int64)
    keys = np.clip(pos[:, None, None] - block * b + 1, 0, block)
    keys = np.where(b >= 0, keys, 0).sum(axis=2)            # [T, Hkv]
    fwd = float(keys.sum()) * (hq // hkv) * 4 * d
    return {"tokens": int(T), "attended_keys": float(keys.sum()), "fwd_flops": fwd,
            "bwd_flops": 2.5 * fwd}
