"""Seeded synthetic inputs for MSA block-sparse attention.

This module is shared by the CUDA path's tests/benchmark and by the CPU oracle.
It holds no arithmetic of the method itself: it only draws random tensors,
sequence lengths and page tables with the shapes and value distributions of the
workloads the MiniMax-M3 pages describe.

Workload recipe (one line per knob):
  * q, k, v, index-q, index-k are drawn N(0, 1) and stored as bf16.
  * Every 128-token key block of every sequence gets one offset vector per index
    head, drawn N(0, 0.5^2), which is added to the pre-norm index keys of all
    tokens of that block, so that block scores separate.
  * Gemma norm weights (q, k, index-q, index-k, one [128] vector each) are drawn
    N(0, 0.1^2) and stored as bf16.
  * The upstream gradient dO is N(0, 1) bf16.
  * Decode caches hold post-prologue values N(0, 1) bf16; the index-key cache
    gets the same per-block offsets; pages are placed in a seeded random
    permutation so that the block table is not the identity.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

D = 128          # head dim (MiniMax-M3.1-Flash, "1. Model Introduction")
BLOCK = 128      # key block size of the indexer
TOPK = 16        # blocks kept per query
ROPE_DIM = 64    # rotated channels
ROPE_BASE = 1.0e7
EPS = 1.0e-6
SCALE = 1.0 / math.sqrt(D)


@dataclasses.dataclass(frozen=True)
class PrefillShape:
    name: str
    seqlens: tuple
    hq: int
    hkv: int
    hi: int
    runs_bwd: bool = False

    @property
    def T(self) -> int:
        return int(sum(self.seqlens))

    @property
    def S(self) -> int:
        return len(self.seqlens)

    @property
    def max_seqlen(self) -> int:
        return int(max(self.seqlens))

    def cu_seqlens(self) -> torch.Tensor:
        cu = [0]
        for L in self.seqlens:
            cu.append(cu[-1] + int(L))
        return torch.tensor(cu, dtype=torch.int32)


@dataclasses.dataclass(frozen=True)
class DecodeShape:
    name: str
    cache_lens: tuple
    hq: int
    hkv: int
    hi: int

    @property
    def B(self) -> int:
        return len(self.cache_lens)


# ---------------------------------------------------------------- sequence lengths

def seqlens_composition(seed: int, total_blocks: int = 128, parts: int = 4,
                        min_blocks: int = 8) -> tuple:
    """A uniform random composition of `total_blocks` 128-token blocks into
    `parts` sequences of at least `min_blocks` blocks each (16,384-token pack of
    4 sequences, each a multiple of 128 and at least 1024 tokens)."""
    rng = np.random.default_rng(seed)
    free = total_blocks - parts * min_blocks
    cuts = np.sort(rng.choice(free + parts - 1, size=parts - 1, replace=False))
    bounds = np.concatenate([[-1], cuts, [free + parts - 1]])
    extra = np.diff(bounds) - 1
    return tuple(int((min_blocks + e) * BLOCK) for e in extra)


def seqlens_uniform_pack(seed: int, total: int = 16384, n: int = 8,
                         lo: int = 512, hi: int = 4096) -> tuple:
    """`n` lengths uniform in [lo, hi], rounded to 128, summing to `total`.

    Eight draws from [512, 4096] average ~18.4k tokens, more than the 16,384-token
    pack holds, so the first n-1 are drawn and the last takes the remainder; the
    draw repeats (same generator) until the remainder also lies in [lo, hi]."""
    rng = np.random.default_rng(seed)
    while True:
        first = rng.integers(lo, hi + 1, size=n - 1)
        first = np.clip(np.rint(first / BLOCK).astype(np.int64) * BLOCK, lo, hi)
        last = total - int(first.sum())
        if lo <= last <= hi:
            return tuple(int(x) for x in first) + (int(last),)


def decode_lens(seed: int, batch: int = 64, lo: int = 8192, hi: int = 32768) -> tuple:
    rng = np.random.default_rng(seed)
    return tuple(int(x) for x in rng.integers(lo, hi + 1, size=batch))


# ---------------------------------------------------------------- the five workloads

def config(idx: int, seed: int = 0):
    """The five workloads: 0 tiny single sequence, 1 one KV group on a 16k pack,
    2 full layer shape on a 16k pack, 3 paged decode, 4 training on a 32k pack."""
    if idx == 0:
        return PrefillShape("tiny-2560-16q1kv", (2560,), 16, 1, 1)
    if idx == 1:
        return PrefillShape("pack16k-4seq-16q1kv", seqlens_composition(seed), 16, 1, 1,
                            runs_bwd=True)
    if idx == 2:
        return PrefillShape("pack16k-8seq-64q4kv", seqlens_uniform_pack(seed), 64, 4, 4)
    if idx == 3:
        return DecodeShape("decode-b64-64q4kv", decode_lens(seed), 64, 4, 4)
    if idx == 4:
        return PrefillShape("pack32k-4seq-64q4kv", (4096, 8192, 8192, 12288), 64, 4, 4,
                            runs_bwd=True)
    raise ValueError(idx)


# ---------------------------------------------------------------- tensors

def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _normal_bf16(shape, g, device, std: float = 1.0) -> torch.Tensor:
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(torch.bfloat16)


def make_prefill(shape: PrefillShape, seed: int = 0, device="cpu",
                 with_grad_out: Optional[bool] = None) -> dict:
    """Pre-norm q, k, v, index-q, index-k (bf16), the four norm weights, cu_seqlens
    and (for training shapes) the upstream gradient dO."""
    device = torch.device(device)
    g = _gen(seed, device)
    T, hq, hkv, hi = shape.T, shape.hq, shape.hkv, shape.hi
    out = {}
    out["q"] = _normal_bf16((T, hq, D), g, device)
    out["k"] = _normal_bf16((T, hkv, D), g, device)
    out["v"] = _normal_bf16((T, hkv, D), g, device)
    out["q_idx"] = _normal_bf16((T, hi, D), g, device)
    kidx = torch.randn((T, hi, D), generator=g, device=device, dtype=torch.float32)
    # one offset vector per (sequence, 128-token block, index head)
    cu = shape.cu_seqlens().tolist()
    for s in range(shape.S):
        L = cu[s + 1] - cu[s]
        nb = (L + BLOCK - 1) // BLOCK
        off = torch.randn((nb, hi, D), generator=g, device=device, dtype=torch.float32) * 0.5
        per_tok = off.repeat_interleave(BLOCK, dim=0)[:L]
        kidx[cu[s]:cu[s + 1]] += per_tok
    out["k_idx"] = kidx.to(torch.bfloat16)
    for name in ("w_q", "w_k", "w_qi", "w_ki"):
        out[name] = _normal_bf16((D,), g, device, std=0.1)
    out["cu_seqlens"] = shape.cu_seqlens().to(device)
    if with_grad_out is None:
        with_grad_out = shape.runs_bwd
    if with_grad_out:
        out["do"] = _normal_bf16((T, hq, D), g, device)
    return out


def make_decode(shape: DecodeShape, seed: int = 0, device="cpu") -> dict:
    """A paged cache (page = one 128-token block; layout [page, kv head, token, dim])
    plus one new post-prologue query token per sequence. cache_lens include the new
    token, whose key/value are already in the cache."""
    device = torch.device(device)
    g = _gen(seed, device)
    B, hq, hkv, hi = shape.B, shape.hq, shape.hkv, shape.hi
    lens = list(shape.cache_lens)
    npages = [(L + BLOCK - 1) // BLOCK for L in lens]
    P = int(sum(npages))
    maxpages = int(max(npages))
    perm = torch.randperm(P, generator=g, device=device).to(torch.int32)
    table = torch.full((B, maxpages), -1, dtype=torch.int32, device=device)
    pos = 0
    for b in range(B):
        table[b, :npages[b]] = perm[pos:pos + npages[b]]
        pos += npages[b]
    out = {
        "q": _normal_bf16((B, hq, D), g, device),
        "q_idx": _normal_bf16((B, hi, D), g, device),
        "k_cache": _normal_bf16((P, hkv, BLOCK, D), g, device),
        "v_cache": _normal_bf16((P, hkv, BLOCK, D), g, device),
    }
    kidx = torch.randn((P, hi, BLOCK, D), generator=g, device=device, dtype=torch.float32)
    kidx += torch.randn((P, hi, 1, D), generator=g, device=device, dtype=torch.float32) * 0.5
    out["kidx_cache"] = kidx.to(torch.bfloat16)
    out["block_table"] = table
    out["cache_lens"] = torch.tensor(lens, dtype=torch.int32, device=device)
    return out


# ---------------------------------------------------------------- narrow-block variant
# The pages' second block-sparse workload ("[1/4] Add MiniMax-M3 support - #4581",
# Kernel tuning): qwen3.8-next's QSA layers with 12 query heads per KV head, head
# dim 256 and 4-token key blocks, timed fwd+bwd on 16k-token packs.  The pages
# give no selection rule for it; the synthetic selection keeps each query's own
# block plus distinct earlier blocks drawn uniformly at random, up to 512 blocks
# (2048 keys, the key budget of the MiniMax layers' 16 x 128).

QSA_D = 256
QSA_BLOCK = 4
QSA_GROUP = 12
QSA_TOPK = 512


@dataclasses.dataclass(frozen=True)
class QsaShape:
    name: str
    seqlens: tuple
    hq: int
    hkv: int
    topk: int

    @property
    def T(self) -> int:
        return int(sum(self.seqlens))

    @property
    def S(self) -> int:
        return len(self.seqlens)

    @property
    def max_seqlen(self) -> int:
        return int(max(self.seqlens))

    def cu_seqlens(self) -> torch.Tensor:
        cu = [0]
        for L in self.seqlens:
            cu.append(cu[-1] + int(L))
        return torch.tensor(cu, dtype=torch.int32)


def qsa_config(idx: int, seed: int = 0) -> QsaShape:
    """0: a ragged 4-sequence pack (an empty-ish 1-token sequence, lengths not
    multiples of the block), top-64, so rows past 256 tokens are sparse;
    1: the 16,384-token pack of the pages' timing (4 sequences, the same length
    draw as the MiniMax pack), top-512; 2: two KV heads (24 q / 2 kv), top-128."""
    if idx == 0:
        return QsaShape("qsa-ragged-12q1kv", (300, 37, 1, 702), 12, 1, 64)
    if idx == 1:
        return QsaShape("qsa-pack16k-4seq-12q1kv", seqlens_composition(seed), 12, 1, QSA_TOPK)
    if idx == 2:
        return QsaShape("qsa-2kv-24q2kv", (1500, 777), 24, 2, 128)
    raise ValueError(idx)


def qsa_selection(seqlens, hkv: int, topk: int, g: torch.Generator, device) -> torch.Tensor:
    """sel [T, hkv, topk] int32: for a token at position p, its own block p // 4
    plus min(topk, p // 4 + 1) - 1 distinct earlier blocks drawn uniformly,
    ascending, padded with -1.  Block ids are relative to the sequence start."""
    device = torch.device(device)
    T = int(sum(seqlens))
    sel = torch.full((T, hkv, topk), -1, dtype=torch.int32, device=device)
    t0 = 0
    for L in seqlens:
        L = int(L)
        nb = (L + QSA_BLOCK - 1) // QSA_BLOCK
        kk = min(topk, nb)
        cols = torch.arange(nb, device=device)
        for a in range(0, L, 1024):
            b = min(L, a + 1024)
            own = (torch.arange(a, b, device=device) // QSA_BLOCK)[:, None]
            for h in range(hkv):
                r = torch.rand((b - a, nb), generator=g, device=device)
                r = torch.where(cols[None] > own, torch.full_like(r, -1.0), r)
                r = torch.where(cols[None] == own, torch.full_like(r, 2.0), r)
                vals, idx = r.topk(kk, dim=1)
                idx = torch.where(vals < 0, torch.full_like(idx, nb), idx)
                idx, _ = idx.sort(dim=1)
                idx = torch.where(idx >= nb, torch.full_like(idx, -1), idx)
                sel[t0 + a:t0 + b, h, :kk] = idx.to(torch.int32)
        t0 += L
    return sel


def make_qsa(shape: QsaShape, seed: int = 0, device="cpu", with_grad_out: bool = True) -> dict:
    """q [T, hq, 256], k and v [T, hkv, 256] bf16 N(0, 1) (the attention inputs; the
    pages name no prologue for this variant), the selection, cu_seqlens and dO."""
    device = torch.device(device)
    g = _gen(seed, device)
    T, hq, hkv = shape.T, shape.hq, shape.hkv
    out = {
        "q": _normal_bf16((T, hq, QSA_D), g, device),
        "k": _normal_bf16((T, hkv, QSA_D), g, device),
        "v": _normal_bf16((T, hkv, QSA_D), g, device),
    }
    out["sel"] = qsa_selection(shape.seqlens, hkv, shape.topk, g, device)
    out["cu_seqlens"] = shape.cu_seqlens().to(device)
    if with_grad_out:
        out["do"] = _normal_bf16((T, hq, QSA_D), g, device)
    return out
