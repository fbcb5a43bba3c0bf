"""GPU parity of the narrow-block variant (4-token blocks, head dim 256, 12 query
heads per KV head; "[1/4] Add MiniMax-M3 support - #4581", Kernel tuning)
against the fp64 oracle run with block=4, on the same seeded inputs and the same
selection.  Small packs (ragged tails, a 1-token sequence, two KV heads) compare
every element; the 16k pack compares sampled rows and key blocks.  Tolerances as
for the 128-token kernels: o max-abs 2e-2 and rel-L2 1e-2, lse max-abs 1e-3,
gradients rel-L2 1e-2."""
import math

import numpy as np
import pytest
import torch

import workloads as W
from oracle import msa_oracle as O

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
SCALE = 1.0 / math.sqrt(W.QSA_D)


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


_CACHE = {}


def inputs(idx, seed=0):
    key = (idx, seed)
    if key not in _CACHE:
        shape = W.qsa_config(idx, seed)
        cpu = W.make_qsa(shape, seed=seed, device="cpu")
        gpu = {k: v.to(DEV) for k, v in cpu.items()}
        _CACHE[key] = (shape, cpu, gpu)
    return _CACHE[key]


def run(m, shape, gpu):
    cu = gpu["cu_seqlens"]
    o, lse = m.msa_qsa_attn_fwd(gpu["q"], gpu["k"], gpu["v"], gpu["sel"], cu, shape.max_seqlen)
    dq, dk, dv = m.msa_qsa_attn_bwd(gpu["q"], gpu["k"], gpu["v"], o, gpu["do"], lse, gpu["sel"],
                                    cu, shape.max_seqlen)
    m.msa_check_status()
    return o, lse, dq, dk, dv


@pytest.mark.parametrize("idx", [0, 2])
def test_qsa_small_matches_oracle(m, idx):
    shape, cpu, gpu = inputs(idx)
    o, lse, dq, dk, dv = run(m, shape, gpu)
    sel = cpu["sel"].numpy()
    cu = cpu["cu_seqlens"].numpy()
    q, k, v, do = (f64(cpu[n]) for n in ("q", "k", "v", "do"))
    oo, olse = O.sparse_attn_fwd(q, k, v, sel, cu, SCALE, block=W.QSA_BLOCK)
    assert_close(f64(o), oo, 2e-2, 1e-2, f"{shape.name} o")
    assert_close(lse.cpu().numpy().astype(np.float64), olse, 1e-3, 1e-4, f"{shape.name} lse")
    rq, rk, rv = O.sparse_attn_bwd(q, k, v, do, sel, cu, SCALE, block=W.QSA_BLOCK)
    for got, want, n in ((dq, rq, "dq"), (dk, rk, "dk"), (dv, rv, "dv")):
        r = rel_l2(f64(got), want)
        assert r <= 1e-2, f"{shape.name} {n}: rel-L2 {r:.3e}"
    # a second call gives the same bits for the forward and dq (no reductions there)
    o2, lse2, dq2, _, _ = run(m, shape, gpu)
    assert torch.equal(o, o2) and torch.equal(lse, lse2) and torch.equal(dq, dq2)


def test_qsa_pack16k_sampled(m):
    shape, cpu, gpu = inputs(1)
    o, lse, dq, dk, dv = run(m, shape, gpu)
    sel = cpu["sel"].numpy()
    cu = cpu["cu_seqlens"].numpy()
    q, k, v, do = (f64(cpu[n]) for n in ("q", "k", "v", "do"))
    rng = np.random.default_rng(5)
    toks = sorted(set(rng.integers(0, shape.T, 40).tolist())
                  | {0, int(cu[1]) - 1, int(cu[1]), shape.T - 1})
    oo, olse = O.sparse_attn_fwd(q, k, v, sel, cu, SCALE, tokens=toks, block=W.QSA_BLOCK)
    assert_close(f64(o[toks]), oo, 2e-2, 1e-2, "pack16k o")
    assert_close(lse[toks].cpu().numpy().astype(np.float64), olse, 1e-3, 1e-4, "pack16k lse")
    last = shape.S - 1
    nb_last = (shape.seqlens[last] + 3) // 4
    short = int(np.argmin(shape.seqlens))
    blocks = [(last, 0, nb_last - 1), (last, 0, nb_last - 40), (short, 0, shape.seqlens[short] // 8)]
    ref = O.sparse_attn_bwd(q, k, v, do, sel, cu, SCALE, dq_tokens=toks[:16], dkv_blocks=blocks,
                            block=W.QSA_BLOCK)
    r = rel_l2(f64(dq[toks[:16]]), ref["dq"])
    assert r <= 1e-2, f"pack16k dq rel-L2 {r:.3e}"
    for (s, g, b), (rk, rv) in zip(blocks, ref["dkv"]):
        k0 = int(cu[s]) + 4 * b
        n = rk.shape[0]
        rk_ = rel_l2(f64(dk[k0:k0 + n, g]), rk)
        rv_ = rel_l2(f64(dv[k0:k0 + n, g]), rv)
        assert rk_ <= 1e-2 and rv_ <= 1e-2, f"block {(s, g, b)}: dk {rk_:.3e} dv {rv_:.3e}"


def test_qsa_long_sequence_sampled(m):
    """A 12,001-token sequence: 1201 query tiles of 10 tokens, more than the
    plan kernel scans in one pass (1024 entries per pass), beside a 5-token
    and a 300-token one; o and lse on sampled rows, dq on a few."""
    shape = W.QsaShape("qsa-long-12q1kv", (12001, 5, 300), 12, 1, 64)
    cpu = W.make_qsa(shape, seed=3, device="cpu")
    gpu = {k: v.to(DEV) for k, v in cpu.items()}
    o, lse, dq, dk, dv = run(m, shape, gpu)
    sel = cpu["sel"].numpy()
    cu = cpu["cu_seqlens"].numpy()
    q, k, v, do = (f64(cpu[n]) for n in ("q", "k", "v", "do"))
    rng = np.random.default_rng(11)
    toks = sorted(set(rng.integers(0, shape.T, 24).tolist())
                  | {0, 10239, 10240, 11999, 12000, 12001, 12005, shape.T - 1})
    oo, olse = O.sparse_attn_fwd(q, k, v, sel, cu, SCALE, tokens=toks, block=W.QSA_BLOCK)
    assert_close(f64(o[toks]), oo, 2e-2, 1e-2, "long o")
    assert_close(lse[toks].cpu().numpy().astype(np.float64), olse, 1e-3, 1e-4, "long lse")
    ref = O.sparse_attn_bwd(q, k, v, do, sel, cu, SCALE, dq_tokens=toks[:8], dkv_blocks=[],
                            block=W.QSA_BLOCK)
    r = rel_l2(f64(dq[toks[:8]]), ref["dq"])
    assert r <= 1e-2, f"long dq rel-L2 {r:.3e}"


def test_qsa_rejects_bad_shapes(m):
    shape, cpu, gpu = inputs(0)
    q12 = gpu["q"][:, :11].contiguous()
    with pytest.raises(m.MSAError):
        m.msa_qsa_attn_fwd(q12, gpu["k"], gpu["v"], gpu["sel"], gpu["cu_seqlens"], shape.max_seqlen)
    with pytest.raises(m.MSAError):
        m.msa_qsa_attn_fwd(gpu["q"], gpu["k"], gpu["v"], gpu["sel"], gpu["cu_seqlens"], 40000)
