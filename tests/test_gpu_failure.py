"""Failure detection on the GPU, without a fault.

Every wait in the library's kernels is bounded: when it runs out the kernel
sets a bit in the device status word and returns, and an index outside its
range is dropped with another bit set.  Here a diagnostic kernel waits on an
mbarrier that nothing completes, and a forward call gets selection ids beyond
the query's own block; both must come back through msa_check_status as errors,
leave the context usable, and (for the ids) drop only the bad entries."""
import math

import numpy as np
import pytest
import torch

import workloads as W
from oracle import msa_oracle as O

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
TIMEOUT, BOUNDS = 4, 5          # MSA_ERR_TIMEOUT, MSA_ERR_BOUNDS


@pytest.fixture(scope="module")
def m():
    import __graft_entry__ as ge
    ge.build()
    import msa_block_sparse_gb300 as mod
    return mod


def f64(t):
    return t.detach().float().cpu().double().numpy()


def test_bounded_wait_runs_out_and_is_reported(m):
    m.msa_check_status()                         # start from a clear status word
    m.msa_selftest_wait()
    with pytest.raises(m.MSAError) as err:
        m.msa_check_status()
    assert err.value.code == TIMEOUT and "site 65535" in str(err.value)
    m.msa_check_status()                         # read-and-clear: nothing left
    # the context still runs kernels correctly afterwards
    x = torch.randn((33, 2, 128), device=DEV).to(torch.bfloat16)
    w = (torch.randn(128, device=DEV) * 0.1).to(torch.bfloat16)
    cu = torch.tensor([0, 20, 33], dtype=torch.int32, device=DEV)
    y = m.msa_qk_norm_rope(x, w, cu)
    m.msa_check_status()
    want = O.qk_norm_rope(f64(x), f64(w), cu.cpu().numpy())
    assert np.max(np.abs(f64(y) - want)) < 0.05


def test_out_of_range_selection_is_reported_and_dropped(m):
    shape = W.PrefillShape("bounds-2seq", (700, 300), 16, 1, 1)
    x = W.make_prefill(shape, seed=3, device="cpu")
    cu = x["cu_seqlens"].numpy()
    sel, _ = O.index_select(f64(x["q_idx"]), f64(x["k_idx"]), cu)
    bad = sel.copy()
    t1, t2 = 650, 10                     # own blocks 5 and 0 of sequence 0
    bad[t1, 0, 6] = 7                    # beyond the own block (and the sequence)
    bad[t2, 0, 1] = 3
    gpu = {n: x[n].to(DEV) for n in ("q", "k", "v", "cu_seqlens")}
    m.msa_check_status()
    o, lse = m.msa_sparse_attn_fwd(gpu["q"], gpu["k"], gpu["v"],
                                   torch.from_numpy(bad.astype(np.int32)).to(DEV),
                                   gpu["cu_seqlens"], shape.max_seqlen)
    with pytest.raises(m.MSAError) as err:
        m.msa_check_status()
    assert err.value.code == BOUNDS
    scale = 1.0 / math.sqrt(128)
    rows = [t1, t2, 0, 699, 700, 999]
    want, _ = O.sparse_attn_fwd(f64(x["q"]), f64(x["k"]), f64(x["v"]), sel, cu, scale,
                                tokens=rows)
    got = f64(o)[rows]
    assert np.max(np.abs(got - want)) < 2e-2
    m.msa_check_status()
