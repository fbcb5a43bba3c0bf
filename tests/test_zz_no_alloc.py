"""msa_decode_step_static: the decode step for callers that cannot allocate
device memory (a serving engine that fixes its GPU memory pool at start-up,
or a plugin that only receives the tensors it computes on).  It keeps its
scratch in a fixed array inside the library instead of a caller workspace.

Called here through the C ABI (ctypes) and compared with msa_decode_step on
the same inputs, twice in a row, so that the second call also shows that the
first call's leftovers in the shared array do no harm.  The file is named to
be collected last."""
import ctypes
import math

import numpy as np
import pytest
import torch

import workloads as W
from oracle import msa_oracle as O
from tests import selection_check as SC

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m():
    import __graft_entry__ as ge
    ge.build()
    import msa_block_sparse_gb300 as mod
    return mod


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _static_call(m, x, o, sel):
    B, Hq = x["q"].shape[0], x["q"].shape[1]
    P, Hkv = x["k_cache"].shape[0], x["k_cache"].shape[1]
    maxp = x["block_table"].shape[1]
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return m.lib().msa_decode_step_static(
        _p(x["q"]), _p(x["q_idx"]), _p(x["k_cache"]), _p(x["v_cache"]), _p(x["kidx_cache"]),
        _p(x["block_table"]), _p(x["cache_lens"]), B, Hq, Hkv, P, maxp, 1.0 / math.sqrt(128),
        _p(o), _p(sel), stream)


def _check_close(got, want):
    g = got.float().cpu().double().numpy()
    w = want.float().cpu().double().numpy()
    err = float(np.max(np.abs(g - w)))
    rel = float(np.linalg.norm(g - w) / np.linalg.norm(w))
    assert err <= 2e-2 and rel <= 1e-2, (err, rel)


@pytest.mark.parametrize("shape", [
    W.DecodeShape("no-alloc-small", (1, 129, 2049, 5000, 300), 32, 2, 2),
    W.config(3),
], ids=["small", "b64"])
def test_static_decode_matches_workspace_decode_twice(m, shape):
    x = {k: v.to("cuda:0") for k, v in W.make_decode(shape, seed=7, device="cuda:0").items()}
    ref_o, ref_sel = m.msa_decode_step(x["q"], x["q_idx"], x["k_cache"], x["v_cache"],
                                       x["kidx_cache"], x["block_table"], x["cache_lens"])
    torch.cuda.synchronize()
    for _ in range(2):
        o = torch.full_like(ref_o, float("nan"))
        sel = torch.full_like(ref_sel, -7)
        rc = _static_call(m, x, o, sel)
        assert rc == 0, m.lib().msa_last_error().decode()
        m.msa_check_status()
        assert torch.equal(sel, ref_sel)
        _check_close(o, ref_o)
    if shape.B <= 8:
        # and against the oracle directly: selections by the near-tie rule,
        # o on the rows whose selection agrees
        f64 = lambda t: t.float().cpu().double().numpy()    # noqa: E731
        lens = x["cache_lens"].cpu().numpy()
        table = x["block_table"].cpu().numpy()
        ro, rsel, rgap = O.decode_step(f64(x["q"]), f64(x["q_idx"]), f64(x["k_cache"]),
                                       f64(x["v_cache"]), f64(x["kidx_cache"]), table, lens,
                                       1.0 / math.sqrt(128))
        gsel = sel.cpu().numpy()
        SC.check_selection(gsel, rsel, rgap, (lens - 1) // 128,
                           SC.decode_scores_of(f64(x["q_idx"]), f64(x["kidx_cache"]), table, lens),
                           "static decode")
        same = np.all(np.all(gsel == rsel, axis=-1), axis=-1)
        assert same.any()
        g = f64(o)[same]
        err = float(np.max(np.abs(g - ro[same])))
        rel = float(np.linalg.norm(g - ro[same]) / np.linalg.norm(ro[same]))
        assert err <= 2e-2 and rel <= 1e-2, (err, rel)


def test_static_decode_rejects_sizes_beyond_its_scratch(m):
    shape = W.DecodeShape("no-alloc-too-big", tuple([200] * 65), 64, 4, 4)   # B * Hkv = 260
    x = {k: v.to("cuda:0") for k, v in W.make_decode(shape, seed=1, device="cuda:0").items()}
    o = torch.empty_like(x["q"])
    sel = torch.empty((shape.B, 4, 16), dtype=torch.int32, device="cuda:0")
    rc = _static_call(m, x, o, sel)
    assert rc == 2 and "B * Hkv <= 256" in m.lib().msa_last_error().decode()
