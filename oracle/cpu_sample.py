"""Times the CPU oracle, as it stands, on a prefill workload, and compares
outputs that the benchmark saved from the CUDA path with the oracle on
sampled rows.

TEST INFRASTRUCTURE: run only by the benchmark's CPU-baseline leg and by its
reference arm (`python -m oracle.cpu_sample ...` prints one JSON line).

Set-up (untimed) draws the pack on the CPU from its seed and runs the oracle
prologue over all of it, since any query needs every key of its sequence.
Timed work for a set of query tokens: the prologue of their q / k / index-q /
index-k rows, index select, the forward and the backward (dq and the tokens'
dk / dv contributions).  The oracle is not changed for this: a set of tokens
is dealt round-robin into equal chunks run by a pool of spawned worker processes, one per
host core used; each worker and the parent run BLAS on one thread (the
variables are set before numpy loads), so "cores" is the process count.
"""
import json
import math
import os
import sys
import time

THREAD_VARS = ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS",
               "NUMEXPR_NUM_THREADS", "BLIS_NUM_THREADS")
for _v in THREAD_VARS:
    os.environ[_v] = "1"
sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))


class Pack:
    """One seeded prefill pack and the oracle prologue over all of it."""

    def __init__(self, config_idx: int = 1, seed: int = 0):
        import numpy as np

        import workloads as W
        from oracle import msa_oracle as O

        self.np, self.O = np, O
        self.shape = W.config(config_idx, seed)
        x = W.make_prefill(self.shape, seed=seed, device="cpu", with_grad_out=True)
        f64 = lambda t: t.float().double().numpy()   # noqa: E731
        self.raw = {n: f64(x[n]) for n in ("q", "k", "q_idx", "k_idx", "w_q", "w_k", "w_qi",
                                            "w_ki")}
        self.v, self.do = f64(x["v"]), f64(x["do"])
        self.cu = x["cu_seqlens"].numpy()
        self.pos = O.positions(self.cu)
        self.q = O.qk_norm_rope(self.raw["q"], self.raw["w_q"], self.cu)
        self.k = O.qk_norm_rope(self.raw["k"], self.raw["w_k"], self.cu)
        self.qi = O.qk_norm_rope(self.raw["q_idx"], self.raw["w_qi"], self.cu)
        self.ki = O.qk_norm_rope(self.raw["k_idx"], self.raw["w_ki"], self.cu)
        self.scale = 1.0 / math.sqrt(128)

    def run(self, toks, keep: bool = False) -> dict:
        """The oracle on query tokens `toks`: per-stage seconds, and with keep
        the selection, gap, o, lse and dq of those tokens."""
        np, O = self.np, self.O
        T = self.shape.T
        t = {}
        t0 = time.perf_counter()
        for n, w in (("q", "w_q"), ("k", "w_k"), ("q_idx", "w_qi"), ("k_idx", "w_ki")):
            O.bf16_round(O.partial_rope(O.gemma_rmsnorm(self.raw[n][toks], self.raw[w]),
                                        self.pos[toks]))
        t["prologue_s"] = time.perf_counter() - t0
        t0 = time.perf_counter()
        sel_s, gap = O.index_select(self.qi, self.ki, self.cu, tokens=toks)
        t["select_s"] = time.perf_counter() - t0
        sel = np.full((T, self.shape.hkv, 16), -1, dtype=np.int64)
        sel[toks] = sel_s
        t0 = time.perf_counter()
        o, lse = O.sparse_attn_fwd(self.q, self.k, self.v, sel, self.cu, self.scale, tokens=toks)
        t["fwd_s"] = time.perf_counter() - t0
        t0 = time.perf_counter()
        dq, _, _ = O.sparse_attn_bwd(self.q, self.k, self.v, self.do, sel, self.cu, self.scale,
                                     only_tokens=toks)
        t["bwd_s"] = time.perf_counter() - t0
        if keep:
            t.update(sel=sel_s, gap=gap, o=o, lse=lse, dq=dq[toks])
        return t


# ------------------------------------------------------------------ worker pool

_PACK = None


def _init_worker(config_idx, seed):
    global _PACK
    _PACK = Pack(config_idx, seed)


def _run_chunk(toks):
    return _PACK.run(toks)


def make_pool(config_idx: int, seed: int, processes: int):
    import multiprocessing as mp
    return mp.get_context("spawn").Pool(processes, _init_worker, (config_idx, seed))


def pooled_seconds(pool, processes: int, toks) -> float:
    """Wall seconds for the pool to run the oracle on `toks`, dealt round-robin
    into one chunk per process (neighbouring tokens cost about the same)."""
    import numpy as np
    toks = np.asarray(toks)
    chunks = [toks[i::processes] for i in range(processes) if len(toks[i::processes])]
    t0 = time.perf_counter()
    pool.map(_run_chunk, chunks, chunksize=1)
    return time.perf_counter() - t0


def host_cores() -> int:
    return len(os.sched_getaffinity(0))


# ------------------------------------------------------------------ parity

def parity(path: str, pack: "Pack", kept: dict, toks) -> dict:
    """Compare the CUDA path's outputs saved in `path` with the oracle on
    sampled rows: selections by the near-tie rule (tests/selection_check.py),
    then o, lse and dq on the rows whose selection agrees."""
    import numpy as np

    import workloads as W
    from oracle import msa_oracle as O
    from tests import selection_check as SC

    z = np.load(path)
    out = {}
    # the timed pack: the whole step on the GPU (prologue, select, fwd, bwd)
    assert np.array_equal(z["cfg1_tokens"], toks)
    gsel = z["cfg1_sel"].astype(np.int64)
    own = pack.pos[toks] // 128
    rep = SC.check_selection(gsel, kept["sel"], kept["gap"], own,
                             SC.prefill_scores_of(pack.qi, pack.ki, pack.cu, toks),
                             "bench pack")
    same = np.all(np.all(gsel == kept["sel"], axis=-1), axis=-1)
    g_o, g_dq = z["cfg1_o"].astype(np.float64), z["cfg1_dq"].astype(np.float64)
    d_o = g_o[same] - kept["o"][same]
    d_dq = g_dq[same] - kept["dq"][same]
    rep.update(
        o_max_abs=float(np.abs(d_o).max()),
        o_rel_l2=float(np.linalg.norm(d_o) / np.linalg.norm(kept["o"][same])),
        lse_max_abs=float(np.abs(z["cfg1_lse"][same] - kept["lse"][same]).max()),
        dq_rel_l2=float(np.linalg.norm(d_dq) / np.linalg.norm(kept["dq"][same])))
    out[pack.shape.name] = rep
    # the other prefill workloads: selections after the GPU prologue
    for key, idx in (("cfg2", 2), ("cfg4", 4)):
        if f"{key}_tokens" not in z:
            continue
        shape = W.config(idx, int(z[f"{key}_seed"]))
        x = W.make_prefill(shape, seed=int(z[f"{key}_seed"]), device="cpu")
        cu = x["cu_seqlens"].numpy()
        f64 = lambda t: t.float().double().numpy()   # noqa: E731
        qi = O.qk_norm_rope(f64(x["q_idx"]), f64(x["w_qi"]), cu)
        ki = O.qk_norm_rope(f64(x["k_idx"]), f64(x["w_ki"]), cu)
        tk = z[f"{key}_tokens"]
        osel, gap = O.index_select(qi, ki, cu, tokens=tk)
        out[shape.name] = SC.check_selection(z[f"{key}_sel"], osel, gap,
                                             O.positions(cu)[tk] // 128,
                                             SC.prefill_scores_of(qi, ki, cu, tk), shape.name)
    # decode: sampled sequences, their pages copied out by the benchmark
    if "dec_q" in z:
        lens, table = z["dec_lens"], z["dec_table"]

        def from_bits(b):        # bf16 bit patterns -> their float32 values (exact)
            return (b.astype(np.uint16).astype(np.uint32) << 16).view(np.float32)

        kc, vc, ic = (from_bits(z[n]) for n in ("dec_k_bits", "dec_v_bits", "dec_kidx_bits"))
        ro, rsel, rgap = O.decode_step(z["dec_q"], z["dec_q_idx"], kc, vc, ic, table, lens,
                                       1.0 / math.sqrt(128))
        gsel = z["dec_sel"].astype(np.int64)
        rep = SC.check_selection(gsel, rsel, rgap, (lens - 1) // 128,
                                 SC.decode_scores_of(z["dec_q_idx"], ic, table, lens),
                                 "decode")
        same = np.all(np.all(gsel == rsel, axis=-1), axis=-1)
        d = z["dec_o"].astype(np.float64)[same] - ro[same]
        rep.update(o_max_abs=float(np.abs(d).max()) if d.size else None,
                   o_rel_l2=float(np.linalg.norm(d) / np.linalg.norm(ro[same])) if d.size else None)
        out[str(z["dec_name"])] = rep
    return out


# ------------------------------------------------------------------ modes

def baseline(config_idx: int, seed: int, n_tokens: int, sample_seed: int, parity_path=None):
    """CPU-baseline leg: the oracle on a random sample of query tokens, on one
    core and on every host core; ms per pack scaled by T / sample."""
    import numpy as np
    pack = Pack(config_idx, seed)
    T = pack.shape.T
    toks = np.sort(np.random.default_rng(sample_seed).choice(T, size=min(n_tokens, T),
                                                             replace=False))
    one = pack.run(toks, keep=parity_path is not None)
    one_s = sum(one[k] for k in ("prologue_s", "select_s", "fwd_s", "bwd_s"))
    cores = host_cores()
    pool = make_pool(config_idx, seed, cores)
    try:
        pooled_seconds(pool, cores, toks[:cores])          # workers warm (imports, set-up)
        all_s = pooled_seconds(pool, cores, toks)
    finally:
        pool.close()
        pool.join()
    res = {"workload": pack.shape.name, "tokens": T, "sample_tokens": int(len(toks)),
           "ms_per_pack": 1e3 * all_s * T / len(toks), "cores": cores,
           "ms_per_pack_1core": 1e3 * one_s * T / len(toks),
           **{k: one[k] for k in ("prologue_s", "select_s", "fwd_s", "bwd_s")}}
    if parity_path:
        res["parity"] = parity(parity_path, pack, one, toks)
    return res


def reference(config_idx: int, seed: int, steps: int, warmup: int, budget_s: float = 150.0):
    """Reference arm: every step runs the oracle on the query tokens of the
    pack (prologue, select, forward, backward) over all host cores.  A step
    covers every token of the pack unless warmup + steps full packs would not
    fit in `budget_s` seconds (estimated from an evenly strided probe of the
    pack); then each step covers an evenly strided subset that fits, and its
    time is scaled to the pack by T / subset (the line says which)."""
    import numpy as np

    import workloads as W
    cores = host_cores()
    T = W.config(config_idx, seed).T
    pool = make_pool(config_idx, seed, cores)
    try:
        probe = np.linspace(0, T - 1, min(T, 32 * cores)).round().astype(np.int64)
        pooled_seconds(pool, cores, probe)                          # workers' set-up
        est = pooled_seconds(pool, cores, probe) * T / len(probe)   # one full pack
        n = T if est * (warmup + steps) <= budget_s else \
            max(cores, int(T * budget_s / (est * (warmup + steps))))
        toks = np.linspace(0, T - 1, n).round().astype(np.int64) if n < T else np.arange(T)
        per = []
        for i in range(warmup + steps):
            s = pooled_seconds(pool, cores, toks)
            if i >= warmup:
                per.append(s)
    finally:
        pool.close()
        pool.join()
    step_s = sum(per) / len(per)
    return {"ms_per_pack": 1e3 * step_s * T / n, "ms_per_step": 1e3 * step_s, "cores": cores,
            "tokens": T, "tokens_per_step": int(n), "scaled": n < T, "steps": steps,
            "warmup": warmup}


if __name__ == "__main__":
    import argparse

    ap = argparse.ArgumentParser()
    ap.add_argument("--mode", choices=["baseline", "reference"], default="baseline")
    ap.add_argument("--config", type=int, default=1)
    ap.add_argument("--tokens", type=int, default=2048)
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--sample-seed", type=int, default=0)
    ap.add_argument("--parity", default=None, help=".npz of CUDA-path outputs to compare")
    ap.add_argument("--steps", type=int, default=3)
    ap.add_argument("--warmup", type=int, default=1)
    ap.add_argument("--budget-s", type=float, default=150.0)
    a = ap.parse_args()
    if a.mode == "baseline":
        r = baseline(a.config, a.seed, a.tokens, a.sample_seed, a.parity)
    else:
        r = reference(a.config, a.seed, a.steps, a.warmup, a.budget_s)
    print(json.dumps(r))
