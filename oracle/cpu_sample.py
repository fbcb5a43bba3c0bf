"""Times the CPU oracle, as it stands, on bounded samples of a prefill workload.

TEST INFRASTRUCTURE: run only by the benchmark's CPU-baseline leg and by its
reference arm (`python -m oracle.cpu_sample ...` prints one JSON line).

Set-up (untimed) draws the pack and runs the oracle prologue over all of it,
since the sampled queries need every key of their sequence.  A timed sample
then takes n random query tokens and runs, for those tokens only, the
prologue of their q / k / index-q / index-k rows, index select, the forward
and the backward (dq and the tokens' dk/dv contributions); each stage's time
is scaled by T / n to a per-pack figure.  BLAS runs single-threaded (the
variables are set before numpy loads), so the figure is one host core's.
"""
import json
import os
import sys
import time

THREAD_VARS = ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS",
               "NUMEXPR_NUM_THREADS", "BLIS_NUM_THREADS")


class Sampler:
    def __init__(self, config_idx: int = 1, seed: int = 0):
        import math

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

    def sample(self, n_tokens: int, sample_seed: int) -> dict:
        np, O = self.np, self.O
        T = self.shape.T
        toks = np.sort(np.random.default_rng(sample_seed).choice(T, size=min(n_tokens, T),
                                                                 replace=False))
        t = {}
        t0 = time.perf_counter()
        for n, w in (("q", "w_q"), ("k", "w_k"), ("q_idx", "w_qi"), ("k_idx", "w_ki")):
            O.bf16_round(O.partial_rope(O.gemma_rmsnorm(self.raw[n][toks], self.raw[w]),
                                        self.pos[toks]))
        t["prologue_s"] = time.perf_counter() - t0
        t0 = time.perf_counter()
        sel_s, _ = O.index_select(self.qi, self.ki, self.cu, tokens=toks)
        t["select_s"] = time.perf_counter() - t0
        sel = np.full((T, self.shape.hkv, 16), -1, dtype=np.int64)
        sel[toks] = sel_s
        t0 = time.perf_counter()
        O.sparse_attn_fwd(self.q, self.k, self.v, sel, self.cu, self.scale, tokens=toks)
        t["fwd_s"] = time.perf_counter() - t0
        t0 = time.perf_counter()
        O.sparse_attn_bwd(self.q, self.k, self.v, self.do, sel, self.cu, self.scale,
                          only_tokens=toks)
        t["bwd_s"] = time.perf_counter() - t0
        frac = T / len(toks)
        ms = 1e3 * frac * sum(t.values())
        return {"ms_per_pack": ms, "sample_tokens": int(len(toks)), "tokens": T,
                "workload": self.shape.name, "threads": 1, **t}


if __name__ == "__main__":
    for var in THREAD_VARS:
        os.environ[var] = "1"
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import argparse

    ap = argparse.ArgumentParser()
    ap.add_argument("--config", type=int, default=1)
    ap.add_argument("--tokens", type=int, default=1024)
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--sample-seed", type=int, default=0)
    a = ap.parse_args()
    print(json.dumps(Sampler(a.config, a.seed).sample(a.tokens, a.sample_seed)))
