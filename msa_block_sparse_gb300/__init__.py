"""MiniMax-M3 MSA block-sparse attention for one NVIDIA GB300 (sm_103a).

The compute lives in libmsa.so (hand-written CUDA kernels behind a C ABI,
include/msa.h); this package holds its build script and a thin ctypes binding
whose functions carry the C names."""
from .api import (  # noqa: F401
    LIB_PATH,
    MSAError,
    lib,
    msa_check_status,
    msa_selftest_wait,
    msa_decode_append,
    msa_decode_step,
    msa_index_select,
    msa_qk_norm_rope,
    msa_qk_norm_rope4,
    msa_qk_norm_rope_bwd,
    msa_sparse_attn_bwd,
    msa_sparse_attn_bwd_prepare,
    msa_qsa_attn_fwd,
    msa_qsa_attn_bwd,
    msa_sparse_attn_fwd,
    msa_trace_begin,
    msa_trace_end,
    workspace_bytes,
)
