"""Host-side checks of the C ABI: the library loads, exports every symbol the
header declares, and rejects bad arguments before launching anything.  No GPU
is needed: every call here fails validation on the host."""
import ctypes
import os
import re

import pytest

from msa_block_sparse_gb300 import api
from msa_block_sparse_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "msa.h")


@pytest.fixture(scope="module")
def lib():
    B.build()
    return api.lib()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"MSA_API\s+[\w\s\*]+?\b(msa_\w+)\s*\(", text)))


def test_header_declares_the_five_calls():
    names = declared_functions()
    for call in ("msa_qk_norm_rope", "msa_index_select", "msa_sparse_attn_fwd",
                 "msa_sparse_attn_bwd", "msa_decode_step", "msa_trace_begin", "msa_trace_end"):
        assert call in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in api._SIGNATURES, f"binding lacks {name}"
    assert lib.msa_abi_version() == 1


def test_workspace_sizes_are_host_only(lib):
    assert lib.msa_index_select_workspace_size(16384, 4, 1, 8192) > 0
    small = lib.msa_sparse_attn_bwd_workspace_size(4096, 1, 16, 1, 4096)
    big = lib.msa_sparse_attn_bwd_workspace_size(32768, 4, 64, 4, 12288)
    # the fp32 dQ accumulator dominates: T * Hq * 128 * 4 bytes
    assert big >= 32768 * 64 * 128 * 4 and small < big
    assert lib.msa_decode_step_workspace_size(64, 64, 4, 256) >= 64 * 4 * 256 * 4
    assert lib.msa_sparse_attn_fwd_workspace_size(0, 1, 16, 1, 1) == 0
    assert lib.msa_qk_norm_rope_bwd_workspace_size(16384, 16) >= 16384 // 16 * 128 * 4
    assert lib.msa_qk_norm_rope_bwd_workspace_size(0, 16) == 0


FAKE = ctypes.c_void_p(1 << 20)   # 16-byte aligned, never dereferenced: validation fails first


def _err(lib):
    return lib.msa_last_error().decode()


def test_null_and_misaligned_pointers_are_rejected(lib):
    rc = lib.msa_qk_norm_rope(None, FAKE, 10, 1, FAKE, FAKE, 1, 64, 1e7, 1e-6, None)
    assert rc == 1 and "x" in _err(lib)
    rc = lib.msa_qk_norm_rope(ctypes.c_void_p((1 << 20) + 2), FAKE, 10, 1, FAKE, FAKE, 1, 64, 1e7,
                              1e-6, None)
    assert rc == 1


def test_unsupported_shapes_are_rejected(lib):
    rc = lib.msa_qk_norm_rope(FAKE, FAKE, 10, 1, FAKE, FAKE, 1, 32, 1e7, 1e-6, None)
    assert rc == 2 and "rope_dim" in _err(lib)
    rc = lib.msa_index_select(FAKE, FAKE, FAKE, 1, 100, 1, 100, 8, FAKE, FAKE, 1 << 20, None)
    assert rc == 2 and "topk" in _err(lib)
    rc = lib.msa_sparse_attn_fwd(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 100, 12, 5, 100, 0.1, FAKE,
                                 FAKE, FAKE, 1 << 20, None)
    assert rc == 1 and "multiple" in _err(lib)
    rc = lib.msa_sparse_attn_fwd(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 100, 48, 1, 100, 0.1, FAKE,
                                 FAKE, FAKE, 1 << 20, None)
    assert rc == 2   # Hq/Hkv = 48 does not divide 128
    rc = lib.msa_sparse_attn_fwd(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 100, 16, 1, 100, 0.1, FAKE,
                                 FAKE, FAKE, 0, None)
    assert rc == 1 and "workspace" in _err(lib)
    rc = lib.msa_sparse_attn_fwd(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 100, 16, 1, 200, 0.1, FAKE,
                                 FAKE, FAKE, 1 << 20, None)
    assert rc == 1 and "max_seqlen" in _err(lib)
    rc = lib.msa_decode_step(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 64, 4, 10, 8, 0.1,
                             FAKE, None, FAKE, 0, None)
    assert rc == 1 and "workspace" in _err(lib)
    rc = lib.msa_decode_step(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 32, 4, 10, 8, 0.1,
                             FAKE, None, FAKE, 1 << 30, None)
    assert rc == 2 and "16" in _err(lib)


def test_training_forward_and_head_limits_are_checked_on_the_host(lib):
    # the training forward needs a backward workspace of the backward's size
    rc = lib.msa_sparse_attn_fwd_train(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 100, 16, 1, 100, 0.1,
                                       FAKE, FAKE, FAKE, 1 << 20, None, 1 << 30, None)
    assert rc == 1 and "bwd_workspace" in _err(lib)
    need = lib.msa_sparse_attn_bwd_workspace_size(100, 1, 16, 1, 100)
    rc = lib.msa_sparse_attn_fwd_train(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 100, 16, 1, 100, 0.1,
                                       FAKE, FAKE, FAKE, 1 << 20, FAKE, need - 1, None)
    assert rc == 1 and "workspace" in _err(lib)
    # the prologue kernels take at most 256 heads per tensor
    rc = lib.msa_qk_norm_rope(FAKE, FAKE, 10, 257, FAKE, FAKE, 1, 64, 1e7, 1e-6, None)
    assert rc == 2 and "256" in _err(lib)
    rc = lib.msa_qk_norm_rope_bwd(FAKE, FAKE, FAKE, FAKE, 10, 257, FAKE, FAKE, 1, 64, 1e7, 1e-6,
                                  FAKE, 1 << 30, None)
    assert rc == 2 and "256" in _err(lib)


def test_python_binding_refuses_cpu_tensors():
    import torch
    x = torch.zeros(4, 1, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        api.msa_qk_norm_rope(x, torch.zeros(128, dtype=torch.bfloat16),
                             torch.tensor([0, 4], dtype=torch.int32))


def test_trace_without_gpu_work_is_empty(lib):
    assert lib.msa_trace_begin() == 0
    buf = ctypes.create_string_buffer(256)
    assert lib.msa_trace_end(buf, 256) == 0
    assert buf.value == b"{}"
