"""Python binding of libmsa.so (ctypes).  Argument marshalling only: every step
of the computation runs in the library's CUDA kernels.  Function names match
the C ABI in include/msa.h; tensors are torch CUDA tensors in the layouts that
header states, outputs and workspaces are allocated here with torch when the
caller does not pass them, and the work is enqueued on the current stream.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmsa.so")

D = 128
TOPK = 16

_c_int, _c_float, _c_size, _vp = ctypes.c_int, ctypes.c_float, ctypes.c_size_t, ctypes.c_void_p

# name -> (restype, argtypes); mirrors include/msa.h
_SIGNATURES = {
    "msa_abi_version": (_c_int, []),
    "msa_last_error": (ctypes.c_char_p, []),
    "msa_check_status": (_c_int, [_vp]),
    "msa_selftest_wait": (_c_int, [_vp]),
    "msa_trace_begin": (_c_int, []),
    "msa_trace_end": (_c_int, [ctypes.c_char_p, _c_size]),
    "msa_qk_norm_rope": (_c_int, [_vp, _vp, _c_int, _c_int, _vp, _vp, _c_int, _c_int, _c_float,
                                  _c_float, _vp]),
    "msa_qk_norm_rope4": (_c_int, [_vp, _vp, _c_int, _vp, _vp, _c_int, _vp, _vp, _vp, _vp,
                                   _c_int, _vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int,
                                   _c_float, _c_float, _vp]),
    "msa_qk_norm_rope_bwd_workspace_size": (_c_size, [_c_int, _c_int]),
    "msa_qk_norm_rope_bwd": (_c_int, [_vp, _vp, _vp, _vp, _c_int, _c_int, _vp, _vp, _c_int,
                                      _c_int, _c_float, _c_float, _vp, _c_size, _vp]),
    "msa_decode_append": (_c_int, [_vp] * 14 + [_c_int] * 6 + [_c_float, _c_float, _vp, _vp, _vp]),
    "msa_index_select_workspace_size": (_c_size, [_c_int, _c_int, _c_int, _c_int]),
    "msa_index_select": (_c_int, [_vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int, _c_int, _vp,
                                  _vp, _c_size, _vp]),
    "msa_index_select_ex": (_c_int, [_vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int, _c_int,
                                     _c_int, _vp, _vp, _c_size, _vp]),
    "msa_sparse_attn_fwd_workspace_size": (_c_size, [_c_int, _c_int, _c_int, _c_int, _c_int]),
    "msa_sparse_attn_fwd": (_c_int, [_vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int,
                                     _c_int, _c_float, _vp, _vp, _vp, _c_size, _vp]),
    "msa_sparse_attn_fwd_train": (_c_int, [_vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int,
                                           _c_int, _c_float, _vp, _vp, _vp, _c_size, _vp, _c_size,
                                           _vp]),
    "msa_sparse_attn_bwd_workspace_size": (_c_size, [_c_int, _c_int, _c_int, _c_int, _c_int]),
    "msa_sparse_attn_bwd": (_c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _c_int, _c_int,
                                     _c_int, _c_int, _c_int, _c_float, _vp, _vp, _vp, _vp,
                                     _c_size, _vp]),
    "msa_sparse_attn_bwd_prepare": (_c_int, [_c_int, _c_int, _c_int, _c_int, _c_int, _vp, _c_size,
                                             _vp]),
    "msa_sparse_attn_bwd_prepared": (_c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _c_int,
                                              _c_int, _c_int, _c_int, _c_int, _c_float, _vp, _vp,
                                              _vp, _vp, _c_size, _vp]),
    "msa_qsa_attn_fwd_workspace_size": (_c_size, [_c_int, _c_int, _c_int, _c_int, _c_int]),
    "msa_qsa_attn_fwd": (_c_int, [_vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int,
                                  _c_int, _c_int, _c_float, _vp, _vp, _vp, _c_size, _vp]),
    "msa_qsa_attn_bwd_workspace_size": (_c_size, [_c_int, _c_int, _c_int, _c_int, _c_int]),
    "msa_qsa_attn_bwd": (_c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _c_int, _c_int,
                                  _c_int, _c_int, _c_int, _c_int, _c_float, _vp, _vp, _vp, _vp,
                                  _c_size, _vp]),
    "msa_decode_step_workspace_size": (_c_size, [_c_int, _c_int, _c_int, _c_int]),
    "msa_decode_step": (_c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int,
                                 _c_int, _c_int, _c_float, _vp, _vp, _vp, _c_size, _vp]),
    "msa_decode_step_ex": (_c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int,
                                    _c_int, _c_int, _c_float, _c_int, _vp, _vp, _vp, _c_size,
                                    _vp]),
    "msa_decode_step_static": (_c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _c_int, _c_int,
                                        _c_int, _c_int, _c_int, _c_float, _vp, _vp, _vp]),
}

STATUS = {0: "MSA_OK", 1: "MSA_ERR_INVALID_ARG", 2: "MSA_ERR_UNSUPPORTED", 3: "MSA_ERR_CUDA",
          4: "MSA_ERR_TIMEOUT", 5: "MSA_ERR_BOUNDS"}

_lib = None


class MSAError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{STATUS.get(code, code)}: {msg}")
        self.code = code


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built (there is no fallback)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        l = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(l, name)
            fn.restype = res
            fn.argtypes = args
        _lib = l
    return _lib


def _check(code: int):
    if code != 0:
        raise MSAError(code, lib().msa_last_error().decode())


def _stream(t: torch.Tensor):
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _ptr(t: Optional[torch.Tensor]):
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _req(t: torch.Tensor, name: str, dtype, shape=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def _workspace(size: int, device, ws: Optional[torch.Tensor]):
    if ws is not None:
        if ws.numel() * ws.element_size() < size:
            raise ValueError(f"workspace needs {size} bytes")
        return ws
    return torch.empty(max(size, 256), dtype=torch.uint8, device=device)


def msa_check_status(device=None) -> None:
    """Synchronizes the current stream and raises if a kernel reported a timeout
    or an out-of-range index since the last check."""
    s = torch.cuda.current_stream(device).cuda_stream
    _check(lib().msa_check_status(ctypes.c_void_p(s)))


# ------------------------------------------------------------------ prologue

def msa_selftest_wait(device=None) -> None:
    """Launch the diagnostic kernel whose bounded wait runs out (~2 s); the next
    msa_check_status raises MSAError (timeout)."""
    s = torch.cuda.current_stream(device).cuda_stream
    _check(lib().msa_selftest_wait(ctypes.c_void_p(s)))


def msa_trace_begin() -> None:
    """Start recording CUDA-event timings around every library kernel launch."""
    _check(lib().msa_trace_begin())


def msa_trace_end() -> dict:
    """Stop recording; {kernel: {"launches": n, "ms": total}} since msa_trace_begin."""
    buf = ctypes.create_string_buffer(1 << 16)
    _check(lib().msa_trace_end(buf, len(buf)))
    import json
    return json.loads(buf.value.decode())


def msa_qk_norm_rope(x, w, cu_seqlens, out: Optional[torch.Tensor] = None, rope_dim: int = 64,
                     rope_base: float = 1.0e7, eps: float = 1.0e-6):
    """x bf16 [T, H, 128] -> out (default: a new tensor; pass out=x for in place):
    gemma RMSNorm with weight w (bf16 [128]) then partial RoPE at each token's
    position in its sequence."""
    T, H = x.shape[0], x.shape[1]
    _req(x, "x", torch.bfloat16, (T, H, D))
    _req(w, "w", torch.bfloat16, (D,))
    _req(cu_seqlens, "cu_seqlens", torch.int32)
    out = torch.empty_like(x) if out is None else out
    _req(out, "out", torch.bfloat16, (T, H, D))
    S = cu_seqlens.numel() - 1
    _check(lib().msa_qk_norm_rope(_ptr(x), _ptr(out), T, H, _ptr(w), _ptr(cu_seqlens), S,
                                  rope_dim, rope_base, eps, _stream(x)))
    return out


def msa_qk_norm_rope_bwd(x, dy, w, cu_seqlens, dx: Optional[torch.Tensor] = None,
                         dw: Optional[torch.Tensor] = None, rope_dim: int = 64,
                         rope_base: float = 1.0e7, eps: float = 1.0e-6,
                         workspace: Optional[torch.Tensor] = None):
    """Gradients of msa_qk_norm_rope: (dx bf16 [T, H, 128], dw fp32 [128]) from
    the prologue input x and dy = dL/dy (pass dx=dy to overwrite dy)."""
    T, H = x.shape[0], x.shape[1]
    _req(x, "x", torch.bfloat16, (T, H, D))
    _req(dy, "dy", torch.bfloat16, (T, H, D))
    _req(w, "w", torch.bfloat16, (D,))
    _req(cu_seqlens, "cu_seqlens", torch.int32)
    dx = torch.empty_like(x) if dx is None else dx
    _req(dx, "dx", torch.bfloat16, (T, H, D))
    dw = torch.empty(D, dtype=torch.float32, device=x.device) if dw is None else dw
    _req(dw, "dw", torch.float32, (D,))
    S = cu_seqlens.numel() - 1
    size = lib().msa_qk_norm_rope_bwd_workspace_size(T, H)
    ws = _workspace(size, x.device, workspace)
    _check(lib().msa_qk_norm_rope_bwd(_ptr(x), _ptr(dy), _ptr(dx), _ptr(dw), T, H, _ptr(w),
                                      _ptr(cu_seqlens), S, rope_dim, rope_base, eps, _ptr(ws),
                                      ws.numel(), _stream(x)))
    return dx, dw


def msa_qk_norm_rope4(q, k, q_idx, k_idx, w_q, w_k, w_qi, w_ki, cu_seqlens, outs=None,
                      rope_dim: int = 64, rope_base: float = 1.0e7, eps: float = 1.0e-6):
    """The prologue of q, k, index-q and index-k in one launch.  `outs` is a
    4-tuple of output tensors (default: new tensors; pass the inputs for in place)."""
    T = q.shape[0]
    Hq, Hkv, Hi = q.shape[1], k.shape[1], q_idx.shape[1]
    _req(q, "q", torch.bfloat16, (T, Hq, D))
    _req(k, "k", torch.bfloat16, (T, Hkv, D))
    _req(q_idx, "q_idx", torch.bfloat16, (T, Hi, D))
    _req(k_idx, "k_idx", torch.bfloat16, (T, Hi, D))
    for n, w in (("w_q", w_q), ("w_k", w_k), ("w_qi", w_qi), ("w_ki", w_ki)):
        _req(w, n, torch.bfloat16, (D,))
    _req(cu_seqlens, "cu_seqlens", torch.int32)
    if outs is None:
        outs = tuple(torch.empty_like(t) for t in (q, k, q_idx, k_idx))
    for o_, t, n in zip(outs, (q, k, q_idx, k_idx), ("q_out", "k_out", "q_idx_out", "k_idx_out")):
        _req(o_, n, torch.bfloat16, tuple(t.shape))
    S = cu_seqlens.numel() - 1
    _check(lib().msa_qk_norm_rope4(_ptr(q), _ptr(outs[0]), Hq, _ptr(k), _ptr(outs[1]), Hkv,
                                   _ptr(q_idx), _ptr(outs[2]), _ptr(k_idx), _ptr(outs[3]), Hi,
                                   _ptr(w_q), _ptr(w_k), _ptr(w_qi), _ptr(w_ki),
                                   _ptr(cu_seqlens), S, T, rope_dim, rope_base, eps,
                                   _stream(q)))
    return tuple(outs)


# ------------------------------------------------------------------ index select

def msa_index_select(q_idx, k_idx, cu_seqlens, max_seqlen: int, topk: int = TOPK,
                     out: Optional[torch.Tensor] = None,
                     workspace: Optional[torch.Tensor] = None, n_init: int = 0) -> torch.Tensor:
    """Selected blocks int32 [T, Hi, 16] (ascending, -1 padded).  n_init > 0 applies
    the init rule (msa_index_select_ex: the first n_init blocks are always kept)."""
    T, Hi = q_idx.shape[0], q_idx.shape[1]
    _req(q_idx, "q_idx", torch.bfloat16, (T, Hi, D))
    _req(k_idx, "k_idx", torch.bfloat16, (T, Hi, D))
    _req(cu_seqlens, "cu_seqlens", torch.int32)
    S = cu_seqlens.numel() - 1
    if out is None:
        out = torch.empty((T, Hi, topk), dtype=torch.int32, device=q_idx.device)
    _req(out, "out", torch.int32, (T, Hi, topk))
    size = lib().msa_index_select_workspace_size(T, S, Hi, max_seqlen)
    ws = _workspace(size, q_idx.device, workspace)
    if n_init:
        _check(lib().msa_index_select_ex(_ptr(q_idx), _ptr(k_idx), _ptr(cu_seqlens), S, T, Hi,
                                         max_seqlen, topk, n_init, _ptr(out), _ptr(ws),
                                         ws.numel(), _stream(q_idx)))
    else:
        _check(lib().msa_index_select(_ptr(q_idx), _ptr(k_idx), _ptr(cu_seqlens), S, T, Hi,
                                      max_seqlen, topk, _ptr(out), _ptr(ws), ws.numel(),
                                      _stream(q_idx)))
    return out


# ------------------------------------------------------------------ attention

def msa_sparse_attn_fwd(q, k, v, sel, cu_seqlens, max_seqlen: int, scale: Optional[float] = None,
                        out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                        workspace: Optional[torch.Tensor] = None,
                        bwd_workspace: Optional[torch.Tensor] = None):
    """Block-sparse attention forward: (o bf16 [T, Hq, 128], lse fp32 [T, Hq]).
    With bwd_workspace (msa_sparse_attn_fwd_train): that backward workspace's
    accumulators are zeroed while the forward runs, for a following
    msa_sparse_attn_bwd(..., workspace=bwd_workspace, prepared=True)."""
    T, Hq, Hkv = q.shape[0], q.shape[1], k.shape[1]
    _req(q, "q", torch.bfloat16, (T, Hq, D))
    _req(k, "k", torch.bfloat16, (T, Hkv, D))
    _req(v, "v", torch.bfloat16, (T, Hkv, D))
    _req(sel, "sel", torch.int32, (T, Hkv, TOPK))
    _req(cu_seqlens, "cu_seqlens", torch.int32)
    S = cu_seqlens.numel() - 1
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((T, Hq), dtype=torch.float32, device=q.device) if lse is None else lse
    _req(out, "out", torch.bfloat16, (T, Hq, D))
    _req(lse, "lse", torch.float32, (T, Hq))
    size = lib().msa_sparse_attn_fwd_workspace_size(T, S, Hq, Hkv, max_seqlen)
    ws = _workspace(size, q.device, workspace)
    if bwd_workspace is None:
        _check(lib().msa_sparse_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(sel), _ptr(cu_seqlens),
                                         S, T, Hq, Hkv, max_seqlen, scale, _ptr(out), _ptr(lse),
                                         _ptr(ws), ws.numel(), _stream(q)))
    else:
        bsize = lib().msa_sparse_attn_bwd_workspace_size(T, S, Hq, Hkv, max_seqlen)
        bws = _workspace(bsize, q.device, bwd_workspace)
        _check(lib().msa_sparse_attn_fwd_train(_ptr(q), _ptr(k), _ptr(v), _ptr(sel),
                                               _ptr(cu_seqlens), S, T, Hq, Hkv, max_seqlen, scale,
                                               _ptr(out), _ptr(lse), _ptr(ws), ws.numel(),
                                               _ptr(bws), bws.numel(), _stream(q)))
    return out, lse


def msa_sparse_attn_bwd_prepare(q, k, cu_seqlens, max_seqlen: int, workspace: torch.Tensor,
                                stream: Optional[torch.cuda.Stream] = None):
    """Clears the fp32 accumulators of `workspace` for one following
    msa_sparse_attn_bwd(..., prepared=True) of the same shapes (q [T, Hq, 128],
    k [T, Hkv, 128]), on `stream` (default: the current stream); the caller
    orders the two (an event when the streams differ)."""
    T, Hq, Hkv = q.shape[0], q.shape[1], k.shape[1]
    S = cu_seqlens.numel() - 1
    size = lib().msa_sparse_attn_bwd_workspace_size(T, S, Hq, Hkv, max_seqlen)
    ws = _workspace(size, q.device, workspace)
    st = ctypes.c_void_p((stream or torch.cuda.current_stream(q.device)).cuda_stream)
    _check(lib().msa_sparse_attn_bwd_prepare(T, S, Hq, Hkv, max_seqlen, _ptr(ws), ws.numel(), st))


def msa_sparse_attn_bwd(q, k, v, o, dout, lse, sel, cu_seqlens, max_seqlen: int,
                        scale: Optional[float] = None, dq=None, dk=None, dv=None,
                        workspace: Optional[torch.Tensor] = None, prepared: bool = False):
    """Block-sparse attention backward: (dq, dk, dv) in bf16.  prepared=True:
    `workspace` was cleared by msa_sparse_attn_bwd_prepare for this call."""
    T, Hq, Hkv = q.shape[0], q.shape[1], k.shape[1]
    _req(q, "q", torch.bfloat16, (T, Hq, D))
    _req(k, "k", torch.bfloat16, (T, Hkv, D))
    _req(v, "v", torch.bfloat16, (T, Hkv, D))
    _req(o, "o", torch.bfloat16, (T, Hq, D))
    _req(dout, "dout", torch.bfloat16, (T, Hq, D))
    _req(lse, "lse", torch.float32, (T, Hq))
    _req(sel, "sel", torch.int32, (T, Hkv, TOPK))
    _req(cu_seqlens, "cu_seqlens", torch.int32)
    S = cu_seqlens.numel() - 1
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    size = lib().msa_sparse_attn_bwd_workspace_size(T, S, Hq, Hkv, max_seqlen)
    if prepared and workspace is None:
        raise ValueError("prepared=True needs the workspace that msa_sparse_attn_bwd_prepare cleared")
    ws = _workspace(size, q.device, workspace)
    call = lib().msa_sparse_attn_bwd_prepared if prepared else lib().msa_sparse_attn_bwd
    _check(call(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _ptr(sel),
                _ptr(cu_seqlens), S, T, Hq, Hkv, max_seqlen, scale, _ptr(dq), _ptr(dk), _ptr(dv),
                _ptr(ws), ws.numel(), _stream(q)))
    return dq, dk, dv


# ------------------------------------------------------------------ decode

def msa_decode_append(q, q_idx, k, v, k_idx, w_q, w_qi, w_k, w_ki, k_cache, v_cache,
                      kidx_cache, block_table, cache_lens, q_out=None, q_idx_out=None,
                      rope_dim: int = 64, rope_base: float = 1.0e7, eps: float = 1.0e-6):
    """Prologue of one new token per sequence (position cache_lens - 1), its k,
    index-k and v written into the paged caches in place; returns (q_out,
    q_idx_out) for msa_decode_step (pass q / q_idx to update them in place)."""
    B, Hq = q.shape[0], q.shape[1]
    P, Hkv = k_cache.shape[0], k_cache.shape[1]
    maxp = block_table.shape[1]
    _req(q, "q", torch.bfloat16, (B, Hq, D))
    for n, t in (("q_idx", q_idx), ("k", k), ("v", v), ("k_idx", k_idx)):
        _req(t, n, torch.bfloat16, (B, Hkv, D))
    for n, w in (("w_q", w_q), ("w_qi", w_qi), ("w_k", w_k), ("w_ki", w_ki)):
        _req(w, n, torch.bfloat16, (D,))
    for n, c in (("k_cache", k_cache), ("v_cache", v_cache), ("kidx_cache", kidx_cache)):
        _req(c, n, torch.bfloat16, (P, Hkv, 128, D))
    _req(block_table, "block_table", torch.int32, (B, maxp))
    _req(cache_lens, "cache_lens", torch.int32, (B,))
    q_out = torch.empty_like(q) if q_out is None else q_out
    q_idx_out = torch.empty_like(q_idx) if q_idx_out is None else q_idx_out
    _check(lib().msa_decode_append(_ptr(q), _ptr(q_idx), _ptr(k), _ptr(v), _ptr(k_idx),
                                   _ptr(w_q), _ptr(w_qi), _ptr(w_k), _ptr(w_ki), _ptr(k_cache),
                                   _ptr(v_cache), _ptr(kidx_cache), _ptr(block_table),
                                   _ptr(cache_lens), B, Hq, Hkv, P, maxp, rope_dim, rope_base, eps,
                                   _ptr(q_out), _ptr(q_idx_out), _stream(q)))
    return q_out, q_idx_out


def msa_decode_step(q, q_idx, k_cache, v_cache, kidx_cache, block_table, cache_lens,
                    scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
                    sel_out: Optional[torch.Tensor] = None,
                    workspace: Optional[torch.Tensor] = None, n_init: int = 0):
    """One decode step: (o bf16 [B, Hq, 128], sel int32 [B, Hkv, 16]).  n_init > 0
    applies the init rule (msa_decode_step_ex)."""
    B, Hq = q.shape[0], q.shape[1]
    P, Hkv = k_cache.shape[0], k_cache.shape[1]
    maxp = block_table.shape[1]
    _req(q, "q", torch.bfloat16, (B, Hq, D))
    _req(q_idx, "q_idx", torch.bfloat16, (B, Hkv, D))
    for n, c in (("k_cache", k_cache), ("v_cache", v_cache), ("kidx_cache", kidx_cache)):
        _req(c, n, torch.bfloat16, (P, Hkv, 128, D))
    _req(block_table, "block_table", torch.int32, (B, maxp))
    _req(cache_lens, "cache_lens", torch.int32, (B,))
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    out = torch.empty_like(q) if out is None else out
    if sel_out is None:
        sel_out = torch.empty((B, Hkv, TOPK), dtype=torch.int32, device=q.device)
    size = lib().msa_decode_step_workspace_size(B, Hq, Hkv, maxp)
    ws = _workspace(size, q.device, workspace)
    if n_init:
        _check(lib().msa_decode_step_ex(_ptr(q), _ptr(q_idx), _ptr(k_cache), _ptr(v_cache),
                                        _ptr(kidx_cache), _ptr(block_table), _ptr(cache_lens), B,
                                        Hq, Hkv, P, maxp, scale, n_init, _ptr(out),
                                        _ptr(sel_out), _ptr(ws), ws.numel(), _stream(q)))
    else:
        _check(lib().msa_decode_step(_ptr(q), _ptr(q_idx), _ptr(k_cache), _ptr(v_cache),
                                     _ptr(kidx_cache), _ptr(block_table), _ptr(cache_lens), B,
                                     Hq, Hkv, P, maxp, scale, _ptr(out), _ptr(sel_out),
                                     _ptr(ws), ws.numel(), _stream(q)))
    return out, sel_out


# ------------------------------------------------------------------ narrow blocks

QSA_D = 256


def msa_qsa_attn_fwd(q, k, v, sel, cu_seqlens, max_seqlen: int, scale: Optional[float] = None,
                     out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                     workspace: Optional[torch.Tensor] = None):
    """Narrow-block (4-token) sparse attention forward, head dim 256, Hq = 12 Hkv:
    (o bf16 [T, Hq, 256], lse fp32 [T, Hq]).  sel int32 [T, Hkv, topk]."""
    T, Hq, Hkv = q.shape[0], q.shape[1], k.shape[1]
    topk = sel.shape[-1]
    _req(q, "q", torch.bfloat16, (T, Hq, QSA_D))
    _req(k, "k", torch.bfloat16, (T, Hkv, QSA_D))
    _req(v, "v", torch.bfloat16, (T, Hkv, QSA_D))
    _req(sel, "sel", torch.int32, (T, Hkv, topk))
    _req(cu_seqlens, "cu_seqlens", torch.int32)
    S = cu_seqlens.numel() - 1
    scale = 1.0 / math.sqrt(QSA_D) if scale is None else scale
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((T, Hq), dtype=torch.float32, device=q.device) if lse is None else lse
    _req(out, "out", torch.bfloat16, (T, Hq, QSA_D))
    _req(lse, "lse", torch.float32, (T, Hq))
    size = lib().msa_qsa_attn_fwd_workspace_size(T, S, Hq, Hkv, max_seqlen)
    ws = _workspace(size, q.device, workspace)
    _check(lib().msa_qsa_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(sel), _ptr(cu_seqlens), S, T,
                                  Hq, Hkv, topk, max_seqlen, scale, _ptr(out), _ptr(lse),
                                  _ptr(ws), ws.numel(), _stream(q)))
    return out, lse


def msa_qsa_attn_bwd(q, k, v, o, dout, lse, sel, cu_seqlens, max_seqlen: int,
                     scale: Optional[float] = None, dq=None, dk=None, dv=None,
                     workspace: Optional[torch.Tensor] = None):
    """Narrow-block sparse attention backward: (dq, dk, dv) in bf16."""
    T, Hq, Hkv = q.shape[0], q.shape[1], k.shape[1]
    topk = sel.shape[-1]
    _req(q, "q", torch.bfloat16, (T, Hq, QSA_D))
    _req(k, "k", torch.bfloat16, (T, Hkv, QSA_D))
    _req(v, "v", torch.bfloat16, (T, Hkv, QSA_D))
    _req(o, "o", torch.bfloat16, (T, Hq, QSA_D))
    _req(dout, "dout", torch.bfloat16, (T, Hq, QSA_D))
    _req(lse, "lse", torch.float32, (T, Hq))
    _req(sel, "sel", torch.int32, (T, Hkv, topk))
    _req(cu_seqlens, "cu_seqlens", torch.int32)
    S = cu_seqlens.numel() - 1
    scale = 1.0 / math.sqrt(QSA_D) if scale is None else scale
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    size = lib().msa_qsa_attn_bwd_workspace_size(T, S, Hq, Hkv, max_seqlen)
    ws = _workspace(size, q.device, workspace)
    _check(lib().msa_qsa_attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse),
                                  _ptr(sel), _ptr(cu_seqlens), S, T, Hq, Hkv, topk, max_seqlen,
                                  scale, _ptr(dq), _ptr(dk), _ptr(dv), _ptr(ws), ws.numel(),
                                  _stream(q)))
    return dq, dk, dv


def workspace_bytes(call: str, *args) -> int:
    """Workspace size of `call` ('qk_norm_rope_bwd', 'index_select', 'sparse_attn_fwd',
    'sparse_attn_bwd', 'qsa_attn_fwd', 'qsa_attn_bwd', 'decode_step') for the given sizes,
    as the C ABI reports it."""
    return int(getattr(lib(), f"msa_{call}_workspace_size")(*args))
