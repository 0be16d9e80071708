"""Exact tiled attention for GB300 (sm_103a): Python binding of libfa_gb300.so.

Every function named ``fa_*`` mirrors the C entry point of the same name in
include/fa.h and only marshals arguments (integers for pointers, a CUDA stream
handle); all of the work runs in the library's CUDA kernels.  There is no
fallback: if the library is not built, importing the binding raises.

The tensor-level helpers at the bottom (``attention_forward``,
``attention_backward``) allocate outputs with PyTorch — PyTorch supplies
device memory and streams only — and call the same entry points.
"""
from __future__ import annotations

import ctypes
import math
import os

__all__ = [
    "FA_OK", "FA_ERR_INVALID_ARG", "FA_ERR_UNSUPPORTED", "FA_ERR_CUDA", "FA_ERR_TIMEOUT", "FA_ERR_WORKSPACE",
    "FAError", "lib", "lib_path", "fa_fwd", "fa_bwd_preprocess", "fa_bwd_workspace_size", "fa_bwd",
    "fa_bwd_noalloc", "FA_NOALLOC_MAX_WORKSPACE_BYTES",
    "fa_status_string", "fa_get_tile_config", "fa_tile_pairs", "fa_debug_set_tile_counter", "fa_debug_set_bwd_split",
    "fa_poll_device_error", "fa_debug_timeout_probe", "fa_selftest_umma", "fa_version",
    "attention_forward", "attention_backward", "check",
]

FA_OK, FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED, FA_ERR_CUDA, FA_ERR_TIMEOUT, FA_ERR_WORKSPACE = range(6)

_HERE = os.path.dirname(os.path.abspath(__file__))
lib_path = os.path.join(_HERE, "libfa_gb300.so")


class FAError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {fa_status_string(status)} ({status})" if what else fa_status_string(status))


def _load():
    if not os.path.exists(lib_path):
        raise ImportError(
            f"{lib_path} is missing: build it with `python exact_tiled_attention_26_gb300/build.py` "
            "(or __graft_entry__.build()); there is no non-CUDA fallback")
    return ctypes.CDLL(lib_path)


lib = _load()

_vp, _i, _f, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
_sig = {
    "fa_fwd": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _vp]),
    "fa_bwd_preprocess": (_i, [_vp, _vp, _vp, _i, _i, _i, _i, _vp]),
    "fa_bwd_workspace_size": (_sz, [_i, _i, _i, _i, _i]),
    "fa_bwd": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _vp, _sz, _vp]),
    "fa_bwd_noalloc": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _vp]),
    "fa_status_string": (ctypes.c_char_p, [_i]),
    "fa_get_tile_config": (_i, [_i, _i, ctypes.POINTER(_i), ctypes.POINTER(_i)]),
    "fa_tile_pairs": (ctypes.c_longlong, [_i, _i, _i, _i]),
    "fa_debug_set_tile_counter": (_i, [_vp]),
    "fa_debug_set_bwd_split": (_i, [_i]),
    "fa_poll_device_error": (_i, [_vp, ctypes.POINTER(_i)]),
    "fa_debug_timeout_probe": (_i, [_i, _vp]),
    "fa_selftest_umma": (_i, [_i, _vp, _vp, _vp, _i, _i, _vp]),
    "fa_version": (_i, []),
}
for _name, (_res, _args) in _sig.items():
    _fn = getattr(lib, _name)
    _fn.restype, _fn.argtypes = _res, _args


# ------------------------------------------------------------------ C entry points

def fa_fwd(Q, K, V, O, L, B, H, N, d, causal, scale, stream):
    return lib.fa_fwd(Q, K, V, O, L, B, H, N, d, int(bool(causal)), scale, stream)


def fa_bwd_preprocess(O, dO, D, B, H, N, d, stream):
    return lib.fa_bwd_preprocess(O, dO, D, B, H, N, d, stream)


def fa_bwd_workspace_size(B, H, N, d, causal):
    return lib.fa_bwd_workspace_size(B, H, N, d, int(bool(causal)))


def fa_bwd(Q, K, V, O, dO, L, D, dQ, dK, dV, B, H, N, d, causal, scale, workspace, workspace_bytes, stream):
    return lib.fa_bwd(Q, K, V, O, dO, L, D, dQ, dK, dV, B, H, N, d, int(bool(causal)), scale, workspace,
                      workspace_bytes, stream)


FA_NOALLOC_MAX_WORKSPACE_BYTES = 16 << 20


def fa_bwd_noalloc(Q, K, V, O, dO, L, D, dQ, dK, dV, B, H, N, d, causal, scale, stream):
    """fa_bwd without a caller-provided workspace (see include/fa.h): for callers
    that cannot allocate device memory; limited to B*H*N*d*4 <= 16 MiB."""
    return lib.fa_bwd_noalloc(Q, K, V, O, dO, L, D, dQ, dK, dV, B, H, N, d, int(bool(causal)), scale, stream)


def fa_status_string(status):
    return lib.fa_status_string(int(status)).decode()


def fa_get_tile_config(d, pass_):
    br, bc = _i(0), _i(0)
    st = lib.fa_get_tile_config(d, pass_, ctypes.byref(br), ctypes.byref(bc))
    return st, br.value, bc.value


def fa_tile_pairs(N, d, causal, pass_):
    return lib.fa_tile_pairs(N, d, int(bool(causal)), pass_)


def fa_debug_set_tile_counter(dev_counter):
    return lib.fa_debug_set_tile_counter(dev_counter)


def fa_debug_set_bwd_split(split):
    return lib.fa_debug_set_bwd_split(split)


def fa_poll_device_error(stream):
    detail = _i(0)
    st = lib.fa_poll_device_error(stream, ctypes.byref(detail))
    return st, detail.value


def fa_debug_timeout_probe(limit_us, stream):
    return lib.fa_debug_timeout_probe(limit_us, stream)


def fa_selftest_umma(mode, A, B, C, K, N, stream):
    return lib.fa_selftest_umma(mode, A, B, C, K, N, stream)


def fa_version():
    return lib.fa_version()


def check(status, what=""):
    if status != FA_OK:
        raise FAError(status, what)


# ------------------------------------------------------------------ tensor helpers

def _stream_handle(device):
    import torch
    return torch.cuda.current_stream(device).cuda_stream


def _check_qkv(*ts):
    import torch
    t0 = ts[0]
    for t in ts:
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous() or t.dim() != 4:
            raise ValueError("expected contiguous bf16 CUDA tensors of shape [B, H, N, d]")
        if t.shape != t0.shape or t.device != t0.device:
            raise ValueError("Q, K, V (and O, dO) must share shape and device")


def attention_forward(q, k, v, causal=False, scale=None):
    """O, L = exact attention of bf16 [B,H,N,d] CUDA tensors (L fp32 [B,H,N])."""
    import torch
    _check_qkv(q, k, v)
    B, H, N, d = q.shape
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    check(fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, N, d, causal, scale,
                 _stream_handle(q.device)), "fa_fwd")
    return o, lse


def attention_backward(q, k, v, o, lse, do, causal=False, scale=None, workspace=None):
    """dQ, dK, dV (bf16) and D (fp32) of exact attention, from the forward's O and L."""
    import torch
    _check_qkv(q, k, v, o, do)
    B, H, N, d = q.shape
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    stream = _stream_handle(q.device)
    D = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    check(fa_bwd_preprocess(o.data_ptr(), do.data_ptr(), D.data_ptr(), B, H, N, d, stream), "fa_bwd_preprocess")
    ws_bytes = fa_bwd_workspace_size(B, H, N, d, causal)
    if workspace is None or workspace.numel() * workspace.element_size() < ws_bytes:
        workspace = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=q.device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    check(fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(), lse.data_ptr(),
                 D.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, N, d, causal, scale,
                 workspace.data_ptr(), workspace.numel() * workspace.element_size(), stream), "fa_bwd")
    return dq, dk, dv, D
