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
    "fa_fwd_ex", "fa_bwd_ex", "fa_bwd_workspace_size_ex", "fa_tile_pairs_ex",
    "fa_bwd_noalloc", "FA_NOALLOC_MAX_WORKSPACE_BYTES",
    "fa_fwd_bwd_host", "fa_fwd_bwd_host_workspace_size", "fa_fwd_bwd_host_chunk_heads",
    "fa_status_string", "fa_get_tile_config", "fa_tile_pairs", "fa_debug_set_tile_counter", "fa_debug_set_bwd_split",
    "fa_debug_set_fwd_form", "fa_selected_forms", "fa_debug_bwd_plan", "fa_debug_set_kernel_events",
    "fa_poll_device_error", "fa_debug_timeout_probe", "fa_selftest_umma", "fa_version",
    "attention_forward", "attention_backward", "attention_fwd_bwd_host", "check",
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
    "fa_fwd_ex": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _f, _vp]),
    "fa_bwd_workspace_size_ex": (_sz, [_i, _i, _i, _i, _i, _i, _i]),
    "fa_bwd_ex": (_i, [_vp] * 10 + [_i] * 7 + [_f, _vp, _sz, _vp]),
    "fa_tile_pairs_ex": (ctypes.c_longlong, [_i, _i, _i, _i, _i, _i]),
    "fa_bwd_preprocess": (_i, [_vp, _vp, _vp, _i, _i, _i, _i, _vp]),
    "fa_bwd_workspace_size": (_sz, [_i, _i, _i, _i, _i]),
    "fa_bwd": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _vp, _sz, _vp]),
    "fa_bwd_noalloc": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _vp]),
    "fa_fwd_bwd_host_chunk_heads": (_i, [_i] * 6),
    "fa_fwd_bwd_host_workspace_size": (_sz, [_i] * 8),
    "fa_fwd_bwd_host": (_i, [_vp] * 9 + [_i] * 7 + [_f, _i, _vp, _sz, _vp]),
    "fa_status_string": (ctypes.c_char_p, [_i]),
    "fa_get_tile_config": (_i, [_i, _i, ctypes.POINTER(_i), ctypes.POINTER(_i)]),
    "fa_tile_pairs": (ctypes.c_longlong, [_i, _i, _i, _i]),
    "fa_debug_set_tile_counter": (_i, [_vp]),
    "fa_debug_set_bwd_split": (_i, [_i]),
    "fa_debug_set_fwd_form": (_i, [_i]),
    "fa_selected_forms": (_i, [_i] * 7 + [ctypes.POINTER(_i)] * 2),
    "fa_debug_bwd_plan": (_i, [_i] * 7 + [ctypes.POINTER(_i), ctypes.POINTER(_sz)]),
    "fa_debug_set_kernel_events": (_i, [_i, _vp, _vp]),
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


def fa_fwd_ex(Q, K, V, O, L, B, H, Nq, Nk, d, causal, window, scale, stream):
    return lib.fa_fwd_ex(Q, K, V, O, L, B, H, Nq, Nk, d, int(bool(causal)), window, scale, stream)


def fa_bwd_workspace_size_ex(B, H, Nq, Nk, d, causal, window):
    return lib.fa_bwd_workspace_size_ex(B, H, Nq, Nk, d, int(bool(causal)), window)


def fa_bwd_ex(Q, K, V, O, dO, L, D, dQ, dK, dV, B, H, Nq, Nk, d, causal, window, scale, workspace, workspace_bytes,
              stream):
    return lib.fa_bwd_ex(Q, K, V, O, dO, L, D, dQ, dK, dV, B, H, Nq, Nk, d, int(bool(causal)), window, scale,
                         workspace, workspace_bytes, stream)


def fa_tile_pairs_ex(Nq, Nk, d, causal, window, pass_):
    return lib.fa_tile_pairs_ex(Nq, Nk, d, int(bool(causal)), window, pass_)


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


def fa_fwd_bwd_host_chunk_heads(B, H, Nq, Nk, d, heads_per_chunk):
    return lib.fa_fwd_bwd_host_chunk_heads(B, H, Nq, Nk, d, heads_per_chunk)


def fa_fwd_bwd_host_workspace_size(B, H, Nq, Nk, d, causal, window, heads_per_chunk):
    return lib.fa_fwd_bwd_host_workspace_size(B, H, Nq, Nk, d, int(bool(causal)), window, heads_per_chunk)


def fa_fwd_bwd_host(Q, K, V, dO, O, L, dQ, dK, dV, B, H, Nq, Nk, d, causal, window, scale, heads_per_chunk, workspace,
                    workspace_bytes, stream):
    """Forward + backward on host arrays, copies overlapped with the kernels (see include/fa.h)."""
    return lib.fa_fwd_bwd_host(Q, K, V, dO, O, L, dQ, dK, dV, B, H, Nq, Nk, d, int(bool(causal)), window, scale,
                               heads_per_chunk, workspace, workspace_bytes, stream)


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


def fa_debug_set_fwd_form(form):
    return lib.fa_debug_set_fwd_form(form)


def fa_selected_forms(B, H, Nq, Nk, d, causal, window):
    """(status, forward form, backward form) the library would run for these sizes and mask."""
    f, b = _i(0), _i(0)
    st = lib.fa_selected_forms(B, H, Nq, Nk, d, int(bool(causal)), window, ctypes.byref(f), ctypes.byref(b))
    return st, f.value, b.value


def fa_debug_bwd_plan(B, H, Nq, Nk, d, causal, window):
    """(status, backward form, workspace bytes) from one reading of the form setting."""
    f, n = _i(0), _sz(0)
    st = lib.fa_debug_bwd_plan(B, H, Nq, Nk, d, int(bool(causal)), window, ctypes.byref(f), ctypes.byref(n))
    return st, f.value, n.value


def fa_debug_set_kernel_events(which, start, stop):
    """Caller-owned CUDA events (raw cudaEvent_t handles, or None) recorded around the main kernel
    launch of later forward (which=0) or backward (which=1) calls."""
    return lib.fa_debug_set_kernel_events(which, start, stop)


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


def _check_tensors(q, k, v, *rest):
    """q [B,H,Nq,d], k and v [B,H,Nk,d], rest (o, do) like q: contiguous bf16 on one CUDA device."""
    import torch
    for t in (q, k, v) + rest:
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous() or t.dim() != 4:
            raise ValueError("expected contiguous bf16 CUDA tensors of shape [B, H, N, d]")
        if t.device != q.device:
            raise ValueError("all tensors must be on one device")
    if k.shape != v.shape or k.shape[:2] != q.shape[:2] or k.shape[3] != q.shape[3]:
        raise ValueError("K and V must be [B, H, Nk, d] with the B, H and d of Q")
    for t in rest:
        if t.shape != q.shape:
            raise ValueError("O and dO must have the shape of Q")


def attention_forward(q, k, v, causal=False, scale=None, window=0):
    """O, L = exact attention of bf16 CUDA tensors q [B,H,Nq,d], k, v [B,H,Nk,d]
    (L fp32 [B,H,Nq]); the mask of fa_fwd_ex (queries at the last Nq positions,
    optional sliding window)."""
    import torch
    _check_tensors(q, k, v)
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    check(fa_fwd_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, Nq, Nk, d, causal,
                    window, scale, _stream_handle(q.device)), "fa_fwd_ex")
    return o, lse


def attention_backward(q, k, v, o, lse, do, causal=False, scale=None, window=0, workspace=None):
    """dQ, dK, dV (bf16) and D (fp32) of exact attention, from the forward's O and L."""
    import torch
    _check_tensors(q, k, v, o, do)
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    stream = _stream_handle(q.device)
    D = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    check(fa_bwd_preprocess(o.data_ptr(), do.data_ptr(), D.data_ptr(), B, H, Nq, d, stream), "fa_bwd_preprocess")
    ws_bytes = fa_bwd_workspace_size_ex(B, H, Nq, Nk, d, causal, window)
    if workspace is None or workspace.numel() * workspace.element_size() < ws_bytes:
        workspace = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=q.device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    check(fa_bwd_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(), lse.data_ptr(),
                    D.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, Nq, Nk, d, causal, window, scale,
                    workspace.data_ptr(), workspace.numel() * workspace.element_size(), stream), "fa_bwd_ex")
    return dq, dk, dv, D


def attention_fwd_bwd_host(q, k, v, do, causal=False, scale=None, window=0, heads_per_chunk=0, device=None):
    """O, L, dQ, dK, dV of exact attention for bf16 CPU tensors q, do [B,H,Nq,d] and
    k, v [B,H,Nk,d], computed on `device` (default: the current CUDA device) by
    fa_fwd_bwd_host.  Returns page-locked CPU tensors once the step has finished.
    Page-locked inputs (Tensor.pin_memory()) let the copies overlap the kernels."""
    import torch
    for t in (q, k, v, do):
        if t.dtype != torch.bfloat16 or t.is_cuda or not t.is_contiguous() or t.dim() != 4:
            raise ValueError("expected contiguous bf16 CPU tensors of shape [B, H, N, d]")
    if k.shape != v.shape or k.shape[:2] != q.shape[:2] or k.shape[3] != q.shape[3] or do.shape != q.shape:
        raise ValueError("K and V must be [B, H, Nk, d] with the B, H and d of Q; dO must have the shape of Q")
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    ws_bytes = fa_fwd_bwd_host_workspace_size(B, H, Nq, Nk, d, causal, window, heads_per_chunk)
    if ws_bytes == ctypes.c_size_t(-1).value:
        check(FA_ERR_INVALID_ARG, "fa_fwd_bwd_host_workspace_size")
    with torch.cuda.device(device):
        ws = torch.empty(max(ws_bytes + 256, 256), dtype=torch.uint8, device=device)
        base = (ws.data_ptr() + 255) // 256 * 256
        o, dq = (torch.empty(q.shape, dtype=torch.bfloat16, pin_memory=True) for _ in range(2))
        dk, dv = (torch.empty(k.shape, dtype=torch.bfloat16, pin_memory=True) for _ in range(2))
        lse = torch.empty((B, H, Nq), dtype=torch.float32, pin_memory=True)
        stream = torch.cuda.current_stream(device)
        check(fa_fwd_bwd_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), do.data_ptr(), o.data_ptr(), lse.data_ptr(),
                              dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, Nq, Nk, d, causal, window, scale,
                              heads_per_chunk, base, ws_bytes, stream.cuda_stream), "fa_fwd_bwd_host")
        stream.synchronize()
        del ws
    return o, lse, dq, dk, dv
