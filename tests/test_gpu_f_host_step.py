"""GPU checks of fa_fwd_bwd_host, the forward + backward step on host arrays with
the copies overlapped: against the device-resident path (the same kernels, so O,
L, dK and dV must agree bit for bit; dQ is summed in fp32 reductions whose order
varies) and against the float64 oracle, over chunk plans that reuse the device
slots, alternate the compute streams and leave a short last chunk."""
import math

import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si
from gpu_util import assert_close, f64, lib, run_gpu

pytestmark = pytest.mark.gpu


def _host_step(Q, K, V, dO, causal, window=0, hpc=0, pinned=True, counter=None):
    fa = lib()
    B, H, Nq, d = Q.shape
    Nk = K.shape[2]
    ins = [t.contiguous() for t in (Q, K, V, dO)]
    if pinned:
        ins = [t.pin_memory() for t in ins]
    O, dQ = (torch.full(Q.shape, 9.0, dtype=torch.bfloat16, pin_memory=pinned) for _ in range(2))
    dK, dV = (torch.full(K.shape, 9.0, dtype=torch.bfloat16, pin_memory=pinned) for _ in range(2))
    L = torch.full((B, H, Nq), 9.0, dtype=torch.float32, pin_memory=pinned)
    ws_bytes = fa.fa_fwd_bwd_host_workspace_size(B, H, Nq, Nk, d, causal, window, hpc)
    ws = torch.empty(ws_bytes + 256, dtype=torch.uint8, device="cuda")
    base = (ws.data_ptr() + 255) // 256 * 256
    s = torch.cuda.current_stream()
    if counter is not None:
        fa.check(fa.fa_debug_set_tile_counter(counter.data_ptr()))
    try:
        fa.check(fa.fa_fwd_bwd_host(*(t.data_ptr() for t in ins), O.data_ptr(), L.data_ptr(), dQ.data_ptr(),
                                    dK.data_ptr(), dV.data_ptr(), B, H, Nq, Nk, d, causal, window, 1 / math.sqrt(d),
                                    hpc, base, ws_bytes, s.cuda_stream), "fa_fwd_bwd_host")
    finally:
        if counter is not None:
            fa.fa_debug_set_tile_counter(None)
    st, detail = fa.fa_poll_device_error(s.cuda_stream)
    fa.check(st, f"device status word (site {detail:#x})")
    return {"O": O, "L": L, "dQ": dQ, "dK": dK, "dV": dV}


def _same_as_device_path(Q, K, V, dO, causal, window, got):
    ref = run_gpu(Q, K, V, dO, causal, window=window)
    for n in ("O", "L", "dK", "dV"):
        assert torch.equal(got[n], ref[n]), n
    # dQ: the same sums in another order, rounded to bf16
    a, b = f64(got["dQ"]), f64(ref["dQ"])
    assert np.linalg.norm(a - b) <= 2e-3 * np.linalg.norm(b)


@pytest.mark.parametrize("hpc", [0, 1, 2, 4, 6])
@pytest.mark.parametrize("d", [64, 128])
def test_chunk_plans_match_device_path(hpc, d):
    """B*H = 6: one chunk per head (six chunks: every slot reused, both compute
    streams), 2, 4 (a short last chunk), 6 (one chunk) and the automatic plan."""
    Q, K, V, dO = si.make_qkvdo(2, 3, 640, d, seed=1100 + hpc + d)
    got = _host_step(Q, K, V, dO, True, hpc=hpc)
    _same_as_device_path(Q, K, V, dO, True, 0, got)


@pytest.mark.parametrize("causal,window,Nq,Nk", [(False, 0, 300, 300), (True, 96, 700, 700), (True, 0, 200, 900),
                                                 (False, 0, 1, 500)])
def test_masks_match_oracle(causal, window, Nq, Nk):
    Q, K, V, dO = si.make_qkvdo(1, 5, max(Nq, Nk), 128, seed=1200 + Nq + window)
    Q, dO = Q[:, :, :Nq].contiguous(), dO[:, :, :Nq].contiguous()
    K, V = K[:, :, :Nk].contiguous(), V[:, :, :Nk].contiguous()
    got = _host_step(Q, K, V, dO, causal, window=window, hpc=2)
    q, k, v, do = (f64(t) for t in (Q, K, V, dO))
    O, L = oracle.standard_attention_fwd(q, k, v, causal, window=window)
    dQ, dK, dV, _ = oracle.standard_attention_bwd(q, k, v, do, causal, window=window)
    assert_close({n: f64(t) for n, t in got.items()}, {"O": O, "L": L, "dQ": dQ, "dK": dK, "dV": dV},
                 f"host step causal={causal} w={window} Nq={Nq} Nk={Nk}")
    _same_as_device_path(Q, K, V, dO, causal, window, got)


def test_pageable_host_arrays():
    """Pageable (not page-locked) host arrays: the copies serialise, the results do not change."""
    Q, K, V, dO = si.make_qkvdo(1, 4, 384, 128, seed=1300)
    got = _host_step(Q, K, V, dO, True, hpc=1, pinned=False)
    _same_as_device_path(Q, K, V, dO, True, 0, got)


def test_no_queries_zero_key_gradients():
    K = torch.randn(1, 3, 200, 64).to(torch.bfloat16)
    Q = torch.empty(1, 3, 0, 64, dtype=torch.bfloat16)
    got = _host_step(Q, K, K.clone(), Q.clone(), True, hpc=1)
    assert (got["dK"] == 0).all() and (got["dV"] == 0).all()


def test_tile_counts_over_chunks():
    fa = lib()
    cnt = torch.zeros(1, dtype=torch.int64, device="cuda")
    Q, K, V, dO = si.make_qkvdo(2, 3, 1000, 128, seed=1400)
    _host_step(Q, K, V, dO, True, hpc=4, counter=cnt)
    per_head = fa.fa_tile_pairs_ex(1000, 1000, 128, True, 0, 0) + fa.fa_tile_pairs_ex(1000, 1000, 128, True, 0, 1)
    assert int(cnt.item()) == 6 * per_head


def test_back_to_back_calls_without_sync():
    """Two steps enqueued on one stream before any synchronisation, sharing the
    internal streams and events: each gets its own results."""
    fa = lib()
    d, B, H, N = 128, 1, 6, 512
    ins = [si.make_qkvdo(B, H, N, d, seed=1500 + i) for i in range(2)]
    s = torch.cuda.current_stream()
    ws_bytes = fa.fa_fwd_bwd_host_workspace_size(B, H, N, N, d, True, 0, 1)
    outs = []
    wss = [torch.empty(ws_bytes + 256, dtype=torch.uint8, device="cuda") for _ in range(2)]
    for (Q, K, V, dO), ws in zip(ins, wss):
        hin = [t.pin_memory() for t in (Q, K, V, dO)]
        o = {n: torch.empty(Q.shape, dtype=torch.bfloat16, pin_memory=True) for n in ("O", "dQ", "dK", "dV")}
        o["L"] = torch.empty((B, H, N), dtype=torch.float32, pin_memory=True)
        base = (ws.data_ptr() + 255) // 256 * 256
        fa.check(fa.fa_fwd_bwd_host(*(t.data_ptr() for t in hin), o["O"].data_ptr(), o["L"].data_ptr(),
                                    o["dQ"].data_ptr(), o["dK"].data_ptr(), o["dV"].data_ptr(), B, H, N, N, d, True, 0,
                                    1 / math.sqrt(d), 1, base, ws_bytes, s.cuda_stream))
        outs.append((hin, o))
    s.synchronize()
    for (Q, K, V, dO), (_, o) in zip(ins, outs):
        _same_as_device_path(Q, K, V, dO, True, 0, o)


def test_tensor_helper_matches_oracle():
    from exact_tiled_attention_26_gb300 import attention_fwd_bwd_host
    Q, K, V, dO = si.make_qkvdo(2, 2, 333, 64, seed=1600)
    o, lse, dq, dk, dv = attention_fwd_bwd_host(*(t.pin_memory() for t in (Q, K, V, dO)), causal=True)
    q, k, v, do = (f64(t) for t in (Q, K, V, dO))
    O, L = oracle.standard_attention_fwd(q, k, v, True)
    dQ, dK, dV, _ = oracle.standard_attention_bwd(q, k, v, do, True)
    assert_close({"O": f64(o), "L": f64(lse), "dQ": f64(dq), "dK": f64(dk), "dV": f64(dv)},
                 {"O": O, "L": L, "dQ": dQ, "dK": dK, "dV": dV}, "attention_fwd_bwd_host")
