"""A seeded sweep over the argument space on the GPU, each case against the
float64 oracle: head size, batch, heads, ragged N_q and N_k, mask (none, causal,
causal with a window of any width, including wider than the keys), the forward
kernel (one or two query tiles per CTA at d = 128), the backward form (one or two
kernels at d >= 64), and the call path (device arrays, or host arrays through
fa_fwd_bwd_host with a random chunking).  Every output element by element and the
exact tile counts."""
import math

import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si
from gpu_util import assert_close, f64, lib, run_gpu

pytestmark = pytest.mark.gpu


def _case(seed):
    rng = np.random.default_rng(5000 + seed)
    d = int(rng.choice([32, 64, 128]))
    B, H = int(rng.integers(1, 3)), int(rng.integers(1, 4))
    causal = bool(rng.integers(0, 2))
    Nk = int(rng.integers(1, 700))
    Nq = int(rng.integers(1, Nk + 1)) if causal else int(rng.integers(1, 700))
    window = int(rng.integers(1, 2 * Nk + 2)) if causal and rng.integers(0, 2) else 0
    split = int(rng.choice([0, 1, 2, 3])) if d >= 64 else 0
    form = int(rng.choice([0, 1, 2, 3])) if d == 128 else int(rng.choice([0, 1, 3]))
    host = bool(rng.integers(0, 3) == 0)
    hpc = int(rng.integers(0, B * H + 1))
    return d, B, H, Nq, Nk, causal, window, split, form, host, hpc


def _host_path(Q, K, V, dO, causal, window, hpc):
    fa = lib()
    B, H, Nq, d = Q.shape
    Nk = K.shape[2]
    ins = [t.contiguous().pin_memory() for t in (Q, K, V, dO)]
    O, dQ = (torch.empty(Q.shape, dtype=torch.bfloat16, pin_memory=True) for _ in range(2))
    dK, dV = (torch.empty(K.shape, dtype=torch.bfloat16, pin_memory=True) for _ in range(2))
    L = torch.empty((B, H, Nq), dtype=torch.float32, pin_memory=True)
    ws_bytes = fa.fa_fwd_bwd_host_workspace_size(B, H, Nq, Nk, d, causal, window, hpc)
    ws = torch.empty(ws_bytes + 256, dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream()
    fa.check(fa.fa_fwd_bwd_host(*(t.data_ptr() for t in ins), O.data_ptr(), L.data_ptr(), dQ.data_ptr(), dK.data_ptr(),
                                dV.data_ptr(), B, H, Nq, Nk, d, causal, window, 1 / math.sqrt(d), hpc,
                                (ws.data_ptr() + 255) // 256 * 256, ws_bytes, s.cuda_stream), "fa_fwd_bwd_host")
    st, detail = fa.fa_poll_device_error(s.cuda_stream)
    fa.check(st, f"device status word (site {detail:#x})")
    return {"O": O, "L": L, "dQ": dQ, "dK": dK, "dV": dV}


@pytest.mark.parametrize("seed", range(48))
def test_sweep(seed):
    d, B, H, Nq, Nk, causal, window, split, form, host, hpc = _case(seed)
    label = (f"seed={seed} d={d} B={B} H={H} Nq={Nq} Nk={Nk} causal={causal} w={window} split={split} form={form} "
             f"host={host} hpc={hpc}")
    Q, K, V, dO = si.make_qkvdo(B, H, max(Nq, Nk), d, seed=6000 + seed)
    Q, dO = Q[:, :, :Nq].contiguous(), dO[:, :, :Nq].contiguous()
    K, V = K[:, :, :Nk].contiguous(), V[:, :, :Nk].contiguous()
    fa = lib()
    fa.check(fa.fa_debug_set_fwd_form(form))
    try:
        if host:
            fa.check(fa.fa_debug_set_bwd_split(split))
            try:
                got = _host_path(Q, K, V, dO, causal, window, hpc)
            finally:
                fa.fa_debug_set_bwd_split(0)
        else:
            got = run_gpu(Q, K, V, dO, causal, counter=True, split=split, window=window)
    finally:
        fa.fa_debug_set_fwd_form(0)
    q, k, v, do = (f64(t) for t in (Q, K, V, dO))
    O, L = oracle.standard_attention_fwd(q, k, v, causal, window=window)
    dQ, dK, dV, _ = oracle.standard_attention_bwd(q, k, v, do, causal, window=window)
    assert_close({n: f64(got[n]) for n in ("O", "L", "dQ", "dK", "dV")},
                 {"O": O, "L": L, "dQ": dQ, "dK": dK, "dV": dV}, label)
    if not host:
        _, br, bc = fa.fa_get_tile_config(d, 0)
        pairs = oracle.causal_tile_pairs(Nq, br, bc, causal, Nk=Nk, window=window)
        assert got["tiles"][0] == B * H * pairs, label
        assert got["tiles"][1] == B * H * fa.fa_tile_pairs_ex(Nq, Nk, d, causal, window, 1), label
