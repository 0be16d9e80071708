"""fa_bwd_noalloc: the backward for callers that cannot allocate device memory
(their device memory is reserved by someone else's pool, or cudaMalloc's device
synchronisation is off limits where they run).  Its fp32 dQ accumulator is a
fixed array inside the library instead of a caller-allocated workspace.

This file is collected last on purpose (tests/test_zz_*), so that a run that
stops at the first failure has already run every other test.  It must also pass
alone in a fresh process.
"""
import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si
from gpu_util import TOL_G_REL, assert_close, f64, lib, rel_frob, stream

pytestmark = pytest.mark.gpu


def _forward_and_D(fa, q, k, v, do, causal):
    B, H, N, d = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    D = torch.empty_like(lse)
    fa.check(fa.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, N, d, causal,
                       d ** -0.5, stream()))
    fa.check(fa.fa_bwd_preprocess(o.data_ptr(), do.data_ptr(), D.data_ptr(), B, H, N, d, stream()))
    return o, lse, D


# split: the backward form (fa_debug_set_bwd_split; 0 = the library's choice).  The
# d = 64 case forces the one-kernel form, which accumulates dQ in the array (the
# library's d = 64 default needs none), so every case exercises the array.
@pytest.mark.parametrize("B,H,N,d,causal,split", [(1, 4, 1000, 128, True, 0), (2, 3, 777, 64, False, 1),
                                                  (1, 1, 256, 32, True, 0)])
def test_noalloc_matches_fa_bwd_twice(B, H, N, d, causal, split):
    """Two calls in a row of the no-allocation entry point give the same dQ, dK,
    dV as fa_bwd with a caller workspace (within the gradient tolerance of the
    other tests; dQ sums in a different order each call, so not bit for bit), and
    both match the float64 oracle.  The second call also shows the shared array is
    cleared between calls."""
    fa = lib()
    fa.check(fa.fa_debug_set_bwd_split(split))
    try:
        _noalloc_twice(fa, B, H, N, d, causal)
    finally:
        fa.fa_debug_set_bwd_split(0)


def _noalloc_twice(fa, B, H, N, d, causal):
    Q, K, V, dO = si.make_qkvdo(B, H, N, d, seed=4242 + N)
    q64, k64, v64, do64 = (f64(t) for t in (Q, K, V, dO))
    dQ, dK, dV, _ = oracle.standard_attention_bwd(q64, k64, v64, do64, causal)
    q, k, v, do = (t.cuda() for t in (Q, K, V, dO))
    o, lse, D = _forward_and_D(fa, q, k, v, do, causal)
    ref = [torch.empty_like(q) for _ in range(3)]
    ws_bytes = fa.fa_bwd_workspace_size(B, H, N, d, causal)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    fa.check(fa.fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(), lse.data_ptr(),
                       D.data_ptr(), *(t.data_ptr() for t in ref), B, H, N, d, causal, d ** -0.5, ws.data_ptr(),
                       ws_bytes, stream()), "fa_bwd")
    for call in range(2):
        got = [torch.full_like(q, float("nan")) for _ in range(3)]
        fa.check(fa.fa_bwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(),
                                   lse.data_ptr(), D.data_ptr(), *(t.data_ptr() for t in got), B, H, N, d, causal,
                                   d ** -0.5, stream()), f"fa_bwd_noalloc call {call}")
        st, detail = fa.fa_poll_device_error(stream())
        fa.check(st, f"device status (site {detail:#x})")
        for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
            err = rel_frob(f64(g.cpu()), f64(r.cpu()))
            assert err <= TOL_G_REL, f"call {call}: {name} rel {err:.3e}"
        assert torch.equal(got[1], ref[1]) and torch.equal(got[2], ref[2])  # dK, dV: same order of sums
        assert_close({n: f64(g.cpu()) for n, g in zip(("dQ", "dK", "dV"), got)}, {"dQ": dQ, "dK": dK, "dV": dV},
                     f"fa_bwd_noalloc call {call} vs oracle")


def test_noalloc_rejects_problems_beyond_its_array():
    fa = lib()
    B, H, N, d = 1, 64, 1024, 128  # 32 MiB of dQ accumulator > 16 MiB
    assert fa.fa_bwd_workspace_size(B, H, N, d, True) > fa.FA_NOALLOC_MAX_WORKSPACE_BYTES
    x = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    p = x.data_ptr()
    assert fa.fa_bwd_noalloc(p, p, p, p, p, p, p, p, p, p, B, H, N, d, True, 0.1, stream()) == fa.FA_ERR_WORKSPACE
    # an empty problem needs no array at all
    assert fa.fa_bwd_noalloc(*([None] * 10), 1, 1, 0, 128, True, 0.1, stream()) == fa.FA_OK
