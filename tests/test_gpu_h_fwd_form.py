"""The forward kernels (fa_debug_set_fwd_form: 1 one query tile per CTA, 2 two
query tiles per CTA taking turns on the tensor pipe (d = 128), 3 one CTA per SM
taking query tiles from a queue) run the same arithmetic on each row in the same
order, so O and L must agree bit for bit; forms 2 and 3 are also checked against
the float64 oracle, over masks, ragged and odd tile counts (a last CTA with one
query tile), N_q != N_k and large logits."""
import math

import pytest
import torch

import oracle
import seeded_inputs as si
from gpu_util import assert_close, f64, lib

pytestmark = pytest.mark.gpu


def _fwd(form, Q, K, V, causal, window, counter=None):
    fa = lib()
    B, H, Nq, d = Q.shape
    Nk = K.shape[2]
    q, k, v = (t.cuda() for t in (Q, K, V))
    o = torch.empty_like(q)
    lse = torch.empty(B, H, Nq, dtype=torch.float32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    fa.check(fa.fa_debug_set_fwd_form(form))
    if counter is not None:
        fa.check(fa.fa_debug_set_tile_counter(counter.data_ptr()))
    try:
        fa.check(fa.fa_fwd_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, Nq, Nk, d,
                              causal, window, 1 / math.sqrt(d), s))
    finally:
        fa.fa_debug_set_fwd_form(0)
        fa.fa_debug_set_tile_counter(None)
    st, detail = fa.fa_poll_device_error(s)
    fa.check(st, f"device status word (site {detail:#x})")
    return o.cpu(), lse.cpu()


def _inputs(B, H, Nq, Nk, seed, qk_mult=1.0, d=128):
    Q, K, V, _ = si.make_qkvdo(B, H, max(Nq, Nk), d, seed=seed, qk_mult=qk_mult)
    return Q[:, :, :Nq].contiguous(), K[:, :, :Nk].contiguous(), V[:, :, :Nk].contiguous()


CASES = [(1, 256, 256, False, 0), (1, 256, 256, True, 0), (2, 384, 384, True, 0), (2, 1000, 1000, True, 0),
         (2, 1000, 1000, False, 0), (2, 129, 129, True, 0), (1, 1, 700, True, 0), (1, 300, 1000, True, 0),
         (2, 1000, 300, False, 0), (2, 777, 777, True, 1), (2, 777, 777, True, 100), (2, 1000, 1000, True, 300),
         (1, 640, 2000, True, 256), (2, 128, 128, True, 0)]


@pytest.mark.parametrize("form", [2, 3])
@pytest.mark.parametrize("H,Nq,Nk,causal,window", CASES)
def test_other_forms_equal_one_tile_form(form, H, Nq, Nk, causal, window):
    Q, K, V = _inputs(1, H, Nq, Nk, seed=1900 + Nq + Nk + window)
    cnt = torch.zeros(2, dtype=torch.int64, device="cuda")
    o1, l1 = _fwd(1, Q, K, V, causal, window, counter=cnt[0:1])
    o2, l2 = _fwd(form, Q, K, V, causal, window, counter=cnt[1:2])
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert cnt[0].item() == cnt[1].item() == H * lib().fa_tile_pairs_ex(Nq, Nk, 128, causal, window, 0)


@pytest.mark.parametrize("d", [32, 64])
@pytest.mark.parametrize("B,H,Nq,Nk,causal,window", [(2, 3, 1000, 1000, True, 0), (1, 5, 300, 700, False, 0),
                                                      (3, 2, 777, 777, True, 100), (1, 1, 1, 300, True, 0),
                                                      (4, 40, 256, 256, True, 0)])
def test_persistent_form_equals_one_tile_form_small_heads(d, B, H, Nq, Nk, causal, window):
    Q, K, V = _inputs(B, H, Nq, Nk, seed=2100 + Nq + d, d=d)
    o1, l1 = _fwd(1, Q, K, V, causal, window)
    o3, l3 = _fwd(3, Q, K, V, causal, window)
    assert torch.equal(o1, o3) and torch.equal(l1, l3)


@pytest.mark.parametrize("form", [2, 3])
@pytest.mark.parametrize("H,Nq,Nk,causal,window,qk", [(2, 1000, 1000, True, 0, 1.0), (2, 700, 700, False, 0, 4.0),
                                                      (2, 900, 900, True, 200, 4.0), (1, 300, 1000, True, 0, 1.0)])
def test_other_forms_match_oracle(form, H, Nq, Nk, causal, window, qk):
    Q, K, V = _inputs(1, H, Nq, Nk, seed=2000 + Nq, qk_mult=qk)
    o, lse = _fwd(form, Q, K, V, causal, window)
    O, L = oracle.standard_attention_fwd(f64(Q), f64(K), f64(V), causal, window=window)
    assert_close({"O": f64(o), "L": f64(lse)}, {"O": O, "L": L}, f"form {form} Nq={Nq} Nk={Nk} w={window}")


@pytest.mark.parametrize("form", [2, 3])
def test_other_forms_long_shape_equal_one_tile_form(form):
    w = si.WORKLOADS["long_1x32x8192x128"]
    Q, K, V, _ = si.make_workload(w)
    o1, l1 = _fwd(1, Q, K, V, True, 0)
    o2, l2 = _fwd(form, Q, K, V, True, 0)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_work_counters_survive_reuse():
    """The persistent kernels take their work counters from a fixed pool of 1024 per
    pass, each launch leaving its counter zeroed for the pool's next round.  Run more
    launches than the pool holds (forward and backward, on one stream, shapes whose
    grids differ so that units are left for the queue), then check a launch of each
    against the one-tile kernels: a counter left non-zero would skip units."""
    fa = lib()
    s = torch.cuda.current_stream().cuda_stream
    B, H, N, d = 2, 16, 1280, 128  # 10 tiles x 32 heads = 320 units per pass: more than one per SM
    Q, K, V, dO = si.make_qkvdo(B, H, N, d, seed=4711)
    q, k, v, do = (t.cuda() for t in (Q, K, V, dO))
    o, lse = torch.empty_like(q), torch.empty(B, H, N, dtype=torch.float32, device="cuda")
    D = torch.empty_like(lse)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(fa.fa_bwd_workspace_size(B, H, N, d, True), dtype=torch.uint8, device="cuda")
    scale = 1 / math.sqrt(d)

    def step():
        fa.check(fa.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, N, d, True,
                           scale, s))
        fa.check(fa.fa_bwd_preprocess(o.data_ptr(), do.data_ptr(), D.data_ptr(), B, H, N, d, s))
        fa.check(fa.fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(), lse.data_ptr(),
                           D.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, N, d, True, scale,
                           ws.data_ptr(), ws.numel(), s))

    fa.check(fa.fa_debug_set_fwd_form(3))
    fa.check(fa.fa_debug_set_bwd_split(3))
    try:
        for _ in range(1100):  # every counter of both pools used at least once, some twice
            step()
        torch.cuda.synchronize()
        got = [t.clone() for t in (o, lse, dk, dv)]
    finally:
        fa.fa_debug_set_fwd_form(0)
        fa.fa_debug_set_bwd_split(0)
    st, detail = fa.fa_poll_device_error(s)
    fa.check(st, f"device status word (site {detail:#x})")
    fa.check(fa.fa_debug_set_fwd_form(1))
    fa.check(fa.fa_debug_set_bwd_split(1))
    try:
        step()
        torch.cuda.synchronize()
    finally:
        fa.fa_debug_set_fwd_form(0)
        fa.fa_debug_set_bwd_split(0)
    for g, r in zip(got, (o, lse, dk, dv)):
        assert torch.equal(g, r)
