"""GPU parity of the general mask against the float64 oracle: sliding windows
("CS324 lecture 8: 03_online_softmax_and_flash.py", window_attention_torch) with
the two-sided whole-tile skip, N_q != N_k with the queries at the last positions
of the key sequence (prefill chunks, decode), keys that no query sees, and the
autograd wrapper.  Every output element by element, and the exact tile counts."""
import math

import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si
from gpu_util import assert_close, f64, lib, rel_frob, run_gpu

pytestmark = pytest.mark.gpu


def _oracle(Q, K, V, dO, causal, window, scale=None):
    q, k, v, do = (f64(t) for t in (Q, K, V, dO))
    O, L = oracle.standard_attention_fwd(q, k, v, causal, scale, window=window)
    dQ, dK, dV, _ = oracle.standard_attention_bwd(q, k, v, do, causal, scale, window=window)
    return {"O": O, "L": L, "dQ": dQ, "dK": dK, "dV": dV}


def _inputs(B, H, Nq, Nk, d, seed, qk_mult=1.0):
    Q, K, V, dO = si.make_qkvdo(B, H, max(Nq, Nk), d, seed=seed, qk_mult=qk_mult)
    return Q[:, :, :Nq].contiguous(), K[:, :, :Nk].contiguous(), V[:, :, :Nk].contiguous(), dO[:, :, :Nq].contiguous()


def _check(Nq, Nk, d, causal, window, seed, split=0, B=1, H=2, qk_mult=1.0):
    Q, K, V, dO = _inputs(B, H, Nq, Nk, d, seed, qk_mult)
    got = run_gpu(Q, K, V, dO, causal, counter=True, split=split, window=window)
    ref = _oracle(Q, K, V, dO, causal, window)
    label = f"Nq={Nq} Nk={Nk} d={d} causal={causal} w={window} split={split}"
    assert_close({n: f64(got[n]) for n in ("O", "L", "dQ", "dK", "dV")}, ref, label)
    fa = lib()
    _, br, bc = fa.fa_get_tile_config(d, 0)
    pairs = oracle.causal_tile_pairs(Nq, br, bc, causal, Nk=Nk, window=window)
    assert got["tiles"][0] == B * H * pairs == B * H * fa.fa_tile_pairs_ex(Nq, Nk, d, causal, window, 0), label
    assert got["tiles"][1] == B * H * fa.fa_tile_pairs_ex(Nq, Nk, d, causal, window, 1), label
    return got


@pytest.mark.parametrize("d", [32, 64, 128])
@pytest.mark.parametrize("N,window", [(300, 1), (300, 64), (300, 127), (300, 128), (300, 129), (1000, 100),
                                      (1000, 500), (1000, 2000), (129, 3)])
def test_sliding_window(d, N, window):
    _check(N, N, d, True, window, seed=400 + N + window + d)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("split", [1, 2, 3])
@pytest.mark.parametrize("N,window", [(1000, 100), (777, 256), (300, 1)])
def test_sliding_window_both_backward_forms(d, split, N, window):
    _check(N, N, d, True, window, seed=500 + N + window, split=split)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("Nq,Nk,causal,window", [
    (1, 1000, True, 0), (1, 1000, False, 0), (1, 1000, True, 37), (7, 300, True, 0), (128, 1000, True, 0),
    (300, 1000, True, 0), (300, 1000, True, 200), (129, 257, True, 0), (1000, 300, False, 0), (64, 1000, False, 0),
    (100, 100, True, 0)])
def test_unequal_lengths(d, Nq, Nk, causal, window):
    _check(Nq, Nk, d, causal, window, seed=600 + Nq + Nk + d)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("split", [1, 2, 3])
def test_unequal_lengths_both_backward_forms(d, split):
    _check(300, 1000, d, True, 0, seed=700, split=split)
    _check(1000, 300, d, False, 0, seed=701, split=split)
    _check(64, 1000, d, True, 32, seed=702, split=split)


@pytest.mark.parametrize("d", [64, 128])
def test_keys_no_query_sees_get_zero_gradients(d):
    """A short window over the last 64 positions of 1000 keys: keys below
    1000 - 64 - 31 are seen by no query, so their dK and dV are exactly zero."""
    got = _check(64, 1000, d, True, 32, seed=800 + d)
    unseen = 1000 - 64 - 31
    assert (got["dK"][:, :, :unseen] == 0).all() and (got["dV"][:, :, :unseen] == 0).all()
    assert (got["dV"][:, :, unseen:] != 0).any()


def test_no_queries_zero_key_gradients():
    fa = lib()
    k = torch.randn(1, 2, 300, 64, device="cuda").to(torch.bfloat16)
    dk = torch.full_like(k, 7.0)
    dv = torch.full_like(k, 7.0)
    s = torch.cuda.current_stream().cuda_stream
    fa.check(fa.fa_bwd_ex(None, k.data_ptr(), k.data_ptr(), None, None, None, None, None, dk.data_ptr(), dv.data_ptr(),
                          1, 2, 0, 300, 64, 1, 0, 0.125, None, 0, s))
    torch.cuda.synchronize()
    assert (dk == 0).all() and (dv == 0).all()


def test_large_logits_with_window():
    _check(640, 640, 128, True, 200, seed=900, qk_mult=4.0)


def test_long_window_sampled_rows():
    """The long shape (1 x 32 heads x 8192 x 128) with a window of 1024: O, L, dQ on
    256 sampled rows of every head, dK and dV of one whole head."""
    w = si.WORKLOADS["long_1x32x8192x128"]
    Q, K, V, dO = si.make_workload(w)
    got = run_gpu(Q, K, V, dO, True, counter=True, window=1024)
    B, H, N, d = Q.shape
    hd = lambda t: f64(t.reshape(B * H, N, d))
    q, k, v, do = hd(Q), hd(K), hd(V), hd(dO)
    rows = si.sample_rows(w, 256)
    O, L, dQ, _ = oracle.rows_fwd_bwd(q, k, v, do, rows, True, window=1024)
    g = {"O": hd(got["O"])[:, rows], "L": f64(got["L"]).reshape(B * H, N)[:, rows], "dQ": hd(got["dQ"])[:, rows]}
    assert_close(g, {"O": O, "L": L, "dQ": dQ}, "long window rows")
    h = 7
    _, dK, dV, _ = oracle.standard_attention_bwd(q[h], k[h], v[h], do[h], True, window=1024)
    assert_close({"dK": hd(got["dK"])[h], "dV": hd(got["dV"])[h]}, {"dK": dK, "dV": dV}, "long window head")
    assert got["tiles"][0] == got["tiles"][1] == B * H * 540


@pytest.mark.parametrize("causal,window,Nq,Nk", [(False, 0, 256, 256), (True, 0, 300, 300), (True, 64, 300, 300),
                                                 (True, 0, 100, 400)])
def test_autograd_wrapper(causal, window, Nq, Nk):
    """flash_attention through torch.autograd: gradients of sum(O * G) against
    the oracle, with L, Q, K, V, O the only saved tensors."""
    from exact_tiled_attention_26_gb300.autograd import flash_attention
    Q, K, V, dO = _inputs(2, 2, Nq, Nk, 128, seed=1000 + Nq)
    q, k, v = (t.cuda().requires_grad_(True) for t in (Q, K, V))
    o = flash_attention(q, k, v, causal=causal, window=window)
    saved = o.grad_fn.saved_tensors
    assert [tuple(t.shape) for t in saved] == [(2, 2, Nq), (2, 2, Nq, 128), (2, 2, Nk, 128), (2, 2, Nk, 128),
                                               (2, 2, Nq, 128)]
    del saved
    o.backward(dO.cuda())
    ref = _oracle(Q, K, V, dO, causal, window)
    assert_close({"O": f64(o.detach().cpu()), "dQ": f64(q.grad.cpu()), "dK": f64(k.grad.cpu()),
                  "dV": f64(v.grad.cpu())}, {n: ref[n] for n in ("O", "dQ", "dK", "dV")}, "autograd")


def test_autograd_in_a_tiny_attention_layer():
    """The wrapper in place of an attention core inside a two-layer model (the
    drop-in of patched_model): the loss and every parameter gradient match the
    same model run with torch's own float32 attention to bf16 accuracy."""
    from exact_tiled_attention_26_gb300.autograd import flash_attention
    torch.manual_seed(0)
    B, T, D, H = 2, 256, 256, 2
    layers = [torch.nn.Linear(D, 3 * D).cuda() for _ in range(2)]

    def model(x, attn):
        for lin in layers:
            q, k, v = lin(x).split(D, dim=2)
            q, k, v = (t.view(B, T, H, D // H).transpose(1, 2) for t in (q, k, v))
            x = x + attn(q, k, v).transpose(1, 2).reshape(B, T, D)
        return x.square().mean()

    x = torch.randn(B, T, D, device="cuda")
    ours = lambda q, k, v: flash_attention(q.to(torch.bfloat16), k.to(torch.bfloat16), v.to(torch.bfloat16),
                                           causal=True).float()
    ref = lambda q, k, v: torch.nn.functional.scaled_dot_product_attention(
        q.to(torch.bfloat16).float(), k.to(torch.bfloat16).float(), v.to(torch.bfloat16).float(), is_causal=True)
    grads = []
    for attn in (ours, ref):
        for lin in layers:
            lin.zero_grad()
        loss = model(x, attn)
        loss.backward()
        grads.append((loss.item(), [p.grad.detach().clone() for lin in layers for p in lin.parameters()]))
    (l0, g0), (l1, g1) = grads
    assert abs(l0 - l1) <= 1e-2 * abs(l1)
    for a, b in zip(g0, g1):
        assert rel_frob(a.double().cpu().numpy(), b.double().cpu().numpy()) <= 3e-2
