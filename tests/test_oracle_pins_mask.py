"""Pins for the oracle's general mask: a sliding window ("CS324 lecture 8:
03_online_softmax_and_flash.py", window_attention_torch: query i sees itself and
the w - 1 keys before it) and N_q != N_k with the queries at the last N_q
positions of the key sequence ("CS349E lecture 11: 03_flash_backward.py",
demo4_causal observation 3: one decoded token sees the whole cache).  Each check
ties the oracle to something other than itself: a pure-Python loop, torch fp64
autograd with an explicitly built mask, closed forms, reductions to the
unmasked/causal cases, central differences, and brute-force tile counts."""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import attention as oa


def _rand(seed, *shape):
    return np.random.default_rng(seed).standard_normal(shape)


def _hidden(Nq, Nk, causal, window):
    """The mask written out entry by entry: position p = i + Nk - Nq."""
    off = Nk - Nq
    return [[(causal and j > i + off) or (window > 0 and j <= i + off - window) for j in range(Nk)]
            for i in range(Nq)]


def _brute(Q, K, V, causal, window, scale):
    """Pure-Python loops with math.exp (no matmul, no max trick)."""
    Nq, d = Q.shape
    Nk = K.shape[0]
    hid = _hidden(Nq, Nk, causal, window)
    O = np.zeros((Nq, V.shape[1]))
    L = np.zeros(Nq)
    for i in range(Nq):
        w = [0.0 if hid[i][j] else math.exp(sum(Q[i, c] * K[j, c] for c in range(d)) * scale) for j in range(Nk)]
        z = math.fsum(w)
        L[i] = math.log(z)
        for c in range(V.shape[1]):
            O[i, c] = math.fsum(w[j] * V[j, c] for j in range(Nk)) / z
    return O, L


def _torch_masked(Q, K, V, dO, causal, window, scale):
    """torch fp64 autograd through softmax with the mask built as in
    window_attention_torch (cols > rows, cols <= rows - w), rows shifted to their
    positions."""
    tq, tk, tv = (torch.tensor(a, requires_grad=True) for a in (Q, K, V))
    Nq, Nk = Q.shape[-2], K.shape[-2]
    s = tq @ tk.transpose(-2, -1) * scale
    rows = torch.arange(Nq)[:, None] + (Nk - Nq)
    cols = torch.arange(Nk)[None, :]
    hide = torch.zeros(Nq, Nk, dtype=torch.bool)
    if causal:
        hide |= cols > rows
    if window > 0:
        hide |= cols <= rows - window
    s = s.masked_fill(hide, float("-inf"))
    lse = torch.logsumexp(s, dim=-1)
    out = torch.softmax(s, dim=-1) @ tv
    out.backward(torch.tensor(dO))
    return (out.detach().numpy(), lse.detach().numpy(), tq.grad.numpy(), tk.grad.numpy(), tv.grad.numpy())


CASES = [  # (Nq, Nk, causal, window)
    (9, 9, True, 3), (9, 9, True, 1), (5, 9, True, 0), (5, 9, True, 4), (1, 9, True, 0), (1, 9, True, 2),
    (9, 5, False, 0), (5, 9, False, 0), (9, 9, True, 20),
]


@pytest.mark.parametrize("Nq,Nk,causal,window", CASES)
def test_masked_forward_brute_force(Nq, Nk, causal, window):
    Q, K, V = _rand(1, Nq, 3), _rand(2, Nk, 3), _rand(3, Nk, 3)
    O, L = oracle.standard_attention_fwd(Q, K, V, causal, scale=0.8, window=window)
    Ob, Lb = _brute(Q, K, V, causal, window, 0.8)
    np.testing.assert_allclose(O, Ob, atol=1e-14)
    np.testing.assert_allclose(L, Lb, atol=1e-14)


@pytest.mark.parametrize("Nq,Nk,causal,window", CASES + [(200, 300, True, 64), (300, 300, True, 37)])
def test_masked_matches_torch_autograd(Nq, Nk, causal, window):
    Q, K, V = _rand(4, 2, Nq, 16), _rand(5, 2, Nk, 16), _rand(6, 2, Nk, 16)
    dO = _rand(7, 2, Nq, 16)
    O, L = oracle.standard_attention_fwd(Q, K, V, causal, window=window)
    dQ, dK, dV, _ = oracle.standard_attention_bwd(Q, K, V, dO, causal, window=window)
    ref = _torch_masked(Q, K, V, dO, causal, window, 1 / math.sqrt(16))
    for a, b in zip((O, L, dQ, dK, dV), ref):
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)


def test_window_one_closed_form():
    """w = 1: each query sees only itself, so O = V, L = s q.k, dV = dO and
    dQ = dK = 0 (dS = P (dP - D) with P = 1 and D = dP_ii)."""
    Q, K, V, dO = (_rand(10 + i, 3, 40, 8) for i in range(4))
    s = 0.3
    O, L = oracle.standard_attention_fwd(Q, K, V, True, scale=s, window=1)
    dQ, dK, dV, _ = oracle.standard_attention_bwd(Q, K, V, dO, True, scale=s, window=1)
    np.testing.assert_allclose(O, V, atol=1e-15)
    np.testing.assert_allclose(L, s * (Q * K).sum(-1), atol=1e-14)
    np.testing.assert_allclose(dV, dO, atol=1e-15)
    assert np.abs(dQ).max() < 1e-15 and np.abs(dK).max() < 1e-15


def test_window_covering_everything_is_causal():
    Q, K, V, dO = (_rand(20 + i, 2, 130, 16) for i in range(4))
    for w in (130, 131, 1000):
        a = oracle.standard_attention_fwd(Q, K, V, True, window=w)
        b = oracle.standard_attention_fwd(Q, K, V, True)
        np.testing.assert_array_equal(a[0], b[0])
        ga = oracle.standard_attention_bwd(Q, K, V, dO, True, window=w)
        gb = oracle.standard_attention_bwd(Q, K, V, dO, True)
        for x, y in zip(ga, gb):
            np.testing.assert_array_equal(x, y)


def test_decode_row_sees_every_key():
    """N_q = 1 with the causal mask: the new token sees the whole cache, so the
    result is the unmasked one (CS349E lecture 11, demo4_causal observation 3)."""
    Q, K, V, dO = _rand(30, 4, 1, 32), _rand(31, 4, 77, 32), _rand(32, 4, 77, 32), _rand(33, 4, 1, 32)
    a = oracle.standard_attention_fwd(Q, K, V, True)
    b = oracle.standard_attention_fwd(Q, K, V, False)
    np.testing.assert_allclose(a[0], b[0], atol=1e-15)
    ga = oracle.standard_attention_bwd(Q, K, V, dO, True)
    gb = oracle.standard_attention_bwd(Q, K, V, dO, False)
    for x, y in zip(ga, gb):
        np.testing.assert_allclose(x, y, atol=1e-15)


@pytest.mark.parametrize("window", [0, 5, 40])
def test_chunked_prefill_equals_full_sequence(window):
    """The last m queries against all keys (bottom-right alignment) are the last
    m rows of the full causal attention; their gradients are those of the full
    problem with dO zero on the first rows."""
    N, m = 90, 23
    Q, K, V, dO = (_rand(40 + i, 2, N, 16) for i in range(4))
    Of, Lf = oracle.standard_attention_fwd(Q, K, V, True, window=window)
    Oc, Lc = oracle.standard_attention_fwd(Q[:, -m:], K, V, True, window=window)
    np.testing.assert_allclose(Oc, Of[:, -m:], atol=1e-14)
    np.testing.assert_allclose(Lc, Lf[:, -m:], atol=1e-14)
    dOz = dO.copy()
    dOz[:, :-m] = 0
    gf = oracle.standard_attention_bwd(Q, K, V, dOz, True, window=window)
    gc = oracle.standard_attention_bwd(Q[:, -m:], K, V, dO[:, -m:], True, window=window)
    np.testing.assert_allclose(gc[0], gf[0][:, -m:], atol=1e-13)
    np.testing.assert_allclose(gc[1], gf[1], atol=1e-13)
    np.testing.assert_allclose(gc[2], gf[2], atol=1e-13)


@pytest.mark.parametrize("Nq,Nk", [(37, 200), (200, 37)])
def test_unmasked_unequal_lengths_match_sdpa(Nq, Nk):
    Q, K, V = _rand(50, 1, 2, Nq, 32), _rand(51, 1, 2, Nk, 32), _rand(52, 1, 2, Nk, 32)
    O, _ = oracle.standard_attention_fwd(Q, K, V, False)
    ref = torch.nn.functional.scaled_dot_product_attention(torch.tensor(Q), torch.tensor(K), torch.tensor(V)).numpy()
    np.testing.assert_allclose(O, ref, atol=1e-12)


def test_windowed_central_differences():
    rng = np.random.default_rng(60)
    Nq, Nk, d, w = 20, 33, 8, 6
    Q, K, V = rng.standard_normal((Nq, d)), rng.standard_normal((Nk, d)), rng.standard_normal((Nk, d))
    G = rng.standard_normal((Nq, d))
    grads = dict(zip("QKV", oracle.standard_attention_bwd(Q, K, V, G, True, window=w)[:3]))
    eps, worst = 1e-6, 0.0
    for name in "QKV":
        for _ in range(6):
            args = {"Q": Q, "K": K, "V": V}
            r, c = int(rng.integers(args[name].shape[0])), int(rng.integers(d))
            p, m = dict(args), dict(args)
            p[name], m[name] = args[name].copy(), args[name].copy()
            p[name][r, c] += eps
            m[name][r, c] -= eps
            fp = np.sum(oracle.standard_attention_fwd(p["Q"], p["K"], p["V"], True, window=w)[0] * G)
            fm = np.sum(oracle.standard_attention_fwd(m["Q"], m["K"], m["V"], True, window=w)[0] * G)
            worst = max(worst, abs((fp - fm) / (2 * eps) - grads[name][r, c]))
    assert worst < 1e-7, worst


@pytest.mark.parametrize("Nq,Nk,causal,window,Br,Bc", [
    (130, 130, True, 17, 32, 32), (130, 130, True, 64, 64, 32), (50, 130, True, 0, 16, 16),
    (50, 130, True, 30, 32, 16), (1, 130, True, 0, 16, 16), (130, 50, False, 0, 32, 64)])
def test_tiled_passes_with_masks_match_standard(Nq, Nk, causal, window, Br, Bc):
    Q, K, V, dO = _rand(70, 2, Nq, 16), _rand(71, 2, Nk, 16), _rand(72, 2, Nk, 16), _rand(73, 2, Nq, 16)
    O, L = oracle.standard_attention_fwd(Q, K, V, causal, window=window)
    Ot, Lt, tiles_f = oracle.flash_forward_tiled(Q, K, V, Br, Bc, causal, window=window)
    np.testing.assert_allclose(Ot, O, atol=1e-13)
    np.testing.assert_allclose(Lt, L, atol=1e-13)
    dQ, dK, dV, _ = oracle.standard_attention_bwd(Q, K, V, dO, causal, window=window)
    tQ, tK, tV, _, tiles_b = oracle.flash_backward_tiled(Q, K, V, O, dO, L, Br, Bc, causal, window=window)
    for a, b in ((tQ, dQ), (tK, dK), (tV, dV)):
        np.testing.assert_allclose(a, b, atol=1e-12)
    n = oracle.causal_tile_pairs(Nq, Br, Bc, causal, Nk=Nk, window=window)
    assert tiles_f == tiles_b == 2 * n


def _brute_tile_pairs(Nq, Nk, Br, Bc, causal, window):
    hid = np.array(_hidden(Nq, Nk, causal, window))
    n = 0
    for i0 in range(0, Nq, Br):
        for j0 in range(0, Nk, Bc):
            n += int((~hid[i0:i0 + Br, j0:j0 + Bc]).any())
    return n


@pytest.mark.parametrize("Nq,Nk", [(256, 256), (300, 300), (100, 300), (1, 300), (129, 1000)])
@pytest.mark.parametrize("window", [0, 1, 64, 100, 128, 129, 1000])
@pytest.mark.parametrize("Br,Bc", [(128, 128), (64, 128), (16, 12)])
def test_two_sided_tile_skip_brute_force(Nq, Nk, window, Br, Bc):
    assert oracle.causal_tile_pairs(Nq, Br, Bc, True, Nk=Nk, window=window) == \
        _brute_tile_pairs(Nq, Nk, Br, Bc, True, window)


@pytest.mark.parametrize("Nq,Nk,causal,window", CASES + [(300, 300, True, 64), (1, 1000, True, 0)])
def test_visible_pairs_brute_force(Nq, Nk, causal, window):
    assert oracle.visible_pairs(Nq, Nk, causal, window) == int((~np.array(_hidden(Nq, Nk, causal, window))).sum())


def test_sliding_window_tile_count_example():
    """N = 8192, w = 1024, 128 x 128 tiles: query tile i sees key tiles
    max(0, i - 8) .. i, i.e. 1 + 2 + ... + 8 for the first eight tiles and 9
    for each of the other 56: 36 + 504 = 540 of the causal 2080."""
    assert oracle.causal_tile_pairs(8192, 128, 128, True, window=1024) == 540
    assert oracle.visible_pairs(8192, 8192, True, 1024) == 1024 * 8192 - 1024 * 1023 // 2


def test_mask_arguments_rejected():
    Q = np.zeros((1, 4, 8))
    with pytest.raises(ValueError):
        oracle.standard_attention_fwd(Q, Q[:, :2], Q[:, :2], True)   # causal with N_q > N_k
    with pytest.raises(ValueError):
        oracle.standard_attention_fwd(Q, Q, Q, False, window=2)      # window without causal


def test_pins_catch_a_window_off_by_one(monkeypatch):
    """A window that keeps one key too many (j >= p - w instead of j > p - w)."""
    def loose(row_ids, cols, causal, off=0, window=0):
        pos = row_ids[:, None] + off
        hide = np.zeros((len(row_ids), len(cols)), dtype=bool)
        if causal:
            hide |= cols[None, :] > pos
        if window > 0:
            hide |= cols[None, :] < pos - window
        return hide
    monkeypatch.setattr(oa, "_masked", loose)
    with pytest.raises(AssertionError):
        test_window_one_closed_form()
    with pytest.raises(AssertionError):
        test_masked_forward_brute_force(9, 9, True, 3)


def test_pins_catch_top_left_alignment(monkeypatch):
    """Aligning unequal lengths top-left (offset 0) instead of bottom-right."""
    monkeypatch.setattr(oa, "_check_mask", lambda Nq, Nk, causal, window: 0)
    with pytest.raises(AssertionError):
        test_decode_row_sees_every_key()
    with pytest.raises(AssertionError):
        test_chunked_prefill_equals_full_sequence(0)
