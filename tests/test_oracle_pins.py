"""Pins for the float64 oracle: each check ties it to something other than itself.

Sources: "CS349E lecture 11: 03_flash_backward.py" (demo1_gradcheck,
demo4_causal), "CS324 lecture 8: 03_online_softmax_and_flash.py"
(demo2_online, demo3_forward, demo4_backward) and "CS336 Assignment 2 notes"
§1.2-§1.4 (FlashAttention-2 forward, whole-tile skip, Equations 13-19).
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import attention as oa

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(seed, *shape):
    return np.random.default_rng(seed).standard_normal(shape)


def _torch_reference(Q, K, V, dO, causal, scale):
    """torch fp64 autograd through softmax(Q K^T s) V: an independent library check
    (the cross-check of the CS324 lecture 8 script, demo4_backward)."""
    tq, tk, tv = (torch.tensor(a, requires_grad=True) for a in (Q, K, V))
    s = tq @ tk.transpose(-2, -1) * scale
    if causal:
        n, m = s.shape[-2:]
        s = s.masked_fill(~torch.tril(torch.ones(n, m, dtype=torch.bool)), float("-inf"))
    lse = torch.logsumexp(s, dim=-1)
    out = torch.softmax(s, dim=-1) @ tv
    out.backward(torch.tensor(dO))
    return (out.detach().numpy(), lse.detach().numpy(), tq.grad.numpy(), tk.grad.numpy(),
            tv.grad.numpy())


# ---------------------------------------------------------------- online softmax

def _read_trace():
    x, block, trace = None, None, []
    with open(os.path.join(GOLDEN, "online_softmax_trace.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if line.startswith("x:"):
                x = [float(v) for v in line[2:].split()]
            elif line.startswith("block:"):
                block = int(line.split()[1])
            else:
                n, m = line.split()
                trace.append((int(n), float(m)))
    return np.array(x), block, trace


def test_online_softmax_worked_trace():
    x, block, golden = _read_trace()
    out, trace = oracle.online_softmax(x, block)
    assert [(n, m) for n, m, _ in trace] == golden
    for n, m, l in trace:
        # denominator after reading n numbers: closed form sum_{k<n} exp(x_k - m)
        assert l == pytest.approx(math.fsum(math.exp(v - m) for v in x[:n]), rel=1e-15)
    assert trace[-1][2] == pytest.approx(math.fsum(math.exp(v - 6.0) for v in x), rel=1e-15)
    ref = np.exp(x - x.max()) / np.exp(x - x.max()).sum()
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-16)


def test_online_softmax_block_sizes_agree():
    x = _rand(3, 1000) * 30
    ref = np.exp(x - x.max()) / np.exp(x - x.max()).sum()
    for block in (1, 3, 64, 1000, 4096):
        out, _ = oracle.online_softmax(x, block)
        np.testing.assert_allclose(out, ref, rtol=1e-13, atol=1e-300)


# ---------------------------------------------------------------- plain definition

def _brute_attention(Q, K, V, causal, scale):
    """Pure-Python triple loop with math.exp: no numpy matmul, no max trick."""
    N, d = Q.shape
    O = np.zeros((N, V.shape[1]))
    L = np.zeros(N)
    for i in range(N):
        w = []
        for j in range(K.shape[0]):
            if causal and j > i:
                w.append(0.0)
                continue
            w.append(math.exp(sum(Q[i, c] * K[j, c] for c in range(d)) * scale))
        z = math.fsum(w)
        L[i] = math.log(z)
        for c in range(V.shape[1]):
            O[i, c] = math.fsum(w[j] * V[j, c] for j in range(K.shape[0])) / z
    return O, L


@pytest.mark.parametrize("causal", [False, True])
def test_standard_fwd_brute_force_tiny(causal):
    Q, K, V = _rand(10, 7, 3), _rand(11, 7, 3), _rand(12, 7, 3)
    O, L = oracle.standard_attention_fwd(Q, K, V, causal, scale=0.7)
    Ob, Lb = _brute_attention(Q, K, V, causal, 0.7)
    np.testing.assert_allclose(O, Ob, atol=1e-14)
    np.testing.assert_allclose(L, Lb, atol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
def test_standard_matches_torch_autograd(causal):
    # N = 128, d = 16 as in the CS324 lecture 8 backward demo; two heads
    Q, K, V, dO = (_rand(20 + i, 2, 128, 16) for i in range(4))
    s = 1 / math.sqrt(16)
    O, L = oracle.standard_attention_fwd(Q, K, V, causal)
    dQ, dK, dV, _ = oracle.standard_attention_bwd(Q, K, V, dO, causal)
    tO, tL, tdQ, tdK, tdV = _torch_reference(Q, K, V, dO, causal, s)
    for a, b in ((O, tO), (L, tL), (dQ, tdQ), (dK, tdK), (dV, tdV)):
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_standard_matches_torch_sdpa(causal):
    Q, K, V = (_rand(30 + i, 1, 3, 200, 32) for i in range(3))
    O, _ = oracle.standard_attention_fwd(Q, K, V, causal)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.tensor(Q), torch.tensor(K), torch.tensor(V), is_causal=causal).numpy()
    np.testing.assert_allclose(O, ref, rtol=0, atol=1e-12)


def test_large_logits_stay_finite_and_exact():
    # Q and K scaled by 4: scores ~16x larger than unit variance (large-logit stress)
    Q, K, V, dO = (_rand(40 + i, 1, 256, 128) for i in range(4))
    Q, K = 4 * Q, 4 * K
    O, L = oracle.standard_attention_fwd(Q, K, V, True)
    dQ, dK, dV, _ = oracle.standard_attention_bwd(Q, K, V, dO, True)
    assert np.isfinite(O).all() and np.isfinite(L).all() and np.isfinite(dK).all()
    tO, tL, tdQ, tdK, tdV = _torch_reference(Q, K, V, dO, True, 1 / math.sqrt(128))
    np.testing.assert_allclose(O, tO, atol=1e-11)
    np.testing.assert_allclose(L, tL, atol=1e-11)
    for a, b in ((dQ, tdQ), (dK, tdK), (dV, tdV)):
        np.testing.assert_allclose(a, b, atol=1e-9 * max(1.0, np.abs(b).max()))


@pytest.mark.parametrize("causal", [False, True])
def test_central_differences(causal):
    """Loss = sum(O * G); 6 random entries each of Q, K and V (18 in all), eps = 1e-6,
    N = 48, d = 16 as in the gradient check of CS349E lecture 11 (demo1_gradcheck)."""
    rng = np.random.default_rng(0)
    N, d = 48, 16
    Q, K, V = (rng.standard_normal((N, d)) for _ in range(3))
    G = rng.standard_normal((N, d))
    dQ, dK, dV, _ = oracle.standard_attention_bwd(Q, K, V, G, causal)
    grads = {"Q": dQ, "K": dK, "V": dV}
    eps = 1e-6
    worst = 0.0
    for name in ("Q", "K", "V"):
        for _ in range(6):
            r, c = int(rng.integers(N)), int(rng.integers(d))
            args_p = {"Q": Q, "K": K, "V": V}
            args_m = dict(args_p)
            Xp, Xm = args_p[name].copy(), args_p[name].copy()
            Xp[r, c] += eps
            Xm[r, c] -= eps
            args_p[name], args_m[name] = Xp, Xm
            fp = np.sum(oracle.standard_attention_fwd(args_p["Q"], args_p["K"], args_p["V"], causal)[0] * G)
            fm = np.sum(oracle.standard_attention_fwd(args_m["Q"], args_m["K"], args_m["V"], causal)[0] * G)
            worst = max(worst, abs((fp - fm) / (2 * eps) - grads[name][r, c]))
    assert worst < 1e-7, worst


def test_D_identity():
    """sum_j P_ij dP_ij == rowsum(dO * O) (CS349E lecture 11 demo1 observations;
    CS336 notes §1.4 Eq 17)."""
    for causal in (False, True):
        Q, K, V, dO = (_rand(50 + i, 2, 2, 300, 64) for i in range(4))
        O, _ = oracle.standard_attention_fwd(Q, K, V, causal)
        _, _, _, D = oracle.standard_attention_bwd(Q, K, V, dO, causal)
        np.testing.assert_allclose(D, (dO * O).sum(-1), rtol=0, atol=1e-12)


def test_single_key_closed_form():
    """N = 1: the only weight is 1, so O = V and L = s q.k."""
    Q, K, V, dO = (_rand(60 + i, 3, 1, 32) for i in range(4))
    O, L = oracle.standard_attention_fwd(Q, K, V, True, scale=0.3)
    np.testing.assert_allclose(O, V, atol=1e-15)
    np.testing.assert_allclose(L, 0.3 * (Q * K).sum(-1), atol=1e-15)
    dQ, dK, dV, _ = oracle.standard_attention_bwd(Q, K, V, dO, True, scale=0.3)
    np.testing.assert_allclose(dV, dO, atol=1e-15)  # dV = P^T dO with P = 1
    np.testing.assert_allclose(dQ, 0 * dQ, atol=1e-15)  # softmax of one score is constant
    np.testing.assert_allclose(dK, 0 * dK, atol=1e-15)


@pytest.mark.parametrize("causal", [False, True])
def test_equal_keys_closed_form(causal):
    """Every key row equal: P is uniform over the visible keys.  Then O_i is the mean
    of the visible V rows, L_i = s q_i.k + ln(#visible), dV_j = sum_{i sees j} dO_i /
    #visible(i), and dQ = 0 because each row of dS sums to zero."""
    N, d, s = 37, 8, 0.5
    Q, V, dO = _rand(70, N, d), _rand(71, N, d), _rand(72, N, d)
    k = _rand(73, d)
    K = np.tile(k, (N, 1))
    O, L = oracle.standard_attention_fwd(Q, K, V, causal, scale=s)
    dQ, _, dV, _ = oracle.standard_attention_bwd(Q, K, V, dO, causal, scale=s)
    cnt = np.arange(1, N + 1) if causal else np.full(N, N)
    Oref = np.cumsum(V, 0) / cnt[:, None] if causal else np.tile(V.mean(0), (N, 1))
    np.testing.assert_allclose(O, Oref, atol=1e-13)
    np.testing.assert_allclose(L, s * Q @ k + np.log(cnt), atol=1e-13)
    w = dO / cnt[:, None]
    dVref = np.cumsum(w[::-1], 0)[::-1] if causal else np.tile(w.sum(0), (N, 1))
    np.testing.assert_allclose(dV, dVref, atol=1e-13)
    np.testing.assert_allclose(dQ, 0 * dQ, atol=1e-13)


def test_row_subsets_match_full():
    Q, K, V, dO = (_rand(80 + i, 2, 500, 32) for i in range(4))
    rows = np.array([0, 3, 255, 256, 499])
    for causal in (False, True):
        O, L = oracle.standard_attention_fwd(Q, K, V, causal)
        dQ, dK, dV, D = oracle.standard_attention_bwd(Q, K, V, dO, causal)
        Or, Lr, dQr, Dr = oracle.rows_fwd_bwd(Q, K, V, dO, rows, causal)
        np.testing.assert_allclose(Or, O[:, rows], atol=1e-13)
        np.testing.assert_allclose(Lr, L[:, rows], atol=1e-13)
        np.testing.assert_allclose(dQr, dQ[:, rows], atol=1e-13)
        np.testing.assert_allclose(Dr, D[:, rows], atol=1e-13)
        dKr, dVr = oracle.key_rows_bwd(Q, K, V, dO, L, D, rows, causal)
        np.testing.assert_allclose(dKr, dK[:, rows], atol=1e-12)
        np.testing.assert_allclose(dVr, dV[:, rows], atol=1e-12)


# ---------------------------------------------------------------- tiled method

@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Br,Bc", [(16, 16), (32, 64), (64, 32), (128, 128), (16, 12), (64, 64)])
def test_tiled_forward_matches_standard(causal, Br, Bc):
    """N = 256, d = 32: the tile sizes of CS324 lecture 8 demo3_forward, plus the
    non-dividing 16 x 12 tiles of the CS349E gradient check; the pages report
    differences of order 1e-16."""
    Q, K, V = (_rand(90 + i, 256, 32) for i in range(3))
    O, L = oracle.standard_attention_fwd(Q, K, V, causal)
    Ot, Lt, tiles = oracle.flash_forward_tiled(Q, K, V, Br, Bc, causal)
    np.testing.assert_allclose(Ot, O, rtol=0, atol=1e-13)
    np.testing.assert_allclose(Lt, L, rtol=0, atol=1e-13)
    assert tiles == oracle.causal_tile_pairs(256, Br, Bc, causal)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,d,Br,Bc", [(128, 16, 32, 32), (48, 16, 16, 12), (100, 8, 64, 32)])
def test_tiled_backward_matches_standard(causal, N, d, Br, Bc):
    Q, K, V, dO = (_rand(100 + i, N, d) for i in range(4))
    O, L = oracle.standard_attention_fwd(Q, K, V, causal)
    dQ, dK, dV, D = oracle.standard_attention_bwd(Q, K, V, dO, causal)
    tdQ, tdK, tdV, tD, tiles = oracle.flash_backward_tiled(Q, K, V, O, dO, L, Br, Bc, causal)
    for a, b in ((tdQ, dQ), (tdK, dK), (tdV, dV), (tD, D)):
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)
    assert tiles == oracle.causal_tile_pairs(N, Br, Bc, causal)


# ---------------------------------------------------------------- tile counts

def _brute_pairs(N, Br, Bc, causal):
    """Count tile pairs holding at least one visible (query, key) entry."""
    n = 0
    for i0 in range(0, N, Br):
        for j0 in range(0, N, Bc):
            rows = range(i0, min(N, i0 + Br))
            cols = range(j0, min(N, j0 + Bc))
            if not causal or any(c <= r for r in rows for c in cols):
                n += 1
    return n


@pytest.mark.parametrize("N", [1, 7, 64, 100, 256, 257, 300])
@pytest.mark.parametrize("Br,Bc", [(64, 64), (128, 128), (64, 128), (128, 64), (16, 12)])
def test_tile_pairs_brute_force(N, Br, Bc):
    for causal in (False, True):
        assert oracle.causal_tile_pairs(N, Br, Bc, causal) == _brute_pairs(N, Br, Bc, causal)


def test_causal_fraction_table():
    with open(os.path.join(GOLDEN, "causal_tile_fraction.txt")) as f:
        rows = [list(map(int, l.split())) for l in f if l.strip() and not l.startswith("#")]
    for N, Br, Bc, pairs, total in rows:
        T = N // Bc
        assert oracle.causal_tile_pairs(N, Br, Bc, True) == pairs == T * (T + 1) // 2
        assert oracle.causal_tile_pairs(N, Br, Bc, False) == total
        assert pairs / total == pytest.approx(0.5 + 0.5 / T, rel=1e-15)


def test_tiny_case_tile_count_at_64_tiles():
    """The tiny case (N = 256) at the 64 x 64 tiles it is written for: 4 tile rows,
    so 4 * 5 / 2 = 10 of the 16 pairs are computed with the causal mask.  The GPU
    runs 128 x 128 tiles there; this count is pinned on the CPU tiled oracle."""
    Q, K, V = (_rand(95 + i, 256, 32) for i in range(3))
    assert oracle.flash_forward_tiled(Q, K, V, 64, 64, True)[2] == oracle.causal_tile_pairs(256, 64, 64, True) == 10
    assert oracle.flash_forward_tiled(Q, K, V, 64, 64, False)[2] == oracle.causal_tile_pairs(256, 64, 64, False) == 16


def test_flop_count():
    # 12 N^2 d standard vs 14 N^2 d recompute for N = 1024, d = 64 (805.3 M vs 939.5 M)
    f, b = oracle.attention_flops(1024, 64, False)
    assert f + b == 14 * 1024 * 1024 * 64
    assert round((f + b) / 1e6, 1) == 939.5
    fc, bc = oracle.attention_flops(1024, 64, True)
    assert (fc, bc) == (f / 2, b / 2)


# ---------------------------------------------------------------- planted mistakes

def _pins_hold():
    """A compact run of the pins above; returns False on the first failure."""
    try:
        test_standard_fwd_brute_force_tiny(True)
        test_standard_matches_torch_autograd(True)
        test_central_differences(True)
        test_equal_keys_closed_form(True)
    except AssertionError:
        return False
    return True


def test_pins_catch_a_flipped_mask(monkeypatch):
    orig = oa._scores

    def flipped(q_rows, row_ids, K, causal, s, off=0, window=0):
        S = (q_rows @ K.T) * s
        if causal:
            cols = np.arange(K.shape[0])[None, :]
            S = np.where(cols < row_ids[:, None] + off, -np.inf, S)  # wrong orientation
        return S
    assert _pins_hold()
    monkeypatch.setattr(oa, "_scores", flipped)
    assert not _pins_hold()
    monkeypatch.setattr(oa, "_scores", orig)


def test_pins_catch_a_dropped_term(monkeypatch):
    real_bwd = oa.standard_attention_bwd

    def no_D(Q, K, V, dO, causal=False, scale=None):
        # plausible slip: dS = P * dP with the rowsum term D dropped.  Then
        # dQ' = dQ + D_i (P K)_i s, where (P K)_i is attention with K as values.
        dQ, dK, dV, D = real_bwd(Q, K, V, dO, causal, scale)
        s = 1 / math.sqrt(np.shape(Q)[-1]) if scale is None else scale
        PK, _ = oa.standard_attention_fwd(Q, K, K, causal, scale)
        return dQ + (D[..., None] * PK) * s, dK, dV, D
    monkeypatch.setattr(oracle, "standard_attention_bwd", no_D)
    assert not _pins_hold()


def test_pins_catch_a_missing_log(monkeypatch):
    monkeypatch.setattr(oa, "_logsumexp_rows", lambda S: S.max(axis=1))
    assert not _pins_hold()
