"""GPU parity of the forms of the d = 64 and d = 128 backward ("CS336 Assignment 2
notes" §1.4): form 1 (one kernel over key tiles, dQ reduced in an fp32 workspace),
form 2 (a key-tile kernel for dK, dV and a query-tile kernel for dQ) and form 3
(form 1 with one CTA per SM taking key tiles from a queue), each against
the float64 oracle, whichever of them is the library's default."""
import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si
from gpu_util import assert_close, f64, lib, rel_frob, run_gpu

pytestmark = pytest.mark.gpu

SPLITS = [1, 2, 3]


def _oracle_full(Q, K, V, dO, causal, scale=None):
    q, k, v, do = (f64(t) for t in (Q, K, V, dO))
    O, L = oracle.standard_attention_fwd(q, k, v, causal, scale)
    dQ, dK, dV, _ = oracle.standard_attention_bwd(q, k, v, do, causal, scale)
    return {"O": O, "L": L, "dQ": dQ, "dK": dK, "dV": dV}


def _grads(got):
    return {n: f64(got[n]) for n in ("dQ", "dK", "dV")}


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("split", SPLITS)
@pytest.mark.parametrize("N", [1, 7, 100, 128, 129, 300, 1000])
@pytest.mark.parametrize("causal", [False, True])
def test_ragged_lengths(d, split, N, causal):
    Q, K, V, dO = si.make_qkvdo(1, 2, N, d, seed=300 + N + d)
    got = run_gpu(Q, K, V, dO, causal, counter=True, split=split)
    ref = _oracle_full(Q, K, V, dO, causal)
    assert_close(_grads(got), {n: ref[n] for n in ("dQ", "dK", "dV")}, f"d={d} split={split} N={N} causal={causal}")
    # the key-tile kernel counts the pairs it computed: the closed form's
    assert got["tiles"][1] == 2 * lib().fa_tile_pairs(N, d, causal, 1)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("split", SPLITS)
@pytest.mark.parametrize("causal", [False, True])
def test_large_logits_and_scale(d, split, causal):
    """Scores ~16x unit variance and a scale other than 1/sqrt(d)."""
    Q, K, V, dO = si.make_qkvdo(2, 2, 640, d, seed=31, qk_mult=4.0)
    got = run_gpu(Q, K, V, dO, causal, scale=0.05, split=split)
    ref = _oracle_full(Q, K, V, dO, causal, scale=0.05)
    assert_close(_grads(got), {n: ref[n] for n in ("dQ", "dK", "dV")}, f"split={split} qk x4")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("split", [1, 3])
@pytest.mark.parametrize("causal", [False, True])
def test_workspace_content_on_entry_does_not_matter(d, split, causal):
    """The one-kernel forms reduce dQ into the fp32 workspace, which the call clears
    first: a workspace full of NaN bit patterns, then the same workspace as the
    first call left it, give the oracle's gradients for two different problems
    (ragged length, three heads)."""
    ws = torch.full((8 << 20,), 0xFF, dtype=torch.uint8, device="cuda")
    for seed in (61, 62):
        Q, K, V, dO = si.make_qkvdo(1, 3, 300, d, seed=seed + d)
        got = run_gpu(Q, K, V, dO, causal, split=split, ws=ws)
        ref = _oracle_full(Q, K, V, dO, causal)
        assert_close(_grads(got), {n: ref[n] for n in ("dQ", "dK", "dV")},
                     f"d={d} split={split} causal={causal} seed={seed}")


@pytest.mark.parametrize("causal", [False, True])
def test_mid_workload_sampled_rows_form2(causal):
    """The mid workload (2 x 16 heads x 4096 x 128) through form 2: dQ on sampled
    query rows, dK and dV of two whole heads."""
    w = si.WORKLOADS["mid_2x16x4096x128"]
    Q, K, V, dO = si.make_workload(w)
    got = run_gpu(Q, K, V, dO, causal, split=2)
    B, H, N, d = Q.shape
    hq = lambda t: f64(t.reshape(B * H, N, d))
    q, k, v, do = hq(Q), hq(K), hq(V), hq(dO)
    rows = si.sample_rows(w, 256)
    _, _, dQ, _ = oracle.rows_fwd_bwd(q, k, v, do, rows, causal)
    assert_close({"dQ": hq(got["dQ"])[:, rows]}, {"dQ": dQ}, "mid form 2 rows")
    for h in (0, 31):
        _, dK, dV, _ = oracle.standard_attention_bwd(q[h], k[h], v[h], do[h], causal)
        assert_close({"dK": hq(got["dK"])[h], "dV": hq(got["dV"])[h]}, {"dK": dK, "dV": dV}, f"mid form 2 head {h}")


@pytest.mark.parametrize("causal", [False, True])
def test_forms_agree_and_form2_is_deterministic(causal):
    """Both forms compute the same gradients (to the rounding of their different
    summation orders); form 2 has no atomics, so repeated calls are bitwise equal."""
    Q, K, V, dO = si.make_qkvdo(1, 4, 2048, 128, seed=41)
    a = run_gpu(Q, K, V, dO, causal, split=1)
    b = run_gpu(Q, K, V, dO, causal, split=2)
    c = run_gpu(Q, K, V, dO, causal, split=2)
    for n in ("dQ", "dK", "dV"):
        assert rel_frob(f64(b[n]), f64(a[n])) <= 1e-2, n
        assert (b[n] == c[n]).all(), n


@pytest.mark.parametrize("causal", [False, True])
def test_small_workload_form2_d64(causal):
    """The small workload (4 x 8 heads x 1024 x 64) through form 2, every gradient."""
    w = si.WORKLOADS["small_4x8x1024x64"]
    Q, K, V, dO = si.make_workload(w)
    got = run_gpu(Q, K, V, dO, causal, counter=True, split=2)
    ref = _oracle_full(Q, K, V, dO, causal)
    assert_close(_grads(got), {n: ref[n] for n in ("dQ", "dK", "dV")}, "small form 2")
    assert got["tiles"][1] == 32 * lib().fa_tile_pairs(1024, 64, causal, 1)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("B,H,N,causal,window", [(2, 3, 1000, True, 0), (1, 5, 700, False, 0), (3, 2, 777, True, 100),
                                                 (4, 40, 256, True, 0), (2, 16, 4096, True, 0)])
def test_persistent_form_equals_form1(B, H, N, causal, window, d):
    """Form 3 runs each key tile exactly as form 1 does: dK and dV agree bit for bit;
    dQ is summed in fp32 reductions whose order varies."""
    Q, K, V, dO = si.make_qkvdo(B, H, N, d, seed=2200 + N + window)
    a = run_gpu(Q, K, V, dO, causal, counter=True, split=1, window=window)
    b = run_gpu(Q, K, V, dO, causal, counter=True, split=3, window=window)
    assert torch.equal(a["dK"], b["dK"]) and torch.equal(a["dV"], b["dV"])
    assert rel_frob(f64(b["dQ"]), f64(a["dQ"])) <= 2e-3
    assert a["tiles"] == b["tiles"]
