"""GPU parity at the full workload sizes, in the launch configuration the benchmark
times.  The float64 oracle cannot afford every output at these lengths, so it
checks:
  * O, L, dQ and D on a seeded sample of 256 query rows of every head (each
    depends on its own row only);
  * dK and dV of whole heads (mid and long shapes) or of 256 sampled key rows of
    one head (very long shape), from the oracle's own L and D of every row;
  * identities that hold at any size: sum_j dV_j = sum_i dO_i, and
    sum_j dK_j = 0 (each row of dS sums to zero);
  * the exact number of tile pairs computed.
"""
import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si
from gpu_util import assert_close, check_D_elementwise, f64, lib, rel_frob, run_gpu

pytestmark = pytest.mark.gpu

_CACHE = {}


def _run(name, causal):
    key = (name, causal)
    if key not in _CACHE:
        _CACHE.clear()  # keep one full-size result in host memory at a time
        w = si.WORKLOADS[name]
        Q, K, V, dO = si.make_workload(w)
        got = run_gpu(Q, K, V, dO, causal, counter=True)
        _CACHE[key] = (w, (Q, K, V, dO), got)
    return _CACHE[key]


def _heads(t):
    B, H, N, d = t.shape
    return t.reshape(B * H, N, d)


CASES = [("mid_2x16x4096x128", False), ("mid_2x16x4096x128", True), ("long_1x32x8192x128", True),
         ("long_1x32x8192x128_qk4", True), ("vlong_1x32x32768x128", True)]
FULL_HEADS = {"mid_2x16x4096x128": [0, 31], "long_1x32x8192x128": [5], "long_1x32x8192x128_qk4": [5]}


@pytest.mark.parametrize("name,causal", CASES)
def test_sampled_rows(name, causal):
    w, (Q, K, V, dO), got = _run(name, causal)
    rows = si.sample_rows(w, 256)
    q, k, v, do = (f64(_heads(t)) for t in (Q, K, V, dO))
    O, L, dQ, D = oracle.rows_fwd_bwd(q, k, v, do, rows, causal)
    g = {n: f64(_heads(got[n]) if got[n].dim() == 4 else got[n].reshape(-1, w.N))[:, rows]
         for n in ("O", "L", "dQ", "D")}
    assert_close({"O": g["O"], "L": g["L"], "dQ": g["dQ"], "D": g["D"]}, {"O": O, "L": L, "dQ": dQ, "D": D},
                 f"{name} causal={causal} rows")


@pytest.mark.parametrize("name,causal", CASES)
def test_D_every_row_elementwise(name, causal):
    """The preprocess step at full size, every row of every head: D_i against
    sum_k dO_ik O_ik in float64 on the GPU's own bf16 O, within 1e-3 * max(1, |D_i|)."""
    w, (Q, K, V, dO), got = _run(name, causal)
    O, D, dOh = _heads(got["O"]), got["D"].reshape(-1, w.N), _heads(dO)
    for h in range(O.shape[0]):  # one head at a time keeps the float64 copies small
        check_D_elementwise(D[h], O[h], dOh[h])


@pytest.mark.parametrize("name,causal", [c for c in CASES if c[0] in FULL_HEADS])
def test_whole_heads(name, causal):
    w, (Q, K, V, dO), got = _run(name, causal)
    for h in FULL_HEADS[name]:
        q, k, v, do = (f64(_heads(t)[h]) for t in (Q, K, V, dO))
        O, L = oracle.standard_attention_fwd(q, k, v, causal)
        dQ, dK, dV, _ = oracle.standard_attention_bwd(q, k, v, do, causal)
        g = {n: f64(_heads(got[n])[h]) for n in ("O", "dQ", "dK", "dV")}
        g["L"] = f64(got["L"].reshape(-1, w.N)[h])
        assert_close(g, {"O": O, "L": L, "dQ": dQ, "dK": dK, "dV": dV}, f"{name} causal={causal} head {h}")


def test_vlong_sampled_key_rows():
    """dK, dV of 256 sampled key rows of head 0 at N = 32768, from the oracle's L
    and D of all 32768 query rows of that head."""
    name = "vlong_1x32x32768x128"
    w, (Q, K, V, dO), got = _run(name, True)
    q, k, v, do = (f64(_heads(t)[:1]) for t in (Q, K, V, dO))
    _, L, _, D = oracle.rows_fwd_bwd(q, k, v, do, np.arange(w.N), True)
    keys = si.sample_rows(w, 256)
    dK, dV = oracle.key_rows_bwd(q, k, v, do, L, D, keys, True)
    gK = f64(_heads(got["dK"])[:1])[:, keys]
    gV = f64(_heads(got["dV"])[:1])[:, keys]
    assert_close({"dK": gK, "dV": gV}, {"dK": dK, "dV": dV}, "vlong keys")


@pytest.mark.parametrize("name,causal", CASES)
def test_identities_every_head(name, causal):
    w, (Q, K, V, dO), got = _run(name, causal)
    dV = f64(_heads(got["dV"]))
    dK = f64(_heads(got["dK"]))
    sum_dO = f64(_heads(dO)).sum(axis=1)
    # sum over keys of dV_j = sum over queries of dO_i (the weights of each row sum to one)
    err_v = np.linalg.norm(dV.sum(axis=1) - sum_dO, axis=-1) / np.linalg.norm(sum_dO, axis=-1)
    assert err_v.max() <= 1e-2, err_v.max()
    # sum over keys of dK_j = 0, up to the rounding of dK and dS (relative to ||dK||_F)
    z = np.linalg.norm(dK.sum(axis=1), axis=-1) / np.linalg.norm(dK, axis=(1, 2))
    assert z.max() <= 5e-2, z.max()


@pytest.mark.parametrize("name,causal", CASES)
def test_tile_pairs_exact(name, causal):
    fa = lib()
    w, _, got = _run(name, causal)
    fwd, bwd = got["tiles"]
    assert fwd == w.B * w.H * fa.fa_tile_pairs(w.N, w.d, causal, 0)
    assert bwd == w.B * w.H * fa.fa_tile_pairs(w.N, w.d, causal, 1)
    _, br, bc = fa.fa_get_tile_config(w.d, 0)
    assert fwd == w.B * w.H * oracle.causal_tile_pairs(w.N, br, bc, causal)
    if causal and w.N % 128 == 0:
        T = w.N // 128
        assert fwd == w.B * w.H * T * (T + 1) // 2


def test_one_head_of_131072_rows():
    """One head of 131072 rows at d = 64, causal: 1024 query and key tiles, the
    largest tile and unit indices of any test.  O, L, dQ and D on 64 sampled rows
    (the first and last among them) against the oracle; dK and dV of the persistent
    backward bit-identical to the two-kernel backward's (the same bf16 P^T and dS^T,
    summed in the same order).  dQ of the two is summed in different orders over up
    to 1024 key tiles (in tensor memory, against fp32 reductions in L2); the fp32
    sums differ by ~1e-5 and flip the bf16 rounding of a fraction of a percent of
    the elements (2.9e-4 relative Frobenius measured), while one key tile's
    contribution missing or counted twice would move it by far more than 2e-3."""
    N, d = 131072, 64
    Q, K, V, dO = si.make_qkvdo(1, 1, N, d, seed=91)
    a = run_gpu(Q, K, V, dO, True, split=3)
    b = run_gpu(Q, K, V, dO, True, split=2)
    rng = np.random.default_rng(92)
    rows = np.unique(np.concatenate([[0, N - 1], rng.choice(N, 62, replace=False)]))
    q, k, v, do = (f64(t.reshape(1, N, d)) for t in (Q, K, V, dO))
    O, L, dQ, D = oracle.rows_fwd_bwd(q, k, v, do, rows, True)
    g = {n: f64(a[n].reshape(1, N, d) if a[n].dim() == 4 else a[n].reshape(1, N))[:, rows]
         for n in ("O", "L", "dQ", "D")}
    assert_close(g, {"O": O, "L": L, "dQ": dQ, "D": D}, "1x1x131072x64 causal rows")
    assert torch.equal(a["dK"], b["dK"]) and torch.equal(a["dV"], b["dV"])
    assert rel_frob(f64(a["dQ"]), f64(b["dQ"])) < 2e-3
