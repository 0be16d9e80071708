"""GPU checks of the building blocks: the tensor-core operand paths, the bounded
waits, and the bandwidth-bound preprocess kernel."""
import numpy as np
import pytest
import torch

import seeded_inputs as si
from gpu_util import lib, stream

pytestmark = pytest.mark.gpu


def _bf16(rng, *shape):
    return torch.from_numpy(rng.standard_normal(shape, dtype=np.float32)).to(torch.bfloat16)


@pytest.mark.parametrize("mode", [0, 1, 2, 3, 4])
@pytest.mark.parametrize("K", [32, 64, 128])
@pytest.mark.parametrize("N", [32, 64, 128])
def test_umma_operand_paths(mode, K, N):
    """One 128 x N x K product per operand layout, against a float64 CPU product
    of the same bf16 values (fp32 accumulation: tolerance 1e-4 relative)."""
    fa = lib()
    rng = np.random.default_rng(1000 + 100 * mode + K + N)
    a_shape = (K, 128) if mode in (3, 4) else (128, K)
    b_shape = (K, N) if mode in (1, 2, 4) else (N, K)
    A, B = _bf16(rng, *a_shape), _bf16(rng, *b_shape)
    Ad, Bd = A.cuda(), B.cuda()
    C = torch.full((128, N), float("nan"), dtype=torch.float32, device="cuda")
    fa.check(fa.fa_selftest_umma(mode, Ad.data_ptr(), Bd.data_ptr(), C.data_ptr(), K, N, stream()), "selftest")
    st, detail = fa.fa_poll_device_error(stream())
    fa.check(st, f"status {detail:#x}")
    a, b = si.to_f64(A), si.to_f64(B)
    a = a.T if mode in (3, 4) else a
    b = b if mode in (1, 2, 4) else b.T
    ref = a @ b
    got = C.cpu().double().numpy()
    err = np.abs(got - ref).max()
    assert err <= 1e-4 * np.abs(ref).max() + 1e-5, f"mode {mode} K {K} N {N}: max err {err}"


def test_bounded_wait_gives_up_and_reports():
    """A wait on a barrier nothing completes ends after its limit (20 ms here) with
    FA_ERR_TIMEOUT in the status word; polling clears it and the context stays usable."""
    fa = lib()
    fa.check(fa.fa_debug_timeout_probe(20000, stream()))
    st, detail = fa.fa_poll_device_error(stream())
    assert st == fa.FA_ERR_TIMEOUT and detail == 0x301
    assert fa.fa_poll_device_error(stream()) == (fa.FA_OK, 0)
    x = torch.ones(1024, device="cuda")
    assert float(x.sum()) == 1024.0


@pytest.mark.parametrize("d", [32, 64, 128])
@pytest.mark.parametrize("rows", [1, 7, 1000, 65536 + 3])
def test_preprocess_rowsum(d, rows):
    """D_i = sum_k dO_ik O_ik on seeded bf16 inputs vs a float64 row sum."""
    fa = lib()
    rng = np.random.default_rng(7 * d + rows)
    O, dO = _bf16(rng, 1, 1, rows, d), _bf16(rng, 1, 1, rows, d)
    D = torch.empty((1, 1, rows), dtype=torch.float32, device="cuda")
    o, do = O.cuda(), dO.cuda()
    fa.check(fa.fa_bwd_preprocess(o.data_ptr(), do.data_ptr(), D.data_ptr(), 1, 1, rows, d, stream()))
    torch.cuda.synchronize()
    ref = (si.to_f64(O) * si.to_f64(dO)).sum(-1)
    np.testing.assert_allclose(D.cpu().double().numpy(), ref, rtol=0, atol=1e-4 * np.sqrt(d))
