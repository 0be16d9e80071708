"""Guard bands around every output: no kernel writes outside [B, H, N, d].

Each output (O, L, D, dQ, dK, dV), the backward's fp32 dQ workspace and the host
step's device workspace are views into a larger buffer with 4 KiB on each side
filled with a fixed byte pattern; inputs are guarded the same way (a kernel must
not write them at all).  After the call the guard bytes must be unchanged.  The
cases are the ones where the edges matter: ragged lengths below and across a tile,
N_q != N_k (a prefill chunk, a decode step), a sliding window, every forward and
backward form, and the step on host buffers (whose host arrays are guarded too).
The values themselves are checked against the oracle elsewhere; here only the
bytes outside the tensors are.
"""
import math

import numpy as np
import pytest
import torch

import seeded_inputs as si
from gpu_util import lib, stream

pytestmark = pytest.mark.gpu

GUARD = 4096
PATTERN = 0xA5


class Guarded:
    """A tensor of `shape` inside a buffer with GUARD bytes of PATTERN on each side."""

    def __init__(self, shape, dtype, device, fill=None):
        esz = torch.empty((), dtype=dtype).element_size()
        self.n = math.prod(shape)
        self.g = GUARD // esz
        kw = {"pin_memory": True} if device == "cpu" else {}
        self.buf = torch.empty(self.n + 2 * self.g, dtype=dtype, device=device, **kw)
        self.buf.view(torch.uint8).fill_(PATTERN)
        self.t = self.buf[self.g:self.g + self.n].view(shape)
        if fill is not None:
            self.t.copy_(fill)

    def ptr(self):
        return self.t.data_ptr() if self.n else None

    def intact(self):
        b = self.buf.view(torch.uint8).cpu().numpy()
        gb = self.g * self.buf.element_size()
        return bool((b[:gb] == PATTERN).all() and (b[len(b) - gb:] == PATTERN).all())


def _device_step(fa, B, H, Nq, Nk, d, causal, window, fwd_form, bwd_split):
    N = max(Nq, Nk)
    Q, K, V, dO = si.make_qkvdo(B, H, N, d, seed=900 + Nq + 7 * Nk + d)
    Q, dO = (t[:, :, :Nq].contiguous() for t in (Q, dO))
    K, V = (t[:, :, :Nk].contiguous() for t in (K, V))
    dev = "cuda"
    g = {n: Guarded(t.shape, torch.bfloat16, dev, t) for n, t in (("Q", Q), ("K", K), ("V", V), ("dO", dO))}
    for n, shape in (("O", (B, H, Nq, d)), ("dQ", (B, H, Nq, d)), ("dK", (B, H, Nk, d)), ("dV", (B, H, Nk, d))):
        g[n] = Guarded(shape, torch.bfloat16, dev)
    for n in ("L", "D"):
        g[n] = Guarded((B, H, Nq), torch.float32, dev)
    fa.check(fa.fa_debug_set_fwd_form(fwd_form))
    fa.check(fa.fa_debug_set_bwd_split(bwd_split))
    try:
        ws_bytes = fa.fa_bwd_workspace_size_ex(B, H, Nq, Nk, d, causal, window)
        g["ws"] = Guarded((max(ws_bytes, 16),), torch.uint8, dev)
        s, scale = stream(), 1.0 / math.sqrt(d)
        fa.check(fa.fa_fwd_ex(g["Q"].ptr(), g["K"].ptr(), g["V"].ptr(), g["O"].ptr(), g["L"].ptr(), B, H, Nq, Nk, d,
                              causal, window, scale, s), "fa_fwd_ex")
        fa.check(fa.fa_bwd_preprocess(g["O"].ptr(), g["dO"].ptr(), g["D"].ptr(), B, H, Nq, d, s), "preprocess")
        fa.check(fa.fa_bwd_ex(*(g[n].ptr() for n in ("Q", "K", "V", "O", "dO", "L", "D", "dQ", "dK", "dV")), B, H, Nq,
                              Nk, d, causal, window, scale, g["ws"].ptr(), ws_bytes, s), "fa_bwd_ex")
    finally:
        fa.fa_debug_set_fwd_form(0)
        fa.fa_debug_set_bwd_split(0)
    st, detail = fa.fa_poll_device_error(s)
    fa.check(st, f"device status (site {detail:#x})")
    torch.cuda.synchronize()
    bad = [n for n, x in g.items() if not x.intact()]
    assert not bad, f"guard bytes changed around {bad}"
    # the inputs are unchanged too
    for n, t in (("Q", Q), ("K", K), ("V", V), ("dO", dO)):
        assert torch.equal(g[n].t.cpu(), t), n
    # and every output element was written (the pattern is not a value these produce)
    for n in ("O", "dQ", "dK", "dV", "L", "D"):
        b = g[n].t.cpu().contiguous().view(torch.uint8).numpy()
        esz = g[n].buf.element_size()
        if b.size:
            assert not (b.reshape(-1, esz) == PATTERN).all(axis=1).any(), f"{n}: an element was never written"


SHAPES = [  # (B, H, Nq, Nk, causal, window)
    (1, 2, 1, 1, True, 0), (1, 2, 7, 7, False, 0), (1, 3, 129, 129, True, 0), (2, 1, 1000, 1000, True, 0),
    (1, 2, 300, 1000, True, 0), (1, 2, 1, 777, True, 0), (1, 2, 1000, 1000, True, 100), (1, 2, 500, 257, False, 0),
]


@pytest.mark.parametrize("d", [32, 64, 128])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_guards_default_forms(d, shape):
    _device_step(lib(), *shape[:4], d, shape[4], shape[5], 0, 0)


@pytest.mark.parametrize("fwd_form,bwd_split", [(1, 1), (2, 2), (3, 3)])
@pytest.mark.parametrize("shape", [(1, 3, 129, 129, True, 0), (2, 1, 1000, 1000, True, 100), (1, 2, 300, 1000, True, 0),
                                   (1, 2, 500, 257, False, 0)], ids=lambda s: "x".join(map(str, s)))
def test_guards_every_form_d128(fwd_form, bwd_split, shape):
    _device_step(lib(), *shape[:4], 128, shape[4], shape[5], fwd_form, bwd_split)


@pytest.mark.parametrize("d", [64, 128])
def test_guards_two_kernel_and_one_kernel_d64(d):
    for split in (1, 2):
        _device_step(lib(), 1, 3, 1000, 1000, d, True, 0, 0, split)


@pytest.mark.parametrize("B,H,Nq,Nk,d,causal,window,hc", [(1, 5, 300, 300, 128, True, 0, 2), (2, 2, 129, 777, 64, True, 0, 1),
                                                       (1, 3, 1000, 1000, 128, True, 100, 0)])
def test_guards_host_step(B, H, Nq, Nk, d, causal, window, hc):
    """fa_fwd_bwd_host: guarded pinned host arrays (in and out) and a guarded device workspace."""
    fa = lib()
    N = max(Nq, Nk)
    Q, K, V, dO = si.make_qkvdo(B, H, N, d, seed=1900 + Nq + Nk)
    Q, dO = (t[:, :, :Nq].contiguous() for t in (Q, dO))
    K, V = (t[:, :, :Nk].contiguous() for t in (K, V))
    g = {n: Guarded(t.shape, torch.bfloat16, "cpu", t) for n, t in (("Q", Q), ("K", K), ("V", V), ("dO", dO))}
    for n, shape in (("O", (B, H, Nq, d)), ("dQ", (B, H, Nq, d)), ("dK", (B, H, Nk, d)), ("dV", (B, H, Nk, d))):
        g[n] = Guarded(shape, torch.bfloat16, "cpu")
    g["L"] = Guarded((B, H, Nq), torch.float32, "cpu")
    ws_bytes = fa.fa_fwd_bwd_host_workspace_size(B, H, Nq, Nk, d, causal, window, hc)
    # 256-byte aligned inside its guards: GUARD is a multiple of 256 and torch's base is aligned
    g["ws"] = Guarded((ws_bytes,), torch.uint8, "cuda")
    assert g["ws"].ptr() % 256 == 0
    s = stream()
    fa.check(fa.fa_fwd_bwd_host(*(g[n].ptr() for n in ("Q", "K", "V", "dO", "O", "L", "dQ", "dK", "dV")), B, H, Nq, Nk,
                                d, causal, window, 1.0 / math.sqrt(d), hc, g["ws"].ptr(), ws_bytes, s), "host step")
    torch.cuda.current_stream().synchronize()
    st, detail = fa.fa_poll_device_error(s)
    fa.check(st, f"device status (site {detail:#x})")
    bad = [n for n, x in g.items() if not x.intact()]
    assert not bad, f"guard bytes changed around {bad}"
    for n, t in (("Q", Q), ("K", K), ("V", V), ("dO", dO)):
        assert torch.equal(g[n].t, t), n
