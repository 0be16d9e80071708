"""The device entry points inside a CUDA graph: forward, preprocess and backward
captured once from one stream (they allocate nothing and never synchronise), then
replayed on new inputs copied into the same buffers.  A replay must give what an
eager call gives on those inputs: O, L, dK, dV bit for bit (dQ is summed in fp32
reductions whose order varies), and match the float64 oracle."""
import math

import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si
from gpu_util import assert_close, f64, lib

pytestmark = pytest.mark.gpu


class _Step:
    def __init__(self, B, H, Nq, Nk, d, causal, window):
        self.fa = lib()
        self.args = (B, H, Nq, Nk, d, causal, window)
        dev = torch.device("cuda")
        self.q, self.do = (torch.empty(B, H, Nq, d, dtype=torch.bfloat16, device=dev) for _ in range(2))
        self.k, self.v = (torch.empty(B, H, Nk, d, dtype=torch.bfloat16, device=dev) for _ in range(2))
        self.o, self.dq = torch.empty_like(self.q), torch.empty_like(self.q)
        self.dk, self.dv = torch.empty_like(self.k), torch.empty_like(self.k)
        self.lse, self.D = (torch.empty(B, H, Nq, dtype=torch.float32, device=dev) for _ in range(2))
        self.ws_bytes = self.fa.fa_bwd_workspace_size_ex(B, H, Nq, Nk, d, causal, window)
        self.ws = torch.empty(max(self.ws_bytes, 16), dtype=torch.uint8, device=dev)
        self.scale = 1 / math.sqrt(d)

    def load(self, Q, K, V, dO):
        for dst, src in zip((self.q, self.k, self.v, self.do), (Q, K, V, dO)):
            dst.copy_(src)

    def run(self, stream):
        fa, (B, H, Nq, Nk, d, causal, window) = self.fa, self.args
        fa.check(fa.fa_fwd_ex(self.q.data_ptr(), self.k.data_ptr(), self.v.data_ptr(), self.o.data_ptr(),
                              self.lse.data_ptr(), B, H, Nq, Nk, d, causal, window, self.scale, stream))
        fa.check(fa.fa_bwd_preprocess(self.o.data_ptr(), self.do.data_ptr(), self.D.data_ptr(), B, H, Nq, d, stream))
        fa.check(fa.fa_bwd_ex(self.q.data_ptr(), self.k.data_ptr(), self.v.data_ptr(), self.o.data_ptr(),
                              self.do.data_ptr(), self.lse.data_ptr(), self.D.data_ptr(), self.dq.data_ptr(),
                              self.dk.data_ptr(), self.dv.data_ptr(), B, H, Nq, Nk, d, causal, window, self.scale,
                              self.ws.data_ptr(), self.ws_bytes, stream))

    def outputs(self):
        return {"O": self.o.cpu(), "L": self.lse.cpu(), "dQ": self.dq.cpu(), "dK": self.dk.cpu(), "dV": self.dv.cpu()}


def _inputs(B, H, Nq, Nk, d, seed):
    Q, K, V, dO = si.make_qkvdo(B, H, max(Nq, Nk), d, seed=seed)
    return Q[:, :, :Nq].contiguous(), K[:, :, :Nk].contiguous(), V[:, :, :Nk].contiguous(), dO[:, :, :Nq].contiguous()


@pytest.mark.parametrize("d,causal,window,Nq,Nk", [(128, True, 0, 700, 700), (128, False, 0, 300, 500),
                                                   (64, True, 0, 640, 640), (128, True, 200, 600, 600),
                                                   (32, True, 0, 300, 300)])
def test_graph_replay_matches_eager(d, causal, window, Nq, Nk):
    B, H = 2, 3
    step = _Step(B, H, Nq, Nk, d, causal, window)
    stream = torch.cuda.current_stream()
    first = [t.cuda() for t in _inputs(B, H, Nq, Nk, d, seed=1700 + d + Nq)]
    second = [t.cuda() for t in _inputs(B, H, Nq, Nk, d, seed=1800 + d + Nq)]
    # eager on the second inputs: the expected values
    step.load(*second)
    step.run(stream.cuda_stream)
    torch.cuda.synchronize()
    eager = step.outputs()
    # capture on the first inputs, then replay on the second
    step.load(*first)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step.run(torch.cuda.current_stream().cuda_stream)
    for _ in range(2):
        step.load(*second)
        g.replay()
    torch.cuda.synchronize()
    st, detail = step.fa.fa_poll_device_error(stream.cuda_stream)
    step.fa.check(st, f"device status word (site {detail:#x})")
    got = step.outputs()
    for n in ("O", "L", "dK", "dV"):
        assert torch.equal(got[n], eager[n]), n
    a, b = f64(got["dQ"]), f64(eager["dQ"])
    assert np.linalg.norm(a - b) <= 2e-3 * np.linalg.norm(b)
    q, k, v, do = (f64(t.cpu()) for t in second)
    O, L = oracle.standard_attention_fwd(q, k, v, causal, window=window)
    dQ, dK, dV, _ = oracle.standard_attention_bwd(q, k, v, do, causal, window=window)
    assert_close({n: f64(t) for n, t in got.items()}, {"O": O, "L": L, "dQ": dQ, "dK": dK, "dV": dV},
                 f"graph replay d={d} causal={causal} w={window}")
