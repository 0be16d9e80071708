"""Host-side checks of fa_fwd_bwd_host (no GPU needed): the chunk plan over the
flattened B*H heads, the device workspace it asks for, and argument errors that
return before any CUDA call."""
import math

import pytest

SHAPES = [(1, 32, 32768, 32768, 128), (2, 16, 4096, 4096, 128), (1, 32, 8192, 8192, 128), (4, 8, 1024, 1024, 64),
          (16, 32, 1, 8192, 128), (1, 32, 2048, 32768, 128), (1, 2, 300, 300, 128), (3, 7, 129, 257, 32),
          (1, 1, 100, 100, 64), (8, 64, 512, 512, 128)]


def _tiles(n):
    return -(-n // 128)


@pytest.mark.parametrize("B,H,Nq,Nk,d", SHAPES)
def test_automatic_chunks(fa_lib, B, H, Nq, Nk, d):
    """Each chunk keeps at least half a wave of 128-row tiles on the 152 SMs (one
    wave before the chunks are evened out), or is the whole batch; there are at most
    32 chunks, and chunks are even (the last one short by fewer heads than there are
    chunks)."""
    BH = B * H
    hc = fa_lib.fa_fwd_bwd_host_chunk_heads(B, H, Nq, Nk, d, 0)
    assert 1 <= hc <= BH
    chunks = math.ceil(BH / hc)
    assert chunks <= 32
    assert hc * chunks - BH < chunks
    assert hc == BH or hc * min(_tiles(Nq), _tiles(Nk)) >= 76


def test_chunk_override_and_errors(fa_lib):
    fa = fa_lib
    assert fa.fa_fwd_bwd_host_chunk_heads(2, 3, 100, 100, 64, 1) == 1
    assert fa.fa_fwd_bwd_host_chunk_heads(2, 3, 100, 100, 64, 4) == 4
    assert fa.fa_fwd_bwd_host_chunk_heads(2, 3, 100, 100, 64, 100) == 6
    assert fa.fa_fwd_bwd_host_chunk_heads(0, 3, 100, 100, 64, 0) == 0
    assert fa.fa_fwd_bwd_host_chunk_heads(2, 3, 100, 100, 64, -1) == -1
    assert fa.fa_fwd_bwd_host_chunk_heads(2, 3, 100, 100, 48, 0) == -1
    assert fa.fa_fwd_bwd_host_chunk_heads(2, 3, 100, 0, 64, 0) == -1


@pytest.mark.parametrize("B,H,Nq,Nk,d", SHAPES)
@pytest.mark.parametrize("hpc", [0, 1, 3])
def test_workspace_holds_the_live_chunks(fa_lib, B, H, Nq, Nk, d, hpc):
    """Device copies of min(4, chunks) chunks (Q, K, V, dO, O, dQ, dK, dV in bf16; L
    and D in fp32), plus one dQ accumulator per compute stream, each array rounded
    up to 256 bytes."""
    fa = fa_lib
    causal = Nq <= Nk
    BH = B * H
    hc = fa.fa_fwd_bwd_host_chunk_heads(B, H, Nq, Nk, d, hpc)
    chunks = math.ceil(BH / hc)
    slots, streams = min(4, chunks), min(2, chunks)
    arrays = hc * (4 * Nq * d * 2 + 4 * Nk * d * 2 + 2 * Nq * 4)
    acc = fa.fa_bwd_workspace_size_ex(1, hc, Nq, Nk, d, causal, 0)
    ws = fa.fa_fwd_bwd_host_workspace_size(B, H, Nq, Nk, d, causal, 0, hpc)
    assert slots * arrays + streams * acc <= ws <= slots * (arrays + 10 * 255) + streams * (acc + 255)
    assert ws % 256 == 0


def test_host_step_argument_errors(fa_lib):
    fa = fa_lib
    p = 4096  # fake addresses: never dereferenced, validation fails first
    ws = fa.fa_fwd_bwd_host_workspace_size(1, 2, 64, 64, 64, 1, 0, 0)
    ptrs = [p] * 9

    def call(ptrs=ptrs, B=1, H=2, Nq=64, Nk=64, d=64, causal=1, window=0, scale=0.125, hpc=0, wsp=p * 16,
             wsb=ws):
        return fa.fa_fwd_bwd_host(*ptrs, B, H, Nq, Nk, d, causal, window, scale, hpc, wsp, wsb, None)

    assert call(d=48) == fa.FA_ERR_UNSUPPORTED
    assert call(scale=0.0) == fa.FA_ERR_INVALID_ARG
    assert call(scale=float("nan")) == fa.FA_ERR_INVALID_ARG
    assert call(causal=0, window=8) == fa.FA_ERR_INVALID_ARG
    assert call(hpc=-1) == fa.FA_ERR_INVALID_ARG
    assert call(Nk=0) == fa.FA_ERR_INVALID_ARG
    for i in range(9):
        assert call(ptrs=[None if j == i else p for j in range(9)]) == fa.FA_ERR_INVALID_ARG, i
    assert call(wsp=None) == fa.FA_ERR_WORKSPACE
    assert call(wsb=ws - 1) == fa.FA_ERR_WORKSPACE
    assert call(wsp=p * 16 + 16) == fa.FA_ERR_WORKSPACE
    # no heads: nothing to do, no CUDA call
    assert call(ptrs=[None] * 9, B=0, wsp=None, wsb=0) == fa.FA_OK
