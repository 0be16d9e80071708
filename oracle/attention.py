"""Oracle for exact tiled attention: plain, slow float64 NumPy on the CPU.

TEST INFRASTRUCTURE.  Only the tests, the smoke check of ``__graft_entry__`` and
the CPU-baseline leg of ``bench.py`` may import this package.  It shares no code
with the CUDA path and the CUDA path never calls it.

Sources (three web pages on FlashAttention):
  [p1] "CS349E lecture 11: 03_flash_backward.py" (functions std_fwd_bwd_io,
       demo1_gradcheck, demo4_causal)
  [p2] "CS324 lecture 8: 03_online_softmax_and_flash.py" (demo2_online,
       demo3_forward, demo4_backward, flash_attention_torch)
  [p3] "CS336 Assignment 2 notes: FlashAttention & DDP", Part 1:
       §1.1 (standard attention), §1.2 (FlashAttention-2 forward),
       §1.3 (Triton kernel: causal whole-tile skip), §1.4 (backward,
       Equations 13-19, two-kernel backward)

Functions and the pins that tie each to something other than itself (all in
tests/test_oracle_pins.py):

  standard_attention_fwd   plain definition of softmax(Q K^T s) V and its
                           logsumexp.  Pinned by torch fp64 autograd and SDPA,
                           the N=1 and equal-keys closed forms, and agreement
                           with flash_forward_tiled.
  standard_attention_bwd   plain softmax-Jacobian backward.  Pinned by central
                           differences, torch fp64 autograd, and the identity
                           sum_j P_ij dP_ij = rowsum(dO * O).
  rows_fwd_bwd / key_rows_bwd
                           the same definitions evaluated on a subset of query
                           rows / key rows.  Pinned by equality with the full
                           functions on small cases.
  online_softmax           streaming (m, l) recurrence.  Pinned by the worked
                           trace on x = [2,-1,3,0.5,6,1,-2,5.5], block 3.
  flash_forward_tiled      FlashAttention-2 forward in the notes' order.
  flash_backward_tiled     Equations 13-19 tile by tile, key/value tiles outer.
  causal_tile_pairs        closed-form count of computed tile pairs (with the
                           two-sided skip of a sliding window).  Pinned by
                           brute force and the fraction 1/2 + 1/(2T).
  visible_pairs            entries the mask leaves visible (the FLOP count of a
                           masked pass).  Pinned by brute force.

The window and N_q != N_k forms of every function are pinned in
tests/test_oracle_pins_mask.py (pure-Python loops, torch fp64 autograd with an
explicit mask, closed forms for w = 1, reductions to the causal and unmasked
cases, chunked prefill, central differences, brute-force tile counts).

Conventions: arrays are [..., N, d]; L is the natural-log logsumexp of the
scaled scores (S already includes the scale).  Q has N_q rows, K and V have
N_k rows (N_q = N_k unless stated).  Query row i sits at sequence position
p_i = i + N_k - N_q: the queries are the last N_q positions of the key
sequence, so the last query (a decoded token) sees every key ([p1]
demo4_causal, observation 3: one new token sees the whole cache); with
N_q = N_k this is the usual top-left alignment, query i sees keys 0..i.
causal: query i sees keys j <= p_i (N_q <= N_k required).  window w > 0 (only
with causal): query i sees keys p_i - w < j <= p_i, itself and the w - 1 before
it ([p2] window_attention_torch: masked where cols > rows or cols <= rows - w).
"""
from __future__ import annotations

import math

import numpy as np

ROW_BLOCK = 256  # rows evaluated at a time, so no N x N array is ever held


def _f64(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64)


def _heads(x: np.ndarray) -> np.ndarray:
    """[..., N, d] -> [BH, N, d] view."""
    return x.reshape((-1,) + x.shape[-2:])


def _scale(d: int, scale) -> float:
    return 1.0 / math.sqrt(d) if scale is None else float(scale)


def _check_mask(Nq: int, Nk: int, causal: bool, window: int) -> int:
    """Validates the mask and returns the position offset N_k - N_q."""
    if window < 0 or (window > 0 and not causal):
        raise ValueError("a sliding window is a causal mask: window > 0 needs causal")
    if causal and Nq > Nk:
        raise ValueError("causal attention needs N_q <= N_k (every query sees at least one key)")
    return Nk - Nq


def _masked(row_ids: np.ndarray, cols: np.ndarray, causal: bool, off: int = 0, window: int = 0) -> np.ndarray:
    """True where key cols[j] is hidden from query row_ids[i] (position p = row + off):
    causal hides j > p ([p2] flash_attention_torch, cols > rows); a window w
    also hides j <= p - w ([p2] window_attention_torch)."""
    pos = row_ids[:, None] + off
    hide = np.zeros((len(row_ids), len(cols)), dtype=bool)
    if causal:
        hide |= cols[None, :] > pos
    if window > 0:
        hide |= cols[None, :] <= pos - window
    return hide


def _scores(q_rows: np.ndarray, row_ids: np.ndarray, K: np.ndarray, causal: bool, s: float, off: int = 0,
            window: int = 0):
    """Scaled scores of some query rows against keys 0 .. len(K)-1, masked.

    S = Q K^T / sqrt(d) ([p3] §1.4 Eq 13); hidden entries are -inf.
    """
    S = (q_rows @ K.T) * s
    if causal or window:
        S = np.where(_masked(row_ids, np.arange(K.shape[0]), causal, off, window), -np.inf, S)
    return S


def _visible(rows: np.ndarray, n_keys: int, causal: bool, off: int = 0) -> int:
    """Keys 0 .. k-1 hold every nonzero weight of these rows.  Under the causal
    mask, keys after the last row's position carry weight exp(-inf) = 0 exactly,
    so leaving them out of the sums changes no value."""
    return min(n_keys, int(rows.max()) + off + 1) if causal else n_keys


def _logsumexp_rows(S: np.ndarray) -> np.ndarray:
    """Safe logsumexp per row: m + ln(sum exp(S - m)) ([p2] demo1_overflow; [p3] §1.2)."""
    m = S.max(axis=1)
    return m + np.log(np.exp(S - m[:, None]).sum(axis=1))


# ---------------------------------------------------------------------------
# Plain definition (no tiling, no online softmax)
# ---------------------------------------------------------------------------

def standard_attention_fwd(Q, K, V, causal: bool = False, scale=None, window: int = 0):
    """O = softmax(Q K^T s) V and L = logsumexp of each row of Q K^T s.

    [p3] §1.1 (S = QK^T, P = softmax(S), O = PV) and §1.2 (L = m + log l), with
    the mask of the module docstring.  Returns (O [..., N_q, d], L [..., N_q]) in
    float64.
    """
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    lead, (N, d) = Q.shape[:-2], Q.shape[-2:]
    off = _check_mask(N, K.shape[-2], causal, window)
    s = _scale(d, scale)
    Qh, Kh, Vh = _heads(Q), _heads(K), _heads(V)
    O = np.empty(Qh.shape[:-1] + (Vh.shape[-1],))
    L = np.empty(Qh.shape[:-1])
    for h in range(Qh.shape[0]):
        for r0 in range(0, N, ROW_BLOCK):
            rows = np.arange(r0, min(N, r0 + ROW_BLOCK))
            kv = _visible(rows, Kh.shape[1], causal, off)
            S = _scores(Qh[h, rows], rows, Kh[h, :kv], causal, s, off, window)
            Lr = _logsumexp_rows(S)
            P = np.exp(S - Lr[:, None])  # softmax of each row
            O[h, rows] = P @ Vh[h, :kv]
            L[h, rows] = Lr
    return O.reshape(lead + O.shape[-2:]), L.reshape(lead + (N,))


def standard_attention_bwd(Q, K, V, dO, causal: bool = False, scale=None, window: int = 0):
    """Gradients of sum(O * dO) with respect to Q, K, V (plain softmax backward).

    P is formed from its definition; then ([p3] §1.4 Equations 15-19, and the
    standard backward of [p1]/[p2] that uses the stored P):
        dV = P^T dO,  dP = dO V^T,
        D_i = sum_j P_ij dP_ij       (the softmax Jacobian term),
        dS = P * (dP - D),  dQ = dS K s,  dK = dS^T Q s.
    Returns (dQ, dK, dV, D) in float64.
    """
    Q, K, V, dO = _f64(Q), _f64(K), _f64(V), _f64(dO)
    lead, (N, d) = Q.shape[:-2], Q.shape[-2:]
    off = _check_mask(N, K.shape[-2], causal, window)
    s = _scale(d, scale)
    Qh, Kh, Vh, dOh = _heads(Q), _heads(K), _heads(V), _heads(dO)
    dQ = np.zeros_like(Qh)
    dK = np.zeros_like(Kh)
    dV = np.zeros_like(Vh)
    D = np.empty(Qh.shape[:-1])
    for h in range(Qh.shape[0]):
        for r0 in range(0, N, ROW_BLOCK):
            rows = np.arange(r0, min(N, r0 + ROW_BLOCK))
            kv = _visible(rows, Kh.shape[1], causal, off)
            S = _scores(Qh[h, rows], rows, Kh[h, :kv], causal, s, off, window)
            P = np.exp(S - _logsumexp_rows(S)[:, None])
            dP = dOh[h, rows] @ Vh[h, :kv].T
            Dr = (P * dP).sum(axis=1)
            dS = P * (dP - Dr[:, None])
            dQ[h, rows] = (dS @ Kh[h, :kv]) * s
            dK[h, :kv] += (dS.T @ Qh[h, rows]) * s
            dV[h, :kv] += P.T @ dOh[h, rows]
            D[h, rows] = Dr
    shp = lead + (N, d)
    return (dQ.reshape(shp), dK.reshape(lead + Kh.shape[-2:]),
            dV.reshape(lead + Vh.shape[-2:]), D.reshape(lead + (N,)))


# ---------------------------------------------------------------------------
# The same definitions on a subset of rows (for sequence lengths where the
# full result is too slow on the CPU)
# ---------------------------------------------------------------------------

def rows_fwd_bwd(Q, K, V, dO, rows, causal: bool = False, scale=None, window: int = 0):
    """O, L, dQ and D of the given query rows of every head.

    Each of these depends only on its own query row (plus all of K and V):
    O_i = P_i V, L_i = logsumexp(S_i), D_i = sum_j P_ij dP_ij and
    dQ_i = sum_j P_ij (dP_ij - D_i) K_j s.   Q, K, V, dO are [BH, N, d].
    Returns arrays [BH, len(rows), ...].
    """
    Q, K, V, dO = _f64(Q), _f64(K), _f64(V), _f64(dO)
    rows = np.asarray(rows)
    d = Q.shape[-1]
    off = _check_mask(Q.shape[-2], K.shape[-2], causal, window)
    s = _scale(d, scale)
    BH = Q.shape[0]
    O = np.empty((BH, len(rows), V.shape[-1]))
    L = np.empty((BH, len(rows)))
    dQ = np.empty((BH, len(rows), d))
    D = np.empty((BH, len(rows)))
    for h in range(BH):
        for b0 in range(0, len(rows), ROW_BLOCK):
            r = rows[b0:b0 + ROW_BLOCK]
            kv = _visible(r, K.shape[1], causal, off)
            S = _scores(Q[h, r], r, K[h, :kv], causal, s, off, window)
            Lr = _logsumexp_rows(S)
            P = np.exp(S - Lr[:, None])
            dP = dO[h, r] @ V[h, :kv].T
            Dr = (P * dP).sum(axis=1)
            O[h, b0:b0 + len(r)] = P @ V[h, :kv]
            L[h, b0:b0 + len(r)] = Lr
            D[h, b0:b0 + len(r)] = Dr
            dQ[h, b0:b0 + len(r)] = ((P * (dP - Dr[:, None])) @ K[h, :kv]) * s
    return O, L, dQ, D


def key_rows_bwd(Q, K, V, dO, L, D, keys, causal: bool = False, scale=None, window: int = 0):
    """dK and dV of the given key rows of every head, from full-length L and D.

    dV_j = sum_i P_ij dO_i and dK_j = sum_i dS_ij Q_i s with
    P_ij = exp(S_ij - L_i) ([p3] §1.4 Eq 14) and dS_ij = P_ij (dP_ij - D_i).
    L and D ([BH, N]) must be the oracle's own (standard_attention_fwd /
    rows_fwd_bwd over all rows).  Returns (dK, dV) as [BH, len(keys), d].
    """
    Q, K, V, dO, L, D = (_f64(x) for x in (Q, K, V, dO, L, D))
    keys = np.asarray(keys)
    N, d = Q.shape[-2:]
    off = _check_mask(N, K.shape[-2], causal, window)
    s = _scale(d, scale)
    BH = Q.shape[0]
    dK = np.zeros((BH, len(keys), d))
    dV = np.zeros((BH, len(keys), V.shape[-1]))
    first = max(0, int(keys.min()) - off) if causal else 0  # rows before the first key's position see none
    for h in range(BH):
        Kk, Vk = K[h, keys], V[h, keys]
        for r0 in range(first - first % ROW_BLOCK, N, ROW_BLOCK):
            rows = np.arange(r0, min(N, r0 + ROW_BLOCK))
            S = (Q[h, rows] @ Kk.T) * s
            if causal or window:
                S = np.where(_masked(rows, keys, causal, off, window), -np.inf, S)
            P = np.exp(S - L[h, rows][:, None])
            dP = dO[h, rows] @ Vk.T
            dS = P * (dP - D[h, rows][:, None])
            dV[h] += P.T @ dO[h, rows]
            dK[h] += (dS.T @ Q[h, rows]) * s
    return dK, dV


# ---------------------------------------------------------------------------
# The method itself, step by step in the pages' order (CPU, float64)
# ---------------------------------------------------------------------------

def online_softmax(x, block: int):
    """Streaming softmax that keeps only the running max m and denominator l.

    [p2] demo2_online and [p3] §1.2: for each block, m_new = max(m, max(block)),
    l <- l * exp(m - m_new) + sum(exp(block - m_new)), m <- m_new; at the end
    softmax = exp(x - m) / l.  Returns (softmax, trace) where trace holds
    (elements read so far, m, l) after each block.
    """
    x = _f64(x)
    m, l = -np.inf, 0.0
    trace = []
    for start in range(0, x.size, block):
        blk = x[start:start + block]
        m_new = max(m, float(blk.max()))
        corr = math.exp(m - m_new) if m != -np.inf else 0.0
        l = l * corr + float(np.exp(blk - m_new).sum())
        m = m_new
        trace.append((min(start + block, x.size), m, l))
    return np.exp(x - m) / l, trace


def _tile_visible(q_first: int, q_last: int, k_first: int, causal: bool, k_last: int = 0, off: int = 0,
                  window: int = 0) -> bool:
    """Whole-tile skip: a key tile whose first key lies after the tile's last
    query position is never read ([p3] §1.3, k_start > q_end; [p2]
    flash_attention_torch visits key blocks j0 < i0 + n_i); with a window, nor is
    a key tile whose last key lies at or before the first query's position minus
    the window (the other side of the band)."""
    if causal and k_first > q_last + off:
        return False
    if window > 0 and k_last <= q_first + off - window:
        return False
    return True


def flash_forward_tiled(Q, K, V, Br: int, Bc: int, causal: bool = False, scale=None, window: int = 0):
    """FlashAttention-2 forward with deferred normalisation, one head at a time.

    [p3] §1.2: per query tile, m = -inf, l = 0, O = 0; per visible key tile
    S = Q_i K_j^T s, m_new = max(m, rowmax S), P = exp(S - m_new),
    l = exp(m - m_new) l + rowsum P, O = exp(m - m_new) O + P V_j, m = m_new;
    finally O = O / l and L = m + log l.  Diagonal tiles get the in-tile mask.
    Returns (O, L, tile pairs computed).
    """
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    lead, (N, d) = Q.shape[:-2], Q.shape[-2:]
    Nk = K.shape[-2]
    off = _check_mask(N, Nk, causal, window)
    s = _scale(d, scale)
    Qh, Kh, Vh = _heads(Q), _heads(K), _heads(V)
    O = np.empty(Qh.shape[:-1] + (Vh.shape[-1],))
    L = np.empty(Qh.shape[:-1])
    tiles = 0
    for h in range(Qh.shape[0]):
        for i0 in range(0, N, Br):
            rows = np.arange(i0, min(N, i0 + Br))
            m = np.full(len(rows), -np.inf)
            l = np.zeros(len(rows))
            acc = np.zeros((len(rows), Vh.shape[-1]))
            for j0 in range(0, Nk, Bc):
                cols = np.arange(j0, min(Nk, j0 + Bc))
                if not _tile_visible(rows[0], rows[-1], j0, causal, cols[-1], off, window):
                    continue
                tiles += 1
                S = (Qh[h, rows] @ Kh[h, cols].T) * s
                if causal or window:
                    S = np.where(_masked(rows, cols, causal, off, window), -np.inf, S)
                m_new = np.maximum(m, S.max(axis=1))
                # a row whose every key so far is masked keeps m = -inf; guard exp(-inf + inf)
                safe = np.where(np.isfinite(m_new), m_new, 0.0)
                P = np.exp(S - safe[:, None])
                corr = np.where(np.isfinite(m), np.exp(m - safe), 0.0)
                l = corr * l + P.sum(axis=1)
                acc = corr[:, None] * acc + P @ Vh[h, cols]
                m = m_new
            O[h, rows] = acc / l[:, None]
            L[h, rows] = m + np.log(l)
    return O.reshape(lead + O.shape[-2:]), L.reshape(lead + (N,)), tiles


def flash_backward_tiled(Q, K, V, O, dO, L, Br: int, Bc: int, causal: bool = False, scale=None, window: int = 0):
    """Recompute backward, key/value tiles in the outer loop, one head at a time.

    D = rowsum(O * dO) once ([p3] §1.4 Eq 17; [p1] demo1_gradcheck), then per
    visible tile pair ([p3] §1.4 Equations 13-19):
        S = Q_i K_j^T s (13), P = exp(S - L_i) (14), dV_j += P^T dO_i (15),
        dP = dO_i V_j^T (16), dS = P * (dP - D_i) (17), dQ_i += dS K_j s (18),
        dK_j += dS^T Q_i s (19).
    dQ_i collects contributions from every key tile, as kernel 1 of the
    two-kernel backward would with atomics ([p3] §1.4).
    Returns (dQ, dK, dV, D, tile pairs computed).
    """
    Q, K, V, O, dO, L = (_f64(x) for x in (Q, K, V, O, dO, L))
    lead, (N, d) = Q.shape[:-2], Q.shape[-2:]
    Nk = K.shape[-2]
    off = _check_mask(N, Nk, causal, window)
    s = _scale(d, scale)
    Qh, Kh, Vh, Oh, dOh = (_heads(x) for x in (Q, K, V, O, dO))
    Lh = L.reshape(-1, N)
    Dh = (Oh * dOh).sum(axis=-1)
    dQ = np.zeros_like(Qh)
    dK = np.zeros_like(Kh)
    dV = np.zeros_like(Vh)
    tiles = 0
    for h in range(Qh.shape[0]):
        for j0 in range(0, Nk, Bc):
            cols = np.arange(j0, min(Nk, j0 + Bc))
            for i0 in range(0, N, Br):
                rows = np.arange(i0, min(N, i0 + Br))
                if not _tile_visible(rows[0], rows[-1], j0, causal, cols[-1], off, window):
                    continue
                tiles += 1
                S = (Qh[h, rows] @ Kh[h, cols].T) * s
                if causal or window:
                    S = np.where(_masked(rows, cols, causal, off, window), -np.inf, S)
                P = np.exp(S - Lh[h, rows][:, None])
                dV[h, cols] += P.T @ dOh[h, rows]
                dP = dOh[h, rows] @ Vh[h, cols].T
                dS = P * (dP - Dh[h, rows][:, None])
                dQ[h, rows] += (dS @ Kh[h, cols]) * s
                dK[h, cols] += (dS.T @ Qh[h, rows]) * s
    shp = lead + (N, d)
    return (dQ.reshape(shp), dK.reshape(lead + Kh.shape[-2:]), dV.reshape(lead + Vh.shape[-2:]),
            Dh.reshape(lead + (N,)), tiles)


def causal_tile_pairs(N: int, Br: int, Bc: int, causal: bool, Nk: int | None = None, window: int = 0) -> int:
    """Number of (query tile, key tile) pairs a tiled pass computes, per head.

    Without the mask every pair: ceil(N/Br) * ceil(Nk/Bc).  With it, query tile
    i (positions p_first .. p_last, p = row + N_k - N_q) sees key tiles up to
    floor(p_last / Bc); for square tiles and N a multiple of the tile this is
    T(T+1)/2, a fraction 1/2 + 1/(2T) of all pairs ([p1] demo4_causal).  A
    window w also drops the key tiles below floor((p_first - w + 1) / Bc).
    """
    Nk = N if Nk is None else Nk
    off = _check_mask(N, Nk, causal, window)
    Tq, Tk = -(-N // Br), -(-Nk // Bc)
    if not causal:
        return Tq * Tk
    n = 0
    for i in range(Tq):
        p_first, p_last = i * Br + off, min((i + 1) * Br, N) - 1 + off
        hi = min(Tk - 1, p_last // Bc)
        lo = max(0, (p_first - window + 1) // Bc) if window > 0 else 0
        n += max(0, hi - lo + 1)
    return n


def attention_flops(N: int, d: int, causal: bool, B: int = 1, H: int = 1):
    """Counted matmul FLOPs: 4 N^2 d forward and 10 N^2 d backward per head
    (two and five N x N x d products at 2 flops per multiply-add; [p1]
    std_fwd_bwd_io and demo3 observations), halved under the causal mask."""
    f = 0.5 if causal else 1.0
    return 4.0 * B * H * N * N * d * f, 10.0 * B * H * N * N * d * f


def visible_pairs(Nq: int, Nk: int, causal: bool, window: int = 0) -> int:
    """Number of (query, key) entries the mask leaves visible, per head: the
    FLOP count of a masked pass is 4 d (forward) and 10 d (backward) times this.
    Counted row by row from the mask's definition."""
    off = _check_mask(Nq, Nk, causal, window)
    n = 0
    for i in range(Nq):
        hi = min(Nk - 1, i + off) if causal else Nk - 1
        lo = max(0, i + off - window + 1) if window > 0 else 0
        n += hi - lo + 1
    return n
