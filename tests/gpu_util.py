"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI and
compare with the float64 oracle on the same seeded bf16 inputs.

Tolerances (element-wise against the oracle run on the bf16-rounded inputs):
  O:  max |err| <= 1e-2 and ||err||_F / ||ref||_F <= 5e-3
  L:  max |err| <= 2e-3
  dQ, dK, dV: ||err||_F / ||ref||_F <= 1e-2

O is returned in bf16, whose own rounding reaches half a bf16 unit in the last
place of |O| (0.0078 for |O| in [2, 4), 0.0156 for |O| in [4, 8)).  The max-abs
bound on O therefore applies to the error beyond that quantum:
|got - ref| - ulp_bf16(ref)/2 <= 1e-2.  A gradient whose exact value is zero
(e.g. dQ and dK with a single key) is checked by its RMS (<= 1e-4) instead of
the relative norm.

With FA_PARITY_LOG set to a file name, every comparison appends its measured
errors to that file as one JSON line: O_max_abs (the raw figure), O_beyond_half_ulp,
O_rel; L_max_abs; D_max_abs and D_rel when D is compared; dQ_rel, dK_rel, dV_rel
(or dX_rms where the exact gradient is zero).
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import torch

import seeded_inputs as si

TOL_O_ABS, TOL_O_REL, TOL_L_ABS, TOL_G_REL = 1e-2, 5e-3, 2e-3, 1e-2
TOL_D_REL = 1e-2  # D end to end (no bound is given for it; it follows from O's)
TOL_D_ELEM = 1e-3  # the preprocess step alone: |D - rowsum(dO * O)| <= 1e-3 * max(1, |D|)


def check_D_elementwise(D_gpu, O_gpu, dO):
    """The preprocess step against its definition on the GPU's own bf16 O: D_i =
    sum_k dO_ik O_ik in float64, element by element.  Returns the largest error
    relative to max(1, |D|)."""
    ref = (f64(dO) * f64(O_gpu)).sum(axis=-1)
    err = np.abs(f64(D_gpu) - ref) / np.maximum(1.0, np.abs(ref))
    worst = float(err.max()) if err.size else 0.0
    assert worst <= TOL_D_ELEM, f"D element-wise {worst:.3e}"
    return worst


def rel_frob(got, ref):
    return float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300))


def half_ulp_bf16(x):
    """Half the spacing of bf16 numbers at |x| (8 significant bits)."""
    ax = np.maximum(np.abs(x), np.finfo(np.float32).tiny)
    return np.ldexp(1.0, np.floor(np.log2(ax)).astype(np.int64) - 8)


def o_excess(got, ref):
    """max(|got - ref| - half a bf16 ulp of ref): the O error beyond output rounding."""
    return float((np.abs(got - ref) - half_ulp_bf16(ref)).max())


def stream():
    return torch.cuda.current_stream().cuda_stream


def lib():
    """The binding; imported here so that collecting GPU tests on a machine
    without the built library does not fail (they are skipped there)."""
    import exact_tiled_attention_26_gb300 as fa
    return fa


def run_gpu(Q, K, V, dO, causal, scale=None, counter=False, split=0, window=0, ws=None):
    """Forward + preprocess + backward through the C ABI (the general-mask entry
    points).  Inputs: bf16 CPU tensors Q, dO [B,H,Nq,d], K, V [B,H,Nk,d].  `split`
    selects the backward form (fa_debug_set_bwd_split; 0 = the library's default).
    `ws`: a device uint8 tensor to use as the backward's workspace, with whatever it
    holds (default: a new one).  Returns CPU tensors and (if asked) the tile-pair
    counts."""
    fa = lib()
    fa.check(fa.fa_debug_set_bwd_split(split))
    B, H, Nq, d = Q.shape
    Nk = K.shape[2]
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    dev = torch.device("cuda")
    q, k, v, do = (t.to(dev) for t in (Q, K, V, dO))
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=dev)
    D = torch.empty((B, H, Nq), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws_bytes = fa.fa_bwd_workspace_size_ex(B, H, Nq, Nk, d, causal, window)
    if ws is None:
        ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    assert ws.numel() >= ws_bytes
    cnt = torch.zeros(2, dtype=torch.int64, device=dev)
    s = stream()
    if counter:
        fa.check(fa.fa_debug_set_tile_counter(cnt.data_ptr()))
    try:
        fa.check(fa.fa_fwd_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, Nq, Nk, d,
                              causal, window, scale, s), "fa_fwd_ex")
        if counter:
            fa.check(fa.fa_debug_set_tile_counter(cnt.data_ptr() + 8))
        fa.check(fa.fa_bwd_preprocess(o.data_ptr(), do.data_ptr(), D.data_ptr(), B, H, Nq, d, s), "preprocess")
        fa.check(fa.fa_bwd_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(), lse.data_ptr(),
                              D.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, Nq, Nk, d, causal, window,
                              scale, ws.data_ptr(), ws.numel(), s), "fa_bwd_ex")
    finally:
        fa.fa_debug_set_bwd_split(0)
        if counter:
            fa.fa_debug_set_tile_counter(None)
    st, detail = fa.fa_poll_device_error(s)
    fa.check(st, f"device status word (site {detail:#x})")
    out = {"O": o, "L": lse, "D": D, "dQ": dq, "dK": dk, "dV": dv}
    out = {n: t.cpu() for n, t in out.items()}
    if counter:
        out["tiles"] = cnt.cpu().tolist()
    return out


def assert_close(got: dict, ref: dict, label=""):
    """got/ref: dicts of float64 arrays with keys among O, L, dQ, dK, dV."""
    msgs = []
    errs = {}
    if "O" in ref:
        ea, ex, er = float(np.abs(got["O"] - ref["O"]).max()), o_excess(got["O"], ref["O"]), rel_frob(got["O"], ref["O"])
        errs.update(O_max_abs=ea, O_beyond_half_ulp=ex, O_rel=er)
        if not (ex <= TOL_O_ABS and er <= TOL_O_REL):
            i = np.unravel_index(np.argmax(np.abs(got["O"] - ref["O"])), ref["O"].shape)
            msgs.append(f"O max-abs {ea:.3e} (beyond output rounding {ex:.3e}, at ref {ref['O'][i]:.4f}) rel {er:.3e}")
    if "L" in ref:
        ea = float(np.abs(got["L"] - ref["L"]).max())
        errs["L_max_abs"] = ea
        if not ea <= TOL_L_ABS:
            msgs.append(f"L max-abs {ea:.3e}")
    if "D" in ref:  # end to end: D from the GPU's own O, against the oracle's D
        ea, er = float(np.abs(got["D"] - ref["D"]).max()), rel_frob(got["D"], ref["D"])
        errs.update(D_max_abs=ea, D_rel=er)
        if not er <= TOL_D_REL:
            msgs.append(f"D rel {er:.3e}")
    for n in ("dQ", "dK", "dV"):
        if n in ref:
            if np.linalg.norm(ref[n]) <= 1e-9:
                rms = float(np.sqrt(np.mean(got[n] ** 2)))
                errs[f"{n}_rms"] = rms
                if not rms <= 1e-4:
                    msgs.append(f"{n} (exactly zero) rms {rms:.3e}")
                continue
            er = rel_frob(got[n], ref[n])
            errs[f"{n}_rel"] = er
            if not er <= TOL_G_REL:
                msgs.append(f"{n} rel {er:.3e}")
    log = os.environ.get("FA_PARITY_LOG")
    if log:  # measured errors, one JSON line per comparison, for the record of a run
        with open(log, "a") as f:
            f.write(json.dumps({"case": label, "pass": not msgs, "errs": errs}) + "\n")
    assert not msgs, f"{label}: " + "; ".join(msgs)
    return errs


def f64(t):
    return si.to_f64(t)
